// Few-token (decode) path of the routed-MoE layer: memory-bound GEMVs over
// the routed experts' MXFP4 weights.
//
// Each warp streams whole weight rows with 128-bit non-coherent loads (one
// 16-byte chunk = one 32-element MXFP4 block per lane and step), converts the
// E2M1 codes to f16 in registers with the hardware e2m1x2 conversion, and
// accumulates f16 x f16 products in fp32 (mixed-precision FMA; the products
// are exact).  The per-block E8M0 scale multiplies each block's partial sum.
// Lanes are then reduced with shuffles.
//
// Activations enter as f16 with a power-of-two prescale per row (so any bf16 /
// fp32 magnitude maps into f16's range without overflow; the scale is undone
// exactly on the fp32 result).  x is exact in f16 after prescaling (bf16 has 8
// significant bits); h loses only its bits beyond f16's 11.
//
// Pages: "DwarfStar実地分析" §GGUFの対応範囲は意図的に狭い (MXFP4 routed experts);
// "284B MoEを128GBノートPCに詰め込む" §プリフィル790 t/sが暴く真のボトルネック
// (generation is memory-bandwidth bound).
#include "common.cuh"
#include "internal.h"

namespace ds4moe {
namespace {

constexpr int kNT = 8;           // tokens per pass (activations staged in shared memory)
constexpr int kThreads = 256;    // 8 warps
constexpr int kGateUpRowsPerItem = 8;   // row pairs per work item (one per warp)
constexpr int kDownRowsPerWarp = 4;
constexpr int kDownRowsPerItem = kDownRowsPerWarp * (kThreads / 32);

__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  if (b == 0u) return __int_as_float(0x00400000);  // 2^-127
  if (b == 255u) return __int_as_float(0x7FC00000);
  return __int_as_float((int)(b << 23));
}

// Shared-memory layout of one staged activation row of K elements as f16:
// 16-byte piece q (elements 8q'..8q'+7 of 32-element block c, q' = 0..3) sits at
// piece index q'*nblk + c, so lane l reading block c = l + 32i hits
// consecutive 16-byte words (no bank conflicts).
__device__ __forceinline__ int piece_index(int c, int q, int nblk) { return q * nblk + c; }

// Stage `nt` activation rows into shared memory as prescaled f16.
// src(row r) is bf16 (is_bf16) or fp32; element offset row_off(tt).
template <bool kBf16>
__device__ void stage_rows(const void* __restrict__ src, const int32_t* __restrict__ rows, int nt, int K,
                           uint4* __restrict__ xs, float* __restrict__ sig) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nblk = K / 32;
  for (int tt = wid; tt < nt; tt += kThreads / 32) {
    const size_t r = (size_t)rows[tt];
    // pass 1: amax over the row
    float amax = 0.f;
    if (kBf16) {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + r * K);
      for (int i = lane; i < K / 8; i += 32) {
        const uint4 v = __ldg(p + i);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          amax = fmaxf(amax, fabsf(__uint_as_float(wv[q] << 16)));
          amax = fmaxf(amax, fabsf(__uint_as_float(wv[q] & 0xFFFF0000u)));
        }
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + r * K);
      for (int i = lane; i < K / 4; i += 32) {
        const float4 v = p[i];
        amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v.x)), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
      }
    }
    amax = warp_max(amax);
    const int s = f16_prescale_exp(amax);
    const float inv = exp2i(-s);
    if (lane == 0) sig[tt] = exp2i(s);
    // pass 2: convert, 8 elements (one 16-byte piece of f16) per step
    uint4* dst = xs + (size_t)tt * (K / 8);
    for (int i = lane; i < K / 8; i += 32) {
      float f[8];
      if (kBf16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + r * K) + i);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[2 * q] = __uint_as_float(wv[q] << 16);
          f[2 * q + 1] = __uint_as_float(wv[q] & 0xFFFF0000u);
        }
      } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + r * K);
        const float4 a = p[2 * i], b = p[2 * i + 1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      }
      uint32_t h[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 hv = __floats2half2_rn(f[2 * q] * inv, f[2 * q + 1] * inv);
        h[q] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      const int c = i >> 2, q = i & 3;  // block c, piece q
      dst[piece_index(c, q, nblk)] = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

// Dot products of R weight rows (MXFP4, K elements each) with nt staged
// activation rows.  acc[r][tt] receives lane-partial sums (reduce afterwards).
template <int R, int CPL>
__device__ __forceinline__ void rows_dot(const uint8_t* const (&codes)[R], const uint8_t* const (&scales)[R],
                                         int nblk, const uint4* __restrict__ xs, int nt,
                                         float (&acc)[R][kNT]) {
  const int lane = threadIdx.x & 31;
  const int xstride = nblk * 4;  // uint4 pieces per staged row
  for (int c0 = 0; c0 < nblk; c0 += 32 * CPL) {
    uint4 cw[R][CPL];
    uint32_t sb[R][CPL];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int q = 0; q < CPL; ++q) {
        const int c = c0 + lane + 32 * q;
        if (c < nblk) {
          cw[r][q] = ldg_nc_v4(codes[r] + (size_t)c * 16);
          sb[r][q] = __ldg(scales[r] + c);
        } else {
          cw[r][q] = make_uint4(0, 0, 0, 0);
          sb[r][q] = 127u;
        }
      }
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int c = c0 + lane + 32 * q;
      if (c >= nblk) break;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        uint32_t wh[16];
        const uint32_t words[4] = {cw[r][q].x, cw[r][q].y, cw[r][q].z, cw[r][q].w};
#pragma unroll
        for (int b = 0; b < 16; ++b) wh[b] = e2m1x2_to_f16x2((words[b >> 2] >> (8 * (b & 3))) & 0xFFu);
        const float sc = e8m0_to_f32(sb[r][q]);
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) {
          if (tt < nt) {
            float p = 0.f;
#pragma unroll
            for (int pq = 0; pq < 4; ++pq) {
              const uint4 xv = xs[(size_t)tt * xstride + piece_index(c, pq, nblk)];
              p = dot2_f16_f32(wh[4 * pq + 0], xv.x, p);
              p = dot2_f16_f32(wh[4 * pq + 1], xv.y, p);
              p = dot2_f16_f32(wh[4 * pq + 2], xv.z, p);
              p = dot2_f16_f32(wh[4 * pq + 3], xv.w, p);
            }
            acc[r][tt] = fmaf(p, sc, acc[r][tt]);
          }
        }
      }
    }
  }
}

// Gate/up + SwiGLU.  Work item = (touched expert, block of 8 row pairs); one
// warp per row pair (gate row i and up row i of the expert).  Also zeroes `out`
// for the down kernel's weighted accumulation.
__global__ void __launch_bounds__(kThreads) decode_gateup_kernel(
    const uint8_t* __restrict__ gate_codes, const uint8_t* __restrict__ gate_scales,
    const uint8_t* __restrict__ up_codes, const uint8_t* __restrict__ up_scales, const void* __restrict__ x,
    float* __restrict__ out, int T, int d, int f, const int32_t* __restrict__ touched,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm_tok, float* __restrict__ h_dec, int E) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* xs = reinterpret_cast<uint4*>(smem);
  __shared__ float sig[kNT];
  __shared__ int32_t rows[kNT];

  {  // zero out[T][d]
    float4* o4 = reinterpret_cast<float4*>(out);
    const size_t n4 = (size_t)T * d / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
      o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int n_touched = touched[E];
  const int nblk_items = f / kGateUpRowsPerItem;
  const int nitems = n_touched * nblk_items;
  const int nblk = d / 32;
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int e = touched[item / nblk_items];
    const int i = (item % nblk_items) * kGateUpRowsPerItem + wid;
    const int p0 = offsets[e], ne = offsets[e + 1] - p0;
    const size_t grow = (size_t)e * f + i;
    const uint8_t* const codes[2] = {gate_codes + grow * (d / 2), up_codes + grow * (d / 2)};
    const uint8_t* const scales[2] = {gate_scales + grow * (d / 32), up_scales + grow * (d / 32)};
    for (int tg = 0; tg < ne; tg += kNT) {
      const int nt = min(kNT, ne - tg);
      __syncthreads();  // previous users of xs / rows are done
      if (threadIdx.x < nt) rows[threadIdx.x] = perm_tok[p0 + tg + threadIdx.x];
      __syncthreads();
      stage_rows<true>(x, rows, nt, d, xs, sig);
      __syncthreads();
      float acc[2][kNT];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) acc[r][tt] = 0.f;
      rows_dot<2, 4>(codes, scales, nblk, xs, nt, acc);
#pragma unroll
      for (int tt = 0; tt < kNT; ++tt) {
        if (tt < nt) {
          const float g = warp_sum(acc[0][tt]) * sig[tt];
          const float u = warp_sum(acc[1][tt]) * sig[tt];
          if (lane == tt) h_dec[(size_t)(p0 + tg + tt) * f + i] = g / (1.f + expf(-g)) * u;
        }
      }
    }
  }
}

// Down projection + weighted combine.  Work item = (touched expert, block of
// 32 output rows); each warp handles 4 rows at once and red-adds
// w[t,j] * y into out[t] (zeroed by the gate/up kernel).
__global__ void __launch_bounds__(kThreads) decode_down_kernel(
    const uint8_t* __restrict__ down_codes, const uint8_t* __restrict__ down_scales, float* __restrict__ out,
    int d, int f, int k, const int32_t* __restrict__ touched, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ perm_tok, const int32_t* __restrict__ perm_slot, const float* __restrict__ topk_w,
    const float* __restrict__ h_dec, int E) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* hs = reinterpret_cast<uint4*>(smem);
  __shared__ float sig[kNT];
  __shared__ int32_t rows[kNT];
  __shared__ float wt[kNT];
  __shared__ int32_t tok[kNT];

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int n_touched = touched[E];
  const int nblk_items = d / kDownRowsPerItem;
  const int nitems = n_touched * nblk_items;
  const int nblk = f / 32;
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int e = touched[item / nblk_items];
    const int m0 = (item % nblk_items) * kDownRowsPerItem + wid * kDownRowsPerWarp;
    const int p0 = offsets[e], ne = offsets[e + 1] - p0;
    const uint8_t* codes[kDownRowsPerWarp];
    const uint8_t* scales[kDownRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kDownRowsPerWarp; ++r) {
      const size_t grow = (size_t)e * d + m0 + r;
      codes[r] = down_codes + grow * (f / 2);
      scales[r] = down_scales + grow * (f / 32);
    }
    for (int tg = 0; tg < ne; tg += kNT) {
      const int nt = min(kNT, ne - tg);
      __syncthreads();
      if (threadIdx.x < nt) {
        const int p = p0 + tg + threadIdx.x;
        const int t = perm_tok[p];
        rows[threadIdx.x] = p;
        tok[threadIdx.x] = t;
        wt[threadIdx.x] = topk_w[(size_t)t * k + perm_slot[p]];
      }
      __syncthreads();
      stage_rows<false>(h_dec, rows, nt, f, hs, sig);
      __syncthreads();
      float acc[kDownRowsPerWarp][kNT];
#pragma unroll
      for (int r = 0; r < kDownRowsPerWarp; ++r)
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) acc[r][tt] = 0.f;
      rows_dot<kDownRowsPerWarp, 2>(codes, scales, nblk, hs, nt, acc);
#pragma unroll
      for (int r = 0; r < kDownRowsPerWarp; ++r)
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) {
          if (tt < nt) {
            const float y = warp_sum(acc[r][tt]) * sig[tt];
            if (lane == tt) red_add_f32(out + (size_t)tok[tt] * d + m0 + r, wt[tt] * y);
          }
        }
    }
  }
}

}  // namespace

static int grid_for(const ds4moe_layer* L, const void* kernel, size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return L->num_sms * per_sm;
}

cudaError_t launch_decode_gateup(const ds4moe_layer* L, const void* x, float* out, int T, cudaStream_t st) {
  const int d = L->cfg.d_model, f = L->cfg.d_ff, E = L->cfg.n_experts;
  const size_t smem = (size_t)kNT * d * 2;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_set = true;
  }
  const int grid = grid_for(L, (const void*)decode_gateup_kernel, smem);
  decode_gateup_kernel<<<grid, kThreads, smem, st>>>(L->w.gate_codes, L->w.gate_scales, L->w.up_codes,
                                                     L->w.up_scales, x, out, T, d, f, L->s.touched, L->s.offsets,
                                                     L->s.perm_tok, L->s.h_dec, E);
  return cudaGetLastError();
}

cudaError_t launch_decode_down(const ds4moe_layer* L, float* out, int T, cudaStream_t st) {
  (void)T;
  const int d = L->cfg.d_model, f = L->cfg.d_ff, E = L->cfg.n_experts, k = L->cfg.top_k;
  const size_t smem = (size_t)kNT * f * 2;
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    attr_set = true;
  }
  const int grid = grid_for(L, (const void*)decode_down_kernel, smem);
  decode_down_kernel<<<grid, kThreads, smem, st>>>(L->w.down_codes, L->w.down_scales, out, d, f, k, L->s.touched,
                                                   L->s.offsets, L->s.perm_tok, L->s.perm_slot, L->s.topk_w,
                                                   L->s.h_dec, E);
  return cudaGetLastError();
}

int decode_launches() { return 4; }

}  // namespace ds4moe
