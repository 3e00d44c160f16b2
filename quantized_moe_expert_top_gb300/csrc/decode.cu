// Few-token (decode) path of the routed-MoE layer: memory-bound GEMVs over
// the routed experts' MXFP4 weights.
//
// Each CTA owns a contiguous run of weight rows of the touched experts and
// streams them through a shared-memory ring: one thread issues bulk copies
// (cp.async.bulk, whole interleaved rows: codes and their E8M0 scales) several
// stages ahead, so many kilobytes per SM are always in flight; eight consumer
// warps each take one row (gate/up: one gate+up row pair) per stage.  A
// consumer lane reads 16-byte chunks (one 32-element MXFP4 block each),
// converts the E2M1 codes to f16 in registers with the hardware e2m1x2
// conversion, multiplies by the activations, scales each block's partial sum
// by its E8M0 scale, and the warp reduces its lanes with shuffles.
//
//   gate/up : x arrives as f16 with a per-token power-of-two prescale (made by
//             the top-k kernel); f16 x f16 products are exact in the fp32
//             mixed-precision FMA, so x enters exactly.  h = SwiGLU(g, u) is
//             stored in fp32.
//   down    : h is used in fp32 (weights converted f16 -> f32); the weighted
//             combine red-adds w[t,j] * y into out[t], which the gate/up kernel
//             zeroed.
// Activations are read through L1 (every warp of an SM reads the same few
// token rows).  Every mbarrier wait is bounded (see the prefill GEMM).
//
// Pages: "DwarfStar実地分析" §GGUFの対応範囲は意図的に狭い (MXFP4 routed experts);
// "284B MoEを128GBノートPCに詰め込む" §プリフィル790 t/sが暴く真のボトルネック
// (generation is memory-bandwidth bound).
#include "common.cuh"
#include "internal.h"

namespace ds4moe {
namespace {

constexpr int kNT = 8;            // tokens per pass over a row
constexpr int kConsumers = 8;     // consumer warps
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kRingBytes = 200 * 1024;
constexpr int kMaxStages = 8;
constexpr int kDnRowsPerWarp = 4;

__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  if (b == 0u) return __int_as_float(0x00400000);  // 2^-127
  if (b == 255u) return __int_as_float(0x7FC00000);
  return __int_as_float((int)(b << 23));
}

__device__ __forceinline__ uint4 ldg_l1(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// Index of h[pair][i] in the piece-transposed fp32 layout the down kernel
// reads: 16-byte piece j (4 floats) of 32-element block c at (j * f/32 + c).
__device__ __forceinline__ size_t h_index(int pair, int i, int f) {
  const int c = i >> 5, j = (i >> 2) & 7;
  return (size_t)pair * f + ((size_t)j * (f >> 5) + c) * 4 + (i & 3);
}

struct Ring {
  uint8_t* buf;
  uint64_t* full;
  uint64_t* empty;
  int stages, stage_bytes;
};

// Producer: stage s of this CTA holds rows [r0 + s*rps, r0 + (s+1)*rps) of the
// global row list (clipped to r1); row r lives at base + grow(r) * pitch where
// consecutive rows of one expert are consecutive in memory.
// With `twin` set every row has a twin `twin_off` bytes further in global
// memory (the up row of a gate row); twins land rps rows after the rows in the
// stage.
template <typename RowAddr>
__device__ void produce(const Ring& R, int r0, int r1, int rps, int pitch, RowAddr row_addr, bool twin,
                        size_t twin_off, uint64_t budget, DeviceStatus* status, volatile int* abort_flag) {
  const int nst = (r1 - r0 + rps - 1) / rps;
  uint32_t issued = 0, parity = 0;
  for (int s = 0; s < nst; ++s) {
    const int slot = s % R.stages;
    const uint32_t ph = (uint32_t)(s / R.stages) & 1u;
    if (!mbar_wait_bounded(&R.empty[slot], ph ^ 1u, budget, abort_flag)) {
      report_timeout(status, kWhereProducerEmpty);
      *abort_flag = 1;
      break;
    }
    const int a = r0 + s * rps, b = min(a + rps, r1);
    mbar_arrive_expect_tx(&R.full[slot], (uint32_t)((b - a) * pitch * (twin ? 2 : 1)));
    uint8_t* dst = R.buf + slot * R.stage_bytes;
    int seg = a;
    while (seg < b) {  // contiguous segments (a block or expert boundary breaks a stage)
      const uint8_t* src = row_addr(seg);
      int end = seg + 1;
      while (end < b && row_addr(end) == src + (size_t)(end - seg) * pitch) ++end;
      bulk_load(dst + (size_t)(seg - a) * pitch, src, (uint32_t)((end - seg) * pitch), &R.full[slot]);
      if (twin)
        bulk_load(dst + (size_t)(rps + seg - a) * pitch, src + twin_off, (uint32_t)((end - seg) * pitch),
                  &R.full[slot]);
      seg = end;
    }
    issued |= 1u << slot;
    parity = (parity & ~(1u << slot)) | (ph << slot);
  }
  if (*abort_flag) {
    for (int slot = 0; slot < R.stages; ++slot)
      if ((issued >> slot) & 1u) {
        volatile int never = 0;
        mbar_wait_bounded(&R.full[slot], (parity >> slot) & 1u, budget, &never);
      }
  }
}

// Consumer side of one stage: wait (lane 0, bounded) and broadcast the outcome.
__device__ __forceinline__ bool consume_wait(const Ring& R, int s, uint64_t budget, DeviceStatus* status,
                                             volatile int* abort_flag) {
  uint32_t ok = 0;
  if ((threadIdx.x & 31) == 0) {
    ok = mbar_wait_bounded(&R.full[s % R.stages], (uint32_t)(s / R.stages) & 1u, budget, abort_flag) ? 1u : 0u;
    if (!ok) {
      report_timeout(status, kWhereMmaFull);
      *abort_flag = 1;
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void consume_release(const Ring& R, int s) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&R.empty[s % R.stages]);
}

__device__ __forceinline__ void cta_range(int total, int& r0, int& r1) {
  const int per = (total + gridDim.x - 1) / gridDim.x;
  r0 = min((int)blockIdx.x * per, total);
  r1 = min(r0 + per, total);
}

__device__ Ring setup_ring(uint8_t* smem_raw, int stage_bytes) {
  Ring R;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  R.stages = min(kMaxStages, kRingBytes / stage_bytes);
  R.stage_bytes = stage_bytes;
  R.full = reinterpret_cast<uint64_t*>(base);
  R.empty = R.full + kMaxStages;
  R.buf = base + 256;
  if (threadIdx.x == 0) {
    for (int i = 0; i < R.stages; ++i) {
      mbar_init(&R.full[i], 1);
      mbar_init(&R.empty[i], kConsumers);
    }
    fence_barrier_init();
  }
  __syncthreads();
  return R;
}

// ------------------------------------------------------------------ gate/up
// Rows = every (gate row i, up row i) pair of every touched expert; stage =
// kConsumers gate rows then their kConsumers up rows, one pair per consumer
// warp.  In the tile-major weight layout gate row i of expert e is row
// (e*f/64 + i/64)*128 + i%64, its up row 64 rows later.
__global__ void __launch_bounds__(kThreads, 1) decode_gateup_kernel(
    const uint8_t* __restrict__ gu, int pitch, const uint4* __restrict__ xh, const float* __restrict__ xsig,
    float* __restrict__ out, int T, int d, int f, const int32_t* __restrict__ touched,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm_tok, float* __restrict__ h_dec, int E,
    DeviceStatus* status, uint64_t budget) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_s;
  volatile int* abort_flag = &abort_s;
  if (threadIdx.x == 0) abort_s = 0;
  {  // zero out[T][d] for the down kernel's accumulation
    float4* o4 = reinterpret_cast<float4*>(out);
    const size_t n4 = (size_t)T * d / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
      o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const Ring R = setup_ring(smem_raw, 2 * kConsumers * pitch);
  int r0, r1;
  cta_range(touched[E] * f, r0, r1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    if (lane == 0)
      produce(
          R, r0, r1, kConsumers, pitch,
          [&](int r) {
            const int i = r % f;
            return gu + (((size_t)__ldg(touched + r / f) * (f / 64) + i / 64) * 128 + i % 64) * pitch;
          },
          true, (size_t)64 * pitch, budget, status, abort_flag);
    return;
  }
  const int cw = warp - 1;
  const int nblk = d / 32;
  const int nst = (r1 - r0 + kConsumers - 1) / kConsumers;
  for (int s = 0; s < nst; ++s) {
    if (!consume_wait(R, s, budget, status, abort_flag)) return;
    const int rp = r0 + s * kConsumers + cw;
    if (rp < r1) {
      const uint8_t* row = R.buf + (s % R.stages) * R.stage_bytes + cw * pitch;
      const uint8_t* urow = row + kConsumers * pitch;
      const int e = __ldg(touched + rp / f), i = rp % f;
      const int p0 = __ldg(offsets + e), ne = __ldg(offsets + e + 1) - p0;
      for (int tg = 0; tg < ne; tg += kNT) {
        const int nt = min(kNT, ne - tg);
        const int my_tok = lane < nt ? __ldg(perm_tok + p0 + tg + lane) : 0;
        int toks[kNT];
        float ag[kNT], au[kNT];
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) {
          toks[tt] = __shfl_sync(0xffffffffu, my_tok, tt);  // warp converged here
          ag[tt] = au[tt] = 0.f;
        }
        for (int c = lane; c < nblk; c += 32) {
          const uint4 gq = lds128(row + 16 * c), uq = lds128(urow + 16 * c);
          const float sg = e8m0_to_f32(row[d / 2 + c]), su = e8m0_to_f32(urow[d / 2 + c]);
          uint32_t wg[16], wu[16];
          const uint32_t g4[4] = {gq.x, gq.y, gq.z, gq.w}, u4[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            wg[b] = e2m1x2_to_f16x2((g4[b >> 2] >> (8 * (b & 3))) & 0xFFu);
            wu[b] = e2m1x2_to_f16x2((u4[b >> 2] >> (8 * (b & 3))) & 0xFFu);
          }
#pragma unroll
          for (int tt = 0; tt < kNT; ++tt) {
            if (tt < nt) {
              const uint4* xr = xh + (size_t)toks[tt] * (d / 8);
              float pg = 0.f, pu = 0.f;
#pragma unroll
              for (int pq = 0; pq < 4; ++pq) {
                const uint4 xv = ldg_l1(xr + pq * nblk + c);
                pg = dot2_f16_f32(wg[4 * pq + 0], xv.x, pg);
                pg = dot2_f16_f32(wg[4 * pq + 1], xv.y, pg);
                pg = dot2_f16_f32(wg[4 * pq + 2], xv.z, pg);
                pg = dot2_f16_f32(wg[4 * pq + 3], xv.w, pg);
                pu = dot2_f16_f32(wu[4 * pq + 0], xv.x, pu);
                pu = dot2_f16_f32(wu[4 * pq + 1], xv.y, pu);
                pu = dot2_f16_f32(wu[4 * pq + 2], xv.z, pu);
                pu = dot2_f16_f32(wu[4 * pq + 3], xv.w, pu);
              }
              ag[tt] = fmaf(pg, sg, ag[tt]);
              au[tt] = fmaf(pu, su, au[tt]);
            }
          }
        }
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) {
          if (tt < nt) {
            const float sig = __ldg(xsig + toks[tt]);
            const float g = warp_sum(ag[tt]) * sig;
            const float u = warp_sum(au[tt]) * sig;
            if (lane == tt) h_dec[h_index(p0 + tg + tt, i, f)] = __fdividef(g, 1.f + __expf(-g)) * u;
          }
        }
      }
    }
    consume_release(R, s);
  }
}

// ------------------------------------------------------------------ down
// Rows = every output row of every touched expert (one dn row each); stage =
// kConsumers * 4 rows, four per consumer warp.
__global__ void __launch_bounds__(kThreads, 1) decode_down_kernel(
    const uint8_t* __restrict__ dn, int pitch, float* __restrict__ out, int d, int f, int k,
    const int32_t* __restrict__ touched, const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm_tok,
    const int32_t* __restrict__ perm_slot, const float* __restrict__ topk_w, const float* __restrict__ h_dec, int E,
    DeviceStatus* status, uint64_t budget) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_s;
  volatile int* abort_flag = &abort_s;
  if (threadIdx.x == 0) abort_s = 0;
  constexpr int rps = kConsumers * kDnRowsPerWarp;
  const Ring R = setup_ring(smem_raw, rps * pitch);
  int r0, r1;
  cta_range(touched[E] * d, r0, r1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    if (lane == 0)
      produce(R, r0, r1, rps, pitch, [&](int r) { return dn + ((size_t)__ldg(touched + r / d) * d + r % d) * pitch; },
              false, 0, budget, status, abort_flag);
    return;
  }
  const int cw = warp - 1;
  const int nblk = f / 32;
  const int nst = (r1 - r0 + rps - 1) / rps;
  for (int s = 0; s < nst; ++s) {
    if (!consume_wait(R, s, budget, status, abort_flag)) return;
    const uint8_t* stage = R.buf + (s % R.stages) * R.stage_bytes;
#pragma unroll 1
    for (int rr = 0; rr < kDnRowsPerWarp; ++rr) {
      const int r = r0 + s * rps + cw * kDnRowsPerWarp + rr;
      if (r >= r1) break;
      const uint8_t* row = stage + (cw * kDnRowsPerWarp + rr) * pitch;
      const int e = __ldg(touched + r / d), m = r % d;
      const int p0 = __ldg(offsets + e), ne = __ldg(offsets + e + 1) - p0;
      for (int tg = 0; tg < ne; tg += kNT) {
        const int nt = min(kNT, ne - tg);
        float acc[kNT];
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) acc[tt] = 0.f;
        for (int c = lane; c < nblk; c += 32) {
          const uint4 cq = lds128(row + 16 * c);
          const float sc = e8m0_to_f32(row[f / 2 + c]);
          float wf[32];
          const uint32_t c4[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const uint32_t h2 = e2m1x2_to_f16x2((c4[b >> 2] >> (8 * (b & 3))) & 0xFFu);
            const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h2));
            wf[2 * b] = v.x;
            wf[2 * b + 1] = v.y;
          }
#pragma unroll
          for (int tt = 0; tt < kNT; ++tt) {
            if (tt < nt) {
              const float* hp = h_dec + (size_t)(p0 + tg + tt) * f;
              float p = 0.f;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint4 hv4 = ldg_l1(hp + ((size_t)j * nblk + c) * 4);
                p = fmaf(wf[4 * j + 0], __uint_as_float(hv4.x), p);
                p = fmaf(wf[4 * j + 1], __uint_as_float(hv4.y), p);
                p = fmaf(wf[4 * j + 2], __uint_as_float(hv4.z), p);
                p = fmaf(wf[4 * j + 3], __uint_as_float(hv4.w), p);
              }
              acc[tt] = fmaf(p, sc, acc[tt]);
            }
          }
        }
#pragma unroll
        for (int tt = 0; tt < kNT; ++tt) {
          if (tt < nt) {
            const float y = warp_sum(acc[tt]);
            if (lane == 0) {
              const int p = p0 + tg + tt;
              const int t = __ldg(perm_tok + p);
              red_add_f32(out + (size_t)t * d + m, __ldg(topk_w + (size_t)t * k + __ldg(perm_slot + p)) * y);
            }
          }
        }
      }
    }
    consume_release(R, s);
  }
}

size_t ring_smem(int stage_bytes) {
  const int stages = kRingBytes / stage_bytes < kMaxStages ? kRingBytes / stage_bytes : kMaxStages;
  return 128 + 256 + (size_t)stages * stage_bytes;
}

}  // namespace

cudaError_t launch_decode_gateup(const ds4moe_layer* L, const void* x, float* out, int T, cudaStream_t st) {
  (void)x;
  const int d = L->cfg.d_model, f = L->cfg.d_ff, E = L->cfg.n_experts;
  const size_t smem = ring_smem(2 * kConsumers * L->w.pitch_gu);
  cudaError_t e = cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_gateup_kernel, L->num_sms, kThreads, smem, st, L->w.gu, L->w.pitch_gu,
                    reinterpret_cast<const uint4*>(L->s.xh), L->s.xsig, out, T, d, f, L->s.touched, L->s.offsets,
                    L->s.perm_tok, L->s.h_dec, E, L->status, (uint64_t)L->cfg.wait_timeout_ms * 1000000ull);
}

cudaError_t launch_decode_down(const ds4moe_layer* L, float* out, int T, cudaStream_t st) {
  (void)T;
  const int d = L->cfg.d_model, f = L->cfg.d_ff, E = L->cfg.n_experts, k = L->cfg.top_k;
  const size_t smem = ring_smem(kConsumers * kDnRowsPerWarp * L->w.pitch_dn);
  cudaError_t e = cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_down_kernel, L->num_sms, kThreads, smem, st, L->w.dn, L->w.pitch_dn, out, d, f, k,
                    L->s.touched, L->s.offsets, L->s.perm_tok, L->s.perm_slot, L->s.topk_w, L->s.h_dec, E, L->status,
                    (uint64_t)L->cfg.wait_timeout_ms * 1000000ull);
}


}  // namespace ds4moe
