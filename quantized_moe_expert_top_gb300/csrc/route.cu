// Routing of the routed-MoE layer: top-k selection with softmax over the
// selected logits, then a deterministic grouping of the (token, slot) pairs
// by expert.
//
// The pages ("DwarfStar実地分析", §GGUFの対応範囲は意図的に狭い) say only that the
// routing itself stays at original precision; the rule implemented here is the
// layer's specification: the k largest fp32 logits per token ordered by
// (value desc, expert index asc), weights = softmax over those k only.
#include "common.cuh"
#include "gemm.cuh"
#include "internal.h"

#include <math.h>

#include <mutex>

namespace ds4moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kMaxK = 8;

// One warp per token.  Lane l holds logits l, l+32, ..., so a lane's own
// entries are in increasing index order.
//
// For the decode path the same warp also prepares the token's activations: x
// as f16 with a power-of-two prescale s (amax * 2^-s lands in [2^14, 2^15), so
// every bf16 value is exact or below f16's subnormal floor), stored in the
// piece-transposed order the decode GEMV reads (16-byte piece q of 32-element
// block c at index q * d/32 + c), and 2^s in xsig[token].
__device__ __forceinline__ void prepare_x_f16(const __nv_bfloat16* __restrict__ x, int token, int d,
                                              uint4* __restrict__ xh, float* __restrict__ xsig, int lane) {
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)token * d);
  const int npieces = d / 8, nblk = d / 32;
  float amax = 0.f;
  for (int i = lane; i < npieces; i += 32) {
    const uint4 v = __ldg(src + i);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wv[q] << 16)), fabsf(__uint_as_float(wv[q] & 0xFFFF0000u))));
  }
  amax = warp_max(amax);
  const int s = f16_prescale_exp(amax);
  const float inv = exp2i(-s);
  if (lane == 0) xsig[token] = exp2i(s);
  uint4* dst = xh + (size_t)token * npieces;
  for (int i = lane; i < npieces; i += 32) {
    const uint4 v = __ldg(src + i);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 hv =
          __floats2half2_rn(__uint_as_float(wv[q] << 16) * inv, __uint_as_float(wv[q] & 0xFFFF0000u) * inv);
      h[q] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    dst[(i & 3) * nblk + (i >> 2)] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// Order key of a logit: unsigned comparison of keys is the comparison of the
// values, with -0 taken as +0 and NaN as -inf (outside the layer's domain).
// Every key is above 0, which marks "no candidate".
__device__ __forceinline__ uint32_t logit_key(float x) {
  if (x != x) x = -INFINITY;
  if (x == 0.f) x = 0.f;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token's logits by one warp (lane l holds entries l, l+32, ...,
// so a lane's own entries are in increasing index order); lane 0 writes the k
// expert indices (value desc, index asc) and their softmax weights to idx[0..k)
// and w[0..k), and the indices also to sidx[0..k) when sidx is given.  Each of
// the k rounds takes the warp's largest key with one redux.sync and, among the
// lanes holding it, the smallest index with a second.
__device__ __forceinline__ void topk_warp(const float* __restrict__ row, int E, int k, int lane,
                                          int32_t* __restrict__ idx, float* __restrict__ w, int* sidx = nullptr) {
  float v[kMaxE / 32];
  uint32_t key[kMaxE / 32];
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    const int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      x = __ldg(row + e);
      if (x != x) x = -INFINITY;
    }
    v[i] = x;
    key[i] = e < E ? logit_key(x) : 0u;  // entries beyond E are never candidates
  }

  float sel_v[kMaxK];
  int sel_e[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) {
      uint32_t bk = 0;
      float bv = -INFINITY;
      uint32_t be = 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i)
        if (key[i] > bk) {  // strict: among equal keys the lane's lower index stays
          bk = key[i];
          bv = v[i];
          be = (uint32_t)(lane + 32 * i);
        }
      const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
      const uint32_t we = __reduce_min_sync(0xffffffffu, bk == wk ? be : 0xFFFFFFFFu);
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i)  // the winner is taken (unrolled: key stays in registers)
        if (we == (uint32_t)(lane + 32 * i)) key[i] = 0u;
      sel_v[j] = __shfl_sync(0xffffffffu, bv, (int)(we & 31u));
      sel_e[j] = (int)we;
    }
  }

  if (lane == 0) {
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) z += expf(sel_v[j] - sel_v[0]);
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        idx[j] = sel_e[j];
        w[j] = expf(sel_v[j] - sel_v[0]) / z;
        if (sidx) sidx[j] = sel_e[j];
      }
    }
  }
}

__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int lds, int T, int E, int k,
                                                         int32_t* __restrict__ idx, float* __restrict__ w,
                                                         const __nv_bfloat16* __restrict__ x, int d,
                                                         uint4* __restrict__ xh, float* __restrict__ xsig) {
  pdl_wait();
  pdl_launch_dependents();
  const int token = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= T) return;
  if (xh != nullptr) prepare_x_f16(x, token, d, xh, xsig, lane);
  topk_warp(logits + (size_t)token * lds, E, k, lane, idx + (size_t)token * k, w + (size_t)token * k);
}

// Inclusive scan of one int per thread over a 256-thread block.
__device__ __forceinline__ int block_scan_incl(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int t = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    if (lane < (int)(blockDim.x >> 5)) warp_tot[lane] = t;
  }
  __syncthreads();
  const int add = wid > 0 ? warp_tot[wid - 1] : 0;
  __syncthreads();
  return v + add;
}

// Grid = E blocks of 256 threads; block e places expert e's pairs in one
// pass over idx: each thread takes a contiguous run of tokens, adds their
// selections to the block's histogram of all experts and counts those equal
// to e; then
//   offsets[e]     = number of pairs with expert < e (exclusive scan of counts)
//   pad_offsets[e] = same over rpp*counts rounded up to 128 rows (rpp = padded
//                    rows per pair: 1, or 2 when x is split into hi + lo rows)
//   rank of pair (t, j) with idx[t,j] == e = number of tokens t' < t that
//   selected e (each token selects an expert at most once): the exclusive
//   scan of the threads' counts plus the order inside a thread's run, so the
//   order is (expert, token) and is independent of thread timing.
__global__ void __launch_bounds__(256) route_group_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ pad_offsets,
                                                          int32_t* __restrict__ perm_tok,
                                                          int32_t* __restrict__ perm_slot, int32_t* __restrict__ inv,
                                                          int32_t* __restrict__ pad_inv,
                                                          int32_t* __restrict__ pad_pair,
                                                          int32_t* __restrict__ touched, int rpp) {
  __shared__ int hist[kMaxE];
  __shared__ int warp_tot[32];
  __shared__ int s_off, s_poff;
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x;
  const int tid = threadIdx.x;

  for (int i = tid; i < kMaxE; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int per = (T + (int)blockDim.x - 1) / (int)blockDim.x;
  const int t0 = min(T, tid * per), t1 = min(T, t0 + per);
  // the thread's selections idx[t0 * k .. t1 * k) are contiguous
  const int p0 = t0 * k, p1 = t1 * k;
  int hits = 0;
  if ((k % 4) == 0 && (reinterpret_cast<uintptr_t>(idx) & 15u) == 0) {
    // eight 16-byte loads in flight per round
    const int4* v4 = reinterpret_cast<const int4*>(idx + p0);
    const int n4 = (p1 - p0) / 4;
    int i = 0;
    for (; i + 8 <= n4; i += 8) {
      int4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(v4 + i + u);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        atomicAdd(&hist[v[u].x], 1);
        atomicAdd(&hist[v[u].y], 1);
        atomicAdd(&hist[v[u].z], 1);
        atomicAdd(&hist[v[u].w], 1);
        hits += (v[u].x == e) + (v[u].y == e) + (v[u].z == e) + (v[u].w == e);
      }
    }
    for (; i < n4; ++i) {
      const int4 v = __ldg(v4 + i);
      atomicAdd(&hist[v.x], 1);
      atomicAdd(&hist[v.y], 1);
      atomicAdd(&hist[v.z], 1);
      atomicAdd(&hist[v.w], 1);
      hits += (v.x == e) + (v.y == e) + (v.z == e) + (v.w == e);
    }
  } else {
    for (int p = p0; p < p1; ++p) {
      const int v = __ldg(idx + p);
      atomicAdd(&hist[v], 1);
      hits += v == e;
    }
  }
  __syncthreads();

  // exclusive scans of counts, padded counts and the touched flag (tid = expert)
  const int c = (tid < E) ? hist[tid] : 0;
  const int pc = (c * rpp + kPadRows - 1) / kPadRows * kPadRows;
  const int inc_c = block_scan_incl(c, warp_tot);
  const int inc_pc = block_scan_incl(pc, warp_tot);
  const int inc_t = block_scan_incl(c > 0 ? 1 : 0, warp_tot);
  if (tid == e) {
    s_off = inc_c - c;
    s_poff = inc_pc - pc;
  }
  if (blockIdx.x == 0 && tid < E) {
    counts[tid] = c;
    offsets[tid] = inc_c - c;
    pad_offsets[tid] = inc_pc - pc;
    if (c > 0) touched[inc_t - 1] = tid;
    if (tid == E - 1) {
      offsets[E] = inc_c;
      pad_offsets[E] = inc_pc;
      touched[E] = inc_t;
    }
  }
  // rank of this thread's first selection of e (the scan's barriers also
  // publish s_off and s_poff)
  int r = block_scan_incl(hits, warp_tot) - hits;
  const int off = s_off, poff = s_poff;
#define DS4_EMIT_PAIR(PAIR)                                   \
  do {                                                        \
    const int pair_ = (PAIR);                                 \
    const int pos_ = off + r, ppos_ = poff + r * rpp;         \
    perm_tok[pos_] = pair_ / k;                               \
    perm_slot[pos_] = pair_ % k;                              \
    inv[pair_] = pos_;                                        \
    pad_inv[pair_] = ppos_;                                   \
    pad_pair[ppos_] = pair_;                                  \
    if (rpp > 1) pad_pair[ppos_ + 1] = pair_; /* rpp <= 2 */   \
    ++r;                                                      \
    --hits;                                                   \
  } while (0)
  if ((k % 4) == 0 && (reinterpret_cast<uintptr_t>(idx) & 15u) == 0) {
    // second pass with batched loads (four 16-byte loads in flight), so a
    // thread holding a selection of e does not wait one load latency per pair
    // up to its last one; selections stay in pair order
    const int4* v4 = reinterpret_cast<const int4*>(idx + p0);
    const int n4 = (p1 - p0) / 4;
    for (int i = 0; i < n4 && hits > 0; i += 4) {
      int4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = i + u < n4 ? __ldg(v4 + i + u) : make_int4(-1, -1, -1, -1);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pb = p0 + 4 * (i + u);
        if (v[u].x == e) DS4_EMIT_PAIR(pb);
        if (v[u].y == e) DS4_EMIT_PAIR(pb + 1);
        if (v[u].z == e) DS4_EMIT_PAIR(pb + 2);
        if (v[u].w == e) DS4_EMIT_PAIR(pb + 3);
      }
    }
  } else {
    for (int pair = p0; pair < p1 && hits > 0; ++pair)
      if (__ldg(idx + pair) == e) DS4_EMIT_PAIR(pair);
  }
#undef DS4_EMIT_PAIR
}

// Grouping of the T*k <= 32 pairs of a few-token call by one warp, without
// block barriers: lane p holds pair p; experts e = lane + 32i are counted and
// scanned in order with warp scans; the rank of pair p is the number of earlier
// pairs with the same expert (a token selects an expert at most once, so these
// are earlier tokens).  The same tables as route_group_kernel, and s_prow[p] =
// the pair's first padded row.
__device__ __forceinline__ void group_warp(const int* idx, int npairs, int E, int k, int rpp, int lane,
                                           int32_t* counts, int32_t* offsets, int32_t* pad_offsets, int32_t* perm_tok,
                                           int32_t* perm_slot, int32_t* inv, int32_t* pad_inv, int32_t* pad_pair,
                                           int32_t* touched, int* s_off, int* s_poff, int* s_prow) {
  // Lane l counts experts 8l .. 8l + 7; one packed inclusive scan of the lane
  // totals (pairs in bits 0-7, padded rows in bits 8-23, touched experts in
  // bits 24-31: npairs <= 32 keeps each field in range) gives every lane its
  // starting offsets.
  static_assert(kMaxE == 8 * 32, "eight experts per lane");
  const int ep = lane < npairs ? idx[lane] : -1;
  int cnt[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) cnt[j] = 0;
  for (int q = 0; q < npairs; ++q) {
    const int eq = __shfl_sync(0xffffffffu, ep, q);
#pragma unroll
    for (int j = 0; j < 8; ++j) cnt[j] += (eq == 8 * lane + j) ? 1 : 0;
  }
  uint32_t tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = 8 * lane + j < E ? cnt[j] : 0;
    cnt[j] = c;
    tot += (uint32_t)c | ((uint32_t)((c * rpp + kPadRows - 1) / kPadRows * kPadRows) << 8) | ((c > 0 ? 1u : 0u) << 24);
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  uint32_t run = incl - tot;  // this lane's exclusive prefix
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = 8 * lane + j;
    const int c = cnt[j];
    if (e < E) {
      const int off = (int)(run & 0xFFu), poff = (int)((run >> 8) & 0xFFFFu);
      counts[e] = c;
      offsets[e] = off;
      pad_offsets[e] = poff;
      s_off[e] = off;
      s_poff[e] = poff;
      if (c > 0) touched[run >> 24] = e;
    }
    run += (uint32_t)c | ((uint32_t)((c * rpp + kPadRows - 1) / kPadRows * kPadRows) << 8) | ((c > 0 ? 1u : 0u) << 24);
  }
  if (lane == 31) {  // totals over all experts
    offsets[E] = (int)(incl & 0xFFu);
    pad_offsets[E] = (int)((incl >> 8) & 0xFFFFu);
    touched[E] = (int)(incl >> 24);
  }
  int r = 0;
  for (int q = 0; q < npairs; ++q) {
    const int eq = __shfl_sync(0xffffffffu, ep, q);
    r += (q < lane && eq == ep) ? 1 : 0;
  }
  __syncwarp();  // s_off, s_poff of every expert written
  if (lane < npairs) {
    const int pos = s_off[ep] + r, ppos = s_poff[ep] + r * rpp;
    perm_tok[pos] = lane / k;
    perm_slot[pos] = lane % k;
    inv[lane] = pos;
    pad_inv[lane] = ppos;
    for (int q = 0; q < rpp; ++q) pad_pair[ppos + q] = lane;
    s_prow[lane] = ppos;
  }
}

// Few-token routing in one block of 1024 threads (T <= kSmallRouteT): warps
// 0..T-1 take the top-k of one token each and warp 0 then groups the pairs
// (group_warp).  Meanwhile, when `quant` is set, warps T..31 quantise x to
// MXFP8 (hi + lo blocks when split == 2) into shared memory and zero out;
// after one block barrier every thread copies blocks of codes and scales into
// the routed pairs' rows.  So a decode step needs one launch before its GEMMs,
// and the routing's serial chain overlaps the quantisation.
__global__ void __launch_bounds__(1024) route_small_kernel(
    const float* __restrict__ logits, int lds, int T, int E, int k, int32_t* __restrict__ idx, float* __restrict__ w,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ pad_offsets,
    int32_t* __restrict__ perm_tok, int32_t* __restrict__ perm_slot, int32_t* __restrict__ inv,
    int32_t* __restrict__ pad_inv, int32_t* __restrict__ pad_pair, int32_t* __restrict__ touched, int split,
    const __nv_bfloat16* __restrict__ x, int d, uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf, int r128,
    float* __restrict__ out, int quant) {
  // [T][d/32 blocks][split][32] codes, then [T][d/32][split] scale bytes
  extern __shared__ __align__(16) uint8_t s_dyn[];
  __shared__ int s_prow[kSmallRouteT * kMaxK];
  __shared__ int s_idx[kSmallRouteT * kMaxK];  // the selections, for the grouping without a global round trip
  __shared__ int s_off[kMaxE], s_poff[kMaxE];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int npairs = T * k;
  const int nblk = d / 32;
  uint8_t* s_codes = s_dyn;
  uint8_t* s_sf = s_dyn + (size_t)T * d * split;

  if (wid < T) {
    topk_warp(logits + (size_t)wid * lds, E, k, lane, idx + (size_t)wid * k, w + (size_t)wid * k, s_idx + wid * k);
    // every token's selection is in s_idx before warp 0 reads it
    if (T > 1) named_bar_sync(1, 32 * T);
    else __syncwarp();
    if (wid == 0)
      group_warp(s_idx, npairs, E, k, split, lane, counts, offsets, pad_offsets, perm_tok, perm_slot, inv, pad_inv,
                 pad_pair, touched, s_off, s_poff, s_prow);
  } else if (quant) {
    const int nthr = (int)blockDim.x - 32 * T;
    for (int task = tid - 32 * T; task < T * nblk; task += nthr) {
      const int t = task / nblk, cb = task % nblk;
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d) + 4 * cb;
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = __ldg(src + q);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          v[8 * q + 2 * h] = __uint_as_float(wv[h] << 16);
          v[8 * q + 2 * h + 1] = __uint_as_float(wv[h] & 0xFFFF0000u);
        }
      }
      uint32_t hi[8], lo[8];
      int s_lo = 0;
      const int s_hi = split == 2 ? mxfp8_split_block(v, hi, lo, s_lo) : mxfp8_block(v, hi);
      uint4* dst = reinterpret_cast<uint4*>(s_codes + (size_t)task * split * 32);
      dst[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      dst[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
      s_sf[task * split] = (uint8_t)(s_hi + 127);
      if (split == 2) {
        dst[2] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        dst[3] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        s_sf[task * split + 1] = (uint8_t)(s_lo + 127);
      }
    }
    float4* o4 = reinterpret_cast<float4*>(out);
    for (int i = tid - 32 * T; i < T * d / 4; i += nthr) o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (!quant) return;
  __syncthreads();

  // Each routed pair's code row (and its lo row) is written in 16-byte
  // pieces, consecutive threads taking consecutive pieces, so a warp stores
  // 512 contiguous bytes; then the row's scales as 32-bit words (four
  // consecutive 32-element blocks share one word of the scale layout).  A
  // thread keeps one piece (word) position and walks the rows, so the index
  // arithmetic is done once, not per store.
  const int pieces = d / 16, words = nblk / 4, nrows = npairs * split;
  if (tid < (int)blockDim.x / pieces * pieces) {  // pieces <= 512 divides the rows among whole groups
    const int piece = tid % pieces, rstep = (int)blockDim.x / pieces;
    const int cb = piece / 2, half16 = (piece % 2) * 16;
    for (int rr = tid / pieces; rr < nrows; rr += rstep) {
      const int p = split == 2 ? rr >> 1 : rr, q = split == 2 ? rr & 1 : 0;
      const int tb = (p / k) * nblk + cb;
      const uint4 v = *reinterpret_cast<const uint4*>(s_codes + ((size_t)tb * split + q) * 32 + half16);
      *reinterpret_cast<uint4*>(xq + (size_t)(s_prow[p] + q) * d + 16 * (size_t)piece) = v;
    }
  }
  if (tid < (int)blockDim.x / words * words) {
    const int g = tid % words, rstep = (int)blockDim.x / words;
    for (int rr = tid / words; rr < nrows; rr += rstep) {
      const int p = split == 2 ? rr >> 1 : rr, q = split == 2 ? rr & 1 : 0;
      const int tb = (p / k) * nblk + 4 * g;
      const uint32_t word = (uint32_t)s_sf[tb * split + q] | ((uint32_t)s_sf[(tb + 1) * split + q] << 8) |
                            ((uint32_t)s_sf[(tb + 2) * split + q] << 16) | ((uint32_t)s_sf[(tb + 3) * split + q] << 24);
      *reinterpret_cast<uint32_t*>(xsf + act_sf_index((size_t)(s_prow[p] + q), 4 * g, r128)) = word;
    }
  }
}

}  // namespace

cudaError_t launch_route_topk(const ds4moe_layer* L, const float* logits, int lds, const void* x, bool prep_x, int T,
                              cudaStream_t st) {
  const int warps_per_block = 8;
  const int blocks = (T + warps_per_block - 1) / warps_per_block;
  return launch_pdl(route_topk_kernel, blocks, 32 * warps_per_block, 0, st, logits, lds, T, L->cfg.n_experts,
                    L->cfg.top_k, L->s.topk_idx, L->s.topk_w, static_cast<const __nv_bfloat16*>(x), L->cfg.d_model,
                    prep_x ? reinterpret_cast<uint4*>(L->s.xh) : nullptr, L->s.xsig);
}

cudaError_t launch_route_group(const ds4moe_layer* L, int T, int rpp, cudaStream_t st) {
  const int E = L->cfg.n_experts, k = L->cfg.top_k;
  const Scratch& s = L->s;
  return launch_pdl(route_group_kernel, E, 256, 0, st, s.topk_idx, T, E, k, s.counts, s.offsets, s.pad_offsets,
                    s.perm_tok, s.perm_slot, s.inv, s.pad_inv, s.pad_pair, s.touched, rpp);
}

cudaError_t launch_route_small(const ds4moe_layer* L, const float* logits, int lds, const void* x, float* out, int T,
                               int split, bool quant, cudaStream_t st) {
  const int E = L->cfg.n_experts, k = L->cfg.top_k;
  const Scratch& s = L->s;
  // dynamic shared memory: the MXFP8 codes and scales of the T rows of x
  // (at most kSmallRouteT x 8192 x 2 split codes + their scales)
  static InitOnce attr_once;
  const cudaError_t e = init_once(attr_once, [] {
    return cudaFuncSetAttribute((const void*)route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmallRouteT * 8192 * 2 + kSmallRouteT * 256 * 2);
  });
  if (e != cudaSuccess) return e;
  const size_t smem = quant ? (size_t)T * L->cfg.d_model * split + (size_t)T * (L->cfg.d_model / 32) * split : 0;
  return launch_pdl(route_small_kernel, 1, 1024, smem, st, logits, lds, T, E, k, s.topk_idx, s.topk_w, s.counts, s.offsets,
                    s.pad_offsets, s.perm_tok, s.perm_slot, s.inv, s.pad_inv, s.pad_pair, s.touched, split,
                    static_cast<const __nv_bfloat16*>(x), L->cfg.d_model, s.xq, s.xsf, (int)(s.pad_rows_max / 128),
                    out, quant ? 1 : 0);
}

}  // namespace ds4moe

// ---------------------------------------------------------------------------
// Routing without device allocation (ds4moe_route_noalloc).
//
// Some callers cannot call cudaMalloc when they route: an engine whose memory
// plan is fixed at start-up and forbids later allocations, or a serving loop
// that cannot pay cudaMalloc's implicit device synchronisation per batch.
// This entry point runs the same two routing kernels with their scratch in a
// file-scope device array instead of layer-owned buffers.  The array is
// sized for T*k <= kNoAllocMaxPairs and E <= 256 and stays resident on every
// GPU that loads this library until the process exits.
namespace ds4moe {
namespace {

constexpr int kNoAllocMaxPairs = 16384;
constexpr int kNoAllocMaxE = 256;
// counts[E] | pad_offsets[E+1] | perm_slot[P] | inv[P] | pad_inv[P] |
// pad_pair[P + E*127] | touched[E+1]
constexpr size_t kNoAllocInts = (size_t)kNoAllocMaxE + (kNoAllocMaxE + 1) + 3 * (size_t)kNoAllocMaxPairs +
                                ((size_t)kNoAllocMaxPairs + (size_t)kNoAllocMaxE * (kPadRows - 1)) +
                                (kNoAllocMaxE + 1);

__device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocInts];

}  // namespace
}  // namespace ds4moe

extern "C" int ds4moe_route_noalloc(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_idx,
                                    float* topk_w, int32_t* offsets, int32_t* perm_tok, ds4moe_stream_t stream) {
  using namespace ds4moe;
  auto misaligned = [](const void* p) { return ((uintptr_t)p & 15u) != 0; };
  if (T < 0 || E < 1 || E > kNoAllocMaxE || k < 1 || k > 8 || k > E) return DS4MOE_ERR_INVALID_ARG;
  if ((int64_t)T * k > kNoAllocMaxPairs) return DS4MOE_ERR_TOO_MANY_TOKENS;
  if (T == 0) {
    // no pairs: every expert's offset is 0 (the other outputs are empty)
    if (!offsets || misaligned(offsets)) return DS4MOE_ERR_INVALID_ARG;
    if (cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
      cudaGetLastError();
      return DS4MOE_ERR_CUDA;
    }
    return DS4MOE_OK;
  }
  if (!logits || !topk_idx || !topk_w || !offsets || !perm_tok) return DS4MOE_ERR_INVALID_ARG;
  if (misaligned(logits) || misaligned(topk_idx) || misaligned(topk_w) || misaligned(offsets) || misaligned(perm_tok))
    return DS4MOE_ERR_INVALID_ARG;

  // Host code must not take the array's address directly (that is a host-side
  // stand-in); the device address is looked up once per device, with that
  // device current, on the first call made on it.
  static std::mutex mu;
  static int32_t* scratch_of[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!scratch_of[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return DS4MOE_ERR_CUDA;
      }
      scratch_of[dev] = static_cast<int32_t*>(p);
    }
    scratch = scratch_of[dev];
  }
  int32_t* counts = scratch;
  int32_t* pad_offsets = counts + kNoAllocMaxE;
  int32_t* perm_slot = pad_offsets + (kNoAllocMaxE + 1);
  int32_t* inv = perm_slot + kNoAllocMaxPairs;
  int32_t* pad_inv = inv + kNoAllocMaxPairs;
  int32_t* pad_pair = pad_inv + kNoAllocMaxPairs;
  int32_t* touched = pad_pair + (kNoAllocMaxPairs + kNoAllocMaxE * (kPadRows - 1));

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int blocks = (T + 7) / 8;
  route_topk_kernel<<<blocks, 256, 0, st>>>(logits, E, T, E, k, topk_idx, topk_w, nullptr, 0, nullptr, nullptr);
  route_group_kernel<<<E, 256, 0, st>>>(topk_idx, T, E, k, counts, offsets, pad_offsets, perm_tok, perm_slot, inv,
                                        pad_inv, pad_pair, touched, 1);
  if (cudaGetLastError() != cudaSuccess) return DS4MOE_ERR_CUDA;
  return DS4MOE_OK;
}
