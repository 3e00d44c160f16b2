// Routing of the routed-MoE layer: top-k selection with softmax over the
// selected logits, then a deterministic grouping of the (token, slot) pairs
// by expert.
//
// The pages ("DwarfStar実地分析", §GGUFの対応範囲は意図的に狭い) say only that the
// routing itself stays at original precision; the rule implemented here is the
// layer's specification: the k largest fp32 logits per token ordered by
// (value desc, expert index asc), weights = softmax over those k only.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace ds4moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kMaxK = 8;

// One warp per token.  Lane l holds logits l, l+32, ..., so a lane's own
// entries are in increasing index order.
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ idx, float* __restrict__ w) {
  const int token = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= T) return;
  const float* row = logits + (size_t)token * E;

  float v[kMaxE / 32];
  uint32_t taken = 0;  // bit i: entry lane+32i already selected, or beyond E
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    const int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      x = __ldg(row + e);
      if (x != x) x = -INFINITY;  // NaN ranks with -inf (outside the layer's domain)
    } else {
      taken |= 1u << i;
    }
    v[i] = x;
  }

  float sel_v[kMaxK];
  int sel_e[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int be = INT_MAX;  // INT_MAX = no candidate
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i) {
        if (!((taken >> i) & 1u) && (be == INT_MAX || v[i] > bv)) {
          bv = v[i];
          be = lane + 32 * i;
        }
      }
      // warp arg-max under the total order (valid, value desc, index asc)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        const bool better = (oe != INT_MAX) && (be == INT_MAX || ov > bv || (ov == bv && oe < be));
        if (better) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      sel_v[j] = bv;
      sel_e[j] = be;
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
        idx[(size_t)token * k + j] = sel_e[j];
        w[(size_t)token * k + j] = expf(sel_v[j] - sel_v[0]) / z;
      }
    }
  }
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

// Grid = E blocks of 256 threads; block e places expert e's pairs.
//   offsets[e]     = number of pairs with expert < e (exclusive scan of counts)
//   pad_offsets[e] = same over counts rounded up to 128 rows
//   rank of pair (t, j) with idx[t,j] == e = number of tokens t' < t that
//   selected e (each token selects an expert at most once), so the order is
//   (expert, token) and is independent of thread timing.
__global__ void __launch_bounds__(256) route_group_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ pad_offsets,
                                                          int32_t* __restrict__ perm_tok,
                                                          int32_t* __restrict__ perm_slot, int32_t* __restrict__ inv,
                                                          int32_t* __restrict__ pad_inv,
                                                          int32_t* __restrict__ pad_pair,
                                                          int32_t* __restrict__ touched) {
  __shared__ int hist[kMaxE];
  __shared__ int warp_tot[32];
  __shared__ int s_off, s_poff;
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  const int npairs = T * k;

  for (int i = tid; i < kMaxE; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int p = tid; p < npairs; p += blockDim.x) atomicAdd(&hist[__ldg(idx + p)], 1);
  __syncthreads();

  // exclusive scans of counts, padded counts and the touched flag (tid = expert)
  const int c = (tid < E) ? hist[tid] : 0;
  const int pc = (c + kPadRows - 1) / kPadRows * kPadRows;
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
  __syncthreads();
  const int off = s_off, poff = s_poff;

  // rank assignment for expert e, 256 tokens at a time
  const int lane = tid & 31, wid = tid >> 5;
  int running = 0;
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + tid;
    int slot = -1;
    if (t < T) {
      for (int j = 0; j < k; ++j)
        if (__ldg(idx + (size_t)t * k + j) == e) slot = j;
    }
    const unsigned ball = __ballot_sync(0xffffffffu, slot >= 0);
    const int in_warp = __popc(ball & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[wid] = __popc(ball);
    __syncthreads();
    int before = 0, total = 0;
    for (int q = 0; q < (int)(blockDim.x >> 5); ++q) {
      const int n = warp_tot[q];
      if (q < wid) before += n;
      total += n;
    }
    if (slot >= 0) {
      const int r = running + before + in_warp;
      const int pos = off + r, ppos = poff + r;
      const int pair = t * k + slot;
      perm_tok[pos] = t;
      perm_slot[pos] = slot;
      inv[pair] = pos;
      pad_inv[pair] = ppos;
      pad_pair[ppos] = pair;
    }
    running += total;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w, cudaStream_t st) {
  const int warps_per_block = 8;
  const int blocks = (T + warps_per_block - 1) / warps_per_block;
  route_topk_kernel<<<blocks, 32 * warps_per_block, 0, st>>>(logits, T, E, k, idx, w);
  return cudaGetLastError();
}

cudaError_t launch_route_group(const ds4moe_layer* L, int T, cudaStream_t st) {
  const int E = L->cfg.n_experts, k = L->cfg.top_k;
  const Scratch& s = L->s;
  route_group_kernel<<<E, 256, 0, st>>>(s.topk_idx, T, E, k, s.counts, s.offsets, s.pad_offsets, s.perm_tok,
                                        s.perm_slot, s.inv, s.pad_inv, s.pad_pair, s.touched);
  return cudaGetLastError();
}

}  // namespace ds4moe
