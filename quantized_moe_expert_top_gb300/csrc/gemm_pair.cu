// Grouped block-scaled GEMMs of the routed experts on CTA pairs
// (tcgen05 cta_group::2): gate/up with the SwiGLU + MXFP8 epilogue, and down
// with the weighted combine back into token order.
//
// "DwarfStar実地分析" §GGUFの対応範囲は意図的に狭い states that on Blackwell CUDA
// the batched expert work runs on FP4 matrix instructions.  Every expert's
// tokens form one GEMM with the weights as the M side (swap-AB): the E2M1
// weights are A (TMA expands the packed nibbles into the 16-byte-aligned layout
// the MMA reads), the E4M3 activations of the expert's tokens are B, with one
// E8M0 scale per 32 K on both, accumulated in fp32 in tensor memory.
//
// Two CTAs of a cluster form a pair and issue one M = 256 MMA: each CTA holds
// 128 weight rows and half of the token rows in its shared memory, and the
// leader (rank 0) issues the MMAs for both.  Each weight and token byte is
// written to and read from shared memory once per pair, which is what bounds a
// single CTA's tile rate, and the smaller stage leaves room for six stage slots.
//
//   gate/up : the pair covers 128 features of one expert; each CTA's 128 rows
//             are the gate rows then the up rows of its 64 features, so its
//             accumulator holds g in lanes 0..63 and u in lanes 64..127 for
//             every token.  The gate warps stage silu(g) in shared memory for
//             the up warps, which form h = silu(g) * u and quantise it to
//             MXFP8 along f (or round it to fp16 for a Q2_K down projection).
//   down    : the pair covers 256 output rows; the epilogue multiplies by the
//             routing weight and red-adds into out[t].
//
// Warp roles per CTA (persistent, one CTA per SM): warp 0 issues the TMA
// loads of both operands (3-D boxes of two K blocks) and, every fourth K
// block, of the scale factors of the next four; warp 1 allocates tensor
// memory and, in the leader, issues the MMAs (the whole warp runs the loop, one
// elected lane issues); warps 2..9 drain the accumulators; warp 10 copies the
// scale factors into tensor memory.  All loads are TMA (async proxy), so the
// tensor core reads them with no proxy fence, and both CTAs' loads complete on
// the leader's barrier.  The accumulator is double-buffered, so a chunk's
// epilogue overlaps the next chunk's main loop.  Every wait is bounded; a wait
// that runs out records DS4MOE_ERR_DEVICE_TIMEOUT in the layer's status word
// and the CTA winds down.
#include "gemm.cuh"

namespace ds4moe {
namespace {

enum class PMode { GateUp, Down };

constexpr int kPStages = 6;     // K = 128 stage slots, loaded and consumed two at a time
constexpr int kPBars = kPStages / 2;
constexpr int kPNMax = 192;     // token columns (N) per chunk, both CTAs together
constexpr int kPEpiWarps = 8;   // two per tensor-memory lane quarter
constexpr int kPCpWarp = 2 + kPEpiWarps;  // the leader's scale-factor copies
constexpr int kPThreads = 32 * (3 + kPEpiWarps);
constexpr int kPAcc1 = 192;     // column of the second accumulator buffer
constexpr int kPSfBase = 384;   // scale-factor slots: SFA 4 + SFB 8 columns each
constexpr int kPSfSlot = 12;
// Scale-factor slots in tensor memory, two per step (one per K = 128 block)
// in issue order, so a slot is rewritten kPBars + 1 steps after its last use:
// the copy thread waits for the MMAs of the step kPBars back (the stage slot
// it reuses), and MMAs complete in issue order.
constexpr int kPSfSlots = 2 * (kPBars + 1);
static_assert(kPAcc1 + kPNMax <= kPSfBase && kPSfBase + kPSfSlots * kPSfSlot <= 512, "tensor memory");
static_assert(kPNMax / 2 <= 128, "token rows per CTA fit the 3-D token maps");
constexpr int kPrefetchSteps = 3;  // weight boxes prefetched into L2 ahead of their load
constexpr int kSfGroup = 4;     // K blocks whose scale factors one pair of TMA loads brings
constexpr int kSfRing = 3;      // scale-factor groups in shared memory
static_assert(kSfGroup % 2 == 0, "scale groups start on a step boundary");

struct PSmem {
  static constexpr int kA = 128 * 128;           // 128 weight rows x 128 K (E2M1 in 8-bit containers)
  static constexpr int kB = (kPNMax / 2) * 128;  // this CTA's half of the token rows
  static constexpr int kStage = kA + kB;
  // A step (two K = 128 blocks) is one slot pair laid out [A0 A1 | B0 B1]:
  // each operand arrives in one 3-D TMA box of two K blocks, B1 right after
  // B0 (nh rows of 128 bytes each).
  static constexpr int kStep = 2 * kStage;
  // scale-factor group: SFA chunks of 4 K blocks (4 x 512) | SFB [4 K blocks][2 row blocks][512]
  static constexpr int kSfA = kSfGroup * kSfChunk;
  static constexpr int kSfGroupBytes = kSfA + kSfGroup * 2 * kSfChunk;
  static constexpr int kSfOff = kPStages * kStage;
  static constexpr int kXchg = kSfOff + kSfRing * kSfGroupBytes;  // gate/up: 4 warp pairs x (silu(g), u) x 8 x 32
  static constexpr int kColOff = kXchg + 4 * 2 * 8 * 32 * 4;   // down: per-column token and weight
  static constexpr int kBarOff = kColOff + kPNMax * 8;
  static constexpr int kTotal = kBarOff + 512 + 1024;          // + barriers, + alignment slack
};
static_assert(PSmem::kStage % 1024 == 0 && (PSmem::kB % 2048) == 0, "stage alignment");
static_assert(PSmem::kTotal <= 227 * 1024, "shared memory");

struct PairArgs {
  int rows_per_expert;  // gate/up: f; down: d
  int r128;             // 128-row blocks of the activation buffers
  int K;                // d (gate/up) or f (down)
  const int32_t* counts;
  const int32_t* touched;
  const int32_t* pad_offsets;
  const int32_t* pad_pair;
  const float* topk_w;
  int E, k, d, f;
  uint8_t* hq;    // gate/up: MXFP8 h codes [rows][f]
  uint8_t* hsf;   // gate/up: h scales (chunk layout)
  __half* h16;    // gate/up: fp16 h for a Q2_K down projection, or nullptr
  float* out;     // down: [T][d]
  DeviceStatus* status;
  uint64_t budget_ns;
  int debug_fault;
  int split;      // token columns per routed pair: 1, or 2 (hi + lo rows)
};

// Work sequence shared by every role of both CTAs of a pair: units
// (touched expert, block pair), expert-major, strided over the pairs; each
// unit's token columns split into chunks that start on a 128-column boundary
// (one chunk when they fit in kPNMax).
struct PairIter {
  int u, nunits, stride, per_e;
  int e, pb, ne, t0, nch;
  const int32_t* counts;
  const int32_t* touched;
  int split;
  __device__ bool first_chunk() {
    for (; u < nunits; u += stride) {
      e = __ldg(touched + u / per_e);
      pb = u % per_e;
      ne = __ldg(counts + e) * split;
      if (ne > 0) {
        t0 = 0;
        nch = ne <= kPNMax ? ne : 128;
        return true;
      }
    }
    return false;
  }
  __device__ bool next() {
    t0 += nch;
    if (t0 < ne) {
      const int rem = ne - t0;
      nch = rem <= kPNMax ? rem : 128;
      return true;
    }
    u += stride;
    return first_chunk();
  }
};

// This CTA's 128-row weight tile of a unit.  Gate/up tiles are [E][f/64]
// (64 gate rows then the same 64 up rows); down tiles are [E][d/128], and the
// peer's tile of the last pair is past the expert when d is an odd multiple of
// 128 (its loads then read zeros or the next expert's rows and scales, which
// are never stored).
template <PMode M>
__device__ __forceinline__ int weight_tile(const PairArgs& a, int e, int pb, uint32_t rank) {
  if (M == PMode::GateUp) return e * (a.f / 64) + 2 * pb + (int)rank;
  return e * (a.d / 128) + 2 * pb + (int)rank;
}

__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// One 16-column slice of the gate/up epilogue for a warp pair (the gate warp
// and the up warp of one feature quarter; lane = feature): each warp stages
// the half of its per-token values that the other warp finishes, then forms
// h = silu(g) * u for its own half of the tokens and stores h in MXFP8 (32
// features = one scale block = the warp's lanes), as hi + lo rows for the
// split activations, or in fp16 for a Q2_K down projection.  SPLIT columns
// make one token.
template <int SPLIT>
__device__ __forceinline__ void gateup_slice(const uint32_t (&r)[16], bool gate, int lane, float* sg, float* su,
                                             int pid, int c0, int nch, int prow, int i, const PairArgs& args) {
  constexpr int kTok = 16 / SPLIT;  // tokens in the slice
  constexpr int kHalf = kTok / 2;   // tokens each warp finishes
  float v[kTok];
#pragma unroll
  for (int jj = 0; jj < kTok; ++jj)
    v[jj] = SPLIT == 2 ? __uint_as_float(r[2 * jj]) + __uint_as_float(r[2 * jj + 1]) : __uint_as_float(r[jj]);
  if (gate) {
#pragma unroll
    for (int jj = 0; jj < kTok; ++jj) v[jj] = silu(v[jj]);
#pragma unroll
    for (int jj = 0; jj < kHalf; ++jj) sg[jj * 32 + lane] = v[kHalf + jj];
  } else {
#pragma unroll
    for (int jj = 0; jj < kHalf; ++jj) su[jj * 32 + lane] = v[jj];
  }
  named_bar_sync(2 + pid, 64);  // both halves staged
  float h[kHalf];
#pragma unroll
  for (int jj = 0; jj < kHalf; ++jj) h[jj] = gate ? v[jj] * su[jj * 32 + lane] : sg[jj * 32 + lane] * v[kHalf + jj];
  named_bar_sync(6 + pid, 64);  // staging free for the next slice
  const int tok0 = c0 / SPLIT + (gate ? 0 : kHalf);  // first token of this warp's half
  // amax of a 32-feature block (the warp's lanes) for all of the warp's
  // tokens at once: a butterfly of shuffles on the magnitudes' bit patterns
  // (unsigned order = float order for non-negative values); lane j then stores
  // the scale byte of token j, one store for all tokens.
  auto block_amax = [&](uint32_t (&am)[kHalf]) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int jj = 0; jj < kHalf; ++jj) am[jj] = max(am[jj], __shfl_xor_sync(0xffffffffu, am[jj], o));
  };
  if constexpr (SPLIT == 2) {
    uint32_t am[kHalf], am2[kHalf], chi[kHalf];
    int s[kHalf];
    float res[kHalf];
#pragma unroll
    for (int jj = 0; jj < kHalf; ++jj) am[jj] = __float_as_uint(fabsf(h[jj]));
    block_amax(am);
#pragma unroll
    for (int jj = 0; jj < kHalf; ++jj) {
      s[jj] = mxfp8_exponent(__uint_as_float(am[jj]));
      chi[jj] = f32x2_to_e4m3x2(h[jj] * exp2i(-s[jj]), 0.f) & 0xFFu;
      res[jj] = h[jj] - e4m3x2_to_f32x2(chi[jj]).x * exp2i_e8m0(s[jj]);
      am2[jj] = __float_as_uint(fabsf(res[jj]));
    }
    block_amax(am2);
    uint32_t sf_mine = 0;  // lane 2j: scale of token j's hi row, lane 2j + 1: of its lo row
#pragma unroll
    for (int jj = 0; jj < kHalf; ++jj) {
      const int s2 = mxfp8_exponent(__uint_as_float(am2[jj]));
      const uint32_t clo = f32x2_to_e4m3x2(res[jj] * exp2i(-s2), 0.f) & 0xFFu;
      if (lane == 2 * jj) sf_mine = (uint32_t)(s[jj] + 127);
      if (lane == 2 * jj + 1) sf_mine = (uint32_t)(s2 + 127);
      const int col = 2 * (tok0 + jj);
      if (col < nch) {
        const size_t row = (size_t)(prow + col);
        args.hq[row * args.f + i] = (uint8_t)chi[jj];
        args.hq[(row + 1) * args.f + i] = (uint8_t)clo;
      }
    }
    if (lane < 2 * kHalf && 2 * tok0 + lane < nch)
      args.hsf[act_sf_index((size_t)(prow + 2 * tok0 + lane), i / 32, args.r128)] = (uint8_t)sf_mine;
  } else {
    if (args.h16 != nullptr) {
#pragma unroll
      for (int jj = 0; jj < kHalf; ++jj)
        if (tok0 + jj < nch) args.h16[(size_t)(prow + tok0 + jj) * args.f + i] = __float2half_rn(h[jj]);
      return;
    }
    uint32_t am[kHalf];
#pragma unroll
    for (int jj = 0; jj < kHalf; ++jj) am[jj] = __float_as_uint(fabsf(h[jj]));
    block_amax(am);
    uint32_t sf_mine = 0;  // lane j: scale of token j
#pragma unroll
    for (int jj = 0; jj < kHalf; ++jj) {
      const int s = mxfp8_exponent(__uint_as_float(am[jj]));
      if (lane == jj) sf_mine = (uint32_t)(s + 127);
      const int col = tok0 + jj;
      if (col < nch)
        args.hq[(size_t)(prow + col) * args.f + i] = (uint8_t)(f32x2_to_e4m3x2(h[jj] * exp2i(-s), 0.f) & 0xFFu);
    }
    if (lane < kHalf && tok0 + lane < nch)
      args.hsf[act_sf_index((size_t)(prow + tok0 + lane), i / 32, args.r128)] = (uint8_t)sf_mine;
  }
}

template <PMode M>
__global__ void __launch_bounds__(kPThreads, 1) pair_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                                                               const __grid_constant__ CUtensorMap tm_sfa,
                                                               const __grid_constant__ CUtensorMap tm_sfb,
                                                               const __grid_constant__ BoxMaps bmaps,
                                                               const PairArgs args) {
  using S = PSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xchg = reinterpret_cast<float*>(smem + S::kXchg);
  int32_t* col_tok = reinterpret_cast<int32_t*>(smem + S::kColOff);
  float* col_w = reinterpret_cast<float*>(col_tok + kPNMax);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);  // leader: all bytes of a slot pair landed
  uint64_t* empty = full + kPBars;                                    // the slot pair's MMAs are done
  uint64_t* acc_full = empty + kPBars;                                // [2] accumulator ready
  uint64_t* acc_empty = acc_full + 2;                                 // [2] leader: both epilogues drained it
  uint64_t* drain = acc_empty + 2;
  uint64_t* never = drain + 1;                                        // fault test: nothing arrives on it
  uint64_t* sf_full = never + 1;                                      // [kSfRing] leader: a scale group landed
  uint64_t* sf_empty = sf_full + kSfRing;                             // [kSfRing] its copies to TMEM are done
  uint64_t* cp_done = sf_empty + kSfRing;                             // [kPBars] leader: a step's scales in TMEM
  uint64_t* cp_drain = cp_done + kPBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cp_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_ok = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int per_e = M == PMode::GateUp ? args.rows_per_expert / 128 : (args.rows_per_expert + 255) / 256;
  const int KB = args.K / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPBars; ++s) {
      mbar_init(&full[s], 1);  // the leader's expect_tx; both CTAs' operand copies count their bytes
      mbar_init(&empty[s], 1);
      mbar_init(&cp_done[s], 1);  // the scale-copy thread's commit once the step's scales are in TMEM
    }
    for (int g = 0; g < kSfRing; ++g) {
      mbar_init(&sf_full[g], 1);
      mbar_init(&sf_empty[g], 1);
    }
    mbar_init(cp_drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * kPEpiWarps);
    }
    mbar_init(drain, 32);  // one commit per lane of the leader's MMA warp
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_sfa);
    prefetch_tmap(&tm_sfb);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or copy
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the routing tables and activations of this forward are complete from here on
  pdl_launch_dependents();
  const int nunits = __ldg(args.touched + args.E) * per_e;
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    // A step loads two K blocks (one when a chunk has an odd count left) into
    // one slot pair, completing on one barrier, so the MMA issuer waits once
    // per eight MMAs.  Every fourth K block (a step boundary) also brings the
    // scale factors of the next four.  The scale ring slot of a group is
    // reused three groups later; a group spans at least one step, so its
    // steps are at least kPBars steps back and done by then.
    if (lane == 0) {
      PairIter it{pair, nunits, npairs, per_e, 0, 0, 0, 0, 0, args.counts, args.touched, args.split};
      // L2 prefetch of this CTA's weight box kPrefetchSteps steps ahead of its load
      PairIter pf{pair, nunits, npairs, per_e, 0, 0, 0, 0, 0, args.counts, args.touched, args.split};
      bool pf_valid = pf.first_chunk();
      int pf_kb = 0;
      auto prefetch_next = [&]() {
        if (!pf_valid) return;
        tma_prefetch_3d(&tm_a, 0, weight_tile<M>(args, pf.e, pf.pb, rank) * 128, pf_kb);
        pf_kb += 2;
        if (pf_kb >= KB) {
          pf_kb = 0;
          pf_valid = pf.next();
        }
      };
      for (int i = 0; i < kPrefetchSteps; ++i) prefetch_next();
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);
      const uint32_t sf_full0 = mapa_shared(smem_u32(sf_full), 0);
      int bar = 0, sf_slot = 0;
      uint32_t phase = 0, sf_phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0, sf_issued = 0, sf_parity = 0;
      bool ok = true;
      for (bool more = it.first_chunk(); more && ok; more = it.next()) {
        const int nh = round32(it.nch) / 2;  // token rows per CTA
        const CUtensorMap* tb = &bmaps.m[nh / 16 - 1];
        const int prow = __ldg(args.pad_offsets + it.e) + it.t0;
        const int brow = prow + (int)rank * nh;
        const int tile = weight_tile<M>(args, it.e, it.pb, rank);
        // 4-bit unpacking loads count their packed global bytes
        const uint32_t stage_bytes = 2u * (128u * 64u + (uint32_t)nh * 128u);
        constexpr uint32_t kSfBytes = 2u * S::kSfGroupBytes;  // both CTAs' scale groups
        for (int kb = 0; kb < KB; kb += 2) {
          if (!mbar_wait_bounded(&empty[bar], phase ^ 1u, args.budget_ns, abort_flag)) {
            report_timeout(args.status, kWhereProducerEmpty);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const bool sf_load = kb % kSfGroup == 0;  // scale factors of K blocks kb .. kb + 3 (zeros past K)
          if (sf_load) {
            // the ring slot's previous group has been copied to TMEM (both CTAs)
            if (!mbar_wait_bounded(&sf_empty[sf_slot], sf_phase ^ 1u, args.budget_ns, abort_flag)) {
              report_timeout(args.status, kWhereProducerEmpty);
              *abort_flag = 1;
              ok = false;
              break;
            }
            const uint32_t g_cl = sf_full0 + 8u * sf_slot;
            if (leader) mbar_arrive_expect_tx(&sf_full[sf_slot], kSfBytes);
            uint8_t* sf = smem + S::kSfOff + sf_slot * S::kSfGroupBytes;
            tma_load_2d_pair(sf, &tm_sfa, g_cl, 0, (tile * KB + kb) * 2);
            tma_load_3d_pair(sf + S::kSfA, &tm_sfb, g_cl, 0, (prow / 128) * 2, kb);
            sf_issued |= 1u << sf_slot;
            sf_parity = (sf_parity & ~(1u << sf_slot)) | (sf_phase << sf_slot);
            if (++sf_slot == kSfRing) {
              sf_slot = 0;
              sf_phase ^= 1u;
            }
          }
          const uint32_t b_cl = full0 + 8u * bar;
          // both K blocks in one box per operand (a block past K reads zeros)
          if (leader) mbar_arrive_expect_tx(&full[bar], stage_bytes * 2);
          uint8_t* st = smem + bar * S::kStep;
          tma_load_3d_pair(st + 2 * S::kA, tb, b_cl, 0, brow, kb);
          tma_load_3d_pair(st, &tm_a, b_cl, 0, tile * 128, kb);
          prefetch_next();
          issued_mask |= 1u << bar;
          issued_parity = (issued_parity & ~(1u << bar)) | (phase << bar);
          if (++bar == kPBars) {
            bar = 0;
            phase ^= 1u;
          }
        }
      }
      if (leader) {
        // The last issued copies of every slot have landed (both CTAs' bytes)
        // before the pair exits: in a normal run these are consumed anyway;
        // after a wait ran out, this is the drain of what is in flight.
        for (int b = 0; b < kPBars; ++b)
          if ((issued_mask >> b) & 1u) {
            volatile int no_abort = 0;
            mbar_wait_bounded(&full[b], (issued_parity >> b) & 1u, args.budget_ns, &no_abort);
          }
        for (int g = 0; g < kSfRing; ++g)
          if ((sf_issued >> g) & 1u) {
            volatile int no_abort = 0;
            mbar_wait_bounded(&sf_full[g], (sf_parity >> g) & 1u, args.budget_ns, &no_abort);
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader) {
      // ---------------------------------------------------------- MMA issuer (leader)
      // The whole warp runs the loop (warp-uniform operands); one elected
      // lane issues each tcgen05 op.
      PairIter it{pair, nunits, npairs, per_e, 0, 0, 0, 0, 0, args.counts, args.touched, args.split};
      int bar = 0, chunk = 0;
      uint32_t phase = 0, acc_phase = 0, sf_seq = 0;
      bool ok = true;
      // Descriptors of stage slot 0; a slot adds its byte offset / 16 to the
      // start-address field, a K step of 32 elements adds 32 bytes.  The scale
      // factors reach tensor memory through the copy thread; this thread
      // waits once per step (operands landed, then scales copied) and issues
      // MMAs only, with no memory access in between.
      const uint32_t st0 = smem_u32(smem);
      const uint64_t adesc0 = smem_desc(st0, 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(st0 + 2 * S::kA, 16, 1024, 2);
      static_assert(S::kXchg < (1 << 18), "descriptor address field");
      constexpr uint32_t kSfIdStep = (1u << 4) | (1u << 29);  // next byte of the 32-bit scale word, A and B
      if (args.debug_fault && blockIdx.x == 0) {
        // Fault test: before its first MMA, the first pair's issuer waits on a
        // barrier that nothing arrives on, so the wait runs out.  Every TMA
        // load of both CTAs is still issued normally (at most kPBars steps,
        // since no slot is ever freed), and the producer's drain below waits
        // for all of them on this CTA's full barriers before the pair exits.
        if (!warp_wait_bounded(never, 0, args.budget_ns, abort_flag)) {
          if (lane == 0) {
            report_timeout(args.status, kWhereMmaFull);
            *abort_flag = 1;
          }
          ok = false;
        }
      }
      for (bool more = ok && it.first_chunk(); more && ok; more = it.next(), ++chunk) {
        const int N = round32(it.nch);
        const int nh = N / 2;  // token rows per CTA (one B block of a step)
        const int buf = chunk & 1;
        const uint32_t acc = tmem + (uint32_t)(buf ? kPAcc1 : 0);
        const uint32_t idesc0 = idesc_mx(256, N, 0);
        if (!warp_wait_bounded(&acc_empty[buf], ((acc_phase >> buf) & 1u) ^ 1u, args.budget_ns, abort_flag)) {
          if (lane == 0) {
            report_timeout(args.status, kWhereMmaAccEmpty);
            *abort_flag = 1;
          }
          break;
        }
        acc_phase ^= 1u << buf;
        tc_fence_after();
        for (int kb = 0; kb < KB; kb += 2) {
          if (!warp_wait_bounded(&full[bar], phase, args.budget_ns, abort_flag) ||
              !warp_wait_bounded(&cp_done[bar], phase, args.budget_ns, abort_flag)) {
            if (lane == 0) {
              report_timeout(args.status, kWhereMmaFull);
              *abort_flag = 1;
            }
            ok = false;
            break;
          }
          tc_fence_after();
          const bool two = KB - kb >= 2;
          const uint32_t slot0 = tmem + kPSfBase + sf_seq * kPSfSlot;
          sf_seq = sf_seq + 1 == kPSfSlots ? 0 : sf_seq + 1;
          const uint32_t slot1 = tmem + kPSfBase + sf_seq * kPSfSlot;
          if (two) sf_seq = sf_seq + 1 == kPSfSlots ? 0 : sf_seq + 1;
          const uint64_t aoff0 = (uint64_t)((bar * S::kStep) >> 4);
          const uint64_t aoff1 = aoff0 + (uint64_t)(S::kA >> 4);
          const uint64_t boff0 = aoff0;                          // bdesc0 points at 2 kA of slot 0
          const uint64_t boff1 = boff0 + (uint64_t)((nh * 128) >> 4);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)  // K = 32 (32 bytes) per instruction
            if (elect_one_sync())
              mma_mxf8f6f4_pair(acc, adesc0 + aoff0 + 2 * jj, bdesc0 + boff0 + 2 * jj,
                                idesc0 + (uint32_t)jj * kSfIdStep, slot0, slot0 + 4, (kb > 0 || jj > 0) ? 1u : 0u);
          if (two) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              if (elect_one_sync())
                mma_mxf8f6f4_pair(acc, adesc0 + aoff1 + 2 * jj, bdesc0 + boff1 + 2 * jj,
                                  idesc0 + (uint32_t)jj * kSfIdStep, slot1, slot1 + 4, 1u);
          }
          if (elect_one_sync()) tc_commit_pair(&empty[bar], 0x3);
          __syncwarp();
          if (++bar == kPBars) {
            bar = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one_sync()) tc_commit_pair(&acc_full[buf], 0x3);
        __syncwarp();
      }
      // every MMA issued lands before tensor memory is freed: each lane
      // commits (a commit tracks the committing lane's own MMAs), the barrier
      // takes 32
      tc_commit_pair(drain, 0x1);
      if (lane == 0) {
        volatile int never = 0;
        mbar_wait_bounded(drain, 0, args.budget_ns, &never);
      }
    }
    __syncwarp();
  } else if (warp == kPCpWarp) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- scale-factor copies (leader)
      // Per step: wait for the stage slot's previous MMAs (so the tensor-memory
      // scale slots this step rewrites are no longer read) and, at a new
      // scale group, for its TMA loads; copy both stages' SFA and SFB chunks
      // into tensor memory (both CTAs) and commit them to cp_done, on which
      // the MMA warp waits.  A group's ring slot is released (sf_empty, both
      // CTAs) once the copies of its last step are done.
      PairIter it{pair, nunits, npairs, per_e, 0, 0, 0, 0, 0, args.counts, args.touched, args.split};
      int bar = 0, groups = 0, gslot = 0;
      uint32_t phase = 0, sf_seq = 0;
      bool ok = true, have_group = false;
      const uint64_t sfdesc0 = smem_desc(smem_u32(smem) + S::kSfOff, 0, 128, 0);
      for (bool more = it.first_chunk(); more && ok; more = it.next()) {
        const int nsf = round32(it.nch) > 128 ? 2 : 1;
        for (int kb = 0; kb < KB; kb += 2) {
          if (!mbar_wait_bounded(&empty[bar], phase ^ 1u, args.budget_ns, abort_flag)) {
            report_timeout(args.status, kWhereProducerEmpty);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (kb % kSfGroup == 0) {
            if (have_group) tc_commit_pair(&sf_empty[gslot], 0x3);  // the previous group's copies are issued
            gslot = groups % kSfRing;
            const uint32_t gphase = (uint32_t)(groups / kSfRing) & 1u;
            ++groups;
            have_group = true;
            if (!mbar_wait_bounded(&sf_full[gslot], gphase, args.budget_ns, abort_flag)) {
              report_timeout(args.status, kWhereMmaFull);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          const int nst = KB - kb >= 2 ? 2 : 1;
          const uint64_t sd = sfdesc0 + (uint64_t)((gslot * S::kSfGroupBytes) >> 4);
          for (int i = 0; i < nst; ++i) {
            const int j = (kb + i) % kSfGroup;
            const uint32_t slot = tmem + kPSfBase + sf_seq * kPSfSlot;
            sf_seq = sf_seq + 1 == kPSfSlots ? 0 : sf_seq + 1;
            tc_cp_32x128b_warpx4_pair(slot, sd + (uint64_t)(j * (kSfChunk >> 4)));  // SFA: this CTA's rows
            for (int c = 0; c < nsf; ++c)  // SFB: all token columns (both CTAs hold them)
              tc_cp_32x128b_warpx4_pair(slot + 4 + 4 * c, sd + (uint64_t)((S::kSfA + (2 * j + c) * kSfChunk) >> 4));
          }
          tc_commit_pair(&cp_done[bar], 0x1);
          if (++bar == kPBars) {
            bar = 0;
            phase ^= 1u;
          }
        }
      }
      if (have_group) tc_commit_pair(&sf_empty[gslot], 0x3);
      // every copy issued lands before tensor memory is freed
      tc_commit_pair(cp_drain, 0x1);
      volatile int no_abort = 0;
      mbar_wait_bounded(cp_drain, 0, args.budget_ns, &no_abort);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                         // tensor-memory lane quarter this warp may access
    const int part = (warp - 2) >> 2;  // which half of the 16-column slices
    const int etid = threadIdx.x - 64;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(acc_empty), 0);
    auto release = [&](int b) {  // the buffer's reads are done: free it for the next chunk
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&acc_empty[b]);
        else mbar_arrive_cluster(acc_empty0 + 8u * b);
      }
    };
    PairIter it{pair, nunits, npairs, per_e, 0, 0, 0, 0, 0, args.counts, args.touched, args.split};
    uint32_t acc_phase = 0;
    int chunk = 0;
    for (bool more = it.first_chunk(); more; more = it.next(), ++chunk) {
      const int N = round32(it.nch);
      const int prow = __ldg(args.pad_offsets + it.e) + it.t0;
      const int buf = chunk & 1;
      // One thread takes the accumulator wait and publishes the outcome, so all
      // epilogue warps leave together (the named barriers need every one).
      named_bar_sync(1, 32 * kPEpiWarps);  // previous chunk's column table no longer read
      if (M == PMode::Down) {
        for (int c = etid; c < it.nch; c += 32 * kPEpiWarps) {
          const int pr = __ldg(args.pad_pair + prow + c);
          col_tok[c] = pr / args.k;
          col_w[c] = __ldg(args.topk_w + pr);
        }
      }
      if (etid == 0) {
        const bool ok = mbar_wait_bounded(&acc_full[buf], (acc_phase >> buf) & 1u, args.budget_ns, abort_flag);
        *epi_ok = ok ? 1 : 0;
        if (!ok) {
          report_timeout(args.status, kWhereEpiAccFull);
          *abort_flag = 1;
        }
      }
      named_bar_sync(1, 32 * kPEpiWarps);
      if (!*epi_ok) break;
      acc_phase ^= 1u << buf;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf ? kPAcc1 : 0) + lane_base;
      if constexpr (M == PMode::Down) {
        const int row = (2 * it.pb + (int)rank) * 128 + q * 32 + lane;  // output feature
        const bool rv = row < args.d;
        for (int c0 = part * 16; c0 < N; c0 += 32) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(acc + (uint32_t)c0, r);
          tmem_ld_wait();
          if (args.split == 2) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int col = c0 + 2 * jj;
              if (rv && col < it.nch)
                red_add_f32(args.out + (size_t)col_tok[col] * args.d + row,
                            col_w[col] * (__uint_as_float(r[2 * jj]) + __uint_as_float(r[2 * jj + 1])));
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int col = c0 + jj;
              if (rv && col < it.nch)
                red_add_f32(args.out + (size_t)col_tok[col] * args.d + row, col_w[col] * __uint_as_float(r[jj]));
            }
          }
        }
      } else {
        // Lanes 0..63 hold gate rows, 64..127 the up rows of the same 64
        // features.  The gate warp and the up warp of one feature quarter
        // each finish half of a 16-column slice: the gate warp the first
        // half (with u from the up warp), the up warp the second half (with
        // silu(g) from the gate warp).
        const bool gate = q < 2;
        const int pid = part * 2 + (q & 1);  // the warp pair of one feature quarter
        float* sg = xchg + pid * (2 * 8 * 32);  // silu(g) of the second half: [8][32]
        float* su = sg + 8 * 32;                // u of the first half: [8][32]
        const int i = it.pb * 128 + (int)rank * 64 + (q & 1) * 32 + lane;  // feature in [0, f)
        for (int c0 = part * 16; c0 < N; c0 += 32) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(acc + (uint32_t)c0, r);
          tmem_ld_wait();
          if (args.split == 2) gateup_slice<2>(r, gate, lane, sg, su, pid, c0, it.nch, prow, i, args);
          else gateup_slice<1>(r, gate, lane, sg, su, pid, c0, it.nch, prow, i, args);
        }
      }
      release(buf);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's accumulator reads and the leader's MMAs are done in both CTAs
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Largest number of resident pairs of a kernel (clusters of two CTAs with
// this shared memory), asked once.
template <PMode M>
int max_pairs(int num_sms) {
  static std::atomic<int> cached{0};
  const int c = cached.load(std::memory_order_relaxed);
  if (c > 0) return c;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(num_sms & ~1));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = PSmem::kTotal;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)pair_gemm_kernel<M>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  cached.store(n, std::memory_order_relaxed);  // every thread computes the same value
  return n;
}

template <PMode M>
cudaError_t launch_pair(const ds4moe_layer* L, const CUtensorMap& a, const CUtensorMap& sfa, const CUtensorMap& sfb,
                        const CUtensorMap* b, const PairArgs& args, cudaStream_t st) {
  // b: the 3-D token-row maps of 16, 32, ..., 128 rows (a CTA holds at most kPNMax / 2 = 96)
  BoxMaps maps;
  for (int i = 0; i < kNumBoxMaps; ++i) maps.m[i] = b[i < 8 ? i : 7];
  static InitOnce attr_once;
  cudaError_t e = init_once(attr_once, [] {
    return cudaFuncSetAttribute((const void*)pair_gemm_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PSmem::kTotal);
  });
  if (e != cudaSuccess) return e;
  const int per_e = M == PMode::GateUp ? args.rows_per_expert / 128 : (args.rows_per_expert + 255) / 256;
  const int units = args.E * per_e;
  const int mp = max_pairs<M>(L->num_sms);
  const int pairs = units < mp ? units : mp;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = PSmem::kTotal;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<M>, a, sfa, sfb, maps, args);
}

PairArgs pair_args(const ds4moe_layer* L, int split) {
  PairArgs a{};
  a.counts = L->s.counts;
  a.touched = L->s.touched;
  a.pad_offsets = L->s.pad_offsets;
  a.pad_pair = L->s.pad_pair;
  a.topk_w = L->s.topk_w;
  a.E = L->cfg.n_experts;
  a.k = L->cfg.top_k;
  a.d = L->cfg.d_model;
  a.f = L->cfg.d_ff;
  a.status = L->status;
  a.r128 = (int)(L->s.pad_rows_max / 128);
  a.debug_fault = L->cfg.debug_fault;
  a.split = split;
  a.budget_ns = L->cfg.debug_fault ? 1000000ull : (uint64_t)L->cfg.wait_timeout_ms * 1000000ull;
  return a;
}

}  // namespace

cudaError_t launch_gemm_gateup(const ds4moe_layer* L, int T, int split, cudaStream_t st) {
  (void)T;
  PairArgs a = pair_args(L, split);
  a.rows_per_expert = L->cfg.d_ff;
  a.K = L->cfg.d_model;
  a.hq = L->s.hq;
  a.hsf = L->s.hsf;
  a.h16 = (L->cfg.down_format == DS4MOE_DOWN_Q2K) ? L->s.h16 : nullptr;
  return launch_pair<PMode::GateUp>(L, L->tm_gu3, L->tm_sfa_gu, L->tm_sfb_x, L->tm_xq3, a, st);
}

cudaError_t launch_gemm_down(const ds4moe_layer* L, float* out, int T, int split, cudaStream_t st) {
  (void)T;
  PairArgs a = pair_args(L, split);
  a.debug_fault = 0;
  a.rows_per_expert = L->cfg.d_model;
  a.K = L->cfg.d_ff;
  a.out = out;
  return launch_pair<PMode::Down>(L, L->tm_dn3, L->tm_sfa_dn, L->tm_sfb_h, L->tm_hq3, a, st);
}

}  // namespace ds4moe
