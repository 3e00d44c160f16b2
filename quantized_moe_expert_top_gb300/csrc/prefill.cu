// Prefill (many-token) path of the routed-MoE layer: grouped block-scaled
// GEMMs on the 5th-generation tensor cores.
//
// "DwarfStar実地分析" §GGUFの対応範囲は意図的に狭い states that on Blackwell CUDA
// the batched expert work runs on FP4 matrix instructions.  Here every expert's
// tokens form one GEMM with the weights as the M side (swap-AB: 128 weight rows
// per tile, the expert's tokens as N, so a ragged token count only pads N to 16):
//
//   gate/up : tcgen05.mma kind::mxf8f6f4 block_scale, A = E2M1 weights (TMA
//             expands the packed nibbles into the 16-byte-aligned layout the
//             MMA reads), B = E4M3 activations, one E8M0 scale per 32 K for
//             both, fp32 accumulators in tensor memory.  Gate and up rows go
//             to two accumulators, so the epilogue has g and u of the same
//             (unit, token) in one thread: it applies SwiGLU and quantises h
//             to MXFP8 along f (or to fp16 for the Q2_K down projection).
//   down    : same MMA on h; the epilogue multiplies by the routing weight and
//             red-adds into out[t] (the weighted combine back to token order).
//
// Warp roles per CTA (persistent, one CTA per SM): warp 0 issues TMA loads,
// warp 1 allocates tensor memory and issues MMAs, warps 2..5 drain the
// accumulators.  Every mbarrier wait is bounded; a wait that runs out records
// DS4MOE_ERR_DEVICE_TIMEOUT in the layer's status word, the CTA drains its
// in-flight copies and MMAs (again bounded), frees its tensor memory and exits.
#include "common.cuh"
#include "internal.h"

namespace ds4moe {
namespace {

// --------------------------------------------------------------- MXFP8 of x
// One warp per token.  Lane l quantises blocks l, l+32, ... of x[t] (32 bf16
// each) to E4M3 with one E8M0 scale (s = floor(log2 amax) - 8, clamped; 0 for
// an all-zero block), then writes the codes and the scale to the k padded rows
// of the token's routed pairs.  Also zeroes out[t] for the down epilogue.
// Activation scales use the K-block-major chunk layout [K/128][rows/128][512]
// so the chunks of consecutive 128-row blocks are adjacent.
__device__ __forceinline__ size_t act_sf_index(size_t row, int kblk, int r128) {
  return ((size_t)(kblk / 4) * r128 + row / 128) * kSfChunk + (row % 32) * 16 + ((row % 128) / 32) * 4 + (kblk % 4);
}

// Two E4M3 codes (low byte first) -> their values as f32.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two) {
  uint32_t h;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "r"(two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// MXFP8 of one 32-value block: E8M0 exponent s (floor(log2 amax) - 8, clamped;
// 0 for an all-zero block) and the 32 codes packed little-endian in 8 words.
__device__ __forceinline__ int mxfp8_block(const float (&v)[32], uint32_t (&packed)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int s = 0;
  if (amax > 0.f) s = max(-127, min(127, floor_log2_f32(amax) - 8));
  const float inv = exp2i(-s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = f32x2_to_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
    const uint32_t hi = f32x2_to_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    packed[i] = lo | (hi << 16);
  }
  return s;
}

__global__ void __launch_bounds__(256) act_quant_kernel(const __nv_bfloat16* __restrict__ x, int T, int d, int k,
                                                        const int32_t* __restrict__ pad_inv, uint8_t* __restrict__ xq,
                                                        uint8_t* __restrict__ xsf, int r128, int split,
                                                        float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  {
    float4* o = reinterpret_cast<float4*>(out + (size_t)t * d);
    for (int i = lane; i < d / 4; i += 32) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  int rows[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) rows[j] = (j < k) ? __ldg(pad_inv + (size_t)t * k + j) : 0;
  const int nblk = d / 32;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  for (int c = lane; c < nblk; c += 32) {
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = __ldg(src + 4 * c + q);
      const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        v[8 * q + 2 * h] = __uint_as_float(wv[h] << 16);
        v[8 * q + 2 * h + 1] = __uint_as_float(wv[h] & 0xFFFF0000u);
      }
    }
    uint32_t packed[8], packed_lo[8];
    const int s = mxfp8_block(v, packed);
    int s_lo = 0;
    if (split == 2) {  // residual after the hi codes, quantised the same way
      const float sc = exp2i(s);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 a = e4m3x2_to_f32x2(packed[i] & 0xFFFFu), b = e4m3x2_to_f32x2(packed[i] >> 16);
        v[4 * i] -= a.x * sc;
        v[4 * i + 1] -= a.y * sc;
        v[4 * i + 2] -= b.x * sc;
        v[4 * i + 3] -= b.y * sc;
      }
      s_lo = mxfp8_block(v, packed_lo);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const size_t r = (size_t)rows[j];
        uint4* dst = reinterpret_cast<uint4*>(xq + r * d + 32 * (size_t)c);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        xsf[act_sf_index(r, c, r128)] = (uint8_t)(s + 127);
        if (split == 2) {
          uint4* dlo = reinterpret_cast<uint4*>(xq + (r + 1) * d + 32 * (size_t)c);
          dlo[0] = make_uint4(packed_lo[0], packed_lo[1], packed_lo[2], packed_lo[3]);
          dlo[1] = make_uint4(packed_lo[4], packed_lo[5], packed_lo[6], packed_lo[7]);
          xsf[act_sf_index(r + 1, c, r128)] = (uint8_t)(s_lo + 127);
        }
      }
    }
  }
}

// --------------------------------------------------------------- GEMM
enum class Mode { GateUp, Down, DownQ2K };

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A/B formats
// (E4M3 = 0, E2M1 = 5), K-major A and B, N >> 3, E8M0 scales, M >> 4, and the
// byte of the 32-bit scale word (one per 32-K step) used for A and B.
__device__ __forceinline__ uint32_t idesc_mx(int N, uint32_t sf_id) {
  constexpr uint32_t kE2M1 = 5, kE4M3 = 0;
  return (sf_id << 4) | (kE2M1 << 7) | (kE4M3 << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(kBM >> 4) << 24) | (sf_id << 29);
}

// Instruction descriptor, kind::f16: f16 A and B, f32 D, K-major, N >> 3, M >> 4.
__device__ __forceinline__ uint32_t idesc_f16(int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// Tensor-memory plan (512 columns): accumulator buffer(s) at columns 0 and
// 256, scale-factor slots from column 448 up.  One pipeline stage covers kKs
// contraction elements (128 bytes of every operand row).
template <Mode M>
struct Cfg;
template <>
struct Cfg<Mode::GateUp> {
  static constexpr int kNumA = 2;       // gate and up tiles
  static constexpr int kNMax = 160;     // token columns per chunk
  static constexpr int kStages = 4;
  static constexpr int kAccBufs = 1;    // G at column 0, U at column 256
  static constexpr int kSfSlot = 16;    // SFA gate 4 + SFA up 4 + SFB 8 columns
  static constexpr int kKs = 128;       // E2M1 / E4M3 elements per stage
  static constexpr int kDeqWarps = 0;
  static constexpr int kEpiWarps = 12;  // three per tensor-memory lane quarter (SwiGLU + MXFP8 epilogue)
};
template <>
struct Cfg<Mode::Down> {
  static constexpr int kNumA = 1;
  static constexpr int kNMax = 192;
  static constexpr int kStages = 4;
  static constexpr int kAccBufs = 2;    // double-buffered: columns 0 and 256
  static constexpr int kSfSlot = 12;    // SFA 4 + SFB 8 columns
  static constexpr int kKs = 128;
  static constexpr int kDeqWarps = 0;
  static constexpr int kEpiWarps = 8;   // two per lane quarter
};
template <>
struct Cfg<Mode::DownQ2K> {
  static constexpr int kNumA = 1;
  static constexpr int kNMax = 192;
  static constexpr int kStages = 4;
  static constexpr int kAccBufs = 2;
  static constexpr int kSfSlot = 0;
  static constexpr int kKs = 64;        // fp16 elements per stage
  static constexpr int kDeqWarps = 4;   // Q2_K -> fp16 producers, one weight row per thread
  static constexpr int kEpiWarps = 8;
};
constexpr int kAccCol2 = 256;
constexpr int kSfBase = 448;
constexpr int kSfSlots = 4;
// Warps: 0 TMA producer, 1 MMA issuer, then the epilogue warps, the Q2_K
// dequant warps, and last one helper warp (scale factors / Q2_K chunks by
// cp.async, L2 prefetch of weight tiles ahead of their TMA load).
template <Mode M>
constexpr int threads_of() { return 64 + 32 * Cfg<M>::kEpiWarps + 32 * Cfg<M>::kDeqWarps + 32; }

// Token-tile tensor maps, one per box height 16, 32, ..., 192 rows.
struct alignas(64) BoxMaps {
  CUtensorMap m[kNumBoxMaps];
};
constexpr int kPrefetchStages = 8;     // weight tiles prefetched into L2 ahead of their load
static_assert(kSfSlots >= Cfg<Mode::GateUp>::kStages && kSfSlots >= Cfg<Mode::Down>::kStages, "scale slots");
static_assert(kSfBase + kSfSlots * Cfg<Mode::GateUp>::kSfSlot <= 512, "tmem");
static_assert(Cfg<Mode::GateUp>::kNMax <= 256 && kAccCol2 + Cfg<Mode::GateUp>::kNMax <= kSfBase, "tmem");
static_assert(kAccCol2 + Cfg<Mode::Down>::kNMax <= kSfBase, "tmem");

template <Mode M>
struct Smem {
  static constexpr int kA = kBM * 128;                    // 16 KB per weight tile (128-byte rows)
  static constexpr int kB = Cfg<M>::kNMax * 128;           // token tile
  static constexpr int kSf = M == Mode::DownQ2K ? 4096    // Q2_K chunk
                                                : (kSfChunk * (Cfg<M>::kNumA + 2) + 1023) / 1024 * 1024;
  static constexpr int kStage = Cfg<M>::kNumA * kA + kB + kSf;
  static constexpr int kColOff = Cfg<M>::kStages * kStage;  // down: per-column (token, weight) table
  static constexpr int kBarOff = kColOff + Cfg<M>::kNMax * 8;
  static constexpr int kTotal = kBarOff + 256 + 1024;       // + barriers, + alignment slack
};
static_assert(Smem<Mode::GateUp>::kStage % 1024 == 0, "stage alignment");
static_assert(Smem<Mode::Down>::kStage % 1024 == 0, "stage alignment");
static_assert(Smem<Mode::DownQ2K>::kStage % 1024 == 0, "stage alignment");

struct GemmArgs {
  // weights
  const uint8_t* sfa;   // chunk-layout scales of the A tile(s): kNumA x 512 B per (tile, K step)
  int rows_per_expert;  // f (gate/up) or d (down)
  int r128;             // 128-row blocks of the activation buffers (scale layout pitch)
  int K;                // d (gate/up) or f (down)
  // activations (B)
  const uint8_t* sfb;   // chunk-layout scales of the B rows
  // routing
  const int32_t* counts;
  const int32_t* touched;  // experts with tokens, ascending, then their number at [E]
  const int32_t* pad_offsets;
  const int32_t* pad_pair;
  const float* topk_w;
  int E, k, d, f;
  const uint8_t* q2k;  // Q2_K down: tile-major chunks
  const uint8_t* wbase;  // weight rows the A tiles come from (L2 prefetch)
  int wpitch;
  // outputs
  uint8_t* hq;    // gate/up: MXFP8 h codes [rows][f]
  uint8_t* hsf;   // gate/up: h scales (chunk layout)
  __half* h16;    // gate/up: fp16 h (Q2_K down), or nullptr
  float* out;     // down: [T][d]
  DeviceStatus* status;
  uint64_t budget_ns;
  int debug_fault;
  int split;  // activation rows (token columns) per routed pair: 1, or 2 (hi + lo)
};

// Work sequence shared by the roles: units u = (touched expert, 128-row
// block), expert-major, strided over the CTAs, so that units are dealt evenly
// whatever experts the tokens chose; each unit's tokens split into chunks that
// start on a 128-token boundary (one chunk when they fit in kNMax).
struct UnitIter {
  int u, nunits, stride, mb_per_e;
  int e, mb, ne, t0, nch;  // ne, t0, nch count token columns (split * routed pairs)
  const int32_t* counts;
  const int32_t* touched;
  int nmax;
  int split;
  __device__ bool first_chunk() {
    for (; u < nunits; u += stride) {
      e = __ldg(touched + u / mb_per_e);
      mb = u % mb_per_e;
      ne = __ldg(counts + e) * split;
      if (ne > 0) {
        t0 = 0;
        nch = ne <= nmax ? ne : 128;
        return true;
      }
    }
    return false;
  }
  __device__ bool next() {
    t0 += nch;
    if (t0 < ne) {
      const int rem = ne - t0;
      nch = rem <= nmax ? rem : 128;
      return true;
    }
    u += stride;
    return first_chunk();
  }
};

// The same sequence one pipeline stage at a time (the producer's L2 prefetch
// cursor runs kPrefetchStages ahead of its load cursor).
struct StageIter {
  UnitIter it;
  int kb, KB;
  bool valid;
  __device__ void start() {
    kb = 0;
    valid = it.first_chunk();
  }
  __device__ void next() {
    if (!valid) return;
    if (++kb < KB) return;
    kb = 0;
    valid = it.next();
  }
};

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

template <Mode M>
__global__ void __launch_bounds__(threads_of<M>(), 1) grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                                                                       const __grid_constant__ BoxMaps bmaps,
                                                                       const GemmArgs args) {
  using C = Cfg<M>;
  using S = Smem<M>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* col_tok = reinterpret_cast<int32_t*>(smem + S::kColOff);
  float* col_w = reinterpret_cast<float*>(col_tok + C::kNMax);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);  // TMA bytes of a stage
  uint64_t* empty = full + C::kStages;
  uint64_t* afull = empty + C::kStages;      // Q2_K: dequantised A tile written
  uint64_t* acc_full = afull + C::kStages;   // [kAccBufs]
  uint64_t* acc_empty = acc_full + 2;        // [kAccBufs]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_ok = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mb_per_e = args.rows_per_expert / kBM;
  const int KB = args.K / C::kKs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1 + 32);  // producer (TMA bytes) + helper lanes (cp.async)
      mbar_init(&empty[s], 1);
      mbar_init(&afull[s], C::kDeqWarps > 0 ? C::kDeqWarps : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    if (M != Mode::DownQ2K) prefetch_tmap(&tm_a);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the routing tables and activations of this forward are complete from here on
  pdl_launch_dependents();
  const int nunits = __ldg(args.touched + args.E) * mb_per_e;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      StageIter ld{{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched, C::kNMax, args.split},
                   0, KB, false};
      ld.start();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool fault_pending = args.debug_fault && blockIdx.x == 0;
      bool ok = true;
      UnitIter it = ld.it;
      for (bool more = ld.valid; more && ok; more = it.next()) {
        // per-chunk constants
        const int N = round16(it.nch);
        const int nsf = (N + 127) / 128;
        // token rows in TMA boxes of 128 / 64 / 32 rows (at most two for N <= 192)
        const CUtensorMap* tb = &bmaps.m[N / 16 - 1];  // one box of exactly N token rows
        const int prow = __ldg(args.pad_offsets + it.e) + it.t0;
        const int arow = (it.e * mb_per_e + it.mb) * kBM * C::kNumA;  // gate+up: 256-row box
        // A 4-bit unpacking load counts its packed global bytes (half the
        // 16 KB it writes to shared memory).
        const uint32_t bytes = (uint32_t)((M == Mode::DownQ2K ? 0 : C::kNumA * S::kA / 2) + N * 128);
        (void)nsf;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, args.budget_ns, abort_flag)) {
            report_timeout(args.status, kWhereProducerEmpty);
            *abort_flag = 1;
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * S::kStage;
          uint8_t* sb = st + C::kNumA * S::kA;
          mbar_arrive_expect_tx(&full[stage], bytes);
          if (fault_pending) {
            fault_pending = false;  // test-only: drop this stage's loads
          } else {
            tma_load_2d(sb, tb, &full[stage], kb * C::kKs, prow);
            if constexpr (M != Mode::DownQ2K) tma_load_2d(st, &tm_a, &full[stage], kb * C::kKs, arow);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        // drain: every issued stage's copies must land before the CTA exits
        for (int s = 0; s < C::kStages; ++s)
          if ((issued_mask >> s) & 1u) {
            volatile int never = 0;
            mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, args.budget_ns, &never);
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      UnitIter it{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched, C::kNMax, args.split};
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;  // acc_phase bit b: phase of accumulator buffer b
      uint32_t sf_seq = 0;  // running stage count; slot = sf_seq % kSfSlots (kSfSlots >= kStages)
      int chunk = 0;
      bool ok = true;
      // Shared-memory descriptors of every stage slot, computed once: K steps
      // add 32 bytes (2 in the 16-byte address field) to the start address.
      // (Only the 14-bit start-address field differs between slots, so a slot
      // is the slot-0 descriptor plus slot * stage size in 16-byte units.)
      const uint32_t st0 = smem_u32(smem);
      const uint64_t adesc0 = smem_desc(st0, 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(st0 + C::kNumA * S::kA, 16, 1024, 2);
      const uint64_t sfdesc0 = smem_desc(st0 + C::kNumA * S::kA + S::kB, 0, 128, 0);
      static_assert(C::kStages * S::kStage < (1 << 18), "descriptor address field");
      for (bool more = it.first_chunk(); more && ok; more = it.next(), ++chunk) {
        const int N = round16(it.nch);
        const int nsf = (N + 127) / 128;
        const int buf = chunk % C::kAccBufs;
        const uint32_t acc0 = tmem + (uint32_t)(buf * kAccCol2);
        const uint32_t idesc0 = M == Mode::DownQ2K ? idesc_f16(N) : idesc_mx(N, 0);
        constexpr uint32_t kSfIdStep = (1u << 4) | (1u << 29);  // next byte of the 32-bit scale word, A and B
        if (!mbar_wait_bounded(&acc_empty[buf], ((acc_phase >> buf) & 1u) ^ 1u, args.budget_ns, abort_flag)) {
          report_timeout(args.status, kWhereMmaAccEmpty);
          *abort_flag = 1;
          break;
        }
        acc_phase ^= 1u << buf;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, args.budget_ns, abort_flag)) {
            report_timeout(args.status, kWhereMmaFull);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if constexpr (M == Mode::DownQ2K) {  // the dequantised A tile is written by the dequant warps
            if (!mbar_wait_bounded(&afull[stage], phase, args.budget_ns, abort_flag)) {
              report_timeout(args.status, kWhereMmaFull);
              *abort_flag = 1;
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint64_t soff = (uint64_t)(stage * (S::kStage >> 4));
          const uint64_t ad = adesc0 + soff, bd = bdesc0 + soff;
          if constexpr (M == Mode::DownQ2K) {
#pragma unroll
            for (int j = 0; j < 4; ++j)  // K = 16 fp16 (32 bytes) per instruction
              mma_f16(acc0, ad + 2 * j, bd + 2 * j, idesc0, (kb > 0 || j > 0) ? 1u : 0u);
          } else {
            // the scale factors were written by cp.async (generic proxy); tcgen05.cp reads through the async proxy
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint32_t slot = tmem + kSfBase + (sf_seq++ % kSfSlots) * C::kSfSlot;
            // scale factors -> tensor memory: A chunk(s) at slot+0 (+4), B chunks after (512 B = 32 units)
            const uint64_t sd = sfdesc0 + soff;
            for (int i = 0; i < C::kNumA + nsf; ++i) tc_cp_32x128b_warpx4(slot + 4 * i, sd + 32 * i);
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // K = 32 (32 bytes) per instruction
              const uint32_t idesc = idesc0 + (uint32_t)j * kSfIdStep;
              const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
              mma_mxf8f6f4(acc0, ad + 2 * j, bd + 2 * j, idesc, slot, slot + 4 * C::kNumA, accum);
              if (C::kNumA > 1)  // up tile: 16 KB (1024 address units) after the gate tile
                mma_mxf8f6f4(acc0 + kAccCol2, ad + 1024 + 2 * j, bd + 2 * j, idesc, slot + 4, slot + 4 * C::kNumA,
                             accum);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      // drain all MMAs this thread issued before tensor memory is freed
      tc_commit(drain);
      volatile int never = 0;
      mbar_wait_bounded(drain, 0, args.budget_ns, &never);
    }
    __syncwarp();
  } else if (warp == threads_of<M>() / 32 - 1) {
    // ------------------------------------------------------------ helper: scale factors / Q2_K chunks
    StageIter sq{{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched, C::kNMax, args.split},
                 0, KB, false};
    sq.start();
    StageIter pf = sq;  // L2 prefetch cursor, kPrefetchStages ahead
    auto l2_prefetch = [&](const StageIter& p) {
      const size_t tile = (size_t)(p.it.e * mb_per_e + p.it.mb) * KB + p.kb;
      if constexpr (M == Mode::DownQ2K) {
        if (lane < kQ2kChunk / 128) prefetch_l2(args.q2k + tile * kQ2kChunk + lane * 128);
      } else {
        const int arow = (p.it.e * mb_per_e + p.it.mb) * kBM * C::kNumA;
        for (int r = lane; r < kBM * C::kNumA; r += 32)
          prefetch_l2(args.wbase + (size_t)(arow + r) * args.wpitch + p.kb * (C::kKs / 2));
        if (lane < C::kNumA * kSfChunk / 128) prefetch_l2(args.sfa + tile * (C::kNumA * kSfChunk) + lane * 128);
      }
    };
    for (int i = 0; i < kPrefetchStages && pf.valid; ++i) {
      l2_prefetch(pf);
      pf.next();
    }
    int stage = 0;
    uint32_t phase = 0;
    while (sq.valid) {
      uint32_t got = 0;
      if (lane == 0) got = mbar_wait_bounded(&empty[stage], phase ^ 1u, args.budget_ns, abort_flag) ? 1u : 0u;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) {
          report_timeout(args.status, kWhereProducerEmpty);
          *abort_flag = 1;
        }
        break;
      }
      uint8_t* ssf = smem + stage * S::kStage + C::kNumA * S::kA + S::kB;
      const size_t tile = (size_t)(sq.it.e * mb_per_e + sq.it.mb) * KB + sq.kb;
      if constexpr (M == Mode::DownQ2K) {
        const uint8_t* src = args.q2k + tile * kQ2kChunk;
        for (int i = lane; i < kQ2kChunk / 16; i += 32) cp_async_16(ssf + 16 * i, src + 16 * i);
      } else {
        const int N = round16(sq.it.nch);
        const int nA = C::kNumA * kSfChunk / 16, nB = ((N + 127) / 128) * kSfChunk / 16;
        const int prow = __ldg(args.pad_offsets + sq.it.e) + sq.it.t0;
        const uint8_t* sfa = args.sfa + tile * (C::kNumA * kSfChunk);
        const uint8_t* sfb = args.sfb + ((size_t)sq.kb * args.r128 + prow / 128) * kSfChunk;
        for (int i = lane; i < nA + nB; i += 32)
          cp_async_16(ssf + 16 * i, i < nA ? sfa + 16 * i : sfb + 16 * (i - nA));
      }
      cp_async_arrive_noinc(&full[stage]);
      if (pf.valid) {
        l2_prefetch(pf);
        pf.next();
      }
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1u;
      }
      sq.next();
    }
    cp_async_wait_all();  // this warp's copies land before the CTA may exit
  } else if (warp >= 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ Q2_K dequant
    if constexpr (M == Mode::DownQ2K) {
      const int r = (warp - 2 - C::kEpiWarps) * 32 + lane;  // weight row of the 128-row tile
      StageIter sq{{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched, C::kNMax, args.split},
                   0, KB, false};
      sq.start();
      int stage = 0;
      uint32_t phase = 0;
      const __half2 k1024 = __float2half2_rn(1024.f);
      while (sq.valid) {
        uint32_t got = 0;
        if (lane == 0) got = mbar_wait_bounded(&full[stage], phase, args.budget_ns, abort_flag) ? 1u : 0u;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          if (lane == 0) {
            report_timeout(args.status, kWhereMmaFull);
            *abort_flag = 1;
          }
          break;
        }
        uint8_t* st = smem + stage * S::kStage;
        const uint8_t* ch = st + S::kA + S::kB;
        const uint4 qv = *reinterpret_cast<const uint4*>(ch + 16 * r);
        const uint32_t scw = *reinterpret_cast<const uint32_t*>(ch + 2048 + 4 * r);
        const uint32_t ddw = *reinterpret_cast<const uint32_t*>(ch + 2560 + 4 * r);
        const float dd = __half2float(__ushort_as_half((unsigned short)(ddw & 0xFFFFu)));
        const float dm = __half2float(__ushort_as_half((unsigned short)(ddw >> 16)));
        const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
        uint8_t* arow = st + r * 128;
#pragma unroll
        for (int sb = 0; sb < 4; ++sb) {  // sub-block sb = weights 16 sb .. 16 sb + 15 of the step
          const uint32_t scb = (scw >> (8 * sb)) & 0xFFu;
          const __half2 a2 = __float2half2_rn(dd * (float)(scb & 15u));
          const __half2 nb2 = __float2half2_rn(-dm * (float)(scb >> 4));
          uint32_t P[8];  // P[n] = {w_n, w_(n+8)}: 2-bit codes 16 bits apart in the word
#pragma unroll
          for (int n = 0; n < 8; ++n) {
            const uint32_t v = ((words[sb] >> (2 * n)) & 0x00030003u) | 0x64006400u;  // f16 1024 + q
            const __half2 q2 = __hsub2(*reinterpret_cast<const __half2*>(&v), k1024);
            const __half2 w2 = __hfma2(q2, a2, nb2);
            P[n] = *reinterpret_cast<const uint32_t*>(&w2);
          }
          const uint4 lo = make_uint4(__byte_perm(P[0], P[1], 0x5410), __byte_perm(P[2], P[3], 0x5410),
                                      __byte_perm(P[4], P[5], 0x5410), __byte_perm(P[6], P[7], 0x5410));
          const uint4 hi = make_uint4(__byte_perm(P[0], P[1], 0x7632), __byte_perm(P[2], P[3], 0x7632),
                                      __byte_perm(P[4], P[5], 0x7632), __byte_perm(P[6], P[7], 0x7632));
          // 16-byte chunks 2 sb and 2 sb + 1 of the row, 128-byte swizzle
          *reinterpret_cast<uint4*>(arow + (((2 * sb) ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(arow + (((2 * sb + 1) ^ (r & 7)) << 4)) = hi;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        sq.next();
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // tensor-memory lane quarter this warp may access
    const int part = (warp - 2) >> 2;   // which share of the 16-column chunks
    constexpr int kParts = C::kEpiWarps / 4;
    const int etid = threadIdx.x - 64;  // index among the epilogue threads
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    UnitIter it{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched, C::kNMax, args.split};
    uint32_t acc_phase = 0;
    int chunk = 0;
    for (bool more = it.first_chunk(); more; more = it.next(), ++chunk) {
      const int N = round16(it.nch);
      const int prow = __ldg(args.pad_offsets + it.e) + it.t0;
      const int buf = chunk % C::kAccBufs;
      uint32_t got = 0;
      if (M != Mode::GateUp) {
        // Per-column token and routing weight, loaded while the MMAs run.  One
        // thread takes the accumulator wait and publishes the outcome, so all
        // epilogue warps leave the loop together (the named barriers need
        // every one of them).
        named_bar_sync(1, 32 * C::kEpiWarps);  // previous chunk's table no longer read
        for (int c = etid; c < it.nch; c += 32 * C::kEpiWarps) {
          const int pair = __ldg(args.pad_pair + prow + c);
          col_tok[c] = pair / args.k;
          col_w[c] = __ldg(args.topk_w + pair);
        }
        if (etid == 0) {
          const bool ok = mbar_wait_bounded(&acc_full[buf], (acc_phase >> buf) & 1u, args.budget_ns, abort_flag);
          *epi_ok = ok ? 1 : 0;
          if (!ok) {
            report_timeout(args.status, kWhereEpiAccFull);
            *abort_flag = 1;
          }
        }
        named_bar_sync(1, 32 * C::kEpiWarps);
        got = (uint32_t)*epi_ok;
        if (!got) break;
      } else {
        if (lane == 0)
          got = mbar_wait_bounded(&acc_full[buf], (acc_phase >> buf) & 1u, args.budget_ns, abort_flag) ? 1u : 0u;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          if (lane == 0) {
            report_timeout(args.status, kWhereEpiAccFull);
            *abort_flag = 1;
          }
          break;
        }
      }
      acc_phase ^= 1u << buf;
      tc_fence_after();
      const uint32_t acc0 = tmem + (uint32_t)(buf * kAccCol2) + lane_base;
      const int unit_row = it.mb * kBM + q * 32 + lane;  // row of this lane inside the expert
      for (int c0 = part * 16; c0 < N; c0 += 16 * kParts) {
        uint32_t r0[16];
        tmem_ld_32x32b_x16(acc0 + (uint32_t)c0, r0);
        if (M == Mode::GateUp) {
          uint32_t r1[16];
          tmem_ld_32x32b_x16(acc0 + (uint32_t)(kAccCol2 + c0), r1);
          tmem_ld_wait();
          const int i = unit_row;  // feature index in [0, f)
          if (args.split == 2) {
            // column pairs (hi, lo) of 8 tokens: add them, SwiGLU, then h -> hi + lo rows again
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const float g = __uint_as_float(r0[2 * jj]) + __uint_as_float(r0[2 * jj + 1]);
              const float u = __uint_as_float(r1[2 * jj]) + __uint_as_float(r1[2 * jj + 1]);
              const float h = __fdividef(g, 1.f + __expf(-g)) * u;
              const float a = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
              int s = 0;
              if (a > 0.f) s = max(-127, min(127, floor_log2_f32(a) - 8));
              const uint32_t chi = f32x2_to_e4m3x2(h * exp2i(-s), 0.f) & 0xFFu;
              const float res = h - e4m3x2_to_f32x2(chi).x * exp2i(s);
              const float a2 = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(res))));
              int s2 = 0;
              if (a2 > 0.f) s2 = max(-127, min(127, floor_log2_f32(a2) - 8));
              const uint32_t clo = f32x2_to_e4m3x2(res * exp2i(-s2), 0.f) & 0xFFu;
              const int col = c0 + 2 * jj;
              if (col < it.nch) {
                const size_t row = (size_t)(prow + col);
                args.hq[row * args.f + i] = (uint8_t)chi;
                args.hq[(row + 1) * args.f + i] = (uint8_t)clo;
                if (lane == 0) {
                  args.hsf[act_sf_index(row, i / 32, args.r128)] = (uint8_t)(s + 127);
                  args.hsf[act_sf_index(row + 1, i / 32, args.r128)] = (uint8_t)(s2 + 127);
                }
              }
            }
            continue;
          }
          float h[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const float g = __uint_as_float(r0[jj]), u = __uint_as_float(r1[jj]);
            h[jj] = __fdividef(g, 1.f + __expf(-g)) * u;
          }
          if (args.h16 != nullptr) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              if (c0 + jj < it.nch) args.h16[(size_t)(prow + c0 + jj) * args.f + i] = __float2half_rn(h[jj]);
          } else {
            uint32_t amax[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) amax[jj] = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h[jj])));
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int col = c0 + jj;
              if (col < it.nch) {
                const float a = __uint_as_float(amax[jj]);
                int s = 0;
                if (a > 0.f) s = max(-127, min(127, floor_log2_f32(a) - 8));
                const size_t row = (size_t)(prow + col);
                args.hq[row * args.f + i] = (uint8_t)(f32x2_to_e4m3x2(h[jj] * exp2i(-s), 0.f) & 0xFFu);
                if (lane == 0) args.hsf[act_sf_index(row, i / 32, args.r128)] = (uint8_t)(s + 127);
              }
            }
          }
        } else {
          tmem_ld_wait();
          const int m = unit_row;  // output feature
          if (args.split == 2) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int col = c0 + 2 * jj;
              if (col < it.nch)
                red_add_f32(args.out + (size_t)col_tok[col] * args.d + m,
                            col_w[col] * (__uint_as_float(r0[2 * jj]) + __uint_as_float(r0[2 * jj + 1])));
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int col = c0 + jj;
              if (col < it.nch)
                red_add_f32(args.out + (size_t)col_tok[col] * args.d + m, col_w[col] * __uint_as_float(r0[jj]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <Mode M>
cudaError_t launch_gemm(const ds4moe_layer* L, const CUtensorMap& a, const CUtensorMap* b, const GemmArgs& args,
                        cudaStream_t st) {
  BoxMaps maps;
  for (int i = 0; i < kNumBoxMaps; ++i) maps.m[i] = b[i];
  static_assert(Smem<M>::kTotal <= 227 * 1024, "shared memory");
  const void* fn = (const void*)grouped_gemm_kernel<M>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<M>::kTotal);
  if (e != cudaSuccess) return e;
  const int units = args.E * (args.rows_per_expert / kBM);
  const int grid = units < L->num_sms ? units : L->num_sms;
  return launch_pdl(grouped_gemm_kernel<M>, grid, threads_of<M>(), Smem<M>::kTotal, st, a, maps, args);
}

}  // namespace

cudaError_t launch_act_quant(const ds4moe_layer* L, const void* x, float* out, int T, int split, cudaStream_t st) {
  const int blocks = (T + 7) / 8;
  return launch_pdl(act_quant_kernel, blocks, 256, 0, st, static_cast<const __nv_bfloat16*>(x), T, L->cfg.d_model,
                    L->cfg.top_k, L->s.pad_inv, L->s.xq, L->s.xsf, (int)(L->s.pad_rows_max / 128), split, out);
}

static GemmArgs base_args(const ds4moe_layer* L) {
  GemmArgs a{};
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
  a.split = 1;
  a.budget_ns = L->cfg.debug_fault ? 1000000ull : (uint64_t)L->cfg.wait_timeout_ms * 1000000ull;
  return a;
}

cudaError_t launch_gemm_gateup(const ds4moe_layer* L, int T, int split, cudaStream_t st) {
  (void)T;
  GemmArgs a = base_args(L);
  a.split = split;
  a.sfa = L->w.gu_sf;
  a.wbase = L->w.gu;
  a.wpitch = L->w.pitch_gu;
  a.rows_per_expert = L->cfg.d_ff;
  a.K = L->cfg.d_model;
  a.sfb = L->s.xsf;
  a.hq = L->s.hq;
  a.hsf = L->s.hsf;
  a.h16 = (L->cfg.down_format == DS4MOE_DOWN_Q2K) ? L->s.h16 : nullptr;
  return launch_gemm<Mode::GateUp>(L, L->tm_gu, L->tm_xq, a, st);
}

cudaError_t launch_gemm_down(const ds4moe_layer* L, float* out, int T, int split, cudaStream_t st) {
  (void)T;
  GemmArgs a = base_args(L);
  a.split = split;
  a.debug_fault = 0;
  a.sfa = L->w.down_sf;
  a.wbase = L->w.dn;
  a.wpitch = L->w.pitch_dn;
  a.rows_per_expert = L->cfg.d_model;
  a.K = L->cfg.d_ff;
  a.sfb = L->s.hsf;
  a.out = out;
  return launch_gemm<Mode::Down>(L, L->tm_down, L->tm_hq, a, st);
}

cudaError_t launch_gemm_down_q2k(const ds4moe_layer* L, float* out, int T, cudaStream_t st) {
  (void)T;
  GemmArgs a = base_args(L);
  a.debug_fault = 0;
  a.q2k = L->w.q2k;
  a.rows_per_expert = L->cfg.d_model;
  a.K = L->cfg.d_ff;
  a.out = out;
  return launch_gemm<Mode::DownQ2K>(L, L->tm_h16[0], L->tm_h16, a, st);
}

int prefill_launches() { return 5; }

}  // namespace ds4moe
