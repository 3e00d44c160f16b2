// Activation quantisation of the GEMM paths and the Q2_K down projection.
//
//   act_quant : x (bf16) -> MXFP8 rows in expert-grouped order for the grouped
//               GEMMs (and, for the few-token path, a second "lo" row holding
//               the MXFP8 residual), and zeroes out[] for the combine.
//   q2k down  : "DwarfStar実地分析" §GGUFの対応範囲は意図的に狭い describes the
//               engine's asymmetric 2-bit scheme with a Q2_K down projection.
//               Dequantisation warps expand each Q2_K tile to fp16 in tensor
//               memory (w = d*sc*q - dmin*m, tcgen05.st), and tcgen05.mma
//               kind::f16 reads it there as the M side (swap-AB) and the fp16
//               h of the expert's tokens from shared memory; the epilogue
//               multiplies by the routing weight and red-adds into out[t].
//               Keeping the weight tile out of shared memory halves that
//               memory's traffic per step, which bounded the kernel.
//
// The Q2_K GEMM is persistent, one CTA per SM: warp 0 issues the TMA loads of
// h, warp 1 allocates tensor memory and issues the MMAs, warps 2..9 drain the
// double-buffered accumulator, warps 10..17 dequantise into tensor memory (two
// groups of four taking alternate 128-weight steps, one thread per weight row),
// warps 18 and 19 stream the Q2_K chunks with bulk copies into a ring of kQRaw
// slots that runs far ahead of the dequantisation, and warp 20 shares the h
// loads with warp 0.  Every mbarrier wait is bounded; a wait that
// runs out records DS4MOE_ERR_DEVICE_TIMEOUT in the layer's status word and
// the CTA drains its in-flight copies and MMAs (again bounded) before it exits.
#include "gemm.cuh"

namespace ds4moe {
namespace {

// --------------------------------------------------------------- MXFP8 of x
// One warp per (token, 1024 elements): lane l quantises one block of 32 bf16
// to E4M3 with one E8M0 scale (s = floor(log2 amax) - 8, clamped; 0 for an
// all-zero block), then writes the codes and the scale to the k padded rows of
// the token's routed pairs (and the residual as a second row when split).
// Also zeroes the warp's part of out[t] for the down epilogue.
__global__ void __launch_bounds__(256) act_quant_kernel(const __nv_bfloat16* __restrict__ x, int T, int d, int k,
                                                        const int32_t* __restrict__ pad_inv, uint8_t* __restrict__ xq,
                                                        uint8_t* __restrict__ xsf, int r128, int split,
                                                        float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  // one warp per (token, 32 consecutive blocks of 32 elements); lane = block
  const int nblk = d / 32, parts = (nblk + 31) / 32;
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int t = gw / parts, part = gw % parts;
  if (t >= T) return;
  {
    float4* o = reinterpret_cast<float4*>(out + (size_t)t * d + (size_t)part * 1024);
    const int n4 = min(1024, d - part * 1024) / 4;
    for (int i = lane; i < n4; i += 32) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int c = part * 32 + lane;
  // lanes past the row leave in whole groups of four (nblk % 4 == 0)
  const unsigned vmask = __ballot_sync(0xffffffffu, c < nblk);
  if (c >= nblk) return;
  int rows[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) rows[j] = (j < k) ? __ldg(pad_inv + (size_t)t * k + j) : 0;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
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
  int s_lo = 0;
  const int s = split == 2 ? mxfp8_split_block(v, packed, packed_lo, s_lo) : mxfp8_block(v, packed);
  // The scales of blocks 4i .. 4i + 3 of a row are 4 consecutive bytes of its
  // scale chunk: lane 4i gathers them and stores one word.
  uint32_t sw = (uint32_t)(s + 127) << (8 * (lane & 3));
  uint32_t sw_lo = (uint32_t)(s_lo + 127) << (8 * (lane & 3));
  sw |= __shfl_xor_sync(vmask, sw, 1);
  sw |= __shfl_xor_sync(vmask, sw, 2);
  sw_lo |= __shfl_xor_sync(vmask, sw_lo, 1);
  sw_lo |= __shfl_xor_sync(vmask, sw_lo, 2);
  if (vmask == 0xffffffffu) {
    // The warp's 32 blocks are 1 KB of a row: staged in shared memory, they
    // go out as two 512-byte contiguous stores per routed row (a lane's own
    // 32 bytes would be two half-sector pieces).
    __shared__ uint4 stage[8][2][64];  // [warp of the block][hi, lo][16-byte piece]
    uint4* sh = stage[(threadIdx.x >> 5) & 7][0];
    uint4* sl = stage[(threadIdx.x >> 5) & 7][1];
    sh[2 * lane] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    sh[2 * lane + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    if (split == 2) {
      sl[2 * lane] = make_uint4(packed_lo[0], packed_lo[1], packed_lo[2], packed_lo[3]);
      sl[2 * lane + 1] = make_uint4(packed_lo[4], packed_lo[5], packed_lo[6], packed_lo[7]);
    }
    __syncwarp();
    const uint4 h0 = sh[lane], h1 = sh[32 + lane];
    uint4 l0 = h0, l1 = h1;
    if (split == 2) {
      l0 = sl[lane];
      l1 = sl[32 + lane];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const size_t r = (size_t)rows[j];
        uint4* dst = reinterpret_cast<uint4*>(xq + r * d + (size_t)part * 1024);
        dst[lane] = h0;
        dst[32 + lane] = h1;
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(xsf + act_sf_index(r, c, r128)) = sw;
        if (split == 2) {
          uint4* dlo = reinterpret_cast<uint4*>(xq + (r + 1) * d + (size_t)part * 1024);
          dlo[lane] = l0;
          dlo[32 + lane] = l1;
          if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(xsf + act_sf_index(r + 1, c, r128)) = sw_lo;
        }
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      const size_t r = (size_t)rows[j];
      uint4* dst = reinterpret_cast<uint4*>(xq + r * d + 32 * (size_t)c);
      dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(xsf + act_sf_index(r, c, r128)) = sw;
      if (split == 2) {
        uint4* dlo = reinterpret_cast<uint4*>(xq + (r + 1) * d + 32 * (size_t)c);
        dlo[0] = make_uint4(packed_lo[0], packed_lo[1], packed_lo[2], packed_lo[3]);
        dlo[1] = make_uint4(packed_lo[4], packed_lo[5], packed_lo[6], packed_lo[7]);
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(xsf + act_sf_index(r + 1, c, r128)) = sw_lo;
      }
    }
  }
}

// --------------------------------------------------------------- Q2_K down GEMM
// Tensor memory (512 columns): accumulator buffers at columns 0 and kQAcc1,
// the fp16 weight tiles of the stages between them.  One pipeline stage covers
// kQKs = 128 contraction elements: two 64-element sub-steps, each a Q2_K
// chunk of the weights and a 128-byte-wide block of h.  Fewer, larger steps
// halve the barrier hand-offs per weight byte, which bounded the kernel.
constexpr int kQNMax = 128;      // token columns per chunk
constexpr int kQStages = 4;
constexpr int kQSub = 2;         // 64-element sub-steps per stage
constexpr int kQKs = 64 * kQSub;  // fp16 elements per stage
constexpr int kQRaw = 12;        // slots of the raw ring, kQSub Q2_K chunks each (72 KB of weights in flight)
constexpr int kQASlot0 = 128;    // tensor-memory columns of the fp16 weight tiles: 32 per sub-step
constexpr int kQDeqWarps = 8;    // kQDeqGroups groups of four: one thread per weight row and step
constexpr int kQDeqGroups = kQDeqWarps / 4;
constexpr int kQEpiWarps = 8;    // kQEpiWarps / 4 per tensor-memory lane quarter
static_assert(kQEpiWarps % 4 == 0, "epilogue warps cover the lane quarters");
constexpr int kQAcc1 = 384;
// The h tiles and the raw chunks are each issued by kQIssuers threads in
// different warps, taking alternate steps.
constexpr int kQIssuers = 2;
constexpr int kQThreads = 64 + 32 * kQEpiWarps + 32 * kQDeqWarps + 32 * (2 * kQIssuers - 1);
static_assert(kQStages % kQIssuers == 0 && kQRaw % kQIssuers == 0, "an issuer owns fixed slots");
static_assert(kQNMax <= kQASlot0 && kQASlot0 + 32 * kQSub * kQStages <= kQAcc1 && kQAcc1 + kQNMax <= 512,
              "tensor memory");

struct QSmem {
  static constexpr int kB = kQSub * kQNMax * 128;  // fp16 token tiles [kQSub][N][128 B] (weights in tensor memory)
  static constexpr int kStage = kB;
  static constexpr int kRawSlot = kQSub * kQ2kChunk;  // bytes of one raw slot
  static constexpr int kRawOff = kQStages * kStage;
  static constexpr int kColOff = kRawOff + kQRaw * kRawSlot;  // per-column (token, routing weight)
  static constexpr int kBarOff = kColOff + kQNMax * 8;
  static constexpr int kTotal = kBarOff + 1024 + 1024;  // barriers (17 + 2 * kQRaw) and flags, alignment slack
};
static_assert(QSmem::kStage % 1024 == 0, "stage alignment");
static_assert(QSmem::kTotal <= 227 * 1024, "shared memory");
static_assert((3 * kQStages + 5 + 2 * kQRaw) * 8 + 16 <= 1024, "barrier area");

struct Q2kArgs {
  const uint8_t* q2k;  // tile-major chunks [E][d/128][f/64][3072]
  const int32_t* counts;
  const int32_t* touched;
  const int32_t* pad_offsets;
  const int32_t* pad_pair;
  const float* topk_w;
  int E, k, d, f;
  int rpp;       // padded activation rows per routed pair (1, or 2 on the few-token path); h has one
                 // row per pair, expert e's first at pad_offsets[e] / rpp
  float* out;
  DeviceStatus* status;
  uint64_t budget_ns;
};

// Work sequence shared by the roles: units (touched expert, 128-row block of
// d), expert-major, strided over the CTAs; each unit's tokens split into chunks
// that start on a 128-token boundary (one chunk when they fit in kQNMax).
struct QIter {
  int u, nunits, stride, mb_per_e;
  int e, mb, ne, t0, nch;
  const int32_t* counts;
  const int32_t* touched;
  __device__ bool first_chunk() {
    for (; u < nunits; u += stride) {
      e = __ldg(touched + u / mb_per_e);
      mb = u % mb_per_e;
      ne = __ldg(counts + e);
      if (ne > 0) {
        t0 = 0;
        nch = ne <= kQNMax ? ne : 128;
        return true;
      }
    }
    return false;
  }
  __device__ bool next() {
    t0 += nch;
    if (t0 < ne) {
      const int rem = ne - t0;
      nch = rem <= kQNMax ? rem : 128;
      return true;
    }
    u += stride;
    return first_chunk();
  }
};


__global__ void __launch_bounds__(kQThreads, 1) q2k_down_kernel(const __grid_constant__ BoxMaps bmaps,
                                                              const Q2kArgs args) {
  using S = QSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* col_tok = reinterpret_cast<int32_t*>(smem + S::kColOff);
  float* col_w = reinterpret_cast<float*>(col_tok + kQNMax);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);  // h tile bytes + the Q2_K chunk copy
  uint64_t* empty = full + kQStages;
  uint64_t* afull = empty + kQStages;     // dequantised weight tile written
  uint64_t* acc_full = afull + kQStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;     // [2]
  uint64_t* drain = acc_empty + 2;
  uint64_t* raw_full = drain + 1;         // [kQRaw] raw chunk landed
  uint64_t* raw_empty = raw_full + kQRaw;  // [kQRaw] raw chunk dequantised
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_empty + kQRaw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_ok = abort_flag + 1;
  uint8_t* raw = smem + S::kRawOff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mb_per_e = args.d / kBM;
  const int KB = args.f / kQKs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full[s], 1);  // producer (TMA bytes of h)
      mbar_init(&empty[s], 1);
      mbar_init(&afull[s], 4);  // the four warps of one dequantising group
    }
    for (int s = 0; s < kQRaw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kQEpiWarps);
    }
    mbar_init(drain, 32);  // one commit per lane of the MMA warp
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the routing tables and h of this forward are complete from here on
  pdl_launch_dependents();
  const int nunits = __ldg(args.touched + args.E) * mb_per_e;
  constexpr int kDeqWarp0 = 2 + kQEpiWarps;
  constexpr int kHelperWarp0 = kDeqWarp0 + kQDeqWarps;  // raw-chunk issuers: warps kHelperWarp0 ..
  constexpr int kProdWarp1 = kHelperWarp0 + kQIssuers;  // h issuers: warp 0, then kProdWarp1 ..
  static_assert(kProdWarp1 + kQIssuers - 1 == kQThreads / 32, "warp roles");
  const bool h_issuer = warp == 0 || warp >= kProdWarp1;
  const bool raw_issuer = warp >= kHelperWarp0 && warp < kProdWarp1;

  if (h_issuer) {
    // ------------------------------------------------------------ TMA producers (h tiles)
    if (lane == 0) {
      const int me = warp == 0 ? 0 : warp - kProdWarp1 + 1;  // takes the steps with step % kQIssuers == me
      QIter it{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched};
      int step = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (bool more = it.first_chunk(); more && ok; more = it.next()) {
        const int N = round16(it.nch);
        const CUtensorMap* tb = &bmaps.m[N / 16 - 1];  // one box of exactly N token rows
        const int prow = __ldg(args.pad_offsets + it.e) / args.rpp + it.t0;  // h row of the chunk's first token
        const uint32_t bytes = (uint32_t)(kQSub * N * 128);
        for (int kb = 0; kb < KB; ++kb, ++step) {
          if (step % kQIssuers != me) continue;
          const int stage = step % kQStages;
          const uint32_t phase = (uint32_t)(step / kQStages) & 1u;
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, args.budget_ns, abort_flag)) {
            report_timeout(args.status, kWhereProducerEmpty);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_3d(smem + stage * S::kStage, tb, &full[stage], 0, prow, kb * kQSub);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        }
      }
      if (*abort_flag) {
        // every stage copy this thread issued lands before the CTA exits
        for (int s = 0; s < kQStages; ++s)
          if ((issued_mask >> s) & 1u) {
            volatile int never = 0;
            mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, args.budget_ns, &never);
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each tcgen05 op.
    QIter it{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched};
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    int chunk = 0;
    bool ok = true;
    // B descriptor of stage slot 0; a slot adds stage * kStage (16-byte units).
    // A (the dequantised weight tile) is read from tensor memory.
    const uint32_t st0 = smem_u32(smem);
    const uint64_t bdesc0 = smem_desc(st0, 16, 1024, 2);
    static_assert(kQStages * S::kStage < (1 << 18), "descriptor address field");
    for (bool more = it.first_chunk(); more && ok; more = it.next(), ++chunk) {
      const int N = round16(it.nch);
      const int buf = chunk & 1;
      const uint32_t acc = tmem + (uint32_t)(buf * kQAcc1);
      const uint32_t idesc = idesc_f16(kBM, N);
      if (!warp_wait_bounded(&acc_empty[buf], ((acc_phase >> buf) & 1u) ^ 1u, args.budget_ns, abort_flag)) {
        if (lane == 0) {
          report_timeout(args.status, kWhereMmaAccEmpty);
          *abort_flag = 1;
        }
        break;
      }
      acc_phase ^= 1u << buf;
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!warp_wait_bounded(&full[stage], phase, args.budget_ns, abort_flag) ||
            !warp_wait_bounded(&afull[stage], phase, args.budget_ns, abort_flag)) {
          if (lane == 0) {
            report_timeout(args.status, kWhereMmaFull);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t soff = (uint64_t)(stage * (S::kStage >> 4));
        const uint32_t a0 = tmem + (uint32_t)(kQASlot0 + 32 * kQSub * stage);
#pragma unroll
        for (int u = 0; u < kQSub; ++u)  // sub-step u: the [N][128 B] h block at u * N * 128 bytes
#pragma unroll
          for (int j = 0; j < 4; ++j)  // K = 16 fp16 per instruction: 8 tensor-memory columns of A, 32 bytes of B
            if (elect_one_sync())
              mma_f16_tmem_a(acc, a0 + 32 * u + 8 * j, bdesc0 + soff + (uint64_t)(u * N * 8 + 2 * j), idesc,
                             (kb > 0 || u > 0 || j > 0) ? 1u : 0u);
        if (elect_one_sync()) tc_commit(&empty[stage]);
        __syncwarp();
        if (++stage == kQStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one_sync()) tc_commit(&acc_full[buf]);
      __syncwarp();
    }
    // every MMA issued lands before tensor memory is freed: each lane commits
    // (a commit tracks the committing lane's own MMAs) and the barrier takes 32
    tc_commit(drain);
    if (lane == 0) {
      volatile int never = 0;
      mbar_wait_bounded(drain, 0, args.budget_ns, &never);
    }
    __syncwarp();
  } else if (raw_issuer) {
    // ------------------------------------------------------------ raw Q2_K chunks, kQSub per bulk copy
    // The ring runs up to kQRaw steps ahead of the dequantisation, so that many
    // kilobytes of weights are in flight per SM.
    if (lane == 0) {
      const int me = warp - kHelperWarp0;  // takes the steps with step % kQIssuers == me
      QIter it{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched};
      int step = 0, last = -1;  // last: the latest step this thread issued
      bool ok = true;
      for (bool more = it.first_chunk(); more && ok; more = it.next()) {
        const uint8_t* src = args.q2k + (size_t)(it.e * mb_per_e + it.mb) * KB * S::kRawSlot;
        for (int kb = 0; kb < KB; ++kb, ++step) {
          if (step % kQIssuers != me) continue;
          const int slot = step % kQRaw;
          const uint32_t phase = (uint32_t)(step / kQRaw) & 1u;
          if (!mbar_wait_bounded(&raw_empty[slot], phase ^ 1u, args.budget_ns, abort_flag)) {
            report_timeout(args.status, kWhereProducerEmpty);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[slot], S::kRawSlot);
          bulk_load(raw + slot * S::kRawSlot, src + (size_t)kb * S::kRawSlot, S::kRawSlot, &raw_full[slot]);
          last = step;
        }
      }
      // every copy this thread issued lands before the CTA exits: the last one of each of its slots
      for (int sq = last; sq >= 0 && sq > last - kQRaw; sq -= kQIssuers) {
        volatile int no_abort = 0;
        mbar_wait_bounded(&raw_full[sq % kQRaw], (uint32_t)(sq / kQRaw) & 1u, args.budget_ns, &no_abort);
      }
    }
    __syncwarp();
  } else if (warp >= kDeqWarp0) {
    // ------------------------------------------------------------ Q2_K -> fp16 weight tile
    // Four warps, one per tensor-memory lane quarter (row r = 32 (warp % 4) +
    // lane), dequantise one 128-weight step (two Q2_K chunks); the kQDeqGroups
    // groups take alternate steps, so that one group's waits and stores overlap
    // another's arithmetic.
    const int r = (warp & 3) * 32 + lane;  // weight row of the 128-row tile
    const int grp = (warp - kDeqWarp0) >> 2;
    const uint32_t a_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)kQASlot0;
    QIter it{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched};
    bool ok = true;
    int step = 0;  // steps of this CTA over all its chunks
    for (bool more = it.first_chunk(); more && ok; more = it.next()) {
      for (int kb = 0; kb < KB; ++kb, ++step) {
        if (step % kQDeqGroups != grp) continue;
        const int stage = step % kQStages, rslot = step % kQRaw;
        const uint32_t phase = (uint32_t)(step / kQStages) & 1u, rphase = (uint32_t)(step / kQRaw) & 1u;
        // The A slot is free once the MMAs of the step this slot held before
        // are done (empty); the h tile (full) is not needed to dequantise.
        const bool got = warp_wait_bounded(&empty[stage], phase ^ 1u, args.budget_ns, abort_flag) &&
                         warp_wait_bounded(&raw_full[rslot], rphase, args.budget_ns, abort_flag);
        if (!got) {
          if (lane == 0) {
            report_timeout(args.status, kWhereMmaFull);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
#pragma unroll
        for (int u = 0; u < kQSub; ++u) {  // sub-step u: Q2_K chunk u of the slot, tensor-memory columns 32 u ..
          const uint8_t* ch = raw + rslot * S::kRawSlot + u * kQ2kChunk;
          const uint4 qv = *reinterpret_cast<const uint4*>(ch + 16 * r);
          const uint32_t scw = *reinterpret_cast<const uint32_t*>(ch + 2048 + 4 * r);
          const uint32_t ddw = *reinterpret_cast<const uint32_t*>(ch + 2560 + 4 * r);
          const float dd = __half2float(__ushort_as_half((unsigned short)(ddw & 0xFFFFu)));
          const float dm = __half2float(__ushort_as_half((unsigned short)(ddw >> 16)));
          const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
          uint32_t P[2][16];  // the row's 64 weights of the sub-step, two f16 per word
#pragma unroll
          for (int sb = 0; sb < 4; ++sb) {  // sub-block sb: weights 16 sb .. 16 sb + 15 of the sub-step
            const uint32_t scb = (scw >> (8 * sb)) & 0xFFu;
            const __half2 a2 = __float2half2_rn(dd * (float)(scb & 15u));
            const __half2 nb2 = __float2half2_rn(-dm * (float)(scb >> 4));
            // {w_2n, w_2n+1}: the repacked word holds w_2n at bit 2n and w_2n+1 at bit
            // 16 + 2n.  OR-ing the 2-bit field at mantissa bit 2m into the f16 pattern
            // of 2^(10 - 2m) gives exactly 2^(10 - 2m) + q, so one mask-and-or (and
            // one shift per word, for pairs 5..7) extracts a pair without shifting it.
            const uint32_t hi_word = words[sb] >> 10;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
              const int m = n < 5 ? n : n - 5;
              const uint32_t wq = n < 5 ? words[sb] : hi_word;
              const uint32_t mag = (uint32_t)(25 - 2 * m) << 10;  // f16 bits of 2^(10 - 2m)
              const uint32_t v = (wq & (0x00030003u << (2 * m))) | (mag | (mag << 16));
              const __half2 base = __float2half2_rn((float)(1 << (10 - 2 * m)));
              const __half2 q2 = __hsub2(*reinterpret_cast<const __half2*>(&v), base);
              const __half2 w2 = __hfma2(q2, a2, nb2);
              P[sb >> 1][8 * (sb & 1) + n] = *reinterpret_cast<const uint32_t*>(&w2);
            }
          }
          const uint32_t col = (uint32_t)(32 * (kQSub * stage + u));
          tmem_st_32x32b_x16(a_lane + col, P[0]);
          tmem_st_32x32b_x16(a_lane + col + 16, P[1]);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&afull[stage]);
          mbar_arrive(&raw_empty[rslot]);  // this warp's reads of the raw chunk are done
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue: weighted combine
    const int q = warp & 3;            // tensor-memory lane quarter this warp may access
    const int part = (warp - 2) >> 2;  // which half of the 16-column slices
    const int etid = threadIdx.x - 64;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    QIter it{(int)blockIdx.x, nunits, (int)gridDim.x, mb_per_e, 0, 0, 0, 0, 0, args.counts, args.touched};
    uint32_t acc_phase = 0;
    int chunk = 0;
    for (bool more = it.first_chunk(); more; more = it.next(), ++chunk) {
      const int N = round16(it.nch);
      const int prow = __ldg(args.pad_offsets + it.e) + it.t0 * args.rpp;  // padded row of the chunk's first token
      const int buf = chunk & 1;
      // Per-column token and routing weight, loaded while the MMAs run.  One
      // thread takes the accumulator wait and publishes the outcome, so all
      // epilogue warps leave the loop together (the named barrier needs every
      // one of them).
      named_bar_sync(1, 32 * kQEpiWarps);  // previous chunk's table no longer read
      for (int c = etid; c < it.nch; c += 32 * kQEpiWarps) {
        const int pr = __ldg(args.pad_pair + prow + c * args.rpp);
        col_tok[c] = pr / args.k;
        col_w[c] = __ldg(args.topk_w + pr);
      }
      if (etid == 0) {
        const bool ok = mbar_wait_bounded(&acc_full[buf], (acc_phase >> buf) & 1u, args.budget_ns, abort_flag);
        *epi_ok = ok ? 1 : 0;
        if (!ok) {
          report_timeout(args.status, kWhereEpiAccFull);
          *abort_flag = 1;
        }
      }
      named_bar_sync(1, 32 * kQEpiWarps);
      if (!*epi_ok) break;
      acc_phase ^= 1u << buf;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * kQAcc1) + lane_base;
      const int m = it.mb * kBM + q * 32 + lane;  // output feature
      for (int c0 = part * 16; c0 < N; c0 += 16 * (kQEpiWarps / 4)) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(acc + (uint32_t)c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int col = c0 + jj;
          if (col < it.nch)
            red_add_f32(args.out + (size_t)col_tok[col] * args.d + m, col_w[col] * __uint_as_float(r[jj]));
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

// --------------------------------------------------------------- diagnostics
// Copies the `split` activation rows of every routed pair p = t*k + j (token
// order) out of the expert-grouped padded buffers: codes[(p*split + q)][K] and
// scales[(p*split + q)][K/32] from padded row pad_inv[p] + q.  One block per
// output row.
__global__ void gather_act_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, int K, int r128,
                                  const int32_t* __restrict__ pad_inv, int split, uint8_t* __restrict__ codes,
                                  uint8_t* __restrict__ scales) {
  const int orow = blockIdx.x;
  const size_t src = (size_t)__ldg(pad_inv + orow / split) + (size_t)(orow % split);
  const uint4* s4 = reinterpret_cast<const uint4*>(q + src * K);
  uint4* d4 = reinterpret_cast<uint4*>(codes + (size_t)orow * K);
  for (int i = threadIdx.x; i < K / 16; i += blockDim.x) d4[i] = s4[i];
  for (int b = threadIdx.x; b < K / 32; b += blockDim.x) scales[(size_t)orow * (K / 32) + b] = sf[act_sf_index(src, b, r128)];
}

}  // namespace

cudaError_t launch_gather_act(const ds4moe_layer* L, int which, int T, int split, uint8_t* codes, uint8_t* scales,
                              cudaStream_t st) {
  const int K = which == 0 ? L->cfg.d_model : L->cfg.d_ff;
  const uint8_t* q = which == 0 ? L->s.xq : L->s.hq;
  const uint8_t* sf = which == 0 ? L->s.xsf : L->s.hsf;
  const int rows = T * L->cfg.top_k * split;
  gather_act_kernel<<<rows, 128, 0, st>>>(q, sf, K, (int)(L->s.pad_rows_max / 128), L->s.pad_inv, split, codes,
                                          scales);
  return cudaGetLastError();
}

cudaError_t launch_act_quant(const ds4moe_layer* L, const void* x, float* out, int T, int split, cudaStream_t st) {
  const int parts = (L->cfg.d_model / 32 + 31) / 32;  // warps per token
  const int blocks = (T * parts + 7) / 8;
  return launch_pdl(act_quant_kernel, blocks, 256, 0, st, static_cast<const __nv_bfloat16*>(x), T, L->cfg.d_model,
                    L->cfg.top_k, L->s.pad_inv, L->s.xq, L->s.xsf, (int)(L->s.pad_rows_max / 128), split, out);
}

cudaError_t launch_gemm_down_q2k(const ds4moe_layer* L, float* out, int T, int rpp, cudaStream_t st) {
  (void)T;
  static InitOnce attr_once;
  cudaError_t e = init_once(attr_once, [] {
    return cudaFuncSetAttribute((const void*)q2k_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                QSmem::kTotal);
  });
  if (e != cudaSuccess) return e;
  BoxMaps maps;
  for (int i = 0; i < kNumBoxMaps; ++i) maps.m[i] = L->tm_h16[i];
  Q2kArgs a{};
  a.q2k = L->w.q2k;
  a.counts = L->s.counts;
  a.touched = L->s.touched;
  a.pad_offsets = L->s.pad_offsets;
  a.pad_pair = L->s.pad_pair;
  a.topk_w = L->s.topk_w;
  a.E = L->cfg.n_experts;
  a.k = L->cfg.top_k;
  a.d = L->cfg.d_model;
  a.f = L->cfg.d_ff;
  a.rpp = rpp;
  a.out = out;
  a.status = L->status;
  a.budget_ns = (uint64_t)L->cfg.wait_timeout_ms * 1000000ull;
  const int units = a.E * (a.d / kBM);
  const int grid = units < L->num_sms ? units : L->num_sms;
  return launch_pdl(q2k_down_kernel, grid, kQThreads, QSmem::kTotal, st, maps, a);
}


}  // namespace ds4moe
