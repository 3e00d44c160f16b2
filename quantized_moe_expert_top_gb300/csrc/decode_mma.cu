// Few-token (T <= 64) grouped GEMMs of the routed experts on the tensor cores:
// gate/up with split-K partial sums and a SwiGLU + MXFP8 step run by the last
// CTA to finish a tile, and down with the weighted combine back into token
// order.
//
// "284B MoEを128GBノートPCに詰め込む" §プリフィル790 t/sが暴く真のボトルネック: generation
// is memory-bandwidth bound, so at a handful of tokens this path is a stream of
// the touched experts' MXFP4 weights through every SM.  Each CTA (one per SM,
// persistent, cta_group::1) owns its tensor core and issues
// tcgen05.mma.kind::mxf8f6f4.block_scale with the E2M1 weight tile as A
// (M = 128 rows, unpacked by TMA) and the tokens' activation rows as B.  As on
// the pair GEMMs of the prefill path, every activation value is sent as two
// MXFP8 rows, hi = MXFP8(v) and lo = MXFP8(v - hi), and the epilogue adds the
// two columns: activations keep about bf16 precision while the weights stay
// 4-bit.  With at most 64 tokens an expert has at most 128 such rows, so an
// MMA is at most N = 128 wide and costs the same as one of N = 16.
//
// Work items are (touched expert, 128-row weight tile, 128-row token chunk,
// K slice).  The number of K slices S (1, 2, 4 or 8) is chosen on the device
// from the number of tiles, only where it evens out the items per SM by a
// quarter or more (at one token the 256 gate/up tiles of 8 experts run
// unsplit: forced splits of 2, 4 and 8 measured slower).  A pipeline stage
// holds two K = 128 blocks (3-D TMA boxes, one load per operand), so the MMA
// warp waits once per eight MMAs; it runs its loop warp-uniformly and one
// elected lane issues each tcgen05 instruction.
//
//   gate/up : a tile is the 64 gate rows and the 64 up rows of 64 features
//             (the tile-major layout of the layer).  The epilogue adds its
//             partial g and u into an fp32 buffer in HBM/L2 (red.add); the CTA
//             that completes a tile's last K slice (a per-tile counter) forms
//             h = silu(g) * u, writes its hi and lo MXFP8 rows for the down
//             GEMM, and clears the buffer and the counter for the next call.
//   down    : a tile is 128 output rows; the epilogue multiplies by the routing
//             weight and red-adds into out[t] (zeroed by the routing kernel);
//             K slices simply add.
//
// Warp roles per CTA: warp 0 issues the TMA loads, warp 1 allocates tensor
// memory and issues the MMAs, warps 2..5 drain the double-buffered
// accumulator (one tensor-memory lane quarter each).  Every mbarrier wait is
// bounded; a wait that runs out records DS4MOE_ERR_DEVICE_TIMEOUT and the CTA
// winds down after its in-flight copies and MMAs have landed.
#include "gemm.cuh"

namespace ds4moe {
namespace {

enum class DMode { GateUp, Down };

constexpr int kDThreads = 192;
constexpr int kDEpiWarps = 4;
constexpr int kDMaxStages = 8;
constexpr int kDNMax = 128;       // token rows per chunk (hi + lo rows of <= 64 tokens)
constexpr int kDAcc1 = 128;       // tensor-memory column of the second accumulator buffer
constexpr int kDSfBase = 256;     // scale-factor slots: SFA 4 + SFB 4 columns each
constexpr int kDSfSlot = 8;
constexpr int kDSfSlots = 2 * kDMaxStages + 2;  // one per K = 128 block, reused 9 stages later
static_assert(kDSfBase + kDSfSlots * kDSfSlot <= 512, "tensor memory");
constexpr int kDGroup = 4;        // K = 128 blocks whose scales one pair of TMA loads brings
constexpr int kDAStage = 2 * 128 * 128;  // two K = 128 blocks of 128 unpacked E2M1 rows
constexpr int kDSfGroupBytes = 2 * kDGroup * kSfChunk;  // SFA 4 chunks | SFB 4 chunks
constexpr int kDBarBytes = 256;    // barriers and flags
constexpr int kDMiscBytes = 4096;  // epilogue exchange and column tables

struct DMaps {
  CUtensorMap a;      // weights, 3-D {128 K, rows, K/128}, box 128 x 128 rows x 2 blocks
  CUtensorMap sfa;    // weight scale chunks, 4 consecutive K blocks per box
  CUtensorMap sfb;    // activation scale chunks, 1 row block x 4 K blocks per box
  CUtensorMap b[8];   // activations, 3-D {128 K, rows, K/128}, boxes of 16, 32, ..., 128 rows x 2 blocks
};

struct DArgs {
  const int32_t* counts;
  const int32_t* touched;      // [E] touched experts, [E] = their count
  const int32_t* offsets;      // pair position of each expert's first token
  const int32_t* pad_offsets;  // padded activation row of each expert's first token
  const int32_t* pad_pair;
  const float* topk_w;
  int E, k, d, f;
  int KB;        // K = 128 blocks of the contraction
  int tiles;     // 128-row weight tiles per expert
  int nbmax;     // token rows of a B stage slot (multiple of 16, <= 128)
  int nstages;
  int stage_bytes;
  int r128;      // 128-row blocks of the activation buffers
  float* gu_acc;     // gate/up: [pairs][2f] partial g | u sums, zero between calls
  int32_t* tile_cnt; // gate/up: K slices done per (touched expert, tile, chunk)
  int maxch;         // token chunks per expert the counters are sized for
  uint8_t* hq;       // gate/up: MXFP8 h rows (hi, lo) in padded expert order
  uint8_t* hsf;
  __half* h16;       // gate/up with a Q2_K down projection: fp16 h, row pad_offsets[e] / 2 + token (else null)
  float* out;        // down: [T][d]
  DeviceStatus* status;
  uint64_t budget_ns;
};

// Number of K slices: the smallest S in {1, 2, 4, 8} (S | KB, >= 2 blocks
// per slice) whose rounds of items over the grid, in full-K units, are at
// least 25 % fewer than the best smaller choice.  A split costs a cross-CTA
// reduction per item (partial sums through L2, a fence and a counter), which
// takes about as long as a few pipeline stages, so only a large imbalance
// pays for it.
__device__ __forceinline__ int choose_split(int items1, int G, int KB) {
  int best = 1;
  float best_t = (float)((items1 + G - 1) / G);
  for (int s = 2; s <= 8; s *= 2) {
    if (KB % s != 0 || KB / s < 2) break;
    const float t = (float)((items1 * s + G - 1) / G) / (float)s;
    if (t < 0.75f * best_t) {
      best = s;
      best_t = t;
    }
  }
  return best;
}

// The work sequence every role of a CTA walks: items i = blockIdx.x,
// blockIdx.x + G, ... of the concatenation over touched experts of
// (tile, chunk, K slice), K slice fastest.
struct DIter {
  const int32_t* counts;
  const int32_t* touched;
  int U, tiles, S, KB, G;
  int i, ui, base, per_u, e, nrows_e, nch;
  int tile, chunk, ks, kb0, kb1, rows;
  __device__ void load_u() {
    e = __ldg(touched + ui);
    nrows_e = 2 * __ldg(counts + e);
    nch = (nrows_e + kDNMax - 1) / kDNMax;
    per_u = nch * tiles * S;
  }
  __device__ bool seek() {
    while (ui < U) {
      if (i < base + per_u) {
        int r = i - base;
        ks = r % S;
        r /= S;
        chunk = r % nch;
        tile = r / nch;
        kb0 = ks * (KB / S);
        kb1 = kb0 + KB / S;
        rows = min(kDNMax, nrows_e - chunk * kDNMax);
        return true;
      }
      base += per_u;
      if (++ui < U) load_u();
    }
    return false;
  }
  __device__ bool first() {
    i = (int)blockIdx.x;
    ui = 0;
    base = 0;
    per_u = 0;
    if (U > 0) load_u();
    return seek();
  }
  __device__ bool next() {
    i += G;
    return seek();
  }
};

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.f + __expf(-g)); }

template <DMode M>
__global__ void __launch_bounds__(kDThreads, 1) decode_mma_kernel(const __grid_constant__ DMaps maps,
                                                                  const DArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nst = args.nstages;
  const int sf_off = nst * args.stage_bytes;
  const int ring = nst + 1;  // scale groups in shared memory
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sf_off + ring * kDSfGroupBytes);
  uint64_t* empty = full + kDMaxStages;
  uint64_t* acc_full = empty + kDMaxStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* epi_ok = abort_flag + 1;    // the epilogue's accumulator wait succeeded
  volatile int* epi_last = abort_flag + 2;  // this CTA completed the tile's last K slice
  int* s_split = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_units = s_split + 1;
  uint8_t* misc = reinterpret_cast<uint8_t*>(full) + kDBarBytes;   // kDMiscBytes
  float* xg = reinterpret_cast<float*>(misc);                       // gate/up: silu(g) [8 tokens][64 features]
  int32_t* col_tok = reinterpret_cast<int32_t*>(misc + 2048);       // down: token of each column pair
  float* col_w = reinterpret_cast<float*>(misc + 2048 + 4 * (kDNMax / 2));  // down: its routing weight

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kDEpiWarps);
    }
    mbar_init(drain, 32);  // one commit per lane of the MMA warp
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.sfa);
    prefetch_tmap(&maps.sfb);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  // The gate/up GEMM reads routing tables written by the kernel right before it,
  // so it plans after the dependency wait.  The down GEMM follows the gate/up
  // GEMM, which starts only after routing has completed: its routing tables
  // are complete already, so it plans and prefetches its first weight tiles
  // into L2 while the gate/up GEMM finishes, and waits only before it reads h.
  auto plan = [&]() {
    if (threadIdx.x == 0) {
      const int U = __ldg(args.touched + args.E);
      const int nch_total = __ldg(args.pad_offsets + args.E) / kDNMax;  // sum over experts of their chunks
      *s_units = U;
      *s_split = choose_split(nch_total * args.tiles, (int)gridDim.x, args.KB);
    }
  };
  if (M == DMode::GateUp) pdl_wait();
  plan();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int U = *s_units, S = *s_split;
  auto make_iter = [&]() {
    DIter it{};
    it.counts = args.counts;
    it.touched = args.touched;
    it.U = U;
    it.tiles = args.tiles;
    it.S = S;
    it.KB = args.KB;
    it.G = (int)gridDim.x;
    return it;
  };
  uint8_t* sf_base = smem + sf_off;
  if (M == DMode::Down && !(warp == 0 && lane == 0)) pdl_wait();  // the producer waits after its prefetches
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      DIter it = make_iter();
      if (M == DMode::Down) {
        // Prefetch the first weight tiles into L2 while the gate/up GEMM finishes.
        DIter pf = make_iter();
        int n = 0;
        for (bool more = pf.first(); more && n < 4; more = pf.next(), ++n)
          for (int kb = pf.kb0; kb < pf.kb1; kb += 2)
            tma_prefetch_3d(&maps.a, 0, (pf.e * args.tiles + pf.tile) * 128, kb);
        pdl_wait();
      }
      int st = 0, gcount = 0;
      uint32_t ph = 0, issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (bool more = it.first(); more && ok; more = it.next()) {
        const int arow = (it.e * args.tiles + it.tile) * 128;
        const int brow = __ldg(args.pad_offsets + it.e) + it.chunk * kDNMax;
        const int nbx = round16(it.rows);
        const CUtensorMap* bm = &maps.b[nbx / 16 - 1];
        for (int kb = it.kb0; kb < it.kb1; kb += 2) {
          if (!mbar_wait_bounded(&empty[st], ph ^ 1u, args.budget_ns, abort_flag)) {
            report_timeout(args.status, kWhereProducerEmpty);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const bool grp = ((kb - it.kb0) & (kDGroup - 1)) == 0;
          // 4-bit unpacking loads count their packed global bytes
          const uint32_t bytes = 128u * 64u * 2u + (uint32_t)nbx * 256u + (grp ? (uint32_t)kDSfGroupBytes : 0u);
          mbar_arrive_expect_tx(&full[st], bytes);
          uint8_t* sa = smem + st * args.stage_bytes;
          tma_load_3d(sa, &maps.a, &full[st], 0, arow, kb);
          tma_load_3d(sa + kDAStage, bm, &full[st], 0, brow, kb);
          if (grp) {
            uint8_t* sf = sf_base + gcount * kDSfGroupBytes;
            gcount = gcount + 1 == ring ? 0 : gcount + 1;
            tma_load_2d(sf, &maps.sfa, &full[st], 0, ((it.e * args.tiles + it.tile) * args.KB + kb) * 2);
            tma_load_3d(sf + kDGroup * kSfChunk, &maps.sfb, &full[st], 0, (brow / 128) * 2, kb);
          }
          issued_mask |= 1u << st;
          issued_parity = (issued_parity & ~(1u << st)) | (ph << st);
          if (++st == nst) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      // the last issued load of every slot lands before the CTA exits
      for (int s = 0; s < nst; ++s)
        if ((issued_mask >> s) & 1u) {
          volatile int no_abort = 0;
          mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, args.budget_ns, &no_abort);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (warp-uniform operands); one elected lane
    // issues each tcgen05 op.
    {
      DIter it = make_iter();
      int st = 0, gcount = 0, chunk_no = 0;
      uint32_t ph = 0, acc_phase = 0, sf_seq = 0;
      bool ok = true;
      constexpr uint32_t kSfIdStep = (1u << 4) | (1u << 29);  // next byte of the 32-bit scale word, A and B
      const uint32_t s0 = smem_u32(smem);
      const uint32_t sf0 = smem_u32(sf_base);
      for (bool more = it.first(); more && ok; more = it.next(), ++chunk_no) {
        const int nbx = round16(it.rows);
        const int buf = chunk_no & 1;
        const uint32_t acc = tmem + (uint32_t)(buf * kDAcc1);
        const uint32_t idesc0 = idesc_mx(128, nbx, 0);
        if (!warp_wait_bounded(&acc_empty[buf], ((acc_phase >> buf) & 1u) ^ 1u, args.budget_ns, abort_flag)) {
          if (lane == 0) {
            report_timeout(args.status, kWhereMmaAccEmpty);
            *abort_flag = 1;
          }
          break;
        }
        acc_phase ^= 1u << buf;
        tc_fence_after();
        int gslot = 0, gkb0 = it.kb0;
        for (int kb = it.kb0; kb < it.kb1; kb += 2) {
          if (!warp_wait_bounded(&full[st], ph, args.budget_ns, abort_flag)) {
            if (lane == 0) {
              report_timeout(args.status, kWhereMmaFull);
              *abort_flag = 1;
            }
            ok = false;
            break;
          }
          tc_fence_after();
          if (((kb - it.kb0) & (kDGroup - 1)) == 0) {
            gslot = gcount;
            gcount = gcount + 1 == ring ? 0 : gcount + 1;
            gkb0 = kb;
          }
          // No memory access from here to the commit: a load in this thread
          // would wait for the queued MMAs to drain, so the slots are scalars
          // and the two K = 128 blocks are unrolled.
          const bool two = kb + 1 < it.kb1;
          const uint32_t sa = s0 + (uint32_t)(st * args.stage_bytes);
          const uint32_t sfg = sf0 + (uint32_t)(gslot * kDSfGroupBytes);
          const int j0 = kb - gkb0;  // chunk of the scale group
          const uint32_t slot0 = tmem + kDSfBase + sf_seq * kDSfSlot;
          sf_seq = sf_seq + 1 == kDSfSlots ? 0 : sf_seq + 1;
          const uint32_t slot1 = tmem + kDSfBase + sf_seq * kDSfSlot;
          if (two) sf_seq = sf_seq + 1 == kDSfSlots ? 0 : sf_seq + 1;
          if (elect_one_sync()) {
            tc_cp_32x128b_warpx4(slot0, smem_desc(sfg + (uint32_t)(j0 * kSfChunk), 0, 128, 0));
            tc_cp_32x128b_warpx4(slot0 + 4, smem_desc(sfg + (uint32_t)((kDGroup + j0) * kSfChunk), 0, 128, 0));
            if (two) {
              tc_cp_32x128b_warpx4(slot1, smem_desc(sfg + (uint32_t)((j0 + 1) * kSfChunk), 0, 128, 0));
              tc_cp_32x128b_warpx4(slot1 + 4, smem_desc(sfg + (uint32_t)((kDGroup + j0 + 1) * kSfChunk), 0, 128, 0));
            }
          }
          const uint64_t ad0 = smem_desc(sa, 16, 1024, 2);
          const uint64_t bd0 = smem_desc(sa + (uint32_t)kDAStage, 16, 1024, 2);
          const uint64_t ad1 = ad0 + (uint64_t)((128 * 128) >> 4);
          const uint64_t bd1 = bd0 + (uint64_t)((nbx * 128) >> 4);
          const uint32_t first = kb > it.kb0 ? 1u : 0u;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)  // K = 32 (32 bytes) per instruction
            if (elect_one_sync())
              mma_mxf8f6f4(acc, ad0 + 2 * jj, bd0 + 2 * jj, idesc0 + (uint32_t)jj * kSfIdStep, slot0, slot0 + 4,
                           jj > 0 ? 1u : first);
          if (two) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              if (elect_one_sync())
                mma_mxf8f6f4(acc, ad1 + 2 * jj, bd1 + 2 * jj, idesc0 + (uint32_t)jj * kSfIdStep, slot1, slot1 + 4,
                             1u);
          }
          if (elect_one_sync()) tc_commit(&empty[st]);
          __syncwarp();
          if (++st == nst) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one_sync()) tc_commit(&acc_full[buf]);
        __syncwarp();
      }
      // every MMA issued lands before tensor memory is freed: each lane
      // commits (a commit tracks the committing lane's own MMAs), the barrier
      // takes 32
      tc_commit(drain);
      if (lane == 0) {
        volatile int no_abort = 0;
        mbar_wait_bounded(drain, 0, args.budget_ns, &no_abort);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // tensor-memory lane quarter this warp may access
    const int etid = threadIdx.x - 64;
    const int ew = warp - 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    DIter it = make_iter();
    uint32_t acc_phase = 0;
    int chunk_no = 0;
    const int twof = 2 * args.f;
    for (bool more = it.first(); more; more = it.next(), ++chunk_no) {
      const int buf = chunk_no & 1;
      const int nbx = round16(it.rows);
      const int ntok = it.rows / 2;
      // One thread takes the accumulator wait and publishes the outcome, so all
      // epilogue warps leave the loop together; the first barrier keeps that
      // outcome and the column table from being overwritten while a warp still
      // reads the last ones.
      named_bar_sync(1, 32 * kDEpiWarps);
      if constexpr (M == DMode::Down) {
        // token and routing weight of each column pair, read while the MMAs run
        const int prow = __ldg(args.pad_offsets + it.e) + it.chunk * kDNMax;
        for (int t = etid; t < ntok; t += 32 * kDEpiWarps) {
          const int pair = __ldg(args.pad_pair + prow + 2 * t);
          col_tok[t] = pair / args.k;
          col_w[t] = __ldg(args.topk_w + pair);
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
      named_bar_sync(1, 32 * kDEpiWarps);
      if (!*epi_ok) break;
      acc_phase ^= 1u << buf;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * kDAcc1) + lane_base;
      const int r = q * 32 + lane;  // tile row of this thread
      const int tok0 = it.chunk * (kDNMax / 2);
      const int prow0 = __ldg(args.pad_offsets + it.e) + it.chunk * kDNMax;
      if constexpr (M == DMode::Down) {
        float* dst = args.out + it.tile * 128 + r;
        for (int c0 = 0; c0 < nbx; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(acc + (uint32_t)c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int t = c0 / 2 + jj;
            if (t < ntok)
              red_add_f32(dst + (size_t)col_tok[t] * args.d,
                          col_w[t] * (__uint_as_float(v[2 * jj]) + __uint_as_float(v[2 * jj + 1])));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);  // the accumulator is free for the item after next
      } else if (S == 1) {
        // The whole K is in this accumulator: h straight from tensor memory.
        // Rows 0..63 are gate rows (quarters 0, 1), 64..127 the up rows of the
        // same features (quarters 2, 3); the gate warps stage silu(g) for 8
        // tokens at a time and the up warps form h = silu(g) * u and write its
        // hi and lo MXFP8 rows (a 32-feature block is one warp's lanes).
        const bool gate = q < 2;
        const int fq = q & 1;                       // 32-feature block of the tile
        const int i = it.tile * 64 + fq * 32 + lane;  // feature
        for (int c0 = 0; c0 < nbx; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(acc + (uint32_t)c0, v);
          tmem_ld_wait();
          float val[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) val[jj] = __uint_as_float(v[2 * jj]) + __uint_as_float(v[2 * jj + 1]);
          if (gate) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) xg[jj * 64 + fq * 32 + lane] = silu_f(val[jj]);
          }
          named_bar_sync(2, 32 * kDEpiWarps);  // silu(g) of the slice staged
          if (!gate && args.h16 != nullptr) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int t = c0 / 2 + jj;
              if (t < ntok)
                args.h16[(size_t)(prow0 / 2 + t) * args.f + i] = __float2half_rn(xg[jj * 64 + fq * 32 + lane] * val[jj]);
            }
          } else if (!gate) {
            float h[8];
            uint32_t am[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              h[jj] = xg[jj * 64 + fq * 32 + lane] * val[jj];
              am[jj] = __float_as_uint(fabsf(h[jj]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) am[jj] = max(am[jj], __shfl_xor_sync(0xffffffffu, am[jj], o));
            int sx[8];
            float res[8];
            uint32_t chi[8], am2[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              sx[jj] = mxfp8_exponent(__uint_as_float(am[jj]));
              chi[jj] = f32x2_to_e4m3x2(h[jj] * exp2i(-sx[jj]), 0.f) & 0xFFu;
              res[jj] = h[jj] - e4m3x2_to_f32x2(chi[jj]).x * exp2i_e8m0(sx[jj]);
              am2[jj] = __float_as_uint(fabsf(res[jj]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) am2[jj] = max(am2[jj], __shfl_xor_sync(0xffffffffu, am2[jj], o));
            uint32_t sf_mine = 0;  // lane 2j: scale of token j's hi row, lane 2j + 1: of its lo row
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int s2 = mxfp8_exponent(__uint_as_float(am2[jj]));
              const uint32_t clo = f32x2_to_e4m3x2(res[jj] * exp2i(-s2), 0.f) & 0xFFu;
              if (lane == 2 * jj) sf_mine = (uint32_t)(sx[jj] + 127);
              if (lane == 2 * jj + 1) sf_mine = (uint32_t)(s2 + 127);
              const int t = c0 / 2 + jj;
              if (t < ntok) {
                const size_t row = (size_t)(prow0 + 2 * t);
                args.hq[row * args.f + i] = (uint8_t)chi[jj];
                args.hq[(row + 1) * args.f + i] = (uint8_t)clo;
              }
            }
            if (lane < 16 && c0 + lane < it.rows)
              args.hsf[act_sf_index((size_t)(prow0 + c0 + lane), i / 32, args.r128)] = (uint8_t)sf_mine;
          }
          named_bar_sync(2, 32 * kDEpiWarps);  // staging free for the next slice
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      } else {
        // K is split over S CTAs: add this slice's g and u into the fp32
        // buffer; the CTA that completes the tile's last slice forms h.
        float* dst = args.gu_acc + (size_t)(__ldg(args.offsets + it.e) + tok0) * twof + it.tile * 128 + r;
        for (int c0 = 0; c0 < nbx; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(acc + (uint32_t)c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int t = c0 / 2 + jj;
            if (t < ntok) red_add_f32(dst + (size_t)t * twof, __uint_as_float(v[2 * jj]) + __uint_as_float(v[2 * jj + 1]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);  // the accumulator is free for the item after next
        __threadfence();  // this CTA's partial sums are visible before its count
        named_bar_sync(1, 32 * kDEpiWarps);
        int32_t* cnt = args.tile_cnt + ((size_t)it.ui * args.tiles + it.tile) * args.maxch + it.chunk;
        if (etid == 0) *epi_last = (atomicAdd(cnt, 1) == S - 1) ? 1 : 0;
        named_bar_sync(1, 32 * kDEpiWarps);
        if (*epi_last) {
          __threadfence();  // the other K slices' sums are visible from here on
          const int blk = ew & 1;  // 32-feature block of the tile's 64 features
          const int i = it.tile * 64 + blk * 32 + lane;  // feature
          const int pos0 = __ldg(args.offsets + it.e) + tok0;
          for (int t0 = ew >> 1; t0 < ntok; t0 += 8) {
            // four tokens (t0, t0 + 2, ...) per round: their loads are in flight together
            float g[4], u[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const int t = t0 + 2 * b;
              float* src = args.gu_acc + (size_t)(pos0 + t) * twof + it.tile * 128 + blk * 32 + lane;
              g[b] = t < ntok ? __ldcg(src) : 0.f;
              u[b] = t < ntok ? __ldcg(src + 64) : 0.f;
            }
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const int t = t0 + 2 * b;
              if (t >= ntok) break;  // uniform over the warp
              float* src = args.gu_acc + (size_t)(pos0 + t) * twof + it.tile * 128 + blk * 32 + lane;
              __stcg(src, 0.f);
              __stcg(src + 64, 0.f);
              const float h = silu_f(g[b]) * u[b];
              if (args.h16 != nullptr) {
                args.h16[(size_t)(prow0 / 2 + t) * args.f + i] = __float2half_rn(h);
                continue;
              }
              // hi = MXFP8(h), lo = MXFP8(h - hi) over the warp's 32 features
              const int sh = mxfp8_exponent(warp_max(fabsf(h)));
              const uint32_t chi = f32x2_to_e4m3x2(h * exp2i(-sh), 0.f) & 0xFFu;
              const float res = h - e4m3x2_to_f32x2(chi).x * exp2i_e8m0(sh);
              const int s2 = mxfp8_exponent(warp_max(fabsf(res)));
              const uint32_t clo = f32x2_to_e4m3x2(res * exp2i(-s2), 0.f) & 0xFFu;
              const size_t prow = (size_t)(prow0 + 2 * t);
              args.hq[prow * args.f + i] = (uint8_t)chi;
              args.hq[(prow + 1) * args.f + i] = (uint8_t)clo;
              if (lane == 0) {
                args.hsf[act_sf_index(prow, i / 32, args.r128)] = (uint8_t)(sh + 127);
                args.hsf[act_sf_index(prow + 1, i / 32, args.r128)] = (uint8_t)(s2 + 127);
              }
            }
          }
          if (etid == 0) *cnt = 0;  // ready for the next call
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <DMode M>
cudaError_t launch_dec(const ds4moe_layer* L, const DMaps& maps, const DArgs& a0, int T, cudaStream_t st) {
  DArgs a = a0;
  a.nbmax = min(kDNMax, (2 * T + 15) / 16 * 16);
  a.stage_bytes = kDAStage + a.nbmax * 256;
  constexpr int kSmemMax = 227 * 1024;
  constexpr int kFixed = 1024 + kDBarBytes + kDMiscBytes;  // alignment slack, barriers, epilogue tables
  a.nstages = min(kDMaxStages, (kSmemMax - kFixed - kDSfGroupBytes) / (a.stage_bytes + kDSfGroupBytes));
  const int smem = kFixed + a.nstages * a.stage_bytes + (a.nstages + 1) * kDSfGroupBytes;
  static InitOnce attr_once;
  cudaError_t e = init_once(attr_once, [] {
    return cudaFuncSetAttribute((const void*)decode_mma_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemMax);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_mma_kernel<M>, dim3((unsigned)L->num_sms), dim3(kDThreads), (size_t)smem, st, maps, a);
}

DArgs dec_args(const ds4moe_layer* L) {
  DArgs a{};
  a.counts = L->s.counts;
  a.touched = L->s.touched;
  a.offsets = L->s.offsets;
  a.pad_offsets = L->s.pad_offsets;
  a.pad_pair = L->s.pad_pair;
  a.topk_w = L->s.topk_w;
  a.E = L->cfg.n_experts;
  a.k = L->cfg.top_k;
  a.d = L->cfg.d_model;
  a.f = L->cfg.d_ff;
  a.r128 = (int)(L->s.pad_rows_max / 128);
  a.status = L->status;
  a.budget_ns = (uint64_t)L->cfg.wait_timeout_ms * 1000000ull;
  return a;
}

}  // namespace

cudaError_t launch_decmma_gateup(const ds4moe_layer* L, int T, cudaStream_t st) {
  DMaps m;
  m.a = L->tm_gu3;
  m.sfa = L->tm_sfa_gu;
  m.sfb = L->tm_sfb_x1;
  for (int i = 0; i < 8; ++i) m.b[i] = L->tm_xq3[i];
  DArgs a = dec_args(L);
  a.KB = L->cfg.d_model / 128;
  a.tiles = L->cfg.d_ff / 64;
  a.gu_acc = L->s.gu_acc;
  a.tile_cnt = L->s.tile_cnt;
  a.maxch = L->s.dec_maxch;
  a.hq = L->s.hq;
  a.hsf = L->s.hsf;
  a.h16 = L->cfg.down_format == DS4MOE_DOWN_Q2K ? L->s.h16 : nullptr;
  return launch_dec<DMode::GateUp>(L, m, a, T, st);
}

cudaError_t launch_decmma_down(const ds4moe_layer* L, float* out, int T, cudaStream_t st) {
  DMaps m;
  m.a = L->tm_dn3;
  m.sfa = L->tm_sfa_dn;
  m.sfb = L->tm_sfb_h1;
  for (int i = 0; i < 8; ++i) m.b[i] = L->tm_hq3[i];
  DArgs a = dec_args(L);
  a.KB = L->cfg.d_ff / 128;
  a.tiles = L->cfg.d_model / 128;
  a.out = out;
  return launch_dec<DMode::Down>(L, m, a, T, st);
}

}  // namespace ds4moe
