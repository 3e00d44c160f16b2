// Internal declarations of the ds4moe library: the layer object, the device
// buffers it owns, and the launchers of each kernel.  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/ds4moe.h"

namespace ds4moe {

struct DeviceStatus;

// Process-wide launch set-up (a kernel's dynamic shared-memory limit, the
// resident CTA-pair count) done once, safely when several host threads launch
// at the same time; a failed attempt is retried by the next call.
struct InitOnce {
  std::atomic<bool> done{false};
  std::mutex mu;
};
template <typename F>
inline cudaError_t init_once(InitOnce& o, F&& f) {
  if (o.done.load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(o.mu);
  if (o.done.load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = f();
  if (e == cudaSuccess) o.done.store(true, std::memory_order_release);
  return e;
}

// Launches `kernel` on `st` with programmatic stream serialisation, so that
// its blocks can be scheduled while the previous kernel in the stream drains
// (each kernel waits with griddepcontrol.wait before touching shared data).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Tile geometry of the prefill GEMMs.
constexpr int kBM = 128;          // rows of a weight tile (tcgen05 M)
constexpr int kBK = 128;          // contraction elements per pipeline stage
constexpr int kPadRows = 128;     // each expert's token rows start on a 128-row boundary
constexpr int kSfChunk = 512;     // bytes of one scale-factor chunk (128 rows x 4 blocks)
constexpr int kGateUpNMax = 224;  // token columns per gate/up tile (two accumulators in TMEM)
constexpr int kDownNMax = 256;    // token columns per down tile
constexpr int kQ2kChunk = 3072;   // bytes of one Q2_K tile-major chunk
constexpr int kNumBoxMaps = 12;   // token-tile TMA maps with 16, 32, ..., 192-row boxes
constexpr int kSmallRouteT = 4;  // largest T routed (and its activations quantised) by the single-block kernel

// Routing tables and scratch for one forward call (all device memory).
struct Scratch {
  int32_t* topk_idx;     // [Tmax*k]
  float* topk_w;         // [Tmax*k]
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E+1]
  int32_t* pad_offsets;  // [E+1] expert row starts in the 128-row padded order
  int32_t* perm_tok;     // [Tmax*k]
  int32_t* perm_slot;    // [Tmax*k]
  int32_t* inv;          // [Tmax*k]  position of pair (t, j) in (expert, token) order
  int32_t* pad_inv;      // [Tmax*k]  padded row of pair (t, j)
  int32_t* pad_pair;     // [pad_rows_max] pair index t*k+j of a padded row (-1: padding)
  int32_t* touched;      // [E+1] experts with at least one token, then their count at [E]
  __half* xh;            // [Tdec][d] decode-path x as prescaled f16 (piece-transposed rows)
  float* xsig;           // [Tdec] the prescale 2^s of each row of xh
  float* h_dec;          // [Tdec*k][f] decode-path SwiGLU output (fp32, piece-transposed rows)
  uint8_t* xq;           // [pad_rows_max][d]   MXFP8 codes of x, padded expert order
  uint8_t* xsf;          // [d/128][pad_rows_max/128][512] E8M0 scales (tcgen05 chunk layout)
  uint8_t* hq;           // [pad_rows_max][f]   MXFP8 codes of h (MXFP4 down)
  uint8_t* hsf;          // [f/128][pad_rows_max/128][512]
  __half* h16;           // [pad_rows_max][f]   fp16 h (Q2_K down); one row per routed pair, expert e's
                         //   first at pad_offsets[e] / (padded rows per pair)
  float* gu_acc;         // [Tdec*k][2f] DECODE_MMA gate/up partial sums (zero between calls)
  int32_t* tile_cnt;     // [E][f/64][dec_maxch] K slices done per gate/up tile and token chunk
  int dec_maxch;         // 128-row token chunks per expert at the DECODE_MMA token limit
  float* dense_c;        // [Tmax][dense_n] router logits | pad | shared g | shared u (fp32)
  __nv_bfloat16* h_shared;  // [Tmax][fs] shared-expert h (bf16)
  void* blas_ws;         // cuBLAS workspace
  uint8_t* stage_x;      // host-call staging: x [Tmax][d] bf16
  float* stage_logits;   // [Tmax][E]
  float* stage_out;      // [Tmax][d]
  int64_t pad_rows_max;
};

// Weights as the kernels read them (library-owned device copies).
//   gu: per (expert, 128-row block mb): the block's 128 gate rows, then its
//       128 up rows; each row = codes (d/2 B) | E8M0 scales (d/32 B) |
//       padding to pitch_gu (a multiple of 32 B).  The decode path streams
//       rows; one prefill TMA box of 256 rows loads a gate tile and its up tile.
//   dn: one row per (expert, m): codes (f/2 B) | scales (f/32 B) | padding.
struct Weights {
  uint8_t* gu;                       // [E][f/128][2][128][pitch_gu]
  uint8_t* dn;                       // [E][d][pitch_dn] (MXFP4 down)
  int pitch_gu, pitch_dn;
  uint8_t* gu_sf;                    // [E][f/128][d/128][gate 512 B | up 512 B] (prefill)
  uint8_t* down_sf;                  // [E][d/128][f/128][512]
  // Q2_K down, tile-major: one 3072-byte chunk per (expert, 128-row block,
  // 64-weight K step): 128 x 16 B 2-bit codes | 128 x 4 sub-block scale bytes
  // | 128 x (fp16 d | fp16 dmin << 16) of the super-block the step lies in.
  uint8_t* q2k;        // [E][d/128][f/64][3072]
};

}  // namespace ds4moe

struct ds4moe_layer {
  ds4moe_config cfg;
  int device;
  int num_sms;
  ds4moe::Weights w;
  ds4moe::Scratch s;
  ds4moe::DeviceStatus* status;  // device
  // TMA descriptors (64-byte aligned inside the struct)
  CUtensorMap tm_gu;     // 4-bit gate+up weights, box 128 x 128 rows (64 gate + 64 up)
  CUtensorMap tm_down;   // 4-bit down weights, box 128 x 128 rows
  CUtensorMap tm_sfa_gu;  // gate/up weight scale chunks, 4 consecutive K blocks per box
  CUtensorMap tm_sfa_dn;  // down weight scale chunks, same
  CUtensorMap tm_sfb_x;   // x scale chunks: 2 row blocks x 4 K blocks per box
  CUtensorMap tm_sfb_h;   // h scale chunks, same
  CUtensorMap tm_xq[ds4moe::kNumBoxMaps];   // 8-bit x, boxes 128 B x (16 * (i + 1)) rows
  CUtensorMap tm_hq[ds4moe::kNumBoxMaps];   // 8-bit h
  CUtensorMap tm_h16[ds4moe::kNumBoxMaps];  // fp16 h as {64, rows, f/64}, boxes {64, 16 * (i + 1), 2}
  // DECODE_MMA (one CTA per SM): 3-D views {128, rows, K/128} that load two
  // K = 128 blocks per box, and activation scale chunks of one row block
  CUtensorMap tm_gu3;     // gate/up weights, box 128 x 128 rows x 2
  CUtensorMap tm_dn3;     // down weights, same
  CUtensorMap tm_xq3[8];  // x rows, boxes 128 x (16 * (i + 1)) rows x 2
  CUtensorMap tm_hq3[8];  // h rows, same
  CUtensorMap tm_sfb_x1;  // x scale chunks: 1 row block x 4 K blocks per box
  CUtensorMap tm_sfb_h1;  // h scale chunks, same
  bool decmma_ready;      // the maps above are encoded
  void* blas;             // cuBLAS handle (router / shared expert), or null
  __nv_bfloat16* wcat;    // [dense_n][d] router rows | zero rows to a multiple of 4 | shared gate rows | shared up rows
  __nv_bfloat16* wsd;     // [d][fs] shared down
  int dense_n;            // rows of wcat (dense_goff + 2 fs)
  int dense_goff;         // column of the first shared gate output in dense_c (E rounded up to 4 with a shared expert)
  bool last_forward_x;    // the most recent forward computed its logits
  cudaEvent_t ev[12];  // kernel timing events (created when timing is enabled)
  bool timing;
  int last_nk;         // kernels in the most recent forward
  int last_T;
  int last_path;       // DS4MOE_PATH_* of the most recent forward
  int last_split;      // activation rows per routed pair in that forward (1 or 2)
  cudaStream_t last_stream;
  bool has_forward;
  bool prefill_ready;  // tensor maps encoded
  void* owned[48];     // every device allocation, freed by destroy
  int n_owned;
};

namespace ds4moe {

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error; none synchronises.
// `lds` = row stride of logits (E, or the dense_in output's width)
cudaError_t launch_route_topk(const ds4moe_layer* L, const float* logits, int lds, const void* x, bool prep_x, int T,
                              cudaStream_t st);
cudaError_t launch_route_group(const ds4moe_layer* L, int T, int rpp, cudaStream_t st);
// Few-token routing (T <= kSmallRouteT) in one launch, with the activation
// quantisation and the zeroing of out when `quant` is set.
cudaError_t launch_route_small(const ds4moe_layer* L, const float* logits, int lds, const void* x, float* out, int T,
                               int split, bool quant, cudaStream_t st);

cudaError_t launch_decode_gateup(const ds4moe_layer* L, const void* x, float* out, int T, cudaStream_t st);
cudaError_t launch_decode_down(const ds4moe_layer* L, float* out, int T, cudaStream_t st);

// split = 2: every routed pair has two activation rows, hi = MXFP8(v) and
// lo = MXFP8(v - hi); the GEMM epilogues add the two columns back together.
cudaError_t launch_act_quant(const ds4moe_layer* L, const void* x, float* out, int T, int split, cudaStream_t st);
cudaError_t launch_gemm_gateup(const ds4moe_layer* L, int T, int split, cudaStream_t st);
cudaError_t launch_gemm_down(const ds4moe_layer* L, float* out, int T, int split, cudaStream_t st);
// rpp = padded activation rows per routed pair of the routing that preceded
// (1 on the PREFILL path, 2 on DECODE_MMA); h16 holds one row per pair.
cudaError_t launch_gemm_down_q2k(const ds4moe_layer* L, float* out, int T, int rpp, cudaStream_t st);
// DECODE_MMA grouped GEMMs (one CTA per SM, split-K over the touched experts'
// weight tiles); the activation rows are split (hi, lo) as above.
cudaError_t launch_decmma_gateup(const ds4moe_layer* L, int T, cudaStream_t st);
cudaError_t launch_decmma_down(const ds4moe_layer* L, float* out, int T, cudaStream_t st);
// Diagnostics: the `split` MXFP8 rows of every routed pair (token order) of
// the x (which = 0) or h (which = 1) activations of the last forward.
cudaError_t launch_gather_act(const ds4moe_layer* L, int which, int T, int split, uint8_t* codes, uint8_t* scales,
                              cudaStream_t st);

// router projection and shared expert (dense.cu, cuBLAS + one kernel)
cudaError_t launch_dense_in(const ds4moe_layer* L, const void* x, int T, cudaStream_t st);
cudaError_t launch_shared_swiglu(const ds4moe_layer* L, int T, cudaStream_t st);
cudaError_t launch_shared_down(const ds4moe_layer* L, float* out, int T, cudaStream_t st);
cudaError_t dense_create(ds4moe_layer* L, size_t workspace_bytes, void* workspace);
void dense_destroy(ds4moe_layer* L);

// create-time repacking
cudaError_t launch_repack_sf(const uint8_t* scales, uint8_t* sf, int E, int rows, int K, int tile_rows, int row_off,
                             cudaStream_t st);
cudaError_t launch_pack_gu(const ds4moe_weights* w, ds4moe_layer* L, cudaStream_t st);
cudaError_t launch_repack_q2k(const uint8_t* blocks, ds4moe_layer* L, cudaStream_t st);
cudaError_t launch_pack_rows(uint8_t* dst, int pitch, int64_t rows, const uint8_t* s0, int l0, const uint8_t* s1,
                             int l1, const uint8_t* s2, int l2, const uint8_t* s3, int l3, cudaStream_t st);


}  // namespace ds4moe
