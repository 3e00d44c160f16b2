/*
 * ds4moe.h -- C ABI of the routed-MoE expert layer with 4-bit block-scaled
 * experts (GB300 / sm_103a).
 *
 * The operation.  One routed mixture-of-experts feed-forward layer of the
 * DwarfStar (ds4) engine, whose routed experts are stored in MXFP4 (gate, up
 * and down projections) or, in the engine's asymmetric 2-bit scheme, with a
 * Q2_K-style down projection ("DwarfStar実地分析: DeepSeek V4 Flashをローカルで
 * 動かす狭域推論エンジン", §GGUFの対応範囲は意図的に狭い: only the routed experts
 * are quantised, MXFP4 routed experts are used as published, Blackwell CUDA
 * runs batched expert work on FP4 matrix instructions; "DS4 分布式Shell客户端",
 * §模型下载: up/gate and down quantised asymmetrically, native MXFP4 experts).
 * The pages give no formula; this library computes, per call on T tokens:
 *
 *   1. route    idx[t, 0..k) = the k largest router logits of token t, sorted
 *               by (value desc, expert index asc); w[t, j] = softmax of those
 *               k logits only.
 *   2. group    the T*k (token, slot) pairs sorted by (expert, token).
 *   3. gate/up  g = W_gate[e] x_t, u = W_up[e] x_t for every routed (t, e).
 *   4. SwiGLU   h = g * sigmoid(g) * u.
 *   5. down     y = W_down[e] h.
 *   6. combine  out[t] = sum_j w[t, j] * y[t, j]   (fp32).
 *
 * Three execution paths compute it (chosen per call, see ds4moe_path_for):
 *   DECODE_MMA (AUTO for T <= decode_max_tokens): the grouped tcgen05 GEMMs
 *           below with split-precision activations: every x (and h) row is
 *           sent as two MXFP8 rows, hi = MXFP8(v) and lo = MXFP8(v - hi), and
 *           the epilogues add the two products, so activations keep about
 *           bf16 precision while the weights stay 4-bit.
 *   DECODE  (only when forced): memory-streaming GEMVs on the CUDA cores,
 *           weights dequantised in registers, activations at f16/fp32.
 *   PREFILL (AUTO for larger T): grouped block-scaled tcgen05 GEMMs; x and h
 *           are quantised to MXFP8 (E4M3 + one E8M0 scale per 32 values, OCP MX
 *           v1.0 conversion rule) inside the library; with a Q2_K down
 *           projection h is kept in fp16 instead.
 *
 * Formats (OCP Microscaling Formats v1.0).  MXFP4 weight: 32 E2M1 codes along
 * the contraction axis share one E8M0 scale byte (value 2^(b-127)); element
 * 2i is the LOW nibble of byte i.  Q2_K-style super-block (256 weights along
 * the contraction axis, 84 bytes): bytes 0..15 sub-block j scale byte (low
 * nibble sc_j, high nibble m_j), bytes 16..79 2-bit q (weight i at byte
 * 16 + i/4, bits 2*(i%4)), bytes 80..81 fp16 d, 82..83 fp16 dmin; weight =
 * d*sc_j*q - dmin*m_j, j = i/16.
 *
 * Conventions for every call:
 *   - Return value: DS4MOE_OK (0) or a negative DS4MOE_ERR_* code.  A call
 *     that returns INVALID_ARG, UNSUPPORTED or TOO_MANY_TOKENS has enqueued
 *     no GPU work (those checks run on the host first); after DS4MOE_ERR_CUDA
 *     (a launch or copy failed) the work enqueued before the failing step may
 *     still run, and the call's outputs are invalid.
 *   - "device pointer" = global memory of the layer's device; "host pointer"
 *     = CPU memory (pinned memory gives the fastest copies).
 *   - Every device pointer must be 16-byte aligned.
 *   - Calls on one layer must not overlap: a layer owns its scratch buffers,
 *     so use it from one stream at a time.
 *   - One GPU per process: the kernels' launch attributes (dynamic shared
 *     memory size) and the resident CTA-pair count are set up once per process,
 *     on the device of the first layer that runs them; layers on a second
 *     device in the same process are not supported.
 *   - Host threads: that one-time set-up is thread-safe, so different layers
 *     may be driven from different host threads at the same time; one layer
 *     is driven by one thread at a time (its last-call state is not locked). 
 *   - NaN or infinite logits or activations are outside the layer's domain
 *     (the output is then unspecified but the call is memory-safe).
 */
#ifndef DS4MOE_H
#define DS4MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream).  NULL = legacy default stream. */
typedef struct CUstream_st *ds4moe_stream_t;

typedef struct ds4moe_layer ds4moe_layer; /* opaque, owned by the library */

enum {
    DS4MOE_OK = 0,
    DS4MOE_ERR_INVALID_ARG = -1,      /* NULL/misaligned pointer, bad size, bad enum */
    DS4MOE_ERR_UNSUPPORTED = -2,      /* shape the kernels do not cover, or no sm_103 device */
    DS4MOE_ERR_CUDA = -3,             /* a CUDA runtime call failed */
    DS4MOE_ERR_OOM = -4,              /* device allocation failed in create */
    DS4MOE_ERR_TOO_MANY_TOKENS = -5,  /* T > config.max_tokens */
    DS4MOE_ERR_DEVICE_TIMEOUT = -6    /* a kernel's bounded wait ran out (see get_status) */
};

enum { DS4MOE_DOWN_MXFP4 = 0, DS4MOE_DOWN_Q2K = 1 };
enum { DS4MOE_PATH_AUTO = 0, DS4MOE_PATH_DECODE = 1, DS4MOE_PATH_PREFILL = 2, DS4MOE_PATH_DECODE_MMA = 3 };

/* Layer shape and options.  Fill with ds4moe_config_default() first.
 *   d_model    hidden size d; multiple of 128, 128..8192.
 *   n_experts  routed experts E; 1..256.
 *   d_ff       expert intermediate size f; multiple of 128 (MXFP4 down) or
 *              of 256 (Q2_K down), 128..8192.
 *   top_k      experts per token k; 1..min(8, E).
 *   max_tokens largest T a forward call may pass (scratch is sized for it).
 *   down_format      DS4MOE_DOWN_MXFP4 or DS4MOE_DOWN_Q2K.  A Q2_K layer runs
 *                    DECODE_MMA and PREFILL like an MXFP4 one (its down
 *                    projection multiplies fp16 h by weights dequantised to
 *                    fp16 on either path); forcing the CUDA-core DECODE path,
 *                    which streams MXFP4 only, is UNSUPPORTED.
 *   decode_max_tokens  AUTO path choice: T <= this runs DECODE_MMA (default 64).
 *   force_path       DS4MOE_PATH_* (AUTO by default; tests force a path).
 *   debug_fault      0 in production.  1 = in the gate/up GEMM, the first
 *                    CTA pair's MMA issuer waits on a barrier that nothing
 *                    arrives on, and the GEMM's waits give up after ~1 ms, so
 *                    ds4moe_get_status() reports DS4MOE_ERR_DEVICE_TIMEOUT
 *                    (fault-handling test; no fault, the GPU stays usable).
 *   wait_timeout_ms  bound on every device-side wait (default 2000).
 *   has_router       1 = the layer holds a router projection (weights.router)
 *                    and ds4moe_forward_x computes the logits; 0 = logits are
 *                    given to ds4moe_forward (default).
 *   d_ff_shared      intermediate size of one shared expert kept at original
 *                    precision (bf16 weights), added to every token's output;
 *                    0 = none (default).  Multiple of 32, at most 16384. */
typedef struct {
    int32_t d_model, n_experts, d_ff, top_k;
    int32_t max_tokens;
    int32_t down_format;
    int32_t decode_max_tokens;
    int32_t force_path;
    int32_t debug_fault;
    int32_t wait_timeout_ms;
    int32_t has_router;
    int32_t d_ff_shared;
} ds4moe_config;

/* Canonical weight layout, DEVICE pointers, read only during create.
 *   gate_codes, up_codes   uint8 [E][f][d/2]   MXFP4 codes, row = output unit
 *   gate_scales, up_scales uint8 [E][f][d/32]  E8M0 scales
 *   MXFP4 down: down_codes uint8 [E][d][f/2], down_scales uint8 [E][d][f/32]
 *   Q2_K down:  down_codes uint8 [E][d][f/256][84], down_scales = NULL
 * Original-precision parts (bf16 raw bits; NULL when not configured):
 *   router       [E][d]      logits = router . x       (has_router = 1)
 *   shared_gate  [fs][d], shared_up [fs][d], shared_down [d][fs]
 *                            the shared expert's SwiGLU FFN (d_ff_shared = fs) */
typedef struct {
    const uint8_t *gate_codes, *gate_scales;
    const uint8_t *up_codes, *up_scales;
    const uint8_t *down_codes, *down_scales;
    const void *router;
    const void *shared_gate, *shared_up, *shared_down;
} ds4moe_weights;

/* Fills *cfg with defaults (all shape fields 0; decode_max_tokens 64,
 * wait_timeout_ms 2000, everything else 0). */
void ds4moe_config_default(ds4moe_config *cfg);

/* Validates cfg, allocates the layer on the CURRENT CUDA device, copies and
 * repacks the weights into library-owned device memory, and synchronises the
 * device before returning (so the caller may free its weight buffers).
 * On success *out receives the layer; on failure *out is set to NULL and
 * nothing stays allocated.  Errors: INVALID_ARG, UNSUPPORTED (shape or a
 * device other than compute capability 10.3), OOM, CUDA. */
int ds4moe_layer_create(const ds4moe_config *cfg, const ds4moe_weights *weights,
                        ds4moe_layer **out);

/* Enqueues one forward pass on `stream` and returns without synchronising.
 *   x       device, bf16 [T][d] row-major (raw bits; 2 bytes per value)
 *   logits  device, fp32 [T][E] row-major router logits
 *   out     device, fp32 [T][d]; fully overwritten
 *   T       0..max_tokens (T = 0 enqueues nothing)
 * x, logits and out stay owned by the caller and must stay valid until the
 * stream work completes; out must not overlap x or logits (INVALID_ARG).
 * Errors: INVALID_ARG, UNSUPPORTED and TOO_MANY_TOKENS (checked on the host
 * before anything is enqueued), CUDA (a launch failed).  Device-side timeouts
 * surface later through ds4moe_get_status. */
int ds4moe_forward(ds4moe_layer *layer, const void *x, const float *logits, float *out,
                   int32_t T, ds4moe_stream_t stream);

/* The whole layer from x alone ("DwarfStar実地分析", §GGUFの対応範囲は意図的に
 * 狭い: the projections, the routing and the shared expert stay at original
 * precision, the routed experts are quantised): logits = router . x in fp32
 * (bf16 products, fp32 accumulation), then the routed experts as in
 * ds4moe_forward, plus the shared expert when d_ff_shared > 0:
 *   out[t] = sum_j w[t,j] * y[t,j] + Wsd . bf16(silu(Wsg . x) * (Wsu . x)).
 * The layer must have has_router = 1 (else UNSUPPORTED).  x device bf16
 * [T][d], out device fp32 [T][d]; asynchronous on `stream`; errors as
 * ds4moe_forward.  ds4moe_forward itself adds the shared expert too when the
 * layer has one (its routing then uses the given logits). */
int ds4moe_forward_x(ds4moe_layer *layer, const void *x, float *out, int32_t T, ds4moe_stream_t stream);

/* Copies the router logits of the most recent ds4moe_forward_x call (device
 * fp32 [T][E], on `stream`).  Errors: INVALID_ARG (no such call yet, NULL),
 * CUDA. */
int ds4moe_get_logits(ds4moe_layer *layer, float *logits, ds4moe_stream_t stream);

/* The same forward pass on HOST buffers: copies x and logits to
 * library-owned device staging on `stream`, runs ds4moe_forward, copies out
 * back, and synchronises `stream` before returning (out is then valid).
 *   x host bf16 [T][d], logits host fp32 [T][E], out host fp32 [T][d].
 * Errors: as ds4moe_forward, plus DEVICE_TIMEOUT if a kernel gave up. */
int ds4moe_forward_host(ds4moe_layer *layer, const void *x, const float *logits, float *out,
                        int32_t T, ds4moe_stream_t stream);

/* Copies the routing of the most recent forward call (device-to-device, on
 * `stream`) into caller buffers; any pointer may be NULL to skip it.
 *   topk_idx  device int32 [T][k]   selected experts, best first
 *   topk_w    device fp32  [T][k]   softmax weights
 *   offsets   device int32 [E+1]    exclusive prefix sum of per-expert counts
 *   perm_tok  device int32 [T*k]    token of each pair in (expert, token) order
 * Errors: INVALID_ARG (no forward yet), CUDA. */
int ds4moe_get_routing(ds4moe_layer *layer, int32_t *topk_idx, float *topk_w, int32_t *offsets,
                       int32_t *perm_tok, ds4moe_stream_t stream);

/* Diagnostics (the pages have no counterpart): copies out the MXFP8
 * activation rows that the most recent forward fed to its grouped tensor-core
 * GEMMs, so that a test can compare these bytes with an independent
 * quantiser.  Enqueued on `stream` (use the forward's stream).
 *   which   0 = x (MXFP8 along d, K = d), 1 = h = SwiGLU output (MXFP8
 *           along f, K = f; MXFP4 down projection only)
 *   codes   device uint8 [T*k*S][K]   E4M3 codes, 16-byte aligned
 *   scales  device uint8 [T*k*S][K/32] E8M0 scale bytes
 * Rows are in token order of the routed pairs, p = t*k + j (j = slot of the
 * token's top-k), and S rows per pair: S = 1 on the PREFILL path; S = 2 on
 * DECODE_MMA (row 2p = hi = MXFP8(v), row 2p + 1 = lo = MXFP8(v - hi)).
 * Returns S (1 or 2) on success, or INVALID_ARG (no forward yet, bad
 * pointer or `which`), UNSUPPORTED (the last forward ran the DECODE GEMV
 * path, or which = 1 on a Q2_K layer, whose h stays fp16), CUDA. */
int ds4moe_get_act_codes(ds4moe_layer *layer, int32_t which, uint8_t *codes, uint8_t *scales,
                         ds4moe_stream_t stream);

/* Synchronises the stream of the most recent forward, reads and clears the
 * layer's device status word.  Returns DS4MOE_OK, DS4MOE_ERR_DEVICE_TIMEOUT
 * (a bounded wait gave up; that forward's output is invalid) or
 * DS4MOE_ERR_CUDA. */
int ds4moe_get_status(ds4moe_layer *layer);

/* DS4MOE_PATH_DECODE, _PREFILL or _DECODE_MMA for a call with T tokens, or
 * a negative error for a NULL layer / T out of range. */
int ds4moe_path_for(const ds4moe_layer *layer, int32_t T);

/* Number of kernels one ds4moe_forward(T) enqueues (0 for T = 0), or a
 * negative error. */
int ds4moe_launches_per_forward(const ds4moe_layer *layer, int32_t T);

/* Per-kernel timing (diagnostics; off by default).  While enabled, every
 * forward also records a CUDA event on its stream before its first kernel and
 * after each kernel.  ds4moe_kernel_times() synchronises that stream and writes
 * the elapsed milliseconds of each kernel of the most recent forward, in
 * launch order, and returns how many it wrote (at most max_n), or a negative
 * error.  ds4moe_kernel_name(layer, T, i) names the i-th kernel a forward of
 * T tokens enqueues (NULL past the end):
 *   A layer with a router or a shared expert first runs dense_in (one cuBLAS
 *   GEMM: router and shared gate/up rows), and with a shared expert then
 *   shared_swiglu; after the routed kernels below, shared_down (cuBLAS).
 *   DECODE:                route_topk, route_group, decode_gateup, decode_down
 *   DECODE_MMA, T <= 4:    route_small, decode_mma_gateup, decode_mma_down (gemm_down for Q2_K)
 *   DECODE_MMA, T > 4:     route_topk, route_group, act_quant, decode_mma_gateup, decode_mma_down
 *                          (gemm_down for Q2_K)
 *   PREFILL, T <= 4:       route_small, gemm_gateup, gemm_down
 *   PREFILL, T > 4:        route_topk, route_group, act_quant, gemm_gateup, gemm_down */
int ds4moe_set_kernel_timing(ds4moe_layer *layer, int enable);
int ds4moe_kernel_times(ds4moe_layer *layer, float *ms, int max_n);
const char *ds4moe_kernel_name(const ds4moe_layer *layer, int32_t T, int i);

/* Routing alone (steps 1-2 above), allocating nothing.  The pages have no
 * counterpart: this call exists for callers that cannot allocate device
 * memory when they route, such as an engine whose memory plan is fixed at
 * start-up, or a serving loop that cannot afford cudaMalloc's implicit device
 * synchronisation.  It needs no layer.  Its scratch is a file-scope device
 * array sized for T*k <= 16384 and E <= 256 (about 390 KB), which every GPU
 * that loads this library keeps until the process exits.
 *   logits    device fp32 [T][E]
 *   topk_idx  device int32 [T][k] out, topk_w device fp32 [T][k] out
 *   offsets   device int32 [E+1] out, perm_tok device int32 [T*k] out
 * Results equal those of ds4moe_forward's routing (see ds4moe_get_routing).
 * T = 0 writes offsets[0..E] = 0 and nothing else (the other pointers may
 * then be NULL).
 * Enqueued on `stream`; no host synchronisation.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current and keeps it for the rest of the process: make that first call
 * before any stream capture, and make no call after cudaDeviceReset() on that
 * device (the kept address belongs to the destroyed context).  Every call
 * shares the one array and nothing in it needs to start at zero; calls whose
 * GPU work overlaps (two streams, two host threads) race on it, so serialise
 * them.
 * Errors: INVALID_ARG (NULL or misaligned pointer, E or k out of range),
 * TOO_MANY_TOKENS (T*k > 16384), CUDA. */
int ds4moe_route_noalloc(const float *logits, int32_t T, int32_t E, int32_t k, int32_t *topk_idx,
                         float *topk_w, int32_t *offsets, int32_t *perm_tok, ds4moe_stream_t stream);

/* Static, human-readable name of a status code. */
const char *ds4moe_status_string(int status);

/* Frees the layer and everything it owns.  NULL-safe.  The caller must have
 * synchronised every stream the layer was used on. */
void ds4moe_destroy(ds4moe_layer *layer);

#ifdef __cplusplus
}
#endif

#endif /* DS4MOE_H */
