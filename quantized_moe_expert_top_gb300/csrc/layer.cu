// C ABI of the ds4moe library: layer creation (weight copies, repacking,
// TMA descriptors), the forward planner, and the query calls.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "common.cuh"
#include "internal.h"

using namespace ds4moe;

namespace {

// Scale bytes [E][rows][K/32] (one per 32-element block) -> the chunk layout the
// tensor-core scale copy reads: one 512-byte chunk per (weight tile, 128-K
// block), byte (t % 32) * 16 + (t / 32) * 4 + (kblock % 4) for tile row t.
// A tile takes `tile_rows` consecutive rows of the matrix (128, or 64 when the
// gate and up rows of 64 features share a tile) at tile rows row_off.. .
__global__ void repack_sf_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E, int rows, int K,
                                 int tile_rows, int row_off) {
  const int nkb = K / 32;
  const size_t total = (size_t)E * rows * nkb;
  const int tiles_per_e = rows / tile_rows, KB = K / kBK;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int kb = (int)(i % nkb);
    const size_t er = i / nkb;
    const int r = (int)(er % rows);
    const int e = (int)(er / rows);
    const size_t chunk = ((size_t)e * tiles_per_e + r / tile_rows) * KB + kb / 4;
    const int t = r % tile_rows + row_off;
    dst[chunk * kSfChunk + (t % 32) * 16 + (t / 32) * 4 + (kb % 4)] = src[i];
  }
}

// Gate/up rows into the tile-major layout: for expert e and 64-feature block
// fb, the 64 gate rows then the same 64 up rows (one 128-row weight tile of
// the paired GEMM), each codes | scales | padding.
__global__ void pack_gu_kernel(uint8_t* __restrict__ dst, int pitch, int E, int d, int f,
                               const uint8_t* __restrict__ gc, const uint8_t* __restrict__ gs,
                               const uint8_t* __restrict__ uc, const uint8_t* __restrict__ us) {
  const int64_t rows = (int64_t)E * f * 2;
  for (int64_t R = blockIdx.x; R < rows; R += gridDim.x) {
    const int r = (int)(R % 128);
    const int j = r / 64;
    const int64_t t = R / 128;                 // e * (f/64) + fb
    const int64_t src_row = t * 64 + r % 64;   // = e * f + fb * 64 + r % 64
    const uint32_t* c = reinterpret_cast<const uint32_t*>((j ? uc : gc) + src_row * (d / 2));
    const uint32_t* sc = reinterpret_cast<const uint32_t*>((j ? us : gs) + src_row * (d / 32));
    uint32_t* o = reinterpret_cast<uint32_t*>(dst + R * pitch);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) o[i] = c[i];
    for (int i = threadIdx.x; i < d / 128; i += blockDim.x) o[d / 8 + i] = sc[i];
    for (int i = d / 8 + d / 128 + threadIdx.x; i < pitch / 4; i += blockDim.x) o[i] = 0u;
  }
}

// Interleaved rows: row r of dst (pitch bytes) = segment 0 row r (l0 bytes) |
// segment 1 row r (l1) | ... (segments with l = 0 are skipped; lengths and
// pitch are multiples of 4 bytes, sources 4-byte aligned).
__global__ void pack_rows_kernel(uint8_t* __restrict__ dst, int pitch, int64_t rows, const uint8_t* __restrict__ s0,
                                 int l0, const uint8_t* __restrict__ s1, int l1, const uint8_t* __restrict__ s2,
                                 int l2, const uint8_t* __restrict__ s3, int l3) {
  const uint8_t* src[4] = {s0, s1, s2, s3};
  const int len[4] = {l0, l1, l2, l3};
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    uint32_t* d = reinterpret_cast<uint32_t*>(dst + r * pitch);
    int off = 0;
    for (int s = 0; s < 4; ++s) {
      if (len[s] == 0) continue;
      const uint32_t* sp = reinterpret_cast<const uint32_t*>(src[s] + r * len[s]);
      for (int i = threadIdx.x; i < len[s] / 4; i += blockDim.x) d[off / 4 + i] = sp[i];
      off += len[s];
    }
    for (int i = off / 4 + threadIdx.x; i < pitch / 4; i += blockDim.x) d[i] = 0u;
  }
}

// Q2_K super-blocks [E][d][f/256][84] -> tile-major chunks [E][d/128][f/64]
// of 3072 bytes: for row r of the 128-row block and K step kb (64 weights,
// quarter kb % 4 of super-block kb / 4): bytes 16r.. four 32-bit words, one
// per 16-weight sub-block, holding the 2-bit code of local weight i at bit
// 2i for even i and 16 + 2(i - 1) for odd i (so one shift and mask yields the
// codes of two neighbouring weights in the two 16-bit halves); 2048 + 4r..
// the 4 sub-block scale bytes; 2560 + 4r.. d | dmin.
__global__ void repack_q2k_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E, int d, int f) {
  const int KB = f / 64, nsb = f / 256;
  const size_t total = (size_t)E * d * KB;  // one thread per (expert, row, K step)
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int kb = (int)(i % KB);
    const size_t er = i / KB;
    const int row = (int)(er % d);
    const int e = (int)(er / d);
    const uint8_t* blk = src + (((size_t)e * d + row) * nsb + kb / 4) * 84;
    const int q4 = kb % 4, r = row % 128;
    uint8_t* ch = dst + (((size_t)e * (d / 128) + row / 128) * KB + kb) * kQ2kChunk;
    for (int sb = 0; sb < 4; ++sb) {
      uint32_t word = 0;
      for (int i = 0; i < 16; ++i) {  // weight 64 q4 + 16 sb + i of the super-block
        const int wi = 64 * q4 + 16 * sb + i;
        const uint32_t qc = (blk[16 + wi / 4] >> (2 * (wi % 4))) & 3u;
        word |= qc << ((i & 1) * 16 + 2 * (i >> 1));
      }
      for (int b = 0; b < 4; ++b) ch[16 * r + 4 * sb + b] = (uint8_t)(word >> (8 * b));
    }
    for (int b = 0; b < 4; ++b) ch[2048 + 4 * r + b] = blk[4 * q4 + b];
    for (int b = 0; b < 4; ++b) ch[2560 + 4 * r + b] = blk[80 + b];
  }
}

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled get_encode_fn() {
  static std::atomic<PFN_encodeTiled> fn{nullptr};
  PFN_encodeTiled f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = (PFN_encodeTiled)p;
      fn.store(f, std::memory_order_release);  // every thread finds the same entry point
    }
  }
  return f;
}

// 2-D row-major tensor map: inner dimension `inner` elements, `rows` rows,
// row pitch `pitch` bytes, box {box_inner, box_rows}, 128-byte swizzle.
bool encode_2d(CUtensorMap* tm, CUtensorMapDataType dt, void* base, uint64_t inner, uint64_t rows, uint64_t pitch,
               uint32_t box_inner, uint32_t box_rows) {
  PFN_encodeTiled fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view {128 elements, rows, K/128} of a row-major matrix whose rows are
// `pitch` bytes apart and whose K = 128 blocks are `kstride` bytes apart, with
// a box of 128 elements x box_rows rows x 2 blocks (128-byte swizzle): one load
// brings two K = 128 blocks as two consecutive [box_rows][128-byte] tiles.
// fp16 h [rows][f] seen as {64 elements, rows, f / 64 blocks}: one box
// {64, box_rows, 2} brings two consecutive 64-element (128-byte) blocks of
// box_rows rows, each block a 128-byte-swizzled [box_rows][128 B] tile.
bool encode_h16_kpairs(CUtensorMap* tm, void* base, uint64_t rows, uint64_t f, uint32_t box_rows) {
  PFN_encodeTiled fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, f / 64};
  cuuint64_t strides[2] = {f * 2, 128};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool encode_3d_kblocks(CUtensorMap* tm, CUtensorMapDataType dt, void* base, uint64_t rows, uint64_t kblocks,
                       uint64_t pitch, uint64_t kstride, uint32_t box_rows) {
  PFN_encodeTiled fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, rows, kblocks};
  cuuint64_t strides[2] = {pitch, kstride};
  cuuint32_t box[3] = {128, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale-factor chunk arrays as rows of 256 bytes (two rows per 512-byte
// chunk), no swizzle.  Weight scales [tiles][K/128][512]: 2-D, box 256 x 8 =
// the chunks of 4 consecutive K blocks of one tile.  Activation scales
// [K/128][rows/128][512]: 3-D {256, 2 * rows/128, K/128}, box 256 x 4 x 4 =
// 2 row blocks x 4 K blocks.
bool encode_sf_weights(CUtensorMap* tm, void* base, uint64_t chunks) {
  PFN_encodeTiled fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {256, chunks * 2};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, 8};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool encode_sf_acts(CUtensorMap* tm, void* base, uint64_t r128, uint64_t kblocks, uint32_t row_blocks = 2) {
  PFN_encodeTiled fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {256, r128 * 2, kblocks};
  cuuint64_t strides[2] = {256, r128 * 512};
  cuuint32_t box[3] = {256, 2 * row_blocks, 4};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int validate_config(const ds4moe_config* c) {
  if (!c) return DS4MOE_ERR_INVALID_ARG;
  if (c->d_model < 128 || c->d_model > 8192 || c->d_model % 128) return DS4MOE_ERR_UNSUPPORTED;
  if (c->d_ff < 128 || c->d_ff > 8192 || c->d_ff % 128) return DS4MOE_ERR_UNSUPPORTED;
  if (c->n_experts < 1 || c->n_experts > 256) return DS4MOE_ERR_UNSUPPORTED;
  if (c->top_k < 1 || c->top_k > 8 || c->top_k > c->n_experts) return DS4MOE_ERR_UNSUPPORTED;
  if (c->max_tokens < 1 || c->max_tokens > (1 << 20) / c->top_k) return DS4MOE_ERR_INVALID_ARG;
  if (c->down_format != DS4MOE_DOWN_MXFP4 && c->down_format != DS4MOE_DOWN_Q2K) return DS4MOE_ERR_INVALID_ARG;
  if (c->down_format == DS4MOE_DOWN_Q2K && c->d_ff % 256) return DS4MOE_ERR_UNSUPPORTED;
  if (c->decode_max_tokens < 0) return DS4MOE_ERR_INVALID_ARG;
  if (c->force_path < DS4MOE_PATH_AUTO || c->force_path > DS4MOE_PATH_DECODE_MMA) return DS4MOE_ERR_INVALID_ARG;
  if (c->wait_timeout_ms < 1 || c->wait_timeout_ms > 60000) return DS4MOE_ERR_INVALID_ARG;
  if (c->has_router != 0 && c->has_router != 1) return DS4MOE_ERR_INVALID_ARG;
  if (c->d_ff_shared < 0 || c->d_ff_shared > 16384 || c->d_ff_shared % 32) return DS4MOE_ERR_UNSUPPORTED;
  return DS4MOE_OK;
}

template <typename Tp>
int alloc(ds4moe_layer* L, Tp** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  if (L->n_owned >= (int)(sizeof(L->owned) / sizeof(L->owned[0]))) return DS4MOE_ERR_OOM;
  void* q = nullptr;
  if (cudaMalloc(&q, bytes) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_OOM;
  }
  L->owned[L->n_owned++] = q;
  *p = static_cast<Tp*>(q);
  return DS4MOE_OK;
}

int path_of(const ds4moe_layer* L, int T) {
  if (L->cfg.force_path != DS4MOE_PATH_AUTO) return L->cfg.force_path;
  return T <= L->cfg.decode_max_tokens ? DS4MOE_PATH_DECODE_MMA : DS4MOE_PATH_PREFILL;
}

// Names of the kernels one forward of T tokens enqueues, in launch order
// (with_x: the call computes its logits from x).
bool runs_dense_in(const ds4moe_layer* L, bool with_x) {
  return L->dense_n > 0 && (with_x || L->cfg.d_ff_shared > 0);
}

int kernel_list(const ds4moe_layer* L, int T, bool with_x, const char** names) {
  int n = 0;
  const int path = path_of(L, T);
  if (runs_dense_in(L, with_x)) names[n++] = "dense_in";
  if (L->cfg.d_ff_shared > 0) names[n++] = "shared_swiglu";
  if (path == DS4MOE_PATH_DECODE) {
    for (const char* k : {"route_topk", "route_group", "decode_gateup", "decode_down"}) names[n++] = k;
  } else {
    if (T <= kSmallRouteT) {
      names[n++] = "route_small";
    } else {
      for (const char* k : {"route_topk", "route_group", "act_quant"}) names[n++] = k;
    }
    const bool dm = path == DS4MOE_PATH_DECODE_MMA;
    const bool q2k = L->cfg.down_format == DS4MOE_DOWN_Q2K;
    names[n++] = dm ? "decode_mma_gateup" : "gemm_gateup";
    names[n++] = (dm && !q2k) ? "decode_mma_down" : "gemm_down";
  }
  if (L->cfg.d_ff_shared > 0) names[n++] = "shared_down";
  return n;
}

void free_all(ds4moe_layer* L) {
  dense_destroy(L);
  for (int i = 0; i < L->n_owned; ++i) cudaFree(L->owned[i]);
  L->n_owned = 0;
}

}  // namespace

extern "C" {

void ds4moe_config_default(ds4moe_config* cfg) {
  if (!cfg) return;
  memset(cfg, 0, sizeof(*cfg));
  cfg->decode_max_tokens = 64;
  cfg->wait_timeout_ms = 2000;
}

const char* ds4moe_status_string(int s) {
  switch (s) {
    case DS4MOE_OK: return "ok";
    case DS4MOE_ERR_INVALID_ARG: return "invalid argument";
    case DS4MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
    case DS4MOE_ERR_CUDA: return "CUDA runtime error";
    case DS4MOE_ERR_OOM: return "out of device memory";
    case DS4MOE_ERR_TOO_MANY_TOKENS: return "T exceeds max_tokens";
    case DS4MOE_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    default: return "unknown status";
  }
}

int ds4moe_layer_create(const ds4moe_config* cfg, const ds4moe_weights* wts, ds4moe_layer** out) {
  if (!out) return DS4MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc != DS4MOE_OK) return rc;
  if (!wts || !wts->gate_codes || !wts->gate_scales || !wts->up_codes || !wts->up_scales || !wts->down_codes)
    return DS4MOE_ERR_INVALID_ARG;
  if (cfg->down_format == DS4MOE_DOWN_MXFP4 && !wts->down_scales) return DS4MOE_ERR_INVALID_ARG;
  if (cfg->has_router && (!wts->router || !aligned16(wts->router))) return DS4MOE_ERR_INVALID_ARG;
  if (cfg->d_ff_shared > 0 && (!wts->shared_gate || !wts->shared_up || !wts->shared_down ||
                               !aligned16(wts->shared_gate) || !aligned16(wts->shared_up) ||
                               !aligned16(wts->shared_down)))
    return DS4MOE_ERR_INVALID_ARG;
  if (!aligned16(wts->gate_codes) || !aligned16(wts->up_codes) || !aligned16(wts->down_codes) ||
      !aligned16(wts->gate_scales) || !aligned16(wts->up_scales) ||
      (wts->down_scales && !aligned16(wts->down_scales)))
    return DS4MOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS4MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DS4MOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return DS4MOE_ERR_UNSUPPORTED;

  ds4moe_layer* L = new (std::nothrow) ds4moe_layer();
  if (!L) return DS4MOE_ERR_OOM;
  memset((void*)L, 0, sizeof(*L));
  L->cfg = *cfg;
  L->device = dev;
  L->num_sms = prop.multiProcessorCount;

  const int E = cfg->n_experts, d = cfg->d_model, f = cfg->d_ff, k = cfg->top_k, Tm = cfg->max_tokens;
  const size_t gu_codes = (size_t)E * f * (d / 2), gu_scales = (size_t)E * f * (d / 32);
  const size_t dn_codes = (size_t)E * d * (f / 2), dn_scales = (size_t)E * d * (f / 32);
  const int64_t pairs = (int64_t)Tm * k;
  const bool q2k = cfg->down_format == DS4MOE_DOWN_Q2K;
  if (q2k && cfg->force_path == DS4MOE_PATH_DECODE) {
    delete L;  // the CUDA-core GEMV streams MXFP4 only
    return DS4MOE_ERR_UNSUPPORTED;
  }
  // GEMV buffers only when that path is forced; the GEMM buffers serve PREFILL and DECODE_MMA.
  const bool need_dec = !q2k && cfg->force_path == DS4MOE_PATH_DECODE;
  const bool need_pre = cfg->force_path != DS4MOE_PATH_DECODE;
  const bool split_ok = cfg->force_path == DS4MOE_PATH_DECODE_MMA ||
                        (cfg->force_path == DS4MOE_PATH_AUTO && cfg->decode_max_tokens > 0);
  const int Tdec = (cfg->force_path != DS4MOE_PATH_AUTO || Tm < cfg->decode_max_tokens) ? Tm
                                                                                       : cfg->decode_max_tokens;
  // padded activation rows: one per routed pair (PREFILL), two (DECODE_MMA)
  const int64_t split_rows = split_ok ? 2 * (int64_t)Tdec * k : 0;
  const int64_t rows_needed = (pairs > split_rows ? pairs : split_rows) + (int64_t)E * (kPadRows - 1);
  const int64_t pad_rows = (rows_needed + kPadRows - 1) / kPadRows * kPadRows;
  L->s.pad_rows_max = pad_rows;
  L->w.pitch_gu = (d / 2 + d / 32 + 31) / 32 * 32;
  L->w.pitch_dn = (f / 2 + f / 32 + 31) / 32 * 32;

#define TRY(x)                 \
  do {                         \
    rc = (x);                  \
    if (rc != DS4MOE_OK) goto fail; \
  } while (0)
  {
    Weights& w = L->w;
    Scratch& s = L->s;
    TRY(alloc(L, &w.gu, (size_t)E * f * 2 * w.pitch_gu));
    if (need_pre) TRY(alloc(L, &w.gu_sf, 2 * gu_scales));
    if (!q2k) {
      TRY(alloc(L, &w.dn, (size_t)E * d * w.pitch_dn));
      if (need_pre) TRY(alloc(L, &w.down_sf, dn_scales));
    } else {
      TRY(alloc(L, &w.q2k, (size_t)E * (d / 128) * (f / 64) * kQ2kChunk));
    }
    TRY(alloc(L, &s.topk_idx, pairs * 4));
    TRY(alloc(L, &s.topk_w, pairs * 4));
    TRY(alloc(L, &s.counts, (size_t)E * 4));
    TRY(alloc(L, &s.offsets, (size_t)(E + 1) * 4));
    TRY(alloc(L, &s.pad_offsets, (size_t)(E + 1) * 4));
    TRY(alloc(L, &s.perm_tok, pairs * 4));
    TRY(alloc(L, &s.perm_slot, pairs * 4));
    TRY(alloc(L, &s.inv, pairs * 4));
    TRY(alloc(L, &s.pad_inv, pairs * 4));
    TRY(alloc(L, &s.pad_pair, (size_t)pad_rows * 4));
    TRY(alloc(L, &s.touched, (size_t)(E + 1) * 4));
    if (need_dec) {
      TRY(alloc(L, &s.h_dec, (size_t)Tdec * k * f * 4));
      TRY(alloc(L, &s.xh, (size_t)Tdec * d * 2));
      TRY(alloc(L, &s.xsig, (size_t)Tdec * 4));
    }
    if (split_ok) {
      s.dec_maxch = (int)((2 * (int64_t)Tdec + 127) / 128);
      TRY(alloc(L, &s.gu_acc, (size_t)Tdec * k * 2 * f * 4));
      TRY(alloc(L, &s.tile_cnt, (size_t)E * (f / 64) * s.dec_maxch * 4));
    }
    if (need_pre) {
      TRY(alloc(L, &s.xq, (size_t)pad_rows * d));
      TRY(alloc(L, &s.xsf, (size_t)pad_rows * d / 32));
      if (q2k) {
        TRY(alloc(L, &s.h16, (size_t)pad_rows * f * 2));
      } else {
        TRY(alloc(L, &s.hq, (size_t)pad_rows * f));
        TRY(alloc(L, &s.hsf, (size_t)pad_rows * f / 32));
      }
    }
    const int fs = cfg->d_ff_shared;
    // The shared gate block starts on a multiple of four columns (zero rows
    // pad the router block), so that the SwiGLU kernel's 16-byte loads of g
    // and u are aligned for any E.
    L->dense_goff = cfg->has_router ? (fs > 0 ? (E + 3) / 4 * 4 : E) : 0;
    L->dense_n = L->dense_goff + 2 * fs;
    if (L->dense_n > 0) {
      constexpr size_t kBlasWs = 32u << 20;
      TRY(alloc(L, &L->wcat, (size_t)L->dense_n * d * 2));
      TRY(alloc(L, &s.dense_c, (size_t)Tm * L->dense_n * 4));
      TRY(alloc(L, &s.blas_ws, kBlasWs));
      if (fs > 0) {
        TRY(alloc(L, &L->wsd, (size_t)d * fs * 2));
        TRY(alloc(L, &s.h_shared, (size_t)Tm * fs * 2));
      }
      const int npad = cfg->has_router ? L->dense_goff - E : 0;  // zero rows after the router's E
      bool okc = npad == 0 || cudaMemset(L->wcat + (size_t)E * d, 0, (size_t)npad * d * 2) == cudaSuccess;
      if (cfg->has_router)
        okc = okc && cudaMemcpy(L->wcat, wts->router, (size_t)E * d * 2, cudaMemcpyDeviceToDevice) == cudaSuccess;
      if (fs > 0) {
        okc = okc && cudaMemcpy(L->wcat + (size_t)L->dense_goff * d, wts->shared_gate, (size_t)fs * d * 2,
                                cudaMemcpyDeviceToDevice) == cudaSuccess;
        okc = okc && cudaMemcpy(L->wcat + (size_t)(L->dense_goff + fs) * d, wts->shared_up, (size_t)fs * d * 2,
                                cudaMemcpyDeviceToDevice) == cudaSuccess;
        okc = okc && cudaMemcpy(L->wsd, wts->shared_down, (size_t)d * fs * 2, cudaMemcpyDeviceToDevice) == cudaSuccess;
      }
      if (!okc || dense_create(L, kBlasWs, s.blas_ws) != cudaSuccess) {
        rc = DS4MOE_ERR_CUDA;
        goto fail;
      }
    }
    TRY(alloc(L, &s.stage_x, (size_t)Tm * d * 2));
    TRY(alloc(L, &s.stage_logits, (size_t)Tm * E * 4));
    TRY(alloc(L, &s.stage_out, (size_t)Tm * d * 4));
    TRY(alloc(L, &L->status, sizeof(DeviceStatus)));

    cudaStream_t st = nullptr;
    bool ok = cudaMemset(L->status, 0, sizeof(DeviceStatus)) == cudaSuccess;
    ok = ok && cudaMemset(s.pad_pair, 0xFF, (size_t)pad_rows * 4) == cudaSuccess;
    if (split_ok) {
      ok = ok && cudaMemset(s.gu_acc, 0, (size_t)Tdec * k * 2 * f * 4) == cudaSuccess;
      ok = ok && cudaMemset(s.tile_cnt, 0, (size_t)E * (f / 64) * s.dec_maxch * 4) == cudaSuccess;
    }
    if (need_pre) {
      // padding rows of the activation buffers hold zeros (finite codes)
      ok = ok && cudaMemset(s.xq, 0, (size_t)pad_rows * d) == cudaSuccess;
      ok = ok && cudaMemset(s.xsf, 127, (size_t)pad_rows * d / 32) == cudaSuccess;
      if (q2k) {
        ok = ok && cudaMemset(s.h16, 0, (size_t)pad_rows * f * 2) == cudaSuccess;
      } else {
        ok = ok && cudaMemset(s.hq, 0, (size_t)pad_rows * f) == cudaSuccess;
        ok = ok && cudaMemset(s.hsf, 127, (size_t)pad_rows * f / 32) == cudaSuccess;
      }
    }
    if (!ok) {
      rc = DS4MOE_ERR_CUDA;
      goto fail;
    }
    (void)gu_codes;
    (void)dn_codes;
    if (launch_pack_gu(wts, L, st) != cudaSuccess ||
        (!q2k && launch_pack_rows(w.dn, w.pitch_dn, (int64_t)E * d, wts->down_codes, f / 2, wts->down_scales,
                                  f / 32, nullptr, 0, nullptr, 0, st) != cudaSuccess)) {
      rc = DS4MOE_ERR_CUDA;
      goto fail;
    }
    if (need_pre) {
      if (launch_repack_sf(wts->gate_scales, w.gu_sf, E, f, d, 64, 0, st) != cudaSuccess ||
          launch_repack_sf(wts->up_scales, w.gu_sf, E, f, d, 64, 64, st) != cudaSuccess ||
          (!q2k && launch_repack_sf(wts->down_scales, w.down_sf, E, d, f, 128, 0, st) != cudaSuccess)) {
        rc = DS4MOE_ERR_CUDA;
        goto fail;
      }
    }
    if (q2k && launch_repack_q2k(wts->down_codes, L, st) != cudaSuccess) {
      rc = DS4MOE_ERR_CUDA;
      goto fail;
    }
    if (need_pre) {
      bool tm_ok = encode_2d(&L->tm_gu, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w.gu, d, (uint64_t)E * f * 2,
                             w.pitch_gu, 128, 128);
      for (int b = 0; b < kNumBoxMaps; ++b) {
        const uint32_t rows = 16u * (uint32_t)(b + 1);
        tm_ok = tm_ok && encode_2d(&L->tm_xq[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, s.xq, d, pad_rows, d, 128, rows);
        if (!q2k)
          tm_ok = tm_ok && encode_2d(&L->tm_hq[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, s.hq, f, pad_rows, f, 128, rows);
        else
          tm_ok = tm_ok && encode_h16_kpairs(&L->tm_h16[b], s.h16, pad_rows, f, rows);
      }
      if (!q2k)
        tm_ok = tm_ok && encode_2d(&L->tm_down, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w.dn, f, (uint64_t)E * d,
                                   w.pitch_dn, 128, 128);
      const uint64_t r128 = (uint64_t)pad_rows / 128;
      tm_ok = tm_ok && encode_sf_weights(&L->tm_sfa_gu, w.gu_sf, (uint64_t)E * (f / 64) * (d / 128));
      tm_ok = tm_ok && encode_sf_acts(&L->tm_sfb_x, s.xsf, r128, (uint64_t)d / 128);
      if (!q2k) {
        tm_ok = tm_ok && encode_sf_weights(&L->tm_sfa_dn, w.down_sf, (uint64_t)E * (d / 128) * (f / 128));
        tm_ok = tm_ok && encode_sf_acts(&L->tm_sfb_h, s.hsf, r128, (uint64_t)f / 128);
      }
      // 3-D views loading two K = 128 blocks per box (both tensor-core paths):
      // gate/up side for both down formats, then the MXFP4 down side
      tm_ok = tm_ok && encode_3d_kblocks(&L->tm_gu3, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w.gu,
                                         (uint64_t)E * f * 2, (uint64_t)d / 128, w.pitch_gu, 64, 128);
      for (int b = 0; b < 8; ++b)
        tm_ok = tm_ok && encode_3d_kblocks(&L->tm_xq3[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, s.xq, pad_rows,
                                           (uint64_t)d / 128, d, 128, 16u * (uint32_t)(b + 1));
      if (!q2k) {
        tm_ok = tm_ok && encode_3d_kblocks(&L->tm_dn3, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w.dn,
                                           (uint64_t)E * d, (uint64_t)f / 128, w.pitch_dn, 64, 128);
        for (int b = 0; b < 8; ++b)
          tm_ok = tm_ok && encode_3d_kblocks(&L->tm_hq3[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, s.hq, pad_rows,
                                             (uint64_t)f / 128, f, 128, 16u * (uint32_t)(b + 1));
      }
      if (split_ok) {
        tm_ok = tm_ok && encode_sf_acts(&L->tm_sfb_x1, s.xsf, r128, (uint64_t)d / 128, 1);
        if (!q2k) tm_ok = tm_ok && encode_sf_acts(&L->tm_sfb_h1, s.hsf, r128, (uint64_t)f / 128, 1);
        L->decmma_ready = tm_ok;
      }
      if (!tm_ok) {
        rc = DS4MOE_ERR_CUDA;
        goto fail;
      }
      L->prefill_ready = true;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
      rc = DS4MOE_ERR_CUDA;
      goto fail;
    }
  }
#undef TRY
  *out = L;
  return DS4MOE_OK;
fail:
  cudaGetLastError();
  free_all(L);
  delete L;
  return rc;
}

int ds4moe_path_for(const ds4moe_layer* L, int32_t T) {
  if (!L) return DS4MOE_ERR_INVALID_ARG;
  if (T < 0 || T > L->cfg.max_tokens) return DS4MOE_ERR_TOO_MANY_TOKENS;
  return path_of(L, T);
}

int ds4moe_launches_per_forward(const ds4moe_layer* L, int32_t T) {
  const int p = ds4moe_path_for(L, T);
  if (p < 0) return p;
  if (T == 0) return 0;
  const char* names[12];
  return kernel_list(L, T, L->last_forward_x, names);
}

namespace {
// One forward pass; logits == nullptr: computed from x by the router (dense_in).
int enqueue_forward(ds4moe_layer* L, const void* x, const float* logits, float* out, int32_t T,
                    ds4moe_stream_t stream);
}  // namespace

int ds4moe_forward(ds4moe_layer* L, const void* x, const float* logits, float* out, int32_t T,
                   ds4moe_stream_t stream) {
  if (!L) return DS4MOE_ERR_INVALID_ARG;
  if (!logits && T > 0) return DS4MOE_ERR_INVALID_ARG;
  return enqueue_forward(L, x, logits, out, T, stream);
}

int ds4moe_forward_x(ds4moe_layer* L, const void* x, float* out, int32_t T, ds4moe_stream_t stream) {
  if (!L) return DS4MOE_ERR_INVALID_ARG;
  if (!L->cfg.has_router) return DS4MOE_ERR_UNSUPPORTED;
  return enqueue_forward(L, x, nullptr, out, T, stream);
}

int ds4moe_get_logits(ds4moe_layer* L, float* logits, ds4moe_stream_t stream) {
  if (!L || !logits || !L->has_forward || !L->last_forward_x) return DS4MOE_ERR_INVALID_ARG;
  const size_t E = (size_t)L->cfg.n_experts;
  if (cudaMemcpy2DAsync(logits, E * 4, L->s.dense_c, (size_t)L->dense_n * 4, E * 4, (size_t)L->last_T,
                        cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  return DS4MOE_OK;
}

namespace {
int enqueue_forward(ds4moe_layer* L, const void* x, const float* logits, float* out, int32_t T,
                    ds4moe_stream_t stream) {
  if (T < 0) return DS4MOE_ERR_INVALID_ARG;
  if (T > L->cfg.max_tokens) return DS4MOE_ERR_TOO_MANY_TOKENS;
  if (T == 0) return DS4MOE_OK;
  const bool with_x = logits == nullptr;
  if (!x || !out || !aligned16(x) || !aligned16(out) || (logits && !aligned16(logits))) return DS4MOE_ERR_INVALID_ARG;
  {
    // out may not overlap x or logits (the kernels zero and accumulate into out
    // while x and the logits are still being read)
    const uintptr_t o0 = (uintptr_t)out, o1 = o0 + (uintptr_t)T * L->cfg.d_model * 4;
    const uintptr_t x0 = (uintptr_t)x, x1 = x0 + (uintptr_t)T * L->cfg.d_model * 2;
    const uintptr_t l0 = (uintptr_t)logits, l1 = logits ? l0 + (uintptr_t)T * L->cfg.n_experts * 4 : l0;
    if ((o0 < x1 && x0 < o1) || (o0 < l1 && l0 < o1)) return DS4MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int path = path_of(L, T);
  if (path == DS4MOE_PATH_DECODE && !L->s.h_dec) return DS4MOE_ERR_UNSUPPORTED;
  if (path != DS4MOE_PATH_DECODE && !L->prefill_ready) return DS4MOE_ERR_UNSUPPORTED;
  if (path == DS4MOE_PATH_DECODE_MMA && !L->decmma_ready) return DS4MOE_ERR_UNSUPPORTED;
  if (path == DS4MOE_PATH_DECODE_MMA &&
      2 * (int64_t)T * L->cfg.top_k + (int64_t)L->cfg.n_experts * (kPadRows - 1) > L->s.pad_rows_max)
    return DS4MOE_ERR_UNSUPPORTED;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != L->device) return DS4MOE_ERR_INVALID_ARG;

  L->last_stream = st;
  const int split = path == DS4MOE_PATH_DECODE_MMA ? 2 : 1;
  int nk = 0;
  auto mark = [&](cudaError_t e) {
    if (e == cudaSuccess && L->timing) e = cudaEventRecord(L->ev[nk], st);
    ++nk;
    return e;
  };
  cudaError_t e = L->timing ? cudaEventRecord(L->ev[0], st) : cudaSuccess;
  nk = 1;
  int lds = L->cfg.n_experts;
  if (runs_dense_in(L, with_x)) {
    if (e == cudaSuccess) e = mark(launch_dense_in(L, x, T, st));
    if (with_x) {
      logits = L->s.dense_c;
      lds = L->dense_n;
    }
  }
  if (L->cfg.d_ff_shared > 0 && e == cudaSuccess) e = mark(launch_shared_swiglu(L, T, st));
  if (path == DS4MOE_PATH_DECODE) {
    if (e == cudaSuccess) e = mark(launch_route_topk(L, logits, lds, x, true, T, st));
    if (e == cudaSuccess) e = mark(launch_route_group(L, T, split, st));
    if (e == cudaSuccess) e = mark(launch_decode_gateup(L, x, out, T, st));
    if (e == cudaSuccess) e = mark(launch_decode_down(L, out, T, st));
  } else {
    if (T <= kSmallRouteT) {
      // routing and the activations in one launch
      if (e == cudaSuccess) e = mark(launch_route_small(L, logits, lds, x, out, T, split, true, st));
    } else {
      if (e == cudaSuccess) e = mark(launch_route_topk(L, logits, lds, x, false, T, st));
      if (e == cudaSuccess) e = mark(launch_route_group(L, T, split, st));
      if (e == cudaSuccess) e = mark(launch_act_quant(L, x, out, T, split, st));
    }
    const bool q2k = L->cfg.down_format == DS4MOE_DOWN_Q2K;
    if (path == DS4MOE_PATH_DECODE_MMA) {
      if (e == cudaSuccess) e = mark(launch_decmma_gateup(L, T, st));
      if (e == cudaSuccess) e = mark(q2k ? launch_gemm_down_q2k(L, out, T, 2, st) : launch_decmma_down(L, out, T, st));
    } else {
      if (e == cudaSuccess) e = mark(launch_gemm_gateup(L, T, split, st));
      if (e == cudaSuccess)
        e = mark(q2k ? launch_gemm_down_q2k(L, out, T, 1, st) : launch_gemm_down(L, out, T, split, st));
    }
  }
  if (L->cfg.d_ff_shared > 0 && e == cudaSuccess) e = mark(launch_shared_down(L, out, T, st));
  L->last_nk = nk - 1;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  L->last_T = T;
  L->last_path = path;
  L->last_split = split;
  L->last_forward_x = with_x;
  L->has_forward = true;
  return DS4MOE_OK;
}
}  // namespace

int ds4moe_forward_host(ds4moe_layer* L, const void* x, const float* logits, float* out, int32_t T,
                        ds4moe_stream_t stream) {
  if (!L) return DS4MOE_ERR_INVALID_ARG;
  if (T < 0) return DS4MOE_ERR_INVALID_ARG;
  if (T > L->cfg.max_tokens) return DS4MOE_ERR_TOO_MANY_TOKENS;
  if (T == 0) return DS4MOE_OK;
  if (!x || !logits || !out) return DS4MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * L->cfg.d_model * 2, lb = (size_t)T * L->cfg.n_experts * 4,
               ob = (size_t)T * L->cfg.d_model * 4;
  if (cudaMemcpyAsync(L->s.stage_x, x, xb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(L->s.stage_logits, logits, lb, cudaMemcpyHostToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  int rc = ds4moe_forward(L, L->s.stage_x, L->s.stage_logits, L->s.stage_out, T, stream);
  if (rc != DS4MOE_OK) return rc;
  if (cudaMemcpyAsync(out, L->s.stage_out, ob, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  return ds4moe_get_status(L);  // synchronises the stream, reads and clears the status word
}

int ds4moe_get_routing(ds4moe_layer* L, int32_t* topk_idx, float* topk_w, int32_t* offsets, int32_t* perm_tok,
                       ds4moe_stream_t stream) {
  if (!L || !L->has_forward) return DS4MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t pairs = (size_t)L->last_T * L->cfg.top_k;
  bool ok = true;
  if (topk_idx) ok = ok && cudaMemcpyAsync(topk_idx, L->s.topk_idx, pairs * 4, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
  if (topk_w) ok = ok && cudaMemcpyAsync(topk_w, L->s.topk_w, pairs * 4, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
  if (offsets)
    ok = ok && cudaMemcpyAsync(offsets, L->s.offsets, (size_t)(L->cfg.n_experts + 1) * 4, cudaMemcpyDeviceToDevice,
                               st) == cudaSuccess;
  if (perm_tok) ok = ok && cudaMemcpyAsync(perm_tok, L->s.perm_tok, pairs * 4, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  return DS4MOE_OK;
}

int ds4moe_get_act_codes(ds4moe_layer* L, int32_t which, uint8_t* codes, uint8_t* scales, ds4moe_stream_t stream) {
  if (!L || !L->has_forward || (which != 0 && which != 1) || !codes || !scales || !aligned16(codes))
    return DS4MOE_ERR_INVALID_ARG;
  if (L->last_path == DS4MOE_PATH_DECODE) return DS4MOE_ERR_UNSUPPORTED;         // the GEMV path has no MXFP8 rows
  if (which == 1 && L->cfg.down_format == DS4MOE_DOWN_Q2K) return DS4MOE_ERR_UNSUPPORTED;  // h stays fp16 there
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != L->device) return DS4MOE_ERR_INVALID_ARG;
  if (launch_gather_act(L, which, L->last_T, L->last_split, codes, scales,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  return L->last_split;
}

int ds4moe_get_status(ds4moe_layer* L) {
  if (!L) return DS4MOE_ERR_INVALID_ARG;
  if (L->has_forward && cudaStreamSynchronize(L->last_stream) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  DeviceStatus hs;
  if (cudaMemcpy(&hs, L->status, sizeof(hs), cudaMemcpyDeviceToHost) != cudaSuccess) return DS4MOE_ERR_CUDA;
  if (hs.code != kStatusOk) {
    DeviceStatus z;
    memset(&z, 0, sizeof(z));
    if (cudaMemcpy(L->status, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return DS4MOE_ERR_CUDA;
    // a call that gave up may have left partial sums and tile counts behind;
    // the next call expects them at zero
    if (L->s.gu_acc) {
      const ds4moe_config& c = L->cfg;
      const int Tdec = (c.force_path != DS4MOE_PATH_AUTO || c.max_tokens < c.decode_max_tokens) ? c.max_tokens
                                                                                              : c.decode_max_tokens;
      if (cudaMemset(L->s.gu_acc, 0, (size_t)Tdec * c.top_k * 2 * c.d_ff * 4) != cudaSuccess ||
          cudaMemset(L->s.tile_cnt, 0, (size_t)c.n_experts * (c.d_ff / 64) * L->s.dec_maxch * 4) != cudaSuccess ||
          cudaDeviceSynchronize() != cudaSuccess)
        return DS4MOE_ERR_CUDA;
    }
    return DS4MOE_ERR_DEVICE_TIMEOUT;
  }
  return DS4MOE_OK;
}

int ds4moe_set_kernel_timing(ds4moe_layer* L, int enable) {
  if (!L) return DS4MOE_ERR_INVALID_ARG;
  if (enable && !L->ev[0]) {
    for (int i = 0; i < 12; ++i)
      if (cudaEventCreate(&L->ev[i]) != cudaSuccess) {
        cudaGetLastError();
        return DS4MOE_ERR_CUDA;
      }
  }
  L->timing = enable != 0;
  return DS4MOE_OK;
}

int ds4moe_kernel_times(ds4moe_layer* L, float* ms, int max_n) {
  if (!L || !ms || max_n < 0) return DS4MOE_ERR_INVALID_ARG;
  if (!L->timing || !L->has_forward) return DS4MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(L->last_stream) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  const int n = L->last_nk < max_n ? L->last_nk : max_n;
  for (int i = 0; i < n; ++i)
    if (cudaEventElapsedTime(&ms[i], L->ev[i], L->ev[i + 1]) != cudaSuccess) {
      cudaGetLastError();
      return DS4MOE_ERR_CUDA;
    }
  return n;
}

const char* ds4moe_kernel_name(const ds4moe_layer* L, int32_t T, int i) {
  if (!L || T <= 0 || T > L->cfg.max_tokens || i < 0) return nullptr;
  const char* names[12];
  const int n = kernel_list(L, T, L->last_forward_x, names);
  return i < n ? names[i] : nullptr;
}

void ds4moe_destroy(ds4moe_layer* L) {
  if (!L) return;
  for (int i = 0; i < 12; ++i)
    if (L->ev[i]) cudaEventDestroy(L->ev[i]);
  free_all(L);
  delete L;
}

}  // extern "C"

namespace ds4moe {

cudaError_t launch_repack_sf(const uint8_t* scales, uint8_t* sf, int E, int rows, int K, int tile_rows, int row_off,
                             cudaStream_t st) {
  const size_t total = (size_t)E * rows * (K / 32);
  const int blocks = (int)((total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536);
  repack_sf_kernel<<<blocks, 256, 0, st>>>(scales, sf, E, rows, K, tile_rows, row_off);
  return cudaGetLastError();
}

cudaError_t launch_pack_gu(const ds4moe_weights* w, ds4moe_layer* L, cudaStream_t st) {
  const int64_t rows = (int64_t)L->cfg.n_experts * L->cfg.d_ff * 2;
  const int grid = (int)(rows < 65536 ? rows : 65536);
  pack_gu_kernel<<<grid, 128, 0, st>>>(L->w.gu, L->w.pitch_gu, L->cfg.n_experts, L->cfg.d_model, L->cfg.d_ff,
                                       w->gate_codes, w->gate_scales, w->up_codes, w->up_scales);
  return cudaGetLastError();
}

cudaError_t launch_pack_rows(uint8_t* dst, int pitch, int64_t rows, const uint8_t* s0, int l0, const uint8_t* s1,
                             int l1, const uint8_t* s2, int l2, const uint8_t* s3, int l3, cudaStream_t st) {
  const int grid = (int)(rows < 65536 ? rows : 65536);
  pack_rows_kernel<<<grid, 128, 0, st>>>(dst, pitch, rows, s0, l0, s1, l1, s2, l2, s3, l3);
  return cudaGetLastError();
}

cudaError_t launch_repack_q2k(const uint8_t* blocks, ds4moe_layer* L, cudaStream_t st) {
  const size_t n = (size_t)L->cfg.n_experts * L->cfg.d_model * (L->cfg.d_ff / 64);
  const int grid = (int)((n + 255) / 256 < 65536 ? (n + 255) / 256 : 65536);
  repack_q2k_kernel<<<grid, 256, 0, st>>>(blocks, L->w.q2k, L->cfg.n_experts, L->cfg.d_model, L->cfg.d_ff);
  return cudaGetLastError();
}

}  // namespace ds4moe
