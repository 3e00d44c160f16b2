// The layer's original-precision parts: the router projection and the shared
// expert.
//
// "DwarfStar実地分析" §GGUFの対応範囲は意図的に狭い: only the routed experts are
// quantised; the shared expert, the projections and the routing stay at the
// model's original precision (bf16 weights and activations).  Their two
// dense products are plain bf16 GEMMs and run in cuBLAS (fp32 accumulation on
// the tensor cores):
//
//   dense_in    C[T][N] = x[T][d] . Wcat[N][d]^T with Wcat = [router (E rows) |
//               shared gate (fs rows) | shared up (fs rows)], one pass over x;
//               the routing reads its logits as the first E columns of C.
//   shared_down out[T][d] += h[T][fs] . Wd[d][fs]^T (beta = 1), after the
//               routed combine has written out.
//
// Between them shared_swiglu_kernel forms h = silu(g) * u in fp32 and rounds
// it to bf16 (round to nearest even), the activation precision of the model.
#include <cublas_v2.h>

#include "common.cuh"
#include "internal.h"

namespace ds4moe {
namespace {

// One thread per 4 consecutive features of a token: g and u from the dense_in
// output, h = bf16(silu(g) * u).
__global__ void __launch_bounds__(256) shared_swiglu_kernel(const float* __restrict__ c, int ldc, int goff, int fs,
                                                            int T, __nv_bfloat16* __restrict__ h) {
  pdl_wait();
  pdl_launch_dependents();
  const int per_tok = fs / 4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * per_tok; i += gridDim.x * blockDim.x) {
    const int t = i / per_tok, j = (i % per_tok) * 4;
    const float4 g = *reinterpret_cast<const float4*>(c + (size_t)t * ldc + goff + j);
    const float4 u = *reinterpret_cast<const float4*>(c + (size_t)t * ldc + goff + fs + j);
    const float gv[4] = {g.x, g.y, g.z, g.w}, uv[4] = {u.x, u.y, u.z, u.w};
    __nv_bfloat16 r[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) r[q] = __float2bfloat16_rn(gv[q] / (1.f + expf(-gv[q])) * uv[q]);
    *reinterpret_cast<uint2*>(h + (size_t)t * fs + j) =
        make_uint2((uint32_t)__bfloat16_as_ushort(r[0]) | ((uint32_t)__bfloat16_as_ushort(r[1]) << 16),
                   (uint32_t)__bfloat16_as_ushort(r[2]) | ((uint32_t)__bfloat16_as_ushort(r[3]) << 16));
  }
}

}  // namespace

cudaError_t launch_dense_in(const ds4moe_layer* L, const void* x, int T, cudaStream_t st) {
  cublasHandle_t h = static_cast<cublasHandle_t>(L->blas);
  if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  const float one = 1.f, zero = 0.f;
  // column-major view: C^T (N x T) = Wcat (N x d, stored as d x N) ^T . x^T (d x T)
  const cublasStatus_t s = cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, L->dense_n, T, L->cfg.d_model, &one, L->wcat,
                                        CUDA_R_16BF, L->cfg.d_model, x, CUDA_R_16BF, L->cfg.d_model, &zero, L->s.dense_c,
                                        CUDA_R_32F, L->dense_n, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  return s == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

cudaError_t launch_shared_swiglu(const ds4moe_layer* L, int T, cudaStream_t st) {
  const int fs = L->cfg.d_ff_shared;
  const int n = T * (fs / 4);
  const int blocks = (n + 255) / 256 < 4 * L->num_sms ? (n + 255) / 256 : 4 * L->num_sms;
  return launch_pdl(shared_swiglu_kernel, dim3((unsigned)blocks), dim3(256), 0, st, (const float*)L->s.dense_c,
                    L->dense_n, L->dense_goff, fs, T, L->s.h_shared);
}

cudaError_t launch_shared_down(const ds4moe_layer* L, float* out, int T, cudaStream_t st) {
  cublasHandle_t h = static_cast<cublasHandle_t>(L->blas);
  if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  const float one = 1.f;
  const int d = L->cfg.d_model, fs = L->cfg.d_ff_shared;
  // out^T (d x T) += Wd (d x fs, stored as fs x d) ^T . h^T (fs x T)
  const cublasStatus_t s = cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, d, T, fs, &one, L->wsd, CUDA_R_16BF, fs,
                                        L->s.h_shared, CUDA_R_16BF, fs, &one, out, CUDA_R_32F, d, CUBLAS_COMPUTE_32F,
                                        CUBLAS_GEMM_DEFAULT);
  return s == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

cudaError_t dense_create(ds4moe_layer* L, size_t workspace_bytes, void* workspace) {
  cublasHandle_t h = nullptr;
  if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  L->blas = h;
  // a library-owned workspace, so that a forward call never allocates
  if (cublasSetWorkspace(h, workspace, workspace_bytes) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  return cudaSuccess;
}

void dense_destroy(ds4moe_layer* L) {
  if (L->blas) cublasDestroy(static_cast<cublasHandle_t>(L->blas));
  L->blas = nullptr;
}

}  // namespace ds4moe
