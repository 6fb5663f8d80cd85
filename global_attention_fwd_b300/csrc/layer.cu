// layer.cu -- a whole gated sliding-window attention layer from the hidden states.
//
// "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ", and the hyper.ai
// summary of arXiv 2609.13356, section "方法": GatedSWA(h) = o_proj(A_SWA(q, k, v) ⊙
// σ(g_proj(h))), with q, k, v and the gate projected in parallel from the normalised
// hidden state h, QK RMSNorm and partial RoPE on q and k.
//
//   q = h W_q, k = h W_k, v = h W_v, g = h W_g   (four GEMMs, bf16 in, fp32 accumulate,
//                                                 bf16 out: the attention's inputs)
//   a = A_SWA(q, k, v) ⊙ σ(g)                     (swa_prefill, this library's kernels)
//   y = a W_o                                     (GEMM)
//
// The projections are plain dense GEMMs and run on cuBLASLt with the caller's
// workspace; everything between them is the library's own attention path.  Row-major
// Y[M x N] = X[M x K] W[K x N] is issued as the column-major product
// Y^T = W^T X^T, so no operand is transposed or copied.
#include <cublasLt.h>

#include <cstring>
#include <mutex>

#include "zg_kernels.cuh"

namespace zg {
namespace {

cublasLtHandle_t lt_handle() {
    static std::once_flag once;
    static cublasLtHandle_t h = nullptr;
    std::call_once(once, [] {
        if (cublasLtCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
    });
    return h;
}

// Y[M x N] = X[M x K] W[K x N], all bf16 row-major, fp32 accumulation.
bool gemm_bf16(const void* X, const void* W, void* Y, long long M, long long N, long long K, void* ws, size_t ws_bytes,
               cudaStream_t s) {
    cublasLtHandle_t h = lt_handle();
    if (!h) return false;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    bool ok = cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS &&
              // column-major views: W^T is N x K (ld N), X^T is K x M (ld K), Y^T is N x M (ld N)
              cublasLtMatrixLayoutCreate(&a, CUDA_R_16BF, N, K, N) == CUBLAS_STATUS_SUCCESS &&
              cublasLtMatrixLayoutCreate(&b, CUDA_R_16BF, K, M, K) == CUBLAS_STATUS_SUCCESS &&
              cublasLtMatrixLayoutCreate(&c, CUDA_R_16BF, N, M, N) == CUBLAS_STATUS_SUCCESS &&
              cublasLtMatmulPreferenceCreate(&pref) == CUBLAS_STATUS_SUCCESS &&
              cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                                   sizeof(ws_bytes)) == CUBLAS_STATUS_SUCCESS;
    cublasLtMatmulHeuristicResult_t heur;
    int found = 0;
    if (ok) {
        std::memset(&heur, 0, sizeof(heur));
        ok = cublasLtMatmulAlgoGetHeuristic(h, op, a, b, c, c, pref, 1, &heur, &found) == CUBLAS_STATUS_SUCCESS &&
             found > 0;
    }
    if (ok) {
        const float alpha = 1.0f, beta = 0.0f;
        ok = cublasLtMatmul(h, op, &alpha, W, a, X, b, &beta, Y, c, Y, c, &heur.algo, ws, ws_bytes, s) ==
             CUBLAS_STATUS_SUCCESS;
    }
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (c) cublasLtMatrixLayoutDestroy(c);
    if (b) cublasLtMatrixLayoutDestroy(b);
    if (a) cublasLtMatrixLayoutDestroy(a);
    if (op) cublasLtMatmulDescDestroy(op);
    return ok;
}

}  // namespace

size_t layer_gemm_workspace_bytes() { return static_cast<size_t>(32) << 20; }

bool layer_gemm(const void* X, const void* W, void* Y, long long M, long long N, long long K, void* ws,
                size_t ws_bytes, cudaStream_t s) {
    return gemm_bf16(X, W, Y, M, N, K, ws, ws_bytes, s);
}

}  // namespace zg
