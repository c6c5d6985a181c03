// W4A16 fallback: the weights' MXFP4 values expanded to bf16 and one plain
// bf16 matrix multiplication (page "Huawei MACaQ: Choosing GGUF or vLLM and
// Avoiding Setup Mistakes", section "vLLM checkpoints have different
// constraints": the documented weight-only fallback expands weights for a
// BF16 matmul and is slower than W4A4).  The activation transform and the
// weight expansion are this library's kernels (quant.cu); the GEMM itself is
// a plain library bf16 GEMM (cuBLASLt, fp32 accumulation) whose plan is
// chosen once per shape and cached.
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"

namespace macaq {

namespace {

struct LtPlan {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
    cublasLtMatmulAlgo_t algo{};
    bool ok = false;
};

// key: device, M, N, K, ldx, ldy, workspace cap
using PlanKey = std::tuple<int, int64_t, int64_t, int64_t, int64_t, int64_t, size_t>;

std::mutex g_lt_mu;
cublasLtHandle_t g_lt[64] = {};
std::map<PlanKey, LtPlan> g_plans;

void destroy(LtPlan &p)
{
    if (p.c) cublasLtMatrixLayoutDestroy(p.c);
    if (p.b) cublasLtMatrixLayoutDestroy(p.b);
    if (p.a) cublasLtMatrixLayoutDestroy(p.a);
    if (p.op) cublasLtMatmulDescDestroy(p.op);
    p = LtPlan{};
}

// Y[M, N] (row-major, pitch ldy) = Xt[M, K] (pitch ldx) . Wd[N, K]^T.  In
// cuBLASLt's column-major terms: D (N x M, ld ldy) = A^T . B with A = Wd
// viewed as K x N (ld K) and B = Xt viewed as K x M (ld ldx).
bool make_plan(cublasLtHandle_t h, int64_t M, int64_t N, int64_t K, int64_t ldx, int64_t ldy,
               size_t ws_cap, LtPlan &p)
{
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    if (cublasLtMatmulDescCreate(&p.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) return false;
    if (cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) != CUBLAS_STATUS_SUCCESS)
        return false;
    if (cublasLtMatrixLayoutCreate(&p.a, CUDA_R_16BF, K, N, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&p.b, CUDA_R_16BF, K, M, ldx) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&p.c, CUDA_R_16BF, N, M, ldy) != CUBLAS_STATUS_SUCCESS)
        return false;
    cublasLtMatmulPreference_t pref = nullptr;
    if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) return false;
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_cap, sizeof(ws_cap));
    cublasLtMatmulHeuristicResult_t res{};
    int found = 0;
    const cublasStatus_t st = cublasLtMatmulAlgoGetHeuristic(h, p.op, p.a, p.b, p.c, p.c, pref, 1, &res, &found);
    cublasLtMatmulPreferenceDestroy(pref);
    if (st != CUBLAS_STATUS_SUCCESS || found < 1 || res.workspaceSize > ws_cap) return false;
    p.algo = res.algo;
    p.ok = true;
    return true;
}

}  // namespace

cudaError_t launch_bf16_gemm_nt(const uint16_t *Xt, int64_t ldx, const uint16_t *Wd, int64_t M, int64_t N,
                                int64_t K, uint16_t *Y, int64_t ldy, void *ws, size_t ws_bytes,
                                cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cublasLtHandle_t h;
    LtPlan plan;
    {
        std::lock_guard<std::mutex> lock(g_lt_mu);
        if (!g_lt[dev] && cublasLtCreate(&g_lt[dev]) != CUBLAS_STATUS_SUCCESS) {
            g_lt[dev] = nullptr;
            return cudaErrorUnknown;
        }
        h = g_lt[dev];
        const PlanKey key{dev, M, N, K, ldx, ldy, ws_bytes};
        auto it = g_plans.find(key);
        if (it == g_plans.end()) {
            LtPlan p;
            if (!make_plan(h, M, N, K, ldx, ldy, ws_bytes, p)) {
                destroy(p);
                return cudaErrorNotSupported;
            }
            it = g_plans.emplace(key, p).first;
        }
        plan = it->second;
    }
    const float alpha = 1.0f, beta = 0.0f;
    const cublasStatus_t st = cublasLtMatmul(h, plan.op, &alpha, Wd, plan.a, Xt, plan.b, &beta, Y, plan.c, Y,
                                             plan.c, &plan.algo, ws, ws_bytes, stream);
    return st == CUBLAS_STATUS_SUCCESS ? cudaGetLastError() : cudaErrorUnknown;
}

}  // namespace macaq
