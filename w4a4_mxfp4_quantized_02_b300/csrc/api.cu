// C ABI of the MACaQ W4A4 library: argument checks, then launches.  Every
// check runs on the host before anything is enqueued; nothing here allocates,
// frees or synchronises (except the two documented error helpers).
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "macaq.h"

using namespace macaq;

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1024;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

macaq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MACAQ_OK : MACAQ_ERR_CUDA; }

macaq_status check_k(int64_t K)
{
    if (K <= 0 || K % 32 != 0) return MACAQ_ERR_INVALID_ARG;
    if (K > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    return MACAQ_OK;
}

macaq_status check_rows(int64_t rows)
{
    if (rows < 0) return MACAQ_ERR_INVALID_ARG;
    if (rows > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    return MACAQ_OK;
}

#define MACAQ_TRY(expr)                       \
    do {                                      \
        macaq_status s__ = (expr);            \
        if (s__ != MACAQ_OK) return s__;      \
    } while (0)

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// scratch the W4A16 bf16 GEMM may use (part of its workspace)

}  // namespace

extern "C" {

const char *macaq_status_string(macaq_status s)
{
    switch (s) {
    case MACAQ_OK: return "ok";
    case MACAQ_ERR_INVALID_ARG: return "invalid argument";
    case MACAQ_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case MACAQ_ERR_UNSUPPORTED: return "unsupported size";
    case MACAQ_ERR_WORKSPACE: return "workspace missing or too small";
    case MACAQ_ERR_CUDA: return "CUDA error";
    case MACAQ_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

size_t macaq_scale_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K <= 0 || K % 32 != 0) return 0;
    return tiled_scale_bytes(rows, K);
}

int64_t macaq_grouped_padded_rows(int64_t rows, int64_t E)
{
    if (rows < 0 || E <= 0) return 0;
    return grouped_padded_rows(rows, E);
}

macaq_status macaq_balance_scales(const void *Xc, int64_t ldxc, const int32_t *xc_rows, int64_t Mc,
                                  const void *W, int64_t N, int64_t K, float *s, float *inv_s,
                                  macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(Mc));
    MACAQ_TRY(check_rows(N));
    if (!s || !inv_s || (Mc > 0 && !Xc) || (N > 0 && !W)) return MACAQ_ERR_INVALID_ARG;
    if (Mc > 0 && ldxc < K) return MACAQ_ERR_INVALID_ARG;
    if ((Xc && !aligned16(Xc)) || (W && !aligned16(W)) || !aligned16(s) || !aligned16(inv_s) ||
        (Mc > 0 && ldxc % 8 != 0))
        return MACAQ_ERR_ALIGNMENT;
    return from_cuda(launch_balance(static_cast<const uint16_t *>(Xc), ldxc, xc_rows, Mc,
                                    static_cast<const uint16_t *>(W), N, K, s, inv_s,
                                    static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_quant_act_hb(const void *X, int64_t ldx, const float *inv_s, int64_t M, int64_t K,
                                int64_t hadamard_block, uint8_t *a_codes, uint8_t *a_scales,
                                macaq_stream_t stream)
{
    if (hadamard_block != 32 && hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_k(K));
    if (K % hadamard_block != 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_rows(M));
    if (M == 0) return MACAQ_OK;
    if (!X || !inv_s || !a_codes || !a_scales || ldx < K) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(inv_s) || !aligned16(a_codes) || !aligned16(a_scales) ||
        ldx % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(X);
    a.ld_src = ldx;
    a.f = inv_s;
    a.K = K;
    a.rows_valid = M;
    a.rows_out = pad_rows(M);
    a.E = 1;
    a.codes = a_codes;
    a.scales = a_scales;
    a.had = static_cast<int32_t>(hadamard_block);
    return from_cuda(launch_quant(QuantMode::Dense, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_quant_weight_hb(const void *W, const float *s, int64_t N, int64_t K,
                                   int64_t hadamard_block, uint8_t *w_codes, uint8_t *w_scales,
                                   macaq_stream_t stream)
{
    return macaq_quant_act_hb(W, K, s, N, K, hadamard_block, w_codes, w_scales, stream);
}

macaq_status macaq_quant_act(const void *X, int64_t ldx, const float *inv_s, int64_t M, int64_t K,
                             uint8_t *a_codes, uint8_t *a_scales, macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(M));
    if (M == 0) return MACAQ_OK;
    if (!X || !inv_s || !a_codes || !a_scales || ldx < K) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(inv_s) || !aligned16(a_codes) || !aligned16(a_scales) ||
        ldx % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(X);
    a.ld_src = ldx;
    a.f = inv_s;
    a.K = K;
    a.rows_valid = M;
    a.rows_out = pad_rows(M);
    a.E = 1;
    a.codes = a_codes;
    a.scales = a_scales;
    return from_cuda(launch_quant(QuantMode::Dense, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_quant_weight(const void *W, const float *s, int64_t N, int64_t K,
                                uint8_t *w_codes, uint8_t *w_scales, macaq_stream_t stream)
{
    return macaq_quant_act(W, K, s, N, K, w_codes, w_scales, stream);
}

macaq_status macaq_quant_weight_grouped(const void *W, const float *s, int64_t E, int64_t N,
                                        int64_t K, uint8_t *w_codes, uint8_t *w_scales,
                                        macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(N));
    if (E < 0) return MACAQ_ERR_INVALID_ARG;
    if (E == 0 || N == 0) return MACAQ_OK;
    if (E * pad_rows(N) > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    if (!W || !s || !w_codes || !w_scales) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(s) || !aligned16(w_codes) || !aligned16(w_scales))
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(W);
    a.ld_src = K;
    a.f = s;
    a.K = K;
    a.rows_valid = N;
    a.group_rows_pad = pad_rows(N);
    a.rows_out = E * pad_rows(N);
    a.E = static_cast<int32_t>(E);
    a.codes = w_codes;
    a.scales = w_scales;
    a.scale_group_stride = tiled_scale_bytes(N, K);
    return from_cuda(launch_quant(QuantMode::WeightGrouped, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_quant_weight_grouped_hb(const void *W, const float *s, int64_t E, int64_t N, int64_t K,
                                           int64_t hadamard_block, uint8_t *w_codes, uint8_t *w_scales,
                                           macaq_stream_t stream)
{
    if (hadamard_block == 32) return macaq_quant_weight_grouped(W, s, E, N, K, w_codes, w_scales, stream);
    if (hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_k(K));
    if (K % 64 != 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_rows(N));
    if (E < 0) return MACAQ_ERR_INVALID_ARG;
    if (E == 0 || N == 0) return MACAQ_OK;
    if (E * pad_rows(N) > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    if (!W || !s || !w_codes || !w_scales) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(s) || !aligned16(w_codes) || !aligned16(w_scales)) return MACAQ_ERR_ALIGNMENT;
    // expert by expert through the dense transform (offline preparation)
    const size_t sbytes = tiled_scale_bytes(N, K);
    for (int64_t e = 0; e < E; ++e) {
        const uint16_t *We = static_cast<const uint16_t *>(W) + e * N * K;
        MACAQ_TRY(macaq_quant_weight_hb(We, s + e * K, N, K, 64, w_codes + e * N * (K / 2), w_scales + e * sbytes,
                                        stream));
    }
    return MACAQ_OK;
}

namespace {
macaq_status w4a4_gemm(const uint8_t *a_codes, const uint8_t *a_scales, const uint8_t *w_codes,
                       const uint8_t *w_scales, int64_t M, int64_t N, int64_t K, void *Y, int64_t ldy,
                       bool weight_early, macaq_stream_t stream);
}  // namespace

macaq_status macaq_w4a4_gemm(const uint8_t *a_codes, const uint8_t *a_scales,
                             const uint8_t *w_codes, const uint8_t *w_scales, int64_t M, int64_t N,
                             int64_t K, void *Y, int64_t ldy, macaq_stream_t stream)
{
    return w4a4_gemm(a_codes, a_scales, w_codes, w_scales, M, N, K, Y, ldy, false, stream);
}

namespace {
macaq_status w4a4_gemm(const uint8_t *a_codes, const uint8_t *a_scales, const uint8_t *w_codes,
                       const uint8_t *w_scales, int64_t M, int64_t N, int64_t K, void *Y, int64_t ldy,
                       bool weight_early, macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(M));
    MACAQ_TRY(check_rows(N));
    if (M == 0 || N == 0) return MACAQ_OK;
    if (!a_codes || !a_scales || !w_codes || !w_scales || !Y || ldy < N) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) || !aligned16(w_scales) ||
        !aligned16(Y) || ldy % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    GemmArgs g{};
    g.a_codes = a_codes;
    g.a_scales = a_scales;
    g.w_codes = w_codes;
    g.w_scales = w_scales;
    g.M = M;
    g.a_rows = M;
    g.N = N;
    g.K = K;
    g.E = 0;
    g.Y = Y;
    g.ldy = ldy;
    g.weight_early = weight_early;
    return from_cuda(launch_gemm(g, static_cast<cudaStream_t>(stream)));
}
}  // namespace

size_t macaq_linear_workspace_bytes(int64_t M, int64_t K)
{
    if (M < 0 || K <= 0 || K % 32 != 0) return 0;
    return align256(static_cast<size_t>(M) * static_cast<size_t>(K / 2)) + tiled_scale_bytes(M, K);
}

macaq_status macaq_linear(const void *X, int64_t ldx, const float *inv_s, const uint8_t *w_codes,
                          const uint8_t *w_scales, int64_t M, int64_t N, int64_t K, void *Y,
                          int64_t ldy, void *workspace, size_t ws_bytes, macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(M));
    MACAQ_TRY(check_rows(N));
    if (M == 0 || N == 0) return MACAQ_OK;
    if (!X || !inv_s || !w_codes || !w_scales || !Y || ldx < K || ldy < N) return MACAQ_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < macaq_linear_workspace_bytes(M, K)) return MACAQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MACAQ_ERR_ALIGNMENT;
    if (M <= kFusedLinearMaxRows) {
        // a few token rows (decode): one launch, the transform inside the GEMM
        // (the same checks as the two calls below make)
        if (!aligned16(X) || !aligned16(inv_s) || ldx % 8 != 0 || !aligned16(w_codes) ||
            !aligned16(w_scales) || !aligned16(Y) || ldy % 8 != 0)
            return MACAQ_ERR_ALIGNMENT;
        GemmArgs g{};
        g.w_codes = w_codes;
        g.w_scales = w_scales;
        g.M = M;
        g.a_rows = M;
        g.N = N;
        g.K = K;
        g.E = 0;
        g.Y = Y;
        g.ldy = ldy;
        return from_cuda(launch_linear_fused(g, static_cast<const uint16_t *>(X), ldx, inv_s,
                                             static_cast<cudaStream_t>(stream)));
    }
    uint8_t *a_codes = static_cast<uint8_t *>(workspace);
    uint8_t *a_scales = a_codes + align256(static_cast<size_t>(M) * static_cast<size_t>(K / 2));
    MACAQ_TRY(macaq_quant_act(X, ldx, inv_s, M, K, a_codes, a_scales, stream));
    // the GEMM follows its own transform, which lets it start only after
    // everything before the layer has completed: its weight may load early
    return w4a4_gemm(a_codes, a_scales, w_codes, w_scales, M, N, K, Y, ldy, true, stream);
}

macaq_status macaq_transform_act_bf16(const void *X, int64_t ldx, const float *inv_s, int64_t M,
                                      int64_t K, int64_t hadamard_block, void *Xt, int64_t ldxt,
                                      macaq_stream_t stream)
{
    if (hadamard_block != 32 && hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_k(K));
    if (K % hadamard_block != 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_rows(M));
    if (M == 0) return MACAQ_OK;
    if (!X || !inv_s || !Xt || ldx < K || ldxt < K) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(inv_s) || !aligned16(Xt) || ldx % 8 != 0 || ldxt % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(X);
    a.ld_src = ldx;
    a.f = inv_s;
    a.K = K;
    a.rows_valid = M;
    a.rows_out = M;
    a.E = 1;
    a.codes = static_cast<uint8_t *>(Xt);
    a.scales = nullptr;
    a.had = static_cast<int32_t>(hadamard_block);
    a.out_kind = kOutBf16;
    a.ld_out = ldxt;
    return from_cuda(launch_quant(QuantMode::Dense, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_dequant_weight_bf16(const uint8_t *w_codes, const uint8_t *w_scales, int64_t N,
                                       int64_t K, void *Wd, macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(N));
    if (N == 0) return MACAQ_OK;
    if (!w_codes || !w_scales || !Wd) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(w_codes) || !aligned16(w_scales) || !aligned16(Wd)) return MACAQ_ERR_ALIGNMENT;
    return from_cuda(launch_dequant_bf16(w_codes, w_scales, N, K, static_cast<uint16_t *>(Wd),
                                         static_cast<cudaStream_t>(stream)));
}

size_t macaq_w4a16_linear_workspace_bytes(int64_t M, int64_t K)
{
    if (M < 0 || K <= 0 || K % 32 != 0) return 0;
    return align256(static_cast<size_t>(M) * static_cast<size_t>(K) * 2);
}

macaq_status macaq_w4a16_gemm(const void *Xt, int64_t ldxt, const uint8_t *w_codes, const uint8_t *w_scales,
                              int64_t M, int64_t N, int64_t K, void *Y, int64_t ldy, macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(M));
    MACAQ_TRY(check_rows(N));
    if (M == 0 || N == 0) return MACAQ_OK;
    if (!Xt || !w_codes || !w_scales || !Y || ldxt < K || ldy < N) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(Xt) || !aligned16(w_codes) || !aligned16(w_scales) || !aligned16(Y) || ldxt % 8 != 0 ||
        ldy % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    W4A16Args g{};
    g.Xt = Xt;
    g.ldx = ldxt;
    g.w_codes = w_codes;
    g.w_scales = w_scales;
    g.M = M;
    g.N = N;
    g.K = K;
    g.Y = Y;
    g.ldy = ldy;
    return from_cuda(launch_w4a16_gemm(g, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_w4a16_linear(const void *X, int64_t ldx, const float *inv_s, const uint8_t *w_codes,
                                const uint8_t *w_scales, int64_t M, int64_t N, int64_t K, int64_t hadamard_block,
                                void *Y, int64_t ldy, void *workspace, size_t ws_bytes, macaq_stream_t stream)
{
    if (hadamard_block != 32 && hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_k(K));
    if (K % hadamard_block != 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_rows(M));
    MACAQ_TRY(check_rows(N));
    if (M == 0 || N == 0) return MACAQ_OK;
    if (!X || !inv_s || !w_codes || !w_scales || !Y || ldx < K || ldy < N) return MACAQ_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < macaq_w4a16_linear_workspace_bytes(M, K)) return MACAQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MACAQ_ERR_ALIGNMENT;
    if (!aligned16(X) || !aligned16(w_codes) || !aligned16(w_scales) || !aligned16(Y) || ldx % 8 != 0 ||
        ldy % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    uint8_t *xt = static_cast<uint8_t *>(workspace);
    MACAQ_TRY(macaq_transform_act_bf16(X, ldx, inv_s, M, K, hadamard_block, xt, K, stream));
    return macaq_w4a16_gemm(xt, K, w_codes, w_scales, M, N, K, Y, ldy, stream);
}

macaq_status macaq_transform_f32(const void *X, int64_t ldx, const float *f, int64_t M, int64_t K,
                                 int64_t hadamard_block, float *Y, int64_t ldy, macaq_stream_t stream)
{
    if (hadamard_block != 32 && hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_k(K));
    if (K % hadamard_block != 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_rows(M));
    if (M == 0) return MACAQ_OK;
    if (!X || !f || !Y || ldx < K || ldy < K) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(f) || !aligned16(Y) || ldx % 8 != 0 || ldy % 4 != 0)
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(X);
    a.ld_src = ldx;
    a.f = f;
    a.K = K;
    a.rows_valid = M;
    a.rows_out = M;
    a.E = 1;
    a.codes = reinterpret_cast<uint8_t *>(Y);
    a.scales = nullptr;
    a.had = static_cast<int32_t>(hadamard_block);
    a.out_kind = kOutF32;
    a.ld_out = ldy;
    return from_cuda(launch_quant(QuantMode::Dense, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_flip_hessian(const float *A, int64_t Mc, int64_t K, float damp, float *H,
                                macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(Mc));
    if (!H || (Mc > 0 && !A)) return MACAQ_ERR_INVALID_ARG;
    if ((A && !aligned16(A)) || !aligned16(H)) return MACAQ_ERR_ALIGNMENT;
    return from_cuda(launch_flip_hessian(A, Mc, K, damp, H, static_cast<cudaStream_t>(stream)));
}

size_t macaq_flip_refine_workspace_bytes(int64_t N, int64_t K)
{
    if (N < 0 || K <= 0 || K % 32 != 0) return 0;
    return 2 * align256(static_cast<size_t>(N) * static_cast<size_t>(K) * 4);
}

namespace {

macaq_status check_flip(const float *H, int64_t N, int64_t K, const uint8_t *w_codes, const uint8_t *w_scales,
                        void *workspace, size_t ws_bytes)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(N));
    if (flip_rows_per_cta(K) < 1) return MACAQ_ERR_UNSUPPORTED;
    if (N == 0) return MACAQ_OK;
    if (!H || !w_codes || !w_scales) return MACAQ_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < macaq_flip_refine_workspace_bytes(N, K)) return MACAQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || !aligned16(H) || !aligned16(w_codes) ||
        !aligned16(w_scales))
        return MACAQ_ERR_ALIGNMENT;
    return MACAQ_OK;
}

float *flip_g(void *workspace, int64_t N, int64_t K)
{
    return reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                     align256(static_cast<size_t>(N) * static_cast<size_t>(K) * 4));
}

}  // namespace

macaq_status macaq_flip_prepare(const float *Wt, const float *H, int64_t N, int64_t K,
                                const uint8_t *w_codes, const uint8_t *w_scales, void *workspace,
                                size_t ws_bytes, macaq_stream_t stream)
{
    MACAQ_TRY(check_flip(H, N, K, w_codes, w_scales, workspace, ws_bytes));
    if (N == 0) return MACAQ_OK;
    if (!Wt) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(Wt)) return MACAQ_ERR_ALIGNMENT;
    return from_cuda(launch_flip_prepare(Wt, H, N, K, w_codes, w_scales, static_cast<float *>(workspace),
                                         flip_g(workspace, N, K), static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_flip_sweeps(const float *H, int64_t N, int64_t K, int32_t sweeps, uint8_t *w_codes,
                               const uint8_t *w_scales, int32_t *flips, void *workspace, size_t ws_bytes,
                               macaq_stream_t stream)
{
    if (sweeps < 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_flip(H, N, K, w_codes, w_scales, workspace, ws_bytes));
    if (N == 0) return MACAQ_OK;
    if (flips && (reinterpret_cast<uintptr_t>(flips) & 3u)) return MACAQ_ERR_ALIGNMENT;
    return from_cuda(launch_flip_sweeps(H, flip_g(workspace, N, K), N, K, sweeps, w_codes, w_scales, flips,
                                        static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_flip_refine(const float *Wt, const float *H, int64_t N, int64_t K, int32_t sweeps,
                               uint8_t *w_codes, const uint8_t *w_scales, int32_t *flips,
                               void *workspace, size_t ws_bytes, macaq_stream_t stream)
{
    if (sweeps < 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(macaq_flip_prepare(Wt, H, N, K, w_codes, w_scales, workspace, ws_bytes, stream));
    return macaq_flip_sweeps(H, N, K, sweeps, w_codes, w_scales, flips, workspace, ws_bytes, stream);
}

macaq_status macaq_quant_act_grouped_hb(const void *X, int64_t ldx, const int32_t *row_src,
                                        const int32_t *expert_offsets, const float *inv_s, int64_t rows,
                                        int64_t E, int64_t K, int64_t hadamard_block, uint8_t *a_codes,
                                        uint8_t *a_scales, macaq_stream_t stream)
{
    if (hadamard_block != 32 && hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_k(K));
    if (K % hadamard_block != 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_rows(rows));
    if (E <= 0) return MACAQ_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MACAQ_ERR_UNSUPPORTED;
    if (grouped_padded_rows(rows, E) > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    if (!expert_offsets || !inv_s || !a_codes || !a_scales) return MACAQ_ERR_INVALID_ARG;
    if (rows > 0 && (!X || !row_src || ldx < K)) return MACAQ_ERR_INVALID_ARG;
    if ((X && !aligned16(X)) || !aligned16(inv_s) || !aligned16(a_codes) || !aligned16(a_scales) ||
        (X && ldx % 8 != 0))
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(X);
    a.ld_src = ldx;
    a.row_src = row_src;
    a.offsets = expert_offsets;
    a.f = inv_s;
    a.K = K;
    a.rows_valid = rows;
    a.rows_out = grouped_padded_rows(rows, E);
    a.E = static_cast<int32_t>(E);
    a.codes = a_codes;
    a.scales = a_scales;
    a.had = static_cast<int32_t>(hadamard_block);
    return from_cuda(launch_quant(QuantMode::ActGrouped, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_quant_act_grouped(const void *X, int64_t ldx, const int32_t *row_src,
                                     const int32_t *expert_offsets, const float *inv_s,
                                     int64_t rows, int64_t E, int64_t K, uint8_t *a_codes,
                                     uint8_t *a_scales, macaq_stream_t stream)
{
    return macaq_quant_act_grouped_hb(X, ldx, row_src, expert_offsets, inv_s, rows, E, K, 32, a_codes, a_scales,
                                      stream);
}

macaq_status macaq_quant_act_grouped_silu_hb(const void *GU, int64_t ldgu, const int32_t *expert_offsets,
                                             const float *inv_s, int64_t rows, int64_t E, int64_t F,
                                             int64_t hadamard_block, uint8_t *a_codes, uint8_t *a_scales,
                                             macaq_stream_t stream)
{
    if (hadamard_block != 32 && hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_k(F));
    if (F % hadamard_block != 0) return MACAQ_ERR_INVALID_ARG;
    MACAQ_TRY(check_rows(rows));
    if (E <= 0) return MACAQ_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MACAQ_ERR_UNSUPPORTED;
    if (grouped_padded_rows(rows, E) > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    if (!expert_offsets || !inv_s || !a_codes || !a_scales) return MACAQ_ERR_INVALID_ARG;
    if (rows > 0 && (!GU || ldgu < 2 * F)) return MACAQ_ERR_INVALID_ARG;
    if ((GU && !aligned16(GU)) || !aligned16(inv_s) || !aligned16(a_codes) || !aligned16(a_scales) ||
        (GU && ldgu % 8 != 0))
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(GU);
    a.ld_src = ldgu;
    a.row_src = nullptr;
    a.offsets = expert_offsets;
    a.f = inv_s;
    a.K = F;
    a.rows_valid = rows;
    a.rows_out = grouped_padded_rows(rows, E);
    a.E = static_cast<int32_t>(E);
    a.codes = a_codes;
    a.scales = a_scales;
    a.had = static_cast<int32_t>(hadamard_block);
    return from_cuda(launch_quant(QuantMode::ActGroupedSilu, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_quant_act_grouped_silu(const void *GU, int64_t ldgu, const int32_t *expert_offsets,
                                          const float *inv_s, int64_t rows, int64_t E, int64_t F,
                                          uint8_t *a_codes, uint8_t *a_scales, macaq_stream_t stream)
{
    return macaq_quant_act_grouped_silu_hb(GU, ldgu, expert_offsets, inv_s, rows, E, F, 32, a_codes, a_scales,
                                           stream);
}

macaq_status macaq_quant_act_silu(const void *GU, int64_t ldgu, const float *inv_s, int64_t M, int64_t F,
                                  uint8_t *a_codes, uint8_t *a_scales, macaq_stream_t stream)
{
    MACAQ_TRY(check_k(F));
    MACAQ_TRY(check_rows(M));
    if (M == 0) return MACAQ_OK;
    if (!GU || !inv_s || !a_codes || !a_scales || ldgu < 2 * F) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(GU) || !aligned16(inv_s) || !aligned16(a_codes) || !aligned16(a_scales) || ldgu % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    QuantArgs a{};
    a.src = static_cast<const uint16_t *>(GU);
    a.ld_src = ldgu;
    a.row_src = nullptr;
    a.offsets = nullptr;  // one group: all M rows
    a.f = inv_s;
    a.K = F;
    a.rows_valid = M;
    a.rows_out = pad_rows(M);
    a.E = 1;
    a.codes = a_codes;
    a.scales = a_scales;
    return from_cuda(launch_quant(QuantMode::ActGroupedSilu, a, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_grouped_w4a4_gemm(const uint8_t *a_codes, const uint8_t *a_scales,
                                     const uint8_t *w_codes, const uint8_t *w_scales,
                                     const int32_t *expert_offsets, int64_t rows, int64_t E,
                                     int64_t N, int64_t K, void *Y, int64_t ldy,
                                     macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(rows));
    MACAQ_TRY(check_rows(N));
    if (E <= 0) return MACAQ_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MACAQ_ERR_UNSUPPORTED;
    if (grouped_padded_rows(rows, E) > kMaxDim || E * N > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    if (rows == 0 || N == 0) return MACAQ_OK;
    if (!a_codes || !a_scales || !w_codes || !w_scales || !expert_offsets || !Y || ldy < N)
        return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) || !aligned16(w_scales) ||
        !aligned16(Y) || ldy % 8 != 0)
        return MACAQ_ERR_ALIGNMENT;
    GemmArgs g{};
    g.a_codes = a_codes;
    g.a_scales = a_scales;
    g.w_codes = w_codes;
    g.w_scales = w_scales;
    g.offsets = expert_offsets;
    g.M = rows;
    g.a_rows = grouped_padded_rows(rows, E);
    g.N = N;
    g.K = K;
    g.E = static_cast<int32_t>(E);
    g.Y = Y;
    g.ldy = ldy;
    return from_cuda(launch_gemm(g, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_interleave_gate_up(const void *W_gu, int64_t E, int64_t F, int64_t K, void *W_out,
                                      macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(F));
    if (E < 0 || F % 64 != 0) return MACAQ_ERR_INVALID_ARG;
    if (E == 0 || F == 0) return MACAQ_OK;
    if (E * 2 * F > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    if (!W_gu || !W_out || W_gu == W_out) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(W_gu) || !aligned16(W_out)) return MACAQ_ERR_ALIGNMENT;
    return from_cuda(launch_interleave_gate_up(static_cast<const uint16_t *>(W_gu), E, F, K,
                                               static_cast<uint16_t *>(W_out), static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_grouped_w4a4_gemm_swiglu(const uint8_t *a_codes, const uint8_t *a_scales,
                                            const uint8_t *w_codes, const uint8_t *w_scales,
                                            const int32_t *expert_offsets, int64_t rows, int64_t E, int64_t F,
                                            int64_t K, const float *inv_s, int64_t hadamard_block,
                                            uint8_t *h_codes, uint8_t *h_scales, macaq_stream_t stream)
{
    MACAQ_TRY(check_k(K));
    MACAQ_TRY(check_rows(rows));
    MACAQ_TRY(check_rows(F));
    if (hadamard_block != 32 && hadamard_block != 64) return MACAQ_ERR_INVALID_ARG;
    if (E <= 0 || F % 64 != 0) return MACAQ_ERR_INVALID_ARG;
    if (E > kMaxExperts) return MACAQ_ERR_UNSUPPORTED;
    if (grouped_padded_rows(rows, E) > kMaxDim || E * 2 * F > kMaxDim) return MACAQ_ERR_UNSUPPORTED;
    if (rows == 0 || F == 0) return MACAQ_OK;
    if (!a_codes || !a_scales || !w_codes || !w_scales || !expert_offsets || !inv_s || !h_codes || !h_scales)
        return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) || !aligned16(w_scales) ||
        !aligned16(inv_s) || !aligned16(h_codes) || !aligned16(h_scales))
        return MACAQ_ERR_ALIGNMENT;
    GemmArgs g{};
    g.a_codes = a_codes;
    g.a_scales = a_scales;
    g.w_codes = w_codes;
    g.w_scales = w_scales;
    g.offsets = expert_offsets;
    g.M = rows;
    g.a_rows = grouped_padded_rows(rows, E);
    g.N = 2 * F;
    g.K = K;
    g.E = static_cast<int32_t>(E);
    g.Y = nullptr;
    g.ldy = 0;
    g.epi = hadamard_block == 64 ? 2 : 1;
    g.h_codes = h_codes;
    g.h_scales = h_scales;
    g.h_f = inv_s;
    return from_cuda(launch_gemm(g, static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_moe_combine(const void *Y, int64_t ldy, int64_t y_rows, const int32_t *tok_rows,
                               const float *tok_weights, int64_t T, int64_t topk, int64_t N, void *out,
                               int64_t ldo, macaq_stream_t stream)
{
    MACAQ_TRY(check_rows(T));
    MACAQ_TRY(check_rows(N));
    MACAQ_TRY(check_rows(y_rows));
    if (topk <= 0 || topk > 1024 || N % 8 != 0) return MACAQ_ERR_INVALID_ARG;
    if (T == 0 || N == 0) return MACAQ_OK;
    if (!Y || !tok_rows || !tok_weights || !out || ldy < N || ldo < N) return MACAQ_ERR_INVALID_ARG;
    if (!aligned16(Y) || !aligned16(out) || ldy % 8 != 0 || ldo % 8 != 0 ||
        (reinterpret_cast<uintptr_t>(tok_rows) & 3u) || (reinterpret_cast<uintptr_t>(tok_weights) & 3u))
        return MACAQ_ERR_ALIGNMENT;
    return from_cuda(launch_moe_combine(static_cast<const uint16_t *>(Y), ldy, y_rows, tok_rows, tok_weights, T,
                                        topk, N, static_cast<uint16_t *>(out), ldo,
                                        static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_check_device_error(macaq_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return MACAQ_ERR_CUDA;
    unsigned flags = 0, qflags = 0, fflags = 0;
    if (read_and_clear_device_error(&flags) != cudaSuccess) return MACAQ_ERR_CUDA;
    if (read_and_clear_quant_error(&qflags) != cudaSuccess) return MACAQ_ERR_CUDA;
    if (read_and_clear_flip_error(&fflags) != cudaSuccess) return MACAQ_ERR_CUDA;
    return (flags | qflags | fflags) ? MACAQ_ERR_TIMEOUT : MACAQ_OK;
}

macaq_status macaq_set_wait_timeout_ns(uint64_t ns)
{
    return from_cuda(set_wait_timeout_ns(ns));
}

macaq_status macaq_debug_wait_probe(macaq_stream_t stream)
{
    return from_cuda(launch_wait_probe(static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_debug_mma_rate(int32_t bn, int32_t iters, int32_t ctas, const void *src,
                                  uint64_t *out, macaq_stream_t stream)
{
    const int32_t n = bn & 0xffff, mode = bn >> 16;
    if (n < 16 || n > 256 || n % 16 != 0 || mode < 0 || mode > 3 || iters <= 0 || ctas <= 0 || !out)
        return MACAQ_ERR_INVALID_ARG;
    if (mode == 3 && (!src || !aligned16(src))) return MACAQ_ERR_INVALID_ARG;
    return from_cuda(launch_mma_rate(bn, iters, reinterpret_cast<unsigned long long *>(out),
                                     static_cast<const uint8_t *>(src), ctas,
                                     static_cast<cudaStream_t>(stream)));
}

macaq_status macaq_debug_e2m1(const float *t, int64_t n, uint8_t *codes, macaq_stream_t stream)
{
    if (n < 0) return MACAQ_ERR_INVALID_ARG;
    if (n == 0) return MACAQ_OK;
    if (!t || !codes) return MACAQ_ERR_INVALID_ARG;
    return from_cuda(launch_debug_e2m1(t, n, codes, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
