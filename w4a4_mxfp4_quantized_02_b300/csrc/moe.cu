// MoE combine: each token's output is the weighted sum of its top-k expert
// rows (the rows the grouped down-projection GEMM wrote in expert-sorted
// order).  out[t, n] = bf16( fp32 fused multiply-add chain over k = 0 ..
// topk-1 of w[t, k] * Y[rows[t, k], n], from +0 ); the order of the choices
// is the caller's, so the result does not depend on the launch.  The pages
// run the routed experts' projections in W4A4 (page "Huawei MACaQ Is an
// Open-Source Model Quantizer", section "MACaQ Backends") and state no
// combine arithmetic; this is the plain reading.
//
// One thread per token and 8 output columns: topk independent 16-byte row
// loads (coalesced along the row across a warp), 8 accumulators, one 16-byte
// store.  Bound by HBM: every expert row is read once, every token row
// written once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace macaq {

namespace {

// kTopk > 0: the choice count fixed at compile time, all rows loaded before
// the chain (kTopk loads in flight per thread); 0: any count, in a loop.
template <int kTopk>
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint16_t *Y, int64_t ldy, int64_t y_rows,
                                                           const int32_t *rows, const float *w, int64_t T,
                                                           int32_t topk, int64_t N, uint16_t *out, int64_t ldo)
{
    const int64_t n8 = N / 8;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (idx >= T * n8) return;
    const int64_t t = idx / n8, c = idx - (idx / n8) * n8;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    auto accumulate = [&](float wk, const uint4 &v) {
        const uint32_t word[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc[2 * j] = __fmaf_rn(wk, __uint_as_float(word[j] << 16), acc[2 * j]);
            acc[2 * j + 1] = __fmaf_rn(wk, __uint_as_float(word[j] & 0xffff0000u), acc[2 * j + 1]);
        }
    };
    if (kTopk > 0) {
        uint4 v[kTopk > 0 ? kTopk : 1];
        bool ok[kTopk > 0 ? kTopk : 1];
#pragma unroll
        for (int k = 0; k < kTopk; ++k) {
            const int64_t r = rows[t * kTopk + k];
            ok[k] = r >= 0 && r < y_rows;  // outside the expert rows: contributes nothing
            if (ok[k]) v[k] = *reinterpret_cast<const uint4 *>(Y + r * ldy + 8 * c);
        }
#pragma unroll
        for (int k = 0; k < kTopk; ++k)
            if (ok[k]) accumulate(w[t * kTopk + k], v[k]);
    } else {
#pragma unroll 4
        for (int32_t k = 0; k < topk; ++k) {
            const int64_t r = rows[t * topk + k];
            if (r < 0 || r >= y_rows) continue;  // outside the expert rows: contributes nothing
            accumulate(w[t * topk + k], *reinterpret_cast<const uint4 *>(Y + r * ldy + 8 * c));
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
        o[j] = *reinterpret_cast<const uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(out + t * ldo + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_moe_combine(const uint16_t *Y, int64_t ldy, int64_t y_rows, const int32_t *rows,
                               const float *w, int64_t T, int64_t topk, int64_t N, uint16_t *out, int64_t ldo,
                               cudaStream_t stream)
{
    const int64_t n = T * (N / 8);
    const int64_t blocks = (n + 255) / 256;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kern = topk == 8 ? moe_combine_kernel<8> : topk == 4 ? moe_combine_kernel<4>
                                   : topk == 2 ? moe_combine_kernel<2> : moe_combine_kernel<0>;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, Y, ldy, y_rows, rows, w, T, static_cast<int32_t>(topk), N,
                                         out, ldo);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// ------------------------------------------------ gate/up row interleave
//
// Weight preparation for the fused gate+up epilogue: W_gu [E, 2F, K] (gate
// rows 0 .. F-1, up rows F .. 2F-1 of each expert) -> W_out [E, 2F, K] with
// output row 128c + j = gate row 64c + j and output row 128c + 64 + j = up
// row 64c + j (j < 64), so that every 128 output rows hold gate and up of the
// same 64 channels.  A row copy per warp (16-byte loads and stores).
namespace {

__global__ void __launch_bounds__(256) interleave_gate_up_kernel(const uint4 *w, int64_t E, int64_t F,
                                                                 int64_t k16, uint4 *out)
{
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= E * 2 * F) return;
    const int64_t e = row / (2 * F), n = row - e * 2 * F;
    const int64_t c = n >> 7, j = n & 127;
    const int64_t src = (j < 64) ? 64 * c + j : F + 64 * c + (j - 64);
    const uint4 *s = w + (e * 2 * F + src) * k16;
    uint4 *d = out + row * k16;
    for (int64_t i = threadIdx.x & 31; i < k16; i += 32) d[i] = s[i];
}

}  // namespace

cudaError_t launch_interleave_gate_up(const uint16_t *w, int64_t E, int64_t F, int64_t K, uint16_t *out,
                                      cudaStream_t stream)
{
    const int64_t rows = E * 2 * F;
    interleave_gate_up_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(w), E, F, K / 8, reinterpret_cast<uint4 *>(out));
    return cudaGetLastError();
}

}  // namespace macaq
