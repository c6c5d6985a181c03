// Declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "macaq.h"

namespace macaq {

constexpr int64_t kRowTile = 128;     // rows per scale tile / GEMM M tile
constexpr int64_t kMaxExperts = 256;  // grouped kernels keep expert offsets in shared memory

inline int64_t pad_rows(int64_t rows) { return (rows + kRowTile - 1) / kRowTile * kRowTile; }
inline int64_t pad_scale_cols(int64_t K) { return (K / 32 + 7) / 8 * 8; }
inline size_t tiled_scale_bytes(int64_t rows, int64_t K)
{
    return static_cast<size_t>(pad_rows(rows)) * static_cast<size_t>(pad_scale_cols(K));
}
inline int64_t grouped_padded_rows(int64_t rows, int64_t E)
{
    return pad_rows(rows + (kRowTile - 1) * E);
}

// ActGroupedSilu: the grouped activation transform of h = SiLU(g) * u read from
// a [rows, 2F] gate|up matrix in sorted row order (K = F).
constexpr int32_t kOutMx = 0, kOutBf16 = 1, kOutF32 = 2;

enum class QuantMode : int { Dense = 0, WeightGrouped = 1, ActGrouped = 2, ActGroupedSilu = 3 };

struct QuantArgs {
    const uint16_t *src;      // bf16 bits
    int64_t ld_src;           // row pitch of src in elements
    const int32_t *row_src;   // ActGrouped: token row of each sorted row
    const int32_t *offsets;   // ActGrouped: expert offsets [E+1]
    const float *f;           // balance factors; group g uses f + g*K
    int64_t K;
    int64_t rows_valid;       // Dense: M; WeightGrouped: N per expert; ActGrouped: sorted rows
    int64_t rows_out;         // output row positions to visit (padded space)
    int64_t group_rows_pad;   // WeightGrouped: pad_rows(N)
    int32_t E;
    uint8_t *codes;
    uint8_t *scales;
    size_t scale_group_stride;  // WeightGrouped: tiled_scale_bytes(N, K)
    int32_t had = 32;           // Hadamard block: 32, or 64 (Dense only)
    int32_t out_kind = 0;       // Dense only: kOutMx, or kOutBf16 / kOutF32 (the transform into
    int64_t ld_out = 0;         //   codes viewed as bf16 / float [rows, ld_out])
};

cudaError_t launch_quant(QuantMode mode, const QuantArgs &a, cudaStream_t stream);
cudaError_t launch_dequant_bf16(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t K,
                                uint16_t *out, cudaStream_t stream);


// Flip Refinement: H = A^T A (+ damp on the diagonal) of fp32 calibration rows
// a [m, k]; the descent over rows wt [n, k] of round-to-nearest codes (in/out)
// with tiled scales: prepare writes r = wt - q and g = r H ([n, k] fp32
// each), the sweeps read g.
int64_t flip_rows_per_cta(int64_t k);
cudaError_t launch_flip_hessian(const float *a, int64_t m, int64_t k, float damp, float *h, cudaStream_t stream);
cudaError_t launch_flip_prepare(const float *wt, const float *h, int64_t n, int64_t k, const uint8_t *codes,
                               const uint8_t *scales, float *r, float *g, cudaStream_t stream);
cudaError_t launch_flip_sweeps(const float *h, const float *g, int64_t n, int64_t k, int32_t sweeps,
                               uint8_t *codes, const uint8_t *scales, int32_t *flips, cudaStream_t stream);
cudaError_t read_and_clear_flip_error(unsigned *flags);

// MoE combine: out[t, :] = bf16(fma chain over k of w[t, k] * Y[rows[t, k], :]).
cudaError_t launch_moe_combine(const uint16_t *Y, int64_t ldy, int64_t y_rows, const int32_t *rows,
                               const float *w, int64_t T, int64_t topk, int64_t N, uint16_t *out, int64_t ldo,
                               cudaStream_t stream);

// W_gu [E, 2F, K] bf16 -> rows interleaved in chunks of 64 channels (gate
// then up), the layout the fused gate+up GEMM epilogue reads.
cudaError_t launch_interleave_gate_up(const uint16_t *w, int64_t E, int64_t F, int64_t K, uint16_t *out,
                                      cudaStream_t stream);

cudaError_t launch_balance(const uint16_t *xc, int64_t ldxc, const int32_t *xc_rows, int64_t mc,
                           const uint16_t *w, int64_t n, int64_t k, float *s, float *inv_s,
                           cudaStream_t stream);

cudaError_t launch_debug_e2m1(const float *t, int64_t n, uint8_t *codes, cudaStream_t stream);

struct GemmArgs {
    const uint8_t *a_codes;
    const uint8_t *a_scales;
    const uint8_t *w_codes;
    const uint8_t *w_scales;
    const int32_t *offsets;  // grouped only
    int64_t M;               // dense: rows of A; grouped: sorted rows (rows of Y)
    int64_t a_rows;          // rows of the A code tensor (grouped: padded capacity)
    int64_t N, K;
    int32_t E;               // 0 = dense
    void *Y;
    int64_t ldy;
    // grouped gate+up with interleaved weight rows (N = 2F): epi 1 / 2 write
    // the down input h = SiLU(g) * u as MXFP4 (Hadamard block 32 / 64) into
    // h_codes / h_scales with the down balance factors h_f [E, F]; Y unused
    int32_t epi = 0;
    uint8_t *h_codes = nullptr;
    uint8_t *h_scales = nullptr;
    const float *h_f = nullptr;
    // the weight was complete before the preceding kernel on the stream
    // started, and that kernel lets dependents start only after its own
    // grid-dependency wait (the transform kernels do): the few-rows GEMM then
    // issues the weight's first stages before its wait.  Set only by
    // macaq_linear, whose GEMM always follows its own transform.
    bool weight_early = false;
};

cudaError_t launch_gemm(const GemmArgs &g, cudaStream_t stream);

// The whole dense layer for a few token rows in one launch: the few-rows GEMM
// forms its token operand from X bf16 [M, ldx] and the balance factors inv_s
// [K] (Hadamard block 32) stage by stage, instead of reading a_codes /
// a_scales (which it ignores).  Every CTA transforms all M rows of its K
// range, so the work grows with M while the weight stream it hides behind
// does not: at K = 5120, N = 25600 one launch took 15.2-16.1 us for M = 1..4
// and 18.9 us for M = 6 against 20.6-21.3 us for the transform and GEMM
// launches, but 21.8 us for M = 8 against 20.9.  Returns
// cudaErrorNotSupported for larger M.
constexpr int64_t kFusedLinearMaxRows = 6;
cudaError_t launch_linear_fused(const GemmArgs &g, const uint16_t *X, int64_t ldx, const float *inv_s,
                                cudaStream_t stream);

// W4A16: Y[M, N] = Xt[M, K] . Wd[N, K]^T with Wd the bf16 expansion of the
// MXFP4 weight (codes [N, K/2], tiled scales), expanded tile by tile in
// shared memory; bf16 products, fp32 accumulation (tcgen05 kind::f16).
struct W4A16Args {
    const void *Xt;
    int64_t ldx;
    const uint8_t *w_codes;
    const uint8_t *w_scales;
    int64_t M, N, K;
    void *Y;
    int64_t ldy;
};
cudaError_t launch_w4a16_gemm(const W4A16Args &g, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda
// link), interleave none, 256-byte L2 promotion, zero fill out of bounds.
bool encode_tensor_map(CUtensorMap *m, CUtensorMapDataType dt, uint32_t rank, const void *base,
                       const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                       CUtensorMapSwizzle sw);

cudaError_t read_and_clear_device_error(unsigned *flags);
cudaError_t read_and_clear_quant_error(unsigned *flags);
cudaError_t set_wait_timeout_ns(uint64_t ns);
cudaError_t launch_wait_probe(cudaStream_t stream);
cudaError_t launch_mma_rate(int bn, int iters, unsigned long long *out, const uint8_t *src, int ctas,
                            cudaStream_t stream);

}  // namespace macaq
