/*
 * macaq.h -- C ABI of the MACaQ W4A4 (MXFP4) linear-layer library for B300
 * (sm_103a).
 *
 * The method (MACaQ page "What is MACaQ quantization", section "How MACaQ
 * works"): each linear layer balances its input channels with a per-channel
 * scale, rotates each block of 32 channels with a Hadamard transform whose
 * inverse is folded into the weights ahead of time (so the output is unchanged
 * before rounding), and runs in W4A4 MXFP4 (FAQ "What is W4A4 quantization":
 * 4-bit floats in blocks of 32 sharing one scale).  Scale and rotation run
 * online at inference time (same section, closing paragraph).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is device memory owned by the caller (unless the
 *   comment says host).  The library allocates and frees nothing.
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means the
 *   legacy default stream).  No entry point synchronises, except
 *   macaq_check_device_error and macaq_set_wait_timeout_ns.
 * - Arguments are validated on the host before any launch; a rejected call
 *   launches nothing and returns the matching MACAQ_ERR_* code.  A failed
 *   launch returns MACAQ_ERR_CUDA.
 * - bf16 means IEEE bfloat16 bits (uint16).  Inputs must be finite.
 * - All pointers must be 16-byte aligned; leading dimensions (ldx, ldy) are
 *   counted in elements and must be multiples of 8.  K must be a positive
 *   multiple of 32.  M, N, rows may be 0 (nothing is launched).
 *
 * MXFP4 data layout
 * -----------------
 * codes   [rows, K/2] uint8, row-major, row pitch K/2 bytes.  Byte i of a row
 *         holds element 2i in its low nibble and element 2i+1 in its high
 *         nibble.  A nibble is E2M1: sign<<3 | exponent(2)<<1 | mantissa(1),
 *         magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7.
 * scales  one E8M0 byte (2^(byte-127)) per 32 consecutive elements of a row,
 *         stored TILED: rows pad to a multiple of 128, scale columns (K/32)
 *         to a multiple of 8, padding bytes are 0.  Tile (rb, ka) holds rows
 *         128*rb .. 128*rb+127 and scale columns 4*ka .. 4*ka+3 in 512
 *         contiguous bytes at offset (rb * nka + ka) * 512, nka = padded
 *         columns / 4; within a tile, row 32*q + p, column c is byte
 *         16*p + 4*q + c.  Size: macaq_scale_bytes(rows, K).
 * The value of element (r, j) is E2M1(code) * 2^(scale - 127).
 */
#ifndef MACAQ_H
#define MACAQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MACAQ_OK = 0,
    MACAQ_ERR_INVALID_ARG = 1,  /* null pointer, negative size, K % 32 != 0 */
    MACAQ_ERR_ALIGNMENT = 2,    /* pointer not 16-byte aligned, ld % 8 != 0 */
    MACAQ_ERR_UNSUPPORTED = 3,  /* size outside the supported range */
    MACAQ_ERR_WORKSPACE = 4,    /* workspace missing or too small */
    MACAQ_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
    MACAQ_ERR_TIMEOUT = 6       /* a device-side wait ran out (see below) */
} macaq_status;

typedef void *macaq_stream_t; /* cudaStream_t */

/* Human-readable name of a status code (static string). */
const char *macaq_status_string(macaq_status s);

/* Bytes of a tiled scale array for `rows` rows of K elements. */
size_t macaq_scale_bytes(int64_t rows, int64_t K);

/* ----------------------------------------------------------- balance */

/* Per-channel balance scales from calibration data (offline preparation).
 * Source: section "How MACaQ works", step "Channel balancing" (a per-channel
 * scale evens out the size of the input channels).
 *   s[j]     = fp32( clamp( sqrt(cx_j / cw_j), 1e-2, 1e2 ) ), ratio and root in
 *              fp64; cx_j = max_m |Xc[m, j]|, cw_j = max_n |W[n, j]|; cw_j = 0
 *              gives 1e2, cx_j = cw_j = 0 gives 1.
 *   inv_s[j] = 1.0f / s[j] (IEEE fp32 division).
 * Xc      bf16 [Mc, ldxc]: calibration rows.  If xc_rows is not NULL, row m
 *         of the batch is Xc row xc_rows[m] (int32, device), else row m.
 * W       bf16 [N, K], row pitch K.
 * s,inv_s fp32 [K] outputs.  Mc >= 0, N >= 0. */
macaq_status macaq_balance_scales(const void *Xc, int64_t ldxc, const int32_t *xc_rows,
                                  int64_t Mc, const void *W, int64_t N, int64_t K,
                                  float *s, float *inv_s, macaq_stream_t stream);

/* ------------------------------------------------- transform + MXFP4 */

/* Online activation transform (the hot path's first half).
 * Source: section "How MACaQ works" (balance, then 32-channel block Hadamard,
 * run online) and FAQ "What is W4A4 quantization" (MXFP4).
 * For each row m and 32-block b (j = 32b + i):
 *   v_i = fp32(X[m, j]) * inv_s[j]                        (fp32, rounded)
 *   v  <- butterflies at stride 1, 2, 4, 8, 16: (a, b) -> (a + b, a - b)
 *   y_i = v_i * fp32(1/sqrt 32)
 *   se  = clamp(floor(log2 max_i |y_i|) - 2, -127, 127)   (all-zero: -127)
 *   code_i = E2M1(y_i * 2^-se), round to nearest, ties to even code,
 *            saturate at 6, sign kept (also on values that round to 0)
 * X       bf16 [M, ldx]; inv_s fp32 [K].
 * a_codes [M, K/2]; a_scales tiled, macaq_scale_bytes(M, K) bytes (every
 *         byte written, padding included). */
macaq_status macaq_quant_act(const void *X, int64_t ldx, const float *inv_s, int64_t M,
                             int64_t K, uint8_t *a_codes, uint8_t *a_scales,
                             macaq_stream_t stream);

/* Offline weight preparation: the same transform with factor s (the inverse
 * balance and the Hadamard folded into the weights, section "How MACaQ works",
 * "A small Hadamard transform"), then MXFP4.
 * W [N, K] bf16 row pitch K; s fp32 [K]; w_codes [N, K/2];
 * w_scales macaq_scale_bytes(N, K) bytes. */
macaq_status macaq_quant_weight(const void *W, const float *s, int64_t N, int64_t K,
                                uint8_t *w_codes, uint8_t *w_scales, macaq_stream_t stream);

/* The transform with a Hadamard block of `hadamard_block` channels: 32 (as
 * macaq_quant_act / macaq_quant_weight) or 64.  The 64-channel block is the
 * recipe's "--had-block 64" option (page "Huawei MACaQ Is an Open-Source
 * Model Quantizer", llama.cpp recipe): the normalised Sylvester matrix of order
 * 64 (butterflies at strides 1 .. 32, then x 1/8 exactly) replaces H32, so one
 * Hadamard block spans two MX blocks; the MXFP4 encoding (blocks of 32, E8M0
 * scales, E2M1 codes, the same layouts) and macaq_w4a4_gemm are unchanged.
 * Activations and weights of one layer must use the same block (the fold).
 * K % hadamard_block == 0 (else MACAQ_ERR_INVALID_ARG); other arguments,
 * layouts and errors as macaq_quant_act / macaq_quant_weight. */
macaq_status macaq_quant_act_hb(const void *X, int64_t ldx, const float *inv_s, int64_t M, int64_t K,
                                int64_t hadamard_block, uint8_t *a_codes, uint8_t *a_scales,
                                macaq_stream_t stream);
macaq_status macaq_quant_weight_hb(const void *W, const float *s, int64_t N, int64_t K,
                                   int64_t hadamard_block, uint8_t *w_codes, uint8_t *w_scales,
                                   macaq_stream_t stream);

/* Grouped (per-expert) weight preparation: E experts, W [E, N, K] bf16,
 * s [E, K] fp32 (expert e uses row e); w_codes [E, N, K/2]; w_scales holds E
 * consecutive tiled arrays of macaq_scale_bytes(N, K) bytes each. */
macaq_status macaq_quant_weight_grouped(const void *W, const float *s, int64_t E, int64_t N,
                                        int64_t K, uint8_t *w_codes, uint8_t *w_scales,
                                        macaq_stream_t stream);

/* The grouped weight preparation with a Hadamard block of 32 or 64 channels
 * (see macaq_quant_act_hb; K % hadamard_block == 0); arguments and layouts as
 * macaq_quant_weight_grouped. */
macaq_status macaq_quant_weight_grouped_hb(const void *W, const float *s, int64_t E, int64_t N, int64_t K,
                                           int64_t hadamard_block, uint8_t *w_codes, uint8_t *w_scales,
                                           macaq_stream_t stream);

/* ------------------------------------------------------------ GEMM */

/* Block-scaled MXFP4 x MXFP4 GEMM with bf16 output (the hot path's second
 * half; W4A4 is the default inference mode, page "Huawei MACaQ", section
 * "MACaQ Backends").
 *   Y[m, n] = bf16_rn( sum_k A(m, k) * Wq(n, k) ), each operand an E2M1 code
 *             times its block's 2^(scale-127); products exact, accumulation
 *             in fp32 on the tensor cores (tcgen05, kind::mxf4).
 * a_codes [M, K/2], a_scales tiled for M rows; w_codes [N, K/2], w_scales
 * tiled for N rows; Y bf16 [M, ldy], ldy >= N. */
macaq_status macaq_w4a4_gemm(const uint8_t *a_codes, const uint8_t *a_scales,
                             const uint8_t *w_codes, const uint8_t *w_scales, int64_t M,
                             int64_t N, int64_t K, void *Y, int64_t ldy, macaq_stream_t stream);

/* Workspace bytes macaq_linear needs for M rows of K channels. */
size_t macaq_linear_workspace_bytes(int64_t M, int64_t K);

/* The whole online layer: macaq_quant_act into `workspace`, then
 * macaq_w4a4_gemm, both on `stream`.  Y = X diag(1/s) H (W diag(s) H)^T up
 * to MXFP4 rounding.  workspace: device, ws_bytes >=
 * macaq_linear_workspace_bytes(M, K), 256-byte aligned, contents scratch.
 * Up to 6 token rows (decode) both steps run as one kernel -- the GEMM forms
 * the transformed token rows itself, stage by stage -- and the workspace is
 * left untouched; Y is bit for bit the two calls' result either way. */
macaq_status macaq_linear(const void *X, int64_t ldx, const float *inv_s,
                          const uint8_t *w_codes, const uint8_t *w_scales, int64_t M,
                          int64_t N, int64_t K, void *Y, int64_t ldy, void *workspace,
                          size_t ws_bytes, macaq_stream_t stream);

/* macaq_linear for callers that cannot allocate device memory at the call
 * site -- for example a plugin whose host framework owns every device
 * allocation, or a runtime that fixes its device memory at start-up.  The
 * workspace is instead a scratch array of MACAQ_LINEAR_STATIC_SCRATCH_BYTES
 * inside the library's own module image; every GPU that loads the library
 * holds that array until the process exits.  The pages describe no such
 * entry point: it exists only for these callers.
 * Arguments as macaq_linear, without workspace / ws_bytes.  A problem whose
 * macaq_linear_workspace_bytes(M, K) exceeds the array is rejected with
 * MACAQ_ERR_WORKSPACE before anything is launched.  Nothing is allocated:
 * the first call on a device looks up the array's device address (make that
 * first call before any stream capture).  The address belongs to the CUDA
 * context current at the call: each context that loads the library holds its
 * own copy of the array, and a call made under a different context than the
 * previous one on that device (after cudaDeviceReset, or under a caller's own
 * driver-API context) looks the address up again, so that call too belongs
 * before any stream capture.  All calls in one context share the one array,
 * so calls that can overlap on the GPU (different streams without ordering)
 * race; the array keeps the last call's contents, which no call depends on. */
#define MACAQ_LINEAR_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
macaq_status macaq_linear_no_alloc(const void *X, int64_t ldx, const float *inv_s,
                                   const uint8_t *w_codes, const uint8_t *w_scales, int64_t M,
                                   int64_t N, int64_t K, void *Y, int64_t ldy,
                                   macaq_stream_t stream);

/* ---------------------------------------------------- grouped (MoE) */

/* Rows of the expert-padded layout the grouped kernels use for `rows`
 * expert-sorted rows over E experts: every expert's rows start on a multiple
 * of 128 (an upper bound; the exact layout follows expert_offsets). */
int64_t macaq_grouped_padded_rows(int64_t rows, int64_t E);

/* Grouped activation transform for routed MoE experts (the routed experts
 * run W4A4, page "Huawei MACaQ", section "MACaQ Backends").
 * Rows are sorted by expert: sorted row r belongs to expert e for
 * expert_offsets[e] <= r < expert_offsets[e+1] (int32 [E+1], device,
 * nondecreasing, offsets[0] = 0, offsets[E] = rows) and reads token row
 * X[row_src[r]] (int32 [rows], device).  It is transformed with inv_s row e
 * (fp32 [E, K]) and written to padded row p = P_e + (r - offsets[e]) with
 * P_e = sum_{e' < e} 128 * ceil(count_e' / 128).
 * a_codes [P, K/2], a_scales tiled for P rows, P =
 * macaq_grouped_padded_rows(rows, E).  Scale bytes of padding rows are 0;
 * code bytes of padding rows are left unspecified.  E <= 256. */
macaq_status macaq_quant_act_grouped(const void *X, int64_t ldx, const int32_t *row_src,
                                     const int32_t *expert_offsets, const float *inv_s,
                                     int64_t rows, int64_t E, int64_t K, uint8_t *a_codes,
                                     uint8_t *a_scales, macaq_stream_t stream);

/* macaq_quant_act_grouped with a Hadamard block of 32 or 64 channels (the
 * 64-channel block of macaq_quant_act_hb, the recipe's "--had-block 64");
 * K % hadamard_block == 0. */
macaq_status macaq_quant_act_grouped_hb(const void *X, int64_t ldx, const int32_t *row_src,
                                        const int32_t *expert_offsets, const float *inv_s, int64_t rows,
                                        int64_t E, int64_t K, int64_t hadamard_block, uint8_t *a_codes,
                                        uint8_t *a_scales, macaq_stream_t stream);

/* Grouped activation transform of a gated MLP's down-projection input,
 * fused with its SwiGLU step.  GU bf16 [rows, ldgu] holds, in sorted row
 * order, the gate (columns 0..F-1) and up (columns F..2F-1) outputs of the
 * grouped gate+up GEMM; row r is first turned into
 *   h_j = bf16_rn( SiLU(g_j) * u_j ),  SiLU(g) = g / (1 + e^-g)
 * in fp32 (e^x by Cody-Waite range reduction and a degree-8 Taylor
 * polynomial, every operation rounded to nearest), then transformed exactly as
 * macaq_quant_act_grouped transforms token rows (balance with inv_s row e,
 * fp32 [E, F]; 32-point Hadamard; MXFP4) into padded row P_e + r - offsets[e].
 * The pages state no gated-MLP arithmetic: the SwiGLU form and its fp32 / bf16
 * rounding are this library's reading (the value an unfused layer would store
 * in bf16, re-read by the transform).  The routed experts it serves run W4A4
 * (page "Huawei MACaQ", section "MACaQ Backends").  a_codes [P, F/2],
 * a_scales tiled for P rows, P = macaq_grouped_padded_rows(rows, E); padding
 * rows as in macaq_quant_act_grouped.  F % 32 == 0, ldgu >= 2F, ldgu % 8 == 0,
 * GU 16-byte aligned, E <= 256. */
macaq_status macaq_quant_act_grouped_silu(const void *GU, int64_t ldgu, const int32_t *expert_offsets,
                                          const float *inv_s, int64_t rows, int64_t E, int64_t F,
                                          uint8_t *a_codes, uint8_t *a_scales, macaq_stream_t stream);

/* macaq_quant_act_grouped_silu with a Hadamard block of 32 or 64 channels;
 * F % hadamard_block == 0. */
macaq_status macaq_quant_act_grouped_silu_hb(const void *GU, int64_t ldgu, const int32_t *expert_offsets,
                                             const float *inv_s, int64_t rows, int64_t E, int64_t F,
                                             int64_t hadamard_block, uint8_t *a_codes, uint8_t *a_scales,
                                             macaq_stream_t stream);

/* The same fused SwiGLU transform for a dense gated MLP (the down
 * projection's input h = bf16(SiLU(g) * u), SiLU and rounding as
 * macaq_quant_act_grouped_silu): GU bf16 [M, ldgu] holds gate columns
 * 0 .. F-1 and up columns F .. 2F-1 of each row; inv_s fp32 [F]; output as
 * macaq_quant_act of h (a_codes [M, F/2], a_scales macaq_scale_bytes(M, F)
 * bytes).  Equals macaq_quant_act of the bf16 h, without writing h. */
macaq_status macaq_quant_act_silu(const void *GU, int64_t ldgu, const float *inv_s, int64_t M, int64_t F,
                                  uint8_t *a_codes, uint8_t *a_scales, macaq_stream_t stream);

/* Grouped GEMM: for each expert e and sorted row r of e,
 *   Y[r, n] = bf16_rn( sum_k A(P_e + r - offsets[e], k) * Wq_e(n, k) )
 * with A from macaq_quant_act_grouped and Wq_e from
 * macaq_quant_weight_grouped (w_codes [E, N, K/2], w_scales E tiled arrays).
 * Y bf16 [rows, ldy] in sorted row order.  E <= 256. */
macaq_status macaq_grouped_w4a4_gemm(const uint8_t *a_codes, const uint8_t *a_scales,
                                     const uint8_t *w_codes, const uint8_t *w_scales,
                                     const int32_t *expert_offsets, int64_t rows, int64_t E,
                                     int64_t N, int64_t K, void *Y, int64_t ldy,
                                     macaq_stream_t stream);

/* The gate+up projection of a routed gated MLP with its output written
 * directly as the down projection's MXFP4 input (the routed experts run W4A4,
 * page "Huawei MACaQ Is an Open-Source Model Quantizer", section "MACaQ
 * Backends"; the scale and rotation run online at inference time, page "What
 * is MACaQ quantization", section "How MACaQ works", closing paragraph): the
 * grouped GEMM's epilogue forms, per sorted row r of expert e and channel j,
 *   g = bf16_rn(gate GEMM output), u = bf16_rn(up GEMM output),
 *   h_j = bf16_rn( SiLU(g) * u )          (as macaq_quant_act_grouped_silu)
 * and runs the activation transform on h with the down projection's balance
 * factors inv_s row e (fp32 [E, F]; Hadamard block 32 or 64, MXFP4) into
 * padded row P_e + r - offsets[e] -- exactly the codes and scales that
 * macaq_grouped_w4a4_gemm with bf16 output followed by
 * macaq_quant_act_grouped_silu(_hb) produce, without writing the bf16
 * gate|up matrix.
 * a_codes / a_scales: the grouped token transform (macaq_quant_act_grouped);
 * w_codes [E, 2F, K/2] and w_scales (E tiled arrays of 2F rows): the gate and
 * up weights prepared with macaq_quant_weight_grouped(_hb) from the rows
 * macaq_interleave_gate_up arranged; h_codes [P, F/2] and h_scales tiled for
 * P = macaq_grouped_padded_rows(rows, E) rows of F channels, as
 * macaq_quant_act_grouped_silu writes them (scale bytes of padding rows 0,
 * codes of padding rows unspecified).  F % 64 == 0, K % 32 == 0, E <= 256,
 * hadamard_block 32 or 64 (F % 64 == 0 covers both). */
macaq_status macaq_grouped_w4a4_gemm_swiglu(const uint8_t *a_codes, const uint8_t *a_scales,
                                            const uint8_t *w_codes, const uint8_t *w_scales,
                                            const int32_t *expert_offsets, int64_t rows, int64_t E, int64_t F,
                                            int64_t K, const float *inv_s, int64_t hadamard_block,
                                            uint8_t *h_codes, uint8_t *h_scales, macaq_stream_t stream);

/* Weight preparation for macaq_grouped_w4a4_gemm_swiglu: W_gu bf16
 * [E, 2F, K] with each expert's gate rows 0 .. F-1 and up rows F .. 2F-1 ->
 * W_out bf16 [E, 2F, K] whose rows 128c .. 128c+63 are gate rows 64c ..
 * 64c+63 and rows 128c+64 .. 128c+127 the up rows of the same channels (a
 * row permutation; no arithmetic).  F % 64 == 0; W_gu and W_out distinct,
 * 16-byte aligned, row pitch K. */
macaq_status macaq_interleave_gate_up(const void *W_gu, int64_t E, int64_t F, int64_t K, void *W_out,
                                      macaq_stream_t stream);

/* ------------------------------------------------ W4A16 fallback */

/* The weight-only fallback (page "Huawei MACaQ: Choosing GGUF or vLLM and
 * Avoiding Setup Mistakes", section "vLLM checkpoints have different
 * constraints": the W4A16 mode expands the weights for a BF16 matrix
 * multiplication and is slower than W4A4).  The weights are the same MXFP4
 * checkpoint (macaq_quant_weight / _hb); the activations keep the online
 * transform but are not quantised: the fp32 transform is rounded once to
 * bf16 (this library's reading; the pages state no W4A16 arithmetic).
 *
 * macaq_transform_act_bf16: Xt[m, k] = bf16_rn(y) with y the normalised
 * transform of macaq_quant_act (hadamard_block 32) or macaq_quant_act_hb
 * (64).  X bf16 [M, ldx]; inv_s fp32 [K]; Xt bf16 [M, ldxt], ldxt >= K, a
 * multiple of 8; only the first K columns of each row are written.  Errors as
 * macaq_quant_act_hb. */
macaq_status macaq_transform_act_bf16(const void *X, int64_t ldx, const float *inv_s, int64_t M,
                                      int64_t K, int64_t hadamard_block, void *Xt, int64_t ldxt,
                                      macaq_stream_t stream);

/* Weight expansion on its own: Wd[n, k] = the MXFP4 value (E2M1 code times
 * 2^(scale - 127)) as bf16, exact for every scale an fp32 input can produce.
 * w_codes [N, K/2] and tiled w_scales as macaq_quant_weight writes them; Wd
 * bf16 [N, K] (row pitch K), 16-byte aligned.  The W4A16 GEMM below does
 * not need it (it expands tiles on chip); it is the checkpoint's bf16 form
 * for callers that want one. */
macaq_status macaq_dequant_weight_bf16(const uint8_t *w_codes, const uint8_t *w_scales, int64_t N,
                                       int64_t K, void *Wd, macaq_stream_t stream);

/* The W4A16 GEMM: Y[m, n] = bf16_rn( sum_k Xt(m, k) * Wd(n, k) ), Wd(n, k) the
 * bf16 value of the MXFP4 weight (as macaq_dequant_weight_bf16), expanded
 * tile by tile in shared memory so the weight is read at 4.25 bits per
 * value; bf16 products accumulated in fp32 on the tensor cores.  Xt bf16
 * [M, ldxt] (ldxt >= K); w_codes [N, K/2] and tiled w_scales from
 * macaq_quant_weight(_hb); Y bf16 [M, ldy] (ldy >= N); ldxt and ldy
 * multiples of 8, pointers 16-byte aligned. */
macaq_status macaq_w4a16_gemm(const void *Xt, int64_t ldxt, const uint8_t *w_codes, const uint8_t *w_scales,
                              int64_t M, int64_t N, int64_t K, void *Y, int64_t ldy, macaq_stream_t stream);

/* Workspace bytes macaq_w4a16_linear needs for M rows of K channels (the
 * bf16 transform of the activations). */
size_t macaq_w4a16_linear_workspace_bytes(int64_t M, int64_t K);

/* The W4A16 layer: macaq_transform_act_bf16 into `workspace`, then
 * macaq_w4a16_gemm, both on `stream`.  w_codes / w_scales prepared with the
 * same hadamard_block; Y bf16 [M, ldy], ldy >= N, a multiple of 8; workspace
 * as macaq_linear (256-byte aligned, ws_bytes >=
 * macaq_w4a16_linear_workspace_bytes(M, K)). */
macaq_status macaq_w4a16_linear(const void *X, int64_t ldx, const float *inv_s, const uint8_t *w_codes,
                                const uint8_t *w_scales, int64_t M, int64_t N, int64_t K,
                                int64_t hadamard_block, void *Y, int64_t ldy, void *workspace, size_t ws_bytes,
                                macaq_stream_t stream);

/* --------------------------------------------- Flip Refinement (offline) */

/* The fp32 transform itself (no rounding to MXFP4): Y[m, k] = the normalised
 * transform y of macaq_quant_act (hadamard_block 32) / macaq_quant_act_hb (64)
 * of X with factor f (1/s for activations, s for weights).  X bf16 [M, ldx];
 * Y fp32 [M, ldy], ldy >= K, a multiple of 4; only the first K columns of each
 * row are written.  The rotated rows Flip Refinement works on. */
macaq_status macaq_transform_f32(const void *X, int64_t ldx, const float *f, int64_t M, int64_t K,
                                 int64_t hadamard_block, float *Y, int64_t ldy, macaq_stream_t stream);

/* Flip Refinement (page "What is MACaQ quantization", section "How MACaQ
 * works", step "Flip Refinement": instead of plain round to nearest, a
 * Hessian-aware coordinate descent moves single 4-bit weight codes to an
 * adjacent value when that lowers the layer's error on calibration data).
 * Reading: in the rotated space the layer output is A . Wt^T, with A the
 * calibration rows through the activation transform and Wt the weight rows
 * through the weight transform (macaq_transform_f32 with 1/s and s); the
 * error of one weight row with dequantised codes q is
 *   E(q) = (Wt - q)^T H (Wt - q),  H = A^T A (+ damp on the diagonal).
 *
 * macaq_flip_hessian: H[i, j] = fp32 fused multiply-add chain over the
 * calibration rows r = 0 .. Mc-1 of A[r, i] * A[r, j] (from +0), then + damp
 * (one fp32 add) where i == j.  A fp32 [Mc, K] row pitch K; H fp32 [K, K]
 * (symmetric bit for bit), 4 K^2 bytes, caller-owned. */
macaq_status macaq_flip_hessian(const float *A, int64_t Mc, int64_t K, float damp, float *H,
                                macaq_stream_t stream);

/* Workspace bytes macaq_flip_refine needs for N rows of K channels. */
size_t macaq_flip_refine_workspace_bytes(int64_t N, int64_t K);

/* The descent, per weight row: r = Wt - q, g = H r (a fused multiply-add
 * chain over k); `sweeps` passes over k = 0 .. K-1; at each k the two
 * neighbours of q_k on the signed E2M1 grid (-6 .. -0.5, 0, 0.5 .. 6 times the
 * block's scale, which never changes) are scored dE = D (D H_kk - 2 g_k)
 * (fp32, one rounding per operation; D the move), the lower strictly negative
 * score is taken (ties to the lower value), and g -= D H[k, :].  A move onto
 * zero keeps the sign of the side it came from (code 0x8 from below).  The
 * pages do not fix the number of passes; the recipe's --vq-sweeps default of 2
 * is the natural choice.
 * Wt fp32 [N, K] row pitch K; H from macaq_flip_hessian; w_codes [N, K/2]
 * (in: round-to-nearest codes from macaq_quant_weight / _hb, out: refined)
 * and tiled w_scales (read only) for the same Wt; flips: int32 [N] moves per
 * row, or NULL.  workspace: device, >= macaq_flip_refine_workspace_bytes(N, K),
 * 256-byte aligned.  K above 48736 is MACAQ_ERR_UNSUPPORTED (a row's state
 * lives in shared memory).  A row whose warps fail to meet within 2 s stops
 * without writing its codes and macaq_check_device_error reports
 * MACAQ_ERR_TIMEOUT. */
macaq_status macaq_flip_refine(const float *Wt, const float *H, int64_t N, int64_t K, int32_t sweeps,
                               uint8_t *w_codes, const uint8_t *w_scales, int32_t *flips,
                               void *workspace, size_t ws_bytes, macaq_stream_t stream);

/* macaq_flip_refine in its two launches.  macaq_flip_prepare: r = Wt - q of
 * the current codes and g = H r (fused multiply-add chain over k) into
 * `workspace`.  macaq_flip_sweeps: the passes, starting from the g that
 * macaq_flip_prepare left in the same workspace (it does not write g back:
 * more passes later start with a new macaq_flip_prepare, whose g is computed
 * afresh and so may differ in its last bits from a continued descent).
 * Arguments and errors as macaq_flip_refine. */
macaq_status macaq_flip_prepare(const float *Wt, const float *H, int64_t N, int64_t K,
                                const uint8_t *w_codes, const uint8_t *w_scales, void *workspace,
                                size_t ws_bytes, macaq_stream_t stream);
macaq_status macaq_flip_sweeps(const float *H, int64_t N, int64_t K, int32_t sweeps, uint8_t *w_codes,
                               const uint8_t *w_scales, int32_t *flips, void *workspace, size_t ws_bytes,
                               macaq_stream_t stream);

/* ------------------------------------------------------ MoE combine */

/* The routed layer's output: token t's row is the weighted sum of the expert
 * rows of its top-k choices (the rows macaq_grouped_w4a4_gemm wrote, in
 * expert-sorted order).  The pages run the routed projections in W4A4 (page
 * "Huawei MACaQ Is an Open-Source Model Quantizer", section "MACaQ
 * Backends") and give no combine arithmetic; reading:
 *   out[t, n] = bf16_rn( fp32 fused multiply-add chain over k = 0 .. topk-1
 *               of tok_weights[t, k] * Y[tok_rows[t, k], n], from +0 )
 * Y bf16 [y_rows, ldy]; tok_rows int32 [T, topk] (row of each choice; rows
 * outside [0, y_rows) contribute nothing); tok_weights fp32 [T, topk]; out
 * bf16 [T, ldo].  N % 8 == 0, ldy and ldo multiples of 8, Y and out 16-byte
 * aligned; 0 < topk <= 1024. */
macaq_status macaq_moe_combine(const void *Y, int64_t ldy, int64_t y_rows, const int32_t *tok_rows,
                               const float *tok_weights, int64_t T, int64_t topk, int64_t N, void *out,
                               int64_t ldo, macaq_stream_t stream);

/* --------------------------------------------------- device errors */

/* Every device-side wait of the GEMM kernels is bounded in time.  A wait that
 * runs out sets a device error flag and the kernel returns early (its output
 * is then undefined) instead of hanging.
 * macaq_check_device_error synchronises `stream`, reads and clears the flag
 * of the current device, and returns MACAQ_ERR_TIMEOUT if it was set. */
macaq_status macaq_check_device_error(macaq_stream_t stream);

/* Sets the bound of each device-side wait on the current device, in
 * nanoseconds (default 4e9).  Synchronous. */
macaq_status macaq_set_wait_timeout_ns(uint64_t ns);

/* Test hook for the bounded wait: launches one thread that waits on a
 * barrier nothing ever signals; it gives up after the configured bound and
 * sets the device error flag. */
macaq_status macaq_debug_wait_probe(macaq_stream_t stream);

/* Test hook for the element encoder: codes[i] = E2M1 code of t[i] (fp32, any
 * finite value; |t| > 6 saturates), as the quantisation kernels compute it.
 * t fp32 [n], codes uint8 [n]. */
macaq_status macaq_debug_e2m1(const float *t, int64_t n, uint8_t *codes,
                              macaq_stream_t stream);

/* Tensor-core rate probe: `ctas` CTAs (at most one per SM) each issue
 * 4 * iters back-to-back block-scaled MXFP4 MMAs of shape 128 x bn x 64 on
 * operands already in shared memory.  out (device uint64 [2 * ctas]) receives
 * per CTA the elapsed SM cycles and nanoseconds.  Low 16 bits of bn: N (16 <= N <= 256,
 * N % 16 == 0); bits 16 and up: 0 = MMAs only, 1 = also the six scale-factor
 * copies a 256-wide K stage needs before its four MMAs, 2 = also one
 * tcgen05.commit per stage, 3 = MMAs while another thread streams 16 KB bulk
 * copies from `src` (device, >= 1 MiB, 16-byte aligned) into shared memory;
 * out then has 3 * ctas entries, the last ctas being bytes copied per CTA.
 * src may be NULL for modes 0..2. */
macaq_status macaq_debug_mma_rate(int32_t bn, int32_t iters, int32_t ctas, const void *src,
                                  uint64_t *out, macaq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MACAQ_H */
