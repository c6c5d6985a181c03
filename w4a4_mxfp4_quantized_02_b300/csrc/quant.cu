// Balance + 32-channel block Hadamard + MXFP4 encode, and the calibration of
// the per-channel balance scales.
//
// MACaQ page "What is MACaQ quantization", section "How MACaQ works": a
// per-channel scale balances the input channels, a block Hadamard over 32
// channels spreads outliers (its inverse is folded into the weights), and the
// result is stored as MXFP4 (FAQ "What is W4A4 quantization": 4-bit floats in
// blocks of 32 sharing one scale).
//
// Design: one thread owns one 32-channel block of a row, so the whole
// 32-point butterfly network runs in that thread's registers (no shuffles),
// and the thread keeps its 32 balance factors in registers across the rows it
// visits.  A CTA covers a slab of consecutive blocks of one row (coalesced
// 64-byte-per-thread loads, 16-byte code stores) and walks a run of rows two
// at a time so each thread has 128 bytes of loads in flight.  Scale bytes of
// four neighbouring blocks are gathered with two shuffles into one 32-bit
// store in the tiled scale layout.
//
// Every arithmetic step uses explicitly rounded intrinsics (and the file is
// built with -fmad=false) so the codes are bit-exact against an fp32 CPU
// statement of the same steps.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace macaq {
namespace {

// fp32 nearest to 2^-2.5 = 1/sqrt(32).
constexpr float kInvSqrt32 = 0x1.6a09e6p-3f;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> one byte of two E2M1 codes (lo in bits 0..3, hi in bits 4..7),
// round to nearest even, saturating.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
#ifdef MACAQ_SOFT_E2M1
    auto enc = [](float t) -> uint32_t {
        const uint32_t s = (__float_as_uint(t) >> 31) << 3;
        const float a = fabsf(t);
        uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.0f);
        return s | m;
    };
    return enc(lo) | (enc(hi) << 4);
#else
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r;
#endif
}

// Packed fp32x2 multiply / add / subtract, each lane rounded to nearest even.
// The code generator fuses a packed multiply feeding a packed add into a
// packed FMA (single rounding) even with an explicit .rn modifier and
// -fmad=false, which would break bit-exactness.  So a packed multiply is only
// ever used where no add consumes its result, and every product that feeds an
// add is formed with scalar __fmul_rn.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 z, x, y;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 add2_rn(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %5};\n\t"
        "add.rn.f32x2 z, x, y;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 sub2_rn(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %5};\n\t"
        "sub.rn.f32x2 z, x, y;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// One 32-element block: balance, butterflies (stride 1, 2, 4, 8, 16),
// normalise, E8M0 scale, E2M1 codes.  raw: 16 words of bf16 pairs (element
// 2i in the low half of word i); f[i] = (f_i, f_{i+16}).  Returns the scale
// byte.
//
// Register layout: v[i] = (element i, element i + 16), so the stages at
// strides 2, 4 and 8 pair whole float2 registers and run as packed fp32x2
// adds (each lane rounded to nearest, exactly like two scalar adds); stride 1
// (whose inputs are products) and stride 16 (which pairs the two halves of a
// register) run as scalar adds.
//
// Scale and encode: the block maximum of |y| = |v * c| (c = fp32(1/sqrt 32))
// equals RN(max|v| * c) because rounding is monotone, so one multiply gives
// it.  The element to encode is RN(v * c) * 2^-se; when -124 <= se <= 122 it
// equals RN(v * (c * 2^-se)) for every element that can get a non-zero code
// (the constant c * 2^-se is exact and normal, products below the normal
// range round to a zero code either way), so one packed multiply per pair
// suffices.  Outside that range the two roundings are done separately.
__device__ __forceinline__ uint32_t quant_block(const uint32_t (&raw)[16], const float2 (&f)[16],
                                                uint4 &codes)
{
    float2 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t w0 = raw[i >> 1];
        const uint32_t w1 = raw[8 + (i >> 1)];
        const float x0 = (i & 1) ? bf16hi(w0) : bf16lo(w0);
        const float x1 = (i & 1) ? bf16hi(w1) : bf16lo(w1);
        v[i] = make_float2(__fmul_rn(x0, f[i].x), __fmul_rn(x1, f[i].y));
    }
    // stride 1 in scalar form: its operands are products (see mul2_rn)
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float2 a = v[i];
        const float2 b = v[i + 1];
        v[i] = make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
        v[i + 1] = make_float2(__fsub_rn(a.x, b.x), __fsub_rn(a.y, b.y));
    }
#pragma unroll
    for (int h = 2; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            const float2 a = v[i];
            const float2 b = v[i + h];
            v[i] = add2_rn(a, b);
            v[i + h] = sub2_rn(a, b);
        }
    }
    float vmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = v[i].x;
        const float b = v[i].y;
        v[i].x = __fadd_rn(a, b);
        v[i].y = __fsub_rn(a, b);
        vmax = fmax3(fabsf(v[i].x), fabsf(v[i].y), vmax);
    }
    const float amax = __fmul_rn(vmax, kInvSqrt32);
    // se = max(floor(log2 amax) - 2, -127) -> byte = max(exponent field - 2, 0)
    const int ef = static_cast<int>(__float_as_uint(amax) >> 23);
    const uint32_t sbyte = static_cast<uint32_t>(ef > 2 ? ef - 2 : 0);
    const int se = static_cast<int>(sbyte) - 127;
    if (se >= -124 && se <= 122) {
        // c * 2^-se: exponent field of c (124) moved by -se
        const float g = __int_as_float(__float_as_int(kInvSqrt32) - se * (1 << 23));
        const float2 g2 = make_float2(g, g);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = mul2_rn(v[i], g2);
    } else {
        const float c = kInvSqrt32;
        const float inv = __uint_as_float((254u - sbyte) << 23);  // 2^-se, normal
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = mul2_rn(v[i], make_float2(c, c));
            v[i] = mul2_rn(v[i], make_float2(inv, inv));
        }
    }
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t b[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = 4 * q + k;  // output byte: elements 2j, 2j+1
            const float lo = (j < 8) ? v[2 * j].x : v[2 * j - 16].y;
            const float hi = (j < 8) ? v[2 * j + 1].x : v[2 * j - 15].y;
            b[k] = e2m1x2(lo, hi);
        }
        w[q] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
    }
    codes = make_uint4(w[0], w[1], w[2], w[3]);
    return sbyte;
}

// 64 bytes of one row's block: two 256-bit loads when 32-byte aligned,
// otherwise four 128-bit loads.
template <bool kWide>
__device__ __forceinline__ void load_block(const uint16_t *src, uint32_t (&r)[16])
{
    if (kWide) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                         : "=r"(r[8 * h + 0]), "=r"(r[8 * h + 1]), "=r"(r[8 * h + 2]),
                           "=r"(r[8 * h + 3]), "=r"(r[8 * h + 4]), "=r"(r[8 * h + 5]),
                           "=r"(r[8 * h + 6]), "=r"(r[8 * h + 7])
                         : "l"(src + 16 * h));
        }
    } else {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 t = __ldg(s4 + j);
            r[4 * j + 0] = t.x;
            r[4 * j + 1] = t.y;
            r[4 * j + 2] = t.z;
            r[4 * j + 3] = t.w;
        }
    }
}

struct RowRef {
    const uint16_t *src;   // row start (nullptr when the row is padding)
    uint8_t *codes;        // row start of codes
    uint8_t *scale_base;   // tiled scale array this row belongs to
    int64_t srow;          // row index inside that tiled array
    int32_t group;         // balance-factor row
};

template <QuantMode MODE>
__device__ __forceinline__ RowRef resolve_row(const QuantArgs &a, int64_t p, const int32_t *s_off,
                                              const int32_t *s_poff)
{
    RowRef r;
    const int64_t half_k = a.K / 2;
    if (MODE == QuantMode::Dense) {
        const bool valid = p < a.rows_valid;
        r.src = valid ? a.src + p * a.ld_src : nullptr;
        r.codes = a.codes + p * half_k;
        r.scale_base = a.scales;
        r.srow = p;
        r.group = 0;
    } else if (MODE == QuantMode::WeightGrouped) {
        const int64_t g = p / a.group_rows_pad;
        const int64_t n = p - g * a.group_rows_pad;
        const bool valid = n < a.rows_valid;
        const int64_t row = g * a.rows_valid + n;
        r.src = valid ? a.src + row * a.ld_src : nullptr;
        r.codes = a.codes + row * half_k;
        r.scale_base = a.scales + g * a.scale_group_stride;
        r.srow = n;
        r.group = static_cast<int32_t>(g);
    } else {
        // expert e with s_poff[e] <= p < s_poff[e+1]
        int lo = 0, hi = a.E;  // invariant: s_poff[lo] <= p, answer in [lo, hi)
        if (p >= s_poff[a.E]) {
            lo = a.E;
        } else {
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_poff[mid] <= p) lo = mid; else hi = mid;
            }
        }
        r.codes = a.codes + p * half_k;
        r.scale_base = a.scales;
        r.srow = p;
        if (lo >= a.E) {
            r.src = nullptr;
            r.group = 0;
        } else {
            const int64_t j = p - s_poff[lo];
            const int64_t cnt = s_off[lo + 1] - s_off[lo];
            r.group = lo;
            r.src = (j < cnt) ? a.src + static_cast<int64_t>(a.row_src[s_off[lo] + j]) * a.ld_src
                              : nullptr;
        }
    }
    return r;
}

template <QuantMode MODE, bool kWide>
__global__ void __launch_bounds__(256) quant_kernel(QuantArgs a, int64_t rows_per_cta)
{
    constexpr int R = 2;  // rows per iteration (loads of all R rows in flight together)
    __shared__ int32_t s_off[kMaxExperts + 1];
    __shared__ int32_t s_poff[kMaxExperts + 1];
    if (MODE == QuantMode::ActGrouped) {
        for (int e = threadIdx.x; e <= a.E; e += blockDim.x) s_off[e] = a.offsets[e];
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t acc = 0;
            s_poff[0] = 0;
            for (int e = 0; e < a.E; ++e) {
                const int32_t cnt = s_off[e + 1] - s_off[e];
                acc += (cnt + 127) / 128 * 128;
                s_poff[e + 1] = acc;
            }
        }
        __syncthreads();
    }

    const int64_t nkb = a.K / 32;
    const int64_t nka = ((nkb + 7) / 8 * 8) / 4;
    const int64_t nkb_pad = nka * 4;
    const int64_t kb = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool has_kb = kb < nkb;
    const int lane = threadIdx.x & 31;
    const bool writes_scale = (lane & 3) == 0 && kb < nkb_pad;

    float2 f[16];
    int32_t cur_group = -1;

    const int64_t p_begin = static_cast<int64_t>(blockIdx.y) * rows_per_cta;
    const int64_t p_end = min(p_begin + rows_per_cta, a.rows_out);

    for (int64_t p = p_begin; p < p_end; p += R) {
        RowRef rr[R];
        uint32_t raw[R][16];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int64_t pu = p + u;
            if (pu < p_end) {
                rr[u] = resolve_row<MODE>(a, pu, s_off, s_poff);
            } else {
                rr[u].src = nullptr;
                rr[u].codes = nullptr;
                rr[u].scale_base = nullptr;
                rr[u].srow = 0;
                rr[u].group = cur_group;
            }
            if (rr[u].src != nullptr && has_kb) {
                load_block<kWide>(rr[u].src + 32 * kb, raw[u]);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) raw[u][j] = 0u;
            }
        }
#pragma unroll
        for (int u = 0; u < R; ++u) {
            if (p + u >= p_end) break;  // uniform across the CTA
            const bool valid = rr[u].src != nullptr;
            if (valid && rr[u].group != cur_group) {
                cur_group = rr[u].group;
                if (has_kb) {
                    const float4 *f4 = reinterpret_cast<const float4 *>(a.f + cur_group * a.K + 32 * kb);
                    float ff[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 t = __ldg(f4 + j);
                        ff[4 * j + 0] = t.x;
                        ff[4 * j + 1] = t.y;
                        ff[4 * j + 2] = t.z;
                        ff[4 * j + 3] = t.w;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) f[i] = make_float2(ff[i], ff[i + 16]);
                }
            }
            uint32_t sbyte = 0;
            if (valid && has_kb) {
                uint4 codes;
                sbyte = quant_block(raw[u], f, codes);
                *reinterpret_cast<uint4 *>(rr[u].codes + 16 * kb) = codes;
            }
            // gather the scale bytes of 4 neighbouring blocks into one word
            uint32_t word = sbyte << (8 * (lane & 3));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            if (writes_scale) {
                const int64_t r = rr[u].srow;
                const int64_t off = ((r / 128) * nka + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4;
                *reinterpret_cast<uint32_t *>(rr[u].scale_base + off) = word;
            }
        }
    }
}

// ---------------------------------------------------------------- balance

__global__ void __launch_bounds__(256) balance_kernel(const uint16_t *xc, int64_t ldxc,
                                                      const int32_t *xc_rows, int64_t mc,
                                                      const uint16_t *w, int64_t n, int64_t k,
                                                      float *s, float *inv_s)
{
    __shared__ float red_x[8][64];
    __shared__ float red_w[8][64];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t c = static_cast<int64_t>(blockIdx.x) * 64 + 2 * lane;
    float mx0 = 0.f, mx1 = 0.f, mw0 = 0.f, mw1 = 0.f;
    if (c < k) {
        for (int64_t m = warp; m < mc; m += 8) {
            const int64_t row = xc_rows ? static_cast<int64_t>(xc_rows[m]) : m;
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(xc + row * ldxc + c));
            mx0 = fmaxf(mx0, fabsf(bf16lo(v)));
            mx1 = fmaxf(mx1, fabsf(bf16hi(v)));
        }
        for (int64_t r = warp; r < n; r += 8) {
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(w + r * k + c));
            mw0 = fmaxf(mw0, fabsf(bf16lo(v)));
            mw1 = fmaxf(mw1, fabsf(bf16hi(v)));
        }
    }
    red_x[warp][2 * lane] = mx0;
    red_x[warp][2 * lane + 1] = mx1;
    red_w[warp][2 * lane] = mw0;
    red_w[warp][2 * lane + 1] = mw1;
    __syncthreads();
    if (threadIdx.x < 64) {
        const int64_t col = static_cast<int64_t>(blockIdx.x) * 64 + threadIdx.x;
        if (col < k) {
            float cx = 0.f, cw = 0.f;
            for (int i = 0; i < 8; ++i) {
                cx = fmaxf(cx, red_x[i][threadIdx.x]);
                cw = fmaxf(cw, red_w[i][threadIdx.x]);
            }
            double r;
            if (cw == 0.f) {
                r = (cx == 0.f) ? 1.0 : 1e2;
            } else {
                r = __dsqrt_rn(__ddiv_rn(static_cast<double>(cx), static_cast<double>(cw)));
                r = r < 1e-2 ? 1e-2 : r;
                r = r > 1e2 ? 1e2 : r;
            }
            const float sv = __double2float_rn(r);
            s[col] = sv;
            inv_s[col] = __fdiv_rn(1.0f, sv);
        }
    }
}

__global__ void debug_e2m1_kernel(const float *t, int64_t n, uint8_t *codes)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) codes[i] = static_cast<uint8_t>(e2m1x2(t[i], 0.0f) & 0xf);
}

}  // namespace

cudaError_t launch_quant(QuantMode mode, const QuantArgs &a, cudaStream_t stream)
{
    const int64_t nkb_pad = pad_scale_cols(a.K);
    // lanes per CTA: a multiple of 32 covering nkb_pad in as few slabs as
    // possible with the least idle lanes (at most 256 lanes per CTA)
    int64_t best_t = 32, best_waste = -1;
    const int64_t min_slabs = (nkb_pad + 255) / 256;
    for (int64_t slabs = min_slabs; slabs <= min_slabs + 4; ++slabs) {
        const int64_t t = ((nkb_pad + slabs - 1) / slabs + 31) / 32 * 32;
        const int64_t waste = t * slabs - nkb_pad;
        if (t <= 256 && (best_waste < 0 || waste < best_waste)) {
            best_waste = waste;
            best_t = t;
        }
    }
    const int64_t slabs = (nkb_pad + best_t - 1) / best_t;
    // rows per CTA: aim for about 8 resident-CTA waves worth of work items
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t target_ctas = static_cast<int64_t>(sms) * 8;
    int64_t rows_per_cta = (a.rows_out * slabs + target_ctas - 1) / target_ctas;
    rows_per_cta = rows_per_cta < 2 ? 2 : rows_per_cta;
    rows_per_cta = rows_per_cta > 64 ? 64 : rows_per_cta;
    rows_per_cta = (rows_per_cta + 1) / 2 * 2;
    const int64_t row_ctas = (a.rows_out + rows_per_cta - 1) / rows_per_cta;
    if (row_ctas > 65535) {
        rows_per_cta = (a.rows_out + 65534) / 65535;
        rows_per_cta = (rows_per_cta + 1) / 2 * 2;
    }
    dim3 grid(static_cast<unsigned>(slabs),
              static_cast<unsigned>((a.rows_out + rows_per_cta - 1) / rows_per_cta));
    dim3 block(static_cast<unsigned>(best_t));
    const bool wide = (reinterpret_cast<uintptr_t>(a.src) % 32 == 0) && ((a.ld_src * 2) % 32 == 0);
#define MACAQ_LAUNCH_QUANT(M)                                                              \
    if (wide)                                                                              \
        quant_kernel<M, true><<<grid, block, 0, stream>>>(a, rows_per_cta);                \
    else                                                                                   \
        quant_kernel<M, false><<<grid, block, 0, stream>>>(a, rows_per_cta);
    switch (mode) {
    case QuantMode::Dense:
        MACAQ_LAUNCH_QUANT(QuantMode::Dense)
        break;
    case QuantMode::WeightGrouped:
        MACAQ_LAUNCH_QUANT(QuantMode::WeightGrouped)
        break;
    case QuantMode::ActGrouped:
        MACAQ_LAUNCH_QUANT(QuantMode::ActGrouped)
        break;
    }
#undef MACAQ_LAUNCH_QUANT
    return cudaGetLastError();
}

cudaError_t launch_balance(const uint16_t *xc, int64_t ldxc, const int32_t *xc_rows, int64_t mc,
                           const uint16_t *w, int64_t n, int64_t k, float *s, float *inv_s,
                           cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>((k + 63) / 64));
    balance_kernel<<<grid, 256, 0, stream>>>(xc, ldxc, xc_rows, mc, w, n, k, s, inv_s);
    return cudaGetLastError();
}

cudaError_t launch_debug_e2m1(const float *t, int64_t n, uint8_t *codes, cudaStream_t stream)
{
    const int64_t blocks = (n + 255) / 256;
    debug_e2m1_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(t, n, codes);
    return cudaGetLastError();
}

}  // namespace macaq
