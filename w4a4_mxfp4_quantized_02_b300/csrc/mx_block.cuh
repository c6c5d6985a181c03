// The per-block arithmetic of the activation transform, shared by the
// transform kernels and the GEMM epilogue that writes MXFP4 directly: the
// balance multiply, the 32-point (and 64-point) Hadamard butterflies, the E8M0
// scale and the E2M1 encode, and the SwiGLU step h = bf16(SiLU(g) * u).
//
// MACaQ page "What is MACaQ quantization", section "How MACaQ works": a
// per-channel scale balances the input channels and a block Hadamard over 32
// channels spreads outliers before the values are stored as MXFP4 (FAQ "What
// is W4A4 quantization": 4-bit floats in blocks of 32 sharing one scale).
//
// Every arithmetic step is an explicitly rounded intrinsic, and no packed
// multiply ever feeds a packed add (the code generator would contract the pair
// into one fused multiply-add whatever the flags), so any unit that includes
// this header computes the same bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace macaq {
namespace mx {

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

// ------------------------------------------------------------- SwiGLU step
//
// h = bf16( SiLU(g) * u ), SiLU(g) = g / (1 + e^-g), the value an unfused
// layer would store.  In fp32, every operation rounded to nearest (every fused
// multiply-add explicit):
//   e^x, x = -g: Cody-Waite range reduction x = n ln2 + r (ln2 split into a
//     16-bit head, so n * head is exact, and a tail; both steps fused
//     multiply-adds), the Taylor series of e^r to r^8 / 8! by Horner with
//     fused multiply-adds (|r| <= 0.35, truncation below 2^-30 relative),
//     then one multiply by 2^n (x clamped to [-87, 88] so that 2^n is a
//     normal float; below -87, e^x no longer changes 1 + e^x; above the fp32
//     overflow point 88.72 it is taken as infinite, so SiLU(g) = -0);
//   1 / (1 + e^x): the hardware reciprocal estimate refined by one
//     Newton-Raphson step r <- r + r (1 - d r);
//   SiLU(g) = g * r, then times u, then rounded once to bf16.
// Relative error before the bf16 rounding, for g >= -80: at most about
// 2 + 0.5 + 1 + 0.5 + 0.5 = 4.5 fp32 ulps (below 2^-20.8), so the result can
// differ from the exactly rounded h only where the exact value lies that close
// to a bf16 rounding boundary.  The two elements of a bf16 word go through
// the polynomial as one packed pair.
__device__ __forceinline__ float pow2i(int k)  // 2^k, -126 <= k <= 127
{
    return __int_as_float((k + 127) << 23);
}

__device__ __forceinline__ float rcp_estimate(float d)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// 1 / d for 1 <= d < inf: the estimate and one Newton-Raphson step
__device__ __forceinline__ float recip_nr(float d)
{
    const float r0 = rcp_estimate(d);
    const float e1 = __fmaf_rn(-d, r0, 1.0f);
    return __fmaf_rn(r0, e1, r0);
}

// e^x for the two elements of a pair, x clamped to [-87, 88]
__device__ __forceinline__ float2 exp_f32x2(float2 x)
{
    const float2 xc = make_float2(fminf(fmaxf(x.x, -87.0f), 88.0f), fminf(fmaxf(x.y, -87.0f), 88.0f));
    const float2 t = __fmul2_rn(xc, make_float2(0x1.715476p+0f, 0x1.715476p+0f));
    const float2 fn = make_float2(rintf(t.x), rintf(t.y));
    const float2 nfn = make_float2(-fn.x, -fn.y);
    float2 r = __ffma2_rn(nfn, make_float2(0x1.62e4p-1f, 0x1.62e4p-1f), xc);
    r = __ffma2_rn(nfn, make_float2(0x1.7f7d1cp-20f, 0x1.7f7d1cp-20f), r);
    float2 q = make_float2(0x1.a01a02p-16f, 0x1.a01a02p-16f);
    q = __ffma2_rn(q, r, make_float2(0x1.a01a02p-13f, 0x1.a01a02p-13f));
    q = __ffma2_rn(q, r, make_float2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    q = __ffma2_rn(q, r, make_float2(0x1.111112p-7f, 0x1.111112p-7f));
    q = __ffma2_rn(q, r, make_float2(0x1.555556p-5f, 0x1.555556p-5f));
    q = __ffma2_rn(q, r, make_float2(0x1.555556p-3f, 0x1.555556p-3f));
    q = __ffma2_rn(q, r, make_float2(0x1.0p-1f, 0x1.0p-1f));
    q = __ffma2_rn(q, r, make_float2(0x1.0p+0f, 0x1.0p+0f));
    q = __ffma2_rn(q, r, make_float2(0x1.0p+0f, 0x1.0p+0f));
    return __fmul2_rn(q, make_float2(pow2i(static_cast<int>(fn.x)), pow2i(static_cast<int>(fn.y))));
}

// Two bf16 words of gate and up values -> the word of the two h values
// (element 2i in the low half).
__device__ __forceinline__ uint32_t silu_mul_word(uint32_t gw, uint32_t uw)
{
    const float2 g = make_float2(bf16lo(gw), bf16hi(gw));
    const float2 e = exp_f32x2(make_float2(-g.x, -g.y));
    const float dx = __fadd_rn(1.0f, e.x), dy = __fadd_rn(1.0f, e.y);
    // beyond the overflow point of e^-g the quotient is a signed zero
    const float rx = (-g.x > 88.72283935546875f) ? 0.0f : recip_nr(dx);
    const float ry = (-g.y > 88.72283935546875f) ? 0.0f : recip_nr(dy);
    const float2 sl = __fmul2_rn(g, make_float2(rx, ry));
    // a product feeding another product (no add): no contraction possible
    const float2 p = __fmul2_rn(sl, make_float2(bf16lo(uw), bf16hi(uw)));
    const __nv_bfloat162 h = __floats2bfloat162_rn(p.x, p.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The same transform as quant_block with the natural register pairing
// v[i] = (element 2i, element 2i+1): the stride-1 stage (fed by products, so
// scalar) pairs the halves of a register, strides 2, 4, 8, 16 pair whole
// registers i and i + h/2 and run as packed adds; the bf16 words and the
// output bytes already come in this pairing.
//
// kH64: the block is one half of a 64-channel Hadamard block whose other half
// is held by the neighbouring lane (lane ^ 1; the even lane holds the lower
// half).  After the five 32-point stages the stride-32 stage pairs element i
// of the two halves through a shuffle, and the normalisation is the exact
// 1/8; the MX block stays these 32 values.
// Packed fp32x2 subtraction, each lane rounded to nearest.
__device__ __forceinline__ float2 fsub2_rn(float2 a, float2 b)
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

__device__ __forceinline__ float max3_f32(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <bool kH64>
__device__ __forceinline__ void hadamard_block_pairs(const uint32_t (&raw)[16], const float2 (&f)[16],
                                                     float2 (&v)[16])
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        // one packed multiply for the pair; the stride-1 stage that consumes it
        // is scalar, so no packed add follows a packed multiply here
        const float2 ab = __fmul2_rn(make_float2(bf16lo(raw[i]), bf16hi(raw[i])), f[i]);
        v[i] = make_float2(__fadd_rn(ab.x, ab.y), __fsub_rn(ab.x, ab.y));
    }
#pragma unroll
    for (int hh = 1; hh < 16; hh <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & hh) continue;
            const float2 a = v[i];
            const float2 b = v[i + hh];
            // sums of sums: no multiply feeds these adds, so the packed
            // intrinsics cannot be contracted into an FMA
            v[i] = __fadd2_rn(a, b);
            v[i + hh] = fsub2_rn(a, b);
        }
    }
    if (kH64) {
        const unsigned mask = __activemask();
        // lower half: own + partner; upper half: partner - own.  As p + sgn * v
        // with sgn = +-1 the product is exact, so one fused multiply-add gives
        // exactly the rounded sum or difference.
        const float sgn = (threadIdx.x & 1u) ? -1.0f : 1.0f;
        const float2 sgn2 = make_float2(sgn, sgn);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 p = make_float2(__shfl_xor_sync(mask, v[i].x, 1), __shfl_xor_sync(mask, v[i].y, 1));
            v[i] = __ffma2_rn(sgn2, v[i], p);
        }
    }
}

// The W4A16 activation: the normalised transform rounded once to bf16
// (element 2i in the low half of word i).
// The 32-channel transform with the block maximum of |v| taken from the last
// butterfly stage: for its pairs (a, b) -> (a + b, a - b), max(|RN(a + b)|,
// |RN(a - b)|) = RN(|a| + |b|) because rounding to nearest is monotone and
// symmetric, so eight packed adds of magnitudes and a short max chain give the
// maximum of all 32 outputs exactly.
__device__ __forceinline__ float hadamard32_pairs_amax(const uint32_t (&raw)[16], const float2 (&f)[16],
                                                       float2 (&v)[16])
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 ab = __fmul2_rn(make_float2(bf16lo(raw[i]), bf16hi(raw[i])), f[i]);
        v[i] = make_float2(__fadd_rn(ab.x, ab.y), __fsub_rn(ab.x, ab.y));
    }
#pragma unroll
    for (int hh = 1; hh < 8; hh <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & hh) continue;
            const float2 a = v[i];
            const float2 b = v[i + hh];
            v[i] = __fadd2_rn(a, b);
            v[i + hh] = fsub2_rn(a, b);
        }
    }
    float2 t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 a = v[i];
        const float2 b = v[i + 8];
        v[i] = __fadd2_rn(a, b);
        v[i + 8] = fsub2_rn(a, b);
        t[i] = __fadd2_rn(make_float2(fabsf(a.x), fabsf(a.y)), make_float2(fabsf(b.x), fabsf(b.y)));
    }
    float m = max3_f32(t[0].x, t[0].y, t[1].x);
    m = max3_f32(m, t[1].y, t[2].x);
    m = max3_f32(m, t[2].y, t[3].x);
    m = max3_f32(m, t[3].y, t[4].x);
    m = max3_f32(m, t[4].y, t[5].x);
    m = max3_f32(m, t[5].y, t[6].x);
    m = max3_f32(m, t[6].y, t[7].x);
    return fmaxf(m, t[7].y);
}

template <bool kH64>
__device__ __forceinline__ void bf16_block_pairs(const uint32_t (&raw)[16], const float2 (&f)[16],
                                                 uint32_t (&out)[16])
{
    constexpr float kNorm = kH64 ? 0.125f : kInvSqrt32;
    float2 v[16];
    hadamard_block_pairs<kH64>(raw, f, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 y = __fmul2_rn(v[i], make_float2(kNorm, kNorm));
        const __nv_bfloat162 b = __floats2bfloat162_rn(y.x, y.y);
        out[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
}

// Scale and encode one 32-element block held as v[i] = (element 2i,
// element 2i+1) after the butterflies (unnormalised): the block maximum, the
// E8M0 byte, the normalise-and-scale multiply and the E2M1 codes (element 2i
// in the low nibble of byte i).  kH64: the 64-channel normalisation 1/8.
// The same with the block maximum of |v| already known.
template <bool kH64>
__device__ __forceinline__ uint32_t encode_block_pairs_vmax(float2 (&v)[16], float vmax, uint4 &codes)
{
    constexpr float kNorm = kH64 ? 0.125f : kInvSqrt32;
    const float amax = __fmul_rn(vmax, kNorm);
    const int ef = static_cast<int>(__float_as_uint(amax) >> 23);
    const uint32_t sbyte = static_cast<uint32_t>(ef > 2 ? ef - 2 : 0);
    const int se = static_cast<int>(sbyte) - 127;
    if (se >= -124 && se <= 122) {
        const float g = __int_as_float(__float_as_int(kNorm) - se * (1 << 23));
        const float2 g2 = make_float2(g, g);
        // the scaled values feed only the encoder: no add follows this multiply
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __fmul2_rn(v[i], g2);
    } else {
        const float c = kNorm;
        const float inv = __uint_as_float((254u - sbyte) << 23);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = __fmul2_rn(v[i], make_float2(c, c));
            v[i] = __fmul2_rn(v[i], make_float2(inv, inv));
        }
    }
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t b0 = e2m1x2(v[4 * q].x, v[4 * q].y);
        const uint32_t b1 = e2m1x2(v[4 * q + 1].x, v[4 * q + 1].y);
        const uint32_t b2 = e2m1x2(v[4 * q + 2].x, v[4 * q + 2].y);
        const uint32_t b3 = e2m1x2(v[4 * q + 3].x, v[4 * q + 3].y);
        w[q] = __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
    }
    codes = make_uint4(w[0], w[1], w[2], w[3]);
    return sbyte;
}

template <bool kH64>
__device__ __forceinline__ uint32_t encode_block_pairs(float2 (&v)[16], uint4 &codes)
{
    float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        m0 = fmaxf(m0, fabsf(v[i].x));
        m1 = fmaxf(m1, fabsf(v[i].y));
    }
    return encode_block_pairs_vmax<kH64>(v, fmaxf(m0, m1), codes);
}

template <bool kH64>
__device__ __forceinline__ uint32_t quant_block_pairs(const uint32_t (&raw)[16], const float2 (&f)[16],
                                                      uint4 &codes)
{
    float2 v[16];
    if constexpr (kH64) {
        hadamard_block_pairs<kH64>(raw, f, v);
        return encode_block_pairs<kH64>(v, codes);
    } else {
        const float vmax = hadamard32_pairs_amax(raw, f, v);
        return encode_block_pairs_vmax<false>(v, vmax, codes);
    }
}

// A whole 64-channel Hadamard block held by one thread (two MX blocks): the
// 32-point butterflies of each half, then the stride-32 stage between the
// halves (lower: a + b, upper: a - b, each one rounding -- the same values
// the lane-pair form above forms through a shuffle), then each half scaled and
// encoded as its own MX block with the exact 1/8 normalisation.
__device__ __forceinline__ void quant_block64_pairs(const uint32_t (&raw_lo)[16], const uint32_t (&raw_hi)[16],
                                                    const float2 (&f_lo)[16], const float2 (&f_hi)[16],
                                                    uint4 &codes_lo, uint4 &codes_hi, uint32_t &s_lo,
                                                    uint32_t &s_hi)
{
    float2 lo[16], hi[16];
    hadamard_block_pairs<false>(raw_lo, f_lo, lo);
    hadamard_block_pairs<false>(raw_hi, f_hi, hi);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 a = lo[i];
        const float2 b = hi[i];
        lo[i] = __fadd2_rn(a, b);
        hi[i] = __fadd2_rn(a, make_float2(-b.x, -b.y));
    }
    s_lo = encode_block_pairs<true>(lo, codes_lo);
    s_hi = encode_block_pairs<true>(hi, codes_hi);
}

}  // namespace mx
}  // namespace macaq
