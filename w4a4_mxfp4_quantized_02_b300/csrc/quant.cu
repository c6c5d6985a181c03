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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "mx_block.cuh"
#include "ptx.cuh"

namespace macaq {

// Set when a wait in a quantisation kernel runs out (reported through
// macaq_check_device_error).
__device__ unsigned int g_quant_error_flags;

namespace {

using namespace mx;

constexpr uint64_t kQuantWaitNs = 2000000000ull;

// Bounded wait on a TMA barrier; false (and the error flag) after kQuantWaitNs.
__device__ __forceinline__ bool quant_wait(uint32_t bar, uint32_t parity)
{
    if (ptx::mbar_try_wait(bar, parity, 100000)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity, 100000)) return true;
        if (ptx::globaltimer() - t0 > kQuantWaitNs) {
            atomicOr(&g_quant_error_flags, 1u);
            return false;
        }
    }
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
    // launched with programmatic stream serialisation: wait for the previous
    // kernel before touching memory, then let the next kernel start (after the
    // wait: see the dense TMA kernel)
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
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


// ------------------------------------------------ TMA-staged dense variant

// Dense rows through a TMA ring.  X is viewed as [rows][blocks][32 values];
// one box per stage brings RT rows x TB blocks (64 bytes each, 64-byte
// swizzle so the four 16-byte reads of 8 neighbouring threads hit distinct
// banks) into shared memory.  Consumer thread c = ty * TB + tx owns block tx
// of the slab in row ty of every group of RT rows and keeps its 32 balance
// factors in registers; the last warp only issues the loads, STAGES groups
// ahead.  Warps run decoupled: each consumer warp waits on a stage's "full"
// barrier through one lane and releases it on the stage's "empty" barrier.
// Consumer threads of a TMA transform CTA (plus one producer warp): 20 warps,
// 96 registers each, so the warps of the one resident CTA hide more latency.
constexpr int kTmaConsumersMax = 640;
constexpr int kTmaThreadsMax = kTmaConsumersMax + 32;
// The grouped kernel takes its balance factors from a shared-memory table of
// the first experts of its rows (up to four, as shared memory allows; L1 for
// any further expert): up to 20 consumer warps, as the dense kernel; 16 when
// it also forms the SwiGLU step (more registers per thread).
__host__ __device__ constexpr int grouped_consumers_max(bool silu) { return silu ? 512 : 640; }
constexpr int kGroupedFacSlotsMax = 4;

// kOut: kOutMx writes MXFP4 codes and scales; kOutBf16 the normalised
// transform as bf16 (the W4A16 activation) to a.codes viewed as bf16
// [rows, ld_out]; kOutF32 the same values in fp32 (the rotated rows Flip
// Refinement works on) to a.codes viewed as float [rows, ld_out].
template <int STAGES, bool kH64, int kOut>
__global__ void __launch_bounds__(kTmaThreadsMax, 1) quant_dense_tma_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                  QuantArgs a, int32_t groups, int32_t TB,
                                                                  int32_t RT)
{
    extern __shared__ uint8_t qsmem_raw[];
    const uint32_t raw_base = ptx::smem_u32(qsmem_raw);
    uint8_t *qsmem = qsmem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(qsmem);
    const int NC = TB * RT;  // consumer threads
    const int cwarps = NC / 32;
    const uint32_t stage_bytes = static_cast<uint32_t>(NC * 64);
    const uint32_t full0 = sbase + STAGES * stage_bytes;
    const uint32_t empty0 = full0 + 8 * STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(qsmem + STAGES * stage_bytes + 16 * STAGES);
    // the slab's balance factors: block tx's 32 floats at 128 * tx, its 16-byte
    // chunk c stored at position (c + tx) mod 8 (conflict-free reads)
    const uint32_t ftab = sbase + STAGES * stage_bytes + 16 * STAGES + 16;
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int32_t slab0 = static_cast<int32_t>(blockIdx.x) * TB;

    if (t == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, static_cast<uint32_t>(cwarps));
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // launched with programmatic stream serialisation: wait for the previous
    // kernel (which may produce X or still read the codes) before touching
    // global memory, and only then let the next kernel start -- so a GEMM
    // launched right after a transform starts only once everything before the
    // transform has completed, and may load its weight before its own wait
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    const int32_t my_groups = blockIdx.y < static_cast<uint32_t>(groups)
                                  ? (groups - 1 - static_cast<int32_t>(blockIdx.y)) / static_cast<int32_t>(gridDim.y) + 1
                                  : 0;

    if (t >= NC) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            int32_t j = 0;
            for (; j < my_groups; ++j) {
                const int s = j % STAGES;
                if (j >= STAGES && !quant_wait(empty0 + 8 * s, static_cast<uint32_t>(j / STAGES - 1) & 1u)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int32_t g = static_cast<int32_t>(blockIdx.y) + j * static_cast<int32_t>(gridDim.y);
                ptx::mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes);
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(sbase + s * stage_bytes),
                    "l"(&tmX), "r"(full0 + 8 * s), "r"(0), "r"(slab0), "r"(g * RT)
                    : "memory");
            }
            // every issued copy must land before the CTA exits
            for (int32_t k = (j > STAGES ? j - STAGES : 0); k < j; ++k)
                quant_wait(full0 + 8 * (k % STAGES), static_cast<uint32_t>(k / STAGES) & 1u);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    // The consumers fill the balance-factor table while the producer's first
    // copies are in flight, and sync among themselves on a named barrier.
    for (int idx = t; idx < TB * 8; idx += NC) {
        const int bx = idx >> 3, c = idx & 7;
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (slab0 + bx < a.K / 32) v4 = __ldg(reinterpret_cast<const float4 *>(a.f + 32 * (slab0 + bx)) + c);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ftab + 128 * bx + 16 * ((c + bx) & 7)),
                     "f"(v4.x), "f"(v4.y), "f"(v4.z), "f"(v4.w)
                     : "memory");
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory");
    const int tx = t % TB, ty = t / TB;
    const int64_t nkb = a.K / 32;
    const int64_t nka = ((nkb + 7) / 8 * 8) / 4;
    const int64_t nkb_pad = nka * 4;
    const int64_t kb = static_cast<int64_t>(slab0) + tx;
    const bool has_kb = kb < nkb;
    const bool writes_scale = (lane & 3) == 0 && kb < nkb_pad;
    const uint32_t fbase = ftab + 128 * tx;
    const uint32_t swz = (static_cast<uint32_t>(t) >> 1) & 3u;  // 64-byte row t of a stage
    const int64_t half_k = a.K / 2;

    for (int32_t j = 0; j < my_groups; ++j) {
        const int s = j % STAGES;
        int ok = 1;
        if (lane == 0) {
            ok = quant_wait(full0 + 8 * s, static_cast<uint32_t>(j / STAGES) & 1u) ? 1 : 0;
            if (!ok) *abort_flag = 1;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int32_t g = static_cast<int32_t>(blockIdx.y) + j * static_cast<int32_t>(gridDim.y);
        const int64_t r = static_cast<int64_t>(g) * RT + ty;  // row (padded space)
        uint32_t sbyte = 0;
        if (r < a.rows_valid && has_kb) {
            uint32_t raw[16];
            const uint32_t base = sbase + s * stage_bytes + static_cast<uint32_t>(t) * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t x0, x1, x2, x3;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                             : "r"(base + 16 * (c ^ swz)));
                raw[4 * c] = x0;
                raw[4 * c + 1] = x1;
                raw[4 * c + 2] = x2;
                raw[4 * c + 3] = x3;
            }
            // the stage is no longer needed by this warp once its reads are done
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty0 + 8 * s);
            float2 f[16];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float x0, x1, x2, x3;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(x0), "=f"(x1), "=f"(x2), "=f"(x3)
                             : "r"(fbase + 16 * ((c + tx) & 7)));
                f[2 * c] = make_float2(x0, x1);
                f[2 * c + 1] = make_float2(x2, x3);
            }
            if (kOut == kOutBf16) {
                // W4A16: the bf16 transform, 64 bytes of row r at block kb
                uint32_t w[16];
                bf16_block_pairs<kH64>(raw, f, w);
                uint4 *dst = reinterpret_cast<uint4 *>(a.codes + (r * a.ld_out + 32 * kb) * 2);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            } else if (kOut == kOutF32) {
                // the fp32 transform, 128 bytes of row r at block kb
                constexpr float kNorm = kH64 ? 0.125f : kInvSqrt32;
                float2 v[16];
                hadamard_block_pairs<kH64>(raw, f, v);
                float4 *dst = reinterpret_cast<float4 *>(a.codes + (r * a.ld_out + 32 * kb) * 4);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float2 y0 = __fmul2_rn(v[2 * q], make_float2(kNorm, kNorm));
                    const float2 y1 = __fmul2_rn(v[2 * q + 1], make_float2(kNorm, kNorm));
                    dst[q] = make_float4(y0.x, y0.y, y1.x, y1.y);
                }
            } else {
                uint4 codes;
                sbyte = quant_block_pairs<kH64>(raw, f, codes);
                *reinterpret_cast<uint4 *>(a.codes + r * half_k + 16 * kb) = codes;
            }
        } else {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty0 + 8 * s);
        }
        if (kOut != kOutMx) continue;
        uint32_t word = sbyte << (8 * (lane & 3));
        word |= __shfl_xor_sync(0xffffffffu, word, 1);
        word |= __shfl_xor_sync(0xffffffffu, word, 2);
        if (writes_scale && r < a.rows_out) {
            const int64_t off = ((r / 128) * nka + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4;
            *reinterpret_cast<uint32_t *>(a.scales + off) = word;
        }
    }
}

// ------------------------------------------- TMA-staged grouped activations
//
// The expert-grouped activation transform (MoE): output row p of the
// expert-padded layout takes token row row_src[offsets[e] + j] (e = the
// expert whose padded range holds p, j = p - its first padded row) through
// the transform with that expert's balance factors; padding rows get zero
// scales and no codes.  The stage layout and the consumer are those of the
// dense kernel; the producer lands each row of a stage with its own TMA box
// (one row high), so the rows can come from anywhere in X.  Only the experts'
// real rows run through the pipeline (padding is a fifth of the padded rows
// at 4096 tokens x top-8 of 128 experts); each CTA resolves its rows (token
// row, expert, padded destination row) once, up front, into a table in
// shared memory, and afterwards writes the zero scales of padding rows.
// kSilu: the rows are the sorted rows of a [rows, 2F] gate|up matrix; each
// stage lands the gate and the up slab of every row and the consumer forms
// h = SiLU(g) * u before the transform.

template <int STAGES, bool kSilu, bool kH64>
__global__ void __launch_bounds__(grouped_consumers_max(kSilu) + 32, 1) quant_grouped_tma_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                    QuantArgs a, int32_t groups, int32_t TB,
                                                                    int32_t RT, int32_t per_cta, int32_t fac_slots)
{
    extern __shared__ uint8_t qsmem_raw[];
    const uint32_t raw_base = ptx::smem_u32(qsmem_raw);
    uint8_t *qsmem = qsmem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(qsmem);
    const int NC = TB * RT;
    const int cwarps = NC / 32;
    const uint32_t row_bytes = static_cast<uint32_t>(TB * 64);
    const uint32_t stage_bytes = static_cast<uint32_t>(NC * 64) * (kSilu ? 2u : 1u);
    const uint32_t full0 = sbase + STAGES * stage_bytes;
    const uint32_t empty0 = full0 + 8 * STAGES;
    uint8_t *misc = qsmem + STAGES * stage_bytes + 16 * STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc);
    int32_t *s_off = reinterpret_cast<int32_t *>(misc + 16);
    int32_t *s_poff = s_off + (kMaxExperts + 1);
    int32_t *m_src = s_poff + (kMaxExperts + 1);  // token row, -2 past the end
    int32_t *m_exp = m_src + per_cta * RT;
    int32_t *m_dst = m_exp + per_cta * RT;        // padded output row
    // factor table: slot x TB blocks x 32 floats, block bx's 16-byte chunk c at
    // position (c + bx) mod 8 (conflict-free reads)
    const uint32_t ftab = (ptx::smem_u32(m_dst + per_cta * RT) + 15u) & ~15u;
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int32_t slab0 = static_cast<int32_t>(blockIdx.x) * TB;

    if (t == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, static_cast<uint32_t>(cwarps));
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    // no offsets: one group of all rows (the dense SwiGLU input)
    for (int e = t; e <= a.E; e += blockDim.x)
        s_off[e] = a.offsets ? a.offsets[e] : (e == 0 ? 0 : static_cast<int32_t>(a.rows_valid));
    __syncthreads();
    if (t == 0) {
        int32_t acc = 0;
        s_poff[0] = 0;
        for (int e = 0; e < a.E; ++e) {
            acc += (s_off[e + 1] - s_off[e] + 127) / 128 * 128;
            s_poff[e + 1] = acc;
        }
    }
    __syncthreads();

    // A contiguous range of row groups per CTA (consecutive rows mostly share
    // an expert, so the balance factors are reloaded rarely), dealt over the
    // experts' real rows in sorted order; padding rows and the rest of the
    // padded capacity only need zero scales, written after the pipeline.
    const int64_t used = s_poff[a.E];
    const int64_t r0 = s_off[0], nreal = static_cast<int64_t>(s_off[a.E]) - s_off[0];
    const int32_t groups_real = static_cast<int32_t>((nreal + RT - 1) / RT);
    const int32_t per = (groups_real + static_cast<int32_t>(gridDim.y) - 1) / static_cast<int32_t>(gridDim.y);
    const int32_t g0 = static_cast<int32_t>(blockIdx.y) * per;
    const int32_t my_groups = g0 < groups_real ? min(per, groups_real - g0) : 0;
    (void)groups;
    (void)per_cta;
    // row i of local group j is sorted row r0 + (g0 + j) * RT + i
    for (int idx = t; idx < my_groups * RT; idx += blockDim.x) {
        const int j = idx / RT, i = idx - (idx / RT) * RT;
        const int64_t r = r0 + (static_cast<int64_t>(g0) + j) * RT + i;
        int32_t src = -2, ex = 0, dst = -1;
        if (r < s_off[a.E]) {
            int lo = 0, hi = a.E;  // s_off[lo] <= r < s_off[lo + 1] (the last such expert)
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= r) lo = mid; else hi = mid;
            }
            ex = lo;
            dst = static_cast<int32_t>(s_poff[lo] + (r - s_off[lo]));
            src = kSilu ? static_cast<int32_t>(r) : a.row_src[r];
        }
        m_src[idx] = src;
        m_exp[idx] = ex;
        m_dst[idx] = dst;
    }
    __syncthreads();

    if (t >= NC) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            int32_t j = 0;
            for (; j < my_groups; ++j) {
                const int s = j % STAGES;
                if (j >= STAGES && !quant_wait(empty0 + 8 * s, static_cast<uint32_t>(j / STAGES - 1) & 1u)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                uint32_t nvalid = 0;
                for (int i = 0; i < RT; ++i) nvalid += m_src[j * RT + i] >= 0 ? 1u : 0u;
                ptx::mbar_arrive_expect_tx(full0 + 8 * s, nvalid * row_bytes * (kSilu ? 2u : 1u));
                for (int i = 0; i < RT; ++i) {
                    const int32_t src = m_src[j * RT + i];
                    if (src < 0) continue;
                    asm volatile(
                        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(sbase + s * stage_bytes + i * row_bytes),
                        "l"(&tmX), "r"(full0 + 8 * s), "r"(0), "r"(slab0), "r"(src)
                        : "memory");
                    if (kSilu) {
                        // the up slab: K / 32 blocks further along the row
                        asm volatile(
                            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                            " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(sbase + s * stage_bytes + (RT + i) * row_bytes),
                            "l"(&tmX), "r"(full0 + 8 * s), "r"(0), "r"(slab0 + static_cast<int32_t>(a.K / 32)),
                            "r"(src)
                            : "memory");
                    }
                }
            }
            for (int32_t k = (j > STAGES ? j - STAGES : 0); k < j; ++k)
                quant_wait(full0 + 8 * (k % STAGES), static_cast<uint32_t>(k / STAGES) & 1u);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int tx = t % TB, ty = t / TB;
    const int64_t nkb = a.K / 32;
    const int64_t nka = ((nkb + 7) / 8 * 8) / 4;
    const int64_t nkb_pad = nka * 4;
    const int64_t kb = static_cast<int64_t>(slab0) + tx;
    const bool has_kb = kb < nkb;
    const bool writes_scale = (lane & 3) == 0 && kb < nkb_pad;
    const uint32_t swz = (static_cast<uint32_t>(t) >> 1) & 3u;
    const int64_t half_k = a.K / 2;
    // the factors of this CTA's first experts (its rows are sorted by expert),
    // filled while the producer's first copies are in flight
    const int32_t e_lo = my_groups > 0 ? m_exp[0] : 0;
    for (int idx = t; idx < fac_slots * TB * 8; idx += NC) {
        const int slot = idx / (TB * 8), rem = idx - slot * (TB * 8);
        const int bx = rem >> 3, c = rem & 7;
        const int32_t e = e_lo + slot;
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < a.E && slab0 + bx < nkb)
            v4 = __ldg(reinterpret_cast<const float4 *>(a.f + static_cast<int64_t>(e) * a.K + 32 * (slab0 + bx)) + c);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                         ftab + static_cast<uint32_t>(slot * TB * 128 + 128 * bx + 16 * ((c + bx) & 7))),
                     "f"(v4.x), "f"(v4.y), "f"(v4.z), "f"(v4.w)
                     : "memory");
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NC) : "memory");

    for (int32_t j = 0; j < my_groups; ++j) {
        const int s = j % STAGES;
        int ok = 1;
        if (lane == 0) {
            ok = quant_wait(full0 + 8 * s, static_cast<uint32_t>(j / STAGES) & 1u) ? 1 : 0;
            if (!ok) *abort_flag = 1;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int32_t src = m_src[j * RT + ty];
        const int32_t ex = m_exp[j * RT + ty];
        const int64_t p = m_dst[j * RT + ty];
        uint32_t sbyte = 0;
        const bool valid = src >= 0 && has_kb;
        uint32_t raw[16];
        uint32_t up[kSilu ? 16 : 1];
        if (valid) {
            const uint32_t base = sbase + s * stage_bytes + static_cast<uint32_t>(t) * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t x0, x1, x2, x3;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                             : "r"(base + 16 * (c ^ swz)));
                raw[4 * c] = x0;
                raw[4 * c + 1] = x1;
                raw[4 * c + 2] = x2;
                raw[4 * c + 3] = x3;
            }
            if (kSilu) {
                // the up slab sits NC rows of 64 bytes later (same swizzle phase)
                const uint32_t ubase = base + static_cast<uint32_t>(NC) * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t x0, x1, x2, x3;
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                                 : "r"(ubase + 16 * (c ^ swz)));
                    up[4 * c] = x0;
                    up[4 * c + 1] = x1;
                    up[4 * c + 2] = x2;
                    up[4 * c + 3] = x3;
                }
            }
        }
        // the stage is no longer needed by this warp once its reads are done
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty0 + 8 * s);
        if (valid) {
            if (kSilu) {
#pragma unroll
                for (int i = 0; i < 16; ++i) raw[i] = silu_mul_word(raw[i], up[i]);
            }
            // the row's expert factors: from the table, or from L1 for an
            // expert past the table's slots
            float2 f[16];
            const int slot = ex - e_lo;
            if (slot < fac_slots) {
                const uint32_t fb = ftab + static_cast<uint32_t>(slot * TB * 128 + 128 * tx);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x0, x1, x2, x3;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(x0), "=f"(x1), "=f"(x2), "=f"(x3)
                                 : "r"(fb + 16 * ((c + tx) & 7)));
                    f[2 * c] = make_float2(x0, x1);
                    f[2 * c + 1] = make_float2(x2, x3);
                }
            } else {
                const float4 *f4 = reinterpret_cast<const float4 *>(a.f + static_cast<int64_t>(ex) * a.K + 32 * kb);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v4 = __ldg(f4 + q);
                    f[2 * q] = make_float2(v4.x, v4.y);
                    f[2 * q + 1] = make_float2(v4.z, v4.w);
                }
            }
            uint4 codes;
            sbyte = quant_block_pairs<kH64>(raw, f, codes);
            *reinterpret_cast<uint4 *>(a.codes + p * half_k + 16 * kb) = codes;
        }
        uint32_t word = sbyte << (8 * (lane & 3));
        word |= __shfl_xor_sync(0xffffffffu, word, 1);
        word |= __shfl_xor_sync(0xffffffffu, word, 2);
        if (writes_scale && src >= 0) {
            const int64_t off = ((p / 128) * nka + kb / 4) * 512 + (p % 32) * 16 + ((p % 128) / 32) * 4;
            *reinterpret_cast<uint32_t *>(a.scales + off) = word;
        }
    }
    // zero scales for the padding rows of this CTA's experts ...
    if (writes_scale) {
        for (int e = static_cast<int>(blockIdx.y); e < a.E; e += static_cast<int>(gridDim.y)) {
            for (int64_t p = static_cast<int64_t>(s_poff[e]) + (s_off[e + 1] - s_off[e]) + ty; p < s_poff[e + 1];
                 p += RT) {
                const int64_t off = ((p / 128) * nka + kb / 4) * 512 + (p % 32) * 16 + ((p % 128) / 32) * 4;
                *reinterpret_cast<uint32_t *>(a.scales + off) = 0u;
            }
        }
    }
    // ... and for the padded capacity past the experts' rows
    if (writes_scale) {
        for (int64_t p = used + static_cast<int64_t>(blockIdx.y) * RT + ty; p < a.rows_out;
             p += static_cast<int64_t>(gridDim.y) * RT) {
            const int64_t off = ((p / 128) * nka + kb / 4) * 512 + (p % 32) * 16 + ((p % 128) / 32) * 4;
            *reinterpret_cast<uint32_t *>(a.scales + off) = 0u;
        }
    }
}

// ------------------------------------------------------------ W4A16 weights

// MXFP4 codes and tiled scales -> bf16 values (each E2M1 value times its
// E8M0 power of two; exact in bf16 for scales an fp32 input can produce).
// One thread per block of 32 values: 16 code bytes in, 64 bytes out.
__global__ void __launch_bounds__(256) dequant_bf16_kernel(const uint8_t *codes, const uint8_t *scales,
                                                           int64_t rows, int64_t K, uint16_t *out)
{
    const int64_t nkb = K / 32;
    const int64_t nka = ((nkb + 7) / 8 * 8) / 4;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= rows * nkb) return;
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int64_t r = idx / nkb, kb = idx - (idx / nkb) * nkb;
    const uint8_t sb = scales[((r / 128) * nka + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4)];
    // 2^se with se = sb - 127 (sb = 0 gives 2^-127, a subnormal)
    const float p2 = sb > 0 ? __int_as_float(static_cast<int>(sb) << 23) : __int_as_float(1 << 22);
    const uint4 c4 = *reinterpret_cast<const uint4 *>(codes + r * (K / 2) + 16 * kb);
    const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t byte = (cw[i >> 2] >> (8 * (i & 3))) & 0xffu;
        float v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t c = (byte >> (4 * h)) & 0xfu;
            const uint32_t m = c & 7u;
            // E2M1 magnitude m: 0, 0.5, 1, 1.5, 2, 3, 4, 6
            const float mag = m < 2 ? 0.5f * static_cast<float>(m)
                                    : __int_as_float(static_cast<int>(((m >> 1) + 126) << 23) | static_cast<int>((m & 1u) << 22));
            v[h] = __fmul_rn((c & 8u) ? -mag : mag, p2);
        }
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[0], v[1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(out + r * K + 32 * kb);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
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

#define MACAQ_TRY_CUDA(expr)                   \
    do {                                       \
        cudaError_t e__ = (expr);              \
        if (e__ != cudaSuccess) return e__;    \
    } while (0)

// Launch with programmatic stream serialisation (the kernel itself waits for
// its predecessor with griddepcontrol.wait before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Per-device facts the launches need, queried once: the SM count, and the
// dynamic shared memory each TMA kernel variant has been opened up to.
struct QuantDevice {
    int sms = 0;
    int smem_set[30] = {};
};
QuantDevice g_qdev[64];
std::mutex g_qdev_mu;

cudaError_t quant_device(int *sms)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_qdev_mu);
    if (g_qdev[dev].sms == 0) {
        err = cudaDeviceGetAttribute(&g_qdev[dev].sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
    }
    *sms = g_qdev[dev].sms;
    return cudaSuccess;
}

template <typename Kern>
cudaError_t open_smem(Kern kern, int slot, int64_t smem)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_qdev_mu);
    if (g_qdev[dev].smem_set[slot] < smem) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        g_qdev[dev].smem_set[slot] = static_cast<int>(smem);
    }
    return cudaSuccess;
}

// Stage shape of the TMA kernels: TB blocks of 32 values (a slab of the row)
// by RT rows, consumer threads TB * RT <= 512 and a whole number of warps
// (a warp may span rows; TB is a multiple of 8, so every group of four
// neighbouring blocks sharing a scale word lies in one row), a stage of at
// most 32 KB, and the fewest idle blocks over the slabs that cover the row.
bool pick_tma_tile(int64_t nkb_pad, int64_t max_consumers, int64_t max_slab_bytes, int64_t *tb_out,
                   int64_t *rt_out)
{
    int64_t best_waste = -1;
    const int64_t s0 = (nkb_pad + 255) / 256;
    for (int64_t slabs = s0; slabs <= s0 + 8; ++slabs) {
        const int64_t tb = ((nkb_pad + slabs - 1) / slabs + 7) / 8 * 8;
        if (tb > 256) continue;
        int64_t rt = 0;
        for (int64_t r = (max_consumers / tb < 32 ? max_consumers / tb : 32); r >= 1; --r) {
            if ((tb * r) % 32 == 0 && tb * r * 64 <= max_slab_bytes) {
                rt = r;
                break;
            }
        }
        if (rt == 0) continue;
        const int64_t waste = tb * slabs - nkb_pad;
        if (best_waste < 0 || waste < best_waste) {
            best_waste = waste;
            *tb_out = tb;
            *rt_out = rt;
        }
    }
    return best_waste >= 0;
}

cudaError_t launch_quant_dense_tma(const QuantArgs &a, cudaStream_t stream, bool *done)
{
    *done = false;
    const int64_t nkb = a.K / 32;
    const int64_t nkb_pad = pad_scale_cols(a.K);
    int64_t tb = 0, rt = 0;
    if (!pick_tma_tile(nkb_pad, kTmaConsumersMax, 40960, &tb, &rt)) return cudaSuccess;
    const int64_t slabs = (nkb_pad + tb - 1) / tb;
    const int64_t stage = tb * rt * 64;
    const int64_t fixed = 16 + tb * 128 + 1024;  // abort flag, balance-factor table, alignment
    const int stages = (6 * stage + 16 * 6 + fixed <= 200 * 1024) ? 6 : 4;
    const int64_t smem = stages * stage + 16 * stages + fixed;
    if (smem > 210 * 1024) return cudaSuccess;  // fall through to the register-staged kernel
    CUtensorMap tm;
    const uint64_t dims[3] = {32, static_cast<uint64_t>(nkb), static_cast<uint64_t>(a.rows_valid)};
    const uint64_t strides[2] = {64, static_cast<uint64_t>(a.ld_src) * 2};
    const uint32_t box[3] = {32, static_cast<uint32_t>(tb), static_cast<uint32_t>(rt)};
    if (!encode_tensor_map(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.src, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaSuccess;
    int sms = 148;
    MACAQ_TRY_CUDA(quant_device(&sms));
    const int64_t groups = (a.rows_out + rt - 1) / rt;
    int64_t ctas_y = sms / slabs;  // one CTA per SM: never a partial second wave
    ctas_y = ctas_y < 1 ? 1 : ctas_y;
    ctas_y = ctas_y > groups ? groups : ctas_y;
    void (*kern)(CUtensorMap, QuantArgs, int32_t, int32_t, int32_t);
    if (a.out_kind == kOutBf16)
        kern = a.had == 64 ? (stages == 6 ? quant_dense_tma_kernel<6, true, kOutBf16> : quant_dense_tma_kernel<4, true, kOutBf16>)
                           : (stages == 6 ? quant_dense_tma_kernel<6, false, kOutBf16> : quant_dense_tma_kernel<4, false, kOutBf16>);
    else if (a.out_kind == kOutF32)
        kern = a.had == 64 ? (stages == 6 ? quant_dense_tma_kernel<6, true, kOutF32> : quant_dense_tma_kernel<4, true, kOutF32>)
                           : (stages == 6 ? quant_dense_tma_kernel<6, false, kOutF32> : quant_dense_tma_kernel<4, false, kOutF32>);
    else
        kern = a.had == 64 ? (stages == 6 ? quant_dense_tma_kernel<6, true, kOutMx> : quant_dense_tma_kernel<4, true, kOutMx>)
                           : (stages == 6 ? quant_dense_tma_kernel<6, false, kOutMx> : quant_dense_tma_kernel<4, false, kOutMx>);
    MACAQ_TRY_CUDA(open_smem(kern, (stages == 6 ? 0 : 1) + (a.had == 64 ? 8 : 0) + 10 * a.out_kind, smem));
    dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(ctas_y));
    dim3 block(static_cast<unsigned>(tb * rt + 32));
    MACAQ_TRY_CUDA(launch_pdl(kern, grid, block, static_cast<size_t>(smem), stream, tm, a,
                              static_cast<int32_t>(groups), static_cast<int32_t>(tb), static_cast<int32_t>(rt)));
    *done = true;
    return cudaGetLastError();
}

cudaError_t launch_quant_grouped_tma(const QuantArgs &a, bool silu, cudaStream_t stream, bool *done)
{
    *done = false;
    const int64_t nkb = a.K / 32;
    const int64_t nkb_pad = pad_scale_cols(a.K);
    int64_t tb = 0, rt = 0;
    // SwiGLU rows land two slabs (gate and up) per row
    if (!pick_tma_tile(nkb_pad, grouped_consumers_max(silu), silu ? 32768 : 40960, &tb, &rt)) return cudaSuccess;
    const int64_t slabs = (nkb_pad + tb - 1) / tb;
    const int64_t stage = tb * rt * 64 * (silu ? 2 : 1);
    int sms = 148;
    MACAQ_TRY_CUDA(quant_device(&sms));
    const int64_t groups = (a.rows_out + rt - 1) / rt;
    int64_t ctas_y = sms / slabs;
    ctas_y = ctas_y < 1 ? 1 : ctas_y;
    ctas_y = ctas_y > groups ? groups : ctas_y;
    const int64_t per_cta = (groups + ctas_y - 1) / ctas_y;
    ctas_y = (groups + per_cta - 1) / per_cta;
    const int64_t max_rows = per_cta * rt;
    if (max_rows > 4096) return cudaSuccess;  // row table too large: register-staged kernel
    // the most factor-table slots (4, 2, 1) beside the deepest ring that fits
    int stages = 0, slots = 0;
    int64_t smem = 0;
    for (int sl = kGroupedFacSlotsMax; sl >= 1 && stages == 0; sl /= 2) {
        const int64_t fixed = 16 + 2 * (kMaxExperts + 1) * 4 + 3 * max_rows * 4 + 16 + sl * tb * 128 + 1024;
        const int st = (6 * stage + 16 * 6 + fixed <= 200 * 1024) ? 6 : (4 * stage + 16 * 4 + fixed <= 210 * 1024) ? 4 : 3;
        if (st * stage + 16 * st + fixed <= 210 * 1024) {
            stages = st;
            slots = sl;
            smem = st * stage + 16 * st + fixed;
        }
    }
    if (stages == 0) return cudaSuccess;
    CUtensorMap tm;
    // the token rows are whatever row_src names (valid by contract): no row bound
    // (SwiGLU: the gate|up row holds 2 * K / 32 blocks)
    const uint64_t dims[3] = {32, static_cast<uint64_t>(silu ? 2 * nkb : nkb), 0x7fffffffull};
    const uint64_t strides[2] = {64, static_cast<uint64_t>(a.ld_src) * 2};
    const uint32_t box[3] = {32, static_cast<uint32_t>(tb), 1};
    if (!encode_tensor_map(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.src, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaSuccess;
    void (*kern)(CUtensorMap, QuantArgs, int32_t, int32_t, int32_t, int32_t, int32_t);
    if (a.had == 64)
        kern = silu ? (stages == 6 ? quant_grouped_tma_kernel<6, true, true>
                                   : stages == 4 ? quant_grouped_tma_kernel<4, true, true>
                                                 : quant_grouped_tma_kernel<3, true, true>)
                    : (stages == 6 ? quant_grouped_tma_kernel<6, false, true>
                                   : stages == 4 ? quant_grouped_tma_kernel<4, false, true>
                                                 : quant_grouped_tma_kernel<3, false, true>);
    else
        kern = silu ? (stages == 6 ? quant_grouped_tma_kernel<6, true, false>
                                   : stages == 4 ? quant_grouped_tma_kernel<4, true, false>
                                                 : quant_grouped_tma_kernel<3, true, false>)
                    : (stages == 6 ? quant_grouped_tma_kernel<6, false, false>
                                   : stages == 4 ? quant_grouped_tma_kernel<4, false, false>
                                                 : quant_grouped_tma_kernel<3, false, false>);
    MACAQ_TRY_CUDA(open_smem(kern, (stages == 6 ? 0 : stages == 4 ? 1 : 2) + (silu ? 3 : 0) + (a.had == 64 ? 22 : 2), smem));
    dim3 grid(static_cast<unsigned>(slabs), static_cast<unsigned>(ctas_y));
    dim3 block(static_cast<unsigned>(tb * rt + 32));
    MACAQ_TRY_CUDA(launch_pdl(kern, grid, block, static_cast<size_t>(smem), stream, tm, a,
                              static_cast<int32_t>(groups), static_cast<int32_t>(tb), static_cast<int32_t>(rt),
                              static_cast<int32_t>(per_cta), static_cast<int32_t>(slots)));
    *done = true;
    return cudaGetLastError();
}

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
    // a few rows (decode): the register-staged kernel spreads them over more
    // CTAs than the TMA ring's row groups, for a shorter launch
    const bool few_rows = a.rows_valid <= 64 && a.had == 32 && a.out_kind == kOutMx;
    if (mode == QuantMode::Dense && (a.ld_src * 2) % 16 == 0 && a.rows_valid >= 1 && !few_rows) {
        bool done = false;
        cudaError_t err = launch_quant_dense_tma(a, stream, &done);
        if (err != cudaSuccess || done) return err;
    }
    if ((mode == QuantMode::ActGrouped || mode == QuantMode::ActGroupedSilu) && (a.ld_src * 2) % 16 == 0 &&
        a.rows_valid >= 1) {
        bool done = false;
        cudaError_t err = launch_quant_grouped_tma(a, mode == QuantMode::ActGroupedSilu, stream, &done);
        if (err != cudaSuccess || done) return err;
    }
    if (mode == QuantMode::ActGroupedSilu) return a.rows_valid >= 1 ? cudaErrorNotSupported : cudaSuccess;
    if (a.had == 64 || a.out_kind != kOutMx) return a.rows_valid >= 1 ? cudaErrorNotSupported : cudaSuccess;
    const int64_t slabs = (nkb_pad + best_t - 1) / best_t;
    // rows per CTA: aim for about 8 resident-CTA waves worth of work items
    int sms = 148;
    MACAQ_TRY_CUDA(quant_device(&sms));
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
        MACAQ_TRY_CUDA(launch_pdl(quant_kernel<M, true>, grid, block, 0, stream, a, rows_per_cta)); \
    else                                                                                   \
        MACAQ_TRY_CUDA(launch_pdl(quant_kernel<M, false>, grid, block, 0, stream, a, rows_per_cta));
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

cudaError_t read_and_clear_quant_error(unsigned *flags)
{
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_quant_error_flags, sizeof(unsigned));
    if (err != cudaSuccess) return err;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_quant_error_flags, &zero, sizeof(unsigned));
}

cudaError_t launch_debug_e2m1(const float *t, int64_t n, uint8_t *codes, cudaStream_t stream)
{
    const int64_t blocks = (n + 255) / 256;
    debug_e2m1_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(t, n, codes);
    return cudaGetLastError();
}

cudaError_t launch_dequant_bf16(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t K,
                                uint16_t *out, cudaStream_t stream)
{
    const int64_t n = rows * (K / 32);
    const int64_t blocks = (n + 255) / 256;
    MACAQ_TRY_CUDA(launch_pdl(dequant_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                              codes, scales, rows, K, out));
    return cudaGetLastError();
}

}  // namespace macaq
