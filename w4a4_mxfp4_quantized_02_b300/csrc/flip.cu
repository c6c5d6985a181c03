// Flip Refinement (page "What is MACaQ quantization", section "How MACaQ
// works", step "Flip Refinement": instead of plain round to nearest, a
// Hessian-aware coordinate descent moves single 4-bit weight codes to an
// adjacent value when that lowers the layer's error on calibration data).
//
// In the rotated space the layer output is A . Wt^T (A: calibration rows
// through the activation transform, Wt: weight rows through the weight
// transform, both fp32).  For one weight row with dequantised codes q the
// calibration error is E(q) = (Wt - q)^T H (Wt - q), H = A^T A (+ damp on the
// diagonal).  With r = Wt - q and g = H r, moving q_k by D changes E by
// D (D H_kk - 2 g_k); coordinates are visited in order, `sweeps` times; of the
// two adjacent values on the signed E2M1 grid (scale unchanged) the one with
// the larger strict decrease is taken, ties to the lower, and g -= D H[k, :].
//
// The codes depend on every bit of g, so every sum here is a chain of fused
// multiply-adds in a fixed order (the order of the definition: calibration
// rows for H, coordinates for g) and every other step one IEEE rounding; the
// unit is compiled without FMA contraction.
//
// Kernels:
//   flip_residual_kernel  r = Wt - q (fp32), q from codes and tiled scales
//   sgemm_seq_kernel      C = A . B on CUDA cores, each output a sequential
//                         FMA chain over the inner index (H = A^T A, G = R H)
//   flip_sweep_kernel     the descent: rows of a CTA each keep g, codes and
//                         scale bytes in shared memory; blocks of 32
//                         coordinates are decided in registers against the
//                         diagonal piece of H, then their moves are applied to
//                         all of g at once (rows of the row meet at a bounded
//                         shared-memory barrier twice per block)
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace macaq {

namespace {

// 2^(sb - 127) as fp32 (sb = 0 gives the subnormal 2^-127)
__device__ __forceinline__ float e8m0_value(uint32_t sb)
{
    return sb > 0 ? __int_as_float(static_cast<int>(sb) << 23) : __int_as_float(1 << 22);
}

// E2M1 magnitude of a magnitude code 0 .. 7: 0, 0.5, 1, 1.5, 2, 3, 4, 6
__device__ __forceinline__ float e2m1_magnitude(uint32_t m)
{
    return m < 2 ? 0.5f * static_cast<float>(m)
                 : __int_as_float(static_cast<int>(((m >> 1) + 126) << 23) | static_cast<int>((m & 1u) << 22));
}

// signed grid position of a code (-7 .. 7; both zeros at 0) and its value
__device__ __forceinline__ int e2m1_position(uint32_t code)
{
    const int m = static_cast<int>(code & 7u);
    return (code & 8u) ? -m : m;
}

__device__ __forceinline__ float position_value(int pos)
{
    const float v = e2m1_magnitude(static_cast<uint32_t>(pos < 0 ? -pos : pos));
    return pos < 0 ? -v : v;
}

__device__ __forceinline__ size_t tiled_scale_offset(int64_t row, int64_t kb, int64_t nka)
{
    return static_cast<size_t>(((row / 128) * nka + kb / 4) * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + (kb % 4));
}

// --------------------------------------------------------------- residual

__global__ void __launch_bounds__(256) flip_residual_kernel(const float *wt, const uint8_t *codes,
                                                            const uint8_t *scales, int64_t n, int64_t k,
                                                            float *r)
{
    const int64_t nkb = k / 32;
    const int64_t nka = ((nkb + 7) / 8 * 8) / 4;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // one 32-block
    if (idx >= n * nkb) return;
    const int64_t row = idx / nkb, kb = idx - row * nkb;
    const float p = e8m0_value(scales[tiled_scale_offset(row, kb, nka)]);
    const uint4 c4 = *reinterpret_cast<const uint4 *>(codes + row * (k / 2) + 16 * kb);
    const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
    const float4 *src = reinterpret_cast<const float4 *>(wt + row * k + 32 * kb);
    float4 *dst = reinterpret_cast<float4 *>(r + row * k + 32 * kb);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 w = src[q];
        const uint32_t two = cw[q >> 1] >> (16 * (q & 1));  // the 4 codes of elements 4q .. 4q+3
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(position_value(e2m1_position((two >> (4 * e)) & 0xfu)), p);
        dst[q] = make_float4(__fsub_rn(w.x, v[0]), __fsub_rn(w.y, v[1]), __fsub_rn(w.z, v[2]), __fsub_rn(w.w, v[3]));
    }
}

// ------------------------------------------------- sequential-order SGEMM

constexpr int kSgBM = 128, kSgBN = 128, kSgBK = 8, kSgThreads = 256;

// C[i, j] = fma-chain over l = 0 .. L-1 of A(i, l) * B(l, j), starting at +0,
// then + diag_add where i == j (one fp32 add; only when add_diag).
// A(i, l) = a[l * lda + i] (kAT) or a[i * lda + l]; B(l, j) = b[l * ldb + j];
// C[i * ldc + j].  M, N, L multiples of 4 where they index a contiguous
// dimension; all pitches multiples of 4, pointers 16-byte aligned.
// Each thread owns an 8 x 8 block of C (rows 4ty.. and 64+4ty.., columns
// 4tx.. and 64+4tx..) and walks l in order, so each output's FMA chain is the
// definition's whatever the tiling; the next 8-deep slab of A and B is
// fetched into registers while the current one is consumed (two shared
// buffers, one barrier per slab).
template <bool kAT>
__global__ void __launch_bounds__(kSgThreads) sgemm_seq_kernel(const float *a, int64_t lda, const float *b,
                                                                int64_t ldb, float *c, int64_t ldc, int64_t M,
                                                                int64_t N, int64_t L, bool add_diag, float diag_add)
{
    __shared__ __align__(16) float As[2][kSgBK][kSgBM];
    __shared__ __align__(16) float Bs[2][kSgBK][kSgBN];
    const int t = threadIdx.x;
    const int tx = t % 16, ty = t / 16;
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * kSgBM;
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kSgBN;
    float acc[8][8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[u][v] = 0.0f;

    // one float4 of A and one of B per thread and slab
    const int a_l = kAT ? t / 32 : (t % 2) * 4;   // slab row (kAT) or first of 4 l
    const int a_i = kAT ? (t % 32) * 4 : t / 2;   // first of 4 i (kAT) or the i
    const int b_l = t / 32, b_j = (t % 32) * 4;
    auto fetch = [&](int64_t l0, float4 &ra, float4 &rb) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kAT) {
            const int64_t gl = l0 + a_l, gi = i0 + a_i;
            ra = (gl < L && gi < M) ? *reinterpret_cast<const float4 *>(a + gl * lda + gi) : z;
        } else {
            const int64_t gl = l0 + a_l, gi = i0 + a_i;
            ra = (gl < L && gi < M) ? *reinterpret_cast<const float4 *>(a + gi * lda + gl) : z;
        }
        const int64_t gl = l0 + b_l, gj = j0 + b_j;
        rb = (gl < L && gj < N) ? *reinterpret_cast<const float4 *>(b + gl * ldb + gj) : z;
    };
    auto stash = [&](int buf, const float4 &ra, const float4 &rb) {
        if (kAT) {
            *reinterpret_cast<float4 *>(&As[buf][a_l][a_i]) = ra;
        } else {
            As[buf][a_l][a_i] = ra.x;
            As[buf][a_l + 1][a_i] = ra.y;
            As[buf][a_l + 2][a_i] = ra.z;
            As[buf][a_l + 3][a_i] = ra.w;
        }
        *reinterpret_cast<float4 *>(&Bs[buf][b_l][b_j]) = rb;
    };

    float4 ra, rb;
    fetch(0, ra, rb);
    stash(0, ra, rb);
    __syncthreads();
    int buf = 0;
    for (int64_t l0 = 0; l0 < L; l0 += kSgBK) {
        const bool more = l0 + kSgBK < L;
        if (more) fetch(l0 + kSgBK, ra, rb);
        auto step = [&](int ll) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][ll][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][ll][64 + 4 * ty]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][ll][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][ll][64 + 4 * tx]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[u][v] = __fmaf_rn(av[u], bv[v], acc[u][v]);
        };
        if (L - l0 >= kSgBK) {
#pragma unroll
            for (int ll = 0; ll < kSgBK; ++ll) step(ll);
        } else {
            for (int ll = 0; ll < static_cast<int>(L - l0); ++ll) step(ll);
        }
        if (more) {
            stash(buf ^ 1, ra, rb);
            __syncthreads();
            buf ^= 1;
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int64_t gi = i0 + (u < 4 ? 4 * ty + u : 64 + 4 * ty + u - 4);
        if (gi >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t gj = j0 + 64 * h + 4 * tx;
            if (gj >= N) continue;
            float x[4] = {acc[u][4 * h], acc[u][4 * h + 1], acc[u][4 * h + 2], acc[u][4 * h + 3]};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (add_diag && gi == gj + q) x[q] = __fadd_rn(x[q], diag_add);
            *reinterpret_cast<float4 *>(c + gi * ldc + gj) = make_float4(x[0], x[1], x[2], x[3]);
        }
    }
}

// ------------------------------------------------------------------ descent

constexpr int kFlipThreads = 512;
constexpr int kFlushRB = 8;  // float4 of g per thread per pass of the block update
constexpr uint64_t kFlipWaitNs = 2000000000ull;  // a row barrier gives up after 2 s
constexpr int64_t kFlipSmemMax = 220 * 1024;

__device__ unsigned int g_flip_error_flags;

// per-row shared-memory header: barrier arrival count, generation, abort flag
struct RowSync {
    unsigned count;
    unsigned gen;
    unsigned abort;
    unsigned pad;
};

// Shared memory of one row: header, g [K], codes [K/2], scale bytes [K/32]
// (padded to 16 bytes), the 32 x 32 diagonal block of H for the current
// coordinate block, and the block's moves (coordinate, step).
inline __host__ __device__ int64_t flip_row_bytes(int64_t k)
{
    return 16 + 4 * k + (k / 2) + ((k / 32 + 15) / 16) * 16 + 32 * 32 * 4 + 32 * 4 + 32 * 4;
}

// Barrier of the `warps` warps of one row: lane 0 of each warp arrives on a
// shared-memory counter; the last arrival resets it and advances the
// generation the others spin on.  A spin that runs past kFlipWaitNs sets the
// row's abort flag and the device error flag and returns false (the caller
// then leaves without writing results).
__device__ __forceinline__ bool row_barrier(RowSync *rs, int warps, int lane)
{
    __syncwarp();
    if (warps == 1) return true;
    int ok = 1;
    if (lane == 0) {
        volatile unsigned *gen = &rs->gen;
        volatile unsigned *abort_flag = &rs->abort;
        const unsigned my_gen = *gen;
        __threadfence_block();
        if (atomicAdd(&rs->count, 1u) == static_cast<unsigned>(warps - 1)) {
            atomicExch(&rs->count, 0u);
            __threadfence_block();
            atomicAdd(&rs->gen, 1u);
        } else {
            const uint64_t t0 = ptx::globaltimer();
            for (uint32_t spin = 0; *gen == my_gen; ++spin) {
                if (*abort_flag) {
                    ok = 0;
                    break;
                }
                if ((spin & 255u) == 255u && ptx::globaltimer() - t0 > kFlipWaitNs) {
                    *abort_flag = 1u;
                    atomicOr(&g_flip_error_flags, 1u);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence_block();
        if (*abort_flag) ok = 0;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// Rows blockIdx.x * RC + i (i < RC), each handled by WR = 16 / RC warps.
//
// The coordinates are taken in blocks of 32 (one MX block, one scale).  Within
// a block, lane l of every warp of the row holds coordinate c0 + l: its code
// and gv, its g plus the block's moves so far; a move at coordinate kk with
// step D updates every lane's gv by one fused multiply-add with H[c0+kk,
// c0+l] (the block's 32 x 32 diagonal piece of H, in shared memory), so each
// decision sees exactly the g the one-move-at-a-time definition has.  After
// the block the row's threads apply the block's moves, in order, to every
// entry of g (rows c0 + kk of H, streamed from global memory), write the
// block's codes back and load the next diagonal piece.  Each entry of g thus
// receives the moves' fused multiply-adds in move order, bit for bit the
// definition.  Every thread of the row passes the same two barriers per block,
// whatever the moves.
__global__ void __launch_bounds__(kFlipThreads, 1) flip_sweep_kernel(const float *H, const float *G,
                                                                     uint8_t *codes, const uint8_t *scales,
                                                                     int32_t *flips, int64_t n, int64_t k,
                                                                     int32_t sweeps, int32_t RC)
{
    extern __shared__ float4 fsmem4[];
    const int WR = 16 / RC;
    const int threads = 32 * WR;
    const int group = threadIdx.x / threads;
    const int gt = threadIdx.x % threads;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * RC + group;
    uint8_t *base = reinterpret_cast<uint8_t *>(fsmem4) + group * flip_row_bytes(k);
    RowSync *rs = reinterpret_cast<RowSync *>(base);
    float *g = reinterpret_cast<float *>(base + 16);
    uint8_t *cs = base + 16 + 4 * k;
    uint8_t *sb = cs + k / 2;
    float *hblk = reinterpret_cast<float *>(sb + ((k / 32 + 15) / 16) * 16);  // [32][32]
    int32_t *mv_k = reinterpret_cast<int32_t *>(hblk + 32 * 32);
    float *mv_d = reinterpret_cast<float *>(mv_k + 32);
    const int64_t nkb = k / 32;
    const int64_t nka = ((nkb + 7) / 8 * 8) / 4;

    if (gt == 0) {
        rs->count = 0;
        rs->gen = 0;
        rs->abort = 0;
    }
    __syncthreads();
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (row >= n) return;  // the whole row group leaves together

    for (int64_t j = gt; j < k / 4; j += threads)
        reinterpret_cast<float4 *>(g)[j] = reinterpret_cast<const float4 *>(G + row * k)[j];
    for (int64_t j = gt; j < k / 32; j += threads)
        reinterpret_cast<uint4 *>(cs)[j] = reinterpret_cast<const uint4 *>(codes + row * (k / 2))[j];
    for (int64_t j = gt; j < nkb; j += threads) sb[j] = scales[tiled_scale_offset(row, j, nka)];
    for (int e = gt; e < 32 * 32; e += threads) hblk[e] = H[static_cast<int64_t>(e >> 5) * k + (e & 31)];
    if (!row_barrier(rs, WR, lane)) return;

    int32_t moves = 0;
    const bool writer = gt < 32;  // warp 0 of the row writes codes and the move list
    for (int32_t sw = 0; sw < sweeps; ++sw) {
        for (int64_t b = 0; b < nkb; ++b) {
            const int64_t c0 = 32 * b;
            float gv = g[c0 + lane];
            const uint32_t byte = cs[(c0 + lane) >> 1];
            uint32_t code = (lane & 1) ? (byte >> 4) : (byte & 0xfu);
            const float hkk_mine = hblk[lane * 33];
            const float p = e8m0_value(sb[b]);
            int cnt = 0;
            for (int kk = 0; kk < 32; ++kk) {
                const float gk = __shfl_sync(0xffffffffu, gv, kk);
                const uint32_t ck = __shfl_sync(0xffffffffu, code, kk);
                const float hkk = __shfl_sync(0xffffffffu, hkk_mine, kk);
                const int pos = e2m1_position(ck);
                const float t = position_value(pos);
                const float two_g = __fmul_rn(2.0f, gk);
                int best = 0;
                float best_de = 0.0f, best_d = 0.0f;
#pragma unroll
                for (int dir = -1; dir <= 1; dir += 2) {
                    const int np = pos + dir;
                    if (np < -7 || np > 7) continue;
                    const float d = __fmul_rn(__fsub_rn(position_value(np), t), p);
                    const float de = __fmul_rn(d, __fsub_rn(__fmul_rn(d, hkk), two_g));
                    if (de < 0.0f && (best == 0 || de < best_de)) {
                        best = dir;
                        best_de = de;
                        best_d = d;
                    }
                }
                if (best == 0) continue;
                const int npos = pos + best;
                // a move onto zero keeps the sign of the side it came from
                const uint32_t nc = npos > 0 ? static_cast<uint32_t>(npos)
                                             : npos < 0 ? (8u | static_cast<uint32_t>(-npos)) : (pos < 0 ? 8u : 0u);
                if (lane == kk) code = nc;
                gv = __fmaf_rn(-best_d, hblk[kk * 32 + lane], gv);
                if (writer && lane == 0) {
                    mv_k[cnt] = kk;
                    mv_d[cnt] = best_d;
                }
                ++cnt;
                ++moves;
            }
            // every thread of the row is done with this block's g, codes,
            // diagonal piece and (previous) move list
            if (!row_barrier(rs, WR, lane)) return;
            const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
            if (writer && (lane & 1) == 0) cs[(c0 + lane) >> 1] = static_cast<uint8_t>(code | (hi << 4));
            if (cnt > 0) {
                // kFlushRB float4 of g per thread in registers; for each move
                // (in order) their kFlushRB rows-of-H loads are independent
                float4 *g4 = reinterpret_cast<float4 *>(g);
                const int64_t k4 = k / 4;
                for (int64_t j0 = gt; j0 < k4; j0 += kFlushRB * threads) {
                    float4 x[kFlushRB];
#pragma unroll
                    for (int q = 0; q < kFlushRB; ++q) {
                        const int64_t j = j0 + q * threads;
                        if (j < k4) x[q] = g4[j];
                    }
#pragma unroll 2
                    for (int m = 0; m < cnt; ++m) {
                        const float nd = -mv_d[m];
                        const float4 *hrow = reinterpret_cast<const float4 *>(H + (c0 + mv_k[m]) * k);
                        float4 h[kFlushRB];
#pragma unroll
                        for (int q = 0; q < kFlushRB; ++q) {
                            const int64_t j = j0 + q * threads;
                            if (j < k4) h[q] = __ldg(hrow + j);
                        }
#pragma unroll
                        for (int q = 0; q < kFlushRB; ++q) {
                            x[q].x = __fmaf_rn(nd, h[q].x, x[q].x);
                            x[q].y = __fmaf_rn(nd, h[q].y, x[q].y);
                            x[q].z = __fmaf_rn(nd, h[q].z, x[q].z);
                            x[q].w = __fmaf_rn(nd, h[q].w, x[q].w);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kFlushRB; ++q) {
                        const int64_t j = j0 + q * threads;
                        if (j < k4) g4[j] = x[q];
                    }
                }
            }
            // the diagonal piece of the next block (wrapping to block 0)
            const int64_t n0 = b + 1 < nkb ? c0 + 32 : 0;
            for (int e = gt; e < 32 * 32; e += threads) hblk[e] = H[(n0 + (e >> 5)) * k + n0 + (e & 31)];
            if (!row_barrier(rs, WR, lane)) return;
        }
    }
    for (int64_t j = gt; j < k / 32; j += threads)
        reinterpret_cast<uint4 *>(codes + row * (k / 2))[j] = reinterpret_cast<const uint4 *>(cs)[j];
    if (gt == 0 && flips) flips[row] = moves;
}

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

}  // namespace

int64_t flip_rows_per_cta(int64_t k)
{
    for (int rc = 16; rc >= 1; rc /= 2)
        if (rc * flip_row_bytes(k) <= kFlipSmemMax) return rc;
    return 0;
}

cudaError_t read_and_clear_flip_error(unsigned *flags)
{
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_flip_error_flags, sizeof(unsigned));
    if (err != cudaSuccess) return err;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_flip_error_flags, &zero, sizeof(unsigned));
}

cudaError_t launch_flip_hessian(const float *a, int64_t m, int64_t k, float damp, float *h, cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>((k + kSgBN - 1) / kSgBN), static_cast<unsigned>((k + kSgBM - 1) / kSgBM));
    // A(i, l) = a[l, i]: rows of H are channels, the inner index the calibration row
    sgemm_seq_kernel<true><<<grid, kSgThreads, 0, stream>>>(a, k, a, k, h, k, k, k, m, true, damp);
    return cudaGetLastError();
}

cudaError_t launch_flip_prepare(const float *wt, const float *h, int64_t n, int64_t k, const uint8_t *codes,
                               const uint8_t *scales, float *r, float *g, cudaStream_t stream)
{
    const int64_t blocks = (n * (k / 32) + 255) / 256;
    flip_residual_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(wt, codes, scales, n, k, r);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    // G = R . H: g of every row, each entry a chain over the coordinates
    dim3 grid(static_cast<unsigned>((k + kSgBN - 1) / kSgBN), static_cast<unsigned>((n + kSgBM - 1) / kSgBM));
    sgemm_seq_kernel<false><<<grid, kSgThreads, 0, stream>>>(r, k, h, k, g, k, n, k, k, false, 0.0f);
    return cudaGetLastError();
}

cudaError_t launch_flip_sweeps(const float *h, const float *g, int64_t n, int64_t k, int32_t sweeps,
                               uint8_t *codes, const uint8_t *scales, int32_t *flips, cudaStream_t stream)
{
    const int64_t rc = flip_rows_per_cta(k);
    if (rc < 1) return cudaErrorNotSupported;
    const size_t smem = static_cast<size_t>(rc * flip_row_bytes(k));
    cudaError_t err = cudaFuncSetAttribute(flip_sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int64_t ctas = (n + rc - 1) / rc;
    err = launch_pdl(flip_sweep_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kFlipThreads), smem, stream, h, g,
                     codes, scales, flips, n, k, sweeps, static_cast<int32_t>(rc));
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace macaq
