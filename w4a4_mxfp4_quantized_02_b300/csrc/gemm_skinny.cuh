// Skinny dense GEMM: few token rows (decode), many weight rows.
//
// Included by gemm.cu (it shares that unit's error flags, wait helpers and
// tensor-map encoder).  With M <= 64 a 128- or 256-row token tile would waste
// most of each MMA and, worse, leave most SMs without weight bytes to stream:
// decode is bound by reading Wq once.  So the roles of the operands swap:
// the MMA's M = 128 rows are weight rows (one n-tile per CTA) and its N = NT
// columns are the token rows (NT = 16, 32 or 64, rows past M read as zeros),
//     D[n, m] = sum_k Wq[n, k] * A[m, k]   (=  Y[m, n]),
// both operands K-major E2M1 with E8M0 scales per 32 values, exactly the
// block-scaled product the prefill kernels compute with A and B exchanged.
//
// One CTA streams one 128-row weight tile through a STAGES-deep TMA ring.
// When there are too few n-tiles to keep every SM streaming, a cluster of KS
// CTAs splits K: rank r covers stages [r*nks/KS, (r+1)*nks/KS), keeps its fp32
// partial in its own shared memory, and rank 0 adds the partials in rank
// order (a fixed order: the result does not depend on timing) through
// distributed shared memory before rounding to bf16.
//
// Warps: 0 TMA producer, 1 MMA issuer, 2 scale copier, 3..6 epilogue (tensor
// memory lanes 0..127 = the tile's weight rows).
//
// FUSED (the whole online layer for a few token rows, NT = 16): the token
// operand is not read from a transformed copy in HBM but formed inside the
// kernel, stage by stage, from the bf16 rows of X.  Eight transform warps
// (3..10; 3..6 then run the epilogue), in four groups that each take every
// fourth stage, run the work items (stage, token row, 32-value block): each
// item the balance, 32-point Hadamard, E8M0 scale and E2M1 codes of one
// block -- the activation transform of the layer, the same arithmetic as the
// standalone transform -- stored as 16 code bytes into the stage's
// 128-byte-swizzled token tile and a scale byte into its scale atoms, in the
// byte positions the TMA copies of the transformed operand would have.  Each
// item then arrives on the stage's "full" barrier, which so completes once
// the weight copies and all of the stage's items are in.  The weight stream
// thus starts right after the grid-dependency wait, with no separate
// transform launch before it.

namespace skinny {

constexpr int kEpiWarp0 = 3;
constexpr int kXformWarps = 8;  // FUSED: warps 3 .. 10 form the token tiles ...
constexpr int kXformGroups = 4;  // ... in four groups of two warps, each its own stages
constexpr int kXformGroupThreads = kXformWarps * 32 / kXformGroups;
constexpr int kTmemCols = 128;
__host__ __device__ constexpr int skinny_threads(bool fused) { return (fused ? kEpiWarp0 + kXformWarps : 7) * 32; }

template <int NT, int STAGES>
struct Layout {
    static constexpr int KB = 128;                    // operand bytes per row per stage
    static constexpr int W_STAGE = 128 * KB;          // 128 weight rows
    static constexpr int X_STAGE = NT * KB;           // NT token rows
    static constexpr int SF_STAGE = 2 * SF_ATOM;      // two 4-scale atoms (K = 256)
    static constexpr int SF_COLS = 16;                // tensor-memory columns per stage (W 8, X 8)
    static constexpr int OFF_W = 0;
    static constexpr int OFF_X = OFF_W + STAGES * W_STAGE;
    static constexpr int OFF_SFW = OFF_X + STAGES * X_STAGE;
    static constexpr int OFF_SFX = OFF_SFW + STAGES * SF_STAGE;
    // fp32 partial [128][NT + 1] of a K-split cluster: written once every MMA
    // has completed and every copy has landed, so it reuses the weight stages
    static constexpr int OFF_PART = OFF_W;
    static constexpr int PART_LD = NT + 1;
    static_assert(128 * PART_LD * 4 <= STAGES * W_STAGE, "partial must fit the weight stages");
    static constexpr int OFF_BAR = OFF_SFX + STAGES * SF_STAGE;
    static constexpr int NUM_BARS = 3 * STAGES + 3;
    static constexpr int OFF_MISC = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(OFF_X % 1024 == 0 && X_STAGE % 1024 == 0, "swizzled tiles need 1 KB alignment");
    static_assert(NT + STAGES * SF_COLS <= kTmemCols, "tensor memory overflow");
};

struct Params {
    const uint8_t *sfw;   // tiled weight scales
    const uint8_t *sfx;   // tiled token scales (one 128-row block)
    uint16_t *Y;
    int64_t ldy;
    int32_t M, N;
    int32_t num_kstages;
    int32_t nka;          // 4-scale atoms per 128-row block
    // FUSED: the layer input X bf16 [M, ldx] and the balance factors 1/s [K]
    const uint16_t *x;
    int64_t ldx;
    const float *inv;
    int32_t nkb;          // 32-value blocks of K
    // the weight was complete before the preceding kernel started (a
    // transform that lets this kernel start only after its own wait): the
    // producer issues the weight's first stages before the grid-dependency wait
    int32_t weight_early;
};

// FUSED asks for registers that let two of its CTAs share an SM (as the
// unfused kernel's fit), so 200 weight tiles still run in one wave.
template <int NT, int STAGES, bool FUSED = false>
__global__ void __launch_bounds__(skinny_threads(FUSED), FUSED ? 2 : 1)
    gemm_mxf4_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                            const Params p)
{
    using L = Layout<NT, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_base = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto ready_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
    const uint32_t acc_full = bar_base + 8u * (3 * STAGES);
    const uint32_t drain_bar = acc_full + 8u;
    const uint32_t drain_bar2 = acc_full + 16u;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
    float *part = reinterpret_cast<float *>(smem + L::OFF_PART);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t wait_ns = g_wait_ns;
    const uint32_t ks_rank = cluster_ctarank();
    const uint32_t KS = gridDim.x / static_cast<uint32_t>((p.N + 127) / 128);  // cluster size
    const int32_t n0 = static_cast<int32_t>(blockIdx.x / KS) * 128;
    const int nks = p.num_kstages;
    const int ks_begin = static_cast<int>((static_cast<int64_t>(nks) * ks_rank) / KS);
    const int ks_end = static_cast<int>((static_cast<int64_t>(nks) * (ks_rank + 1)) / KS);
    const int my_stages = ks_end - ks_begin;

    // FUSED: token rows 0 .. xrows-1 are formed in the kernel (8 items per
    // row and stage); the rest of each token tile and every scale byte not
    // rewritten per stage stay zero, set once here
    const int xrows = FUSED ? (p.M < NT ? p.M : NT) : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), FUSED ? 1u + 8u * static_cast<uint32_t>(xrows) : 1u);
            mbar_init(empty_bar(s), 1);
            mbar_init(ready_bar(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain_bar, 1);
        mbar_init(drain_bar2, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (FUSED) {
        for (int i = threadIdx.x; i < STAGES * (L::X_STAGE + L::SF_STAGE) / 16; i += blockDim.x) {
            const int s = i / ((L::X_STAGE + L::SF_STAGE) / 16);
            const int o = (i - s * ((L::X_STAGE + L::SF_STAGE) / 16)) * 16;
            const uint32_t addr = o < L::X_STAGE ? sbase + L::OFF_X + s * L::X_STAGE + o
                                                 : sbase + L::OFF_SFX + s * L::SF_STAGE + (o - L::X_STAGE);
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::OFF_MISC, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_launch_dependents();
    const bool weight_early = !FUSED && p.weight_early != 0;
    // (with weight_early the producer thread waits itself, after issuing the
    // weight's first stages)
    if (!(weight_early && threadIdx.x == 0)) griddep_wait();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            constexpr uint32_t kBytes = FUSED ? L::W_STAGE + L::SF_STAGE : L::W_STAGE + L::X_STAGE + 2 * L::SF_STAGE;
            const uint8_t *sfw = p.sfw + static_cast<size_t>(n0 / 128) * p.nka * SF_ATOM;
            uint32_t issued = 0, last_parity = 0;
            // the first round of stages: the slots are free; the weight part
            // may go before the grid-dependency wait, the token part not
            const int pre = weight_early ? (my_stages < STAGES ? my_stages : STAGES) : 0;
            for (int i = 0; i < pre; ++i) {
                const int ks = ks_begin + i;
                mbar_arrive_expect_tx(full_bar(i), kBytes);
                tma_load_2d(sbase + L::OFF_W + i * L::W_STAGE, &tmW, full_bar(i), ks * L::KB, n0);
                bulk_load(sbase + L::OFF_SFW + i * L::SF_STAGE, sfw + static_cast<size_t>(2 * ks) * SF_ATOM,
                          L::SF_STAGE, full_bar(i));
            }
            if (weight_early) griddep_wait();
            for (int i = 0; i < pre; ++i) {
                const int ks = ks_begin + i;
                tma_load_2d(sbase + L::OFF_X + i * L::X_STAGE, &tmX, full_bar(i), ks * L::KB, 0);
                bulk_load(sbase + L::OFF_SFX + i * L::SF_STAGE, p.sfx + static_cast<size_t>(2 * ks) * SF_ATOM,
                          L::SF_STAGE, full_bar(i));
                issued |= 1u << i;  // first pass of the ring: parity 0
            }
            for (int i = pre; i < my_stages; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
                if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kErrProducer, wait_ns)) break;
                const int ks = ks_begin + i;
                const uint32_t fb = full_bar(s);
                mbar_arrive_expect_tx(fb, kBytes);
                tma_load_2d(sbase + L::OFF_W + s * L::W_STAGE, &tmW, fb, ks * L::KB, n0);
                bulk_load(sbase + L::OFF_SFW + s * L::SF_STAGE, sfw + static_cast<size_t>(2 * ks) * SF_ATOM,
                          L::SF_STAGE, fb);
                if (!FUSED) {
                    tma_load_2d(sbase + L::OFF_X + s * L::X_STAGE, &tmX, fb, ks * L::KB, 0);
                    bulk_load(sbase + L::OFF_SFX + s * L::SF_STAGE,
                              p.sfx + static_cast<size_t>(2 * ks) * SF_ATOM, L::SF_STAGE, fb);
                }
                issued |= 1u << s;
                last_parity = (last_parity & ~(1u << s)) | (ph << s);
            }
            for (int s = 0; s < STAGES; ++s) {
                if (issued & (1u << s)) {
                    wait_fixed(full_bar(s), (last_parity >> s) & 1u);
                    wait_fixed(empty_bar(s), (last_parity >> s) & 1u);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint64_t w_desc0 = smem_desc(sbase + L::OFF_W, 16, 8 * L::KB, kSwizzle128B);
            const uint64_t x_desc0 = smem_desc(sbase + L::OFF_X, 16, 8 * L::KB, kSwizzle128B);
            const uint32_t idesc0 = idesc_mxf4(128, NT, 0, 0);
            const uint32_t idesc2 = idesc_mxf4(128, NT, 2, 2);
            bool ok = true;
            for (int i = 0; i < my_stages; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
                if (!wait_bounded(ready_bar(s), ph, abort_flag, kErrMma, wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sfw_t = tmem + NT + s * L::SF_COLS;
                const uint32_t sfx_t = sfw_t + 8;
                const uint64_t wd = w_desc0 + ((s * L::W_STAGE) >> 4);
                const uint64_t xd = x_desc0 + ((s * L::X_STAGE) >> 4);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tc_mma_mxf4(tmem, wd + 2 * j, xd + 2 * j, (j & 1) ? idesc2 : idesc0,
                                sfw_t + 4 * (j >> 1), sfx_t + 4 * (j >> 1), (i > 0 || j > 0) ? 1u : 0u);
                tc_commit(empty_bar(s));
            }
            if (ok && my_stages > 0) tc_commit(acc_full);
            tc_commit(drain_bar);
            wait_fixed(drain_bar, 0);
        }
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0) {
            // ------------------------------------------------ scale copier
            for (int i = 0; i < my_stages; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
                if (!wait_bounded(full_bar(s), ph, abort_flag, kErrMma, wait_ns)) break;
                const uint32_t sfw_t = tmem + NT + s * L::SF_COLS;
                const uint64_t dw = smem_desc(sbase + L::OFF_SFW + s * L::SF_STAGE, 0, 128, kSwizzleNone);
                const uint64_t dx = smem_desc(sbase + L::OFF_SFX + s * L::SF_STAGE, 0, 128, kSwizzleNone);
#pragma unroll
                for (int at = 0; at < 2; ++at) {
                    tc_cp_32x128b_warpx4(sfw_t + 4 * at, dw + at * (SF_ATOM >> 4));
                    tc_cp_32x128b_warpx4(sfw_t + 8 + 4 * at, dx + at * (SF_ATOM >> 4));
                }
                tc_commit(ready_bar(s));
            }
            tc_commit(drain_bar2);
            wait_fixed(drain_bar2, 0);
        }
        __syncwarp();
    } else {
        if constexpr (FUSED) {
            // ------------------------------------------------ token transform
            // The transform warps form four groups of two; group g takes stages
            // g, g + 4, g + 8, ... in order, its 64 threads the stage's items
            // (row r, block b) in turn.  A stage's buffers are free once the
            // MMAs of stage i - STAGES have read them ("empty", a parity wait).
            // A parity wait cannot tell a phase from the one two before it, so
            // no thread may wait more than one phase ahead: a thread's previous
            // stage was at most 4 <= STAGES stages earlier, and its wait then
            // proved every stage up to STAGES before that consumed.
            // Item (i, r, b): the 16 code bytes at row r, 16-byte chunk b of the
            // stage's token tile (128-byte swizzle: chunk b sits at b ^ (r % 8))
            // and the scale byte at block b of row r in the stage's two scale
            // atoms (row 32q + p, block c of an atom at byte 16p + 4q + c);
            // blocks past K get zero codes and a zero scale.
            static_assert(kXformGroups <= STAGES, "a transform group may run at most one ring ahead");
            const int tid = static_cast<int>(threadIdx.x) - kEpiWarp0 * 32;
            const int grp = tid / kXformGroupThreads, gt = tid % kXformGroupThreads;
            const int per_stage = 8 * xrows;
            bool ok = true;
            for (int i = grp; i < my_stages && ok; i += kXformGroups) {
                const int s = i % STAGES;
                const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
                for (int item = gt; item < per_stage; item += kXformGroupThreads) {
                    const int r = item >> 3, b = item & 7;
                    const int32_t kblk = (ks_begin + i) * 8 + b;
                    uint4 codes = make_uint4(0u, 0u, 0u, 0u);
                    uint32_t sbyte = 0;
                    if (kblk < p.nkb) {
                        uint32_t raw[16];
                        float2 f[16];
                        const uint4 *src = reinterpret_cast<const uint4 *>(
                            p.x + static_cast<int64_t>(r) * p.ldx + 32 * static_cast<int64_t>(kblk));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 w = __ldg(src + j);
                            raw[4 * j + 0] = w.x;
                            raw[4 * j + 1] = w.y;
                            raw[4 * j + 2] = w.z;
                            raw[4 * j + 3] = w.w;
                        }
                        const float4 *f4 = reinterpret_cast<const float4 *>(p.inv + 32 * static_cast<int64_t>(kblk));
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 a4 = __ldg(f4 + j);
                            f[2 * j] = make_float2(a4.x, a4.y);
                            f[2 * j + 1] = make_float2(a4.z, a4.w);
                        }
                        sbyte = mx::quant_block_pairs<false>(raw, f, codes);
                    }
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kErrEpilogue, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t xa = sbase + L::OFF_X + s * L::X_STAGE + r * L::KB + ((b ^ (r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(xa), "r"(codes.x),
                                 "r"(codes.y), "r"(codes.z), "r"(codes.w)
                                 : "memory");
                    const uint32_t sa = sbase + L::OFF_SFX + s * L::SF_STAGE + (b >> 2) * SF_ATOM +
                                        16 * (r & 31) + 4 * (r >> 5) + (b & 3);
                    asm volatile("st.shared.u8 [%0], %1;" ::"r"(sa), "r"(sbyte) : "memory");
                    // the tensor core reads both through the async proxy
                    fence_proxy_async_smem();
                    mbar_arrive(full_bar(s));
                }
            }
            // lanes leave the loop at different times (each waited for its own
            // stages); what follows -- tcgen05.ld and the cluster barriers --
            // is .aligned and must be reached by the whole warp together
            __syncwarp();
        }
    }
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;                 // tensor-memory lanes 32q..32q+31
        const int row = 32 * q + lane;          // weight row within the tile
        float acc[NT];
        bool have = false;
        if (my_stages > 0 && warp_wait_bounded(acc_full, 0, abort_flag, kErrEpilogue, wait_ns)) {
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16);
            if constexpr (NT == 16) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(taddr, r);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) acc[c] = __uint_as_float(r[c]);
            } else {
#pragma unroll
                for (int h = 0; h < NT / 32; ++h) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + 32 * h, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) acc[32 * h + c] = __uint_as_float(r[c]);
                }
            }
            have = true;
        }
        if (!have) {
#pragma unroll
            for (int c = 0; c < NT; ++c) acc[c] = 0.0f;
        }
        if (KS > 1) {
#pragma unroll
            for (int c = 0; c < NT; ++c) part[row * L::PART_LD + c] = acc[c];
        }
        tc_fence_before();
        // partials of the whole cluster are in place (a no-op wait for KS = 1)
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (ks_rank == 0) {
            if (KS > 1) {
                // rank order: rank 0's own partial first, then ranks 1, 2, ...
                for (uint32_t r = 1; r < KS; ++r) {
                    const uint32_t base = mapa_shared(smem_u32(part + row * L::PART_LD), r);
#pragma unroll
                    for (int c = 0; c < NT; ++c) acc[c] = __fadd_rn(acc[c], ld_shared_cluster_f32(base + 4 * c));
                }
            }
            const int32_t n = n0 + row;
            if (n < p.N) {
                const int mmax = p.M < NT ? p.M : NT;
#pragma unroll
                for (int c = 0; c < NT; ++c) {
                    if (c < mmax) {
                        const __nv_bfloat16 b = __float2bfloat16_rn(acc[c]);
                        p.Y[static_cast<int64_t>(c) * p.ldy + n] = *reinterpret_cast<const uint16_t *>(&b);
                    }
                }
            }
        }
        // peers keep their shared memory until rank 0 has read it
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }

    if (warp < kEpiWarp0 || warp >= kEpiWarp0 + 4) {
        // the non-epilogue warps take part in the epilogue's two cluster barriers
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace skinny
