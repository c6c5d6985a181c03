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

namespace skinny {

constexpr int kThreads = 7 * 32;
constexpr int kEpiWarp0 = 3;
constexpr int kTmemCols = 128;

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
};

template <int NT, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(ready_bar(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain_bar, 1);
        mbar_init(drain_bar2, 1);
        *abort_flag = 0;
        fence_mbar_init();
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
    griddep_wait();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            constexpr uint32_t kBytes = L::W_STAGE + L::X_STAGE + 2 * L::SF_STAGE;
            const uint8_t *sfw = p.sfw + static_cast<size_t>(n0 / 128) * p.nka * SF_ATOM;
            uint32_t issued = 0, last_parity = 0;
            for (int i = 0; i < my_stages; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = static_cast<uint32_t>(i / STAGES) & 1u;
                if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kErrProducer, wait_ns)) break;
                const int ks = ks_begin + i;
                const uint32_t fb = full_bar(s);
                mbar_arrive_expect_tx(fb, kBytes);
                tma_load_2d(sbase + L::OFF_W + s * L::W_STAGE, &tmW, fb, ks * L::KB, n0);
                tma_load_2d(sbase + L::OFF_X + s * L::X_STAGE, &tmX, fb, ks * L::KB, 0);
                bulk_load(sbase + L::OFF_SFW + s * L::SF_STAGE, sfw + static_cast<size_t>(2 * ks) * SF_ATOM,
                          L::SF_STAGE, fb);
                bulk_load(sbase + L::OFF_SFX + s * L::SF_STAGE, p.sfx + static_cast<size_t>(2 * ks) * SF_ATOM,
                          L::SF_STAGE, fb);
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

    if (warp < kEpiWarp0) {
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
