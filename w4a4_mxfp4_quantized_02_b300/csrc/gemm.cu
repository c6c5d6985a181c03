// Block-scaled MXFP4 x MXFP4 GEMM (dense and grouped-by-expert) on the
// 5th-generation tensor cores of sm_103a.
//
// MACaQ runs its linear layers in W4A4 MXFP4 (page "Huawei MACaQ Is an
// Open-Source Model Quantizer", section "MACaQ Backends": W4A4 is the default
// inference mode; routed MoE experts run W4A4).  Y = A . Wq^T with both
// operands E2M1 codes scaled per 32 elements by E8M0 powers of two.
//
// Kernels, warp-specialised, one CTA per SM:
//   gemm_mxf4_pair_kernel   dense and expert-grouped Y: persistent CTA pairs
//                           (tcgen05 cta_group::2) on 256 x 256 tiles; see the
//                           comment at the kernel.
//   gemm_mxf4_skinny_kernel up to 64 token rows (decode): weight rows on the
//                           MMA's M side; gemm_skinny.cuh.
// Common shape:
//   warp 0      TMA producer: per 256-wide K stage, A and B tiles (128-byte
//               rows, 128B-swizzled) and the scale tiles (512-byte atoms) into
//               a ring of STAGES shared-memory buffers guarded by mbarriers.
//   warp 1      MMA issuer (one thread): tcgen05.mma.kind::mxf4.block_scale
//               (K = 64 per instruction) accumulating in tensor memory;
//               tcgen05.commit frees the stage.
//   warp 2      scale copier: tcgen05.cp 32x128b.warpx4 of the stage's scale
//               atoms into tensor memory, committed to "scales ready".  In
//               the MMA thread these copies would stall the tensor pipe: a
//               barrier wait issued after them waits for them to finish.
//   epilogue    tcgen05.ld of the fp32 accumulator into registers, release of
//               the accumulator, bf16 rounding and stores.
// Every mbarrier wait is bounded in time; a wait that runs out sets a device
// error flag and the CTA leaves in order (drains its copies and MMAs, frees
// tensor memory).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "mx_block.cuh"
#include "ptx.cuh"

#ifndef MACAQ_TRACE
#define MACAQ_TRACE(slot, idx)
#define MACAQ_TRACE_EDGE(which)
#endif

namespace macaq {

__device__ unsigned int g_error_flags;
__device__ unsigned long long g_wait_ns = 4000000000ull;

namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int SF_ATOM = 512;
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 3;  // warps 0..2: TMA producer, MMA issuer, scale copier
// The gate+up epilogue with 32-channel blocks (EPI 1) runs sixteen warps, two
// per lane quarter and column half, each taking one block of a 64-channel chunk.
__host__ __device__ constexpr int pair_epi_warps(int epi) { return epi == 1 ? 2 * NUM_EPI_WARPS : NUM_EPI_WARPS; }
__host__ __device__ constexpr int pair_threads(int epi) { return (EPI_WARP0 + pair_epi_warps(epi)) * 32; }
constexpr int TMEM_COLS = 512;
constexpr int SF_TMEM_BASE = 256;
constexpr int EPI_BUF = 32 * 32;  // 32 rows x 16 bf16

constexpr unsigned kErrProducer = 1u, kErrMma = 2u, kErrEpilogue = 4u, kErrDrain = 8u,
                   kErrProbe = 16u;
constexpr uint64_t kDrainNs = 2000000000ull;
constexpr uint32_t kPollHintNs = 20000;  // longest hardware sleep per poll

struct Params {
    const int32_t *offsets;  // grouped: expert row offsets [E+1]
    uint16_t *Y;
    int64_t ldy;
    int32_t E;
    int32_t M;               // rows of Y (grouped: sorted rows)
    int32_t N;
    int32_t num_kstages;     // 256-wide K stages
    int32_t num_nb;          // 256-column blocks
    int32_t n_rb;            // 128-row scale blocks of one weight
    int32_t num_full;        // whole 256-column tiles run first ...
    int32_t num_split;       // ... then the last num_split tiles as two 128-column halves
    int32_t n_fastest;       // tile order: column blocks fastest (else row-pair blocks)
    int32_t band;            // dense, column blocks fastest: row-pair blocks per band (0: none)
    // EPI != 0 (grouped gate+up with interleaved weight rows): the epilogue
    // writes the down projection's input h = SiLU(g) * u as MXFP4 instead of Y
    uint8_t *h_codes;        // [P, F/2], padded rows
    uint8_t *h_scales;       // tiled for P rows of F channels
    const float *h_f;        // down balance factors [E, F]
    int32_t F;
    int32_t h_nka;           // scale atoms per 128-row block of the down input
    int32_t h_pad_cols;      // padded scale columns of F
};

struct Tile {
    int32_t a_row;      // row coordinate in the A code tensor (= scale row block * 128)
    int32_t n0;
    int32_t expert;
    int32_t y_row0;     // first output row
    int32_t rows_valid; // rows of this tile that exist in Y
    int32_t ncols;      // 256, or 128 for half of a split tile
};

// Wait for the phase of `bar` with parity `parity`.  Each poll lets the
// thread sleep in hardware until the phase completes (up to a short hint), so
// waiting threads do not compete with the tensor cores for shared memory.
// The clock starts after the first miss; past limit_ns the wait gives up,
// raising the CTA's abort flag and the device error flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             unsigned code, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity, kPollHintNs)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity, kPollHintNs)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            atomicOr(&g_error_flags, code);
            *abort_flag = 1;
            return false;
        }
    }
}

// The same wait taken by lane 0 of a warp on behalf of the whole warp.
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag, unsigned code,
                                                  uint64_t limit_ns)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, abort_flag, code, limit_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ bool wait_fixed(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity, kPollHintNs)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity, kPollHintNs)) return true;
        if (globaltimer() - t0 > kDrainNs) {
            atomicOr(&g_error_flags, kErrDrain);
            return false;
        }
    }
}

// ------------------------------------------------------------ CTA-pair GEMM
//
// Dense GEMM on CTA pairs (tcgen05 cta_group::2).  A pair computes a 256 x 256
// tile of Y: rank r holds rows 128r..128r+127 of the tile's A and the same
// 128 rows of B (its half of the N = 256 columns); rank 0 issues one
// M = 256, N = 256, K = 64 MMA per k step, which reads both CTAs' shared
// memory and accumulates each CTA's 128 x 256 block in its own tensor
// memory.  Per 256-wide K stage a CTA so loads 32 KB of operands instead of
// the 48 KB a single-CTA M = 128, N = 256 tile needs, and the scale copies of
// one stage serve both halves of the tile.
//
// Roles (the same warps in both CTAs):
//   warp 0      TMA producer of this CTA's stage buffers (A rows, B rows,
//               A's scales, and B's scales for all 256 columns).  Both CTAs'
//               copies signal rank 0's "full" barrier (TMA .cta_group::2),
//               so it completes only when both halves of the stage are in.
//   warp 1      rank 0: MMA issuer.
//   warp 2      rank 0: scale copier (tcgen05.cp into both CTAs' tensor
//               memory, each from its own shared memory).
//   warps 3..10 epilogue, each CTA for its own 128 rows; release of the
//               accumulator is an arrival on rank 0's barrier (warps 3..18
//               for the gate+up epilogue with 32-channel blocks, EPI 1).
template <int STAGES>
struct PairLayout {
    static constexpr int BN = 256;           // tile columns (both CTAs)
    static constexpr int KB = 128;           // operand bytes per row per stage
    static constexpr int KATOMS = KB / 64;
    static constexpr int KSTEPS = KB / 32;           // MMAs (K = 64) per stage
    static constexpr int A_STAGE = BM * KB;          // this CTA's 128 rows of A
    static constexpr int B_STAGE = (BN / 2) * KB;    // this CTA's 128 rows of B
    static constexpr int SFA_STAGE = KATOMS * SF_ATOM;
    static constexpr int SFB_STAGE = (BN / 128) * KATOMS * SF_ATOM;  // all 256 columns
    static constexpr int SF_COLS = 4 * KATOMS + 4 * KATOMS * (BN / 128);
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
    static constexpr int OFF_EPI = OFF_SFB + STAGES * SFB_STAGE;
    // store staging per epilogue warp: one 32 x 16 buffer beside six stages;
    // beside five (short K: the next tile's accumulator is full after three or
    // four stages) four, beside four all eight of a warp's 16-column pieces,
    // written in batches that one proxy fence each publishes to the store unit
    static constexpr int EPI_NBUF = STAGES >= 6 ? 1 : STAGES == 5 ? 4 : 8;
    static constexpr int OFF_BAR = OFF_EPI + NUM_EPI_WARPS * EPI_NBUF * EPI_BUF;
    static constexpr int NUM_BARS = 3 * STAGES + 4;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_OFFS = OFF_MISC + 16;  // grouped: expert tables
    static constexpr int BYTES = OFF_OFFS + 3 * (static_cast<int>(kMaxExperts) + 1) * 4;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(OFF_EPI % 1024 == 0, "epilogue buffers must be 1 KB aligned");
    static_assert(STAGES * A_STAGE >= NUM_EPI_WARPS * 8 * EPI_BUF, "last tile's staging must fit the A ring");
    static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= TMEM_COLS, "tensor memory overflow");
    static_assert(ALLOC <= 232448, "shared memory");
};

// GROUPED (MoE): the rows of A are expert-grouped (each expert's rows start on
// a multiple of 128 of the padded layout, sorted rows in Y), B is [E, N, K/2].
// A pair tile is two consecutive 128-row blocks of one expert's rows; a rank
// whose block lies past its expert's rows computes nothing that is stored.
//
// EPI (grouped only): 0 stores bf16 Y; 1 and 2 are the gate+up projection of
// a gated MLP whose weight rows come interleaved in chunks of 64 channels
// (tile columns 128c .. 128c+63 are gate rows 64c .., the next 64 up rows of
// the same channels).  Each epilogue warp then holds gate and up of 64
// channels for its 32 rows, and each thread, owning one row, forms
// h = bf16(SiLU(bf16(g)) * bf16(u)) -- the values the unfused layer would
// store and re-read -- and runs the down input's transform on it in its own
// registers: balance with the expert's down factors, 32-point butterflies
// (EPI 1) or the 64-channel block (EPI 2), E8M0 scale, E2M1 codes, written to
// the down input's padded rows.  Padding rows of an expert's last block get
// zero scales; a block past the expert's rows writes nothing.
template <int STAGES, bool GROUPED, int EPI = 0>
__global__ void __launch_bounds__(pair_threads(EPI), 1)
    gemm_mxf4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmB64, const __grid_constant__ CUtensorMap tmY,
                          const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                          const Params p)
{
    using L = PairLayout<STAGES>;
    constexpr int BN = L::BN;
    constexpr int KB = L::KB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_base = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto ready_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
    const uint32_t acc_full = bar_base + 8u * (3 * STAGES);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t drain_bar = acc_full + 16u;
    const uint32_t drain_bar2 = acc_full + 24u;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    MACAQ_TRACE_EDGE(0);
    const uint64_t wait_ns = g_wait_ns;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t first_unit = blockIdx.x >> 1;
    const int64_t unit_stride = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // (rank 0's) stage is full once both CTAs' copies have landed
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);  // one MMA commit, arriving in both CTAs
            mbar_init(ready_bar(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * pair_epi_warps(EPI));  // every epilogue warp of the pair
        mbar_init(drain_bar, 1);
        mbar_init(drain_bar2, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(sbase + L::OFF_MISC, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_launch_dependents();

    int32_t *s_off = reinterpret_cast<int32_t *>(smem + L::OFF_OFFS);  // expert row offsets
    int32_t *s_ppb = s_off + (kMaxExperts + 1);    // pair-tiles before expert e
    int32_t *s_pst = s_ppb + (kMaxExperts + 1);    // first padded row of expert e
    int32_t num_mp = (p.M + 2 * BM - 1) / (2 * BM);
    int32_t num_full = p.num_full, num_split = p.num_split;
    const int nks = p.num_kstages;
    // scale atoms of stage st -> its tensor-memory slot (A: atom `at` at column
    // 4*at; B: atom `at` of row block r at 4*(2*at + r)), in both CTAs; a
    // 128-column unit reads only B's first row block
    auto copy_scales = [&](uint32_t st, bool whole) {
        const uint64_t da = smem_desc(sbase + L::OFF_SFA + st * L::SFA_STAGE, 0, 128, kSwizzleNone);
        const uint64_t db = smem_desc(sbase + L::OFF_SFB + st * L::SFB_STAGE, 0, 128, kSwizzleNone);
        const uint32_t sfa_t = tmem + SF_TMEM_BASE + st * L::SF_COLS;
        const uint32_t sfb_t = sfa_t + 4 * L::KATOMS;
        constexpr uint32_t kAtom = SF_ATOM >> 4;
#pragma unroll
        for (int at = 0; at < L::KATOMS; ++at) {
            tc_cp_pair_32x128b_warpx4(sfa_t + 4 * at, da + at * kAtom);
#pragma unroll
            for (int r = 0; r < BN / 128; ++r)
                if (r == 0 || whole)
                    tc_cp_pair_32x128b_warpx4(sfb_t + at * 4 * (BN / 128) + 4 * r, db + (r * L::KATOMS + at) * kAtom);
        }
    };
    // Tiles t run over (pair m-block t % num_mp (m fastest), n-block t / num_mp),
    // or with n_fastest over (pair m-block t / num_nb, n-block t % num_nb).
    // Units 0 .. num_full-1 are whole tiles; when the tiles do not fill the
    // last round of pairs, the remaining num_split tiles run as two units of
    // 128 columns each, so the last round takes about half as long.
    auto tile_of = [&](int64_t u, Tile &ti) {
        int64_t t = u;
        int32_t half = -1;
        if (u >= num_full) {
            t = num_full + (u - num_full) / 2;
            half = static_cast<int32_t>((u - num_full) & 1);
        }
        int32_t mp, nb;
        if (!GROUPED && p.band > 0) {
            const int64_t band_tiles = static_cast<int64_t>(p.band) * p.num_nb;
            const int32_t b = static_cast<int32_t>(t / band_tiles);
            const int32_t r = static_cast<int32_t>(t - b * band_tiles);
            const int32_t rows_in_band = min(p.band, num_mp - b * p.band);
            mp = b * p.band + r % rows_in_band;
            nb = r / rows_in_band;
        } else {
            mp = static_cast<int32_t>(p.n_fastest ? t / p.num_nb : t % num_mp);
            nb = static_cast<int32_t>(p.n_fastest ? t % p.num_nb : t / num_mp);
        }
        ti.n0 = nb * BN + (half > 0 ? BN / 2 : 0);
        ti.ncols = half < 0 ? BN : BN / 2;
        if (!GROUPED) {
            ti.a_row = mp * 2 * BM + static_cast<int32_t>(rank) * BM;
            ti.expert = 0;
            ti.y_row0 = ti.a_row;
            ti.rows_valid = min(BM, p.M - ti.a_row);
        } else {
            int lo = 0, hi = p.E;  // s_ppb[lo] <= mp < s_ppb[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_ppb[mid] <= mp) lo = mid; else hi = mid;
            }
            const int32_t blk = 2 * (mp - s_ppb[lo]) + static_cast<int32_t>(rank);
            ti.expert = lo;
            ti.a_row = s_pst[lo] + blk * BM;
            ti.y_row0 = s_off[lo] + blk * BM;
            ti.rows_valid = min(BM, s_off[lo + 1] - s_off[lo] - blk * BM);
        }
    };

    if (!GROUPED && warp == 0 && lane == 0 && first_unit < static_cast<int64_t>(num_full) + 2 * num_split) {
        // The weight does not depend on the kernel this one may overlap (A
        // does): start the first unit's weight stages towards L2 meanwhile.  A
        // prefetch is only a hint; the loads after the wait read the latest data.
        Tile ti;
        tile_of(first_unit, ti);
        const int32_t brow = ti.n0 + static_cast<int32_t>(rank) * (ti.ncols / 2);
        for (int ks = 0; ks < min(nks, STAGES); ++ks)
            tma_prefetch_2d(ti.ncols == BN ? &tmB : &tmB64, ks * KB, brow);
    }
    griddep_wait();

    if (GROUPED) {
        for (int e = threadIdx.x; e <= p.E; e += static_cast<int>(blockDim.x)) s_off[e] = p.offsets[e];
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t pairs = 0, rows = 0;
            for (int e = 0; e < p.E; ++e) {
                const int32_t blocks = (s_off[e + 1] - s_off[e] + BM - 1) / BM;
                s_ppb[e] = pairs;
                s_pst[e] = rows;
                pairs += (blocks + 1) / 2;
                rows += blocks * BM;
            }
            s_ppb[p.E] = pairs;
            s_pst[p.E] = rows;
        }
        __syncthreads();
        // the same last-round split as the host makes for dense problems
        num_mp = s_ppb[p.E];
        const int32_t tiles = num_mp * p.num_nb;
        const int32_t pairs = static_cast<int32_t>(gridDim.x >> 1);
        const int32_t rem = tiles % pairs;
        num_full = tiles;
        num_split = 0;
        if (rem > 0 && 2 * rem <= pairs) {
            num_full = tiles - rem;
            num_split = rem;
        }
    }
    const int64_t total_units = static_cast<int64_t>(num_full) + 2 * static_cast<int64_t>(num_split);
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // Every box is loaded whole (rows or scale blocks past the end of a
            // tensor are filled with zeros), so each CTA lands the same bytes
            // per stage.  Rows of A / B past the end are never stored.
            constexpr uint32_t kStageBytes = L::A_STAGE + L::B_STAGE + L::SFA_STAGE + L::SFB_STAGE;
            constexpr uint32_t kHalfBytes = kStageBytes - L::B_STAGE / 2;
            const uint32_t full0 = mapa_shared(full_bar(0), 0);
            uint32_t it = 0;
            uint32_t issued = 0;
            uint32_t last_parity = 0;
            for (int64_t u = first_unit; u < total_units; u += unit_stride) {
                Tile ti;
                tile_of(u, ti);
                const int32_t a_rb = ti.a_row / BM;
                // B's scale row blocks: the experts' tiled arrays follow one another
                const int32_t n_rb0 = ti.expert * p.n_rb + ti.n0 / 128;
                const bool whole = ti.ncols == BN;
                bool ok = true;
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    const int s = static_cast<int>(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    MACAQ_TRACE(0, it);
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kErrProducer, wait_ns)) {
                        ok = false;
                        break;
                    }
                    MACAQ_TRACE(1, it);
                    const uint32_t fb = full0 + 8u * s;
                    if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * (whole ? kStageBytes : kHalfBytes));
                    tma_load_2d_pair(sbase + L::OFF_A + s * L::A_STAGE, &tmA, fb, ks * KB, ti.a_row);
                    // this CTA's half of the tile's columns (64 of a 128-column unit)
                    const int32_t brow = ti.n0 + static_cast<int32_t>(rank) * (ti.ncols / 2);
                    if (GROUPED)
                        tma_load_3d_pair(sbase + L::OFF_B + s * L::B_STAGE, whole ? &tmB : &tmB64, fb, ks * KB,
                                         brow, ti.expert);
                    else
                        tma_load_2d_pair(sbase + L::OFF_B + s * L::B_STAGE, whole ? &tmB : &tmB64, fb, ks * KB,
                                         brow);
                    // scale blocks: (256 B, 2, k atom, 128-row block) views of the tiled layout
                    tma_load_4d_pair(sbase + L::OFF_SFA + s * L::SFA_STAGE, &tmSFA, fb, 0, 0,
                                     L::KATOMS * ks, a_rb);
                    tma_load_4d_pair(sbase + L::OFF_SFB + s * L::SFB_STAGE, &tmSFB, fb, 0, 0,
                                     L::KATOMS * ks, n_rb0);
                    issued |= 1u << s;
                    last_parity = (last_parity & ~(1u << s)) | (ph << s);
                }
                if (!ok) break;
            }
            // the copies issued into this CTA must land, and rank 0's MMAs must
            // have released every stage, before the CTA may leave (a stage is
            // released only after it landed in both CTAs)
            for (int s = 0; s < STAGES; ++s) {
                if (issued & (1u << s)) {
                    if (leader) wait_fixed(full_bar(s), (last_parity >> s) & 1u);
                    wait_fixed(empty_bar(s), (last_parity >> s) & 1u);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (rank 0)
            const uint64_t a_desc0 = smem_desc(sbase + L::OFF_A, 16, 8 * KB, kSwizzle128B);
            const uint64_t b_desc0 = smem_desc(sbase + L::OFF_B, 16, 8 * KB, kSwizzle128B);
            const uint32_t idesc0 = idesc_mxf4(2 * BM, BN, 0, 0);
            const uint32_t idesc2 = idesc_mxf4(2 * BM, BN, 2, 2);
            const uint32_t hdesc0 = idesc_mxf4(2 * BM, BN / 2, 0, 0);
            const uint32_t hdesc2 = idesc_mxf4(2 * BM, BN / 2, 2, 2);
            const uint32_t sf_t0 = tmem + SF_TMEM_BASE;
            constexpr uint32_t kAStep = L::A_STAGE >> 4, kBStep = L::B_STAGE >> 4;
            uint32_t st = 0, ph = 0, tc = 0;
            bool ok = true;
            for (int64_t u = first_unit; u < total_units && ok; u += unit_stride, ++tc) {
                const bool whole = u < num_full;
                const uint32_t d0 = whole ? idesc0 : hdesc0, d2 = whole ? idesc2 : hdesc2;
                for (int ks = 0; ks < nks; ++ks) {
                    MACAQ_TRACE(2, tc * nks + ks);
                    if (!wait_bounded(ready_bar(static_cast<int>(st)), ph, abort_flag, kErrMma, wait_ns)) {
                        ok = false;
                        break;
                    }
                    MACAQ_TRACE(3, tc * nks + ks);
                    if (ks == 0) {
                        // both CTAs' epilogues must have drained the previous accumulator
                        MACAQ_TRACE(4, tc);
                        if (!wait_bounded(acc_empty, (tc & 1u) ^ 1u, abort_flag, kErrMma, wait_ns)) {
                            ok = false;
                            break;
                        }
                        MACAQ_TRACE(5, tc);
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = sf_t0 + st * L::SF_COLS;
                    const uint32_t sfb_t = sfa_t + 4 * L::KATOMS;
                    const uint64_t ad = a_desc0 + st * kAStep;
                    const uint64_t bd = b_desc0 + st * kBStep;
#pragma unroll
                    for (int j = 0; j < L::KSTEPS; ++j)
                        tc_mma_mxf4_pair(tmem, ad + 2 * j, bd + 2 * j, (j & 1) ? d2 : d0,
                                         sfa_t + 4 * (j >> 1), sfb_t + 4 * (BN / 128) * (j >> 1),
                                         (ks > 0 || j > 0) ? 1u : 0u);
                    // the stage's buffers in both CTAs may be refilled once these MMAs read them
                    tc_commit_pair_mc(empty_bar(static_cast<int>(st)), 3);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) tc_commit_pair_mc(acc_full, 3);
            }
            tc_commit_pair(drain_bar);
            wait_fixed(drain_bar, 0);
        }
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ scale copier (rank 0)
            uint32_t st = 0, ph = 0, it = 0;
            bool ok = true;
            for (int64_t u = first_unit; u < total_units && ok; u += unit_stride) {
                const bool whole = u < num_full;
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    // both CTAs' data of the stage have landed
                    MACAQ_TRACE(9, it);
                    if (!wait_bounded(full_bar(static_cast<int>(st)), ph, abort_flag, kErrMma, wait_ns)) {
                        ok = false;
                        break;
                    }
                    MACAQ_TRACE(10, it);
                    copy_scales(st, whole);
                    tc_commit_pair(ready_bar(static_cast<int>(st)));
                    MACAQ_TRACE(11, it);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            tc_commit_pair(drain_bar2);
            wait_fixed(drain_bar2, 0);
        }
        __syncwarp();
    } else if constexpr (EPI == 1) {
        // ------------------------------------ epilogue: gate+up, 32-channel blocks
        // warp (q, half, sub): rows 32q.. of this CTA, channels 32 sub .. of the
        // 64-channel chunk in columns half * 128 .. (gate columns 32 sub .., up
        // columns 64 + 32 sub ..): one MX block of h per row
        const int ew = warp - EPI_WARP0;
        const int q = warp & 3;
        const int half = (ew >> 2) & 1;
        const int sub = ew >> 3;
        const uint32_t leader_acc_empty = mapa_shared(acc_empty, 0);
        uint32_t tc = 0;
        for (int64_t u = first_unit; u < total_units; u += unit_stride, ++tc) {
            Tile ti;
            tile_of(u, ti);
            if (warp == EPI_WARP0) MACAQ_TRACE(6, tc);
            if (!warp_wait_bounded(acc_full, tc & 1u, abort_flag, kErrEpilogue, wait_ns)) break;
            if (warp == EPI_WARP0) MACAQ_TRACE(7, tc);
            tc_fence_after();
            uint32_t g[32], up[32];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + half * 128 + 32 * sub;
            tmem_ld_32x32b_x32(taddr, g);
            tmem_ld_32x32b_x32(taddr + 64, up);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_acc_empty);
            if (warp == EPI_WARP0) MACAQ_TRACE(8, tc);

            if (ti.rows_valid <= 0 || half * 128 >= ti.ncols) continue;
            const int32_t c0 = ((ti.n0 + half * 128) >> 7) * 64 + 32 * sub;  // this warp's 32 channels
            if (c0 >= p.F) continue;
            const int r = 32 * q + lane;
            const int64_t prow = static_cast<int64_t>(ti.a_row) + r;
            uint32_t sbyte = 0;
            if (r < ti.rows_valid) {
                uint32_t h[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __nv_bfloat162 gb = __floats2bfloat162_rn(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
                    const __nv_bfloat162 ub =
                        __floats2bfloat162_rn(__uint_as_float(up[2 * i]), __uint_as_float(up[2 * i + 1]));
                    h[i] = mx::silu_mul_word(*reinterpret_cast<const uint32_t *>(&gb),
                                             *reinterpret_cast<const uint32_t *>(&ub));
                }
                const float4 *f4 = reinterpret_cast<const float4 *>(p.h_f + static_cast<int64_t>(ti.expert) * p.F + c0);
                float2 f[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 a4 = __ldg(f4 + j);
                    f[2 * j] = make_float2(a4.x, a4.y);
                    f[2 * j + 1] = make_float2(a4.z, a4.w);
                }
                uint4 codes;
                sbyte = mx::quant_block_pairs<false>(h, f, codes);
                *reinterpret_cast<uint4 *>(p.h_codes + prow * (p.F / 2) + c0 / 2) = codes;
            }
            // the row's scale byte (zero on padding rows), and after the last
            // block the row's padding scale columns
            const int64_t rb = (prow >> 7) * p.h_nka;
            const int64_t in_atom = (prow & 31) * 16 + ((prow & 127) >> 5) * 4;
            const int32_t kb = c0 / 32;
            p.h_scales[(rb + (kb >> 2)) * 512 + in_atom + (kb & 3)] = static_cast<uint8_t>(sbyte);
            if (c0 + 32 == p.F) {
                for (int32_t k2 = kb + 1; k2 < p.h_pad_cols; ++k2)
                    p.h_scales[(rb + (k2 >> 2)) * 512 + in_atom + (k2 & 3)] = 0;
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue
        const int ew = warp - EPI_WARP0;
        const int q = warp & 3;
        const int half = ew >> 2;
        const uint32_t ebuf = sbase + L::OFF_EPI + ew * L::EPI_NBUF * EPI_BUF;
        const uint32_t leader_acc_empty = mapa_shared(acc_empty, 0);
        uint32_t tc = 0, chunk = 0;
        for (int64_t u = first_unit; u < total_units; u += unit_stride, ++tc) {
            Tile ti;
            tile_of(u, ti);
            if (warp == EPI_WARP0) MACAQ_TRACE(6, tc);
            if (!warp_wait_bounded(acc_full, tc & 1u, abort_flag, kErrEpilogue, wait_ns)) break;
            if (warp == EPI_WARP0) MACAQ_TRACE(7, tc);
            tc_fence_after();
            uint32_t acc[4][32];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + 32 * c, acc[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_acc_empty);
            if (warp == EPI_WARP0) MACAQ_TRACE(8, tc);

            const int row0 = 32 * q;
            if constexpr (EPI != 0) {
                if (ti.rows_valid <= 0 || half * 128 >= ti.ncols) continue;
                const int32_t c0 = ((ti.n0 + half * 128) >> 7) * 64;  // this warp's 64 channels
                if (c0 >= p.F) continue;
                const int r = row0 + lane;
                const int64_t prow = static_cast<int64_t>(ti.a_row) + r;
                uint32_t sw = 0;
                if (r < ti.rows_valid) {
                    uint32_t hlo[16], hhi[16];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int gc = 2 * i, uc = 64 + 2 * i;
                        const __nv_bfloat162 gb = __floats2bfloat162_rn(__uint_as_float(acc[gc >> 5][gc & 31]),
                                                                        __uint_as_float(acc[gc >> 5][(gc & 31) + 1]));
                        const __nv_bfloat162 ub = __floats2bfloat162_rn(__uint_as_float(acc[uc >> 5][uc & 31]),
                                                                        __uint_as_float(acc[uc >> 5][(uc & 31) + 1]));
                        const uint32_t hw = mx::silu_mul_word(*reinterpret_cast<const uint32_t *>(&gb),
                                                              *reinterpret_cast<const uint32_t *>(&ub));
                        if (i < 16) hlo[i] = hw; else hhi[i - 16] = hw;
                    }
                    const float4 *f4 = reinterpret_cast<const float4 *>(
                        p.h_f + static_cast<int64_t>(ti.expert) * p.F + c0);
                    float2 flo[16], fhi[16];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 a4 = __ldg(f4 + j);
                        const float4 b4 = __ldg(f4 + 8 + j);
                        flo[2 * j] = make_float2(a4.x, a4.y);
                        flo[2 * j + 1] = make_float2(a4.z, a4.w);
                        fhi[2 * j] = make_float2(b4.x, b4.y);
                        fhi[2 * j + 1] = make_float2(b4.z, b4.w);
                    }
                    uint4 clo, chi;
                    uint32_t slo, shi;
                    if constexpr (EPI == 1) {
                        slo = mx::quant_block_pairs<false>(hlo, flo, clo);
                        shi = mx::quant_block_pairs<false>(hhi, fhi, chi);
                    } else {
                        mx::quant_block64_pairs(hlo, hhi, flo, fhi, clo, chi, slo, shi);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(p.h_codes + prow * (p.F / 2) + c0 / 2);
                    dst[0] = clo;
                    dst[1] = chi;
                    sw = slo | (shi << 8);
                }
                // the row's two scale bytes (zero on padding rows), and on the
                // last chunk the row's padding scale columns
                const int64_t rb = (prow >> 7) * p.h_nka;
                const int64_t in_atom = (prow & 31) * 16 + ((prow & 127) >> 5) * 4;
                const int32_t kb0 = c0 / 32;
                *reinterpret_cast<uint16_t *>(p.h_scales + (rb + (kb0 >> 2)) * 512 + in_atom + (kb0 & 3)) =
                    static_cast<uint16_t>(sw);
                if (c0 + 64 == p.F) {
                    for (int32_t kb = kb0 + 2; kb < p.h_pad_cols; ++kb)
                        p.h_scales[(rb + (kb >> 2)) * 512 + in_atom + (kb & 3)] = 0;
                }
                continue;
            }
            const bool any_row = row0 < ti.rows_valid;
            if (!any_row || half * 128 >= ti.ncols) continue;
            // Grouped: rows past an expert's last row belong to the next expert
            // in Y, so a warp with some of them stores row by row.
            const bool use_tma = !GROUPED || row0 + 32 <= ti.rows_valid;
            const bool my_row = row0 + lane < ti.rows_valid;
            // Staging in batches of NB 16-column pieces (1 KB each) from sbuf:
            // each batch is written, published to the store unit with one proxy
            // fence and stored, after the previous batch's stores have read it.
            auto store_batched = [&](auto nb_c, uint32_t sbuf) {
                constexpr int NB = decltype(nb_c)::value;
#pragma unroll
                for (int c0 = 0; c0 < 8; c0 += NB) {
                    // the previous batch's stores must be done reading the staging
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    int nchunks = 0;
#pragma unroll
                    for (int c = c0; c < c0 + NB; ++c) {
                        if (ti.n0 + half * 128 + 16 * c >= p.N) break;
                        uint32_t packed[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float lo = __uint_as_float(acc[c >> 1][(c & 1) * 16 + 2 * i]);
                            const float hi = __uint_as_float(acc[c >> 1][(c & 1) * 16 + 2 * i + 1]);
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                            packed[i] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        const uint32_t buf = sbuf + (c - c0) * EPI_BUF;
                        const uint32_t sw = (lane >> 2) & 1;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 32 + 16 * sw),
                                     "r"(packed[0]), "r"(packed[1]), "r"(packed[2]), "r"(packed[3])
                                     : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 32 + 16 * (1 ^ sw)),
                                     "r"(packed[4]), "r"(packed[5]), "r"(packed[6]), "r"(packed[7])
                                     : "memory");
                        ++nchunks;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        // rows past M and columns past N are clipped by the stores
                        for (int c = 0; c < nchunks; ++c)
                            tma_store_2d(&tmY, sbuf + c * EPI_BUF, ti.n0 + half * 128 + 16 * (c0 + c),
                                         ti.y_row0 + row0);
                        bulk_commit();
                    }
                    if (nchunks < NB) break;
                }
            };
            if (use_tma && u + unit_stride >= total_units) {
                // The CTA's last tile: the accumulator is full, so every MMA has
                // read its stages, and no stage is loaded again; the A part of
                // the operand ring (at least 80 KB) stages all eight of this
                // warp's pieces at once (8 KB per warp).
                store_batched(std::integral_constant<int, 8>{}, sbase + L::OFF_A + ew * 8 * EPI_BUF);
            } else if (L::EPI_NBUF >= 4 && use_tma) {
                store_batched(std::integral_constant<int, L::EPI_NBUF>{}, ebuf);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int32_t ncol = ti.n0 + half * 128 + 16 * c;
                    if (ncol >= p.N) break;
                    uint32_t packed[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float lo = __uint_as_float(acc[c >> 1][(c & 1) * 16 + 2 * i]);
                        const float hi = __uint_as_float(acc[c >> 1][(c & 1) * 16 + 2 * i + 1]);
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                        packed[i] = *reinterpret_cast<const uint32_t *>(&b2);
                    }
                    if (!use_tma) {
                        if (my_row) {
                            uint16_t *dst = p.Y + static_cast<int64_t>(ti.y_row0 + row0 + lane) * p.ldy + ncol;
                            if (ncol + 16 <= p.N) {
                                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
                                d4[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                                d4[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                            } else {
                                for (int i = 0; i < 16 && ncol + i < p.N; ++i)
                                    dst[i] = static_cast<uint16_t>(packed[i >> 1] >> (16 * (i & 1)));
                            }
                        }
                    } else {
                        // rows past M and columns past N are clipped by the store
                        const uint32_t buf = ebuf + (chunk % L::EPI_NBUF) * EPI_BUF;
                        ++chunk;
                        // the store that last read this buffer must be done with it
                        if (lane == 0) {
                            bulk_wait_read_le<L::EPI_NBUF - 1>();
                        }
                        __syncwarp();
                        const uint32_t sw = (lane >> 2) & 1;
                        const uint32_t r0 = buf + lane * 32 + 16 * (0 ^ sw);
                        const uint32_t r1 = buf + lane * 32 + 16 * (1 ^ sw);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(r0), "r"(packed[0]),
                                     "r"(packed[1]), "r"(packed[2]), "r"(packed[3])
                                     : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(r1), "r"(packed[4]),
                                     "r"(packed[5]), "r"(packed[6]), "r"(packed[7])
                                     : "memory");
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmY, buf, ncol, ti.y_row0 + row0);
                            bulk_commit();
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    __syncthreads();
    MACAQ_TRACE_EDGE(1);
    // neither CTA may leave (or free tensor memory) while its peer can still
    // touch its shared memory, barriers or tensor memory
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, TMEM_COLS);
}

#include "gemm_skinny.cuh"
#include "gemm_w4a16.cuh"

__global__ void wait_probe_kernel()
{
    __shared__ alignas(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        wait_bounded(smem_u32(&bar), 0, &abort_flag, kErrProbe, g_wait_ns);
    }
}


// Tensor-core rate probe: one CTA per SM issues `iters` x 4 back-to-back
// kind::mxf4 block-scaled MMAs (M=128, N=bn, K=64) on operands resident in
// shared memory and reports the elapsed SM cycles and nanoseconds.
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int bn_mode, int iters, unsigned long long *out, const uint8_t *src)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    // A 16 KB | B 32 KB | SFA 1 KB | SFB 2 KB | barrier | tmem slot
    const uint32_t a_s = sbase, b_s = sbase + 16384, sfa_s = sbase + 49152, sfb_s = sbase + 50176;
    const int bn = bn_mode & 0xffff;
    const uint32_t bar = sbase + 52224;
    const uint32_t bar2 = sbase + 52240;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + 52232);
    for (int i = threadIdx.x; i < 52224 / 4; i += blockDim.x) {
        const uint32_t x = static_cast<uint32_t>(i) * 2654435761u;
        // codes: any byte is a finite E2M1 pair; scales: keep near 2^0
        reinterpret_cast<uint32_t *>(smem)[i] = (i < 49152 / 4) ? x : 0x7f7f7f7fu;
    }
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_init(bar2, 1);
        mbar_init(sbase + 52256, 1);
        *reinterpret_cast<volatile int *>(smem + 52264) = 0;
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(sbase + 52232, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        const uint32_t sfa_t = tmem + 256, sfb_t = tmem + 264;
        for (int at = 0; at < 2; ++at) {
            tc_cp_32x128b_warpx4(sfa_t + 4 * at, smem_desc(sfa_s + at * 512, 0, 128, kSwizzleNone));
            for (int r = 0; r < 2; ++r)
                tc_cp_32x128b_warpx4(sfb_t + at * 8 + 4 * r,
                                     smem_desc(sfb_s + r * 1024 + at * 512, 0, 128, kSwizzleNone));
        }
        const int nsf = (bn + 127) / 128;
        const int mode = bn_mode >> 16;
        const long long c0 = clock64();
        const uint64_t t0 = globaltimer();
        for (int it = 0; it < iters; ++it) {
            if (mode >= 1) {
                // the scale copies one 256-wide K stage of the GEMM issues
                const uint32_t sa = tmem + SF_TMEM_BASE + (it & 3) * 24, sb = sa + 8;
                for (int at = 0; at < 2; ++at) {
                    tc_cp_32x128b_warpx4(sa + 4 * at, smem_desc(sfa_s + at * 512, 0, 128, kSwizzleNone));
                    for (int r = 0; r < 2; ++r)
                        tc_cp_32x128b_warpx4(sb + at * 8 + 4 * r,
                                             smem_desc(sfb_s + r * 1024 + at * 512, 0, 128, kSwizzleNone));
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t sf_id = (j & 1) * 2;
                tc_mma_mxf4(tmem, smem_desc(a_s + 32 * j, 16, 1024, kSwizzle128B),
                            smem_desc(b_s + 32 * j, 16, 1024, kSwizzle128B),
                            idesc_mxf4(BM, static_cast<uint32_t>(bn), sf_id, sf_id),
                            sfa_t + 4 * (j >> 1), sfb_t + 4 * nsf * (j >> 1), (it | j) != 0 ? 1u : 0u);
            }
            if (mode >= 2) tc_commit(bar2);
        }
        tc_commit(bar);
        wait_fixed(bar, 0);
        const long long c1 = clock64();
        const uint64_t t1 = globaltimer();
        out[2 * blockIdx.x] = static_cast<unsigned long long>(c1 - c0);
        out[2 * blockIdx.x + 1] = t1 - t0;
        *reinterpret_cast<volatile int *>(smem + 52264) = 1;
    }
    if (threadIdx.x == 64 && (bn_mode >> 16) == 3 && src != nullptr) {
        // shared-memory write traffic next to the MMAs: 16 KB bulk copies from
        // an L2-resident buffer into a 64 KB region, four in flight
        const uint32_t region = sbase + 53248, lbar = sbase + 52256;
        uint64_t bytes = 0;
        uint32_t ph = 0;
        while (*reinterpret_cast<volatile int *>(smem + 52264) == 0) {
            mbar_arrive_expect_tx(lbar, 4 * 16384);
            for (int i = 0; i < 4; ++i)
                bulk_load(region + i * 16384, src + ((bytes / 16384 + i) % 64) * 16384, 16384, lbar);
            wait_fixed(lbar, ph);
            ph ^= 1;
            bytes += 4 * 16384;
        }
        out[2 * gridDim.x + blockIdx.x] = bytes;
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}


// ------------------------------------------------------------- host side

bool encode(CUtensorMap *m, CUtensorMapDataType dt, uint32_t rank, const void *base,
            const uint64_t *dims, const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle sw)
{
    return encode_tensor_map(m, dt, rank, base, dims, strides, box, sw);
}

bool encode_4d(CUtensorMap *m, const void *base, const uint64_t *dims, const uint64_t *strides,
               const uint32_t *box)
{
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
}

struct DeviceInfo {
    int sms = 0;
    bool attr_set[16] = {};
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

// Dense (GROUPED = false) or expert-grouped GEMM on CTA pairs; EPI as the kernel.
template <int STAGES, bool GROUPED, int EPI = 0>
cudaError_t launch_pair(const GemmArgs &g, cudaStream_t stream, int slot)
{
    using L = PairLayout<STAGES>;
    constexpr int BN = L::BN, KB = L::KB;
    constexpr CUtensorMapSwizzle kSw = CU_TENSOR_MAP_SWIZZLE_128B;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kern = gemm_mxf4_pair_kernel<STAGES, GROUPED, EPI>;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        DeviceInfo &di = g_dev[dev];
        if (di.sms == 0) {
            err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
            if (err != cudaSuccess) return err;
        }
        if (!di.attr_set[slot]) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
            if (err != cudaSuccess) return err;
            di.attr_set[slot] = true;
        }
    }
    const int sms = g_dev[dev].sms;

    const uint64_t kb = static_cast<uint64_t>(g.K / 2);
    // A: 128-row boxes; B: each CTA's 128 rows (64 for a split tile's halves),
    // per expert when grouped; Y: 32 x 16 store boxes
    CUtensorMap tmA, tmB, tmB64, tmY;
    {
        uint64_t dims[2] = {kb, static_cast<uint64_t>(g.a_rows)};
        uint64_t strides[1] = {kb};
        uint32_t box[2] = {KB, BM};
        if (!encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g.a_codes, dims, strides, box, kSw))
            return cudaErrorInvalidValue;
    }
    for (int which = 0; which < 2; ++which) {
        CUtensorMap *m = which == 0 ? &tmB : &tmB64;
        const uint32_t rows = which == 0 ? BN / 2 : BN / 4;
        if (GROUPED) {
            uint64_t dims[3] = {kb, static_cast<uint64_t>(g.N), static_cast<uint64_t>(g.E)};
            uint64_t strides[2] = {kb, kb * static_cast<uint64_t>(g.N)};
            uint32_t box[3] = {KB, rows, 1};
            if (!encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, g.w_codes, dims, strides, box, kSw))
                return cudaErrorInvalidValue;
        } else {
            uint64_t dims[2] = {kb, static_cast<uint64_t>(g.N)};
            uint64_t strides[1] = {kb};
            uint32_t box[2] = {KB, rows};
            if (!encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g.w_codes, dims, strides, box, kSw))
                return cudaErrorInvalidValue;
        }
    }
    if (EPI == 0) {
        uint64_t dims[2] = {static_cast<uint64_t>(g.N), static_cast<uint64_t>(g.M)};
        uint64_t strides[1] = {static_cast<uint64_t>(g.ldy) * 2};
        uint32_t box[2] = {16, 32};
        if (!encode(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.Y, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_32B))
            return cudaErrorInvalidValue;
    } else {
        std::memset(&tmY, 0, sizeof(tmY));  // no bf16 output: never read
    }
    // Scale blocks: the tiled layout viewed as (256 B, 2 halves of a 512-byte
    // atom, k atom, 128-row block); grouped weights: the experts' tiled arrays
    // one after another.
    CUtensorMap tmSFA, tmSFB;
    {
        const uint64_t nka = static_cast<uint64_t>(pad_scale_cols(g.K) / 4);
        uint64_t strides[3] = {256, 512, nka * 512};
        uint64_t dims_a[4] = {256, 2, nka, static_cast<uint64_t>(pad_rows(g.a_rows) / 128)};
        uint32_t box_a[4] = {256, 2, 2, 1};
        if (!encode_4d(&tmSFA, g.a_scales, dims_a, strides, box_a)) return cudaErrorInvalidValue;
        const uint64_t experts = GROUPED ? static_cast<uint64_t>(g.E) : 1;
        uint64_t dims_b[4] = {256, 2, nka, experts * static_cast<uint64_t>(pad_rows(g.N) / 128)};
        uint32_t box_b[4] = {256, 2, 2, 2};
        if (!encode_4d(&tmSFB, g.w_scales, dims_b, strides, box_b)) return cudaErrorInvalidValue;
    }

    Params p;
    p.offsets = g.offsets;
    p.Y = static_cast<uint16_t *>(g.Y);
    p.ldy = g.ldy;
    p.E = g.E;
    p.M = static_cast<int32_t>(g.M);
    p.N = static_cast<int32_t>(g.N);
    p.num_kstages = static_cast<int32_t>((g.K + 2 * KB - 1) / (2 * KB));
    p.num_nb = static_cast<int32_t>((g.N + BN - 1) / BN);
    p.n_rb = static_cast<int32_t>((g.N + 127) / 128);
    p.h_codes = g.h_codes;
    p.h_scales = g.h_scales;
    p.h_f = g.h_f;
    p.F = static_cast<int32_t>(g.N / 2);
    p.h_nka = static_cast<int32_t>(pad_scale_cols(g.N / 2) / 4);
    p.h_pad_cols = static_cast<int32_t>(pad_scale_cols(g.N / 2));
    // column blocks fastest when A would not stay in L2 across a pass over
    // the column blocks: grouped A (each expert's rows then meet all of its
    // weight tiles in a row, so an expert's weight tile is read once for both
    // of its pair tiles), and dense A of more than half of L2
    p.n_fastest = (GROUPED || static_cast<uint64_t>(g.a_rows) * kb > (64ull << 20)) ? 1 : 0;
    // dense with a large A: tiles go in bands of `band` row-pair blocks, row
    // pairs fastest inside a band and the column blocks swept band by band, so
    // that a round of tiles touches a few column blocks of B and one band of A
    // (which stays in L2 while the band's columns pass), not all of B
    // (a band of about 40 MB of A: 12 row pairs at K = 25600, 3-5 % faster
    // than sweeping all column blocks per row pair on the down projection)
    p.band = 0;
    if (!GROUPED && p.n_fastest) {
        const uint64_t pair_bytes = 2 * BM * (kb + kb / 16);
        int64_t band = static_cast<int64_t>((40ull << 20) / (pair_bytes ? pair_bytes : 1));
        band = band < 2 ? 2 : band;
        p.band = static_cast<int32_t>(band);
    }

    const int64_t pairs_max = sms / 2;
    int64_t units;
    if (GROUPED) {
        // at most (padded blocks / 2 + one odd block per expert) pair tiles per
        // column block; the kernel counts the exact number and splits its tail
        units = (g.a_rows / BM / 2 + g.E) * p.num_nb;
        p.num_full = static_cast<int32_t>(units);
        p.num_split = 0;
    } else {
        units = static_cast<int64_t>((g.M + 2 * BM - 1) / (2 * BM)) * p.num_nb;
        p.num_full = static_cast<int32_t>(units);
        p.num_split = 0;
        // tiles that would run in a last, partly filled round of pairs run as
        // two 128-column halves instead (when the halves fit in that round)
        const int64_t rem = units % pairs_max;
        if (rem > 0 && 2 * rem <= pairs_max) {
            p.num_full = static_cast<int32_t>(units - rem);
            p.num_split = static_cast<int32_t>(rem);
            units += rem;
        }
    }
    int64_t pairs = units < pairs_max ? units : pairs_max;
    if (pairs < 1) pairs = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(pair_threads(EPI));
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmB64, tmY, tmSFA, tmSFB, p);
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}
}  // namespace

bool encode_tensor_map(CUtensorMap *m, CUtensorMapDataType dt, uint32_t rank, const void *base,
                       const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                       CUtensorMapSwizzle sw)
{
    auto fn = encode_fn();
    if (!fn) return false;
    uint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, dt, rank, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FUSED: x / ldx / inv carry the layer input and balance factors, and the
// kernel forms the token operand itself (a_codes / a_scales unused).
template <int NT, int STAGES, bool FUSED = false>
cudaError_t launch_skinny(const GemmArgs &g, cudaStream_t stream, int slot, const uint16_t *x = nullptr,
                          int64_t ldx = 0, const float *inv = nullptr)
{
    using L = skinny::Layout<NT, STAGES>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kern = skinny::gemm_mxf4_skinny_kernel<NT, STAGES, FUSED>;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        DeviceInfo &di = g_dev[dev];
        if (di.sms == 0) {
            err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
            if (err != cudaSuccess) return err;
        }
        if (!di.attr_set[slot]) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
            if (err != cudaSuccess) return err;
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (err != cudaSuccess) return err;
            di.attr_set[slot] = true;
        }
    }
    const int sms = g_dev[dev].sms;
    const uint64_t kb = static_cast<uint64_t>(g.K / 2);
    CUtensorMap tmW, tmX;
    {
        uint64_t dims[2] = {kb, static_cast<uint64_t>(g.N)};
        uint64_t strides[1] = {kb};
        uint32_t box[2] = {128, 128};
        if (!encode(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g.w_codes, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (FUSED) {
        std::memset(&tmX, 0, sizeof(tmX));  // the token operand is formed in the kernel: never read
    } else {
        uint64_t dims[2] = {kb, static_cast<uint64_t>(g.M)};
        uint64_t strides[1] = {kb};
        uint32_t box[2] = {128, NT};
        if (!encode(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g.a_codes, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    skinny::Params p;
    p.sfw = g.w_scales;
    p.sfx = g.a_scales;
    p.x = x;
    p.ldx = ldx;
    p.inv = inv;
    p.nkb = static_cast<int32_t>(g.K / 32);
    p.weight_early = (!FUSED && g.weight_early) ? 1 : 0;
    p.Y = static_cast<uint16_t *>(g.Y);
    p.ldy = g.ldy;
    p.M = static_cast<int32_t>(g.M);
    p.N = static_cast<int32_t>(g.N);
    p.num_kstages = static_cast<int32_t>((g.K + 255) / 256);
    p.nka = static_cast<int32_t>(pad_scale_cols(g.K) / 4);
    // split K over a cluster while there are fewer weight tiles than SMs
    const int64_t n_tiles = (g.N + 127) / 128;
    int ks = 1;
    while (n_tiles * ks < sms && ks < 8 && 2 * ks <= p.num_kstages) ks *= 2;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_tiles * ks));
    cfg.blockDim = dim3(skinny::skinny_threads(FUSED));
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, p);
}

// W4A16: token tile NT (16 .. 256); RS raw stages and XS expanded tiles as
// shared memory allows (small tiles: two CTAs per SM, the epilogue in the
// expander warps).
template <int NT, int RS, int XS, bool kSepEpi>
cudaError_t launch_w4a16_tile(const W4A16Args &g, cudaStream_t stream, int slot)
{
    using L = w4a16::Layout<NT, RS, XS, kSepEpi>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kern = w4a16::gemm_w4a16_kernel<NT, RS, XS, kSepEpi>;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        DeviceInfo &di = g_dev[dev];
        if (di.sms == 0) {
            err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
            if (err != cudaSuccess) return err;
        }
        if (!di.attr_set[slot]) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
            if (err != cudaSuccess) return err;
            // all of the unified L1 as shared memory, so that two CTAs of the
            // small-tile variants fit on an SM
            err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
            if (err != cudaSuccess) return err;
            di.attr_set[slot] = true;
        }
    }
    const int sms = g_dev[dev].sms;
    CUtensorMap tmX, tmWc;
    {
        uint64_t dims[2] = {static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M)};
        uint64_t strides[1] = {static_cast<uint64_t>(g.ldx) * 2};
        uint32_t box[2] = {64, NT};
        if (!encode(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.Xt, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        uint64_t dims[2] = {static_cast<uint64_t>(g.K / 2), static_cast<uint64_t>(g.N)};
        uint64_t strides[1] = {static_cast<uint64_t>(g.K / 2)};
        uint32_t box[2] = {32, 128};
        if (!encode(&tmWc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, g.w_codes, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    w4a16::Params p;
    p.sfw = g.w_scales;
    p.Y = static_cast<uint16_t *>(g.Y);
    p.ldy = g.ldy;
    p.M = static_cast<int32_t>(g.M);
    p.N = static_cast<int32_t>(g.N);
    p.num_kstages = static_cast<int32_t>((g.K + 63) / 64);
    p.nka = static_cast<int32_t>(pad_scale_cols(g.K) / 4);
    p.n_wb = static_cast<int32_t>((g.N + 127) / 128);
    const int64_t tiles = static_cast<int64_t>((g.M + NT - 1) / NT) * p.n_wb;
    if (tiles > (int64_t{1} << 30)) return cudaErrorInvalidValue;
    p.n_tiles = static_cast<int32_t>(tiles);
    // CTAs resident per SM by shared memory (1 KB reserved per CTA): every
    // tile gets its own CTA while they all fit, else a persistent grid
    int smem_sm = 0;
    err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (err != cudaSuccess) return err;
    int per_sm = smem_sm / (L::ALLOC + 1024);
    per_sm = per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm);
    const int64_t slots = static_cast<int64_t>(sms) * per_sm;
    const int64_t grid = tiles < slots ? tiles : slots;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(L::THREADS);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmX, tmWc, p);
}

cudaError_t launch_w4a16_gemm(const W4A16Args &g, cudaStream_t stream)
{
    if (g.M <= 16) return launch_w4a16_tile<16, 8, 3, false>(g, stream, 8);
    if (g.M <= 32) return launch_w4a16_tile<32, 6, 3, false>(g, stream, 9);
    if (g.M <= 64) return launch_w4a16_tile<64, 4, 3, false>(g, stream, 10);
    if (g.M <= 128) return launch_w4a16_tile<128, 6, 3, true>(g, stream, 11);
    return launch_w4a16_tile<256, 4, 3, true>(g, stream, 12);
}

cudaError_t launch_gemm(const GemmArgs &g, cudaStream_t stream)
{
    // a few token rows: weight rows on the MMA's M side (decode)
    if (g.E == 0 && g.M <= 16) return launch_skinny<16, 5>(g, stream, 4);
    if (g.E == 0 && g.M <= 32) return launch_skinny<32, 5>(g, stream, 5);
    if (g.E == 0 && g.M <= 64) return launch_skinny<64, 4>(g, stream, 6);
    // everything else: CTA pairs on 256 x 256 tiles (grouped: per-expert B)
    if (g.E > 0 && g.epi == 1) return launch_pair<6, true, 1>(g, stream, 0);
    if (g.E > 0 && g.epi == 2) return launch_pair<6, true, 2>(g, stream, 1);
    // at most four 256-wide K stages per tile: five stages and batched store
    // staging (four 16-column pieces per warp and proxy fence)
    const bool short_k = g.K <= 4 * 256;
    if (g.E > 0) return short_k ? launch_pair<5, true>(g, stream, 13) : launch_pair<6, true>(g, stream, 7);
    return short_k ? launch_pair<5, false>(g, stream, 14) : launch_pair<6, false>(g, stream, 3);
}

cudaError_t launch_linear_fused(const GemmArgs &g, const uint16_t *X, int64_t ldx, const float *inv_s,
                                cudaStream_t stream)
{
    if (g.E != 0 || g.M > kFusedLinearMaxRows) return cudaErrorNotSupported;
    return launch_skinny<16, 5, true>(g, stream, 15, X, ldx, inv_s);
}

cudaError_t read_and_clear_device_error(unsigned *flags)
{
    cudaError_t err = cudaMemcpyFromSymbol(flags, g_error_flags, sizeof(unsigned));
    if (err != cudaSuccess) return err;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_error_flags, &zero, sizeof(unsigned));
}

cudaError_t set_wait_timeout_ns(uint64_t ns)
{
    const unsigned long long v = ns;
    return cudaMemcpyToSymbol(g_wait_ns, &v, sizeof(v));
}

cudaError_t launch_wait_probe(cudaStream_t stream)
{
    wait_probe_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t launch_mma_rate(int bn, int iters, unsigned long long *out, const uint8_t *src, int ctas,
                            cudaStream_t stream)
{
    const int smem = 53248 + 65536 + 1024;
    cudaError_t err = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    mma_rate_kernel<<<ctas, 128, smem, stream>>>(bn, iters, out, src);
    return cudaGetLastError();
}


}  // namespace macaq
