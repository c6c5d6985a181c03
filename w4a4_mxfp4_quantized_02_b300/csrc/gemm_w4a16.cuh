// W4A16 GEMM: bf16 activations times MXFP4 weights expanded to bf16 on chip.
//
// The weight-only fallback (page "Huawei MACaQ: Choosing GGUF or vLLM and
// Avoiding Setup Mistakes", section "vLLM checkpoints have different
// constraints": the weights are expanded for a BF16 matrix multiplication).
// Here the expansion happens in shared memory, tile by tile, so the weights
// are read from HBM at 4.25 bits per value (codes plus E8M0 scales), never as
// a bf16 copy:
//     Y[m, n] = bf16_rn( sum_k Xt[m, k] * Wd(n, k) ),  Wd(n, k) = E2M1 code
//               times 2^(scale - 127), exactly representable in bf16,
// products of bf16 values accumulated in fp32 on the tensor cores
// (tcgen05 kind::f16).
//
// Included by gemm.cu (it shares that unit's error flags, wait helpers and
// tensor-map encoder).  Roles swap as in the few-rows kernel: the MMA's
// M = 128 rows are weight rows (one 128-row weight block per tile), its N = NT
// columns token rows (16 .. 256; rows past M read as zeros).  Tiles
// (token block, weight block) run weight blocks fastest, persistently.
//
// Two rings: RS stages of what TMA brings per 64-wide K stage (the NT x 64
// bf16 activation tile, 128-byte swizzled; the 128 x 32-byte code tile; the
// 512-byte scale atom of the weight block), and XS buffers of expanded weight
// tiles (128 x 64 bf16 in the 128-byte swizzled K-major layout the MMA
// reads), so many raw stages stay in flight while only a few expanded tiles
// take shared memory.
// Warps: 0 TMA producer, 1 MMA issuer, 2..9 expanders (thread t expands
// block t & 1 of weight row t >> 1: 16 code bytes and one scale byte into 32
// bf16 values), then the epilogue (tensor-memory lanes = the tile's weight
// rows): warps 10..13 of their own when kSepEpi, else expander warps 2..5
// after each tile's stages (fewer warps: two CTAs fit on an SM).
namespace w4a16 {

constexpr int kExpWarp0 = 2;
constexpr int kExpWarps = 8;

template <int NT, int RS, int XS, bool kSepEpi>
struct Layout {
    static constexpr int THREADS = (kExpWarp0 + kExpWarps + (kSepEpi ? 4 : 0)) * 32;
    static constexpr int EPI_WARP0 = kSepEpi ? kExpWarp0 + kExpWarps : kExpWarp0;
    static constexpr int KB = 128;                    // bytes of bf16 per row per stage (64 values)
    static constexpr int X_STAGE = NT * KB;           // token rows
    static constexpr int WX_STAGE = 128 * KB;         // expanded weight rows
    static constexpr int WC_STAGE = 128 * 32;         // weight codes (64 values per row)
    static constexpr int SF_STAGE = SF_ATOM;          // one scale atom (128 rows x 4 blocks)
    static constexpr int OFF_X = 0;
    static constexpr int OFF_WX = OFF_X + RS * X_STAGE;
    static constexpr int OFF_WC = OFF_WX + XS * WX_STAGE;
    static constexpr int OFF_SF = OFF_WC + RS * WC_STAGE;
    static constexpr int OFF_BAR = OFF_SF + RS * SF_STAGE;
    static constexpr int NUM_BARS = 2 * RS + 2 * XS + 3;
    static constexpr int OFF_MISC = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;
    static constexpr int TMEM_COLS = NT < 32 ? 32 : NT;
    static_assert(X_STAGE % 1024 == 0 && WX_STAGE % 1024 == 0, "swizzled tiles need 1 KB alignment");
    static_assert(ALLOC <= 232448, "shared memory");
};

struct Params {
    const uint8_t *sfw;   // tiled weight scales
    uint16_t *Y;
    int64_t ldy;
    int32_t M, N;
    int32_t num_kstages;  // 64-wide K stages
    int32_t nka;          // 4-scale atoms per 128-row block
    int32_t n_wb;         // 128-row weight blocks
    int32_t n_tiles;
};

// One code byte (two E2M1 values) times 2^(s - 127) as a bf16 pair (element
// 2i in the low half): E2M1 -> f16 (exact), f16 -> fp32 (exact), times the
// power of two (exact: the product has two significant bits and stays above
// 2^-149), fp32 -> bf16 (exact: two significant bits, above bf16's 2^-133).
__device__ __forceinline__ uint32_t expand_byte(uint32_t byte, float scale)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 b;\n\t"
        "cvt.u8.u32 b, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
        : "=r"(h2)
        : "r"(byte));
    const float2 v = __fmul2_rn(make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu))),
                                            __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)))),
                                make_float2(scale, scale));
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t *>(&b);
}

__device__ __forceinline__ float e8m0_value(uint32_t s)
{
    // 2^(s - 127); s = 0 is the subnormal 2^-127
    return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}

// The epilogue of one tile by one warp (tensor-memory lanes 32q .. 32q+31):
// weight row n = w0 + 32q + lane, token columns -> Y[tok0 + c][n].  Releases
// the accumulator (an arrival on acc_empty) once its columns are loaded.
template <int NT>
__device__ __forceinline__ void epilogue_tile(uint32_t tmem, int q, int lane, int32_t w0, int32_t tok0,
                                              const Params &p, uint32_t acc_empty)
{
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const int32_t n = w0 + 32 * q + lane;
    const int32_t mmax = min(NT, p.M - tok0);
    if constexpr (NT == 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr, r);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        if (n < p.N) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                if (c < mmax) {
                    const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(r[c]));
                    p.Y[static_cast<int64_t>(tok0 + c) * p.ldy + n] = *reinterpret_cast<const uint16_t *>(&b);
                }
            }
        }
    } else {
#pragma unroll 1
        for (int h = 0; h < NT / 32; ++h) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + 32 * h, r);
            tmem_ld_wait();
            if (h == NT / 32 - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            if (n < p.N) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if (32 * h + c < mmax) {
                        const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(r[c]));
                        p.Y[static_cast<int64_t>(tok0 + 32 * h + c) * p.ldy + n] =
                            *reinterpret_cast<const uint16_t *>(&b);
                    }
                }
            }
        }
    }
}

template <int NT, int RS, int XS, bool kSepEpi>
__global__ void __launch_bounds__(Layout<NT, RS, XS, kSepEpi>::THREADS, 1)
    gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWc,
                      const Params p)
{
    using L = Layout<NT, RS, XS, kSepEpi>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_base = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (RS + s); };
    auto xfull_bar = [&](int e) { return bar_base + 8u * (2 * RS + e); };
    auto xempty_bar = [&](int e) { return bar_base + 8u * (2 * RS + XS + e); };
    const uint32_t acc_full = bar_base + 8u * (2 * RS + 2 * XS);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t drain_bar = acc_full + 16u;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t wait_ns = g_wait_ns;
    const int nks = p.num_kstages;

    if (threadIdx.x == 0) {
        abort_flag[1] = 1;
        abort_flag[2] = 1;
        for (int s = 0; s < RS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int e = 0; e < XS; ++e) {
            mbar_init(xfull_bar(e), kExpWarps);  // one arrival per expander warp
            mbar_init(xempty_bar(e), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);                // one arrival per epilogue warp
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::OFF_MISC, L::TMEM_COLS);
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
            constexpr uint32_t kBytes = L::X_STAGE + L::WC_STAGE + L::SF_STAGE;
            uint32_t it = 0, issued = 0, last_parity = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
                const int32_t w0 = (t % p.n_wb) * 128, tok0 = (t / p.n_wb) * NT;
                const uint8_t *sfw = p.sfw + static_cast<size_t>(w0 / 128) * p.nka * SF_ATOM;
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    const int s = static_cast<int>(it % RS);
                    const uint32_t ph = (it / RS) & 1u;
                    MACAQ_TRACE(0, it);
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, kErrProducer, wait_ns)) {
                        ok = false;
                        break;
                    }
                    MACAQ_TRACE(1, it);
                    const uint32_t fb = full_bar(s);
                    mbar_arrive_expect_tx(fb, kBytes);
                    tma_load_2d(sbase + L::OFF_X + s * L::X_STAGE, &tmX, fb, ks * 64, tok0);
                    tma_load_2d(sbase + L::OFF_WC + s * L::WC_STAGE, &tmWc, fb, ks * 32, w0);
                    bulk_load(sbase + L::OFF_SF + s * L::SF_STAGE, sfw + static_cast<size_t>(ks / 2) * SF_ATOM,
                              L::SF_STAGE, fb);
                    issued |= 1u << s;
                    last_parity = (last_parity & ~(1u << s)) | (ph << s);
                }
            }
            for (int s = 0; s < RS; ++s) {
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
            const uint64_t w_desc0 = smem_desc(sbase + L::OFF_WX, 16, 8 * L::KB, kSwizzle128B);
            const uint64_t x_desc0 = smem_desc(sbase + L::OFF_X, 16, 8 * L::KB, kSwizzle128B);
            constexpr uint32_t idesc = idesc_bf16(128, NT);
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int32_t t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tc) {
                // the epilogue must have drained the previous tile's accumulator
                if (!wait_bounded(acc_empty, (tc & 1u) ^ 1u, abort_flag, kErrMma, wait_ns)) break;
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    const int s = static_cast<int>(it % RS);
                    const int e = static_cast<int>(it % XS);
                    // the expanded tile (its expanders saw the raw stage land)
                    MACAQ_TRACE(2, it);
                    if (!wait_bounded(xfull_bar(e), (it / XS) & 1u, abort_flag, kErrMma, wait_ns)) {
                        ok = false;
                        break;
                    }
                    MACAQ_TRACE(3, it);
                    tc_fence_after();
                    const uint64_t wd = w_desc0 + ((e * L::WX_STAGE) >> 4);
                    const uint64_t xd = x_desc0 + ((s * L::X_STAGE) >> 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tc_mma_f16(tmem, wd + 2 * j, xd + 2 * j, idesc, (ks > 0 || j > 0) ? 1u : 0u);
                    tc_commit(empty_bar(s));
                    tc_commit(xempty_bar(e));
                }
                if (ok) tc_commit(acc_full);
            }
            tc_commit(drain_bar);
            wait_fixed(drain_bar, 0);
        }
        __syncwarp();
    } else if (warp < kExpWarp0 + kExpWarps) {
        // ---------------------------------------------------- expanders
        // One leader thread waits on the stage's barriers; the expander warps
        // then start together from a named CTA barrier (cheaper than eight
        // warps each waking on the same mbarrier, one after another).
        const int t = threadIdx.x - kExpWarp0 * 32;
        const int row = t >> 1, half = t & 1;  // block `half` of weight row `row`
        const uint32_t swz = static_cast<uint32_t>(row) & 7u;
        const uint32_t sf_off = static_cast<uint32_t>((row & 31) * 16 + (row >> 5) * 4 + half);
        const bool epi = !kSepEpi && warp < kExpWarp0 + 4;
        // the leader's verdict per stage, in two slots by stage parity: a slot
        // is rewritten only two stages later, after every expander has read it
        // (all of them pass the next stage's named barrier in between)
        volatile int *go = abort_flag + 1;
        uint32_t it = 0, tc = 0;
        bool ok = true;
        for (int32_t tl = blockIdx.x; tl < p.n_tiles && ok; tl += gridDim.x, ++tc) {
            for (int ks = 0; ks < nks; ++ks, ++it) {
                const int s = static_cast<int>(it % RS);
                const int e = static_cast<int>(it % XS);
                if (t == 0) {
                    MACAQ_TRACE(4, it);
                    const bool got = wait_bounded(full_bar(s), (it / RS) & 1u, abort_flag, kErrMma, wait_ns) &&
                                     wait_bounded(xempty_bar(e), ((it / XS) & 1u) ^ 1u, abort_flag, kErrMma,
                                                  wait_ns);
                    MACAQ_TRACE(6, it);
                    go[it & 1u] = got ? 1 : 0;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kExpWarps * 32) : "memory");
                if (!go[it & 1u]) {
                    ok = false;
                    break;
                }
                const uint4 cw = *reinterpret_cast<const uint4 *>(smem + L::OFF_WC + s * L::WC_STAGE + row * 32 +
                                                                  16 * half);
                const float sc = e8m0_value(smem[L::OFF_SF + s * L::SF_STAGE + sf_off + 2 * (ks & 1)]);
                const uint32_t dst = sbase + L::OFF_WX + e * L::WX_STAGE + row * L::KB;
                const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // 16-byte chunk 4 half + c: values 8 (4 half + c) .., from code word c
                    const uint32_t w = words[c];
                    const uint32_t o0 = expand_byte(w & 0xffu, sc), o1 = expand_byte((w >> 8) & 0xffu, sc);
                    const uint32_t o2 = expand_byte((w >> 16) & 0xffu, sc), o3 = expand_byte(w >> 24, sc);
                    const uint32_t chunk = static_cast<uint32_t>(4 * half + c);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + ((chunk ^ swz) << 4)),
                                 "r"(o0), "r"(o1), "r"(o2), "r"(o3)
                                 : "memory");
                }
                // the tensor core reads these stores through the async proxy
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(xfull_bar(e));
                if (lane == 0 && warp == kExpWarp0) MACAQ_TRACE(7, it);
                if (lane == 0 && warp == kExpWarp0 + kExpWarps - 1) MACAQ_TRACE(8, it);
            }
            if (epi && ok) {
                const int32_t w0 = (tl % p.n_wb) * 128, tok0 = (tl / p.n_wb) * NT;
                if (!warp_wait_bounded(acc_full, tc & 1u, abort_flag, kErrEpilogue, wait_ns)) break;
                tc_fence_after();
                epilogue_tile<NT>(tmem, warp & 3, lane, w0, tok0, p, acc_empty);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        uint32_t tc = 0;
        for (int32_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++tc) {
            const int32_t w0 = (t % p.n_wb) * 128, tok0 = (t / p.n_wb) * NT;
            if (!warp_wait_bounded(acc_full, tc & 1u, abort_flag, kErrEpilogue, wait_ns)) break;
            tc_fence_after();
            epilogue_tile<NT>(tmem, warp & 3, lane, w0, tok0, p, acc_empty);
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

}  // namespace w4a16
