// gemm.cu -- persistent, warp-specialised q6_K / q4_K x q8 MMQ GEMM for sm_103a.
//
// Y[t,j] = sum over 32-value chunks c of d_a[t,c] * (scale terms of row j, chunk c)
// applied to the exact integer sub-block dots I[t,j,.]:
//   q6_K: Y += d_a * (dsc0 * I_h0 + dsc1 * I_h1)   (two 16-value sub-blocks per chunk,
//         the dsc pair of "r56 - q6_K A-side bundle ...", §2.2)
//   q4_K: Y += d_a * (dsc * I - ssum * dmn)        (one 32-value chunk)
//
// Structure of one CTA (one per SM, persistent over 128-token x 128-row tiles):
//   warp 0     producer: bulk async copies (cp.async.bulk, no multicast) of the
//              pre-swizzled A/B operand tiles into a STAGES-deep ring and of the
//              token/weight scale pairs into an SSTAGES-deep ring, completion
//              counted on mbarriers (full/empty pairs with phase bits).
//   warp 1     allocates TMEM; one thread issues tcgen05.mma kind::f16 (integer
//              codes held exactly as f16, f32 accumulation in TMEM), one fresh
//              accumulator per sub-block, rotating over TMEM slots, and commits
//              each slot to a "full" mbarrier.
//   warps 2-9  promotion: tcgen05.ld of a finished slot, release the slot, then
//              apply the f32 scales into register accumulators; store Y per tile.
// The multi-stage ring replaces the pages' one-deep double buffer and group-count
// waits ("r45 ...", §2.2; "r58 ...", §2.2 and §6 lesson 2: one tile of
// lookahead cannot cover the global-to-shared latency); tails need no zero-fill
// at copy time because the prepass and the repack pad the planes with zero rows
// ("r45 ...", §2.3; "r56 ...", §2.4), and Y stores are predicated.
//
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel sets
// the sticky error word, every role leaves its loop, waits (bounded) for its own
// copies and MMAs in flight, and the CTA frees TMEM and exits.
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "mmq_internal.h"
#include "ptx.cuh"

namespace mmq {
namespace {

constexpr int BM = 128;             // tokens per tile (TMEM lanes)
constexpr int BN = 128;             // weight rows per tile (MMA N)
constexpr int BK = TILE_K;          // values per stage: two 32-value chunks
constexpr int STAGES = 5;           // operand ring depth
constexpr int SSTAGES = 8;          // scale ring depth
constexpr int NUM_THREADS = 320;
constexpr int PROMO_WARP0 = 2;
constexpr int NUM_PROMO_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

constexpr int SCALE_STAGE_BYTES = 2 * BM * 8;   // two chunks x 128 entries x 8 B
constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * TILE_BYTES;
constexpr int SMEM_AS = SMEM_B + STAGES * TILE_BYTES;
constexpr int SMEM_WS = SMEM_AS + SSTAGES * SCALE_STAGE_BYTES;
constexpr int SMEM_BAR = SMEM_WS + SSTAGES * SCALE_STAGE_BYTES;
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = BAR_FULL + STAGES;
constexpr int BAR_SFULL = BAR_EMPTY + STAGES;
constexpr int BAR_SEMPTY = BAR_SFULL + SSTAGES;
constexpr int BAR_TFULL = BAR_SEMPTY + SSTAGES;
constexpr int BAR_TEMPTY = BAR_TFULL + 4;
constexpr int BAR_DRAIN = BAR_TEMPTY + 4;
constexpr int NUM_BARS = BAR_DRAIN + 1;
constexpr int SMEM_TMEMPTR = SMEM_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = SMEM_TMEMPTR + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;    // slack for 1024-byte alignment
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(SMEM_B % 1024 == 0 && SMEM_A % 1024 == 0, "operand tiles need 1024-byte alignment");

struct GemmArgs {
    const uint8_t* A;    // activation code tiles  [num_m][nkb][16 KiB]
    const uint8_t* AS;   // token scale pairs      [num_m][nchunk][128] x {f32 d, i32 ssum}
    const uint8_t* B;    // weight code tiles      [num_n][nkb][16 KiB]
    const uint8_t* WS;   // weight scale pairs     [num_n][nchunk][128] x {f32, f32}
    float* out;          // Y [M][ldy], or the dot dump [M][od][nsub]
    int ldy;
    int M, od, id;
    int num_m, num_n;
    int vec_store;       // Y is 16-byte aligned and ldy % 4 == 0
};

// Bounded wait that ignores the error word (used only to drain our own copies /
// MMAs in flight before the CTA exits; those always complete).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(&g_error_word, 1u);
            return;
        }
    }
}

template <int TYPE, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const GemmArgs g)
{
    constexpr bool Q4 = (TYPE == 12);
    constexpr int NSLOT = Q4 ? 4 : 2;          // TMEM accumulator slots
    constexpr int SLOT_COLS = Q4 ? BN : 2 * BN; // q6_K: two sub-block accumulators per chunk

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nkb = g.id / BK;
    const int nchunk = g.id / CHUNK;
    const int num_tiles = g.num_m * g.num_n;
    auto bar = [&](int i) -> uint32_t { return sbase + SMEM_BAR + 8u * static_cast<uint32_t>(i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(BAR_FULL + s), 1);
            mbar_init(bar(BAR_EMPTY + s), 1);
        }
        for (int s = 0; s < SSTAGES; ++s) {
            mbar_init(bar(BAR_SFULL + s), 1);
            mbar_init(bar(BAR_SEMPTY + s), NUM_PROMO_WARPS);
        }
        for (int k = 0; k < 4; ++k) {
            mbar_init(bar(BAR_TFULL + k), 1);
            mbar_init(bar(BAR_TEMPTY + k), NUM_PROMO_WARPS);
        }
        mbar_init(bar(BAR_DRAIN), 1);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(sbase + SMEM_TMEMPTR, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + SMEM_TMEMPTR);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t n_ops = 0, n_sc = 0;  // fills issued on each ring
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m = tile % g.num_m, n = tile / g.num_m;
                const uint8_t* Ab = g.A + static_cast<size_t>(m) * nkb * TILE_BYTES;
                const uint8_t* Bb = g.B + static_cast<size_t>(n) * nkb * TILE_BYTES;
                const uint8_t* ASb = g.AS + static_cast<size_t>(m) * nchunk * BM * 8;
                const uint8_t* WSb = g.WS + static_cast<size_t>(n) * nchunk * BN * 8;
                for (int kb = 0; kb < nkb; ++kb) {
                    const uint32_t s = n_ops % STAGES;
                    if (!mbar_wait(bar(BAR_EMPTY + s), ((n_ops / STAGES) & 1u) ^ 1u, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(BAR_FULL + s), 2 * TILE_BYTES);
                    bulk_g2s(sbase + SMEM_A + s * TILE_BYTES, Ab + static_cast<size_t>(kb) * TILE_BYTES,
                             TILE_BYTES, bar(BAR_FULL + s));
                    bulk_g2s(sbase + SMEM_B + s * TILE_BYTES, Bb + static_cast<size_t>(kb) * TILE_BYTES,
                             TILE_BYTES, bar(BAR_FULL + s));
                    ++n_ops;
                    const uint32_t ss = n_sc % SSTAGES;
                    if (!mbar_wait(bar(BAR_SEMPTY + ss), ((n_sc / SSTAGES) & 1u) ^ 1u, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(BAR_SFULL + ss), 2 * SCALE_STAGE_BYTES);
                    bulk_g2s(sbase + SMEM_AS + ss * SCALE_STAGE_BYTES,
                             ASb + static_cast<size_t>(kb) * SCALE_STAGE_BYTES, SCALE_STAGE_BYTES,
                             bar(BAR_SFULL + ss));
                    bulk_g2s(sbase + SMEM_WS + ss * SCALE_STAGE_BYTES,
                             WSb + static_cast<size_t>(kb) * SCALE_STAGE_BYTES, SCALE_STAGE_BYTES,
                             bar(BAR_SFULL + ss));
                    ++n_sc;
                }
            }
            // Our copies must have landed before the CTA may exit.
            for (uint32_t i = (n_ops > STAGES ? n_ops - STAGES : 0); i < n_ops; ++i)
                drain_wait(bar(BAR_FULL + i % STAGES), (i / STAGES) & 1u);
            for (uint32_t i = (n_sc > SSTAGES ? n_sc - SSTAGES : 0); i < n_sc; ++i)
                drain_wait(bar(BAR_SFULL + i % SSTAGES), (i / SSTAGES) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            uint32_t it = 0, ch = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                for (int kb = 0; kb < nkb; ++kb) {
                    const uint32_t s = it % STAGES;
                    if (!mbar_wait(bar(BAR_FULL + s), (it / STAGES) & 1u, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a0 = sdesc_k_sw128(sbase + SMEM_A + s * TILE_BYTES);
                    const uint64_t b0 = sdesc_k_sw128(sbase + SMEM_B + s * TILE_BYTES);
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const uint32_t slot = ch % NSLOT;
                        if (!mbar_wait(bar(BAR_TEMPTY + slot), ((ch / NSLOT) & 1u) ^ 1u, WAIT_LIMIT_NS)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + slot * SLOT_COLS;
                        // K advance inside the 128-byte swizzled row: +32 bytes per 16 values
                        // (descriptor address field counts 16-byte units).
                        const uint64_t ak = a0 + static_cast<uint64_t>(4 * cc);
                        const uint64_t bk = b0 + static_cast<uint64_t>(4 * cc);
                        if (Q4) {
                            umma_f16(d, ak, bk, idesc, 0u);
                            umma_f16(d, ak + 2, bk + 2, idesc, 1u);
                        } else {
                            umma_f16(d, ak, bk, idesc, 0u);
                            umma_f16(d + BN, ak + 2, bk + 2, idesc, 0u);
                        }
                        umma_commit(bar(BAR_TFULL + slot));
                        ++ch;
                    }
                    if (!ok)
                        break;
                    umma_commit(bar(BAR_EMPTY + s));  // operand stage free once these MMAs finish
                    ++it;
                }
            }
            umma_commit(bar(BAR_DRAIN));  // every MMA issued so far has completed
            drain_wait(bar(BAR_DRAIN), 0u);
        }
        __syncwarp();
    } else if (warp >= PROMO_WARP0) {
        // ------------------------------------------------------------ promotion
        const int pw = warp - PROMO_WARP0;            // 0..7
        const int q = warp & 3;                        // TMEM lane quarter this warp may read
        const int hcol = pw >> 2;                      // which 64 of the 128 columns
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        uint32_t it = 0, ch = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            const int m = tile % g.num_m, n = tile / g.num_m;
            const int row = m * BM + row_in_tile;
            const int jb = n * BN + hcol * 64;
            float acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i)
                acc[i] = 0.0f;
            for (int kb = 0; kb < nkb; ++kb) {
                const uint32_t ss = it % SSTAGES;
                if (!mbar_wait(bar(BAR_SFULL + ss), (it / SSTAGES) & 1u, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                const uint2* tsc = reinterpret_cast<const uint2*>(smem + SMEM_AS + ss * SCALE_STAGE_BYTES);
                const float4* wsc = reinterpret_cast<const float4*>(smem + SMEM_WS + ss * SCALE_STAGE_BYTES);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const uint32_t slot = ch % NSLOT;
                    if (!mbar_wait(bar(BAR_TFULL + slot), (ch / NSLOT) & 1u, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint2 ts = tsc[cc * BM + row_in_tile];
                    const float da = __uint_as_float(ts.x);
                    const float4* w4 = wsc + (cc * BN + hcol * 64) / 2;  // two columns per float4
                    const int sub = 2 * kb + cc;                          // chunk index along id
                    if (Q4) {
                        const float sf = static_cast<float>(static_cast<int>(ts.y));  // ssum
#pragma unroll
                        for (int gq = 0; gq < 4; ++gq) {  // four groups of 16 columns
                            float I[16];
                            tmem_ld16_wait(lane_addr + slot * SLOT_COLS + hcol * 64 + gq * 16, I);
                            if (gq == 3) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0)
                                    mbar_arrive(bar(BAR_TEMPTY + slot));
                            }
                            if (MODE == GEMM_DOTS) {
                                if (row < g.M) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        const int j = jb + gq * 16 + i;
                                        if (j < g.od)
                                            g.out[(static_cast<size_t>(row) * g.od + j) * nchunk + sub] = I[i];
                                    }
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; i += 2) {
                                    const float4 w = w4[gq * 8 + i / 2];
                                    float* a = acc + gq * 16 + i;
                                    // d_a * (dsc * I - ssum * dmn)
                                    a[0] = fmaf(da, fmaf(I[i], w.x, -sf * w.y), a[0]);
                                    a[1] = fmaf(da, fmaf(I[i + 1], w.z, -sf * w.w), a[1]);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int p = 0; p < 4; ++p) {  // four groups of 16 columns, both sub-blocks
                            float I0[16], I1[16];
                            const uint32_t c0 = lane_addr + slot * SLOT_COLS + hcol * 64 + p * 16;
                            tmem_ld16x2_wait(c0, c0 + BN, I0, I1);
                            if (p == 3) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0)
                                    mbar_arrive(bar(BAR_TEMPTY + slot));
                            }
                            if (MODE == GEMM_DOTS) {
                                if (row < g.M) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        const int j = jb + p * 16 + i;
                                        if (j < g.od) {
                                            float* dst = g.out + (static_cast<size_t>(row) * g.od + j) * (2 * nchunk);
                                            dst[2 * sub] = I0[i];
                                            dst[2 * sub + 1] = I1[i];
                                        }
                                    }
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; i += 2) {
                                    const float4 w = w4[p * 8 + i / 2];
                                    float* a = acc + p * 16 + i;
                                    a[0] = fmaf(da, fmaf(I1[i], w.y, I0[i] * w.x), a[0]);
                                    a[1] = fmaf(da, fmaf(I1[i + 1], w.w, I0[i + 1] * w.z), a[1]);
                                }
                            }
                        }
                    }
                    ++ch;
                }
                if (!ok)
                    break;
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(BAR_SEMPTY + ss));
                ++it;
            }
            if (!ok)
                break;
            if (MODE == GEMM_Y && row < g.M) {
                float* yrow = g.out + static_cast<size_t>(row) * g.ldy;
#pragma unroll
                for (int i = 0; i < 64; i += 4) {
                    const int j = jb + i;
                    if (g.vec_store && j + 3 < g.od) {
                        *reinterpret_cast<float4*>(yrow + j) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (j + k < g.od)
                                yrow[j + k] = acc[i + k];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int TYPE, int MODE>
cudaError_t launch_typed(const GemmArgs& a, int grid, cudaStream_t s)
{
    static std::atomic<uint64_t> attr_set_mask{0};  // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set_mask.load() & bit)) {
        e = cudaFuncSetAttribute(gemm_kernel<TYPE, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess)
            return e;
        attr_set_mask.fetch_or(bit);
    }
    gemm_kernel<TYPE, MODE><<<grid, NUM_THREADS, SMEM_ALLOC, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(int type, GemmMode mode, const void* packed, int od, int id, const void* qa,
                        const void* scales, int M, float* out, int ldy, cudaStream_t s, const char** path_label)
{
    const WeightPlanes wp = weight_planes(od, id);
    GemmArgs a;
    a.A = static_cast<const uint8_t*>(qa);
    a.AS = static_cast<const uint8_t*>(scales);
    a.B = static_cast<const uint8_t*>(packed) + wp.code_off;
    a.WS = static_cast<const uint8_t*>(packed) + wp.scale_off;
    a.out = out;
    a.ldy = ldy;
    a.M = M;
    a.od = od;
    a.id = id;
    a.num_m = ceil_div(M, BM);
    a.num_n = ceil_div(od, BN);
    a.vec_store = ((reinterpret_cast<uintptr_t>(out) & 15u) == 0 && (ldy & 3) == 0) ? 1 : 0;

    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    const int tiles = a.num_m * a.num_n;
    const int grid = tiles < nsm ? tiles : nsm;

    if (type == 14) {
        if (path_label)
            *path_label = "q6_K: persistent tcgen05.mma kind::f16 128x128x16 (exact int codes), "
                          "cp.async.bulk 5-stage ring, TMEM 2x2 sub-block slots, f32 dsc-pair promotion";
        return mode == GEMM_Y ? launch_typed<14, GEMM_Y>(a, grid, s) : launch_typed<14, GEMM_DOTS>(a, grid, s);
    }
    if (path_label)
        *path_label = "q4_K: persistent tcgen05.mma kind::f16 128x128x16 (exact int codes), "
                      "cp.async.bulk 5-stage ring, TMEM 4 chunk slots, f32 dsc/dmn promotion";
    return mode == GEMM_Y ? launch_typed<12, GEMM_Y>(a, grid, s) : launch_typed<12, GEMM_DOTS>(a, grid, s);
}

cudaError_t gemm_read_and_clear_error(cudaStream_t s, unsigned int* word)
{
    *word = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return e;
    e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned int));
    if (e != cudaSuccess)
        return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned int));
}

}  // namespace mmq
