// gemm.cu -- persistent, warp-specialised q6_K / q4_K x q8 MMQ GEMM for sm_103a.
//
// What it computes (per token t, weight row j, 32-value chunk c of super-block sb):
//   q4_K: Y = sum_sb d_sb * sum_{c in sb} d_a[t,c] * I'[t,j,c]  -  sum_c ma[t,c] * dmn[j,c]
//         I' = sum over the chunk of (sc_c * q) * q_a   (integer; sc folded into the codes)
//         ma = d_a * ssum, dmn = dmin * m_c
//   q6_K: Y = sum_sb d_sb * sum_{c in sb} d_a[t,c] * I'[t,j,c]
//         I' = sum of (sc * q) * q_a over the chunk when the codes are folded, else
//         sc0 * I_0 + sc1 * I_1 from one accumulator per 16-value sub-block.
// This is the q6_K/q4_K formula with the integer sub-block scale moved into the
// integer dot and the f16 super-block scale factored out of the chunk sum; every
// dot is an exact integer below 2^24.  The q4_K min term is a contraction over
// chunks (K = id/32); it runs on the tensor cores in tf32 with both operands split
// hi + lo (hi*hi + hi*lo + lo*hi, relative error ~2^-21 per product).
//
// One CTA per SM, persistent over 128-token x 128-row tiles; 18 warps:
//   warp 0      producer: cp.async.bulk copies (no multicast) of the pre-swizzled
//               f16 operand tiles into a STAGES-deep ring, token scale pairs into an
//               SSTAGES ring, and per-super-block data (d, min-term operands, q6_K
//               sub-block scales) into an SBR ring; completion on mbarriers.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma kind::f16 (f16-held
//               integer codes, f32 accumulate) into rotating per-chunk TMEM slots,
//               and (q4_K) kind::tf32 into a per-tile min-term accumulator.
//   warps 2-17  promotion: tcgen05.ld of a finished chunk slot, release it,
//               inner += d_a * I'; per super-block acc += d * inner; at tile end
//               (q4_K) acc -= min term; store Y.  Each warp owns one TMEM lane
//               quarter (warp % 4) and 32 of the 128 columns.
// The multi-stage rings replace the pages' one-deep double buffer and group-count
// waits ("r45 ...", §2.2; "r58 ...", §2.2 and §6 lesson 2: one tile of lookahead
// cannot cover the global-to-shared latency); registration-time planes remove the
// staging ALU the pages attribute stalls to ("r56 ...", §1-§2.2); tails need no
// zero-fill at copy time because the prepass and the repack pad the planes with
// zero rows ("r45 ...", §2.3; "r56 ...", §2.4), and Y stores are predicated.
//
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel sets
// the sticky error word, every role leaves its loop, waits (bounded) for its own
// copies and MMAs in flight, and the CTA frees TMEM and exits.
#include <cuda_fp16.h>

#include <atomic>

#include "mmq_internal.h"
#include "ptx.cuh"

namespace mmq {
namespace {

constexpr int BM = 128;             // tokens per tile (TMEM lanes)
constexpr int BN = 128;             // weight rows per tile (MMA N)
constexpr int BK = TILE_K;          // values per stage: two 32-value chunks
constexpr int STAGES = 5;           // operand ring depth
constexpr int SSTAGES = 8;          // token-scale ring depth (entries of one stage)
constexpr int SBR = 2;              // super-block ring depth
constexpr int NUM_WARPS = 18;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int PROMO_WARP0 = 2;
constexpr int NUM_PROMO_WARPS = 16;
constexpr int COLS_PER_WARP = BN / 4;   // 32
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t MIN_COL = 384;   // q4_K min-term accumulator columns [384, 512)
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

constexpr int SCALE_STAGE_BYTES = 2 * BM * 8;      // {d, ssum} for two chunks x 128 tokens
constexpr int SB_SBD_BYTES = BN * 4;               // d per row
constexpr int SB_AM_BYTES = 2 * TF32_TILE_BYTES;   // q4_K: token min-term operand hi, lo
constexpr int SB_BM_BYTES = 2 * TF32_TILE_BYTES;   // q4_K: weight min-term operand hi, lo
constexpr int SB_SC_BYTES = 16 * BN * 4;           // q6_K: sub-block scales
constexpr int SB_BYTES = SB_AM_BYTES + SB_BM_BYTES + SB_SBD_BYTES;
static_assert(SB_BYTES >= SB_SBD_BYTES + SB_SC_BYTES, "super-block entry");

constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * TILE_BYTES;
constexpr int SMEM_AS = SMEM_B + STAGES * TILE_BYTES;
constexpr int SMEM_SB = SMEM_AS + SSTAGES * SCALE_STAGE_BYTES;
constexpr int SMEM_BAR = SMEM_SB + SBR * SB_BYTES;
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = BAR_FULL + STAGES;
constexpr int BAR_SFULL = BAR_EMPTY + STAGES;
constexpr int BAR_SEMPTY = BAR_SFULL + SSTAGES;
constexpr int BAR_SBFULL = BAR_SEMPTY + SSTAGES;
constexpr int BAR_SBEMPTY = BAR_SBFULL + SBR;
constexpr int BAR_TFULL = BAR_SBEMPTY + SBR;
constexpr int BAR_TEMPTY = BAR_TFULL + 4;
constexpr int BAR_MINFULL = BAR_TEMPTY + 4;
constexpr int BAR_MINEMPTY = BAR_MINFULL + 1;
constexpr int BAR_DRAIN = BAR_MINEMPTY + 1;
constexpr int NUM_BARS = BAR_DRAIN + 1;
constexpr int SMEM_TMEMPTR = SMEM_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = SMEM_TMEMPTR + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;    // slack for 1024-byte alignment
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(SMEM_B % 1024 == 0 && SMEM_AS % 16 == 0 && SMEM_SB % 16 == 0 && SB_BYTES % 16 == 0, "alignment");

struct GemmArgs {
    const uint8_t* A;     // activation code tiles      [num_m][nkb][16 KiB]
    const uint8_t* AS;    // token scale pairs          [num_m][nchunk][128] x {f32 d, i32 ssum}
    const uint8_t* AM;    // token min-term tiles       [num_m][nsb][hi 4 KiB, lo 4 KiB]
    const uint8_t* B;     // weight code tiles          [num_n][nkb][16 KiB]
    const uint8_t* SBD;   // weight d per super-block   [num_n][nsb][128] f32
    const uint8_t* AUX;   // q4_K min-term tiles [num_n][nsb][8 KiB]; q6_K scales [num_n][nsb][16][128]
    const unsigned int* FLAG;
    float* out;           // Y [M][ldy], or the dot dump [M][od][nsub]
    int ldy;
    int M, od, id;
    int num_m, num_n;
    int vec_store;        // Y is 16-byte aligned and ldy % 4 == 0
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

// Shared-memory descriptor of a 128 x 8 tf32 tile in the no-swizzle K-major
// core-matrix layout of tf32_tile_byte(): K-direction core-matrix stride 128 B
// (leading byte offset), 8-row group stride 256 B (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_tf32_tile(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128u >> 4) << 16;
    d |= static_cast<uint64_t>(256u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;  // layout type 0: no swizzle
}

__host__ __device__ constexpr uint32_t idesc_tf32_f32(int m, int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// TYPE 12 = q4_K, 14 = q6_K; MODE GEMM_Y or GEMM_DOTS (raw per-chunk dots).
template <int TYPE, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const GemmArgs g)
{
    constexpr bool Q4 = (TYPE == 12);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nkb = g.id / BK;
    const int nchunk = g.id / CHUNK;
    const int nsb = g.id / QK_K;
    const int num_tiles = g.num_m * g.num_n;
    // q6_K codes hold sc*q (one accumulator per chunk) unless some |sc| > 64.
    const bool folded = Q4 || (__ldg(g.FLAG) != 0u);
    const uint32_t nslot = Q4 ? 3u : (folded ? 4u : 2u);       // TMEM chunk slots
    const uint32_t slot_cols = (Q4 || folded) ? BN : 2 * BN;
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
        for (int s = 0; s < SBR; ++s) {
            mbar_init(bar(BAR_SBFULL + s), 1);
            mbar_init(bar(BAR_SBEMPTY + s), NUM_PROMO_WARPS + (Q4 ? 1 : 0));
        }
        for (int k = 0; k < 4; ++k) {
            mbar_init(bar(BAR_TFULL + k), 1);
            mbar_init(bar(BAR_TEMPTY + k), NUM_PROMO_WARPS);
        }
        mbar_init(bar(BAR_MINFULL), 1);
        mbar_init(bar(BAR_MINEMPTY), NUM_PROMO_WARPS);
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
            uint32_t n_ops = 0, n_sc = 0, n_sb = 0;  // fills issued on each ring
            const uint32_t sb_tx = Q4 ? (SB_AM_BYTES + SB_BM_BYTES + SB_SBD_BYTES)
                                      : (SB_SBD_BYTES + (folded ? 0 : SB_SC_BYTES));
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m = tile % g.num_m, n = tile / g.num_m;
                const uint8_t* Ab = g.A + static_cast<size_t>(m) * nkb * TILE_BYTES;
                const uint8_t* Bb = g.B + static_cast<size_t>(n) * nkb * TILE_BYTES;
                const uint8_t* ASb = g.AS + static_cast<size_t>(m) * nchunk * BM * 8;
                for (int kb = 0; kb < nkb; ++kb) {
                    if ((kb & 3) == 0) {  // a new super-block
                        const int sb = kb >> 2;
                        const uint32_t e = n_sb % SBR;
                        if (!mbar_wait(bar(BAR_SBEMPTY + e), ((n_sb / SBR) & 1u) ^ 1u, WAIT_LIMIT_NS)) {
                            ok = false;
                            break;
                        }
                        // The promotion warps read this entry with ordinary loads before
                        // releasing it; order those reads before the bulk copy's writes.
                        fence_proxy_async_smem();
                        const uint32_t dst = sbase + SMEM_SB + e * SB_BYTES;
                        mbar_arrive_expect_tx(bar(BAR_SBFULL + e), sb_tx);
                        bulk_g2s(dst, g.SBD + (static_cast<size_t>(n) * nsb + sb) * SB_SBD_BYTES, SB_SBD_BYTES,
                                 bar(BAR_SBFULL + e));
                        if (Q4) {
                            bulk_g2s(dst + SB_SBD_BYTES, g.AM + (static_cast<size_t>(m) * nsb + sb) * SB_AM_BYTES,
                                     SB_AM_BYTES, bar(BAR_SBFULL + e));
                            bulk_g2s(dst + SB_SBD_BYTES + SB_AM_BYTES,
                                     g.AUX + (static_cast<size_t>(n) * nsb + sb) * SB_BM_BYTES, SB_BM_BYTES,
                                     bar(BAR_SBFULL + e));
                        } else if (!folded) {
                            bulk_g2s(dst + SB_SBD_BYTES, g.AUX + (static_cast<size_t>(n) * nsb + sb) * SB_SC_BYTES,
                                     SB_SC_BYTES, bar(BAR_SBFULL + e));
                        }
                        ++n_sb;
                    }
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
                    fence_proxy_async_smem();  // same ordering for the token-scale ring
                    mbar_arrive_expect_tx(bar(BAR_SFULL + ss), SCALE_STAGE_BYTES);
                    bulk_g2s(sbase + SMEM_AS + ss * SCALE_STAGE_BYTES,
                             ASb + static_cast<size_t>(kb) * SCALE_STAGE_BYTES, SCALE_STAGE_BYTES,
                             bar(BAR_SFULL + ss));
                    ++n_sc;
                }
            }
            // Our copies must have landed before the CTA may exit.
            for (uint32_t i = (n_ops > STAGES ? n_ops - STAGES : 0); i < n_ops; ++i)
                drain_wait(bar(BAR_FULL + i % STAGES), (i / STAGES) & 1u);
            for (uint32_t i = (n_sc > SSTAGES ? n_sc - SSTAGES : 0); i < n_sc; ++i)
                drain_wait(bar(BAR_SFULL + i % SSTAGES), (i / SSTAGES) & 1u);
            for (uint32_t i = (n_sb > SBR ? n_sb - SBR : 0); i < n_sb; ++i)
                drain_wait(bar(BAR_SBFULL + i % SBR), (i / SBR) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            constexpr uint32_t idesc_t = idesc_tf32_f32(BM, BN);
            uint32_t it = 0, ch = 0, n_sb = 0, tiles = 0;
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
                        const uint32_t slot = ch % nslot;
                        if (!mbar_wait(bar(BAR_TEMPTY + slot), ((ch / nslot) & 1u) ^ 1u, WAIT_LIMIT_NS)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + slot * slot_cols;
                        // K advance inside the 128-byte swizzled rows: 32 bytes per 16 values
                        // (the descriptor's address field counts 16-byte units).
                        const uint64_t ak = a0 + static_cast<uint64_t>(4 * cc);
                        const uint64_t bk = b0 + static_cast<uint64_t>(4 * cc);
                        umma_f16(d, ak, bk, idesc, 0u);
                        if (folded)
                            umma_f16(d, ak + 2, bk + 2, idesc, 1u);
                        else
                            umma_f16(d + BN, ak + 2, bk + 2, idesc, 0u);
                        umma_commit(bar(BAR_TFULL + slot));
                        ++ch;
                    }
                    if (!ok)
                        break;
                    umma_commit(bar(BAR_EMPTY + s));  // operand stage free once these MMAs finish
                    ++it;
                    if (Q4 && (kb & 3) == 3) {
                        // min-term contraction of this super-block: 8 chunks, hi/lo split
                        const uint32_t e = n_sb % SBR;
                        if (!mbar_wait(bar(BAR_SBFULL + e), (n_sb / SBR) & 1u, WAIT_LIMIT_NS)) {
                            ok = false;
                            break;
                        }
                        if (kb == 3 && !mbar_wait(bar(BAR_MINEMPTY), (tiles & 1u) ^ 1u, WAIT_LIMIT_NS)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t am = sbase + SMEM_SB + e * SB_BYTES + SB_SBD_BYTES;
                        const uint32_t bm = am + SB_AM_BYTES;
                        const uint64_t ahi = sdesc_tf32_tile(am), alo = sdesc_tf32_tile(am + TF32_TILE_BYTES);
                        const uint64_t bhi = sdesc_tf32_tile(bm), blo = sdesc_tf32_tile(bm + TF32_TILE_BYTES);
                        const uint32_t dmin_acc = tmem_base + MIN_COL;
                        umma_tf32(dmin_acc, ahi, bhi, idesc_t, kb == 3 ? 0u : 1u);
                        umma_tf32(dmin_acc, ahi, blo, idesc_t, 1u);
                        umma_tf32(dmin_acc, alo, bhi, idesc_t, 1u);
                        umma_commit(bar(BAR_SBEMPTY + e));
                        ++n_sb;
                    }
                }
                if (ok && Q4)
                    umma_commit(bar(BAR_MINFULL));
                ++tiles;
            }
            umma_commit(bar(BAR_DRAIN));  // every MMA issued so far has completed
            drain_wait(bar(BAR_DRAIN), 0u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ promotion
        const int pw = warp - PROMO_WARP0;              // 0..15
        const int q = warp & 3;                          // TMEM lane quarter this warp may read
        const int cg = pw >> 2;                          // which 32 of the 128 columns
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        uint32_t it = 0, ch = 0, n_sb = 0, tiles = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            const int m = tile % g.num_m, n = tile / g.num_m;
            const int row = m * BM + row_in_tile;
            const int jb = n * BN + cg * COLS_PER_WARP;
            float acc[COLS_PER_WARP], inner[COLS_PER_WARP];
#pragma unroll
            for (int i = 0; i < COLS_PER_WARP; ++i) {
                acc[i] = 0.0f;
                inner[i] = 0.0f;
            }
            for (int kb = 0; kb < nkb; ++kb) {
                const uint32_t e = n_sb % SBR;
                const uint8_t* sbe = smem + SMEM_SB + e * SB_BYTES;
                if ((kb & 3) == 0) {
                    if (!mbar_wait(bar(BAR_SBFULL + e), (n_sb / SBR) & 1u, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int i = 0; i < COLS_PER_WARP; ++i)
                        inner[i] = 0.0f;
                }
                const uint32_t ss = it % SSTAGES;
                if (!mbar_wait(bar(BAR_SFULL + ss), (it / SSTAGES) & 1u, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                const uint2* tsc = reinterpret_cast<const uint2*>(smem + SMEM_AS + ss * SCALE_STAGE_BYTES);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const uint32_t slot = ch % nslot;
                    if (!mbar_wait(bar(BAR_TFULL + slot), (ch / nslot) & 1u, WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float da = __uint_as_float(tsc[cc * BM + row_in_tile].x);
                    const int c = 2 * kb + cc;                  // chunk index along id
                    const uint32_t col0 = lane_addr + slot * slot_cols + cg * COLS_PER_WARP;
                    if (folded) {
                        float I0[16], I1[16];
                        tmem_ld16x2_wait(col0, col0 + 16, I0, I1);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(bar(BAR_TEMPTY + slot));
                        if (MODE == GEMM_DOTS) {
                            if (row < g.M) {
#pragma unroll
                                for (int i = 0; i < COLS_PER_WARP; ++i) {
                                    const int j = jb + i;
                                    if (j < g.od)
                                        g.out[(static_cast<size_t>(row) * g.od + j) * nchunk + c] =
                                            i < 16 ? I0[i] : I1[i - 16];
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                inner[i] = fmaf(da, I0[i], inner[i]);
                                inner[16 + i] = fmaf(da, I1[i], inner[16 + i]);
                            }
                        }
                    } else {
                        // q6_K with plain codes: one accumulator per 16-value sub-block,
                        // I' = sc0 * I_0 + sc1 * I_1 (exact: |I'| < 2^24).
                        const float* scp = reinterpret_cast<const float*>(sbe + SB_SBD_BYTES);
                        const int s0 = 2 * (c & 7);
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            float h0[8], h1[8];
                            tmem_ld8x2_wait(col0 + p * 8, col0 + BN + p * 8, h0, h1);
                            if (p == 3) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0)
                                    mbar_arrive(bar(BAR_TEMPTY + slot));
                            }
                            if (MODE == GEMM_DOTS) {
                                if (row < g.M) {
#pragma unroll
                                    for (int i = 0; i < 8; ++i) {
                                        const int j = jb + p * 8 + i;
                                        if (j < g.od) {
                                            float* dst = g.out + (static_cast<size_t>(row) * g.od + j) * (2 * nchunk);
                                            dst[2 * c] = h0[i];
                                            dst[2 * c + 1] = h1[i];
                                        }
                                    }
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const int col = cg * COLS_PER_WARP + p * 8 + i;
                                    const float u = fmaf(h1[i], scp[(s0 + 1) * BN + col], h0[i] * scp[s0 * BN + col]);
                                    inner[p * 8 + i] = fmaf(da, u, inner[p * 8 + i]);
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
                if ((kb & 3) == 3) {
                    // acc += d * inner  (d per weight row of this super-block)
                    const float4* d4 = reinterpret_cast<const float4*>(sbe) + cg * (COLS_PER_WARP / 4);
#pragma unroll
                    for (int i = 0; i < COLS_PER_WARP; i += 4) {
                        const float4 dv = d4[i / 4];
                        acc[i] = fmaf(dv.x, inner[i], acc[i]);
                        acc[i + 1] = fmaf(dv.y, inner[i + 1], acc[i + 1]);
                        acc[i + 2] = fmaf(dv.z, inner[i + 2], acc[i + 2]);
                        acc[i + 3] = fmaf(dv.w, inner[i + 3], acc[i + 3]);
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar(BAR_SBEMPTY + e));
                    ++n_sb;
                }
            }
            if (!ok)
                break;
            if (Q4) {
                if (!mbar_wait(bar(BAR_MINFULL), tiles & 1u, WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float m0[16], m1[16];
                const uint32_t mc = lane_addr + MIN_COL + cg * COLS_PER_WARP;
                tmem_ld16x2_wait(mc, mc + 16, m0, m1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(BAR_MINEMPTY));
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    acc[i] -= m0[i];
                    acc[16 + i] -= m1[i];
                }
            }
            ++tiles;
            if (MODE == GEMM_Y && row < g.M) {
                float* yrow = g.out + static_cast<size_t>(row) * g.ldy;
#pragma unroll
                for (int i = 0; i < COLS_PER_WARP; i += 4) {
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
    const ActPlanes ap = act_planes(M, id);
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    const uint8_t* sc = static_cast<const uint8_t*>(scales);
    GemmArgs a;
    a.A = static_cast<const uint8_t*>(qa);
    a.AS = sc + ap.pair_off;
    a.AM = sc + ap.am_off;
    a.B = pk + wp.code_off;
    a.SBD = pk + wp.sbd_off;
    a.AUX = pk + wp.aux_off;
    a.FLAG = reinterpret_cast<const unsigned int*>(pk + wp.flag_off);
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
            *path_label = "q6_K: persistent tcgen05.mma kind::f16 128x128x16 on scale-folded exact int codes "
                          "(plain codes + per-sub-block slots when |sc| > 64), cp.async.bulk rings, "
                          "f32 d_a per chunk / d per super-block";
        return mode == GEMM_Y ? launch_typed<14, GEMM_Y>(a, grid, s) : launch_typed<14, GEMM_DOTS>(a, grid, s);
    }
    if (path_label)
        *path_label = "q4_K: persistent tcgen05.mma kind::f16 128x128x16 on scale-folded exact int codes, "
                      "tf32 hi/lo min-term side contraction in TMEM, cp.async.bulk rings, "
                      "f32 d_a per chunk / d per super-block";
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
