// gemm.cu -- persistent, warp-specialised q6_K / q4_K x q8 MMQ GEMM for sm_103a.
//
// What it computes (per token t, weight row j, 32-value chunk c of super-block sb):
//   q4_K: Y = sum_sb d_sb * sum_{c in sb} d_a[t,c] * I'[t,j,c]  -  sum_c ma[t,c] * dmn[j,c]
//         I' = sum over the chunk of (sc_c * q) * q_a   (integer; sc folded into the codes)
//         ma = d_a * ssum, dmn = dmin * m_c
//   q6_K: Y = sum_sb d_sb * sum_{c in sb} d_a[t,c] * I'[t,j,c]
//         I' = sum of (sc * q) * q_a over the chunk: one MMA per 16 values on the
//         folded codes sc * q, or, when some |sc| > 64, two on the exact tiles sc * l
//         and 16 sc (h - 2) whose sum is sc * q (l, h the low 4 and high 2 bits of
//         q + 32) into the same accumulator.
// This is the q6_K/q4_K formula with the integer sub-block scale moved into the
// integer dot and the f16 super-block scale factored out of the chunk sum; every
// dot is an exact integer below 2^24.  The q4_K min term is a contraction over
// chunks (K = id/32); it runs on the tensor cores in tf32 with both operands split
// hi + lo (hi*hi + hi*lo + lo*hi, relative error ~2^-21 per product).
//
// One CTA per SM, persistent over 128-token x 128-row tiles; 12 warps in three
// warpgroups.  The control warpgroup gives up registers (setmaxnreg) so that each
// promotion thread can keep its 64 tile accumulators, 64 super-block partial sums
// and one 64-column chunk load in registers:
//   warp 0      producer: cp.async.bulk copies (no multicast) of the pre-swizzled
//               f16 operand tiles into a STAGES-deep ring, and once per super-block
//               the token scales of its 8 chunks and the weight d into an SBR ring
//               (two weight tiles per stage for two-tile q6_K); for q4_K, after a tile's last
//               k-block, the min-term operands of every super-block through the
//               operand ring; completion on mbarriers.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma kind::f16 (f16-held
//               integer codes, f32 accumulate) into two 256-column TMEM items that are
//               synchronised as units: an item is one 64-value k-block (its two
//               chunks' accumulators side by side), so the issuing thread waits,
//               fences and commits once per two chunks.  q4_K: the min term
//               sum_c (d_a*ssum)(dmin*m) carries
//               no per-super-block factor, so it is a kind::tf32 contraction after the
//               tile's last k-block (three MMAs per super-block, hi/lo split) into one
//               item per MIN_GROUP_SB super-blocks.
//   warps 2-3   idle (they only lend their registers).
//   warps 4-11  promotion: each owns one TMEM lane quarter (warp % 4) and 64 of the
//               128 columns; per item: wait, tcgen05.ld of its chunks, one release,
//               inner += d_a * I' (packed f32x2 FMAs); per super-block acc += d * inner;
//               per tile acc -= the q4_K min-term items; store Y (or, for the two
//               K-halves of a last-round tile, add into a zeroed Y).
// Per-chunk scaling forces one TMEM round trip per 32-value chunk; what it costs is
// set by the synchronisation, not the tensor pipe.  Measured on GB300, the issuing
// thread's wait + fence + commit cost about 80 cycles on top of a chunk's 128 cycles
// of MMA even when the wait is already satisfied, so the items are made as large as
// TMEM allows while still double-buffered (two items of 256 columns); that took the
// q4_K 11008x4096 GEMM from about 700 to about 600 SM cycles per chunk.
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
#include "route.h"
#include "ptx.cuh"

namespace mmq {
namespace {

constexpr int BM = 128;             // tokens per tile (TMEM lanes)
constexpr int BN = 128;             // weight rows per tile (MMA N)
constexpr int BK = TILE_K;          // values per stage: two 32-value chunks
constexpr int STAGES = 4;           // operand ring depth
constexpr int SBR = 3;              // super-block ring depth
constexpr int NUM_WARPS = 12;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int PROMO_WARP0 = 4;
constexpr int NUM_PROMO_WARPS = 8;
constexpr int COLS_PER_WARP = BN / 2;   // 64
constexpr uint32_t TMEM_COLS = 512;
// Register split: the launch gives every thread LAUNCH_REGS; the control warpgroup
// drops to CTRL_REGS and the two promotion warpgroups grow to PROMO_REGS out of the
// same pool (the host checks the compiled count before launching).
constexpr int LAUNCH_REGS = 168;
constexpr int CTRL_REGS = 56;
constexpr int PROMO_REGS = 224;
static_assert(CTRL_REGS * 128 + PROMO_REGS * 256 <= LAUNCH_REGS * NUM_THREADS, "register split");

// One super-block ring entry: weight d per row, the token scale pairs of the
// super-block's 8 chunks.
constexpr int SB_SBD_OFF = 0;
constexpr int SB_SBD_BYTES = BN * 4;
constexpr int SB_AS_OFF = SB_SBD_OFF + SB_SBD_BYTES;
constexpr int SB_AS_BYTES = 8 * BM * 8;            // {d, ssum} x 8 chunks x 128 tokens
constexpr int SB_BYTES = SB_AS_OFF + SB_AS_BYTES;
// q4_K min-term operands per super-block (token hi, lo tiles; weight hi, lo tiles),
// streamed through the operand ring after a tile's last k-block.
// q4_K min term: super-blocks per TMEM item (one f32 subtraction by the promotion each);
// shapes with id <= 64 * 256 take one item per tile.
constexpr int MIN_GROUP_SB = 64;
constexpr int MIN_AM_BYTES = 2 * TF32_TILE_BYTES;
constexpr int MIN_BM_BYTES = 2 * TF32_TILE_BYTES;
static_assert(MIN_AM_BYTES <= TILE_BYTES && MIN_BM_BYTES <= TILE_BYTES, "min-term operands fit a stage");

constexpr int B_STAGE = 2 * TILE_BYTES;          // one weight tile, or the two exact q6_K tiles
constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * TILE_BYTES;
constexpr int SMEM_SB = SMEM_B + STAGES * B_STAGE;
constexpr int SMEM_BAR = SMEM_SB + SBR * SB_BYTES;
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = BAR_FULL + STAGES;
constexpr int BAR_SBFULL = BAR_EMPTY + STAGES;
constexpr int BAR_SBEMPTY = BAR_SBFULL + SBR;
constexpr int BAR_TFULL = BAR_SBEMPTY + SBR;
constexpr int BAR_TEMPTY = BAR_TFULL + 4;
constexpr int BAR_DRAIN = BAR_TEMPTY + 4;
constexpr int NUM_BARS = BAR_DRAIN + 1;
constexpr int SMEM_TMEMPTR = SMEM_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = SMEM_TMEMPTR + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;    // slack for 1024-byte alignment
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(SMEM_B % 1024 == 0 && SMEM_SB % 16 == 0 && SB_BYTES % 16 == 0 && SMEM_BAR % 8 == 0,
              "alignment");


struct GemmArgs {
    const uint8_t* A;     // activation code tiles      [num_m][nkb][16 KiB]
    const uint8_t* AS;    // token scale pairs          [num_m][nchunk][128] x {f32 d, i32 ssum}
    const uint8_t* AM;    // token min-term tiles       [num_m][nsb][hi 4 KiB, lo 4 KiB]
    const uint8_t* B;     // weight code tiles          [num_n][nkb][16 KiB]
    const uint8_t* B2;    // q6_K second code tiles     [num_n][nkb][16 KiB] (two-tile codes)
    const uint8_t* SBD;   // weight d per super-block   [num_n][nsb][128] f32
    const uint8_t* AUX;   // q4_K min-term tiles [num_n][nsb][8 KiB]
    const unsigned int* FLAG;
    float* out;           // Y [M][ldy], or the dot dump [M][od][nsub]
    int ldy;
    int M, od, id;
    int num_m, num_n;
    int units;            // work units of the launch (see unit_of)
    int full_units;       // units below this are whole tiles
    int nsb_half;         // split units: super-blocks [0, nsb_half) and [nsb_half, nsb)
    int vec_store;        // Y is 16-byte aligned and ldy % 4 == 0
    unsigned int* err;    // the library's sticky error word
    unsigned long long wait_ns;   // limit of each bounded wait
    int withhold;         // verification: operand fill CTA 0's producer leaves out (-1: none)
};

// Bounded wait that ignores the error word (used only to drain our own copies /
// MMAs in flight before the CTA exits; those always complete).
__device__ __forceinline__ void drain_wait(const GemmArgs& g, uint32_t bar, uint32_t parity)
{
    mbar_drain_wait(bar, parity, WAIT_LIMIT_NS, g.err);
}

// Bounded wait of the single producer / MMA thread.
__device__ __forceinline__ bool ctl_wait(const GemmArgs& g, uint32_t bar, uint32_t parity)
{
    return mbar_wait(bar, parity, g.wait_ns, g.err);
}

// Bounded wait by a whole warp; the verdict is made warp-uniform so that every lane
// takes the same branch after it.
__device__ __forceinline__ bool warp_wait(const GemmArgs& g, uint32_t bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, g.wait_ns, g.err));
}

// Verification: the operand fill of this CTA's producer that is left out (never
// armed, never copied) so that the consumers' wait for it runs out; ~0 for none.
__device__ __forceinline__ uint32_t withheld_fill(const GemmArgs& g)
{
    return (blockIdx.x == 0 && g.withhold >= 0) ? static_cast<uint32_t>(g.withhold) : ~0u;
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

template <int R>
__device__ __forceinline__ void regs_grow()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_shrink()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(R));
}

// Work unit u of a launch: tile (m, n) and its super-block range [sb0, sb1).  Units
// below full_units are whole tiles, taken in order; each later pair of units is the
// two K-halves of one tile of the last round, whose partial sums are added into a
// zeroed Y (two addends: the order cannot change the sum).  Splitting the last
// round's tiles keeps SMs busy that would otherwise idle while it runs.
struct Unit {
    int m, n, sb0, sb1;
    bool half;
};
__device__ __forceinline__ Unit unit_of(const GemmArgs& g, int u, int nsb)
{
    Unit w;
    int tile;
    if (u < g.full_units) {
        tile = u;
        w.sb0 = 0;
        w.sb1 = nsb;
        w.half = false;
    } else {
        const int v = u - g.full_units;
        tile = g.full_units + (v >> 1);
        w.half = true;
        w.sb0 = (v & 1) ? g.nsb_half : 0;
        w.sb1 = (v & 1) ? nsb : g.nsb_half;
    }
    w.m = tile % g.num_m;
    w.n = tile / g.num_m;
    return w;
}

// Position in a ring of N entries: entry index and the phase parity of its barriers.
template <uint32_t N>
struct RingPos {
    uint32_t i = 0, ph = 0;
    __device__ __forceinline__ void next()
    {
        if (++i == N) {
            i = 0;
            ph ^= 1u;
        }
    }
};

// The three roles of one CTA.  TYPE 12 = q4_K, 14 = q6_K; MODE GEMM_Y or GEMM_DOTS;
// TILES = 1 (codes sc * q) or 2 (q6_K with some |sc| > 64: tiles sc * l and
// 16 sc (h - 2), two MMAs per 16 values into the same accumulator).
template <int TYPE, int MODE, int TILES>
__device__ __forceinline__ void gemm_roles(const GemmArgs& g, uint8_t* smem, uint32_t sbase, uint32_t tmem_base,
                                           int warp, int lane)
{
    constexpr bool Q4 = (TYPE == 12);
    // TMEM holds two 256-column items, synchronised as units: one 64-value k-block (its
    // two chunks' accumulators side by side); q4_K's min term takes an item of its own
    // per tile.
    constexpr uint32_t ITEM_COLS = 2 * BN;
    const int nkb = g.id / BK;
    const int nchunk = g.id / CHUNK;
    const int nsb = g.id / QK_K;
    auto bar = [&](int i) -> uint32_t { return sbase + SMEM_BAR + 8u * static_cast<uint32_t>(i); };

    if (warp < PROMO_WARP0) {
        regs_shrink<CTRL_REGS>();
        // One thread of warp 0 produces and one thread of warp 1 issues MMAs; the other
        // lanes of the control warpgroup wait at the CTA's final barrier.
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------------- producer
            RingPos<STAGES> op;
            RingPos<SBR> sb;
            uint32_t n_ops = 0, n_sb = 0;  // fills issued on each ring
            constexpr uint32_t sb_tx = SB_SBD_BYTES + SB_AS_BYTES;
            const uint32_t skip = withheld_fill(g);
            bool ok = true;
            for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
                const Unit w = unit_of(g, u, nsb);
                const int m = w.m, n = w.n;
                const uint8_t* Ab = g.A + static_cast<size_t>(m) * nkb * TILE_BYTES;
                const uint8_t* Bb = g.B + static_cast<size_t>(n) * nkb * TILE_BYTES;
                const uint8_t* B2b = (TILES == 2) ? g.B2 + static_cast<size_t>(n) * nkb * TILE_BYTES : nullptr;
                const uint8_t* ASb = g.AS + static_cast<size_t>(m) * nchunk * BM * 8;
                for (int kb = 4 * w.sb0; kb < 4 * w.sb1; ++kb) {
                    if ((kb & 3) == 0) {  // a new super-block
                        const int s = kb >> 2;
                        if (!ctl_wait(g, bar(BAR_SBEMPTY + sb.i), sb.ph ^ 1u)) {
                            ok = false;
                            break;
                        }
                        // The promotion warps read this entry with ordinary loads before
                        // releasing it; order those reads before the bulk copy's writes.
                        fence_proxy_async_smem();
                        const uint32_t dst = sbase + SMEM_SB + sb.i * SB_BYTES;
                        const uint32_t fb = bar(BAR_SBFULL + sb.i);
                        mbar_arrive_expect_tx(fb, sb_tx);
                        bulk_g2s(dst + SB_SBD_OFF, g.SBD + (static_cast<size_t>(n) * nsb + s) * SB_SBD_BYTES,
                                 SB_SBD_BYTES, fb);
                        bulk_g2s(dst + SB_AS_OFF, ASb + static_cast<size_t>(s) * SB_AS_BYTES, SB_AS_BYTES, fb);
                        sb.next();
                        ++n_sb;
                    }
                    if (!ctl_wait(g, bar(BAR_EMPTY + op.i), op.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    if (n_ops == skip) {
                        op.next();
                        ++n_ops;
                        continue;
                    }
                    const uint32_t fo = bar(BAR_FULL + op.i);
                    mbar_arrive_expect_tx(fo, (1 + TILES) * TILE_BYTES);
                    bulk_g2s(sbase + SMEM_A + op.i * TILE_BYTES, Ab + static_cast<size_t>(kb) * TILE_BYTES,
                             TILE_BYTES, fo);
                    bulk_g2s(sbase + SMEM_B + op.i * B_STAGE, Bb + static_cast<size_t>(kb) * TILE_BYTES,
                             TILE_BYTES, fo);
                    if (TILES == 2)
                        bulk_g2s(sbase + SMEM_B + op.i * B_STAGE + TILE_BYTES,
                                 B2b + static_cast<size_t>(kb) * TILE_BYTES, TILE_BYTES, fo);
                    op.next();
                    ++n_ops;
                }
                if (Q4 && ok) {
                    // The tile's min-term operands, one super-block per stage: token hi/lo
                    // tiles in the A slot, weight hi/lo tiles in the B slot.
                    for (int s = w.sb0; s < w.sb1; ++s) {
                        if (!ctl_wait(g, bar(BAR_EMPTY + op.i), op.ph ^ 1u)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fo = bar(BAR_FULL + op.i);
                        mbar_arrive_expect_tx(fo, MIN_AM_BYTES + MIN_BM_BYTES);
                        bulk_g2s(sbase + SMEM_A + op.i * TILE_BYTES,
                                 g.AM + (static_cast<size_t>(m) * nsb + s) * MIN_AM_BYTES, MIN_AM_BYTES, fo);
                        bulk_g2s(sbase + SMEM_B + op.i * B_STAGE,
                                 g.AUX + (static_cast<size_t>(n) * nsb + s) * MIN_BM_BYTES, MIN_BM_BYTES, fo);
                        op.next();
                        ++n_ops;
                    }
                }
            }
            // Our copies must have landed before the CTA may exit.
            for (uint32_t i = (n_ops > STAGES ? n_ops - STAGES : 0); i < n_ops; ++i)
                if (i != skip)
                    drain_wait(g, bar(BAR_FULL + i % STAGES), (i / STAGES) & 1u);
            for (uint32_t i = (n_sb > SBR ? n_sb - SBR : 0); i < n_sb; ++i)
                drain_wait(g, bar(BAR_SBFULL + i % SBR), (i / SBR) & 1u);
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            constexpr uint32_t idesc_t = idesc_tf32_f32(BM, BN);
            RingPos<STAGES> op;
            RingPos<2> item;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
                const Unit w = unit_of(g, u, nsb);
                for (int kb = 4 * w.sb0; kb < 4 * w.sb1; ++kb) {
                    if (!ctl_wait(g, bar(BAR_FULL + op.i), op.ph)) {
                        ok = false;
                        break;
                    }
                    const uint64_t a0 = sdesc_k_sw128(sbase + SMEM_A + op.i * TILE_BYTES);
                    const uint64_t b0 = sdesc_k_sw128(sbase + SMEM_B + op.i * B_STAGE);
                    const uint64_t b1 = sdesc_k_sw128(sbase + SMEM_B + op.i * B_STAGE + TILE_BYTES);
                    // K advance inside the 128-byte swizzled rows: 32 bytes per 16 values
                    // (the descriptor's address field counts 16-byte units).
                    // one item per k-block: one wait, one fence, one commit for two chunks
                    if (!ctl_wait(g, bar(BAR_TEMPTY + item.i), item.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + item.i * ITEM_COLS;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        umma_f16(d + cc * BN, a0 + 4u * cc, b0 + 4u * cc, idesc, 0u);
                        umma_f16(d + cc * BN, a0 + 4u * cc + 2, b0 + 4u * cc + 2, idesc, 1u);
                        if (TILES == 2) {
                            umma_f16(d + cc * BN, a0 + 4u * cc, b1 + 4u * cc, idesc, 1u);
                            umma_f16(d + cc * BN, a0 + 4u * cc + 2, b1 + 4u * cc + 2, idesc, 1u);
                        }
                    }
                    umma_commit(bar(BAR_TFULL + item.i));
                    item.next();
                    umma_commit(bar(BAR_EMPTY + op.i));  // operand stage free once these MMAs finish
                    op.next();
                }
                // Min-term contraction of the tile, sum over chunks of (d_a*ssum)(dmin*m),
                // one super-block (8 chunks, hi/lo split) per stage, into one item per
                // MIN_GROUP_SB super-blocks that the promotion subtracts in f32: the tensor
                // core's own accumulation then never chains more than 3 * MIN_GROUP_SB MMAs.
                for (int g0 = w.sb0; Q4 && ok && g0 < w.sb1; g0 += MIN_GROUP_SB) {
                    const int g1 = min(g0 + MIN_GROUP_SB, w.sb1);
                    if (!ctl_wait(g, bar(BAR_TEMPTY + item.i), item.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t d = tmem_base + item.i * ITEM_COLS;
                    for (int s = g0; s < g1; ++s) {
                        if (!ctl_wait(g, bar(BAR_FULL + op.i), op.ph)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t am = sbase + SMEM_A + op.i * TILE_BYTES;
                        const uint32_t bm = sbase + SMEM_B + op.i * B_STAGE;
                        const uint64_t ahi = sdesc_tf32_tile(am), alo = sdesc_tf32_tile(am + TF32_TILE_BYTES);
                        const uint64_t bhi = sdesc_tf32_tile(bm), blo = sdesc_tf32_tile(bm + TF32_TILE_BYTES);
                        umma_tf32(d, ahi, bhi, idesc_t, s > g0 ? 1u : 0u);
                        umma_tf32(d, ahi, blo, idesc_t, 1u);
                        umma_tf32(d, alo, bhi, idesc_t, 1u);
                        umma_commit(bar(BAR_EMPTY + op.i));
                        op.next();
                    }
                    if (!ok)
                        break;
                    umma_commit(bar(BAR_TFULL + item.i));
                    item.next();
                }
            }
            umma_commit(bar(BAR_DRAIN));  // every MMA issued so far has completed
            drain_wait(g, bar(BAR_DRAIN), 0u);
        }
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------------- promotion
    regs_grow<PROMO_REGS>();
    const int pw = warp - PROMO_WARP0;              // 0..7
    const int q = warp & 3;                          // TMEM lane quarter this warp may read
    const int hc = pw >> 2;                          // which 64 of the 128 columns
    const int row_in_tile = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    RingPos<2> item;
    RingPos<SBR> sb;
    auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar(BAR_TEMPTY + item.i));
        item.next();
    };
    bool ok = true;
    for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
        const Unit w = unit_of(g, u, nsb);
        const int m = w.m, n = w.n;
        const int row = m * BM + row_in_tile;
        const int jb = n * BN + hc * COLS_PER_WARP;
        float2 acc[COLS_PER_WARP / 2];
#pragma unroll
        for (int i = 0; i < COLS_PER_WARP / 2; ++i)
            acc[i] = make_float2(0.0f, 0.0f);
        for (int s = w.sb0; s < w.sb1; ++s) {
            const uint8_t* sbe = smem + SMEM_SB + sb.i * SB_BYTES;
            if (!warp_wait(g, bar(BAR_SBFULL + sb.i), sb.ph)) {
                ok = false;
                break;
            }
            const uint2* tsc = reinterpret_cast<const uint2*>(sbe + SB_AS_OFF);
            float2 inner[COLS_PER_WARP / 2];
#pragma unroll
            for (int i = 0; i < COLS_PER_WARP / 2; ++i)
                inner[i] = make_float2(0.0f, 0.0f);
            for (int k2 = 0; k2 < 4 && ok; ++k2) {             // the super-block's four k-blocks
                if (!warp_wait(g, bar(BAR_TFULL + item.i), item.ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col0 = lane_addr + item.i * ITEM_COLS + hc * COLS_PER_WARP;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int k = 2 * k2 + cc;
                    const int c = 8 * s + k;                    // chunk index along id
                    float I[COLS_PER_WARP];
                    tmem_ld64_wait(col0 + cc * BN, I);
                    if (cc == 1)
                        release();                              // both chunks are in registers
                    if (MODE == GEMM_Y) {
                        const float da = __uint_as_float(tsc[k * BM + row_in_tile].x);
                        const float2 da2 = make_float2(da, da);
#pragma unroll
                        for (int i = 0; i < COLS_PER_WARP / 2; ++i)
                            inner[i] = ffma2(da2, make_float2(I[2 * i], I[2 * i + 1]), inner[i]);
                    } else if (row < g.M) {
#pragma unroll
                        for (int i = 0; i < COLS_PER_WARP; ++i) {
                            const int j = jb + i;
                            if (j < g.od)
                                g.out[(static_cast<size_t>(row) * g.od + j) * nchunk + c] = I[i];
                        }
                    }
                }
            }
            if (!ok)
                break;
            // acc += d * inner  (d per weight row of this super-block)
            if (MODE == GEMM_Y) {
                const float4* d4 = reinterpret_cast<const float4*>(sbe + SB_SBD_OFF) + hc * (COLS_PER_WARP / 4);
#pragma unroll
                for (int i = 0; i < COLS_PER_WARP / 4; ++i) {
                    const float4 dv = d4[i];
                    acc[2 * i] = ffma2(make_float2(dv.x, dv.y), inner[2 * i], acc[2 * i]);
                    acc[2 * i + 1] = ffma2(make_float2(dv.z, dv.w), inner[2 * i + 1], acc[2 * i + 1]);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(BAR_SBEMPTY + sb.i));
            sb.next();
        }
        if (!ok)
            break;
        // acc -= the tile's min term, one item per MIN_GROUP_SB super-blocks
        for (int g0 = w.sb0; Q4 && g0 < w.sb1; g0 += MIN_GROUP_SB) {
            if (!warp_wait(g, bar(BAR_TFULL + item.i), item.ph)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float mn[COLS_PER_WARP];
            tmem_ld64_wait(lane_addr + item.i * ITEM_COLS + hc * COLS_PER_WARP, mn);
            release();
            if (MODE == GEMM_Y) {
#pragma unroll
                for (int i = 0; i < COLS_PER_WARP / 2; ++i)
                    acc[i] = ffma2(make_float2(-1.0f, -1.0f), make_float2(mn[2 * i], mn[2 * i + 1]), acc[i]);
            }
        }
        if (!ok)
            break;
        if (MODE == GEMM_Y && row < g.M) {
            float* yrow = g.out + static_cast<size_t>(row) * g.ldy;
#pragma unroll
            for (int i = 0; i < COLS_PER_WARP; i += 4) {
                const int j = jb + i;
                const float2 lo = acc[i / 2], hi = acc[i / 2 + 1];
                if (w.half) {
                    if (g.vec_store && j + 3 < g.od) {
                        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(yrow + j), "f"(lo.x),
                                     "f"(lo.y), "f"(hi.x), "f"(hi.y)
                                     : "memory");
                    } else {
                        const float v[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (j + k < g.od)
                                atomicAdd(yrow + j + k, v[k]);
                    }
                } else if (g.vec_store && j + 3 < g.od) {
                    *reinterpret_cast<float4*>(yrow + j) = make_float4(lo.x, lo.y, hi.x, hi.y);
                } else {
                    const float v[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (j + k < g.od)
                            yrow[j + k] = v[k];
                }
            }
        }
    }
}

template <int TYPE, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const GemmArgs g)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sbase + SMEM_BAR + 8u * static_cast<uint32_t>(i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(BAR_FULL + s), 1);
            mbar_init(bar(BAR_EMPTY + s), 1);
        }
        for (int s = 0; s < SBR; ++s) {
            mbar_init(bar(BAR_SBFULL + s), 1);
            mbar_init(bar(BAR_SBEMPTY + s), NUM_PROMO_WARPS);
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
    // A dependent launch: the set-up above overlapped the end of the kernel ahead (the
    // prepass, or the repack that wrote the flag); nothing global is read before it has
    // completed, and the next kernel may be scheduled from here on.
    grid_dep_wait();
    grid_dep_launch();

    if constexpr (TYPE == 14) {
        // q6_K codes hold sc*q in one tile unless some |sc| > 64 (then two exact tiles);
        // the repack recorded which in the flag word (uniform for the launch).
        if (__ldg(g.FLAG) != 0u)
            gemm_roles<14, MODE, 1>(g, smem, sbase, tmem_base, warp, lane);
        else
            gemm_roles<14, MODE, 2>(g, smem, sbase, tmem_base, warp, lane);
    } else {
        gemm_roles<12, MODE, 1>(g, smem, sbase, tmem_base, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

constexpr int ZERO_ROWS = 16;   // rows of Y a zeroing block clears

// Zeroes Y over the tiles [first, first + count) of a launch (rows < M, columns < od).
__global__ void __launch_bounds__(256) zero_tiles_kernel(float* __restrict__ Y, int ldy, int M, int od, int num_m,
                                                         int first)
{
    // Y may still be written by the kernel ahead (a GEMM into the same buffer).
    grid_dep_wait();
    grid_dep_launch();
    // block (tile, row group of ZERO_ROWS rows); consecutive threads take consecutive columns
    const int tile = first + blockIdx.x;
    const int m = tile % num_m, n = tile / num_m;
    const int r0 = blockIdx.y * ZERO_ROWS;
    const int r_end = min(r0 + ZERO_ROWS, M - m * BM), c_end = min(BN, od - n * BN);
    for (int e = threadIdx.x; e < ZERO_ROWS * BN; e += blockDim.x) {
        const int r = r0 + e / BN, c = e % BN;
        if (r < r_end && c < c_end)
            Y[static_cast<size_t>(m * BM + r) * ldy + n * BN + c] = 0.0f;
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
        // The setmaxnreg split draws on the registers the launch reserved; a build
        // that compiled to fewer per thread would make the promotion wait forever.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, gemm_kernel<TYPE, MODE>);
        if (e != cudaSuccess)
            return e;
        if (fa.numRegs < LAUNCH_REGS)
            return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(gemm_kernel<TYPE, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess)
            return e;
        attr_set_mask.fetch_or(bit);
    }
    count_launch();
    return launch_dependent_smem(gemm_kernel<TYPE, MODE>, dim3(grid), dim3(NUM_THREADS), SMEM_ALLOC, s, a);
}

}  // namespace

std::atomic<int> g_large_m_kernel{0};

void select_large_m_kernel(int which) { g_large_m_kernel.store(which); }
int large_m_kernel() { return g_large_m_kernel.load(); }

cudaError_t launch_gemm(int type, GemmMode mode, const void* packed, int od, int id, const void* qa,
                        const void* scales, int M, float* out, int ldy, cudaStream_t s, const char** path_label)
{
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    // Y goes to the super-block kernel or to this chunk kernel by a round-count cost
    // model of both (two-tile q6_K always here); both read the one- or two-tile q6_K
    // codes, so the fold state recorded at registration only steers the speed.
    const int sel = g_large_m_kernel.load();
    const bool sb_first =
        mode == GEMM_Y &&
        (sel == 2 || (sel == 0 && M > FT_MAX_M &&
                      prefer_superblock(type, od, id, M, nsm,
                                        type == 14 ? packed_fold_state(dev, packed, type, od, id) : 1)));
    WaitCtl wc;
    bool injected = false;
    e = take_wait_ctl(&wc, &injected);
    if (e != cudaSuccess)
        return e;
    // Few tokens: the few-token GEMM (compact codes widened into tensor memory, one TMEM
    // accumulator per super-block), unless a tile kernel was selected.  No cluster split
    // under a wait-timeout injection: a cluster barrier has no time limit.
    if (mode == GEMM_Y && M <= FT_MAX_M && (sel == 0 || sel == 3 || sel == 4))
        return launch_gemm_ft(type, packed, od, id, qa, scales, M, out, ldy, s, wc, !injected && sel != 3,
                              path_label);
    if (sb_first) {
        e = launch_gemm_sb(type, packed, od, id, qa, scales, M, out, ldy, s, wc);
        if (e == cudaSuccess && path_label)
            *path_label = type == 12
                              ? "q4_K: super-block tcgen05 GEMM, 128x256 tiles, activation operand p*d_a*q_a split "
                                "f16 hi+lo in shared memory, one TMEM accumulator per super-block, tf32 hi/lo min term"
                              : "q6_K: super-block tcgen05 GEMM, 128x256 tiles, activation operand p*d_a*q_a split "
                                "f16 hi+lo in shared memory, one TMEM accumulator per super-block; codes sc*q in one "
                                "f16 tile (every |sc| <= 64) or two exact tiles sc*l and 16*sc*(h-2)";
        return e;
    }
    const WeightPlanes wp = weight_planes(type, od, id);
    const ActPlanes ap = act_planes(M, id);
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    const uint8_t* sc = static_cast<const uint8_t*>(scales);
    GemmArgs a;
    a.A = static_cast<const uint8_t*>(qa);
    a.AS = sc + ap.pair_off;
    a.AM = sc + ap.am_off;
    a.B = pk + wp.code_off;
    a.B2 = pk + wp.code2_off;
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
    a.err = wc.err;
    a.wait_ns = wc.limit_ns;
    a.withhold = wc.withhold_fill;

    const int tiles = a.num_m * a.num_n;
    int grid = tiles < nsm ? tiles : nsm;
    a.units = tiles;
    a.full_units = tiles;
    a.nsb_half = 0;
    const int rem = tiles % grid;
    const int nsb = id / QK_K;
    // Tiles run as two K-halves added into a zeroed Y (two addends: the order cannot
    // change the sum): every tile when the launch has at most half as many tiles as SMs
    // (decode-tail shapes), else the last round's tiles when they fill at most half.
    int split = 0;
    if (mode == GEMM_Y && !sb_first && nsb >= 2) {
        if (2 * tiles <= nsm)
            split = tiles;
        else if (tiles > grid && rem > 0 && 2 * rem <= grid)
            split = rem;
    }
    if (split > 0) {
        a.full_units = tiles - split;
        a.units = a.full_units + 2 * split;
        a.nsb_half = nsb / 2;
        grid = a.units < nsm ? a.units : nsm;
        count_launch();
        e = launch_dependent(zero_tiles_kernel, dim3(static_cast<unsigned>(split), BM / ZERO_ROWS), dim3(256), s, out,
                             ldy, M, od, a.num_m, a.full_units);
        if (e != cudaSuccess)
            return e;
    }

    if (type == 14) {
        if (path_label)
            *path_label = "q6_K: chunk GEMM, tcgen05.mma kind::f16 128x128x16 on exact int codes (sc*q in one f16 "
                          "tile, or two exact tiles sc*l and 16*sc*(h-2)), two 256-column TMEM items, f32 d_a per "
                          "chunk / d per super-block";
        return mode == GEMM_Y ? launch_typed<14, GEMM_Y>(a, grid, s) : launch_typed<14, GEMM_DOTS>(a, grid, s);
    }
    if (path_label)
        *path_label = "q4_K: chunk GEMM, tcgen05.mma kind::f16 128x128x16 on scale-folded exact int codes, two "
                      "256-column TMEM items, tf32 hi/lo min term per tile, f32 d_a per chunk / d per super-block";
    return mode == GEMM_Y ? launch_typed<12, GEMM_Y>(a, grid, s) : launch_typed<12, GEMM_DOTS>(a, grid, s);
}

}  // namespace mmq
