// gemm_sb.cu -- super-block-accumulating q4_K / q6_K x q8 GEMM for sm_103a (the
// default large-M path for scale-folded weight codes).
//
// The per-32-value activation scale d_a is what forces the chunk-granular kernel
// (gemm.cu) to take one TMEM round trip and one f32 FMA per accumulator element
// per chunk.  This kernel moves d_a onto the activation operand instead, so that
// the tensor core sums a whole 256-value super-block into one accumulator:
//
//   a[t,k] = p[t,sb] * d_a[t,c(k)] * q_a[t,k] = s * q_a,   s = s_hi + s_lo (f16 pair)
//   a     ~= hi + lo,  hi = rn_f16(s_hi*q_a),  lo = rn_f16(s_hi*q_a - hi + s_lo*q_a)
//   D[t,j] = sum_{k in sb} hi[t,k] * w[j,k] + lo[t,k] * w[j,k]   (tensor core, f32)
//   Y[t,j] = sum_sb d_sb[j] * D[t,j] / p[t,sb]   -   sum_c (d_a*ssum)[t,c] * (dmin*m)[j,c]
//
// w = sc*q are the registration-time scale-folded integer codes (exact in f16), so
// every product hi*w, lo*w is exact and the only roundings are the split (about
// 2^-21 relative per activation value) and the f32 sums: far inside the
// 1e-5 bound on Y, and no longer bit-comparable per chunk (the per-chunk integer
// dots are checked on gemm.cu, which keeps that form).  p = 2^e is chosen per
// (token, super-block) from the largest d_a so that 127 * max d_a * p <= 2^14:
// hi stays finite and lo stays out of the f16 subnormal range for every value
// within 2^17 of the super-block's largest.  The q4_K min term is the same tf32
// hi/lo contraction over chunks as in gemm.cu, per tile in items of 64 super-blocks.
//
// One CTA per SM, persistent over 128-token x 256-row tiles (N = 256: two 128-row
// weight tiles side by side); 16 warps in four warpgroups:
//   warp 0      producer: cp.async.bulk of the f16 activation code tile (on its own
//               barrier) and the two weight code tiles of each 64-value k-block into
//               a 3-deep ring, with an L2 prefetch of the tiles the stage takes next;
//               the super-block entries (weight d of 256 rows, token {d, ssum} of its
//               8 chunks) into a 3-deep ring; then the q4_K min-term operands, two
//               super-blocks per stage, prefetched into L2 when the tile starts.
//   warp 1      allocates TMEM (two 256-column items); one thread issues per k-block
//               eight tcgen05.mma kind::f16 128x256x16 (hi and lo for each 16 values)
//               into the item of the current super-block, commits the stage, and
//               commits the item after the super-block's fourth k-block.
//   warps 2-3   idle (they lend their registers).
//   warps 4-7   converter: thread r owns token row r of the tile; per super-block it
//               derives p from the row's 8 chunk scales and publishes 1/p; per
//               k-block it reads its row's 64 codes from the stage (all eight 16-byte
//               groups first), writes hi in place and lo into the stage's second slot
//               (same swizzled positions), fences the async proxy and arrives on the
//               stage's CONV barrier.
//   warps 8-15  promotion: each owns one TMEM lane quarter (warp % 4) and 128 of the
//               256 columns; per super-block: wait, four tcgen05.ld (16x256b shape,
//               64 columns), release, acc += d_sb * (D / p); per tile acc -= the q4_K
//               min-term items; store Y (or, for K-halves, add into a zeroed Y) as float2,
//               whole 32-byte sectors per quad.
// The synchronisation count per tensor-core FLOP is 8x lower than in gemm.cu and
// the promotion does one FMA pair per accumulator element per super-block rather
// than one FMA per chunk; the tensor pipe does twice the MMAs (hi and lo).
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

constexpr int BM = 128;               // tokens per tile (TMEM lanes, MMA M)
constexpr int BN = 256;               // weight rows per tile (MMA N): two 128-row tiles
constexpr int SBR = 3;                // super-block ring depth
constexpr int NUM_WARPS = 16;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int CONV_WARP0 = 4;
constexpr int NUM_CONV_WARPS = 4;
constexpr int PROMO_WARP0 = 8;
constexpr int NUM_PROMO_WARPS = 8;
constexpr int COLS_PER_WARP = BN / 2;  // 128
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ITEM_COLS = BN;     // one super-block accumulator
// Register split out of the launch's 128 x 512: control 56, converter 56,
// promotion 200 (128 tile accumulators + one 32-column load per thread).
constexpr int LAUNCH_REGS = 128;
constexpr int CTRL_REGS = 56;
constexpr int CONV_REGS = 56;
constexpr int PROMO_REGS = 200;
static_assert(CTRL_REGS * 128 + CONV_REGS * 128 + PROMO_REGS * 256 <= LAUNCH_REGS * NUM_THREADS, "register split");

// One operand stage: activation codes (converted in place to hi), lo, and the two
// weight tiles.  For a q4_K min-term stage the first slot holds the token tf32
// hi/lo tiles and the weight slot the weight tf32 tiles [hi n0 | hi n1 | lo n0 | lo n1].
constexpr int ST_A = 0;
constexpr int ST_LO = TILE_BYTES;
constexpr int ST_B = 2 * TILE_BYTES;
constexpr int MIN_AM_BYTES = 2 * TF32_TILE_BYTES;      // token hi, lo
constexpr int MIN_BM_BYTES = 2 * TF32_TILE_BYTES;      // per 128-row weight tile: hi, lo
// Min-term super-blocks per stage: a stage of one super-block holds only 384 cycles of
// tensor work, too little to cover the copy latency of the next.
constexpr int MIN_PER_STAGE = 2;
// Min-term super-blocks per TMEM item, each subtracted by the promotion in f32, so that the
// tensor core's own accumulation never chains more than 3 * MIN_GROUP_SB MMAs; shapes with
// id <= 64 * 256 take one item per tile.  A multiple of MIN_PER_STAGE: no stage straddles
// two items.
constexpr int MIN_GROUP_SB = 64;
static_assert(MIN_GROUP_SB % MIN_PER_STAGE == 0, "min-term groups hold whole stages");

// One super-block entry: weight d of the 256 rows, then {d, ssum} of the 8 chunks
// for the 128 tokens ([chunk][token]) (both copied in), then 1/p per token (written
// by the converter).
constexpr int SB_SBD_OFF = 0;
constexpr int SB_SBD_BYTES = BN * 4;
constexpr int SB_AS_OFF = SB_SBD_OFF + SB_SBD_BYTES;
constexpr int SB_AS_BYTES = 8 * BM * 8;
constexpr int SB_IP_OFF = SB_AS_OFF + SB_AS_BYTES;
constexpr int SB_IP_BYTES = BM * 4;
constexpr int SB_COPY_BYTES = SB_SBD_BYTES + SB_AS_BYTES;
constexpr int SB_BYTES = SB_IP_OFF + SB_IP_BYTES;

// Shared-memory plan of a launch, by the number of exact weight tiles per k-block:
// TILES = 1 (codes sc * q): 3 stages of [A | lo | B n0 | B n1]; TILES = 2 (q6_K with
// some |sc| > 64: tiles sc * l and 16 sc (h - 2)): 2 stages of [A | lo | B n0 | B n1 |
// B2 n0 | B2 n1].
template <int TILES>
struct SbL {
    static constexpr int STAGES = TILES == 1 ? 3 : 2;         // operand ring depth
    static constexpr int STAGE_BYTES = (2 + 2 * TILES) * TILE_BYTES;
    static constexpr int SMEM_ST = 0;
    static constexpr int SMEM_SB = SMEM_ST + STAGES * STAGE_BYTES;
    static constexpr int SMEM_BAR = SMEM_SB + SBR * SB_BYTES;
    static constexpr int BAR_FULL = 0;                      // the stage's activation (or min-term token) tile
    static constexpr int BAR_FULLB = BAR_FULL + STAGES;     // the stage's weight tiles
    static constexpr int BAR_CONV = BAR_FULLB + STAGES;
    static constexpr int BAR_EMPTY = BAR_CONV + STAGES;
    static constexpr int BAR_SBFULL = BAR_EMPTY + STAGES;
    static constexpr int BAR_SBEMPTY = BAR_SBFULL + SBR;
    static constexpr int BAR_IPREADY = BAR_SBEMPTY + SBR;
    static constexpr int BAR_TFULL = BAR_IPREADY + SBR;
    static constexpr int BAR_TEMPTY = BAR_TFULL + 2;
    static constexpr int BAR_DRAIN = BAR_TEMPTY + 2;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr int SMEM_TMEMPTR = SMEM_BAR + NUM_BARS * 8;
    static constexpr int SMEM_USED = SMEM_TMEMPTR + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;    // slack for 1024-byte alignment
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(STAGE_BYTES % 1024 == 0 && SMEM_SB % 1024 == 0 && SB_BYTES % 16 == 0 && SMEM_BAR % 8 == 0,
                  "alignment");
};
constexpr int SMEM_ALLOC = SbL<1>::SMEM_ALLOC > SbL<2>::SMEM_ALLOC ? SbL<1>::SMEM_ALLOC : SbL<2>::SMEM_ALLOC;
static_assert(MIN_PER_STAGE * MIN_AM_BYTES <= TILE_BYTES && MIN_PER_STAGE * 2 * MIN_BM_BYTES <= 2 * TILE_BYTES,
              "min-term operands fit a stage");

struct SbArgs {
    const uint8_t* A;     // activation code tiles      [num_m][nkb][16 KiB]
    const uint8_t* AS;    // token scale pairs          [num_m][nchunk][128] x {f32 d, i32 ssum}
    const uint8_t* AM;    // token min-term tiles       [num_m][nsb][hi 4 KiB, lo 4 KiB]
    const uint8_t* B;     // weight code tiles          [num_n128][nkb][16 KiB]
    const uint8_t* B2;    // q6_K second code tiles     [num_n128][nkb][16 KiB] (two-tile codes)
    const uint8_t* SBD;   // weight d per super-block   [num_n128][nsb][128] f32
    const uint8_t* AUX;   // q4_K min-term tiles        [num_n128][nsb][hi 4 KiB, lo 4 KiB]
    const unsigned int* FLAG;
    float* Y;             // [M][ldy]
    int ldy;
    int M, od, id;
    int num_m, num_n;     // num_n counts 256-row tiles
    int num_n128;         // 128-row weight tiles in the packed planes
    int units, full_units, nsb_half;
    int vec_store;        // Y is 8-byte aligned and ldy is even (float2 stores)
    unsigned int* err;    // the library's sticky error word
    unsigned long long wait_ns;   // limit of each bounded wait
    int withhold;         // verification: operand fill CTA 0's producer leaves out (-1: none)
};

__device__ __forceinline__ void drain_wait(const SbArgs& g, uint32_t bar, uint32_t parity)
{
    mbar_drain_wait(bar, parity, WAIT_LIMIT_NS, g.err);
}

__device__ __forceinline__ bool ctl_wait(const SbArgs& g, uint32_t bar, uint32_t parity)
{
    return mbar_wait(bar, parity, g.wait_ns, g.err);
}

__device__ __forceinline__ bool warp_wait(const SbArgs& g, uint32_t bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, g.wait_ns, g.err));
}

// 128 x 8 tf32 tile, no swizzle, K-major core matrices (see tf32_tile_byte): K-direction
// core-matrix stride 128 B, 8-row group stride 256 B.  Two such tiles back to back form
// the 256-row operand.
__device__ __forceinline__ uint64_t sdesc_tf32(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128u >> 4) << 16;
    d |= static_cast<uint64_t>(256u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}

__host__ __device__ constexpr uint32_t idesc_tf32(int m, int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
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

// tcgen05.ld.16x256b.x8 and its wait: 16 TMEM lanes from the address's lane, 64
// columns from its column; thread t receives, for n = 0..7, v[4n], v[4n+1] = lane
// t/4, columns 8n + 2(t%4) + {0, 1}, and v[4n+2], v[4n+3] = lane 8 + t/4, the same
// columns.
__device__ __forceinline__ void tmem_ld16x256b_x8_wait(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Power-of-two operand scale of one (token, super-block) from the largest of its 8
// chunk scales dmax >= 0: the f32 exponent field of p is min(260 - E, 253), E the
// exponent field of dmax, so that 127 * dmax * p < 2^14; 1/p is exact and normal.
__device__ __forceinline__ uint32_t p_field(float dmax)
{
    const int E = static_cast<int>((__float_as_uint(dmax) >> 23) & 0xFFu);
    return static_cast<uint32_t>(min(260 - E, 253));
}

// Work unit u: tile (m, n) and its super-block range [sb0, sb1); units from
// full_units on are the two K-halves of the tiles of the last round.
struct Unit {
    int m, n, sb0, sb1;
    bool half;
};
__device__ __forceinline__ Unit unit_of(const SbArgs& g, int u, int nsb)
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

// hi + lo split of s * c for the two f16 integer codes in `cbits` (|c| <= 127), in
// f16x2 arithmetic with s = s_hi + s_lo (two f16 values): hi = rn(s_hi*c); the
// residual s_hi*c - hi is exact in one fma; lo = rn(residual + s_lo*c).  About 21
// significant bits of s*c survive in hi + lo while s_hi >= 2^-14 (|lo| <= 2^-10 |s c|).
__device__ __forceinline__ void split_pair(uint32_t cbits, __half2 s_hi, __half2 s_lo, uint32_t& hi, uint32_t& lo)
{
    const __half2 c = *reinterpret_cast<const __half2*>(&cbits);
    const __half2 h = __hmul2_rn(s_hi, c);
    const __half2 r = __hfma2(s_hi, c, __hneg2(h));
    const __half2 l = __hfma2(s_lo, c, r);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <int TYPE, int TILES>
__device__ __forceinline__ void sb_roles(const SbArgs& g, uint8_t* smem, uint32_t sbase, uint32_t tmem_base,
                                         int warp, int lane)
{
    using L = SbL<TILES>;
    constexpr bool Q4 = (TYPE == 12);
    const int nkb = g.id / TILE_K;
    const int nchunk = g.id / CHUNK;
    const int nsb = g.id / QK_K;
    auto bar = [&](int i) -> uint32_t { return sbase + L::SMEM_BAR + 8u * static_cast<uint32_t>(i); };

    if (warp < CONV_WARP0) {
        regs_shrink<CTRL_REGS>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ producer
            RingPos<L::STAGES> op;
            RingPos<SBR> sb;
            uint32_t n_ops = 0, n_sb = 0;
            // verification only: the fill of this CTA that is left out (never armed,
            // never copied), so that the consumers' wait for it runs out
            const uint32_t skip = (blockIdx.x == 0 && g.withhold >= 0) ? static_cast<uint32_t>(g.withhold) : ~0u;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
                const Unit w = unit_of(g, u, nsb);
                const int m = w.m;
                const int n0 = 2 * w.n;
                const int n1 = (2 * w.n + 1 < g.num_n128) ? 2 * w.n + 1 : n0;  // odd count: repeat (never stored)
                const uint8_t* Ab = g.A + static_cast<size_t>(m) * nkb * TILE_BYTES;
                const uint8_t* B0 = g.B + static_cast<size_t>(n0) * nkb * TILE_BYTES;
                const uint8_t* B1 = g.B + static_cast<size_t>(n1) * nkb * TILE_BYTES;
                const uint8_t* B20 = TILES == 2 ? g.B2 + static_cast<size_t>(n0) * nkb * TILE_BYTES : nullptr;
                const uint8_t* B21 = TILES == 2 ? g.B2 + static_cast<size_t>(n1) * nkb * TILE_BYTES : nullptr;
                const uint8_t* ASb = g.AS + static_cast<size_t>(m) * nchunk * BM * 8;
                if (Q4) {
                    // the tile's min-term operands, consumed after its last k-block
                    const uint32_t mb = static_cast<uint32_t>(w.sb1 - w.sb0) * MIN_AM_BYTES;
                    bulk_prefetch_l2(g.AM + (static_cast<size_t>(m) * nsb + w.sb0) * MIN_AM_BYTES, mb);
                    bulk_prefetch_l2(g.AUX + (static_cast<size_t>(n0) * nsb + w.sb0) * MIN_BM_BYTES, mb);
                    if (n1 != n0)
                        bulk_prefetch_l2(g.AUX + (static_cast<size_t>(n1) * nsb + w.sb0) * MIN_BM_BYTES, mb);
                }
                for (int kb = 4 * w.sb0; kb < 4 * w.sb1; ++kb) {
                    if ((kb & 3) == 0) {
                        const int s = kb >> 2;
                        if (!ctl_wait(g, bar(L::BAR_SBEMPTY + sb.i), sb.ph ^ 1u)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();   // after the consumers' ordinary loads
                        const uint32_t dst = sbase + L::SMEM_SB + sb.i * SB_BYTES;
                        const uint32_t fb = bar(L::BAR_SBFULL + sb.i);
                        mbar_arrive_expect_tx(fb, SB_COPY_BYTES);
                        bulk_g2s(dst + SB_SBD_OFF, g.SBD + (static_cast<size_t>(n0) * nsb + s) * 512, 512, fb);
                        bulk_g2s(dst + SB_SBD_OFF + 512, g.SBD + (static_cast<size_t>(n1) * nsb + s) * 512, 512, fb);
                        bulk_g2s(dst + SB_AS_OFF, ASb + static_cast<size_t>(s) * SB_AS_BYTES, SB_AS_BYTES, fb);
                        sb.next();
                        ++n_sb;
                    }
                    if (!ctl_wait(g, bar(L::BAR_EMPTY + op.i), op.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    if (n_ops == skip) {
                        op.next();
                        ++n_ops;
                        continue;
                    }
                    fence_proxy_async_smem();       // after the converter's ordinary stores
                    const uint32_t st = sbase + L::SMEM_ST + op.i * L::STAGE_BYTES;
                    // the activation tile completes on its own barrier so that the converter
                    // starts while the weight tiles are still in flight
                    const uint32_t fo = bar(L::BAR_FULL + op.i), fw = bar(L::BAR_FULLB + op.i);
                    const size_t ko = static_cast<size_t>(kb) * TILE_BYTES;
                    mbar_arrive_expect_tx(fo, TILE_BYTES);
                    bulk_g2s(st + ST_A, Ab + ko, TILE_BYTES, fo);
                    mbar_arrive_expect_tx(fw, 2 * TILES * TILE_BYTES);
                    bulk_g2s(st + ST_B, B0 + ko, TILE_BYTES, fw);
                    bulk_g2s(st + ST_B + TILE_BYTES, B1 + ko, TILE_BYTES, fw);
                    if (TILES == 2) {
                        bulk_g2s(st + ST_B + 2 * TILE_BYTES, B20 + ko, TILE_BYTES, fw);
                        bulk_g2s(st + ST_B + 3 * TILE_BYTES, B21 + ko, TILE_BYTES, fw);
                    }
                    if (kb + L::STAGES < 4 * w.sb1) {
                        // warm L2 with the tiles of the k-block this stage takes next
                        // (measured: about 3.5 % off the launch)
                        const size_t kp = static_cast<size_t>(kb + L::STAGES) * TILE_BYTES;
                        bulk_prefetch_l2(B0 + kp, TILE_BYTES);
                        bulk_prefetch_l2(B1 + kp, TILE_BYTES);
                        if (TILES == 2) {
                            bulk_prefetch_l2(B20 + kp, TILE_BYTES);
                            bulk_prefetch_l2(B21 + kp, TILE_BYTES);
                        }
                        bulk_prefetch_l2(Ab + kp, TILE_BYTES);
                    }
                    op.next();
                    ++n_ops;
                }
                if (Q4 && ok) {
                    // MIN_PER_STAGE super-blocks per stage: token tiles of super-block
                    // s + e at ST_A + e * 8 KiB, weight tiles [hi n0 | hi n1 | lo n0 | lo n1]
                    // at ST_B + e * 16 KiB
                    for (int s = w.sb0; s < w.sb1; s += MIN_PER_STAGE) {
                        const int ne = min(MIN_PER_STAGE, w.sb1 - s);
                        if (!ctl_wait(g, bar(L::BAR_EMPTY + op.i), op.ph ^ 1u)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_smem();
                        const uint32_t st = sbase + L::SMEM_ST + op.i * L::STAGE_BYTES;
                        const uint32_t fo = bar(L::BAR_FULL + op.i), fw = bar(L::BAR_FULLB + op.i);
                        mbar_arrive_expect_tx(fo, ne * MIN_AM_BYTES);
                        bulk_g2s(st + ST_A, g.AM + (static_cast<size_t>(m) * nsb + s) * MIN_AM_BYTES,
                                 ne * MIN_AM_BYTES, fo);
                        mbar_arrive_expect_tx(fw, ne * 2 * MIN_BM_BYTES);
                        for (int e = 0; e < ne; ++e) {
                            const uint8_t* x0 = g.AUX + (static_cast<size_t>(n0) * nsb + s + e) * MIN_BM_BYTES;
                            const uint8_t* x1 = g.AUX + (static_cast<size_t>(n1) * nsb + s + e) * MIN_BM_BYTES;
                            const uint32_t bb = st + ST_B + e * 2 * MIN_BM_BYTES;
                            bulk_g2s(bb, x0, TF32_TILE_BYTES, fw);
                            bulk_g2s(bb + TF32_TILE_BYTES, x1, TF32_TILE_BYTES, fw);
                            bulk_g2s(bb + 2 * TF32_TILE_BYTES, x0 + TF32_TILE_BYTES, TF32_TILE_BYTES, fw);
                            bulk_g2s(bb + 3 * TF32_TILE_BYTES, x1 + TF32_TILE_BYTES, TF32_TILE_BYTES, fw);
                        }
                        op.next();
                        ++n_ops;
                    }
                }
            }
            for (uint32_t i = (n_ops > L::STAGES ? n_ops - L::STAGES : 0); i < n_ops; ++i) {
                if (i == skip)
                    continue;
                drain_wait(g, bar(L::BAR_FULL + i % L::STAGES), (i / L::STAGES) & 1u);
                drain_wait(g, bar(L::BAR_FULLB + i % L::STAGES), (i / L::STAGES) & 1u);
            }
            for (uint32_t i = (n_sb > SBR ? n_sb - SBR : 0); i < n_sb; ++i)
                drain_wait(g, bar(L::BAR_SBFULL + i % SBR), (i / SBR) & 1u);
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            constexpr uint32_t idesc_t = idesc_tf32(BM, BN);
            RingPos<L::STAGES> op;
            RingPos<2> item;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
                const Unit w = unit_of(g, u, nsb);
                for (int kb = 4 * w.sb0; kb < 4 * w.sb1; ++kb) {
                    const int k2 = kb & 3;
                    if (k2 == 0 && !ctl_wait(g, bar(L::BAR_TEMPTY + item.i), item.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    if (!ctl_wait(g, bar(L::BAR_CONV + op.i), op.ph) || !ctl_wait(g, bar(L::BAR_FULLB + op.i), op.ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = sbase + L::SMEM_ST + op.i * L::STAGE_BYTES;
                    const uint64_t ah = sdesc_k_sw128(st + ST_A);
                    const uint64_t al = sdesc_k_sw128(st + ST_LO);
                    const uint64_t b = sdesc_k_sw128(st + ST_B);
                    const uint64_t b2 = sdesc_k_sw128(st + ST_B + 2 * TILE_BYTES);
                    const uint32_t d = tmem_base + item.i * ITEM_COLS;
                    // 16 values per step: +32 bytes (two 16-byte units) inside the swizzled rows
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        umma_f16(d, ah + 2u * kk, b + 2u * kk, idesc, (k2 | kk) ? 1u : 0u);
                        umma_f16(d, al + 2u * kk, b + 2u * kk, idesc, 1u);
                        if (TILES == 2) {   // the second exact tile: sc*l + 16 sc (h - 2) = sc*q
                            umma_f16(d, ah + 2u * kk, b2 + 2u * kk, idesc, 1u);
                            umma_f16(d, al + 2u * kk, b2 + 2u * kk, idesc, 1u);
                        }
                    }
                    umma_commit(bar(L::BAR_EMPTY + op.i));
                    op.next();
                    if (k2 == 3) {
                        umma_commit(bar(L::BAR_TFULL + item.i));
                        item.next();
                    }
                }
                for (int g0 = w.sb0; Q4 && ok && g0 < w.sb1; g0 += MIN_GROUP_SB) {
                    const int g1 = min(g0 + MIN_GROUP_SB, w.sb1);
                    if (!ctl_wait(g, bar(L::BAR_TEMPTY + item.i), item.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t d = tmem_base + item.i * ITEM_COLS;
                    for (int s = g0; s < g1; s += MIN_PER_STAGE) {
                        const int ne = min(MIN_PER_STAGE, g1 - s);
                        if (!ctl_wait(g, bar(L::BAR_CONV + op.i), op.ph) || !ctl_wait(g, bar(L::BAR_FULLB + op.i), op.ph)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = sbase + L::SMEM_ST + op.i * L::STAGE_BYTES;
                        for (int e = 0; e < ne; ++e) {
                            const uint32_t aa = st + ST_A + e * MIN_AM_BYTES;
                            const uint32_t bb = st + ST_B + e * 2 * MIN_BM_BYTES;
                            const uint64_t ahi = sdesc_tf32(aa), alo = sdesc_tf32(aa + TF32_TILE_BYTES);
                            const uint64_t bhi = sdesc_tf32(bb), blo = sdesc_tf32(bb + 2 * TF32_TILE_BYTES);
                            mma_tf32(d, ahi, bhi, idesc_t, (s + e > g0) ? 1u : 0u);
                            mma_tf32(d, ahi, blo, idesc_t, 1u);
                            mma_tf32(d, alo, bhi, idesc_t, 1u);
                        }
                        umma_commit(bar(L::BAR_EMPTY + op.i));
                        op.next();
                    }
                    if (!ok)
                        break;
                    umma_commit(bar(L::BAR_TFULL + item.i));
                    item.next();
                }
            }
            umma_commit(bar(L::BAR_DRAIN));
            drain_wait(g, bar(L::BAR_DRAIN), 0u);
        }
        __syncwarp();
        return;
    }

    if (warp < PROMO_WARP0) {
        // ---------------------------------------------------------------- converter
        regs_shrink<CONV_REGS>();
        const int r = (warp - CONV_WARP0) * 32 + lane;    // token row of the tile
        const uint32_t row_off = static_cast<uint32_t>(r) * 128u;
        const uint32_t sw = static_cast<uint32_t>(r & 7);
        RingPos<L::STAGES> op;
        RingPos<SBR> sb;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
            const Unit w = unit_of(g, u, nsb);
            for (int s = w.sb0; ok && s < w.sb1; ++s) {
                if (!warp_wait(g, bar(L::BAR_SBFULL + sb.i), sb.ph)) {
                    ok = false;
                    break;
                }
                const uint2* pr = reinterpret_cast<const uint2*>(smem + L::SMEM_SB + sb.i * SB_BYTES + SB_AS_OFF);
                float da[8];
                float dmax = 0.0f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    da[k] = __uint_as_float(pr[k * BM + r].x);
                    dmax = fmaxf(dmax, da[k]);
                }
                const uint32_t pf = p_field(dmax);
                const float p = __uint_as_float(pf << 23);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    da[k] *= p;                   // s = d_a * p, exact
                // 1/p (exact) for the promotion warps
                reinterpret_cast<float*>(smem + L::SMEM_SB + sb.i * SB_BYTES + SB_IP_OFF)[r] =
                    __uint_as_float((254u - pf) << 23);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(L::BAR_IPREADY + sb.i));
                    mbar_arrive(bar(L::BAR_SBEMPTY + sb.i));
                }
                sb.next();
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    if (!warp_wait(g, bar(L::BAR_FULL + op.i), op.ph)) {
                        ok = false;
                        break;
                    }
                    // s of the k-block's two chunks as f16 pairs s_hi + s_lo
                    __half2 shi[2], slo[2];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const float sk = da[2 * k2 + cc];
                        const __half hh = __float2half_rn(sk);
                        shi[cc] = __half2half2(hh);
                        slo[cc] = __half2half2(__float2half_rn(sk - __half2float(hh)));
                    }
                    uint8_t* st = smem + L::SMEM_ST + op.i * L::STAGE_BYTES;
                    // all eight 16-byte groups of the row first (one shared-memory
                    // latency per k-block), then convert and store
                    uint4 c[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)         // logical group j = values 8j..8j+7
                        c[j] = *reinterpret_cast<const uint4*>(st + ST_A + row_off + ((static_cast<uint32_t>(j) ^ sw) << 4));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t off = row_off + ((static_cast<uint32_t>(j) ^ sw) << 4);
                        const int k = j >> 2;              // chunk of the k-block
                        uint4 h, l;
                        split_pair(c[j].x, shi[k], slo[k], h.x, l.x);
                        split_pair(c[j].y, shi[k], slo[k], h.y, l.y);
                        split_pair(c[j].z, shi[k], slo[k], h.z, l.z);
                        split_pair(c[j].w, shi[k], slo[k], h.w, l.w);
                        *reinterpret_cast<uint4*>(st + ST_A + off) = h;
                        *reinterpret_cast<uint4*>(st + ST_LO + off) = l;
                    }
                    fence_proxy_async_smem();           // ordinary stores -> tensor-core reads
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar(L::BAR_CONV + op.i));
                    op.next();
                }
            }
            if (Q4 && ok) {
                // min-term stages pass through unchanged
                for (int s = w.sb0; s < w.sb1; s += MIN_PER_STAGE) {
                    if (!warp_wait(g, bar(L::BAR_FULL + op.i), op.ph)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar(L::BAR_CONV + op.i));
                    op.next();
                }
            }
        }
        return;
    }

    // -------------------------------------------------------------------- promotion
    // TMEM is read with the 16x256b shape, so that the four threads of a quad hold
    // eight consecutive columns of one row: each thread owns rows
    // q*32 + 16h + 8rho + quad (h, rho in {0, 1}) and, of the warp's 128 columns,
    // 8n + 2*qi + {0, 1} (n = 0..15), and a warp's Y stores write whole 32-byte
    // sectors of 8 rows.
    regs_grow<PROMO_REGS>();
    const int pw = warp - PROMO_WARP0;                  // 0..7
    const int q = warp & 3;                              // TMEM lane quarter
    const int hc = pw >> 2;                              // which 128 of the 256 columns
    const int quad = lane >> 2, qi = lane & 3;
    const uint32_t qaddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + hc * COLS_PER_WARP;
    RingPos<2> item;
    RingPos<SBR> sb;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
        const Unit w = unit_of(g, u, nsb);
        float2 acc[2][2][16];     // [h][rho][n]
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int rho = 0; rho < 2; ++rho)
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    acc[h][rho][n] = make_float2(0.0f, 0.0f);
        // One item per super-block: acc += d_sb * (D / p); for q4_K one more item per
        // MIN_GROUP_SB super-blocks of the tile, the min term, taken with d = 1 and
        // 1/p = -1 (acc -= min term).
        const int s_end = Q4 ? w.sb1 + (w.sb1 - w.sb0 + MIN_GROUP_SB - 1) / MIN_GROUP_SB : w.sb1;
        for (int s = w.sb0; s < s_end; ++s) {
            const bool min_item = Q4 && s >= w.sb1;
            float ip[2][2] = {{-1.0f, -1.0f}, {-1.0f, -1.0f}};
            const float2* d2 = nullptr;
            if (!min_item) {
                if (!warp_wait(g, bar(L::BAR_SBFULL + sb.i), sb.ph) || !warp_wait(g, bar(L::BAR_IPREADY + sb.i), sb.ph)) {
                    ok = false;
                    break;
                }
                const uint8_t* sbe = smem + L::SMEM_SB + sb.i * SB_BYTES;
                const float* ipr = reinterpret_cast<const float*>(sbe + SB_IP_OFF);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int rho = 0; rho < 2; ++rho)
                        ip[h][rho] = ipr[q * 32 + 16 * h + 8 * rho + quad];
                d2 = reinterpret_cast<const float2*>(sbe + SB_SBD_OFF) + hc * (COLS_PER_WARP / 2) + qi;
            }
            if (!warp_wait(g, bar(L::BAR_TFULL + item.i), item.ph)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t col0 = qaddr + item.i * ITEM_COLS;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int gq = 0; gq < 2; ++gq) {
                    float D[32];
                    tmem_ld16x256b_x8_wait(col0 + (static_cast<uint32_t>(16 * h) << 16) + 64 * gq, D);
                    if (h == 1 && gq == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(bar(L::BAR_TEMPTY + item.i));
                        item.next();
                    }
#pragma unroll
                    for (int n2 = 0; n2 < 8; ++n2) {
                        const int n = 8 * gq + n2;
                        const float2 dv = min_item ? make_float2(1.0f, 1.0f) : d2[4 * n];
#pragma unroll
                        for (int rho = 0; rho < 2; ++rho) {
                            const float2 u2 = ffma2(make_float2(ip[h][rho], ip[h][rho]),
                                                    make_float2(D[4 * n2 + 2 * rho], D[4 * n2 + 2 * rho + 1]),
                                                    make_float2(0.0f, 0.0f));
                            acc[h][rho][n] = ffma2(dv, u2, acc[h][rho][n]);
                        }
                    }
                }
            }
            if (!min_item) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(L::BAR_SBEMPTY + sb.i));
                sb.next();
            }
        }
        if (!ok)
            break;
        const int jb = w.n * BN + hc * COLS_PER_WARP + 2 * qi;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int rho = 0; rho < 2; ++rho) {
                const int row = w.m * BM + q * 32 + 16 * h + 8 * rho + quad;
                if (row >= g.M)
                    continue;
                float* yrow = g.Y + static_cast<size_t>(row) * g.ldy;
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    const int j = jb + 8 * n;
                    const float2 v = acc[h][rho][n];
                    if (g.vec_store && j + 1 < g.od) {
                        if (w.half)
                            asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(yrow + j), "f"(v.x), "f"(v.y)
                                         : "memory");
                        else
                            *reinterpret_cast<float2*>(yrow + j) = v;
                    } else {
                        if (j < g.od) {
                            if (w.half)
                                atomicAdd(yrow + j, v.x);
                            else
                                yrow[j] = v.x;
                        }
                        if (j + 1 < g.od) {
                            if (w.half)
                                atomicAdd(yrow + j + 1, v.y);
                            else
                                yrow[j + 1] = v.y;
                        }
                    }
                }
            }
    }
}

// Barrier set-up, TMEM, the roles, TMEM release, for one shared-memory plan.
template <int TYPE, int TILES>
__device__ __forceinline__ void sb_body(const SbArgs& g, uint8_t* smem, uint32_t sbase, int warp, int lane)
{
    using L = SbL<TILES>;
    auto bar = [&](int i) -> uint32_t { return sbase + L::SMEM_BAR + 8u * static_cast<uint32_t>(i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(bar(L::BAR_FULL + s), 1);
            mbar_init(bar(L::BAR_FULLB + s), 1);
            mbar_init(bar(L::BAR_CONV + s), NUM_CONV_WARPS);
            mbar_init(bar(L::BAR_EMPTY + s), 1);
        }
        for (int s = 0; s < SBR; ++s) {
            mbar_init(bar(L::BAR_SBFULL + s), 1);
            mbar_init(bar(L::BAR_SBEMPTY + s), NUM_CONV_WARPS + NUM_PROMO_WARPS);
            mbar_init(bar(L::BAR_IPREADY + s), NUM_CONV_WARPS);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(bar(L::BAR_TFULL + k), 1);
            mbar_init(bar(L::BAR_TEMPTY + k), NUM_PROMO_WARPS);
        }
        mbar_init(bar(L::BAR_DRAIN), 1);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::SMEM_TMEMPTR, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + L::SMEM_TMEMPTR);

    // A dependent launch: the set-up above may overlap the kernel ahead on the stream (the
    // prepass that writes the activation planes, or a kernel still reading Y); nothing is
    // read or written in global memory before it has completed.  The next kernel may be
    // scheduled as this grid's CTAs finish.
    grid_dep_wait();
    grid_dep_launch();
    sb_roles<TYPE, TILES>(g, smem, sbase, tmem_base, warp, lane);

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int TYPE>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_sb_kernel(const SbArgs g)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if constexpr (TYPE == 14) {
        // q6_K codes hold sc*q in one tile unless some |sc| > 64 (then two exact tiles);
        // the repack recorded which in the flag word (uniform for the launch).  The flag
        // is read only once the kernel ahead, which may be the repack, has completed.
        grid_dep_wait();
        if (__ldg(g.FLAG) != 0u)
            sb_body<14, 1>(g, smem, sbase, warp, lane);
        else
            sb_body<14, 2>(g, smem, sbase, warp, lane);
    } else {
        sb_body<12, 1>(g, smem, sbase, warp, lane);
    }
}

constexpr int ZERO_ROWS = 16;   // rows of Y a zeroing block clears

// Zeroes Y over the 128 x 256 tiles [first, first + count) (rows < M, columns < od).
__global__ void __launch_bounds__(256) sb_zero_tiles_kernel(float* __restrict__ Y, int ldy, int M, int od, int num_m,
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

template <int TYPE>
cudaError_t launch_sb_typed(const SbArgs& a, int grid, cudaStream_t s)
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
        e = cudaFuncGetAttributes(&fa, gemm_sb_kernel<TYPE>);
        if (e != cudaSuccess)
            return e;
        if (fa.numRegs < LAUNCH_REGS)
            return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(gemm_sb_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess)
            return e;
        attr_set_mask.fetch_or(bit);
    }
    count_launch();
    return launch_dependent_smem(gemm_sb_kernel<TYPE>, dim3(static_cast<unsigned>(grid)), dim3(NUM_THREADS),
                                 static_cast<size_t>(SMEM_ALLOC), s, a);
}

}  // namespace

cudaError_t launch_gemm_sb(int type, const void* packed, int od, int id, const void* qa, const void* scales, int M,
                           float* Y, int ldy, cudaStream_t s, const WaitCtl& wc)
{
    const WeightPlanes wp = weight_planes(type, od, id);
    const ActPlanes ap = act_planes(M, id);
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    const uint8_t* sc = static_cast<const uint8_t*>(scales);
    SbArgs a;
    a.A = static_cast<const uint8_t*>(qa);
    a.AS = sc + ap.pair_off;
    a.AM = sc + ap.am_off;
    a.B = pk + wp.code_off;
    a.B2 = pk + wp.code2_off;
    a.SBD = pk + wp.sbd_off;
    a.AUX = pk + wp.aux_off;
    a.FLAG = reinterpret_cast<const unsigned int*>(pk + wp.flag_off);
    a.Y = Y;
    a.ldy = ldy;
    a.M = M;
    a.od = od;
    a.id = id;
    a.num_m = ceil_div(M, BM);
    a.num_n = ceil_div(od, BN);
    a.num_n128 = ceil_div(od, TILE_ROWS);
    a.vec_store = ((reinterpret_cast<uintptr_t>(Y) & 7u) == 0 && (ldy & 1) == 0) ? 1 : 0;
    a.err = wc.err;
    a.wait_ns = wc.limit_ns;
    a.withhold = wc.withhold_fill;

    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    const int tiles = a.num_m * a.num_n;
    int grid = tiles < nsm ? tiles : nsm;
    a.units = tiles;
    a.full_units = tiles;
    a.nsb_half = 0;
    const int rem = tiles % grid;
    const int nsb = id / QK_K;
    // two K-halves added into a zeroed Y: every tile when there are at most half as
    // many tiles as SMs, else the last round's tiles when they fill at most half
    int split = 0;
    if (nsb >= 2) {
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
        e = launch_dependent(sb_zero_tiles_kernel, dim3(static_cast<unsigned>(split), BM / ZERO_ROWS), dim3(256), s, Y,
                             ldy, M, od, a.num_m, a.full_units);
        if (e != cudaSuccess)
            return e;
    }
    return type == 14 ? launch_sb_typed<14>(a, grid, s) : launch_sb_typed<12>(a, grid, s);
}

}  // namespace mmq
