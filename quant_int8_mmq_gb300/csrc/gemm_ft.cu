// gemm_ft.cu -- few-token q4_K / q6_K x q8 GEMM for sm_103a (1 <= M <= 64 tokens):
// the decode and prompt-tail shapes, where the weights are read once and their
// stream from HBM is the whole cost.
//
// What it computes is the formula of the super-block kernel (gemm_sb.cu) with the
// operands swapped, so that the weight rows fill the 128 TMEM lanes and the tokens are
// the MMA's N (16 * ceil(M/16) columns):
//
//   D[j,t] = sum_{k in stage} W[j,k] * (hi[t,k] + lo[t,k])      (tcgen05 kind::f16, f32 TMEM)
//   Y[t,j] = sum_sb d_sb[j] * (sum of the super-block's stage D[j,t]) * (1/p[t,sb])
//            -  sum_sb sum_c dmin_sb[j] * m_c[j] * (d_a*ssum)[t,c]            (q4_K)
//
// hi + lo = p * d_a * q_a is the activation operand the prepass writes for few tokens
// (about 21 significant bits per value, p a power of two per token and super-block);
// W is the integer-scaled weight code, exact in f16:
//   q4_K: W = sc_c * q                           (|W| <= 945, one tile)
//   q6_K whose every |sc| <= 64 (the packed flag says so):
//         W = sc * q                             (|W| <= 2048, one tile, one fma from
//         1024 + 4 (q + 32))
//   q6_K otherwise:
//         W = (sc * l) / 4  +  4 * sc * (h - 2)  (two tiles, l and h the low 4 and high 2
//         bits of q + 32; sc * l / 4 is a quarter-integer
//         below 480 in magnitude and 4 sc (h - 2) an integer of at most 1024, both exact
//         for any int8 sc), so the sum of the two tiles is sc * q / 4 and the promotion
//         uses 4/p.
// Every product W * hi, W * lo is exact; the roundings are the split of the activation
// operand, the f32 sums and the promotion (the 1e-5 bound on Y holds with margin).  The
// q4_K min term is a contraction over only 8 chunks per super-block: the promotion
// threads take it on the CUDA cores, two tokens per f32x2 FMA against the chunk-major
// d_a*ssum values the prepass wrote (a tf32 hi/lo tensor-core form, as in the
// super-block kernel, was slower here once the FMAs were paired).
//
// The weights come from the compact code plane (0.5 B per value for q4_K, 1 for q6_K:
// one byte 4 (q + 32), which a mask alone puts under the exponent) and are widened to
// f16 by converter warps, the unpacking of "r56 - q6_K A-side
// bundle ..." §1 / "r58 - q4_K BT spec ..." §3.2 done in the GEMM instead of at
// registration.  Each f16 pair comes from one 32-bit word with a mask, an OR of the
// exponent of 1024 (0x6400, so the field lands in the mantissa: 1024 + field) and one
// f16x2 fma or add/multiply that removes the 1024 and applies the integer scale; no
// value is ever inexact.  The widened tiles go straight from registers to tensor
// memory (tcgen05.st), where the MMA reads its A operand; only the compact codes and
// the tokens pass through shared memory.
//
// At these N an MMA costs the issuing thread a fixed ~50 ns whatever its width, and
// MMAs from different threads into different accumulators overlap on the tensor
// pipe, so two warps issue: stage g (a super-block, or for two-tile q6_K half of one)
// goes to issuer g % 2, into its own accumulator item; the promotion adds the items
// of a super-block.  A stage is large because each mbarrier hand-off between roles
// costs a few hundred cycles whatever the stage carries: 128 TMEM columns of widened
// weights (double-buffered), the tokens of a whole super-block in one bulk copy, and
// one MMA covering the hi and the lo rows of the tokens.
//
// One CTA per SM, persistent over 128-row weight tiles (or, when the tiles are few,
// one cluster of S CTAs per tile along K whose partial sums meet in rank 0 through
// distributed shared memory, in rank order); 16 warps:
//   warp 0       producer: compact codes of each stage into a ring (bulk copies, L2
//                prefetch four stages ahead) and once per super-block the weight d, the
//                sub-block scales, the tokens' 1/p and (q4_K) the weight dmin and the
//                tokens' d_a*ssum into a ring.
//   warp 1       allocates TMEM (accumulator items in columns [0, 256), two weight
//                buffers of 128 columns), then issues the odd stages.
//   warp 2       producer: the tokens' hi and lo tiles of each super-block into a 2-deep
//                ring.
//   warp 3       issues the even stages: 128 x 2N x 16 MMAs (A = weights from TMEM, B =
//                the N hi and N lo token rows from shared memory in one operand).
//   warps 4-11   converters: thread (row r, half h of the stage) widens its values into
//                the weight buffer and the warp signals the issuers.
//   warps 12-15  promotion: thread = weight row (its TMEM lane), every token: per
//                super-block its stage items' TMEM loads, acc += d * (D * 1/p), and for
//                q4_K acc -= dmin * sum_c m_c * (d_a*ssum)_c; store Y.
//
// Every mbarrier wait is bounded; on expiry the kernel sets the library's error word,
// every role leaves its loop, waits (bounded) for its own copies and MMAs in flight,
// and the CTA frees TMEM and exits.
#include <cuda_fp16.h>

#include <atomic>

#include "mmq_internal.h"
#include "ptx.cuh"

namespace mmq {
namespace {

constexpr int BM = 128;                 // weight rows per tile (MMA M, TMEM lanes)
constexpr int NUM_WARPS = 16;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int CONV_WARP0 = 4;
constexpr int NUM_CONV_WARPS = 8;
constexpr int PROMO_WARP0 = 12;
// Register split for q4_K at 49 to 64 tokens (N = 64), whose promotion threads hold 64
// accumulators and spilled at 128 registers: the control warpgroup gives up registers to
// the promotion warpgroup out of the launch's 128 x 512 (converters keep 128).  Measured on
// GB300: q4_K 11008x4096 M = 56 29.1 -> 24.3 us, 4096x4096 15.8 -> 14.2 us; at N = 48 and
// for q6_K (whose converters keep their spills) it changed nothing or cost 1 %, so those
// keep the uniform 128.  The host launches a split build only if it compiled to 128
// registers per thread, the sum the split assumes.
constexpr int LAUNCH_REGS = 128;
constexpr int CTRL_REGS = 56;
constexpr int CONV_REGS = 128;
constexpr int PROMO_REGS = 200;
static_assert(4 * 32 * CTRL_REGS + 8 * 32 * CONV_REGS + 4 * 32 * PROMO_REGS == LAUNCH_REGS * 512, "register split");
constexpr int NUM_PROMO_WARPS = 4;
constexpr int NUM_ISSUERS = 2;          // warp 3: even stages, warp 1: odd stages
constexpr int PF_STAGES = 4;            // L2 prefetch distance of the compact codes, stages
constexpr int TOK_STAGES = 2;           // token ring depth (super-blocks)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t WBUF_COL0 = 256;     // accumulator items in columns [0, 256), then the two weight buffers
constexpr uint32_t WBUF_COLS = 128;
constexpr int MAX_CLUSTER = 8;
static_assert(MAX_CLUSTER * NUM_PROMO_WARPS <= 32, "one lane per rank flag");
constexpr int SMEM_BUDGET = 227 * 1024 - 2048;   // rings; the rest: barriers, TMEM address, alignment slack
static_assert(WBUF_COL0 + 2 * WBUF_COLS <= TMEM_COLS, "TMEM budget");
// Accumulator items: one MMA covers the hi and the lo token rows (N = 2 x 16*NT columns:
// W*hi in the first half, W*lo in the second), 64 or 128 columns per item.
__host__ __device__ constexpr int items_of(int nt) { return nt <= 2 ? 4 : 2; }
__host__ __device__ constexpr uint32_t item_cols_of(int nt) { return nt <= 2 ? 64u : 128u; }
// K split of the most recent launch from this thread (for its path label).
thread_local int g_last_kslices = 1;

// Super-block ring entry: weight d of the 128 rows, their 16 sub-block scale bytes, 1/p
// of the FT_MAX_M tokens, and for q4_K the rows' dmin and the tokens' 8 values d_a*ssum
// per chunk ([chunk][FT_MAX_M tokens]).
constexpr int SB_SBD_OFF = 0;
constexpr int SB_SC_OFF = SB_SBD_OFF + BM * 4;
constexpr int SB_IP_OFF = SB_SC_OFF + BM * SC_ROW_BYTES;
constexpr int SB_DM_OFF = SB_IP_OFF + FT_MAX_M * 4;
constexpr int SB_FM_OFF = SB_DM_OFF + BM * 4;
__host__ __device__ constexpr int sb_bytes_of(int type) { return type == 12 ? SB_FM_OFF + FT_MAX_M * 32 : SB_DM_OFF; }

// ONE: one weight tile per k-block (q4_K always; q6_K when its codes fold); else two.
template <int TYPE, int NT, bool ONE>
struct Cfg {
    static constexpr int N = 16 * NT;
    static constexpr int TILES = ONE ? 1 : 2;
    static constexpr int ITEMS = items_of(NT);
    static constexpr bool SPLIT_REGS = TYPE == 12 && NT == 4;
    static constexpr uint32_t ITEM_COLS = item_cols_of(NT);
    static_assert(ITEMS * ITEM_COLS == WBUF_COL0 && 2 * N <= static_cast<int>(ITEM_COLS), "items");
    static_assert(TYPE == 14 || ONE, "q4_K has one tile");
    static constexpr int KPS = ONE ? 4 : 2;                          // k-blocks per stage
    static constexpr int SPS = 4 / KPS;                              // stages per super-block
    static_assert(KPS * 32 * TILES == static_cast<int>(WBUF_COLS), "a stage fills one weight buffer");
    static constexpr int RAW_BYTES = KPS * cw_kblock_bytes(TYPE);    // compact codes of a stage
    static constexpr int TOK_KB_BYTES = 2 * N * 128;                 // hi rows, lo rows of a k-block
    static constexpr int TOK_SLOT = 4 * TOK_KB_BYTES;                // a super-block of tokens
    static constexpr int SB_BYTES = sb_bytes_of(TYPE);
    static constexpr int SBR = TYPE == 12 ? 6 : 8;                   // super-block ring depth
    static constexpr int FIXED = TOK_STAGES * TOK_SLOT + SBR * SB_BYTES;
    static constexpr int RAW_FIT = (SMEM_BUDGET - FIXED) / RAW_BYTES;
    static constexpr int RAW_STAGES = RAW_FIT > 4 ? 4 : RAW_FIT;     // compact-code ring depth
    static_assert(RAW_STAGES >= 2, "shared memory budget");
    static constexpr int SMEM_TOK = 0;
    static constexpr int SMEM_RAW = SMEM_TOK + TOK_STAGES * TOK_SLOT;
    static constexpr int SMEM_SB = SMEM_RAW + RAW_STAGES * RAW_BYTES;
    static constexpr int SMEM_BAR = SMEM_SB + SBR * SB_BYTES;
    static constexpr int BAR_RFULL = 0;
    static constexpr int BAR_REMPTY = BAR_RFULL + RAW_STAGES;
    static constexpr int BAR_TKFULL = BAR_REMPTY + RAW_STAGES;
    static constexpr int BAR_TKEMPTY = BAR_TKFULL + TOK_STAGES;
    static constexpr int BAR_AEMPTY = BAR_TKEMPTY + TOK_STAGES;
    static constexpr int BAR_WCONV = BAR_AEMPTY + 2;
    static constexpr int BAR_SBFULL = BAR_WCONV + 2;
    static constexpr int BAR_SBEMPTY = BAR_SBFULL + SBR;
    static constexpr int BAR_TFULL = BAR_SBEMPTY + SBR;
    static constexpr int BAR_TEMPTY = BAR_TFULL + ITEMS;
    static constexpr int BAR_DRAIN = BAR_TEMPTY + ITEMS;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr int SMEM_TMEMPTR = SMEM_BAR + NUM_BARS * 8;
    static constexpr int SMEM_ALLOC = SMEM_TMEMPTR + 16 + 1024;      // slack for 1024-byte alignment
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(TOK_SLOT % 1024 == 0 && TOK_KB_BYTES % 1024 == 0 && SMEM_RAW % 16 == 0 &&
                      RAW_BYTES % 16 == 0 && SMEM_SB % 16 == 0 && SB_BYTES % 16 == 0 && SMEM_BAR % 8 == 0,
                  "alignment");
    // cluster K split: partial sums (rows x FT_MAX_M tokens) and the promotion warps' ok
    // flags, in the idle token and compact rings
    static constexpr int OKF_OFF = BM * FT_MAX_M * 4;
    static_assert(OKF_OFF + NUM_PROMO_WARPS * 4 <= SMEM_SB, "partial sums fit the idle rings");
};

// Dynamic shared memory of a launch: the larger of the q6_K layouts (the kernel picks
// one from the packed flag).
template <int TYPE, int NT>
constexpr int smem_alloc_of()
{
    return TYPE == 12 ? Cfg<12, NT, true>::SMEM_ALLOC
                      : (Cfg<14, NT, true>::SMEM_ALLOC > Cfg<14, NT, false>::SMEM_ALLOC ? Cfg<14, NT, true>::SMEM_ALLOC
                                                                                       : Cfg<14, NT, false>::SMEM_ALLOC);
}

struct FtArgs {
    const uint8_t* CW;    // compact codes        [num_n][nkb][words][128][16 B]
    const uint8_t* SC;    // sub-block scales     [num_n][nsb][128][16 B]
    const uint8_t* SBD;   // weight d             [num_n][nsb][128] f32
    const uint8_t* DM;    // q4_K weight dmin     [num_n][nsb][128] f32
    const unsigned int* FLAG;   // q6_K: word 0 = 1 if every |sc| <= 64
    const uint8_t* TQ;    // token hi/lo tiles    [nkb][hi n_tok rows | lo n_tok rows][128 B]
    const uint8_t* IP;    // token 1/p            [nsb][FT_MAX_M] f32
    const uint8_t* FM;    // token d_a*ssum       [nsb][8][FT_MAX_M] f32
    float* Y;
    int ldy;
    int M, od, id;
    int n_tok;
    int num_n;            // 128-row weight tiles
    int units;            // num_n * kslices
    int kslices;          // CTAs per tile along K (a cluster), 1 = none
    unsigned int* err;
    unsigned long long wait_ns;
    int withhold;         // verification: compact fill CTA 0's producer leaves out (-1: none)
};

struct Unit {
    int n, sb0, sb1;
};
__device__ __forceinline__ Unit unit_of(const FtArgs& g, int u, int nsb)
{
    Unit w;
    const int r = u % g.kslices;
    w.n = u / g.kslices;
    w.sb0 = r * nsb / g.kslices;
    w.sb1 = (r + 1) * nsb / g.kslices;
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

__device__ __forceinline__ bool ctl_wait(const FtArgs& g, uint32_t bar, uint32_t parity)
{
    return mbar_wait(bar, parity, g.wait_ns, g.err);
}
__device__ __forceinline__ bool warp_wait(const FtArgs& g, uint32_t bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, g.wait_ns, g.err));
}
__device__ __forceinline__ void drain_wait(const FtArgs& g, uint32_t bar, uint32_t parity)
{
    mbar_drain_wait(bar, parity, WAIT_LIMIT_NS, g.err);
}

__device__ __forceinline__ uint32_t lop_or(uint32_t x, uint32_t mask)   // (x & mask) | 0x64006400
{
    return (x & mask) | 0x64006400u;
}
__device__ __forceinline__ uint32_t h2u(__half2 v) { return *reinterpret_cast<const uint32_t*>(&v); }
// Pairs of f32 as one f32x2 instruction each (two IEEE operations, each rounded as its
// scalar form): (x, y) = (a, b) + (c, d); (x, y) = (a, b) * (c, d); and below
// (x, y) = fma(m, (fx, fy), (x, y)).
__device__ __forceinline__ void fadd2(float& x, float& y, float a, float b, float c, float d)
{
    asm("{\n\t.reg .b64 p, q;\n\t"
        "mov.b64 p, {%2, %3};\n\t"
        "mov.b64 q, {%4, %5};\n\t"
        "add.rn.f32x2 p, p, q;\n\t"
        "mov.b64 {%0, %1}, p;\n\t}"
        : "=f"(x), "=f"(y)
        : "f"(a), "f"(b), "f"(c), "f"(d));
}
__device__ __forceinline__ void fmul2(float& x, float& y, float a, float b, float c, float d)
{
    asm("{\n\t.reg .b64 p, q;\n\t"
        "mov.b64 p, {%2, %3};\n\t"
        "mov.b64 q, {%4, %5};\n\t"
        "mul.rn.f32x2 p, p, q;\n\t"
        "mov.b64 {%0, %1}, p;\n\t}"
        : "=f"(x), "=f"(y)
        : "f"(a), "f"(b), "f"(c), "f"(d));
}
__device__ __forceinline__ void ffma2(float& x, float& y, float m, float fx, float fy)
{
    asm("{\n\t.reg .b64 a, b, c;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 b, {%2, %2};\n\t"
        "mov.b64 c, {%3, %4};\n\t"
        "fma.rn.f32x2 a, b, c, a;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "+f"(x), "+f"(y)
        : "f"(m), "f"(fx), "f"(fy));
}
__device__ __forceinline__ __half2 u2h(uint32_t v) { return *reinterpret_cast<const __half2*>(&v); }

// q4_K: the 8 codes of one unit (nibble word x) times sc as four f16 pairs.  Fields at
// bits 0-3 give 1024 + q, fields at bits 4-7 give 1024 + 16 q; one fma removes the
// 1024 and applies sc (c1 = sc, a1 = -1024 sc; c16 = sc/16, a16 = -64 sc), exactly.
__device__ __forceinline__ uint4 widen_q4(uint32_t x, __half2 c1, __half2 a1, __half2 c16, __half2 a16)
{
    const uint32_t xh = x >> 8;
    uint4 o;
    o.x = h2u(__hfma2(u2h(lop_or(x, 0x000F000Fu)), c1, a1));
    o.y = h2u(__hfma2(u2h(lop_or(x, 0x00F000F0u)), c16, a16));
    o.z = h2u(__hfma2(u2h(lop_or(xh, 0x000F000Fu)), c1, a1));
    o.w = h2u(__hfma2(u2h(lop_or(xh, 0x00F000F0u)), c16, a16));
    return o;
}

// q6_K, one sub-block word x (16 values, byte 4 (q + 32) each, values 4u + {0, 1} at
// bytes 0, 2 and 4u + {2, 3} at bytes 1, 3 of 32-bit word u): the mask puts 4 (q + 32)
// under the exponent of 1024, so each f16 lane is 1024 + 4 (q + 32), exactly.
//   one tile (every |sc| <= 64): fma(1024 + 4 (q + 32), sc/4, -288 sc) = sc * q
//     (|sc q| <= 2048: exact; 288 sc is 9 * 32 * sc, exact);
//   two tiles: the low 4 bits l alone give fma(1024 + 4 l, sc/16, -64 sc) = sc * l / 4
//     (a quarter-integer below 480) and the high 2 bits h alone give
//     fma(1024 + 64 h, sc/16, -72 sc) = 4 sc (h - 2); both exact for any int8 sc.
__device__ __forceinline__ uint32_t q6_pair(uint32_t w, uint32_t mask, __half2 c, __half2 a)
{
    return h2u(__hfma2(u2h(lop_or(w, mask)), c, a));
}
__device__ __forceinline__ void widen_q6_one(uint4 x, __half2 c, __half2 a, uint4& o0, uint4& o1)
{
    constexpr uint32_t Q = 0x00FC00FCu;
    o0 = make_uint4(q6_pair(x.x, Q, c, a), q6_pair(x.x >> 8, Q, c, a), q6_pair(x.y, Q, c, a),
                    q6_pair(x.y >> 8, Q, c, a));
    o1 = make_uint4(q6_pair(x.z, Q, c, a), q6_pair(x.z >> 8, Q, c, a), q6_pair(x.w, Q, c, a),
                    q6_pair(x.w >> 8, Q, c, a));
}
__device__ __forceinline__ void widen_q6_two(uint4 x, __half2 c, __half2 al, __half2 ah, uint4& l0, uint4& l1,
                                             uint4& h0, uint4& h1)
{
    constexpr uint32_t L = 0x003C003Cu, H = 0x00C000C0u;
    const uint32_t w[8] = {x.x, x.x >> 8, x.y, x.y >> 8, x.z, x.z >> 8, x.w, x.w >> 8};
    l0 = make_uint4(q6_pair(w[0], L, c, al), q6_pair(w[1], L, c, al), q6_pair(w[2], L, c, al), q6_pair(w[3], L, c, al));
    l1 = make_uint4(q6_pair(w[4], L, c, al), q6_pair(w[5], L, c, al), q6_pair(w[6], L, c, al), q6_pair(w[7], L, c, al));
    h0 = make_uint4(q6_pair(w[0], H, c, ah), q6_pair(w[1], H, c, ah), q6_pair(w[2], H, c, ah), q6_pair(w[3], H, c, ah));
    h1 = make_uint4(q6_pair(w[4], H, c, ah), q6_pair(w[5], H, c, ah), q6_pair(w[6], H, c, ah), q6_pair(w[7], H, c, ah));
}

// Four f16 pairs (one 8-value unit) from each of 4 uint4: 16 TMEM columns of one lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint4 (&v)[4])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
        "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y), "r"(v[1].z), "r"(v[1].w),
        "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w), "r"(v[3].x), "r"(v[3].y), "r"(v[3].z), "r"(v[3].w)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem]^T, one 128 x N x 16 kind::f16 step (A: 128 lanes x 8
// columns, each 32-bit column two consecutive K values), issued by one thread.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Work unit u: weight tile n and its super-block range; stage st of the unit covers
// k-blocks [4*sb0 + st*KPS, +KPS).  Stages are numbered across the CTA's units (g);
// stage g goes to issuer g % 2 and accumulator item g % ITEMS, its super-block's
// tokens to slot (g / SPS) % 2.
template <int TYPE, int NT, bool ONE>
__device__ __forceinline__ void ft_roles(const FtArgs& g, uint8_t* smem, uint32_t sbase, uint32_t tmem_base,
                                         int warp, int lane)
{
    using C = Cfg<TYPE, NT, ONE>;
    constexpr bool Q4 = (TYPE == 12);
    constexpr int N = C::N;
    constexpr int KPS = C::KPS;
    constexpr int SPS = C::SPS;
    const int nkb = g.id / TILE_K;
    const int nsb = g.id / QK_K;
    auto bar = [&](int i) -> uint32_t { return sbase + C::SMEM_BAR + 8u * static_cast<uint32_t>(i); };
    const bool clustered = g.kslices > 1;

    if (warp < CONV_WARP0) {
        if constexpr (C::SPLIT_REGS)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(CTRL_REGS));
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ producer: compact codes, super-block entries
            RingPos<C::RAW_STAGES> rp;
            RingPos<C::SBR> sp;
            uint32_t n_raw = 0, n_sb = 0;
            const uint32_t skip = (blockIdx.x == 0 && g.withhold >= 0) ? static_cast<uint32_t>(g.withhold) : ~0u;
            constexpr uint32_t SB_TX = BM * 4 + BM * SC_ROW_BYTES + FT_MAX_M * 4 + (Q4 ? BM * 4 + FT_MAX_M * 32 : 0);
            bool ok = true;
            for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
                const Unit w = unit_of(g, u, nsb);
                const uint8_t* cwb = g.CW + (static_cast<size_t>(w.n) * nkb + 4 * w.sb0) * cw_kblock_bytes(TYPE);
                const int nst = (w.sb1 - w.sb0) * SPS;
                bulk_prefetch_l2(cwb, static_cast<uint32_t>(min(PF_STAGES, nst) * C::RAW_BYTES));
                for (int st = 0; st < nst; ++st) {
                    if (st % SPS == 0) {
                        const int s = w.sb0 + st / SPS;
                        if (!ctl_wait(g, bar(C::BAR_SBEMPTY + sp.i), sp.ph ^ 1u)) {
                            ok = false;
                            break;
                        }
                        // consumers read the entry with ordinary loads; the bulk copy that
                        // refills it is ordered after them only through this proxy fence
                        fence_proxy_async_smem();
                        const uint32_t dst = sbase + C::SMEM_SB + sp.i * C::SB_BYTES;
                        const uint32_t fb = bar(C::BAR_SBFULL + sp.i);
                        mbar_arrive_expect_tx(fb, SB_TX);
                        const size_t ts = static_cast<size_t>(w.n) * nsb + s;
                        bulk_g2s(dst + SB_SBD_OFF, g.SBD + ts * (BM * 4), BM * 4, fb);
                        bulk_g2s(dst + SB_SC_OFF, g.SC + ts * (BM * SC_ROW_BYTES), BM * SC_ROW_BYTES, fb);
                        bulk_g2s(dst + SB_IP_OFF, g.IP + static_cast<size_t>(s) * (FT_MAX_M * 4), FT_MAX_M * 4, fb);
                        if (Q4) {
                            bulk_g2s(dst + SB_DM_OFF, g.DM + ts * (BM * 4), BM * 4, fb);
                            // [chunk][FT_MAX_M tokens]: the whole super-block's 2 KB
                            bulk_g2s(dst + SB_FM_OFF, g.FM + static_cast<size_t>(s) * (FT_MAX_M * 32), FT_MAX_M * 32,
                                     fb);
                        }
                        sp.next();
                        ++n_sb;
                    }
                    if (!ctl_wait(g, bar(C::BAR_REMPTY + rp.i), rp.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    if (st + PF_STAGES < nst)
                        bulk_prefetch_l2(cwb + static_cast<size_t>(st + PF_STAGES) * C::RAW_BYTES, C::RAW_BYTES);
                    if (n_raw == skip) {   // verification: this fill is left out
                        rp.next();
                        ++n_raw;
                        continue;
                    }
                    fence_proxy_async_smem();
                    const uint32_t fb = bar(C::BAR_RFULL + rp.i);
                    mbar_arrive_expect_tx(fb, C::RAW_BYTES);
                    bulk_g2s(sbase + C::SMEM_RAW + rp.i * C::RAW_BYTES, cwb + static_cast<size_t>(st) * C::RAW_BYTES,
                             C::RAW_BYTES, fb);
                    rp.next();
                    ++n_raw;
                }
            }
            for (uint32_t i = (n_raw > C::RAW_STAGES ? n_raw - C::RAW_STAGES : 0); i < n_raw; ++i)
                if (i != skip)
                    drain_wait(g, bar(C::BAR_RFULL + i % C::RAW_STAGES), (i / C::RAW_STAGES) & 1u);
            for (uint32_t i = (n_sb > C::SBR ? n_sb - C::SBR : 0); i < n_sb; ++i)
                drain_wait(g, bar(C::BAR_SBFULL + i % C::SBR), (i / C::SBR) & 1u);
        } else if ((warp == 3 || warp == 1) && lane == 0) {
            // ------------------------------------------------ MMA issuers: stage g with g % 2 == e
            const uint32_t e = warp == 3 ? 0u : 1u;
            constexpr uint32_t idesc = idesc_f16_f32(BM, 2 * N);   // hi and lo token rows at once
            uint32_t gs = 0;                                        // stage number across units
            bool ok = true;
            for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
                const Unit w = unit_of(g, u, nsb);
                const int nst = (w.sb1 - w.sb0) * SPS;
                for (int st = 0; st < nst; ++st, ++gs) {
                    if ((gs & 1u) != e)
                        continue;
                    const uint32_t item = gs % C::ITEMS, iph = (gs / C::ITEMS) & 1u;
                    const uint32_t sg = gs / SPS;                     // super-block number across units
                    const uint32_t slot = sg % TOK_STAGES, tph = (sg / TOK_STAGES) & 1u;
                    if (!ctl_wait(g, bar(C::BAR_TEMPTY + item), iph ^ 1u) ||
                        !ctl_wait(g, bar(C::BAR_TKFULL + slot), tph) ||
                        !ctl_wait(g, bar(C::BAR_WCONV + e), (gs >> 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + item * C::ITEM_COLS;
                    const uint32_t wa = tmem_base + WBUF_COL0 + e * WBUF_COLS;
                    const uint32_t tk = sbase + C::SMEM_TOK + slot * C::TOK_SLOT;
                    const int sst = static_cast<int>(gs % SPS);       // stage within its super-block
#pragma unroll
                    for (int k = 0; k < KPS; ++k) {
                        // the k-block's 2N token rows: N of hi, then N of lo
                        const uint64_t bt = sdesc_k_sw128(tk + (sst * KPS + k) * C::TOK_KB_BYTES);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {       // 16 values per step
                            const uint32_t acol = 32u * k + 8u * kk;
                            umma_f16_ts(d, wa + acol, bt + 2u * kk, idesc, (k | kk) ? 1u : 0u);
                            if (!ONE)
                                umma_f16_ts(d, wa + 64u + acol, bt + 2u * kk, idesc, 1u);
                        }
                    }
                    umma_commit(bar(C::BAR_AEMPTY + e));
                    umma_commit(bar(C::BAR_TFULL + item));
                    umma_commit(bar(C::BAR_TKEMPTY + slot));
                }
            }
            umma_commit(bar(C::BAR_DRAIN));           // every MMA this thread issued has completed
            drain_wait(g, bar(C::BAR_DRAIN), 0u);
        } else if (warp == 2 && lane == 0) {
            // ------------------------------------------------ producer: token tiles
            RingPos<TOK_STAGES> tp;
            uint32_t n_t = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
                const Unit w = unit_of(g, u, nsb);
                for (int s = w.sb0; s < w.sb1; ++s) {
                    if (!ctl_wait(g, bar(C::BAR_TKEMPTY + tp.i), tp.ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar(C::BAR_TKFULL + tp.i);
                    mbar_arrive_expect_tx(fb, C::TOK_SLOT);
                    bulk_g2s(sbase + C::SMEM_TOK + tp.i * C::TOK_SLOT,
                             g.TQ + static_cast<size_t>(4 * s) * C::TOK_KB_BYTES, C::TOK_SLOT, fb);
                    tp.next();
                    ++n_t;
                }
            }
            for (uint32_t i = (n_t > TOK_STAGES ? n_t - TOK_STAGES : 0); i < n_t; ++i)
                drain_wait(g, bar(C::BAR_TKFULL + i % TOK_STAGES), (i / TOK_STAGES) & 1u);
        }
        __syncwarp();
        if (clustered) {
            named_bar_sync(1, NUM_THREADS);
            cluster_sync();
            cluster_sync();
        }
        return;
    }

    if (warp < PROMO_WARP0) {
        // ---------------------------------------------------- converters
        const int cwarp = warp - CONV_WARP0;
        const int q = cwarp & 3;                      // TMEM lane quarter of this warp
        const int r = q * 32 + lane;                  // weight row of the tile
        const int h = cwarp >> 2;                     // half of the stage
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        RingPos<C::RAW_STAGES> rp;
        RingPos<C::SBR> sp;
        RingPos<2> ab;              // weight buffer
        bool ok = true;
        for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
            const Unit w = unit_of(g, u, nsb);
            const int nst = (w.sb1 - w.sb0) * SPS;
            for (int st = 0; st < nst; ++st) {
                const int sst = st % SPS;                  // stage within its super-block
                if (sst == 0 && !warp_wait(g, bar(C::BAR_SBFULL + sp.i), sp.ph)) {
                    ok = false;
                    break;
                }
                const uint8_t* scr = smem + C::SMEM_SB + sp.i * C::SB_BYTES + SB_SC_OFF + r * SC_ROW_BYTES;
                if (!warp_wait(g, bar(C::BAR_RFULL + rp.i), rp.ph)) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = smem + C::SMEM_RAW + rp.i * C::RAW_BYTES;
                // this half's words: q4_K the 4 chunks of k-blocks 2h, 2h+1; q6_K two-tile the
                // 4 sub-block words of k-block h; q6_K one-tile those of k-blocks 2h and 2h+1
                constexpr int NW = Q4 ? 4 : (ONE ? 8 : 4);
                uint4 xw[NW];
                if (Q4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        xw[j] = *reinterpret_cast<const uint4*>(raw + (2 * h + (j >> 1)) * cw_kblock_bytes(TYPE) +
                                                                ((j & 1) * BM + r) * 16);
                } else {
#pragma unroll
                    for (int b = 0; b < NW / 4; ++b) {
                        const uint8_t* kb = raw + ((NW / 4) * h + b) * cw_kblock_bytes(TYPE);
#pragma unroll
                        for (int wd = 0; wd < 4; ++wd)
                            xw[4 * b + wd] = *reinterpret_cast<const uint4*>(kb + (wd * BM + r) * 16);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(C::BAR_REMPTY + rp.i));
                rp.next();
                if (!warp_wait(g, bar(C::BAR_AEMPTY + ab.i), ab.ph ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();   // the MMAs that read this buffer have completed
                const uint32_t wcol = lane_base + WBUF_COL0 + ab.i * WBUF_COLS;
                if (Q4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int cc = 4 * h + j;                 // chunk of the super-block
                        const float sc = static_cast<float>(scr[cc]);
                        const __half2 c1 = __float2half2_rn(sc), a1 = __float2half2_rn(-1024.0f * sc);
                        const __half2 c16 = __float2half2_rn(sc * 0.0625f), a16 = __float2half2_rn(-64.0f * sc);
                        const uint4 o[4] = {widen_q4(xw[j].x, c1, a1, c16, a16), widen_q4(xw[j].y, c1, a1, c16, a16),
                                            widen_q4(xw[j].z, c1, a1, c16, a16), widen_q4(xw[j].w, c1, a1, c16, a16)};
                        tmem_st16(wcol + 64 * h + 16 * j, o);
                    }
                } else {
#pragma unroll
                    for (int b = 0; b < NW / 4; ++b) {
                        const int kbs = ONE ? 2 * h + b : 2 * sst + h;     // k-block of the super-block
                        const int kcol = ONE ? 32 * (2 * h + b) : 32 * h;  // its columns in the buffer
#pragma unroll
                        for (int cw = 0; cw < 2; ++cw) {               // the k-block's two chunks
                            const int cc = 2 * kbs + cw;               // chunk of the super-block
                            uint4 oa[4], ob[4];
#pragma unroll
                            for (int half = 0; half < 2; ++half) {     // 16-value sub-blocks
                                const float sc = static_cast<float>(static_cast<int8_t>(scr[2 * cc + half]));
                                const uint4 x = xw[4 * b + 2 * cw + half];
                                if (ONE) {
                                    widen_q6_one(x, __float2half2_rn(0.25f * sc), __float2half2_rn(-288.0f * sc),
                                                 oa[2 * half], oa[2 * half + 1]);
                                } else {
                                    widen_q6_two(x, __float2half2_rn(0.0625f * sc), __float2half2_rn(-64.0f * sc),
                                                 __float2half2_rn(-72.0f * sc), oa[2 * half], oa[2 * half + 1],
                                                 ob[2 * half], ob[2 * half + 1]);
                                }
                            }
                            tmem_st16(wcol + kcol + 16 * cw, oa);
                            if (!ONE)
                                tmem_st16(wcol + 64 + kcol + 16 * cw, ob);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(C::BAR_WCONV + ab.i));
                ab.next();
                if (sst == SPS - 1) {
                    if (lane == 0)
                        mbar_arrive(bar(C::BAR_SBEMPTY + sp.i));
                    sp.next();
                }
            }
        }
        if (clustered) {
            named_bar_sync(1, NUM_THREADS);
            cluster_sync();
            cluster_sync();
        }
        return;
    }

    // -------------------------------------------------------- promotion
    if constexpr (C::SPLIT_REGS)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(PROMO_REGS));
    const int q = warp & 3;                              // TMEM lane quarter
    const int row = q * 32 + lane;                       // weight row of the tile
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    constexpr float IPS = ONE ? 1.0f : 4.0f;             // two q6_K tiles hold sc * q / 4
    RingPos<C::ITEMS> it;
    RingPos<C::SBR> sp;
    bool ok = true, had_unit = false;
    int n_tile = 0;
    float acc[N];
#pragma unroll
    for (int t = 0; t < N; ++t)
        acc[t] = 0.0f;
    for (int u = blockIdx.x; ok && u < g.units; u += gridDim.x) {
        const Unit w = unit_of(g, u, nsb);
        n_tile = w.n;
        had_unit = true;
#pragma unroll
        for (int t = 0; t < N; ++t)
            acc[t] = 0.0f;
        for (int s = w.sb0; s < w.sb1; ++s) {
            if (!warp_wait(g, bar(C::BAR_SBFULL + sp.i), sp.ph)) {
                ok = false;
                break;
            }
            const uint8_t* sbe = smem + C::SMEM_SB + sp.i * C::SB_BYTES;
            const float dsb = reinterpret_cast<const float*>(sbe + SB_SBD_OFF)[row];
            const float4* ip4 = reinterpret_cast<const float4*>(sbe + SB_IP_OFF);
            // the super-block's SPS stage items: it, it + 1 (mod ITEMS)
            uint32_t ii[SPS];
            bool got = true;
#pragma unroll
            for (int k = 0; k < SPS; ++k) {
                ii[k] = it.i;
                got = got && warp_wait(g, bar(C::BAR_TFULL + it.i), it.ph);
                it.next();
            }
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int gq = 0; gq < NT; ++gq) {
                float Dt[16];              // sum over the stages of W*hi + W*lo, tokens 16gq ..
#pragma unroll
                for (int k = 0; k < SPS; ++k) {
                    float Dh[16], Dl[16];
                    tmem_ld16x2_wait(lane_addr + ii[k] * C::ITEM_COLS + 16 * gq,
                                     lane_addr + ii[k] * C::ITEM_COLS + N + 16 * gq, Dh, Dl);
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        float s0, s1;
                        fadd2(s0, s1, Dh[e], Dh[e + 1], Dl[e], Dl[e + 1]);
                        if (k == 0) {
                            Dt[e] = s0;
                            Dt[e + 1] = s1;
                        } else {
                            fadd2(Dt[e], Dt[e + 1], Dt[e], Dt[e + 1], s0, s1);
                        }
                    }
                }
                if (gq == NT - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int k = 0; k < SPS; ++k)
                            mbar_arrive(bar(C::BAR_TEMPTY + ii[k]));
                    }
                }
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const float4 ipv = ip4[4 * gq + i4];
                    const float ipa[4] = {ipv.x, ipv.y, ipv.z, ipv.w};
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int t = 16 * gq + 4 * i4 + e;
                        float p0, p1;
                        fmul2(p0, p1, Dt[4 * i4 + e], Dt[4 * i4 + e + 1], ipa[e] * IPS, ipa[e + 1] * IPS);
                        ffma2(acc[t], acc[t + 1], dsb, p0, p1);
                    }
                }
            }
            if (Q4) {
                // min term: acc -= sum_c (dmin * m_c) * (d_a * ssum)_c
                const float dmin = reinterpret_cast<const float*>(sbe + SB_DM_OFF)[row];
                const uint2 mw = *reinterpret_cast<const uint2*>(sbe + SB_SC_OFF + row * SC_ROW_BYTES + 8);
                float dmn[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dmn[c] = -__fmul_rn(dmin, static_cast<float>(((c < 4 ? mw.x : mw.y) >> (8 * (c & 3))) & 0xFFu));
                // chunk-major d_a*ssum: four tokens per load, two per f32x2 fma (each token's
                // sum still runs over c = 0..7 in order)
                const float* fmc = reinterpret_cast<const float*>(sbe + SB_FM_OFF);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
#pragma unroll
                    for (int t = 0; t < N; t += 4) {
                        const float4 f = *reinterpret_cast<const float4*>(fmc + c * FT_MAX_M + t);
                        ffma2(acc[t], acc[t + 1], dmn[c], f.x, f.y);
                        ffma2(acc[t + 2], acc[t + 3], dmn[c], f.z, f.w);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(C::BAR_SBEMPTY + sp.i));
            sp.next();
        }
        if (!ok)
            break;
        if (!clustered) {
            const int j = w.n * BM + row;
            if (j < g.od) {
#pragma unroll
                for (int t = 0; t < N; ++t)
                    if (t < g.M)
                        g.Y[static_cast<size_t>(t) * g.ldy + j] = acc[t];
            }
        }
    }
    if (clustered) {
        // The K slices' partial sums meet in rank 0 and are added in rank order.  The CTA
        // barrier lets the producers and the MMA issuers finish draining their copies and
        // MMAs first, so the rings are idle when the partial sums overwrite them.  Each
        // rank leaves one ok flag per promotion warp; rank 0 stores Y only if all are set.
        const uint32_t rank = cluster_ctarank();
        float* scratch = reinterpret_cast<float*>(smem + C::SMEM_TOK);
        named_bar_sync(1, NUM_THREADS);
        if (rank != 0) {
#pragma unroll
            for (int t = 0; t < N; ++t)
                scratch[t * BM + row] = acc[t];
        }
        if (lane == 0)
            reinterpret_cast<int*>(smem + C::SMEM_TOK + C::OKF_OFF)[q] = ok ? 1 : 0;
        cluster_sync();
        if (rank == 0) {
            // every rank's flags at once: lane l reads flag l % 4 of rank l / 4 (S * 4 <= 32)
            uint32_t f = 1u;
            if (lane < g.kslices * NUM_PROMO_WARPS)
                f = ld_cluster_u32(cluster_map(sbase + C::SMEM_TOK + C::OKF_OFF, static_cast<uint32_t>(lane >> 2)) +
                                   4u * static_cast<uint32_t>(lane & 3));
            const bool all_ok = __all_sync(0xffffffffu, f != 0u) && ok && had_unit;
            if (all_ok) {
                for (int rr = 1; rr < g.kslices; ++rr) {
                    const uint32_t rbase = cluster_map(sbase + C::SMEM_TOK, static_cast<uint32_t>(rr));
#pragma unroll
                    for (int t0 = 0; t0 < N; t0 += 16) {
                        float v[16];        // 16 loads in flight before their sums
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            v[t] = ld_cluster_f32(rbase + 4u * static_cast<uint32_t>((t0 + t) * BM + row));
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            acc[t0 + t] += v[t];
                    }
                }
                const int j = n_tile * BM + row;
                if (j < g.od) {
#pragma unroll
                    for (int t = 0; t < N; ++t)
                        if (t < g.M)
                            g.Y[static_cast<size_t>(t) * g.ldy + j] = acc[t];
                }
            }
        }
        cluster_sync();
    }
}

// Barrier set-up, TMEM, the roles, TMEM release, for one layout.
template <int TYPE, int NT, bool ONE>
__device__ __forceinline__ void ft_body(const FtArgs& g, uint8_t* smem, uint32_t sbase, int warp, int lane)
{
    using C = Cfg<TYPE, NT, ONE>;
    auto bar = [&](int i) -> uint32_t { return sbase + C::SMEM_BAR + 8u * static_cast<uint32_t>(i); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::RAW_STAGES; ++s) {
            mbar_init(bar(C::BAR_RFULL + s), 1);
            mbar_init(bar(C::BAR_REMPTY + s), NUM_CONV_WARPS);
        }
        for (int s = 0; s < TOK_STAGES; ++s) {
            mbar_init(bar(C::BAR_TKFULL + s), 1);
            mbar_init(bar(C::BAR_TKEMPTY + s), C::SPS);          // one commit per stage of the super-block
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::BAR_AEMPTY + s), 1);
            mbar_init(bar(C::BAR_WCONV + s), NUM_CONV_WARPS);
        }
        for (int s = 0; s < C::SBR; ++s) {
            mbar_init(bar(C::BAR_SBFULL + s), 1);
            mbar_init(bar(C::BAR_SBEMPTY + s), NUM_CONV_WARPS + NUM_PROMO_WARPS);
        }
        for (int k = 0; k < C::ITEMS; ++k) {
            mbar_init(bar(C::BAR_TFULL + k), 1);
            mbar_init(bar(C::BAR_TEMPTY + k), NUM_PROMO_WARPS);
        }
        mbar_init(bar(C::BAR_DRAIN), NUM_ISSUERS);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(sbase + C::SMEM_TMEMPTR, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + C::SMEM_TMEMPTR);

    // the kernel ahead on the stream (the prepass) writes the token planes; the weight
    // planes are registration-time data
    grid_dep_wait();
    ft_roles<TYPE, NT, ONE>(g, smem, sbase, tmem_base, warp, lane);

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int TYPE, int NT>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_ft_kernel(const FtArgs g)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The next kernel on the stream may be scheduled as SMs free up (it waits for this
    // grid to complete before it touches memory), for q6_K and for clustered launches;
    // and while the kernel ahead of this one finishes, a q6_K CTA warms L2 with its first
    // weights: the compact codes of its first two super-blocks and the first super-
    // block's scales (a prefetch changes no value).  Measured back to back: q6_K
    // 4097x11008 -8 %, q4_K 4096x4096 (clusters) -3 %; the early trigger made the
    // unclustered q4_K 11008x4096 at 40-64 tokens 4-7 % slower, and the q4_K prefetch
    // made no difference.
    if (TYPE == 14 || g.kslices > 1)
        grid_dep_launch();
    if (TYPE == 14 && threadIdx.x == 0 && static_cast<int>(blockIdx.x) < g.units) {
        const int nsb = g.id / QK_K;
        const Unit w = unit_of(g, static_cast<int>(blockIdx.x), nsb);
        const size_t ts = static_cast<size_t>(w.n) * nsb + w.sb0;
        const int nkb = g.id / TILE_K;
        const uint32_t cw_sb = 4u * static_cast<uint32_t>(cw_kblock_bytes(TYPE));
        bulk_prefetch_l2(g.CW + (static_cast<size_t>(w.n) * nkb + 4 * w.sb0) * cw_kblock_bytes(TYPE),
                         (w.sb1 - w.sb0 > 1 ? 2u : 1u) * cw_sb);
        bulk_prefetch_l2(g.SC + ts * (BM * SC_ROW_BYTES), BM * SC_ROW_BYTES);
        bulk_prefetch_l2(g.SBD + ts * (BM * 4), BM * 4);
    }
    if constexpr (TYPE == 12) {
        ft_body<12, NT, true>(g, smem, sbase, warp, lane);
    } else {
        // the packed flag (uniform for the launch) says whether every sub-block scale
        // fits the one-tile form; it is read only once the kernel ahead, which may be the
        // repack that wrote it, has completed
        grid_dep_wait();
        if (__ldg(g.FLAG) != 0u)
            ft_body<14, NT, true>(g, smem, sbase, warp, lane);
        else
            ft_body<14, NT, false>(g, smem, sbase, warp, lane);
    }
}

template <int TYPE, int NT>
cudaError_t set_smem_attr()
{
    static std::atomic<uint64_t> attr_set_mask{0};  // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (attr_set_mask.load() & bit)
        return cudaSuccess;
    if (Cfg<TYPE, NT, true>::SPLIT_REGS) {
        // The setmaxnreg split draws on the registers the launch reserved; a build that
        // compiled to fewer per thread would make the promotion warps wait forever.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, gemm_ft_kernel<TYPE, NT>);
        if (e != cudaSuccess)
            return e;
        if (fa.numRegs < LAUNCH_REGS)
            return cudaErrorInvalidKernelImage;
    }
    e = cudaFuncSetAttribute(gemm_ft_kernel<TYPE, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_alloc_of<TYPE, NT>());
    if (e != cudaSuccess)
        return e;
    attr_set_mask.fetch_or(bit);
    return cudaSuccess;
}

// Clusters of `size` CTAs that can be resident at once (0 if none or the query fails);
// cached per instantiation, size and device ordinal.
template <int TYPE, int NT>
int max_clusters(int size)
{
    static std::atomic<int> cache[MAX_CLUSTER + 1][64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || size < 2 || size > MAX_CLUSTER)
        return 0;
    const int c = cache[size][dev].load();
    if (c != 0)
        return c > 0 ? c : 0;
    int n = 0;
    if (set_smem_attr<TYPE, NT>() == cudaSuccess) {
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = static_cast<unsigned>(size);
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(size));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = smem_alloc_of<TYPE, NT>();
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_ft_kernel<TYPE, NT>, &cfg) != cudaSuccess) {
            n = 0;
            cudaGetLastError();   // clear the failed query's error, and only that one
        }
    } else {
        cudaGetLastError();
    }
    cache[size][dev].store(n > 0 ? n : -1);
    return n;
}

template <int TYPE, int NT>
cudaError_t launch_ft_typed(FtArgs a, int nsm, bool allow_cluster, cudaStream_t s)
{
    cudaError_t e = set_smem_attr<TYPE, NT>();
    if (e != cudaSuccess)
        return e;
    const int nsb = a.id / QK_K;
    a.kslices = 1;
    if (allow_cluster) {
        // the largest cluster along K with one cluster per weight tile resident at once
        constexpr int sizes[5] = {8, 6, 4, 3, 2};
        for (int ks : sizes) {
            if (nsb < ks || static_cast<long long>(a.num_n) * ks > nsm)
                continue;
            if (max_clusters<TYPE, NT>(ks) >= a.num_n) {
                a.kslices = ks;
                break;
            }
        }
    }
    a.units = a.num_n * a.kslices;
    const int grid = a.kslices > 1 ? a.units : (a.num_n < nsm ? a.num_n : nsm);
    cudaLaunchAttribute at[2];
    int na = 0;
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (a.kslices > 1) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = static_cast<unsigned>(a.kslices);
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        ++na;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem_alloc_of<TYPE, NT>();
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = na;
    count_launch();
    e = cudaLaunchKernelEx(&cfg, gemm_ft_kernel<TYPE, NT>, a);
    if (e == cudaSuccess)
        g_last_kslices = a.kslices;
    return e;
}

template <int TYPE>
cudaError_t launch_ft_nt(const FtArgs& a, int nsm, bool allow_cluster, cudaStream_t s)
{
    switch (a.n_tok / 16) {
    case 1: return launch_ft_typed<TYPE, 1>(a, nsm, allow_cluster, s);
    case 2: return launch_ft_typed<TYPE, 2>(a, nsm, allow_cluster, s);
    case 3: return launch_ft_typed<TYPE, 3>(a, nsm, allow_cluster, s);
    default: return launch_ft_typed<TYPE, 4>(a, nsm, allow_cluster, s);
    }
}

}  // namespace

cudaError_t launch_gemm_ft(int type, const void* packed, int od, int id, const void* qa, const void* scales,
                           int M, float* Y, int ldy, cudaStream_t s, const WaitCtl& wc, bool allow_cluster,
                           const char** path_label)
{
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    const WeightPlanes wp = weight_planes(type, od, id);
    const ActPlanes ap = act_planes(M, id);
    const uint8_t* pk = static_cast<const uint8_t*>(packed);
    const uint8_t* sc = static_cast<const uint8_t*>(scales);
    FtArgs a;
    a.CW = pk + wp.cw_off;
    a.SC = pk + wp.sc_off;
    a.SBD = pk + wp.sbd_off;
    a.DM = pk + wp.dm_off;
    a.FLAG = reinterpret_cast<const unsigned int*>(pk + wp.flag_off);
    a.TQ = static_cast<const uint8_t*>(qa) + ap.tq_off;
    a.IP = sc + ap.ip_off;
    a.FM = sc + ap.fm_off;
    a.Y = Y;
    a.ldy = ldy;
    a.M = M;
    a.od = od;
    a.id = id;
    a.n_tok = ft_n(M);
    a.num_n = ceil_div(od, BM);
    a.units = a.num_n;
    a.kslices = 1;
    a.err = wc.err;
    a.wait_ns = wc.limit_ns;
    a.withhold = wc.withhold_fill;
    e = type == 14 ? launch_ft_nt<14>(a, nsm, allow_cluster, s) : launch_ft_nt<12>(a, nsm, allow_cluster, s);
    if (e == cudaSuccess && path_label) {
        static const char* const lab[2][9] = {
            {"q4_K: few-token GEMM (M <= 64): compact 4-bit codes widened to sc*q f16 tiles in tensor memory, "
             "weights as the MMA's A, token operand p*d_a*q_a as f16 hi+lo as N, two MMA issuers with one TMEM "
             "accumulator per stage, min term on the CUDA cores in f32x2 pairs; "
             "K split: none",
             "", "q4_K: few-token GEMM (M <= 64): compact 4-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=2 CTAs",
             "q4_K: few-token GEMM (M <= 64): compact 4-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=3 CTAs",
             "q4_K: few-token GEMM (M <= 64): compact 4-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=4 CTAs",
             "", "q4_K: few-token GEMM (M <= 64): compact 4-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=6 CTAs",
             "", "q4_K: few-token GEMM (M <= 64): compact 4-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=8 CTAs"},
            {"q6_K: few-token GEMM (M <= 64): compact 6-bit codes widened in tensor memory to one sc*q f16 tile "
             "(every |sc| <= 64) or two exact tiles (sc*l/4, 4*sc*(h-2)), weights as the MMA's A, token operand "
             "p*d_a*q_a as f16 hi+lo as N, two MMA issuers with one TMEM accumulator per stage; K split: none",
             "", "q6_K: few-token GEMM (M <= 64): compact 6-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=2 CTAs",
             "q6_K: few-token GEMM (M <= 64): compact 6-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=3 CTAs",
             "q6_K: few-token GEMM (M <= 64): compact 6-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=4 CTAs",
             "", "q6_K: few-token GEMM (M <= 64): compact 6-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=6 CTAs",
             "", "q6_K: few-token GEMM (M <= 64): compact 6-bit codes widened into tensor memory, two MMA issuers; K split: cluster of S=8 CTAs"}};
        *path_label = lab[type == 14 ? 1 : 0][g_last_kslices > 1 ? g_last_kslices : 0];
    }
    return e;
}

}  // namespace mmq
