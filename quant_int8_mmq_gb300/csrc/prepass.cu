// prepass.cu -- activation quantize-transpose prepass.
//
// Per token t and 32-value chunk c: amax = max|x|, d = amax/127 (IEEE f32
// division), q = round(x/d) (IEEE f32 division, ties away from zero, clamped to
// [-127,127]), ssum = sum q; d == 0 gives q = 0.  The codes are written as exact
// f16 integers straight into the tensor-core operand tile layout (128 tokens x 64
// values, 128-byte swizzle), so the GEMM stages them with one bulk copy and no
// conversion; the (d, ssum) pairs go to a tile-major scale plane.  It also writes
// the operand of the q4_K min-term side contraction: ma = d*ssum (one f32
// multiply) split exactly-enough into tf32 hi = rna(ma) and lo = rna(ma - hi),
// in 128 x 8 tf32 tiles per (token tile, super-block).  Padded token rows
// (t >= M) are zero-filled.  For M <= SMALL_M it also writes the codes as int8,
// row-major, in the small_pos order the weight-streaming GEMM consumes.
//
// Sources: the prepass that moved activation quantization and transposition
// out of the GEMM and writes pre-transposed qa8 and d/ssum planes with padded
// rows zeroed ("r45 - cp.async for the q6_K A-side staging ...", §1.1 and §2.3;
// "r56 - q6_K A-side bundle ...", §1).
//
// Mapping: one half-warp per (token row, 256-value super-block); lane l of the half owns
// values 16l..16l+15 (four 16-byte loads), so two lanes share a 32-value chunk and the
// amax and ssum reductions take one shuffle each, and the per-chunk work (the divisor,
// its reciprocal, the scale entries) is spread over 16 values per lane.  A lane's 16
// codes are two 16-byte segments of the swizzled operand tile.  Consecutive half-warps
// take consecutive token rows of one super-block, so the tile rows and the scale
// entries they write are contiguous in HBM.
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "ptx.cuh"

namespace mmq {
namespace {

// round(x/d) as an integer-valued float, clamped to [-127, 127] (the clamp matters
// only for subnormal d, whose rounding can leave |x/d| above 127.5).
__device__ __forceinline__ float quant_one(float x, float d)
{
    const float r = roundf(__fdiv_rn(x, d));
    return fminf(fmaxf(r, -127.0f), 127.0f) + 0.0f;    // + 0: code 0 is +0, never -0
}

// Packed pairs of f32 (the f32x2 arithmetic of sm_100-class SMs: one instruction for two
// IEEE round-to-nearest operations, each rounded as its scalar form would be).
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// Round half away from zero of |y| < 2^23 as trunc(y + sign(y) * (1/2 - 2^-25)): below a
// tie the sum stays under the next integer (its distance to it is at least one ulp of y
// plus 2^-25, while the rounding moves it by at most half an ulp), at a tie or above it
// reaches the next integer (n + 1 - 2^-25 rounds up, to even at n + 1 = 1), and the
// truncation then gives the rounded value; -0 is left as -0.
__device__ __forceinline__ float round_away_small(float y)
{
    const float c = __uint_as_float((__float_as_uint(y) & 0x80000000u) | 0x3EFFFFFFu);
    return truncf(__fadd_rn(y, c));
}

// Eight codes of one chunk with the chunk's divisor shared, two values per instruction:
// rd = 1/d correctly rounded (once per chunk), then Markstein's correction step (P.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34, 1990): q0 = RN(x * rd) is within one ulp of x/d,
// e = x - d * q0 is exact as one FMA, and RN(q0 + e * rd) is the correctly rounded
// quotient RN(x/d) when rd = RN(1/d) and nothing overflows or underflows, which the
// caller guarantees by using this only for d in [2^-100, 2^100].  No clamp is needed:
// for finite x with |x| <= amax and d = RN(amax/127) normal, |x/d| <= 127 (1 + 2^-23),
// so the rounded quotient is at most 127 in magnitude.  q is left as integer-valued
// floats with code 0 as +0.
__device__ __forceinline__ void quant8_shared(const float (&v)[8], float d, float rd, float (&q)[8])
{
    const uint64_t rd2 = f2_pack(rd, rd), nd2 = f2_pack(-d, -d), zero2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t x2 = f2_pack(v[2 * i], v[2 * i + 1]);
        const uint64_t q0 = f2_mul(x2, rd2);
        const uint64_t e = f2_fma(q0, nd2, x2);       // x - d * q0, exact
        const uint64_t y = f2_fma(e, rd2, q0);        // RN(x / d)
        const uint64_t r = f2_add(f2_pack(round_away_small(f2_lo(y)), round_away_small(f2_hi(y))), zero2);
        q[2 * i] = f2_lo(r);
        q[2 * i + 1] = f2_hi(r);
    }
}

// Sum of eight integer-valued floats (exact: |sum| <= 1016).
__device__ __forceinline__ float sum8(const float (&q)[8])
{
    const uint64_t a = f2_add(f2_pack(q[0], q[1]), f2_pack(q[2], q[3]));
    const uint64_t b = f2_add(f2_pack(q[4], q[5]), f2_pack(q[6], q[7]));
    const uint64_t c = f2_add(a, b);
    return __fadd_rn(f2_lo(c), f2_hi(c));
}

__device__ __forceinline__ float tf32_rna(float v)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// The few-token GEMM's activation operand for one token and super-block.  p = 2^e is
// chosen from the largest chunk scale dmax of the super-block so that 127 * dmax * p
// < 2^14 (f32 exponent field of p: min(260 - E, 253), E that of dmax; 1/p is exact and
// normal); s = p * d is exact and is split into f16 s_hi = rn(s), s_lo = rn(s - s_hi);
// each code c (an exact f16 integer, |c| <= 127) gives hi = rn(s_hi * c) and
// lo = rn(s_hi * c - hi + s_lo * c), the residual s_hi * c - hi being exact in one fma,
// so that hi + lo carries about 21 significant bits of s * c.
__device__ __forceinline__ uint32_t ft_p_field(float dmax)
{
    const int E = static_cast<int>((__float_as_uint(dmax) >> 23) & 0xFFu);
    return static_cast<uint32_t>(min(260 - E, 253));
}
__device__ __forceinline__ void ft_split_pair(uint32_t cbits, __half2 s_hi, __half2 s_lo, uint32_t& hi, uint32_t& lo)
{
    const __half2 c = *reinterpret_cast<const __half2*>(&cbits);
    const __half2 h = __hmul2_rn(s_hi, c);
    const __half2 r = __hfma2(s_hi, c, __hneg2(h));
    const __half2 l = __hfma2(s_lo, c, r);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

__global__ void __launch_bounds__(256) quantize_act_kernel(const float* __restrict__ x, int M, int K, int ldx,
                                                           int Mp, int vec4, uint16_t* __restrict__ qa,
                                                           uint2* __restrict__ scales, uint8_t* __restrict__ am,
                                                           int8_t* __restrict__ qa8, uint8_t* __restrict__ tq,
                                                           float* __restrict__ ip, float* __restrict__ fm, int ftn)
{
    // x may come from the kernel ahead, and qa / scales may still be read by it.
    grid_dep_wait();
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int hl = lane & 15;                 // lane within its half-warp: values 16 hl .. 16 hl + 15
    const int nkb = K / TILE_K;
    const int nchunk = K / CHUNK;
    const int nsb = K / QK_K;
    // Item w = sb * Mp + t (token row t, super-block sb), one per half-warp, grid-stride over
    // half-warps; the (t, sb) pair is advanced incrementally (no 64-bit division per item).
    const int stride = gridDim.x * (blockDim.x >> 5) * 2;
    const int w0 = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 2 + (lane >> 4);
    const int st_t = stride % Mp, st_sb = stride / Mp;
    int t = w0 % Mp, sb = w0 / Mp;
    // Both halves run every pass (the shuffles below span whole warps); a half whose items
    // are done computes on zeros and stores nothing.
    while (__any_sync(0xffffffffu, sb < nsb)) {
        const bool valid = sb < nsb;
        const int k0 = sb * QK_K + 16 * hl;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = 0.0f;
        if (valid && t < M) {
            const float* p = x + static_cast<size_t>(t) * ldx + k0;
            if (vec4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 a = __ldcs(reinterpret_cast<const float4*>(p) + u);
                    v[4 * u] = a.x; v[4 * u + 1] = a.y; v[4 * u + 2] = a.z; v[4 * u + 3] = a.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = __ldcs(p + i);
            }
        }
        // the chunk (32 values) is this lane's 16 and its neighbour's (lane ^ 1)
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            a = fmaxf(a, fabsf(v[i]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        const float d = __fdiv_rn(a, 127.0f);
        const bool shared = (d >= 0x1p-100f && d <= 0x1p100f);
        const float rd = shared ? __frcp_rn(d) : 0.0f;
        // codes as integer-valued floats; their chunk sum (|.| <= 4064) is exact in f32
        // (one branch per lane: the 16 values share d, so the division path is never
        // evaluated next to the shared-reciprocal one)
        float q[2][8];
        if (shared) {
#pragma unroll
            for (int g = 0; g < 2; ++g)
                quant8_shared(reinterpret_cast<const float(&)[8]>(v[8 * g]), d, rd, q[g]);
        } else if (d != 0.0f) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                q[i >> 3][i & 7] = quant_one(v[i], d);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                q[i >> 3][i & 7] = 0.0f;
        }
        float sf = __fadd_rn(sum8(q[0]), sum8(q[1]));
        sf += __shfl_xor_sync(0xffffffffu, sf, 1);
        const int s = static_cast<int>(sf);

        const int mt = t / TILE_ROWS, r = t % TILE_ROWS;
        const int kb = k0 / TILE_K;
        const int kk = k0 % TILE_K;               // 16-value segment inside the k-block
        uint8_t* tile = reinterpret_cast<uint8_t*>(qa) + (static_cast<size_t>(mt) * nkb + kb) * TILE_BYTES;
        uint32_t h[2][4];
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i) {       // exact: |q| <= 127 is an f16 integer
                const __half2 p2 = __floats2half2_rn(q[g][2 * i], q[g][2 * i + 1]);
                h[g][i] = *reinterpret_cast<const uint32_t*>(&p2);
            }
        if (valid) {
#pragma unroll
            for (int g = 0; g < 2; ++g)
                *reinterpret_cast<uint4*>(tile + tile_byte(r, kk + 8 * g)) =
                    make_uint4(h[g][0], h[g][1], h[g][2], h[g][3]);
        }
        if (tq != nullptr) {
            // few-token operand: hi and lo tiles of p * d * q for this token row; p from
            // the largest chunk scale of the super-block (its 16 lanes)
            float dm = d;
            dm = fmaxf(dm, __shfl_xor_sync(0xffffffffu, dm, 2));
            dm = fmaxf(dm, __shfl_xor_sync(0xffffffffu, dm, 4));
            dm = fmaxf(dm, __shfl_xor_sync(0xffffffffu, dm, 8));
            if (valid && t < ftn) {
                const uint32_t pf = ft_p_field(dm);
                const float sv = __fmul_rn(d, __uint_as_float(pf << 23));  // exact: a power of two
                const __half shh = __float2half_rn(sv);
                const __half2 s_hi = __half2half2(shh);
                const __half2 s_lo = __half2half2(__float2half_rn(sv - __half2float(shh)));
                uint8_t* kt = tq + static_cast<size_t>(kb) * (2 * ftn * 128);
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    uint32_t hv[4], lv[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        ft_split_pair(h[g][i], s_hi, s_lo, hv[i], lv[i]);
                    const int off = tile_byte(t, kk + 8 * g);
                    *reinterpret_cast<uint4*>(kt + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    *reinterpret_cast<uint4*>(kt + ftn * 128 + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
                }
                if (hl == 0)
                    ip[static_cast<size_t>(sb) * FT_MAX_M + t] = __uint_as_float((254u - pf) << 23);
            }
        }
        if (qa8 != nullptr && valid && t < M) {
            // small_pos order inside each 8-value group: values (0,2,4,6) then (1,3,5,7)
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                int qi[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    qi[i] = static_cast<int>(q[g][i]);
                const uint32_t lo = (qi[0] & 0xFF) | ((qi[2] & 0xFF) << 8) | ((qi[4] & 0xFF) << 16) |
                                    (static_cast<uint32_t>(qi[6] & 0xFF) << 24);
                const uint32_t hi = (qi[1] & 0xFF) | ((qi[3] & 0xFF) << 8) | ((qi[5] & 0xFF) << 16) |
                                    (static_cast<uint32_t>(qi[7] & 0xFF) << 24);
                *reinterpret_cast<uint2*>(qa8 + static_cast<size_t>(t) * K + k0 + 8 * g) = make_uint2(lo, hi);
            }
        }
        if (valid && (hl & 1) == 0) {
            const int c = k0 / CHUNK;
            scales[(static_cast<size_t>(mt) * nchunk + c) * TILE_ROWS + r] =
                make_uint2(__float_as_uint(d), static_cast<uint32_t>(s));
            const float ma = __fmul_rn(d, static_cast<float>(s));
            const float mhi = tf32_rna(ma);
            const float mlo = tf32_rna(__fsub_rn(ma, mhi));
            uint8_t* t0 = am + (static_cast<size_t>(mt) * nsb + sb) * (2 * TF32_TILE_BYTES);
            *reinterpret_cast<float*>(t0 + tf32_tile_byte(r, c & 7)) = mhi;
            *reinterpret_cast<float*>(t0 + TF32_TILE_BYTES + tf32_tile_byte(r, c & 7)) = mlo;
            if (fm != nullptr && t < ftn)
                fm[(static_cast<size_t>(sb) * 8 + (c & 7)) * FT_MAX_M + t] = ma;
        }
        t += st_t;
        sb += st_sb;
        if (t >= Mp) {
            t -= Mp;
            ++sb;
        }
    }
}

}  // namespace

cudaError_t launch_quantize_act(const float* x, int M, int K, int ldx, void* qa, void* scales, cudaStream_t s)
{
    const int Mp = ceil_div(M, TILE_ROWS) * TILE_ROWS;
    const long long warps = (static_cast<long long>(Mp) * (K / QK_K) + 1) / 2;   // one half-warp per item
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (nsm <= 0)
        nsm = 148;
    // 8 warps per block; up to 8 resident blocks per SM worth of grid, grid-stride beyond.
    long long blocks = (warps + 7) / 8;
    const long long cap = static_cast<long long>(nsm) * 8;
    if (blocks > cap)
        blocks = cap;
    const int vec4 = ((ldx % 4) == 0 && (reinterpret_cast<uintptr_t>(x) % 16) == 0) ? 1 : 0;
    const ActPlanes ap = act_planes(M, K);
    uint8_t* sc = static_cast<uint8_t*>(scales);
    count_launch();
    return launch_dependent(
        quantize_act_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), s, x, M, K, ldx, Mp, vec4,
        static_cast<uint16_t*>(qa), reinterpret_cast<uint2*>(sc + ap.pair_off), sc + ap.am_off,
        ap.i8_bytes ? reinterpret_cast<int8_t*>(static_cast<uint8_t*>(qa) + ap.i8_off) : nullptr,
        ap.tq_bytes ? static_cast<uint8_t*>(qa) + ap.tq_off : nullptr,
        ap.ip_bytes ? reinterpret_cast<float*>(sc + ap.ip_off) : nullptr,
        ap.fm_bytes ? reinterpret_cast<float*>(sc + ap.fm_off) : nullptr, ap.tq_bytes ? ft_n(M) : 0);
}

}  // namespace mmq
