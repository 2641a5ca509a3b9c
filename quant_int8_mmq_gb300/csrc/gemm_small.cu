// gemm_small.cu -- weight-streaming q6_K / q4_K x q8 GEMM for a few tokens
// (M <= SMALL_M): the decode and tail shapes, where the tile GEMM would leave most
// SMs idle and the weights, read once, are the whole cost.
//
// What it computes is the q6_K/q4_K formula in its plain per-chunk order
// (32-value chunk c of weight row j and token t):
//   q4_K: Y += d_a * (dsc * I) - ma * dmn,  I = sum q * q_a  (q the 4-bit code),
//         dsc = d * sc_c, dmn = dmin * m_c, ma = d_a * ssum
//   q6_K: Y += d_a * (dsc0 * I_0 + dsc1 * I_1), I_h = sum (q - 32) * q_a over the
//         16-value half h, dsc_h = d * scales[2(c % 8) + h]
// with exact integer dots (dp4a on packed int8 codes) and the f32 scale products
// formed exactly as the repack's pair plane forms them (f16 -> f32 and int -> f32
// conversions, one f32 multiply each).  This is the small-M weight-streaming
// variant the pages rank first after the prefill path (the decode / tail shapes),
// built from the pages' formula ("r56 - q6_K A-side bundle ...", §2.2; "r58 - q4_K
// BT spec ...", §5).
//
// Data: the packed buffer's raw plane (blocks re-laid so that a chunk's codes are
// one aligned 16-byte load, q6_K's high bits one 8-byte load) and the prepass's
// int8 code plane (small_pos order: a word of low or high nibbles of 4 bytes meets
// the four activation codes it multiplies, no byte shuffles).  Bytes read per weight
// value: 0.5625 (q4_K) / 0.875 (q6_K, 14 pad bytes per 224-byte block).
//
// Mapping: one 64-thread CTA (128 for q6_K at M <= 2) per group of R weight rows; its
// threads split the row's 32-value chunks (thread i takes chunks i, i + THREADS, ...),
// every token of the call in registers, and each thread issues the loads of all R rows
// before it computes, so many short CTAs per SM keep the weight stream in flight.  A
// CTA whose rows span at most 16 KB first prefetches them to L2 in one bulk operation.
// The kernel is a dependent launch: its CTAs may start while the kernel ahead (the
// prepass, or another GEMM) finishes, issue that prefetch, and wait for it before they
// read anything an earlier kernel writes.  Partial sums are reduced with a fixed
// butterfly per warp and then in warp order through shared memory, so the result does
// not depend on scheduling.
#include <cuda_fp16.h>

#include "mmq_internal.h"
#include "ptx.cuh"

namespace mmq {
namespace {

// Warps per CTA: 2, except 4 for q6_K at one or two tokens (measured on GB300 with the
// weights streamed from HBM: q6_K 4097x11008 M = 2 15.3 -> 13.2 us with 4; M = 1 equal;
// q4_K and M = 4, 8 as fast or faster with 2, slower with 8).
__host__ __device__ constexpr int small_warps(int type, int mt) { return (type == 14 && mt <= 2) ? 4 : 2; }
constexpr int UNR = 1;             // chunk iterations whose loads are issued together
constexpr int ROWS_FEW = 4;        // rows per CTA for MT <= 2
constexpr int ROWS_MANY = 4;       // rows per CTA for MT > 2
// Largest row-group range a CTA prefetches to L2 in one bulk operation.  Measured on
// GB300 with the weights streamed from HBM (8 rotated copies): the prefetch helps at
// id = 4096 (9-14 KB per CTA; q6_K 32000x4096 M = 1: 25.8 -> 22.9 us, q4_K 11008x4096:
// 6.8 -> 6.3 us) and hurts at q6_K id = 11008 (38.5 KB: 10.0 -> 12.4 us), where the
// demand loads queue behind it.
constexpr uint32_t PREFETCH_MAX_BYTES = 16384;

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
}

// Six-bit field f (0..15) of the 12 q4_K scale bytes read as one little-endian
// 96-bit word (fields 0-7: sc, 8-15: m); w0..w2 hold bytes 0-3, 4-7, 8-11.
__device__ __forceinline__ int q4k_field6(uint32_t w0, uint32_t w1, uint32_t w2, int f)
{
    const int bit = 6 * f;
    const uint64_t lo = static_cast<uint64_t>(w0) | (static_cast<uint64_t>(w1) << 32);
    uint64_t v;
    if (bit < 64) {
        v = lo >> bit;
        if (bit > 58)
            v |= static_cast<uint64_t>(w2) << (64 - bit);
    } else {
        v = static_cast<uint64_t>(w2) >> (bit - 64);
    }
    return static_cast<int>(v & 63u);
}

// q6_K: the four packed codes (q - 32) of the even or odd values of 8-value group
// `i` of a chunk, from the low-nibble word and the group's 16 high-bit bits.
__device__ __forceinline__ void q6k_group(uint32_t ql_word, uint32_t h16, uint32_t& even, uint32_t& odd)
{
    // byte k of w = nibble k of h16 = the 2-bit highs of values 2k (bits 0-1) and 2k+1 (bits 2-3)
    const uint32_t w = __byte_perm(h16 & 0x0F0Fu, (h16 >> 4) & 0x0F0Fu, 0x5140);
    const uint32_t qe = (ql_word & 0x0F0F0F0Fu) | ((w & 0x03030303u) << 4);
    const uint32_t qo = ((ql_word >> 4) & 0x0F0F0F0Fu) | (((w >> 2) & 0x03030303u) << 4);
    even = __vsub4(qe, 0x20202020u);
    odd = __vsub4(qo, 0x20202020u);
}

// q4_K at 5 to 8 tokens forms each row's scale products and int8 code words once per
// chunk rather than once per token.  Measured on GB300 (weights streamed from HBM) over
// ten q4_K shapes: 1-8 % faster at 5 tokens (one shape, 32000x4096, 2 % slower); at 3-4
// tokens the change went either way by shape (-26 % to +17 %), and q6_K was 0-7 % slower
// at every token count, so those keep the per-token form.
template <int TYPE, int MT, int R, int WARPS = small_warps(TYPE, MT), int THREADS = WARPS * 32,
          bool HOIST = (TYPE == 12 && MT == 8)>
__global__ void __launch_bounds__(THREADS) gemm_small_kernel(const uint8_t* __restrict__ raw, int od, int id,
                                                             const int8_t* __restrict__ qa8,
                                                             const uint2* __restrict__ pairs, int M,
                                                             float* __restrict__ Y, int ldy)
{
    constexpr int RB = raw_block_bytes(TYPE);
    __shared__ float part[WARPS][R * MT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunk = id / CHUNK;
    const int nsb = id / QK_K;
    const int j0 = blockIdx.x * R;
    if (tid == 0) {
        // The CTA's rows are contiguous in the raw plane: a short range is put in flight
        // to L2 at once, so that the per-chunk loads below wait on L2, not on HBM.  A
        // prefetch changes no value, so it is issued before the wait on the kernel
        // ahead: the weight stream starts while that kernel finishes.
        const int rows = min(R, od - j0);
        const uint32_t bytes = static_cast<uint32_t>(rows * nsb * RB);
        if (bytes <= PREFETCH_MAX_BYTES)
            bulk_prefetch_l2(raw + static_cast<size_t>(j0) * nsb * RB, bytes);
    }
    grid_dep_launch();
    grid_dep_wait();

    float acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < MT; ++t)
            acc[r][t] = 0.0f;

    for (int c0 = tid; c0 < nchunk; c0 += UNR * THREADS) {
        // the weights of all R rows for UNR chunk iterations first (the stream) ...
        uint4 w0u[UNR][R];
        uint4 w1u[UNR][R];   // q4_K: d | dmin | scales[12];  q6_K: qh (x, y), scale pair (z), d (w)
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int c = min(c0 + u * THREADS, nchunk - 1);   // past the end: a repeat, unused
            const int b = c >> 3, cc = c & 7;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int j = min(j0 + r, od - 1);           // rows past od repeat the last one, unused
                const uint8_t* blk = raw + (static_cast<size_t>(j) * nsb + b) * RB;
                w0u[u][r] = __ldcs(reinterpret_cast<const uint4*>(blk + 16 * cc));
                if (TYPE == 12) {
                    w1u[u][r] = __ldg(reinterpret_cast<const uint4*>(blk + 128));
                } else {
                    const uint2 qh = __ldcs(reinterpret_cast<const uint2*>(blk + 128 + 8 * cc));
                    w1u[u][r] =
                        make_uint4(qh.x, qh.y, __ldg(reinterpret_cast<const unsigned short*>(blk + 192 + 2 * cc)),
                                   __ldg(reinterpret_cast<const unsigned short*>(blk + 208)));
                }
            }
        }
        // ... then, per chunk iteration, every token against every row
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int c = c0 + u * THREADS;
            if (c >= nchunk)
                break;
            const int cc = c & 7;
            const uint4(&w0)[R] = w0u[u];
            const uint4(&w1)[R] = w1u[u];
            if constexpr (HOIST) {
                // each row's scale products and int8 code words once per chunk, then every
                // token against them (the same operations per (row, token) as below)
                float s0[R], s1[R];
                uint32_t qa_[R][4], qb_[R][4];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (TYPE == 12) {
                        const uint4 meta = w1[r];
                        const float d = f16_bits_to_f32(meta.x), dmin = f16_bits_to_f32(meta.x >> 16);
                        s0[r] = __fmul_rn(d, static_cast<float>(q4k_field6(meta.y, meta.z, meta.w, cc)));
                        s1[r] = __fmul_rn(dmin, static_cast<float>(q4k_field6(meta.y, meta.z, meta.w, 8 + cc)));
                        const uint32_t qw[4] = {w0[r].x, w0[r].y, w0[r].z, w0[r].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            qa_[r][i] = qw[i] & 0x0F0F0F0Fu;
                            qb_[r][i] = (qw[i] >> 4) & 0x0F0F0F0Fu;
                        }
                    } else {
                        const float d = f16_bits_to_f32(w1[r].w);
                        s0[r] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w1[r].z & 0xFFu)));
                        s1[r] = __fmul_rn(d, static_cast<float>(static_cast<int8_t>((w1[r].z >> 8) & 0xFFu)));
                        q6k_group(w0[r].x, w1[r].x & 0xFFFFu, qa_[r][0], qb_[r][0]);
                        q6k_group(w0[r].y, w1[r].x >> 16, qa_[r][1], qb_[r][1]);
                        q6k_group(w0[r].z, w1[r].y & 0xFFFFu, qa_[r][2], qb_[r][2]);
                        q6k_group(w0[r].w, w1[r].y >> 16, qa_[r][3], qb_[r][3]);
                    }
                }
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t >= M)
                        break;
                    const uint4* ap = reinterpret_cast<const uint4*>(qa8 + static_cast<size_t>(t) * id + c * CHUNK);
                    const uint4 v0 = __ldg(ap), v1 = __ldg(ap + 1);
                    const uint32_t a[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                    const uint2 pr = __ldg(pairs + static_cast<size_t>(c) * TILE_ROWS + t);
                    const float da = __uint_as_float(pr.x);
                    const float ma = __fmul_rn(da, static_cast<float>(static_cast<int>(pr.y)));
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (TYPE == 12) {
                            int I = 0;
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                I = __dp4a(static_cast<int>(qa_[r][i]), static_cast<int>(a[2 * i]), I);
                                I = __dp4a(static_cast<int>(qb_[r][i]), static_cast<int>(a[2 * i + 1]), I);
                            }
                            acc[r][t] = fmaf(da, __fmul_rn(s0[r], static_cast<float>(I)), acc[r][t]);
                            acc[r][t] = fmaf(-ma, s1[r], acc[r][t]);
                        } else {
                            int I0 = 0, I1 = 0;
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                I0 = __dp4a(static_cast<int>(qa_[r][i]), static_cast<int>(a[2 * i]), I0);
                                I0 = __dp4a(static_cast<int>(qb_[r][i]), static_cast<int>(a[2 * i + 1]), I0);
                                I1 = __dp4a(static_cast<int>(qa_[r][2 + i]), static_cast<int>(a[4 + 2 * i]), I1);
                                I1 = __dp4a(static_cast<int>(qb_[r][2 + i]), static_cast<int>(a[4 + 2 * i + 1]), I1);
                            }
                            const float v = fmaf(s1[r], static_cast<float>(I1), __fmul_rn(s0[r], static_cast<float>(I0)));
                            acc[r][t] = fmaf(da, v, acc[r][t]);
                        }
                    }
                }
                continue;
            }
            // per token: its 8 code words of this chunk, d_a and d_a * ssum, against every row
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= M)
                    break;
                const uint4* ap = reinterpret_cast<const uint4*>(qa8 + static_cast<size_t>(t) * id + c * CHUNK);
                const uint4 v0 = __ldg(ap), v1 = __ldg(ap + 1);
                const uint32_t a[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                const uint2 pr = __ldg(pairs + static_cast<size_t>(c) * TILE_ROWS + t);
                const float da = __uint_as_float(pr.x);
                const float ma = __fmul_rn(da, static_cast<float>(static_cast<int>(pr.y)));
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (TYPE == 12) {
                        const uint4 meta = w1[r];
                        const float d = f16_bits_to_f32(meta.x), dmin = f16_bits_to_f32(meta.x >> 16);
                        const float dsc = __fmul_rn(d, static_cast<float>(q4k_field6(meta.y, meta.z, meta.w, cc)));
                        const float dmn =
                            __fmul_rn(dmin, static_cast<float>(q4k_field6(meta.y, meta.z, meta.w, 8 + cc)));
                        const uint32_t qw[4] = {w0[r].x, w0[r].y, w0[r].z, w0[r].w};
                        int I = 0;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            I = __dp4a(static_cast<int>(qw[i] & 0x0F0F0F0Fu), static_cast<int>(a[2 * i]), I);
                            I = __dp4a(static_cast<int>((qw[i] >> 4) & 0x0F0F0F0Fu), static_cast<int>(a[2 * i + 1]), I);
                        }
                        acc[r][t] = fmaf(da, __fmul_rn(dsc, static_cast<float>(I)), acc[r][t]);
                        acc[r][t] = fmaf(-ma, dmn, acc[r][t]);
                    } else {
                        const float d = f16_bits_to_f32(w1[r].w);
                        const float dsc0 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(w1[r].z & 0xFFu)));
                        const float dsc1 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>((w1[r].z >> 8) & 0xFFu)));
                        uint32_t ev[4], odd[4];
                        q6k_group(w0[r].x, w1[r].x & 0xFFFFu, ev[0], odd[0]);
                        q6k_group(w0[r].y, w1[r].x >> 16, ev[1], odd[1]);
                        q6k_group(w0[r].z, w1[r].y & 0xFFFFu, ev[2], odd[2]);
                        q6k_group(w0[r].w, w1[r].y >> 16, ev[3], odd[3]);
                        int I0 = 0, I1 = 0;
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            I0 = __dp4a(static_cast<int>(ev[i]), static_cast<int>(a[2 * i]), I0);
                            I0 = __dp4a(static_cast<int>(odd[i]), static_cast<int>(a[2 * i + 1]), I0);
                            I1 = __dp4a(static_cast<int>(ev[2 + i]), static_cast<int>(a[4 + 2 * i]), I1);
                            I1 = __dp4a(static_cast<int>(odd[2 + i]), static_cast<int>(a[4 + 2 * i + 1]), I1);
                        }
                        const float u = fmaf(dsc1, static_cast<float>(I1), __fmul_rn(dsc0, static_cast<float>(I0)));
                        acc[r][t] = fmaf(da, u, acc[r][t]);
                    }
                }
            }
        }
    }

    // Fixed butterfly within each warp, then the warps' partials in warp order.
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            float v = acc[r][t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0)
                part[warp][r * MT + t] = v;
        }
    }
    __syncthreads();
    if (tid < R * MT) {
        const int r = tid / MT, t = tid % MT;
        float v = part[0][tid];
#pragma unroll
        for (int w = 1; w < WARPS; ++w)
            v += part[w][tid];
        const int j = j0 + r;
        if (t < M && j < od)
            Y[static_cast<size_t>(t) * ldy + j] = v;
    }
}

template <int TYPE, int MT>
cudaError_t launch_typed(const uint8_t* raw, int od, int id, const int8_t* qa8, const uint2* pairs, int M, float* Y,
                         int ldy, cudaStream_t s)
{
    constexpr int R = (MT <= 2) ? ROWS_FEW : ROWS_MANY;
    count_launch();
    return launch_dependent(gemm_small_kernel<TYPE, MT, R>, dim3(ceil_div(od, R)), dim3(small_warps(TYPE, MT) * 32), s,
                            raw, od, id, qa8, pairs, M, Y, ldy);
}

template <int TYPE>
cudaError_t launch_mt(const uint8_t* raw, int od, int id, const int8_t* qa8, const uint2* pairs, int M, float* Y,
                      int ldy, cudaStream_t s)
{
    if (M <= 1)
        return launch_typed<TYPE, 1>(raw, od, id, qa8, pairs, M, Y, ldy, s);
    if (M <= 2)
        return launch_typed<TYPE, 2>(raw, od, id, qa8, pairs, M, Y, ldy, s);
    if (M <= 4)
        return launch_typed<TYPE, 4>(raw, od, id, qa8, pairs, M, Y, ldy, s);
    return launch_typed<TYPE, 8>(raw, od, id, qa8, pairs, M, Y, ldy, s);
}

}  // namespace

cudaError_t launch_gemm_small(int type, const void* packed, int od, int id, const void* qa, const void* scales,
                              int M, float* Y, int ldy, cudaStream_t s, const char** path_label)
{
    static_assert(SMALL_M == 8, "token-count dispatch above covers 1..8");
    const WeightPlanes wp = weight_planes(type, od, id);
    const ActPlanes ap = act_planes(M, id);
    const uint8_t* raw = static_cast<const uint8_t*>(packed) + wp.raw_off;
    const int8_t* qa8 = reinterpret_cast<const int8_t*>(static_cast<const uint8_t*>(qa) + ap.i8_off);
    const uint2* pairs = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(scales) + ap.pair_off);
    if (path_label)
        *path_label = type == 14 ? "q6_K: weight-streaming path (M <= 8): raw blocks x int8 codes, dp4a integer dots, "
                                   "f32 scales per chunk, CTA per weight-row group"
                                 : "q4_K: weight-streaming path (M <= 8): raw blocks x int8 codes, dp4a integer dots, "
                                   "f32 scales and min term per chunk, CTA per weight-row group";
    if (type == 14)
        return launch_mt<14>(raw, od, id, qa8, pairs, M, Y, ldy, s);
    return launch_mt<12>(raw, od, id, qa8, pairs, M, Y, ldy, s);
}

}  // namespace mmq
