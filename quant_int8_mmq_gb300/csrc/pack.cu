// pack.cu -- registration-time weight repack.
//
// Raw q6_K / q4_K super-blocks -> the planes the GEMM streams (rows >= od zero):
//  codes  f16 integer codes in the tensor-core operand tile layout (128 weight
//         rows x 64 values, 128-byte swizzle) with the integer sub-block scale
//         folded in, exactly:
//           q4_K: sc_c * q  (|.| <= 63 * 15 = 945)
//           q6_K: sc * q    when every |sc| of the tensor is <= 64 (|.| <= 2048);
//                 else sc * l, l the low 4 bits of q + 32 (|.| <= 1920), and
//  codes2 (q6_K) the second tile 16 * sc * (h - 2), h the high 2 bits of q + 32
//         (a multiple of 16 of magnitude <= 4096, exact), so that
//         codes + codes2 = sc * (l + 16 (h - 2)) = sc * q; zero when folded
//  pairs  tile-major f32 scale pairs per (row, chunk), built the way the W_dsc
//         plane is ("r56 - q6_K A-side bundle ...", §2.2 and §2.3): exact f16 -> f32
//         and int -> f32 conversions and exactly one f32 multiply (__fmul_rn, never
//         contracted into an FMA):
//           q6_K {d * scales[2(c%8)], d * scales[2(c%8)+1]}   (the r56 float2 pair)
//           q4_K {d * sc_c, dmin * m_c}     (the q4_K plane "r58 - q4_K BT spec ...",
//                                           §5 names as the next step)
//  sbd    f32 d per (row, super-block): the factor applied once per super-block
//         when the codes carry the integer scale.
//  aux    q4_K: the min-term operand dmn = dmin * m (exact f32, <= 17 significant
//               bits) split exactly into tf32 hi + lo, in 128 x 8 tf32 tiles per
//               (row tile, super-block);
//         q6_K: the 16 int8 sub-block scales as f32 per (row, super-block), used
//               when the codes are not folded.
//  flag   q6_K: word 0 = 1 if the codes are folded, word 1 = max |sc|.
//  dm     q4_K: f32 dmin per (row, super-block), the factor of the few-token GEMM's
//         min term (which multiplies it by m_c on the fly).
//  raw    the raw blocks re-laid for 16-byte loads by the weight-streaming path
//         (few tokens): codes first, then the scale bytes; q4_K keeps 144 bytes,
//         q6_K is padded with zeros to 224.
// The layout follows the GEMM's consumption window: one tile's rows of one chunk
// or super-block are contiguous (the chunk-major principle of r56 §2.2), and the
// codes are unpacked once here instead of in the GEMM's staging (the
// registration-time expansion of r56 §1 and r58 §3.2).
//
// Bit mapping inside ql/qh/qs and the scales[12] packing: the documented reading
// (see include/mmq.h).  One thread per (padded row j, chunk c).
#include <cuda_fp16.h>

#include "mmq_internal.h"

namespace mmq {
namespace {

__device__ __forceinline__ float load_f16_bytes(const uint8_t* p)
{
    const unsigned short bits = static_cast<unsigned short>(p[0] | (static_cast<unsigned>(p[1]) << 8));
    return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ uint32_t half2_bits(int a, int b)
{
    return static_cast<uint32_t>(__half_as_ushort(__int2half_rn(a))) |
           (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(b))) << 16);
}

__device__ __forceinline__ float tf32_rna(float v)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// Six-bit field f (0..15) of the 12 scale bytes read as one little-endian 96-bit word.
__device__ __forceinline__ int q4k_field(const uint8_t* sc12, int f)
{
    const int bit = 6 * f;
    const int byte = bit >> 3, sh = bit & 7;
    unsigned v = static_cast<unsigned>(sc12[byte]) >> sh;
    if (sh > 2)
        v |= static_cast<unsigned>(sc12[byte + 1]) << (8 - sh);
    return static_cast<int>(v & 63u);
}

// The raw blocks of the weight being packed: rows [0, od_a) from a, rows from od_a on
// from b (a fused pack of two weights that share their input), each row-major with
// nsb blocks per row; a plain pack has od_a = od.
struct RawRows {
    const uint8_t* a;
    const uint8_t* b;
    int od_a, nsb, bytes;
    __device__ __forceinline__ const uint8_t* block(int j, int sb) const
    {
        return j < od_a ? a + (static_cast<size_t>(j) * nsb + sb) * bytes
                        : b + (static_cast<size_t>(j - od_a) * nsb + sb) * bytes;
    }
    __device__ __forceinline__ const uint8_t* block(long long linear) const   // row-major block index
    {
        return block(static_cast<int>(linear / nsb), static_cast<int>(linear % nsb));
    }
};

// q6_K: max |sc| over the tensor -> flag word 1 (atomicMax); word 0 is set later.
__global__ void q6k_scale_scan(const RawRows raw, long long nblocks, unsigned int* flag)
{
    unsigned int mx = 0;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < nblocks * 16;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int v = static_cast<int8_t>(raw.block(i >> 4)[192 + (i & 15)]);
        const unsigned int a = static_cast<unsigned int>(v < 0 ? -v : v);
        mx = a > mx ? a : mx;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0 && mx)
        atomicMax(flag + 1, mx);
}

template <int TYPE>
__global__ void __launch_bounds__(256) pack_kernel(const RawRows raw, int od, int id, int Np,
                                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ codes2,
                                                   float2* __restrict__ pairs,
                                                   float* __restrict__ sbd, uint8_t* __restrict__ aux,
                                                   float* __restrict__ dm, unsigned int* __restrict__ flag)
{
    const int nchunk = id / CHUNK;
    const int nkb = id / TILE_K;
    const int nsb = id / QK_K;
    const bool fold = (TYPE == 12) || (flag[1] <= 64u);
    if (TYPE == 14 && blockIdx.x == 0 && threadIdx.x == 0)
        flag[0] = fold ? 1u : 0u;
    const long long total = static_cast<long long>(Np) * nchunk;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % nchunk);
        const int j = static_cast<int>(i / nchunk);
        const int cc = c & 7;       // chunk within its super-block
        const int sb = c >> 3;
        const int nt = j / TILE_ROWS, r = j % TILE_ROWS;
        uint32_t h2[16];            // 32 codes as 16 f16 pairs
        uint32_t g2[16];            // q6_K second tile (zero unless unfolded)
        float2 w = make_float2(0.0f, 0.0f);
        if (j < od) {
            if (TYPE == 14) {  // q6_K
                const uint8_t* b = raw.block(j, sb);
                const uint8_t* ql = b + 16 * cc;   // values 32cc.. use ql bytes 16cc..16cc+15
                const uint8_t* qh = b + 128 + 8 * cc;
                const int s0 = static_cast<int8_t>(b[192 + 2 * cc]);
                const int s1 = static_cast<int8_t>(b[192 + 2 * cc + 1]);
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    const int e0 = 2 * p, e1 = 2 * p + 1;  // values 32cc+e0, 32cc+e1
                    const unsigned lo = ql[p];
                    const unsigned hb = qh[p >> 1];
                    const int l0 = static_cast<int>(lo & 15u), l1 = static_cast<int>(lo >> 4);
                    const int hh0 = static_cast<int>((hb >> (2 * (e0 & 3))) & 3u);
                    const int hh1 = static_cast<int>((hb >> (2 * (e1 & 3))) & 3u);
                    const int sc = p < 8 ? s0 : s1;  // values 0..15 of the chunk use s0
                    if (fold) {
                        h2[p] = half2_bits(sc * (l0 + 16 * hh0 - 32), sc * (l1 + 16 * hh1 - 32));
                        g2[p] = 0u;
                    } else {
                        h2[p] = half2_bits(sc * l0, sc * l1);
                        g2[p] = half2_bits(16 * sc * (hh0 - 2), 16 * sc * (hh1 - 2));
                    }
                }
                const float d = load_f16_bytes(b + 208);
                w = make_float2(__fmul_rn(d, static_cast<float>(s0)), __fmul_rn(d, static_cast<float>(s1)));
                if (cc == 0) {
                    sbd[(static_cast<size_t>(nt) * nsb + sb) * TILE_ROWS + r] = d;
                    float* scp = reinterpret_cast<float*>(aux + (static_cast<size_t>(nt) * nsb + sb) * 8192);
#pragma unroll
                    for (int s = 0; s < 16; ++s)
                        scp[s * TILE_ROWS + r] = static_cast<float>(static_cast<int8_t>(b[192 + s]));
                }
            } else {  // q4_K
                const uint8_t* b = raw.block(j, sb);
                const uint8_t* qs = b + 16 + 16 * cc;
                const int sc = q4k_field(b + 4, cc);
                const int m = q4k_field(b + 4, 8 + cc);
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    const unsigned v = qs[p];
                    h2[p] = half2_bits(sc * static_cast<int>(v & 15u), sc * static_cast<int>(v >> 4));
                    g2[p] = 0u;
                }
                const float d = load_f16_bytes(b + 0);
                const float dmin = load_f16_bytes(b + 2);
                const float dmn = __fmul_rn(dmin, static_cast<float>(m));
                w = make_float2(__fmul_rn(d, static_cast<float>(sc)), dmn);
                if (cc == 0) {
                    sbd[(static_cast<size_t>(nt) * nsb + sb) * TILE_ROWS + r] = d;
                    dm[(static_cast<size_t>(nt) * nsb + sb) * TILE_ROWS + r] = dmin;
                }
                const float hi = tf32_rna(dmn);
                const float lo = __fsub_rn(dmn, hi);  // <= 6 significant bits: exact in tf32
                uint8_t* t0 = aux + (static_cast<size_t>(nt) * nsb + sb) * (2 * TF32_TILE_BYTES);
                *reinterpret_cast<float*>(t0 + tf32_tile_byte(r, cc)) = hi;
                *reinterpret_cast<float*>(t0 + TF32_TILE_BYTES + tf32_tile_byte(r, cc)) = lo;
            }
        } else {
#pragma unroll
            for (int p = 0; p < 16; ++p)
                h2[p] = g2[p] = 0u;
            if (cc == 0)
                sbd[(static_cast<size_t>(nt) * nsb + sb) * TILE_ROWS + r] = 0.0f;
            if (TYPE == 14) {
                if (cc == 0) {
                    float* scp = reinterpret_cast<float*>(aux + (static_cast<size_t>(nt) * nsb + sb) * 8192);
#pragma unroll
                    for (int s = 0; s < 16; ++s)
                        scp[s * TILE_ROWS + r] = 0.0f;
                }
            } else {
                if (cc == 0)
                    dm[(static_cast<size_t>(nt) * nsb + sb) * TILE_ROWS + r] = 0.0f;
                uint8_t* t0 = aux + (static_cast<size_t>(nt) * nsb + sb) * (2 * TF32_TILE_BYTES);
                *reinterpret_cast<float*>(t0 + tf32_tile_byte(r, cc)) = 0.0f;
                *reinterpret_cast<float*>(t0 + TF32_TILE_BYTES + tf32_tile_byte(r, cc)) = 0.0f;
            }
        }
        const int kb = c >> 1, k0 = (c & 1) * CHUNK;
        uint8_t* tile = codes + (static_cast<size_t>(nt) * nkb + kb) * TILE_BYTES;
#pragma unroll
        for (int u = 0; u < 4; ++u)  // four 16-byte units of 8 codes each
            *reinterpret_cast<uint4*>(tile + tile_byte(r, k0 + 8 * u)) =
                make_uint4(h2[4 * u], h2[4 * u + 1], h2[4 * u + 2], h2[4 * u + 3]);
        if (TYPE == 14) {
            uint8_t* tile2 = codes2 + (static_cast<size_t>(nt) * nkb + kb) * TILE_BYTES;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(tile2 + tile_byte(r, k0 + 8 * u)) =
                    make_uint4(g2[4 * u], g2[4 * u + 1], g2[4 * u + 2], g2[4 * u + 3]);
        }
        pairs[(static_cast<size_t>(nt) * nchunk + c) * TILE_ROWS + r] = w;
    }
}

// Raw blocks -> the re-laid raw plane, one 32-bit output word per thread.
//   q4_K in [d 2 | dmin 2 | scales 12 | qs 128]  -> out [qs 128 | d, dmin, scales 16]
//   q6_K in [ql 128 | qh 64 | scales 16 | d 2]   -> out [the same 210 | zeros 14]
template <int TYPE>
__global__ void __launch_bounds__(256) raw_relayout_kernel(const RawRows raw, long long nblocks,
                                                           uint32_t* __restrict__ out)
{
    constexpr int OUTW = raw_block_bytes(TYPE) / 4;
    const long long words = nblocks * OUTW;
    for (long long w = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; w < words;
         w += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long b = w / OUTW;
        const int o = static_cast<int>(w - b * OUTW) * 4;
        const uint8_t* src = raw.block(b);
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int ob = o + k;
            int sb;
            if (TYPE == 12)
                sb = ob < 128 ? ob + 16 : ob - 128;
            else
                sb = ob < Q6K_BYTES ? ob : -1;
            const uint32_t byte = sb >= 0 ? static_cast<uint32_t>(src[sb]) : 0u;
            v |= byte << (8 * k);
        }
        out[w] = v;
    }
}

// Compact codes and sub-block scales for the few-token GEMM, one thread per (padded row
// j, k-block kb), the rows of a tile on consecutive threads.  Bit positions are chosen
// so that the GEMM's converter turns each 32-bit word into f16 pairs with a mask and
// an OR of the exponent 0x6400 (1024 + the field), no per-value shifts:
//   q4_K nibble word (code q) of a 32-value chunk: value 8u + 2p + h (u, p = 0..3,
//     h = 0, 1) at bit 4p + 16h of byte group u (bytes 4u..4u+3);
//   q6_K word of a 16-value sub-block: one byte 4 (q + 32) per value (the six-bit code
//     at bits 2..7, so that 1024 + 4 (q + 32) is exact), value 4u + o (u, o = 0..3) in
//     32-bit word u at byte 2 (o & 1) + (o >> 1): bytes 0, 2 hold values 4u, 4u + 1 and
//     bytes 1, 3 values 4u + 2, 4u + 3, each pair one mask (or a shift and a mask) away
//     from its f16x2 form.
template <int TYPE>
__global__ void __launch_bounds__(256) compact_kernel(const RawRows raw, int od, int id, int Np,
                                                      uint4* __restrict__ cw, uint4* __restrict__ scp)
{
    constexpr int W = cw_words(TYPE);
    const int nkb = id / TILE_K;
    const int nsb = id / QK_K;
    const long long total = static_cast<long long>(Np) * nkb;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i % TILE_ROWS);
        const long long tk = i / TILE_ROWS;
        const int kb = static_cast<int>(tk % nkb);
        const int nt = static_cast<int>(tk / nkb);
        const int j = nt * TILE_ROWS + r;
        const int sb = kb >> 2;
        uint32_t word[W][4];
#pragma unroll
        for (int w = 0; w < W; ++w)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                word[w][u] = 0u;
        static_assert(TYPE == 12 || W == 4, "q6_K: one word per 16-value sub-block");
        uint32_t sc4[4] = {0u, 0u, 0u, 0u};
        if (j < od) {
            const uint8_t* b = raw.block(j, sb);
            for (int hc = 0; hc < 2; ++hc) {
                const int e0 = 64 * (kb & 3) + 32 * hc;      // first value of the chunk in its block
                for (int i2 = 0; i2 < 32; ++i2) {
                    const int e = e0 + i2;
                    if constexpr (TYPE == 12) {
                        const int u = i2 >> 3, pp = (i2 & 7) >> 1, h = i2 & 1;
                        const uint32_t lo4 = (b[16 + e / 2] >> (4 * (e & 1))) & 15u;
                        word[hc][u] |= lo4 << (4 * pp + 16 * h);
                    } else {
                        const uint32_t lo4 = (b[e / 2] >> (4 * (e & 1))) & 15u;
                        const uint32_t hi2 = (b[128 + e / 4] >> (2 * (e & 3))) & 3u;
                        const int i16 = i2 & 15, o = i16 & 3;      // value 4 u6 + o of the sub-block
                        const int u6 = i16 >> 2, byte = 2 * (o & 1) + (o >> 1);
                        word[2 * hc + (i2 >> 4)][u6] |= (4u * (lo4 | (hi2 << 4))) << (8 * byte);
                    }
                }
            }
            if ((kb & 3) == 0) {
                uint8_t v[16];
                if (TYPE == 12) {
                    for (int f = 0; f < 16; ++f) {   // the 16 six-bit fields, little-endian
                        const int bit = 6 * f, byte = bit >> 3, sh = bit & 7;
                        unsigned x = static_cast<unsigned>(b[4 + byte]) >> sh;
                        if (sh > 2)
                            x |= static_cast<unsigned>(b[4 + byte + 1]) << (8 - sh);
                        v[f] = static_cast<uint8_t>(x & 63u);
                    }
                } else {
                    for (int f = 0; f < 16; ++f)
                        v[f] = b[192 + f];
                }
                for (int q = 0; q < 4; ++q)
                    sc4[q] = static_cast<uint32_t>(v[4 * q]) | (static_cast<uint32_t>(v[4 * q + 1]) << 8) |
                             (static_cast<uint32_t>(v[4 * q + 2]) << 16) | (static_cast<uint32_t>(v[4 * q + 3]) << 24);
            }
        }
        uint4* dst = cw + (static_cast<size_t>(nt) * nkb + kb) * (W * TILE_ROWS);
#pragma unroll
        for (int w = 0; w < W; ++w)
            dst[w * TILE_ROWS + r] = make_uint4(word[w][0], word[w][1], word[w][2], word[w][3]);
        if ((kb & 3) == 0)
            scp[(static_cast<size_t>(nt) * nsb + sb) * TILE_ROWS + r] = make_uint4(sc4[0], sc4[1], sc4[2], sc4[3]);
    }
}

}  // namespace

cudaError_t launch_pack(int type, const void* raw_a, int od_a, const void* raw_b, int od, int id, void* packed,
                        cudaStream_t s)
{
    RawRows rb;
    rb.a = static_cast<const uint8_t*>(raw_a);
    rb.b = static_cast<const uint8_t*>(raw_b);
    rb.od_a = od_a;
    rb.nsb = id / QK_K;
    rb.bytes = type == 12 ? Q4K_BYTES : Q6K_BYTES;
    const WeightPlanes wp = weight_planes(type, od, id);
    const int Np = ceil_div(od, TILE_ROWS) * TILE_ROWS;
    const long long total = static_cast<long long>(Np) * (id / CHUNK);
    long long blocks = (total + 255) / 256;
    if (blocks > 65535LL * 8)
        blocks = 65535LL * 8;
    uint8_t* base = static_cast<uint8_t*>(packed);
    unsigned int* flag = reinterpret_cast<unsigned int*>(base + wp.flag_off);
    cudaError_t e = cudaMemsetAsync(flag, 0, wp.flag_bytes, s);
    if (e != cudaSuccess)
        return e;
    float2* pairs = reinterpret_cast<float2*>(base + wp.pair_off);
    float* sbd = reinterpret_cast<float*>(base + wp.sbd_off);
    if (type == 14) {
        const long long nblocks = static_cast<long long>(od) * (id / QK_K);
        long long sblocks = (nblocks * 16 + 255) / 256;
        if (sblocks > 4096)
            sblocks = 4096;
        count_launch();
        q6k_scale_scan<<<static_cast<unsigned>(sblocks), 256, 0, s>>>(rb, nblocks, flag);
        count_launch();
        pack_kernel<14><<<static_cast<unsigned>(blocks), 256, 0, s>>>(rb, od, id, Np, base + wp.code_off,
                                                                        base + wp.code2_off, pairs, sbd,
                                                                        base + wp.aux_off, nullptr, flag);
    } else {
        count_launch();
        pack_kernel<12><<<static_cast<unsigned>(blocks), 256, 0, s>>>(rb, od, id, Np, base + wp.code_off, nullptr,
                                                                        pairs, sbd, base + wp.aux_off,
                                                                        reinterpret_cast<float*>(base + wp.dm_off),
                                                                        flag);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const long long nblocks = static_cast<long long>(od) * (id / QK_K);
    const long long rwords = nblocks * (raw_block_bytes(type) / 4);
    long long rblocks = (rwords + 255) / 256;
    if (rblocks > 65535LL * 8)
        rblocks = 65535LL * 8;
    uint32_t* rout = reinterpret_cast<uint32_t*>(base + wp.raw_off);
    count_launch();
    if (type == 14)
        raw_relayout_kernel<14><<<static_cast<unsigned>(rblocks), 256, 0, s>>>(rb, nblocks, rout);
    else
        raw_relayout_kernel<12><<<static_cast<unsigned>(rblocks), 256, 0, s>>>(rb, nblocks, rout);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const long long citems = static_cast<long long>(Np) * (id / TILE_K);
    long long cblocks = (citems + 255) / 256;
    if (cblocks > 65535LL * 8)
        cblocks = 65535LL * 8;
    uint4* cw = reinterpret_cast<uint4*>(base + wp.cw_off);
    uint4* scp = reinterpret_cast<uint4*>(base + wp.sc_off);
    count_launch();
    if (type == 14)
        compact_kernel<14><<<static_cast<unsigned>(cblocks), 256, 0, s>>>(rb, od, id, Np, cw, scp);
    else
        compact_kernel<12><<<static_cast<unsigned>(cblocks), 256, 0, s>>>(rb, od, id, Np, cw, scp);
    return cudaGetLastError();
}

}  // namespace mmq
