// pack.cu -- registration-time weight repack.
//
// Raw q6_K / q4_K super-blocks -> (1) a code plane of exact f16 integer codes in
// the tensor-core operand tile layout (128 weight rows x 64 values, 128-byte
// swizzle) and (2) a tile-major f32 scale-pair plane, rows >= od zero-filled.
//
// Scale planes are built the way the W_dsc plane is ("r56 - q6_K A-side
// bundle ...", §2.2 and §2.3): exact f16 -> f32 and int -> f32 conversions and
// exactly one f32 multiply (__fmul_rn, never contracted into an FMA), so each
// entry is bit-identical to the scalar product.  The pair per (chunk, row) is
//   q6_K: {d * scales[2(c%8)], d * scales[2(c%8)+1]}   (the r56 float2 pair)
//   q4_K: {d * sc_c, dmin * m_c}                      (the q4_K plane named as the
//          next step in "r58 - q4_K BT spec ...", §5)
// The layout follows the GEMM's consumption window: one tile's 128 rows of one
// chunk are 1 KiB contiguous (the chunk-major principle of r56 §2.2).  Codes are
// unpacked once here instead of in the GEMM's staging (the registration-time
// expansion of r56 §1 / r58 §3.2).
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

template <int TYPE>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t* __restrict__ raw, int od, int id, int Np,
                                                   uint8_t* __restrict__ codes, float2* __restrict__ wscale)
{
    const int nchunk = id / CHUNK;
    const int nkb = id / TILE_K;
    const int nsb = id / QK_K;
    const long long total = static_cast<long long>(Np) * nchunk;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % nchunk);
        const int j = static_cast<int>(i / nchunk);
        const int cc = c & 7;  // chunk within its super-block
        uint32_t h2[16];       // 32 codes as 16 f16 pairs
        float2 w = make_float2(0.0f, 0.0f);
        if (j < od) {
            if (TYPE == 14) {  // q6_K
                const uint8_t* b = raw + (static_cast<size_t>(j) * nsb + (c >> 3)) * Q6K_BYTES;
                const uint8_t* ql = b + 16 * cc;   // values 32cc.. use ql bytes 16cc..16cc+15
                const uint8_t* qh = b + 128 + 8 * cc;
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    const int e0 = 2 * p, e1 = 2 * p + 1;  // values 32cc+e0, 32cc+e1 (e0 even)
                    const unsigned lo = ql[p];
                    const unsigned hb = qh[p >> 1];
                    const int u0 = static_cast<int>((lo & 15u) | (((hb >> (2 * (e0 & 3))) & 3u) << 4));
                    const int u1 = static_cast<int>((lo >> 4) | (((hb >> (2 * (e1 & 3))) & 3u) << 4));
                    h2[p] = half2_bits(u0 - 32, u1 - 32);
                }
                const float d = load_f16_bytes(b + 208);
                const float s0 = static_cast<float>(static_cast<int8_t>(b[192 + 2 * cc]));
                const float s1 = static_cast<float>(static_cast<int8_t>(b[192 + 2 * cc + 1]));
                w = make_float2(__fmul_rn(d, s0), __fmul_rn(d, s1));
            } else {  // q4_K
                const uint8_t* b = raw + (static_cast<size_t>(j) * nsb + (c >> 3)) * Q4K_BYTES;
                const uint8_t* qs = b + 16 + 16 * cc;
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    const unsigned v = qs[p];
                    h2[p] = half2_bits(static_cast<int>(v & 15u), static_cast<int>(v >> 4));
                }
                const float d = load_f16_bytes(b + 0);
                const float dmin = load_f16_bytes(b + 2);
                const float sc = static_cast<float>(q4k_field(b + 4, cc));
                const float m = static_cast<float>(q4k_field(b + 4, 8 + cc));
                w = make_float2(__fmul_rn(d, sc), __fmul_rn(dmin, m));
            }
        } else {
#pragma unroll
            for (int p = 0; p < 16; ++p)
                h2[p] = 0u;
        }
        const int nt = j / TILE_ROWS, r = j % TILE_ROWS;
        const int kb = c >> 1, k0 = (c & 1) * CHUNK;
        uint8_t* tile = codes + (static_cast<size_t>(nt) * nkb + kb) * TILE_BYTES;
#pragma unroll
        for (int u = 0; u < 4; ++u)  // four 16-byte units of 8 codes each
            *reinterpret_cast<uint4*>(tile + tile_byte(r, k0 + 8 * u)) =
                make_uint4(h2[4 * u], h2[4 * u + 1], h2[4 * u + 2], h2[4 * u + 3]);
        wscale[(static_cast<size_t>(nt) * nchunk + c) * TILE_ROWS + r] = w;
    }
}

}  // namespace

cudaError_t launch_pack(int type, const void* raw, int od, int id, void* packed, cudaStream_t s)
{
    const WeightPlanes wp = weight_planes(od, id);
    const int Np = ceil_div(od, TILE_ROWS) * TILE_ROWS;
    const long long total = static_cast<long long>(Np) * (id / CHUNK);
    long long blocks = (total + 255) / 256;
    if (blocks > 65535LL * 8)
        blocks = 65535LL * 8;
    uint8_t* base = static_cast<uint8_t*>(packed);
    float2* ws = reinterpret_cast<float2*>(base + wp.scale_off);
    if (type == 14)
        pack_kernel<14><<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint8_t*>(raw), od, id,
                                                                        Np, base + wp.code_off, ws);
    else
        pack_kernel<12><<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const uint8_t*>(raw), od, id,
                                                                        Np, base + wp.code_off, ws);
    return cudaGetLastError();
}

}  // namespace mmq
