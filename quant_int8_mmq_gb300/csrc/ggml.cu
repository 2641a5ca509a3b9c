// ggml.cu -- GGUF interop: q4_K / q6_K super-blocks in the public ggml (llama.cpp)
// block layout rewritten into the layout mmq_pack_weights reads.
//
// Both layouts put d, dmin, the scales and the code arrays at the same byte offsets
// (q4_K: d@0 dmin@2 scales[12]@4 qs[128]@16; q6_K: ql[128]@0 qh[64]@128
// scales[16]@192 d@208); they differ in where each of the 256 codes sits inside the
// code arrays and in how q4_K packs its eight 6-bit scales and mins:
//   ggml q4_K: value 64j + l (l < 32) is the low nibble of qs[32j + l], value
//              64j + 32 + l its high nibble; sub-block s < 4 keeps sc and m in the low
//              6 bits of S[s] and S[s + 4]; s >= 4 has their low 4 bits in S[s + 4]
//              (sc low nibble, m high nibble) and their top 2 bits in the top bits of
//              S[s - 4] (sc) and S[s] (m).
//   ggml q6_K: value 128n + 32p + l has its low 4 bits in nibble p/2 of
//              ql[64n + 32(p%2) + l] and its high 2 bits at bit 2p of qh[32n + l]; the
//              scales array is indexed by value / 16 in both layouts.
//   target:    value e in nibble e%2 of qs/ql[e/2], q6_K high bits at bit 2(e%4) of
//              qh[e/4], q4_K fields as one little-endian 96-bit word of sixteen 6-bit
//              fields (sc_0..7, m_0..7).
// One warp per block: the block is staged in shared memory first, so the
// conversion may run in place.
#include "mmq_internal.h"

namespace mmq {
namespace {

constexpr int WARPS = 8;
constexpr int STAGE = 224;   // bytes staged per warp (>= 210)

template <int TYPE>
__global__ void __launch_bounds__(WARPS * 32) ggml_to_reading_kernel(const uint8_t* src, size_t nblocks, uint8_t* dst)
{
    constexpr int NB = (TYPE == 12) ? Q4K_BYTES : Q6K_BYTES;
    __shared__ uint8_t stage[WARPS][STAGE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* in = stage[warp];
    for (size_t b = static_cast<size_t>(blockIdx.x) * WARPS + warp; b < nblocks;
         b += static_cast<size_t>(gridDim.x) * WARPS) {
        const uint8_t* s = src + b * NB;
        uint8_t* d = dst + b * NB;
        for (int i = lane; i < NB; i += 32)
            in[i] = s[i];
        __syncwarp();
        if (TYPE == 12) {
            // codes: output byte 16 + i holds values 2i (low nibble) and 2i + 1
            uint8_t code_out[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = lane + 32 * k;
                uint8_t o = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int v = 2 * i + h, j = v / 64, l = v % 64;
                    const int code = (l < 32) ? (in[16 + 32 * j + l] & 15) : (in[16 + 32 * j + l - 32] >> 4);
                    o |= static_cast<uint8_t>(code << (4 * h));
                }
                code_out[k] = o;
            }
            // scales: lane 0 unpacks the 16 six-bit fields and repacks them
            uint8_t sc_out[12];
            if (lane == 0) {
                const uint8_t* S = in + 4;
                unsigned long long lo = 0;   // bits 0..63 of the 96-bit word
                unsigned int hi = 0;         // bits 64..95
                for (int f = 0; f < 16; ++f) {
                    const int s_ = f & 7;
                    int val;
                    if (f < 8)
                        val = (s_ < 4) ? (S[s_] & 63) : ((S[s_ + 4] & 15) | ((S[s_ - 4] >> 6) << 4));
                    else
                        val = (s_ < 4) ? (S[s_ + 4] & 63) : ((S[s_ + 4] >> 4) | ((S[s_] >> 6) << 4));
                    const int bit = 6 * f;
                    for (int t = 0; t < 6; ++t) {
                        if ((val >> t) & 1) {
                            const int bb = bit + t;
                            if (bb < 64)
                                lo |= 1ull << bb;
                            else
                                hi |= 1u << (bb - 64);
                        }
                    }
                }
                for (int k = 0; k < 8; ++k)
                    sc_out[k] = static_cast<uint8_t>(lo >> (8 * k));
                for (int k = 0; k < 4; ++k)
                    sc_out[8 + k] = static_cast<uint8_t>(hi >> (8 * k));
            }
            __syncwarp();          // every lane has read `in` before anything is written
#pragma unroll
            for (int k = 0; k < 4; ++k)
                d[16 + lane + 32 * k] = code_out[k];
            if (lane < 4)
                d[lane] = in[lane];                    // d, dmin
            if (lane == 0)
                for (int k = 0; k < 12; ++k)
                    d[4 + k] = sc_out[k];
        } else {
            // ql: output byte i (0..127) = low 4 bits of values 2i, 2i + 1;
            // qh: output byte 128 + i (0..63) = high 2 bits of values 4i .. 4i + 3
            auto code6 = [&](int v) -> int {
                const int n = v / 128, w = v % 128, p = w / 32, l = w % 32;
                const int byte = in[64 * n + 32 * (p % 2) + l];
                const int low = (p / 2) ? (byte >> 4) : (byte & 15);
                const int high = (in[128 + 32 * n + l] >> (2 * p)) & 3;
                return low | (high << 4);
            };
            uint8_t out[6];
#pragma unroll
            for (int k = 0; k < 6; ++k) {
                const int o = lane + 32 * k;     // output byte 0..191
                uint8_t val = 0;
                if (o < 128) {
                    val = static_cast<uint8_t>((code6(2 * o) & 15) | ((code6(2 * o + 1) & 15) << 4));
                } else {
                    const int i = o - 128;
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        val |= static_cast<uint8_t>(((code6(4 * i + t) >> 4) & 3) << (2 * t));
                }
                out[k] = val;
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 6; ++k)
                d[lane + 32 * k] = out[k];
            if (lane < 18)
                d[192 + lane] = in[192 + lane];        // scales, d
        }
        __syncwarp();              // the stage is reused by the warp's next block
    }
}

}  // namespace

cudaError_t launch_convert_ggml(int type, const void* src, size_t nblocks, void* dst, cudaStream_t s)
{
    if (nblocks == 0)
        return cudaSuccess;
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    size_t grid = (nblocks + WARPS - 1) / WARPS;
    const size_t cap = static_cast<size_t>(nsm > 0 ? nsm : 1) * 16;
    if (grid > cap)
        grid = cap;
    count_launch();
    const uint8_t* in = static_cast<const uint8_t*>(src);
    uint8_t* out = static_cast<uint8_t*>(dst);
    if (type == 12)
        ggml_to_reading_kernel<12><<<static_cast<unsigned>(grid), WARPS * 32, 0, s>>>(in, nblocks, out);
    else
        ggml_to_reading_kernel<14><<<static_cast<unsigned>(grid), WARPS * 32, 0, s>>>(in, nblocks, out);
    return cudaGetLastError();
}

}  // namespace mmq
