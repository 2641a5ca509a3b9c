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
// Mapping: one warp per (token row, 64-value block); lane l owns values 2l, 2l+1,
// so lanes 0-15 hold chunk 2kb and lanes 16-31 chunk 2kb+1.  Consecutive warps
// take consecutive token rows of one 64-value block, so the 128-byte code rows and
// the 8-byte scale entries they write are contiguous in HBM.
#include <cuda_fp16.h>

#include "mmq_internal.h"

namespace mmq {
namespace {

__device__ __forceinline__ int quant_one(float x, float d)
{
    float r = roundf(__fdiv_rn(x, d));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

__device__ __forceinline__ float tf32_rna(float v)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

__global__ void __launch_bounds__(256) quantize_act_kernel(const float* __restrict__ x, int M, int K, int ldx,
                                                           int Mp, int vec2, uint16_t* __restrict__ qa,
                                                           uint2* __restrict__ scales, uint8_t* __restrict__ am,
                                                           int8_t* __restrict__ qa8)
{
    const int lane = threadIdx.x & 31;
    const int nkb = K / TILE_K;
    const int nchunk = K / CHUNK;
    const long long total = static_cast<long long>(Mp) * nkb;
    const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
         w += stride) {
        const int t = static_cast<int>(w % Mp);
        const int kb = static_cast<int>(w / Mp);
        float x0 = 0.0f, x1 = 0.0f;
        if (t < M) {
            const float* p = x + static_cast<size_t>(t) * ldx + static_cast<size_t>(kb) * TILE_K + 2 * lane;
            if (vec2) {
                const float2 v = __ldcs(reinterpret_cast<const float2*>(p));
                x0 = v.x;
                x1 = v.y;
            } else {
                x0 = __ldcs(p);
                x1 = __ldcs(p + 1);
            }
        }
        float a = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float d = __fdiv_rn(a, 127.0f);
        int q0 = 0, q1 = 0;
        if (d != 0.0f) {
            q0 = quant_one(x0, d);
            q1 = quant_one(x1, d);
        }
        int s = q0 + q1;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);

        const int mt = t / TILE_ROWS, r = t % TILE_ROWS;
        uint8_t* tile = reinterpret_cast<uint8_t*>(qa) + (static_cast<size_t>(mt) * nkb + kb) * TILE_BYTES;
        const uint32_t packed = static_cast<uint32_t>(__half_as_ushort(__int2half_rn(q0))) |
                                (static_cast<uint32_t>(__half_as_ushort(__int2half_rn(q1))) << 16);
        *reinterpret_cast<uint32_t*>(tile + tile_byte(r, 2 * lane)) = packed;
        if (qa8 != nullptr && t < M) {
            int8_t* row8 = qa8 + static_cast<size_t>(t) * K;
            const int k0 = kb * TILE_K + 2 * lane;
            row8[small_pos(k0)] = static_cast<int8_t>(q0);
            row8[small_pos(k0 + 1)] = static_cast<int8_t>(q1);
        }
        if ((lane & 15) == 0) {
            const int c = 2 * kb + (lane >> 4);
            scales[(static_cast<size_t>(mt) * nchunk + c) * TILE_ROWS + r] =
                make_uint2(__float_as_uint(d), static_cast<uint32_t>(s));
            const float ma = __fmul_rn(d, static_cast<float>(s));
            const float hi = tf32_rna(ma);
            const float lo = tf32_rna(__fsub_rn(ma, hi));
            uint8_t* t0 = am + (static_cast<size_t>(mt) * (K / QK_K) + c / 8) * (2 * TF32_TILE_BYTES);
            *reinterpret_cast<float*>(t0 + tf32_tile_byte(r, c & 7)) = hi;
            *reinterpret_cast<float*>(t0 + TF32_TILE_BYTES + tf32_tile_byte(r, c & 7)) = lo;
        }
    }
}

}  // namespace

cudaError_t launch_quantize_act(const float* x, int M, int K, int ldx, void* qa, void* scales, cudaStream_t s)
{
    const int Mp = ceil_div(M, TILE_ROWS) * TILE_ROWS;
    const long long warps = static_cast<long long>(Mp) * (K / TILE_K);
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (nsm <= 0)
        nsm = 148;
    // 8 warps per block; up to 8 resident blocks per SM worth of grid, grid-stride beyond.
    long long blocks = (warps + 7) / 8;
    const long long cap = static_cast<long long>(nsm) * 16;
    if (blocks > cap)
        blocks = cap;
    const int vec2 = ((ldx % 2) == 0 && (reinterpret_cast<uintptr_t>(x) % 8) == 0) ? 1 : 0;
    const ActPlanes ap = act_planes(M, K);
    uint8_t* sc = static_cast<uint8_t*>(scales);
    quantize_act_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        x, M, K, ldx, Mp, vec2, static_cast<uint16_t*>(qa), reinterpret_cast<uint2*>(sc + ap.pair_off),
        sc + ap.am_off, ap.i8_bytes ? reinterpret_cast<int8_t*>(static_cast<uint8_t*>(qa) + ap.i8_off) : nullptr);
    return cudaGetLastError();
}

}  // namespace mmq
