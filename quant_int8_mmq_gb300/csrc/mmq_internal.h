// mmq_internal.h -- constants of the plane layouts and the launchers shared by
// the library's translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace mmq {

constexpr int QK_K = 256;          // values per super-block
constexpr int CHUNK = 32;          // values per activation scale / q4_K scale
constexpr int Q6K_BYTES = 210;
constexpr int Q4K_BYTES = 144;

// Operand tiles: 128 rows x 64 values of f16 = 16 KiB, 128-byte swizzled.
constexpr int TILE_ROWS = 128;
constexpr int TILE_K = 64;
constexpr int TILE_BYTES = TILE_ROWS * TILE_K * 2;

constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Byte offset of value k (0..63) of row r (0..127) inside one operand tile.
__host__ __device__ constexpr int tile_byte(int r, int k)
{
    return r * 128 + (((k >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1);
}

struct ActPlanes {       // layout of mmq_quantize_act's outputs
    size_t qa_bytes, scale_bytes;
};
inline ActPlanes act_planes(int M, int K)
{
    const size_t Mp = static_cast<size_t>(ceil_div(M, TILE_ROWS)) * TILE_ROWS;
    return {Mp * static_cast<size_t>(K) * 2, Mp * static_cast<size_t>(K / CHUNK) * 8};
}

struct WeightPlanes {    // layout of mmq_pack_weights' output
    size_t code_off, code_bytes, scale_off, scale_bytes, total;
};
inline WeightPlanes weight_planes(int od, int id)
{
    const size_t Np = static_cast<size_t>(ceil_div(od, TILE_ROWS)) * TILE_ROWS;
    WeightPlanes w;
    w.code_off = 0;
    w.code_bytes = Np * static_cast<size_t>(id) * 2;
    w.scale_off = w.code_bytes;
    w.scale_bytes = Np * static_cast<size_t>(id / CHUNK) * 8;
    w.total = w.scale_off + w.scale_bytes;
    return w;
}

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error; arguments are already validated.
cudaError_t launch_quantize_act(const float* x, int M, int K, int ldx, void* qa, void* scales,
                                cudaStream_t s);
cudaError_t launch_pack(int type, const void* raw, int od, int id, void* packed, cudaStream_t s);

enum GemmMode { GEMM_Y = 0, GEMM_DOTS = 1 };
cudaError_t launch_gemm(int type, GemmMode mode, const void* packed, int od, int id, const void* qa,
                        const void* scales, int M, float* out, int ldy, cudaStream_t s,
                        const char** path_label);

// Reads and clears the GEMM translation unit's sticky error word (stream-ordered,
// then synchronizes the stream).  *word receives the old value.
cudaError_t gemm_read_and_clear_error(cudaStream_t s, unsigned int* word);

}  // namespace mmq
