// mmq_internal.h -- constants of the plane layouts and the launchers shared by
// the library's translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

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

// Byte offset of value k (0..7) of row r (0..127) inside one 128 x 8 tf32 operand
// tile: K-major, no swizzle, 8-row x 16-byte core matrices; the two core matrices
// of an 8-row group are adjacent (K-direction stride 128 B), 8-row groups are
// 256 B apart.
__host__ __device__ constexpr int tf32_tile_byte(int r, int k)
{
    return (r >> 3) * 256 + (k >> 2) * 128 + (r & 7) * 16 + (k & 3) * 4;
}
constexpr int TF32_TILE_BYTES = 128 * 8 * 4;

// Token counts up to SMALL_M take the weight-streaming path; for them the prepass
// also writes int8 codes, row-major, each group of 8 values stored in the order
// (0,2,4,6,1,3,5,7) so that a word of low (or high) weight nibbles meets the four
// activation codes it multiplies.
constexpr int SMALL_M = 8;
__host__ __device__ constexpr int small_pos(int k)   // byte position of value k in its row
{
    return (k & ~7) + ((k & 7) >> 1) + 4 * (k & 1);
}

// Token counts up to FT_MAX_M take the few-token GEMM, whose activation operand the
// prepass writes as well: per 64-value k-block, the FT_N = 16*ceil(M/16) token rows of
// hi = rn_f16(s_hi*q) then of lo = rn_f16(s_hi*q - hi + s_lo*q) (s = p*d, split into
// two f16 values s_hi + s_lo; p a power of two per token and super-block), in the
// 128-byte-swizzled operand layout (row t at t*128); 1/p per (super-block, token),
// FT_MAX_M entries per super-block; and the q4_K min-term operand ma = d*ssum per
// (super-block, token, chunk of the super-block), 8 f32 per token.
constexpr int FT_MAX_M = 64;   // MMQ_FT_MAX_M
__host__ __device__ constexpr int ft_n(int M) { return ((M + 15) / 16) * 16; }

struct ActPlanes {       // layout of mmq_quantize_act's outputs
    size_t tile_bytes;   // f16 code tiles (start of the qa buffer)
    size_t i8_off, i8_bytes;       // M <= SMALL_M: int8 codes [M][K] (small_pos order), else 0
    size_t tq_off, tq_bytes;       // M <= FT_MAX_M: hi/lo operand tiles [K/64][2][FT_N rows], else 0
    size_t qa_bytes;     // tiles + int8 plane + hi/lo tiles
    size_t pair_off, pair_bytes;   // {f32 d, i32 ssum} per (token, chunk)
    size_t am_off, am_bytes;       // tf32 hi/lo tiles of d*ssum per (token tile, super-block)
    size_t ip_off, ip_bytes;       // M <= FT_MAX_M: f32 1/p [K/256][FT_MAX_M], else 0
    size_t fm_off, fm_bytes;       // M <= FT_MAX_M: f32 d*ssum [K/256][8][FT_MAX_M], else 0
    size_t scale_bytes;            // pairs + am + 1/p + d*ssum
};
inline ActPlanes act_planes(int M, int K)
{
    const size_t Mp = static_cast<size_t>(ceil_div(M, TILE_ROWS)) * TILE_ROWS;
    ActPlanes a;
    a.tile_bytes = Mp * static_cast<size_t>(K) * 2;
    a.i8_off = a.tile_bytes;
    a.i8_bytes = (M <= SMALL_M) ? static_cast<size_t>(M) * static_cast<size_t>(K) : 0;
    a.tq_off = a.i8_off + a.i8_bytes;
    a.tq_bytes = (M <= FT_MAX_M) ? static_cast<size_t>(K / TILE_K) * 2 * ft_n(M) * 128 : 0;
    a.qa_bytes = a.tq_off + a.tq_bytes;
    a.pair_off = 0;
    a.pair_bytes = Mp * static_cast<size_t>(K / CHUNK) * 8;
    a.am_off = a.pair_bytes;
    a.am_bytes = Mp / TILE_ROWS * static_cast<size_t>(K / QK_K) * 2 * TF32_TILE_BYTES;
    a.ip_off = a.am_off + a.am_bytes;
    a.ip_bytes = (M <= FT_MAX_M) ? static_cast<size_t>(K / QK_K) * FT_MAX_M * 4 : 0;
    a.fm_off = a.ip_off + a.ip_bytes;
    a.fm_bytes = (M <= FT_MAX_M) ? static_cast<size_t>(K / QK_K) * FT_MAX_M * 8 * 4 : 0;
    a.scale_bytes = a.fm_off + a.fm_bytes;
    return a;
}

// Raw blocks re-laid for 16-byte loads (the weight-streaming path): per row, per
// super-block, q4_K [qs 128 | d 2 | dmin 2 | scales 12] = 144 B, q6_K
// [ql 128 | qh 64 | scales 16 | d 2 | zero 14] = 224 B.
constexpr int RAW4_BYTES = 144;
constexpr int RAW6_BYTES = 224;
__host__ __device__ constexpr int raw_block_bytes(int type) { return type == 12 ? RAW4_BYTES : RAW6_BYTES; }

// Compact code plane (the few-token GEMM's weight operand, widened to f16 in tensor
// memory): per (128-row tile, 64-value k-block) CW_WORDS 16-byte words per row, stored
// word-major ([word][row][16 B]) so that the 128 rows of one word are 2048 contiguous
// bytes.  q4_K: words 0, 1 = the 4-bit codes of the k-block's two chunks; q6_K: word w
// = the 16 values of sub-block w of the k-block, one byte 4 (q + 32) each.  Bit and
// byte positions: see pack.cu.
__host__ __device__ constexpr int cw_words(int type) { return type == 12 ? 2 : 4; }
__host__ __device__ constexpr int cw_kblock_bytes(int type) { return cw_words(type) * TILE_ROWS * 16; }
// Sub-block scale plane: per (128-row tile, super-block) 16 bytes per row, [row][16 B]:
// q4_K the 8 six-bit scales sc_c then the 8 mins m_c (one byte each); q6_K the 16 int8
// scales.
constexpr int SC_ROW_BYTES = 16;

struct WeightPlanes {    // layout of mmq_pack_weights' output
    size_t code_off, code_bytes;   // f16 code tiles (scale-folded where exact)
    size_t pair_off, pair_bytes;   // f32 scale pairs per (row, chunk)
    size_t sbd_off, sbd_bytes;     // f32 d per (row, super-block)
    size_t aux_off, aux_bytes;     // q4_K: tf32 hi/lo tiles of dmin*m; q6_K: f32 scales per sub-block
    size_t flag_off, flag_bytes;   // q6_K: word 0 = 1 if codes hold sc*q, word 1 = max |sc|
    size_t raw_off, raw_bytes;     // re-laid raw blocks [od][id/256]
    size_t cw_off, cw_bytes;       // compact codes [row tile][k-block][word][128][16 B]
    size_t sc_off, sc_bytes;       // sub-block scales [row tile][super-block][128][16 B]
    size_t dm_off, dm_bytes;       // q4_K: f32 dmin per (row, super-block) [row tile][super-block][128]; q6_K: 0
    size_t code2_off, code2_bytes; // q6_K: second f16 tile 16*sc*(h-2) of unfolded codes (zero when folded); q4_K: 0
    size_t total;
};
inline WeightPlanes weight_planes(int type, int od, int id)
{
    const size_t Np = static_cast<size_t>(ceil_div(od, TILE_ROWS)) * TILE_ROWS;
    const size_t nsb = static_cast<size_t>(id / QK_K);
    WeightPlanes w;
    w.code_off = 0;
    w.code_bytes = Np * static_cast<size_t>(id) * 2;
    w.pair_off = w.code_off + w.code_bytes;
    w.pair_bytes = Np * static_cast<size_t>(id / CHUNK) * 8;
    w.sbd_off = w.pair_off + w.pair_bytes;
    w.sbd_bytes = Np * nsb * 4;
    w.aux_off = w.sbd_off + w.sbd_bytes;
    w.aux_bytes = Np * nsb * 64;   // q4_K: 2 x 8 tf32; q6_K: 16 f32
    w.flag_off = w.aux_off + w.aux_bytes;
    w.flag_bytes = 256;
    w.raw_off = w.flag_off + w.flag_bytes;
    w.raw_bytes = static_cast<size_t>(od) * nsb * static_cast<size_t>(raw_block_bytes(type));
    w.cw_off = w.raw_off + ((w.raw_bytes + 255) / 256) * 256;
    w.cw_bytes = (Np / TILE_ROWS) * static_cast<size_t>(id / TILE_K) * cw_kblock_bytes(type);
    w.sc_off = w.cw_off + w.cw_bytes;
    w.sc_bytes = Np * nsb * SC_ROW_BYTES;
    w.dm_off = w.sc_off + w.sc_bytes;
    w.dm_bytes = type == 12 ? Np * nsb * 4 : 0;
    w.code2_off = w.dm_off + w.dm_bytes;
    w.code2_bytes = type == 14 ? Np * static_cast<size_t>(id) * 2 : 0;
    w.total = w.code2_off + w.code2_bytes;
    return w;
}

// ---------------------------------------------------------------- launchers
// Every kernel launch of the library adds to one process-wide counter
// (mmq_launch_count); count_launch is called once per launch attempt.
void count_launch();

// The library's sticky device error word (api.cu): its device address on the
// current device (looked up once per device), and the host-side read-and-clear
// behind mmq_get_device_error (synchronizes the stream first).
cudaError_t device_error_word(unsigned int** word);
cudaError_t read_and_clear_device_error(cudaStream_t s, unsigned int* value);

// What a tile-GEMM launch's bounded waits use: the error word, the time limit of
// each wait, and (verification only) one operand-ring fill that CTA 0's producer
// leaves out, so that the wait for it runs out (-1: none).
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;
struct WaitCtl {
    unsigned int* err;
    unsigned long long limit_ns;
    int withhold_fill;
};
// The WaitCtl of the next tile-GEMM launch: the default limit and no withheld fill,
// unless mmq_debug_inject_wait_timeout armed a one-shot injection, which this call
// consumes.  *injected tells which.
cudaError_t take_wait_ctl(WaitCtl* wc, bool* injected);
// Arms (fill >= 0) or disarms (fill < 0) the one-shot injection.
void arm_wait_injection(int fill, unsigned long long limit_ns);

// Launches `kernel` with programmatic stream serialization: its CTAs may start while
// the kernel ahead of it on `s` finishes, so the kernel calls grid_dep_wait() before
// it touches memory that an earlier kernel may write (only an L2 prefetch may precede
// the wait).  Returns the launch error.
template <typename... P, typename... A>
cudaError_t launch_dependent_smem(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  A&&... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, cudaStream_t s, A&&... args)
{
    return launch_dependent_smem(kernel, grid, block, 0, s, std::forward<A>(args)...);
}

// Each returns cudaSuccess or the launch error; arguments are already validated.
cudaError_t launch_quantize_act(const float* x, int M, int K, int ldx, void* qa, void* scales,
                                cudaStream_t s);
// Repack od rows: rows [0, od_a) from raw_a and rows [od_a, od) from raw_b (a fused
// pack of two weights sharing their input; a plain pack passes od_a = od).
cudaError_t launch_pack(int type, const void* raw_a, int od_a, const void* raw_b, int od, int id, void* packed,
                        cudaStream_t s);
// ggml-layout blocks -> the layout launch_pack reads (src == dst allowed).
cudaError_t launch_convert_ggml(int type, const void* src, size_t nblocks, void* dst, cudaStream_t s);

enum GemmMode { GEMM_Y = 0, GEMM_DOTS = 1 };
// Weight-streaming GEMM for M <= SMALL_M (raw blocks x int8 codes, dp4a).
cudaError_t launch_gemm_small(int type, const void* packed, int od, int id, const void* qa, const void* scales,
                              int M, float* Y, int ldy, cudaStream_t s, const char** path_label);
// Super-block-accumulating GEMM (Y only; q6_K: returns at once for plain codes).
cudaError_t launch_gemm_sb(int type, const void* packed, int od, int id, const void* qa, const void* scales, int M,
                           float* Y, int ldy, cudaStream_t s, const WaitCtl& wc);
// Which kernel takes Y for M > SMALL_M: 0 = the super-block kernel when its tiles
// fill the GPU, else the chunk kernel; 1 = the chunk kernel; 2 = the super-block
// kernel (q6_K plain codes always go to the chunk kernel).
void select_large_m_kernel(int which);
int large_m_kernel();
cudaError_t launch_gemm(int type, GemmMode mode, const void* packed, int od, int id, const void* qa,
                        const void* scales, int M, float* out, int ldy, cudaStream_t s,
                        const char** path_label);
// Few-token GEMM (M <= FT_MAX_M, Y only): compact codes widened in shared memory, the
// prepass's hi/lo token operand, one TMEM accumulator per super-block.
cudaError_t launch_gemm_ft(int type, const void* packed, int od, int id, const void* qa, const void* scales,
                           int M, float* Y, int ldy, cudaStream_t s, const WaitCtl& wc, bool allow_cluster,
                           const char** path_label);


}  // namespace mmq
