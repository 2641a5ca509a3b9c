// api.cu -- the extern "C" entry points declared in include/mmq.h.
//
// Every call validates its arguments on the host first (no CUDA call before an
// argument error is returned), then checks that the current device is an sm_103
// part, then launches on the caller's stream.  Nothing here allocates device
// memory.
#include <atomic>
#include <cstdint>

#include "mmq.h"
#include "mmq_internal.h"
#include "route.h"

namespace mmq {
namespace {
std::atomic<unsigned long long> g_launches{0};

// The sticky device error word of the whole library (one per device the library
// is loaded on).  Kernels receive its address in their arguments; nothing else
// names it in device code.
__device__ unsigned int g_device_error_word;
std::atomic<unsigned int*> g_error_word_addr[64];   // per device ordinal, looked up once

// One-shot wait-timeout injection (verification only): fill index, wait limit.
std::atomic<int> g_inject_fill{-1};
std::atomic<unsigned long long> g_inject_limit_ns{0};
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

cudaError_t device_error_word(unsigned int** word)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64) {
        unsigned int* c = g_error_word_addr[dev].load(std::memory_order_acquire);
        if (c != nullptr) {
            *word = c;
            return cudaSuccess;
        }
    }
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_device_error_word);
    if (e != cudaSuccess)
        return e;
    *word = static_cast<unsigned int*>(a);
    if (dev >= 0 && dev < 64)
        g_error_word_addr[dev].store(*word, std::memory_order_release);
    return cudaSuccess;
}

cudaError_t read_and_clear_device_error(cudaStream_t s, unsigned int* value)
{
    *value = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return e;
    e = cudaMemcpyFromSymbol(value, g_device_error_word, sizeof(unsigned int));
    if (e != cudaSuccess)
        return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(unsigned int));
}

void arm_wait_injection(int fill, unsigned long long limit_ns)
{
    g_inject_limit_ns.store(limit_ns);
    g_inject_fill.store(fill < 0 ? -1 : fill);
}

cudaError_t take_wait_ctl(WaitCtl* wc, bool* injected)
{
    const cudaError_t e = device_error_word(&wc->err);
    if (e != cudaSuccess)
        return e;
    const int fill = g_inject_fill.exchange(-1);
    *injected = fill >= 0;
    wc->withhold_fill = fill;
    wc->limit_ns = *injected ? g_inject_limit_ns.load() : WAIT_LIMIT_NS;
    return cudaSuccess;
}
}  // namespace mmq

namespace {

std::atomic<const char*> g_last_path{"none"};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_k(int K) { return K >= mmq::QK_K && K <= MMQ_MAX_ID && (K % mmq::QK_K) == 0; }

// The verdict per device ordinal is cached (0 unknown, 1 sm_103, 2 other): a
// device's compute capability does not change while the process runs.
std::atomic<unsigned char> g_dev_ok[64];

mmq_status check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_UNSUPPORTED;
    }
    if (dev >= 0 && dev < 64) {
        const unsigned char v = g_dev_ok[dev].load(std::memory_order_relaxed);
        if (v != 0)
            return v == 1 ? MMQ_OK : MMQ_ERR_UNSUPPORTED;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_UNSUPPORTED;
    }
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < 64)
        g_dev_ok[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
    return ok ? MMQ_OK : MMQ_ERR_UNSUPPORTED;
}

mmq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MMQ_OK : MMQ_ERR_CUDA; }

// After a pack: for q6_K, read the fold flag (FLAG word 0) back once, so that GEMM
// calls on this buffer choose their kernel without a device read.  The read waits for
// the stream.  While the stream is being captured into a graph nothing is read and any
// earlier record for the address is dropped (GEMMs then take the codes as folded).
cudaError_t note_fold_state(mmq_type t, const void* packed, int od, int id, cudaStream_t s)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || t != MMQ_Q6_K)
        return e;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess)
        return e;
    if (cap != cudaStreamCaptureStatusNone) {
        mmq::note_packed(dev, packed, static_cast<int>(t), od, id, -1);
        return cudaSuccess;
    }
    const mmq::WeightPlanes wp = mmq::weight_planes(static_cast<int>(t), od, id);
    uint32_t flag = 0;
    e = cudaMemcpyAsync(&flag, static_cast<const uint8_t*>(packed) + wp.flag_off, sizeof(flag),
                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    mmq::note_packed(dev, packed, static_cast<int>(t), od, id, e == cudaSuccess ? (flag != 0 ? 1 : 0) : -1);
    return e;
}

mmq_status check_weight_shape(mmq_type t, int od, int id)
{
    if (t != MMQ_Q4_K && t != MMQ_Q6_K)
        return MMQ_ERR_ARG;
    if (od < 1 || od > MMQ_MAX_OD || !valid_k(id))
        return MMQ_ERR_SHAPE;
    return MMQ_OK;
}

// Token counts up to MMQ_SMALL_M go to the weight-streaming kernel, whose cost grows with
// M (its integer dots are issue-bound), unless the weight is large enough that the
// few-token kernel, whose cost hardly depends on M, is faster.  The crossovers were
// measured on GB300 over q4_K 4096x4096 / 11008x4096 and q6_K 4096x4096 / 4097x11008 /
// 32000x4096 at M = 2..8, and retaken at M = 3..6 after the few-token kernel's promotion
// went to f32x2 pairs (q6_K 4097x11008 M = 4: 17.9 us streaming, 16.8 few-token).
bool takes_streaming_path(mmq_type t, int od, int id, int M)
{
    if (M > mmq::SMALL_M)
        return false;
    const long long w = static_cast<long long>(od) * id;
    constexpr long long W24 = 1ll << 24, W25 = 1ll << 25;
    if (t == MMQ_Q4_K)
        return !(w >= W24 && (M >= 7 || (M >= 5 && w >= W25)));
    return !(w >= W25 && M >= 4);
}

mmq_status gemm_common(mmq_type t, mmq::GemmMode mode, const void* packed, int od, int id, const void* qa,
                       const void* scales, int M, float* out, int ldy, mmq_stream_t s)
{
    mmq_status st = check_weight_shape(t, od, id);
    if (st != MMQ_OK)
        return st;
    if (!packed || !qa || !scales || !out)
        return MMQ_ERR_ARG;
    if (M < 1 || M > MMQ_MAX_M)
        return MMQ_ERR_SHAPE;
    if (mode == mmq::GEMM_Y && ldy < od)
        return MMQ_ERR_ARG;
    if (!aligned(packed, 16) || !aligned(qa, 16) || !aligned(scales, 16) || !aligned(out, 4))
        return MMQ_ERR_ALIGN;
    st = check_device();
    if (st != MMQ_OK)
        return st;
    const char* label = nullptr;
    const cudaError_t e =
        (mode == mmq::GEMM_Y && takes_streaming_path(t, od, id, M) && mmq::large_m_kernel() != 4)
            ? mmq::launch_gemm_small(static_cast<int>(t), packed, od, id, qa, scales, M, out, ldy,
                                     reinterpret_cast<cudaStream_t>(s), &label)
            : mmq::launch_gemm(static_cast<int>(t), mode, packed, od, id, qa, scales, M, out, ldy,
                               reinterpret_cast<cudaStream_t>(s), &label);
    if (label)
        g_last_path.store(label);
    return from_cuda(e);
}

}  // namespace

extern "C" {

mmq_status mmq_act_plane_bytes(int M, int K, size_t* qa_bytes, size_t* scale_bytes)
{
    if (!qa_bytes || !scale_bytes)
        return MMQ_ERR_ARG;
    if (M < 1 || M > MMQ_MAX_M || !valid_k(K))
        return MMQ_ERR_SHAPE;
    const mmq::ActPlanes p = mmq::act_planes(M, K);
    *qa_bytes = p.qa_bytes;
    *scale_bytes = p.scale_bytes;
    return MMQ_OK;
}

mmq_status mmq_quantize_act(const float* x, int M, int K, int ldx, void* qa, void* scales, mmq_stream_t s)
{
    if (!x || !qa || !scales)
        return MMQ_ERR_ARG;
    if (M < 1 || M > MMQ_MAX_M || !valid_k(K))
        return MMQ_ERR_SHAPE;
    if (ldx < K)
        return MMQ_ERR_ARG;
    if (!aligned(x, 4) || !aligned(qa, 16) || !aligned(scales, 16))
        return MMQ_ERR_ALIGN;
    const mmq_status st = check_device();
    if (st != MMQ_OK)
        return st;
    return from_cuda(mmq::launch_quantize_act(x, M, K, ldx, qa, scales, reinterpret_cast<cudaStream_t>(s)));
}

mmq_status mmq_packed_weight_bytes(mmq_type t, int od, int id, size_t* bytes)
{
    if (!bytes)
        return MMQ_ERR_ARG;
    const mmq_status st = check_weight_shape(t, od, id);
    if (st != MMQ_OK)
        return st;
    *bytes = mmq::weight_planes(static_cast<int>(t), od, id).total;
    return MMQ_OK;
}

mmq_status mmq_packed_weight_layout(mmq_type t, int od, int id, size_t offsets[MMQ_NUM_WEIGHT_PLANES],
                                    size_t sizes[MMQ_NUM_WEIGHT_PLANES])
{
    if (!offsets || !sizes)
        return MMQ_ERR_ARG;
    const mmq_status st = check_weight_shape(t, od, id);
    if (st != MMQ_OK)
        return st;
    const mmq::WeightPlanes w = mmq::weight_planes(static_cast<int>(t), od, id);
    offsets[MMQ_PLANE_CODES] = w.code_off;
    sizes[MMQ_PLANE_CODES] = w.code_bytes;
    offsets[MMQ_PLANE_PAIRS] = w.pair_off;
    sizes[MMQ_PLANE_PAIRS] = w.pair_bytes;
    offsets[MMQ_PLANE_SBD] = w.sbd_off;
    sizes[MMQ_PLANE_SBD] = w.sbd_bytes;
    offsets[MMQ_PLANE_AUX] = w.aux_off;
    sizes[MMQ_PLANE_AUX] = w.aux_bytes;
    offsets[MMQ_PLANE_FLAG] = w.flag_off;
    sizes[MMQ_PLANE_FLAG] = w.flag_bytes;
    offsets[MMQ_PLANE_RAW] = w.raw_off;
    sizes[MMQ_PLANE_RAW] = w.raw_bytes;
    offsets[MMQ_PLANE_CW] = w.cw_off;
    sizes[MMQ_PLANE_CW] = w.cw_bytes;
    offsets[MMQ_PLANE_DM] = w.dm_off;
    sizes[MMQ_PLANE_DM] = w.dm_bytes;
    offsets[MMQ_PLANE_CODES2] = w.code2_off;
    sizes[MMQ_PLANE_CODES2] = w.code2_bytes;
    offsets[MMQ_PLANE_SC] = w.sc_off;
    sizes[MMQ_PLANE_SC] = w.sc_bytes;
    return MMQ_OK;
}

mmq_status mmq_act_ft_layout(int M, int K, size_t* tq_offset, size_t* tq_bytes, size_t* ip_offset,
                             size_t* ip_bytes, size_t* fm_offset, size_t* fm_bytes)
{
    if (!tq_offset || !tq_bytes || !ip_offset || !ip_bytes || !fm_offset || !fm_bytes)
        return MMQ_ERR_ARG;
    if (M < 1 || M > MMQ_MAX_M || !valid_k(K))
        return MMQ_ERR_SHAPE;
    const mmq::ActPlanes p = mmq::act_planes(M, K);
    *tq_offset = p.tq_bytes ? p.tq_off : 0;
    *tq_bytes = p.tq_bytes;
    *ip_offset = p.ip_bytes ? p.ip_off : 0;
    *ip_bytes = p.ip_bytes;
    *fm_offset = p.fm_bytes ? p.fm_off : 0;
    *fm_bytes = p.fm_bytes;
    return MMQ_OK;
}

mmq_status mmq_act_scale_layout(int M, int K, size_t* pair_offset, size_t* pair_bytes, size_t* am_offset,
                                size_t* am_bytes)
{
    if (!pair_offset || !pair_bytes || !am_offset || !am_bytes)
        return MMQ_ERR_ARG;
    if (M < 1 || M > MMQ_MAX_M || !valid_k(K))
        return MMQ_ERR_SHAPE;
    const mmq::ActPlanes p = mmq::act_planes(M, K);
    *pair_offset = p.pair_off;
    *pair_bytes = p.pair_bytes;
    *am_offset = p.am_off;
    *am_bytes = p.am_bytes;
    return MMQ_OK;
}

mmq_status mmq_pack_weights(mmq_type t, const void* raw_blocks, int od, int id, void* packed, mmq_stream_t s)
{
    mmq_status st = check_weight_shape(t, od, id);
    if (st != MMQ_OK)
        return st;
    if (!raw_blocks || !packed)
        return MMQ_ERR_ARG;
    if (!aligned(packed, 16))
        return MMQ_ERR_ALIGN;
    st = check_device();
    if (st != MMQ_OK)
        return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    cudaError_t e = mmq::launch_pack(static_cast<int>(t), raw_blocks, od, raw_blocks, od, id, packed, cs);
    if (e == cudaSuccess)
        e = note_fold_state(t, packed, od, id, cs);
    return from_cuda(e);
}

mmq_status mmq_pack_weights_fused(mmq_type t, const void* raw_a, int od_a, const void* raw_b, int od_b, int id,
                                  void* packed, mmq_stream_t s)
{
    if (t != MMQ_Q4_K && t != MMQ_Q6_K)
        return MMQ_ERR_ARG;
    if (od_a < 1 || od_b < 1 || static_cast<long long>(od_a) + od_b > MMQ_MAX_OD)
        return MMQ_ERR_SHAPE;
    mmq_status st = check_weight_shape(t, od_a + od_b, id);
    if (st != MMQ_OK)
        return st;
    if (!raw_a || !raw_b || !packed)
        return MMQ_ERR_ARG;
    if (!aligned(packed, 16))
        return MMQ_ERR_ALIGN;
    st = check_device();
    if (st != MMQ_OK)
        return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    cudaError_t e = mmq::launch_pack(static_cast<int>(t), raw_a, od_a, raw_b, od_a + od_b, id, packed, cs);
    if (e == cudaSuccess)
        e = note_fold_state(t, packed, od_a + od_b, id, cs);
    return from_cuda(e);
}

mmq_status mmq_convert_ggml_blocks(mmq_type t, const void* src, size_t nblocks, void* dst, mmq_stream_t s)
{
    if (t != MMQ_Q4_K && t != MMQ_Q6_K)
        return MMQ_ERR_ARG;
    if (!src || !dst)
        return MMQ_ERR_ARG;
    if (nblocks > (static_cast<size_t>(1) << 40))
        return MMQ_ERR_SHAPE;
    const mmq_status st = check_device();
    if (st != MMQ_OK)
        return st;
    return from_cuda(mmq::launch_convert_ggml(static_cast<int>(t), src, nblocks, dst,
                                              reinterpret_cast<cudaStream_t>(s)));
}

mmq_status mmq_gemm_q6k(const void* packed, int od, int id, const void* qa, const void* scales, int M, float* Y,
                        int ldy, mmq_stream_t s)
{
    return gemm_common(MMQ_Q6_K, mmq::GEMM_Y, packed, od, id, qa, scales, M, Y, ldy, s);
}

mmq_status mmq_gemm_q4k(const void* packed, int od, int id, const void* qa, const void* scales, int M, float* Y,
                        int ldy, mmq_stream_t s)
{
    return gemm_common(MMQ_Q4_K, mmq::GEMM_Y, packed, od, id, qa, scales, M, Y, ldy, s);
}

mmq_status mmq_debug_gemm_dots(mmq_type t, const void* packed, int od, int id, const void* qa, const void* scales,
                               int M, float* dots, mmq_stream_t s)
{
    return gemm_common(t, mmq::GEMM_DOTS, packed, od, id, qa, scales, M, dots, od, s);
}

mmq_status mmq_debug_route(mmq_type t, int od, int id, int M, int fold, int nsm, int* kernel)
{
    mmq_status st = check_weight_shape(t, od, id);
    if (st != MMQ_OK)
        return st;
    if (!kernel || nsm < 1 || fold < -1 || fold > 1)
        return MMQ_ERR_ARG;
    if (M < 1 || M > MMQ_MAX_M)
        return MMQ_ERR_SHAPE;
    if (takes_streaming_path(t, od, id, M))
        *kernel = 0;
    else if (M <= MMQ_FT_MAX_M)
        *kernel = 3;
    else
        *kernel = mmq::prefer_superblock(static_cast<int>(t), od, id, M, nsm, t == MMQ_Q6_K ? fold : 1) ? 2 : 1;
    return MMQ_OK;
}

mmq_status mmq_debug_select_large_m_kernel(int which)
{
    if (which < 0 || which > 4)
        return MMQ_ERR_ARG;
    mmq::select_large_m_kernel(which);
    return MMQ_OK;
}

unsigned long long mmq_launch_count(void) { return mmq::g_launches.load(std::memory_order_relaxed); }

mmq_status mmq_debug_inject_wait_timeout(int fill, unsigned long long limit_ns)
{
    if (fill < 0) {
        mmq::arm_wait_injection(-1, 0);
        return MMQ_OK;
    }
    if (limit_ns < 1000ull || limit_ns > mmq::WAIT_LIMIT_NS)
        return MMQ_ERR_ARG;
    mmq::arm_wait_injection(fill, limit_ns);
    return MMQ_OK;
}

mmq_status mmq_get_device_error(mmq_stream_t s)
{
    const mmq_status st = check_device();
    if (st != MMQ_OK)
        return st;
    unsigned int word = 0;
    const cudaError_t e = mmq::read_and_clear_device_error(reinterpret_cast<cudaStream_t>(s), &word);
    if (e != cudaSuccess)
        return MMQ_ERR_CUDA;
    return word ? MMQ_ERR_TIMEOUT : MMQ_OK;
}

const char* mmq_status_string(mmq_status st)
{
    switch (st) {
    case MMQ_OK: return "MMQ_OK";
    case MMQ_ERR_ARG: return "MMQ_ERR_ARG: invalid argument";
    case MMQ_ERR_SHAPE: return "MMQ_ERR_SHAPE: unsupported shape";
    case MMQ_ERR_ALIGN: return "MMQ_ERR_ALIGN: misaligned pointer";
    case MMQ_ERR_CUDA: return "MMQ_ERR_CUDA: CUDA runtime error";
    case MMQ_ERR_TIMEOUT: return "MMQ_ERR_TIMEOUT: in-kernel wait expired";
    case MMQ_ERR_UNSUPPORTED: return "MMQ_ERR_UNSUPPORTED: no sm_103 device current";
    }
    return "MMQ_ERR_UNKNOWN";
}

const char* mmq_last_path(void) { return g_last_path.load(); }

const char* mmq_version(void) { return "mmq_gb300 0.1.0 (sm_103a, tcgen05 kind::f16 exact-integer MMQ)"; }

}  // extern "C"
