// peaks.cu -- throughput probes on the current GPU (roofline denominators).
// Standalone program: prints one JSON object.
//
//   tcgen05_f16_tflops_n{128,256}: tcgen05.mma kind::f16 (f16 in, f32 accumulate),
//       M=128, K=16, one issuing thread per SM, operands resident in shared memory
//   int8_mma_sync_tops:           legacy warp-level mma.sync m16n8k32 s8 x s8 -> s32
//   ffma_tflops / ffma2_tflops:   scalar fma.rn.f32 and packed fma.rn.f32x2
//   l2_read_gbs:                  repeated reads of a 64 MiB buffer (L2 resident)
//   hbm_read_gbs / hbm_copy_gbs:  reads of / copy between 4 GiB buffers
// Every wait is bounded by the global timer.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstdint>

#include "ptx.cuh"

using namespace mmq;

#define CK(x)                                                                                       \
    do {                                                                                            \
        cudaError_t e_ = (x);                                                                       \
        if (e_ != cudaSuccess) {                                                                    \
            fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
            exit(1);                                                                                \
        }                                                                                           \
    } while (0)

__global__ void __launch_bounds__(128, 1) umma_probe(int iters, int n, unsigned int* err)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t base = raw + pad;
    const uint32_t a_addr = base, b_addr = base + 16384, bar = base + 16384 + 32768, tptr = bar + 8;
    for (int i = threadIdx.x; i < (16384 + 32768) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(tptr, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + 16384 + 32768 + 8);
    if (threadIdx.x == 0) {
        const uint32_t idesc = (n == 256) ? idesc_f16_f32(128, 256) : idesc_f16_f32(128, 128);
        const uint64_t ad = sdesc_k_sw128(a_addr), bd = sdesc_k_sw128(b_addr);
        for (int it = 0; it < iters; ++it) {
            const uint32_t d = tmem + static_cast<uint32_t>((it & 1) * 256);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, 0)) {
            if (globaltimer_ns() - t0 > 2000000000ull) {
                atomicOr(err, 1u);
                break;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

__global__ void imma_probe(int iters, int* out)
{
    int a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 * 5, a3 = a0 * 7, b0 = a0 * 11, b1 = a0 * 13;
    int c[8][4] = {};
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+r"(c[k][0]), "+r"(c[k][1]), "+r"(c[k][2]), "+r"(c[k][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        s += c[k][0] + c[k][1] + c[k][2] + c[k][3];
    if (s == 0x7fffffff)
        out[0] = s;
}

__global__ void ffma_probe(int iters, float* out)
{
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        x[k] = threadIdx.x * 0.001f + k;
    const float a = 0.999f, b = 0.001f;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            x[k] = fmaf(x[k], a, b);
    }
    float s = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        s += x[k];
    if (s == 12345.0f)
        out[0] = s;
}

__global__ void ffma2_probe(int iters, float* out)
{
    uint64_t x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float2 v = make_float2(threadIdx.x * 0.001f + k, k * 0.5f);
        x[k] = *reinterpret_cast<uint64_t*>(&v);
    }
    float2 av = make_float2(0.999f, 0.999f), bv = make_float2(0.001f, 0.001f);
    const uint64_t a = *reinterpret_cast<uint64_t*>(&av), b = *reinterpret_cast<uint64_t*>(&bv);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[k]) : "l"(a), "l"(b));
    }
    float s = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float2 v = *reinterpret_cast<float2*>(&x[k]);
        s += v.x + v.y;
    }
    if (s == 12345.0f)
        out[0] = s;
}

__global__ void read_probe(const uint4* __restrict__ p, size_t n16, int passes, unsigned int* out)
{
    unsigned int acc = 0;
    for (int r = 0; r < passes; ++r)
        for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
             i += static_cast<size_t>(gridDim.x) * blockDim.x) {
            const uint4 v = __ldcg(p + i);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
    if (acc == 0x12345678u)
        out[0] = acc;
}

__global__ void copy_probe(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        __stcs(dst + i, __ldcs(src + i));
}

template <typename F>
static float time_ms(F f, int reps)
{
    cudaEvent_t a, b;
    CK(cudaEventCreate(&a));
    CK(cudaEventCreate(&b));
    f();  // warm-up
    CK(cudaDeviceSynchronize());
    CK(cudaEventRecord(a));
    for (int i = 0; i < reps; ++i)
        f();
    CK(cudaEventRecord(b));
    CK(cudaEventSynchronize(b));
    float ms = 0;
    CK(cudaEventElapsedTime(&ms, a, b));
    CK(cudaGetLastError());
    return ms / reps;
}

int main()
{
    int dev = 0, nsm = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev));
    cudaDeviceProp prop;
    CK(cudaGetDeviceProperties(&prop, dev));
    unsigned int* err;
    int* iout;
    float* fout;
    CK(cudaMalloc(&err, 4));
    CK(cudaMemset(err, 0, 4));
    CK(cudaMalloc(&iout, 4));
    CK(cudaMalloc(&fout, 4));
    printf("{\"gpu\": \"%s\", \"sms\": %d", prop.name, nsm);

    const int smem = 120 * 1024;  // more than half an SM's shared memory: one probe CTA per SM
    CK(cudaFuncSetAttribute(umma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    for (int n : {128, 256}) {
        const int iters = 4096;
        float ms = time_ms([&] { umma_probe<<<nsm, 128, smem>>>(iters, n, err); }, 5);
        double flops = 2.0 * 128 * n * 16 * 4.0 * iters * nsm;
        printf(", \"tcgen05_f16_tflops_n%d\": %.1f", n, flops / (ms * 1e-3) / 1e12);
    }
    {
        const int iters = 2048, blocks = nsm * 8, threads = 256;
        float ms = time_ms([&] { imma_probe<<<blocks, threads>>>(iters, iout); }, 5);
        double ops = 2.0 * 16 * 8 * 32 * 8.0 * iters * (blocks * threads / 32.0);
        printf(", \"int8_mma_sync_tops\": %.1f", ops / (ms * 1e-3) / 1e12);
    }
    {
        const int iters = 8192, blocks = nsm * 8, threads = 256;
        float ms = time_ms([&] { ffma_probe<<<blocks, threads>>>(iters, fout); }, 5);
        double fl = 2.0 * 8 * iters * double(blocks) * threads;
        printf(", \"ffma_tflops\": %.1f", fl / (ms * 1e-3) / 1e12);
        ms = time_ms([&] { ffma2_probe<<<blocks, threads>>>(iters, fout); }, 5);
        fl = 2.0 * 16 * iters * double(blocks) * threads;
        printf(", \"ffma2_tflops\": %.1f", fl / (ms * 1e-3) / 1e12);
    }
    {
        const size_t l2b = 64ull << 20;
        uint4* p;
        CK(cudaMalloc(&p, l2b));
        CK(cudaMemset(p, 1, l2b));
        const int passes = 20;
        float ms = time_ms([&] { read_probe<<<nsm * 4, 512>>>(p, l2b / 16, passes, err); }, 3);
        printf(", \"l2_read_gbs\": %.0f", double(l2b) * passes / (ms * 1e-3) / 1e9);
        CK(cudaFree(p));
    }
    {
        const size_t hb = 4ull << 30;
        uint4 *a, *b;
        CK(cudaMalloc(&a, hb));
        CK(cudaMalloc(&b, hb));
        CK(cudaMemset(a, 1, hb));
        float ms = time_ms([&] { read_probe<<<nsm * 4, 512>>>(a, hb / 16, 1, err); }, 3);
        printf(", \"hbm_read_gbs\": %.0f", double(hb) / (ms * 1e-3) / 1e9);
        ms = time_ms([&] { copy_probe<<<nsm * 4, 512>>>(a, b, hb / 16); }, 3);
        printf(", \"hbm_copy_gbs\": %.0f", 2.0 * double(hb) / (ms * 1e-3) / 1e9);
        CK(cudaFree(a));
        CK(cudaFree(b));
    }
    unsigned int e = 0;
    CK(cudaMemcpy(&e, err, 4, cudaMemcpyDeviceToHost));
    printf(", \"wait_timeouts\": %u}\n", e);
    return 0;
}
