// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarriers, bulk async copies
// (global -> shared, completion counted on an mbarrier), tcgen05 tensor-core MMA
// with TMEM accumulators, TMEM loads, and the bounded wait every kernel uses.
#pragma once

#include <cstdint>

namespace mmq {

// Bits of the library's sticky device error word.  The word itself is one
// __device__ variable of the library (api.cu); a kernel that waits receives its
// device address among its arguments, so every kernel sets the same word and
// mmq_get_device_error reads and clears exactly that one.
constexpr unsigned int ERR_WAIT_EXPIRED = 1u;

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps
// until the phase completes or about hint_ns pass, instead of returning at once.
// A sleeping thread issues nothing, so waiting warps leave the issue slots of
// their scheduler to the warps that share it.
__device__ __forceinline__ uint32_t mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok;
}

// Wait until the phase with the given parity has completed.  Gives up (returns
// false) once the sticky error word *err is set by anyone, or after limit_ns of
// global time, in which case it sets ERR_WAIT_EXPIRED in *err itself.  The error
// word and the global timer are first read after 64 unsuccessful polls, so short
// waits cost one or a few try_wait round trips.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, unsigned int* err)
{
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 63u) == 0) {
            if (*reinterpret_cast<volatile unsigned int*>(err) != 0u)
                return false;
            const uint64_t now = globaltimer_ns();
            if (i == 64u)
                t0 = now;
            else if (now - t0 > limit_ns) {
                atomicOr(err, ERR_WAIT_EXPIRED);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the error word, used only to drain a CTA's own copies
// and MMAs in flight before it exits (those always complete): sleeps between polls
// and gives up after limit_ns, setting ERR_WAIT_EXPIRED.
__device__ __forceinline__ void mbar_drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, unsigned int* err)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, ERR_WAIT_EXPIRED);
            return;
        }
    }
}

// Packed f32x2 fused multiply-add: {a.x*b.x + c.x, a.y*b.y + c.y}, one rounding each.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
          "l"(*reinterpret_cast<uint64_t*>(&c)));
    return *reinterpret_cast<float2*>(&d);
}

// ---------------------------------------------------------------- bulk copy
// Plain (non-tensor) bulk copy global -> this CTA's shared memory; the bytes are
// counted on `bar` (complete_tx).  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Prefetch [src, src + bytes) into L2 (no completion tracking); src 16-byte
// aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start before the
// kernel ahead of it on the stream has finished.  grid_dep_wait() returns once that
// kernel has completed and its memory operations are visible; every access to memory
// that an earlier kernel may write comes after it.  grid_dep_launch() lets the next
// such kernel on the stream start once every CTA of this grid has issued it or exited.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives (release) and waits (acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of this CTA's shared address `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(saddr), "r"(rank));
    return out;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
// Named CTA barrier `id` over `nthreads` threads (a multiple of 32; every thread of each
// participating warp arrives).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// The same barrier, also returning the AND of `v` over the participating threads.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool v)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}\n"
        : "=r"(out)
        : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0u;
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes (stride byte
// offset 1024), leading byte offset unused for this layout, descriptor version 1.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address  [0,14)
    d |= static_cast<uint64_t>(16u >> 4) << 16;             // leading offset [16,30)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;           // stride offset  [32,46)
    d |= static_cast<uint64_t>(1u) << 46;                   // version        [46,48)
    d |= static_cast<uint64_t>(2u) << 61;                   // 128B swizzle   [61,64)
    return d;
}

// Instruction descriptor, kind::f16: f16 A and B, f32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n)
{
    return (1u << 4)                                   // D format: f32
           | (0u << 7) | (0u << 10)                    // A, B format: f16
           | (0u << 15) | (0u << 16)                   // A, B K-major
           | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, one 128 x N x 16 step, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Shared-memory descriptor of a 128 x 8 tf32 tile in the no-swizzle K-major core-matrix
// layout (tf32_tile_byte in mmq_internal.h): K-direction core-matrix stride 128 B
// (leading byte offset), 8-row group stride 256 B (stride byte offset).
__device__ __forceinline__ uint64_t sdesc_tf32_core(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128u >> 4) << 16;
    d |= static_cast<uint64_t>(256u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;   // layout type 0: no swizzle
}

// Instruction descriptor, kind::tf32: tf32 A and B, f32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_acc32(int m, int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one 128 x N x 8 tf32 step, issued by one thread.
__device__ __forceinline__ void umma_tf32_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05 op this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

#define MMQ_R32(i) "=r"(r[(i)])

// Two 8-column loads (columns taddr0.. and taddr1..) with a single wait.
__device__ __forceinline__ void tmem_ld8x2_wait(uint32_t taddr0, uint32_t taddr1, float (&v0)[8], float (&v1)[8])
{
    uint32_t r[8], s[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7),
          "=r"(s[0]), "=r"(s[1]), "=r"(s[2]), "=r"(s[3]), "=r"(s[4]), "=r"(s[5]), "=r"(s[6]), "=r"(s[7])
        : "r"(taddr0), "r"(taddr1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(s[i]);
    }
}

// Four 16-column loads (columns taddr, +16, +32, +48) with a single wait: the 64
// consecutive columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, float (&v)[64])
{
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%65];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%66];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7),
          MMQ_R32(8), MMQ_R32(9), MMQ_R32(10), MMQ_R32(11), MMQ_R32(12), MMQ_R32(13), MMQ_R32(14),
          MMQ_R32(15), MMQ_R32(16), MMQ_R32(17), MMQ_R32(18), MMQ_R32(19), MMQ_R32(20), MMQ_R32(21),
          MMQ_R32(22), MMQ_R32(23), MMQ_R32(24), MMQ_R32(25), MMQ_R32(26), MMQ_R32(27), MMQ_R32(28),
          MMQ_R32(29), MMQ_R32(30), MMQ_R32(31), MMQ_R32(32), MMQ_R32(33), MMQ_R32(34), MMQ_R32(35),
          MMQ_R32(36), MMQ_R32(37), MMQ_R32(38), MMQ_R32(39), MMQ_R32(40), MMQ_R32(41), MMQ_R32(42),
          MMQ_R32(43), MMQ_R32(44), MMQ_R32(45), MMQ_R32(46), MMQ_R32(47), MMQ_R32(48), MMQ_R32(49),
          MMQ_R32(50), MMQ_R32(51), MMQ_R32(52), MMQ_R32(53), MMQ_R32(54), MMQ_R32(55), MMQ_R32(56),
          MMQ_R32(57), MMQ_R32(58), MMQ_R32(59), MMQ_R32(60), MMQ_R32(61), MMQ_R32(62), MMQ_R32(63)
        : "r"(taddr), "r"(taddr + 16), "r"(taddr + 32), "r"(taddr + 48)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i)
        v[i] = __uint_as_float(r[i]);
}

// One 16-column load (columns taddr .. taddr + 15) and its wait.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7),
          MMQ_R32(8), MMQ_R32(9), MMQ_R32(10), MMQ_R32(11), MMQ_R32(12), MMQ_R32(13), MMQ_R32(14),
          MMQ_R32(15)
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads from independent column ranges with a single wait.
__device__ __forceinline__ void tmem_ld16x2_wait(uint32_t taddr0, uint32_t taddr1, float (&v0)[16], float (&v1)[16])
{
    uint32_t r[16], q[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]),
          "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15])
        : "r"(taddr0), "r"(taddr1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(q[i]);
    }
}

// Two 16-column loads (columns taddr .. taddr + 31) with a single wait.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7),
          MMQ_R32(8), MMQ_R32(9), MMQ_R32(10), MMQ_R32(11), MMQ_R32(12), MMQ_R32(13), MMQ_R32(14),
          MMQ_R32(15), MMQ_R32(16), MMQ_R32(17), MMQ_R32(18), MMQ_R32(19), MMQ_R32(20), MMQ_R32(21),
          MMQ_R32(22), MMQ_R32(23), MMQ_R32(24), MMQ_R32(25), MMQ_R32(26), MMQ_R32(27), MMQ_R32(28),
          MMQ_R32(29), MMQ_R32(30), MMQ_R32(31)
        : "r"(taddr), "r"(taddr + 16)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

#undef MMQ_R32

}  // namespace mmq
