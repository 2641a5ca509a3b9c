// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarriers, bulk async copies
// (global -> shared, completion counted on an mbarrier), tcgen05 tensor-core MMA
// with TMEM accumulators, TMEM loads, and the bounded wait every kernel uses.
#pragma once

#include <cstdint>

namespace mmq {

// Sticky device error word of this translation unit (bit 0: a bounded wait
// expired).  Each .cu file that includes this header gets its own copy and
// exposes a host-side reader (see mmq_internal.h).
static __device__ unsigned int g_error_word;

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
// false) once the sticky error word is set by anyone, or after limit_ns of
// global time, in which case it sets the error word itself.  The error word and
// the global timer are first read after 64 unsuccessful polls, so short waits
// cost one or a few try_wait round trips.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 63u) == 0) {
            if (*reinterpret_cast<volatile unsigned int*>(&g_error_word) != 0u)
                return false;
            const uint64_t now = globaltimer_ns();
            if (i == 64u)
                t0 = now;
            else if (now - t0 > limit_ns) {
                atomicOr(&g_error_word, 1u);
                return false;
            }
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

// Same with an L2 eviction-priority hint (createpolicy handle).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
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

// Arrive (once) on `bar` when every tcgen05 op this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

#define MMQ_R32(i) "=r"(r[(i)])

// 32 lanes x 32 consecutive f32 columns from TMEM, then wait for the load:
// thread `lane` of the warp gets columns [taddr.col, +32) of TMEM lane
// (taddr.lane + lane).  The wait sits in the same asm statement so no use of
// the registers can be scheduled before it.
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7),
          MMQ_R32(8), MMQ_R32(9), MMQ_R32(10), MMQ_R32(11), MMQ_R32(12), MMQ_R32(13), MMQ_R32(14),
          MMQ_R32(15), MMQ_R32(16), MMQ_R32(17), MMQ_R32(18), MMQ_R32(19), MMQ_R32(20), MMQ_R32(21),
          MMQ_R32(22), MMQ_R32(23), MMQ_R32(24), MMQ_R32(25), MMQ_R32(26), MMQ_R32(27), MMQ_R32(28),
          MMQ_R32(29), MMQ_R32(30), MMQ_R32(31)
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Two 32-column loads (columns taddr0.. and taddr1..) with a single wait.
__device__ __forceinline__ void tmem_ld32x2_wait(uint32_t taddr0, uint32_t taddr1, float (&v0)[32],
                                                 float (&v1)[32])
{
    uint32_t r[32], s[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7),
          MMQ_R32(8), MMQ_R32(9), MMQ_R32(10), MMQ_R32(11), MMQ_R32(12), MMQ_R32(13), MMQ_R32(14),
          MMQ_R32(15), MMQ_R32(16), MMQ_R32(17), MMQ_R32(18), MMQ_R32(19), MMQ_R32(20), MMQ_R32(21),
          MMQ_R32(22), MMQ_R32(23), MMQ_R32(24), MMQ_R32(25), MMQ_R32(26), MMQ_R32(27), MMQ_R32(28),
          MMQ_R32(29), MMQ_R32(30), MMQ_R32(31),
          "=r"(s[0]), "=r"(s[1]), "=r"(s[2]), "=r"(s[3]), "=r"(s[4]), "=r"(s[5]), "=r"(s[6]), "=r"(s[7]),
          "=r"(s[8]), "=r"(s[9]), "=r"(s[10]), "=r"(s[11]), "=r"(s[12]), "=r"(s[13]), "=r"(s[14]),
          "=r"(s[15]), "=r"(s[16]), "=r"(s[17]), "=r"(s[18]), "=r"(s[19]), "=r"(s[20]), "=r"(s[21]),
          "=r"(s[22]), "=r"(s[23]), "=r"(s[24]), "=r"(s[25]), "=r"(s[26]), "=r"(s[27]), "=r"(s[28]),
          "=r"(s[29]), "=r"(s[30]), "=r"(s[31])
        : "r"(taddr0), "r"(taddr1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(s[i]);
    }
}

// 32 lanes x 16 consecutive f32 columns from TMEM, then wait for the load.
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

// Two 16-column loads (columns taddr0.. and taddr1..) with a single wait.
__device__ __forceinline__ void tmem_ld16x2_wait(uint32_t taddr0, uint32_t taddr1, float (&v0)[16],
                                                 float (&v1)[16])
{
    uint32_t r[16], s[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7),
          MMQ_R32(8), MMQ_R32(9), MMQ_R32(10), MMQ_R32(11), MMQ_R32(12), MMQ_R32(13), MMQ_R32(14),
          MMQ_R32(15), "=r"(s[0]), "=r"(s[1]), "=r"(s[2]), "=r"(s[3]), "=r"(s[4]), "=r"(s[5]), "=r"(s[6]),
          "=r"(s[7]), "=r"(s[8]), "=r"(s[9]), "=r"(s[10]), "=r"(s[11]), "=r"(s[12]), "=r"(s[13]),
          "=r"(s[14]), "=r"(s[15])
        : "r"(taddr0), "r"(taddr1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(s[i]);
    }
}

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

// Issue a 64-column TMEM load (two 32-column loads) without waiting: the
// registers hold the data only after tmem_wait_ld_tied() has run on them.
__device__ __forceinline__ void tmem_ld64_issue(uint32_t taddr, uint32_t (&r)[64])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
        : MMQ_R32(0), MMQ_R32(1), MMQ_R32(2), MMQ_R32(3), MMQ_R32(4), MMQ_R32(5), MMQ_R32(6), MMQ_R32(7), MMQ_R32(8), MMQ_R32(9), MMQ_R32(10), MMQ_R32(11), MMQ_R32(12), MMQ_R32(13), MMQ_R32(14), MMQ_R32(15), MMQ_R32(16), MMQ_R32(17), MMQ_R32(18), MMQ_R32(19), MMQ_R32(20), MMQ_R32(21), MMQ_R32(22), MMQ_R32(23), MMQ_R32(24), MMQ_R32(25), MMQ_R32(26), MMQ_R32(27), MMQ_R32(28), MMQ_R32(29), MMQ_R32(30), MMQ_R32(31), MMQ_R32(32), MMQ_R32(33), MMQ_R32(34), MMQ_R32(35), MMQ_R32(36), MMQ_R32(37), MMQ_R32(38), MMQ_R32(39), MMQ_R32(40), MMQ_R32(41), MMQ_R32(42), MMQ_R32(43), MMQ_R32(44), MMQ_R32(45), MMQ_R32(46), MMQ_R32(47), MMQ_R32(48), MMQ_R32(49), MMQ_R32(50), MMQ_R32(51), MMQ_R32(52), MMQ_R32(53), MMQ_R32(54), MMQ_R32(55), MMQ_R32(56), MMQ_R32(57), MMQ_R32(58), MMQ_R32(59), MMQ_R32(60), MMQ_R32(61), MMQ_R32(62), MMQ_R32(63)
        : "r"(taddr), "r"(taddr + 32)
        : "memory");
}

#define MMQ_T64(i) "+r"(r[(i)])
#define MMQ_K2(i) "+f"(k[(i)].x), "+f"(k[(i)].y)

// Wait for this thread's outstanding TMEM loads.  `r` (the destination of the
// load waited for) and `k` (values whose computation should overlap the load)
// are tied to the wait: the compiler can neither read r before it nor move the
// computation of k after it.
__device__ __forceinline__ void tmem_wait_ld_tied(uint32_t (&r)[64], float2 (&k)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : MMQ_T64(0), MMQ_T64(1), MMQ_T64(2), MMQ_T64(3), MMQ_T64(4), MMQ_T64(5), MMQ_T64(6), MMQ_T64(7), MMQ_T64(8), MMQ_T64(9), MMQ_T64(10), MMQ_T64(11), MMQ_T64(12), MMQ_T64(13), MMQ_T64(14), MMQ_T64(15), MMQ_T64(16), MMQ_T64(17), MMQ_T64(18), MMQ_T64(19), MMQ_T64(20), MMQ_T64(21), MMQ_T64(22), MMQ_T64(23), MMQ_T64(24), MMQ_T64(25), MMQ_T64(26), MMQ_T64(27), MMQ_T64(28), MMQ_T64(29), MMQ_T64(30), MMQ_T64(31), MMQ_T64(32), MMQ_T64(33), MMQ_T64(34), MMQ_T64(35), MMQ_T64(36), MMQ_T64(37), MMQ_T64(38), MMQ_T64(39), MMQ_T64(40), MMQ_T64(41), MMQ_T64(42), MMQ_T64(43), MMQ_T64(44), MMQ_T64(45), MMQ_T64(46), MMQ_T64(47), MMQ_T64(48), MMQ_T64(49), MMQ_T64(50), MMQ_T64(51), MMQ_T64(52), MMQ_T64(53), MMQ_T64(54), MMQ_T64(55), MMQ_T64(56), MMQ_T64(57), MMQ_T64(58), MMQ_T64(59), MMQ_T64(60), MMQ_T64(61), MMQ_T64(62), MMQ_T64(63), MMQ_K2(0), MMQ_K2(1), MMQ_K2(2), MMQ_K2(3), MMQ_K2(4), MMQ_K2(5), MMQ_K2(6), MMQ_K2(7), MMQ_K2(8), MMQ_K2(9), MMQ_K2(10), MMQ_K2(11), MMQ_K2(12), MMQ_K2(13), MMQ_K2(14), MMQ_K2(15), MMQ_K2(16), MMQ_K2(17), MMQ_K2(18), MMQ_K2(19), MMQ_K2(20), MMQ_K2(21), MMQ_K2(22), MMQ_K2(23), MMQ_K2(24), MMQ_K2(25), MMQ_K2(26), MMQ_K2(27), MMQ_K2(28), MMQ_K2(29), MMQ_K2(30), MMQ_K2(31)
                 :
                 : "memory");
}

#undef MMQ_T64
#undef MMQ_K2

#define MMQ_T64A(i) "+r"(a[(i)])
#define MMQ_T64B(i) "+r"(b[(i)])

// Wait for this thread's outstanding TMEM loads into a and b (two loads issued
// with tmem_ld64_issue); both arrays are tied to the wait.
__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&a)[64], uint32_t (&b)[64])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : MMQ_T64A(0), MMQ_T64A(1), MMQ_T64A(2), MMQ_T64A(3), MMQ_T64A(4), MMQ_T64A(5), MMQ_T64A(6), MMQ_T64A(7), MMQ_T64A(8), MMQ_T64A(9), MMQ_T64A(10), MMQ_T64A(11), MMQ_T64A(12), MMQ_T64A(13), MMQ_T64A(14), MMQ_T64A(15), MMQ_T64A(16), MMQ_T64A(17), MMQ_T64A(18), MMQ_T64A(19), MMQ_T64A(20), MMQ_T64A(21), MMQ_T64A(22), MMQ_T64A(23), MMQ_T64A(24), MMQ_T64A(25), MMQ_T64A(26), MMQ_T64A(27), MMQ_T64A(28), MMQ_T64A(29), MMQ_T64A(30), MMQ_T64A(31), MMQ_T64A(32), MMQ_T64A(33), MMQ_T64A(34), MMQ_T64A(35), MMQ_T64A(36), MMQ_T64A(37), MMQ_T64A(38), MMQ_T64A(39), MMQ_T64A(40), MMQ_T64A(41), MMQ_T64A(42), MMQ_T64A(43), MMQ_T64A(44), MMQ_T64A(45), MMQ_T64A(46), MMQ_T64A(47), MMQ_T64A(48), MMQ_T64A(49), MMQ_T64A(50), MMQ_T64A(51), MMQ_T64A(52), MMQ_T64A(53), MMQ_T64A(54), MMQ_T64A(55), MMQ_T64A(56), MMQ_T64A(57), MMQ_T64A(58), MMQ_T64A(59), MMQ_T64A(60), MMQ_T64A(61), MMQ_T64A(62), MMQ_T64A(63), MMQ_T64B(0), MMQ_T64B(1), MMQ_T64B(2), MMQ_T64B(3), MMQ_T64B(4), MMQ_T64B(5), MMQ_T64B(6), MMQ_T64B(7), MMQ_T64B(8), MMQ_T64B(9), MMQ_T64B(10), MMQ_T64B(11), MMQ_T64B(12), MMQ_T64B(13), MMQ_T64B(14), MMQ_T64B(15), MMQ_T64B(16), MMQ_T64B(17), MMQ_T64B(18), MMQ_T64B(19), MMQ_T64B(20), MMQ_T64B(21), MMQ_T64B(22), MMQ_T64B(23), MMQ_T64B(24), MMQ_T64B(25), MMQ_T64B(26), MMQ_T64B(27), MMQ_T64B(28), MMQ_T64B(29), MMQ_T64B(30), MMQ_T64B(31), MMQ_T64B(32), MMQ_T64B(33), MMQ_T64B(34), MMQ_T64B(35), MMQ_T64B(36), MMQ_T64B(37), MMQ_T64B(38), MMQ_T64B(39), MMQ_T64B(40), MMQ_T64B(41), MMQ_T64B(42), MMQ_T64B(43), MMQ_T64B(44), MMQ_T64B(45), MMQ_T64B(46), MMQ_T64B(47), MMQ_T64B(48), MMQ_T64B(49), MMQ_T64B(50), MMQ_T64B(51), MMQ_T64B(52), MMQ_T64B(53), MMQ_T64B(54), MMQ_T64B(55), MMQ_T64B(56), MMQ_T64B(57), MMQ_T64B(58), MMQ_T64B(59), MMQ_T64B(60), MMQ_T64B(61), MMQ_T64B(62), MMQ_T64B(63)
                 :
                 : "memory");
}

#undef MMQ_T64A
#undef MMQ_T64B

// 64 consecutive 32-bit columns of this thread's TMEM lane from registers (two
// 32-column stores); tmem_wait_st() waits for them.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&v)[64])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], "
        "{%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,"
        "%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65};\n"
        :
        : "r"(taddr), "r"(taddr + 32), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]), "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef MMQ_R32

}  // namespace mmq
