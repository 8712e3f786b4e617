// sm103_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_103a)
// features the attention kernels use: mbarriers, TMA tensor loads, tcgen05
// tensor-core MMAs with accumulators in tensor memory (TMEM), TMEM loads and
// stores, the shared-memory matrix descriptor and the instruction descriptor.
// Written from the public PTX ISA description of these instructions.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ne {

// Device status bits (the word is OR-ed; the host maps them to ne_status).
constexpr uint32_t kDevTimeout = 1u;
constexpr uint32_t kDevRange = 2u;
constexpr uint32_t kDevPrecision = 4u;   // more large-norm rows than a CTA records
constexpr uint32_t kDevArg = 8u;         // a device-resident argument out of range

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarrier ---

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Programmatic dependent launch.  griddep_wait: block until every grid this
// one depends on has completed and its memory operations are visible (a
// no-op when the launch had no such dependency).  griddep_launch_dependents:
// allow the next grid in the stream to be scheduled once every CTA of this
// grid has executed it or exited; it grants no memory visibility.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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

__device__ __forceinline__ uint32_t mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// Every wait in the kernels is bounded.  `abort` is a shared-memory flag of
// the CTA: the first wait that runs out sets it and records kDevTimeout in
// the device status word; every later wait of the CTA then gives up at once,
// so all roles leave their loops and the CTA drains and exits.
struct WaitCtl {
    volatile uint32_t *abort;
    uint32_t *status;
    uint64_t limit_ns;
};

static __device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, WaitCtl w)
{
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_test(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1u;
            atomicOr(w.status, kDevTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &w)
{
    if (mbar_test(bar, parity))
        return true;
    return mbar_wait_slow(bar, parity, w);
}

// Bounded wait that does not touch the abort flag: used while draining a
// CTA's own in-flight copies after an abort.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_test(bar, parity))
        if (global_timer_ns() - t0 > limit_ns)
            return false;
    return true;
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the result
// (so warp-collective tcgen05 instructions after it are never divergent).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const WaitCtl &w)
{
    bool ok = mbar_wait(bar, parity, w);
    return __all_sync(0xffffffffu, ok);
}

// The same for a warp off the critical path: between polls the thread is
// suspended until the phase completes or for at most kIdleHintNs, so it does
// not take issue slots from the computing warps of its sub-partition (waking
// costs latency, which such a warp can afford).
constexpr uint32_t kIdleHintNs = 100000;

__device__ __forceinline__ uint32_t mbar_test_idle(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(kIdleHintNs)
        : "memory");
    return ok;
}

__device__ __forceinline__ bool mbar_wait_warp_idle(uint32_t bar, uint32_t parity,
                                                    const WaitCtl &w)
{
    bool ok = true;
    if (!mbar_test_idle(bar, parity)) {
        const uint64_t t0 = global_timer_ns();
        while (true) {
            if (mbar_test_idle(bar, parity))
                break;
            if (*w.abort) {
                ok = false;
                break;
            }
            if (global_timer_ns() - t0 > w.limit_ns) {
                *w.abort = 1u;
                atomicOr(w.status, kDevTimeout);
                ok = false;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// One lane of a fully active warp (the lowest); all 32 lanes must call it.
// Warp-wide issue loops keep descriptor math warp-uniform, and only the
// elected lane issues the tcgen05 instruction.
__device__ __forceinline__ bool elect_one()
{
    uint32_t p;
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(p));
    return p != 0;
}

// -------------------------------------------------------------- fences ---

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's async-proxy (TMA) writes to global memory, already
// complete, before its later generic accesses and those it synchronises with.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ TMA ---

// 16-byte read-only load that is not kept in L1 (a pure streaming pass).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load; coordinates innermost first.  Completion is signalled on
// `bar` as transaction bytes (the caller posts expect_tx for the box size).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Prefetch a 4-D tile into L2 (no shared memory, no completion signal).
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                                   int c3)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// 4-D tiled store from shared memory (bulk-group completion).  Elements
// outside the tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// This thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait0()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------- shared-memory counters ---
// Monotonic per-CTA counters that order hand-offs between warps of different
// roles without a CTA-wide barrier: a writer publishes with release, a reader
// polls with acquire.

__device__ __forceinline__ uint32_t ld_acquire_smem(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_smem(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ void add_release_smem(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v)
                 : "memory");
}

static __device__ __forceinline__ bool counter_wait_slow(const uint32_t *p, uint32_t target,
                                                        WaitCtl w)
{
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (ld_acquire_smem(p) >= target)
            return true;
        if (*w.abort)
            return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1u;
            atomicOr(w.status, kDevTimeout);
            return false;
        }
    }
}

// Warp-uniform bounded wait until *p >= target (every lane polls the same
// word with acquire, so each is ordered after the writer's release).
__device__ __forceinline__ bool counter_wait_warp(const uint32_t *p, uint32_t target,
                                                  const WaitCtl &w)
{
    bool ok = ld_acquire_smem(p) >= target;
    if (!__all_sync(0xffffffffu, ok))
        ok = counter_wait_slow(p, target, w);
    return __all_sync(0xffffffffu, ok);
}

// ----------------------------------------------------------------- TMEM ---

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

// TMEM address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col)
{
    return base + (lane << 16) + col;
}

#define NE_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])

// 32 lanes x 32 consecutive 32-bit columns: lane i of the warp receives row
// (warp's lane quarter)*32 + i, columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : NE_R8(0), NE_R8(8), NE_R8(16), NE_R8(24)
        : "r"(taddr));
}

#define NE_T8(i) "+r"(r[i + 0]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                 "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

// Waits for this thread's outstanding TMEM loads, and ties the registers of
// `r` to the wait so the compiler cannot read them before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    asm volatile("" : NE_T8(0), NE_T8(8), NE_T8(16), NE_T8(24));
}

__device__ __forceinline__ void tmem_ld_wait_only()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_tie(uint32_t (&r)[32])
{
    asm volatile("" : NE_T8(0), NE_T8(8), NE_T8(16), NE_T8(24));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

#define NE_R4(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3])

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : NE_R8(0), NE_R8(8)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_tie16(uint32_t (&r)[16])
{
    asm volatile("" : NE_T8(0), NE_T8(8));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------- tcgen05 ---

// Shared-memory matrix descriptor.  layout: 0 none, 2 = 128-byte swizzle,
// 4 = 64-byte swizzle.  Byte offsets are encoded in 16-byte units.  Bits
// 46..48 hold the fixed value 0b001; the base-offset field stays 0 because
// every operand tile starts on a 1024-byte boundary.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= static_cast<uint64_t>(layout & 7u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with an fp32 accumulator.
// ab_bf16: both operands bf16 (else both fp16).  a_mn / b_mn: the operand is
// stored MN-major (contiguous along M resp. N) instead of K-major.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, bool ab_bf16, bool a_mn,
                                                 bool b_mn)
{
    return (1u << 4)                              // D format: f32
           | ((ab_bf16 ? 1u : 0u) << 7)           // A format: 0 f16, 1 bf16
           | ((ab_bf16 ? 1u : 0u) << 10)          // B format
           | ((a_mn ? 1u : 0u) << 15)             // A major
           | ((b_mn ? 1u : 0u) << 16)             // B major
           | ((N >> 3) << 17)                     // N / 8
           | ((M >> 4) << 24);                    // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T.  A (M = 128 rows in lanes 0..127) is
// packed two 16-bit elements per 32-bit column, element 2c in the low half of
// column c; one K step of 16 elements spans 8 columns.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Per-warpgroup register budget changes (all four warps of the warpgroup
// execute them).  The budgets of all warpgroups must add up to at most the
// registers the block was launched with.
template <uint32_t N>
__device__ __forceinline__ void regs_release()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void regs_claim()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// ------------------------------------------------------------- numerics ---

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Three-way maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed pairs of fp32 values (sm_100+ two-lane FMA / add): one instruction
// for two values.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f32x2_split(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

} // namespace ne
