// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tile loads, and the tcgen05 tensor-core / tensor-memory instructions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mdcn {

// Bits of the device status word (workspace header). A bounded wait that
// gives up sets kStatusTimeout plus the bit of the site that gave up.
constexpr uint32_t kStatusTimeout = 1u << 0;
constexpr uint32_t kSiteTmaEmpty = 1u << 8;
constexpr uint32_t kSiteGatherEmpty = 1u << 9;
constexpr uint32_t kSiteMmaFull = 1u << 10;
constexpr uint32_t kSiteMmaTma = 1u << 11;
constexpr uint32_t kSiteEpilogue = 1u << 12;
constexpr uint32_t kSiteDrain = 1u << 13;
constexpr uint32_t kSiteSelftest = 1u << 14;
constexpr uint32_t kSiteSplitWait = 1u << 15;

// Limit of every pipeline wait in the fused kernel, in SM clock cycles
// (4e9 cycles: about 2 s at the 2.07 GHz maximum clock, longer at lower
// clocks). A correct launch never waits more than microseconds; the limit
// only bounds a bug. The cycle counter is read every 64 polls, so a wait
// that completes is noticed after one mbarrier test, not after a timer read.
constexpr uint64_t kWaitLimitCycles = 4000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of the given parity to complete, for at most
// limit_cycles SM cycles (or until another role of the CTA raised *abort).
// On giving up it records the site in the status word, raises *abort and
// returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint32_t* status, uint32_t site,
                                                  uint64_t limit_cycles = kWaitLimitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (static_cast<uint64_t>(clock64()) - t0 > limit_cycles) {
                *abort = 1;
                if (status) atomicOr(status, kStatusTimeout | site);
                return false;
            }
        }
    }
}

// mbar_wait_bounded for a whole warp: lane 0 polls, every lane gets its result
// (the warp stays converged).
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint32_t* status, uint32_t site,
                                                  uint64_t limit_cycles = kWaitLimitCycles) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort, status, site, limit_cycles) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait for the given phases of two barriers (bar2 = 0: only bar1) by
// a converged warp: every lane polls both barriers each round, so the two
// polls' latencies overlap, and the warp votes; no lane diverges.
__device__ __forceinline__ bool warp_wait2(uint32_t bar1, uint32_t bar2, uint32_t parity, volatile int* abort,
                                           uint32_t* status, uint32_t site,
                                           uint64_t limit_cycles = kWaitLimitCycles) {
    auto ready = [&]() {
        const bool a = mbar_try_wait(bar1, parity);
        const bool b = bar2 == 0u || mbar_try_wait(bar2, parity);
        return __all_sync(0xffffffffu, a && b);
    };
    if (ready()) return true;
    const uint64_t t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (ready()) return true;
        if ((it & 63u) == 0) {
            if (__any_sync(0xffffffffu, *abort != 0)) return false;
            if (__any_sync(0xffffffffu, static_cast<uint64_t>(clock64()) - t0 > limit_cycles)) {
                if ((threadIdx.x & 31) == 0) {
                    *abort = 1;
                    if (status) atomicOr(status, kStatusTimeout | site);
                }
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- registers
// Per-warpgroup register count (all warps of the warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) { return lds_f32(addr); }
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Named barrier over `count` threads (whole warps) that also ANDs a predicate
// across them: every participant gets the same answer.
__device__ __forceinline__ bool bar_red_and(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Waits, for at most kWaitLimitCycles, until a global counter that other CTAs
// raise reaches `target` (acquire: their writes before the raise are then
// visible). On giving up it records the site, raises *abort, returns false.
__device__ __forceinline__ bool wait_count_bounded(const uint32_t* p, uint32_t target, volatile int* abort,
                                                   uint32_t* status, uint32_t site) {
    const uint64_t t0 = clock64();
    for (;;) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if (*abort) return false;
        if (static_cast<uint64_t>(clock64()) - t0 > kWaitLimitCycles) {
            *abort = 1;
            if (status) atomicOr(status, kStatusTimeout | site);
            return false;
        }
        __nanosleep(64);
    }
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- tcgen05
// Tensor-memory allocation: executed by one whole warp; the base address is
// written to shared memory at dst.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart (stride
// byte offset), tile base 1024-byte aligned. Advancing along K inside the
// 128-byte row is done by adding bytes to the start address.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);          // start address >> 4
    d |= static_cast<uint64_t>(1) << 16;                          // leading byte offset (unused for SW128 K-major)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                          // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;                          // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16 / kind::tf32: fp32 accumulator,
// A and B K-major, shape M x N. ab_format: 0 = f16, 1 = bf16, 2 = tf32.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, uint32_t M, uint32_t N) {
    return (1u << 4)                  // D format: f32
           | (ab_format << 7)         // A format
           | (ab_format << 10)        // B format
           | ((N >> 3) << 17)         // N >> 3
           | ((M >> 4) << 24);        // M >> 4
}

// Warp-wide forms of the issue instructions: the whole (converged) warp
// executes them, computing every operand alike, and the lane elect.sync picks
// (the lowest one, so always the same lane) issues. Operands computed by a
// converged warp stay in uniform registers, which the tcgen05 and TMA
// instructions read.
__device__ __forceinline__ void mma_f16_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with the A operand in tensor memory (a_tmem: lane = row of A,
// 32-bit column c = K elements 2c and 2c + 1 of the instruction's 16).
__device__ __forceinline__ void mma_f16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// kind::tf32: A and B fp32 in shared memory, read as tf32.
__device__ __forceinline__ void mma_tf32_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on the mbarrier once every tcgen05 operation the CTA issued so far
// has completed.
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(bar)
        : "memory");
}

// One arrival that also expects `bytes` of asynchronous copies on the barrier.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}"
        ::"r"(bar), "r"(bytes)
        : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on the
// mbarrier as transferred bytes.
__device__ __forceinline__ void tma_load_2d_elect(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                                  uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets TMEM
// lane (taddr.lane + t), columns taddr.col .. +15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 1 or 2 x (32 lanes x 16 columns) TMEM loads issued back to back, one wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, int n, float (&v)[32]) {
    uint32_t r[32];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (k < n) {
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                : "=r"(r[16 * k + 0]), "=r"(r[16 * k + 1]), "=r"(r[16 * k + 2]), "=r"(r[16 * k + 3]),
                  "=r"(r[16 * k + 4]), "=r"(r[16 * k + 5]), "=r"(r[16 * k + 6]), "=r"(r[16 * k + 7]),
                  "=r"(r[16 * k + 8]), "=r"(r[16 * k + 9]), "=r"(r[16 * k + 10]), "=r"(r[16 * k + 11]),
                  "=r"(r[16 * k + 12]), "=r"(r[16 * k + 13]), "=r"(r[16 * k + 14]), "=r"(r[16 * k + 15])
                : "r"(taddr + 16u * k)
                : "memory");
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) r[16 * k + i] = 0u;
        }
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 lanes x 256 bits, repeated over 4 consecutive 8-column blocks: thread t
// writes r[4k], r[4k+1] to lane (taddr.lane + t/4), columns taddr.col + 8k +
// 2(t%4) and + 1, and r[4k+2], r[4k+3] to lane (taddr.lane + 8 + t/4), the
// same columns. taddr.lane must lie in the warp's lane quarter.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Waits until this thread's tensor-memory stores have completed.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 256-bit read-only global load (32-byte aligned address).
__device__ __forceinline__ void ldg256(const void* p, uint4& a, uint4& b) {
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
}

// Round-to-nearest (ties away) fp32 -> tf32, returned as an fp32 bit pattern
// with the low 13 mantissa bits cleared.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

}  // namespace mdcn
