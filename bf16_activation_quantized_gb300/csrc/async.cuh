// async.cuh -- mbarrier, bulk-copy and TMA helpers (sm_100-family PTX).
//
// Every wait is bounded: a wait that has not completed after kWaitLimitNs of
// %globaltimer time sets an error bit in the kernel's error word and returns
// false, and once a CTA has seen a timeout (its shared abort flag is set) all
// later waits return immediately, so a broken pipeline ends the kernel instead
// of hanging the GPU.  A CTA that aborts writes NaN to every output it owns
// (see the kernels), so an incomplete result is never a plausible number.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// Error bits a kernel may record in the library's device error word (read
// back, and cleared, with w4a16_read_error_word).
constexpr int kErrWaitTimeout = 1;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tensor core).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test: true if the phase with the given parity has completed.
// (try_wait may suspend the thread for a while when the phase is incomplete;
// a thread that polls several barriers must not be held on one of them.)
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in the instruction (up to
// kSuspendHintNs) until the phase completes, instead of spinning.
constexpr uint32_t kSuspendHintNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Whether more than limit_ns have passed since *t0 on %globaltimer.  The timer
// is a wall clock that the driver may adjust; a reading below *t0 restarts the
// interval instead of being taken, as an unsigned difference would be, for a
// wait of about 2^64 ns.
__device__ __forceinline__ bool elapsed_beyond(unsigned long long *t0, unsigned long long limit_ns) {
    const unsigned long long now = global_timer_ns();
    if (now < *t0) {
        *t0 = now;
        return false;
    }
    return now - *t0 > limit_ns;
}

// True in exactly one lane of a converged warp (elect.sync over all 32 lanes,
// the lowest active lane).  Single-thread issue of TMA copies, MMAs and
// commits goes through it: measured on GB300, a warp-wide loop that issues
// tcgen05.mma under elect.sync issued an M=128, N=32 MMA every ~26 cycles,
// the same loop under `lane == 0` every ~60 and a loop run by lane 0 alone
// every ~55-100.
__device__ __forceinline__ bool elect_one() {
    uint32_t p = 0;
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}"
        : "=r"(p));
    return p != 0;
}

// Reading %globaltimer is slow (measured on GB300: a producer loop that read
// it once per iteration issued one copy every ~0.5 us), so the bounded waits
// consult it only once every kTimerPollSpins failed polls.
constexpr int kTimerPollSpins = 32;

// Wait for the phase with the given parity to complete.  Returns false on
// timeout (after limit_ns) or when the CTA is already aborting.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int *err_word,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = 0;
    for (int spins = 1;; ++spins) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag) return false;
        if (spins % kTimerPollSpins == 0) {
            if (t0 == 0) {
                t0 = global_timer_ns();
            } else if (elapsed_beyond(&t0, limit_ns)) {
                *abort_flag = 1;
                if (err_word) atomicOr(err_word, kErrWaitTimeout);
                return false;
            }
        }
    }
}

// Wait, ignoring the abort flag, for a phase that copies still in flight will
// complete (used only when aborting, so that no copy lands in shared memory
// after the CTA has exited); gives up after 100 ms.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (elapsed_beyond(&t0, 100000000ull)) break;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Warm L2 with `bytes` of global memory (bytes % 16 == 0, 16-byte aligned);
// nothing is written anywhere, so it is safe before a dependency wait (L2 is
// coherent: a later write by another kernel replaces the prefetched lines).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2-D tiled TMA load: box at (x = innermost element index, y = row) -> shared.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31) == 0; }

}  // namespace w4a16
