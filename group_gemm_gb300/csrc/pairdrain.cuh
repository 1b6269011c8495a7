// pairdrain.cuh -- the exact drain of a CTA pair's TMA loads when its producers stop.
//
// In the CTA-pair kernels both CTAs issue TMA loads into their own shared memory, and every load
// completes on the even CTA's "full" barrier of its stage (that barrier counts both halves). The
// odd CTA cannot see its own loads land, and when the producers stop early (a wait ran out) the
// two may have stopped at different iterations of the same load sequence. Before either CTA may
// leave, every load either issued must have landed, or the copy engine would write into shared
// memory that a later CTA owns.
//
// Both producers count the iterations they issued (iteration i uses stage i % S with phase
// (i / S) & 1) and record, per stage, the odd CTA's share of the bytes of their latest iteration
// there (both compute the same share for the same iteration). At the end of its loop the odd
// producer stores its count and its shares into the even CTA's exchange area and arrives on the
// even CTA's exchange barrier (release at cluster scope). The even producer waits for that arrival
// (acquire at cluster scope) and settles each stage s, with L and O the last iterations the even
// and the odd CTA issued there:
//   L == O  wait for the phase of L: both halves are in flight or landed;
//   L >  O  the odd CTA never issued L (then O == L - S): count its share as arrived
//           (mbarrier.complete_tx), then wait for the phase of L, that is, for the even CTA's half;
//   O >  L  the even CTA never armed O (then O == L + S; the phase of L has completed, since the
//           odd CTA waited for stage s to be freed): arm it with the odd share alone and wait.
// Then all bytes of both CTAs have landed. The odd CTA leaves only through the kernel's final
// cluster barrier, which the even CTA reaches after settling, so neither leaves early. In a run
// that did not stop early, L == O on every stage and every phase has already completed.
//
// Every wait here is bounded: the drains by kDrainTimeoutNs (or the caller's longer limit), the
// wait for the odd producer's count by the caller's limit plus kDrainTimeoutNs. If that count never
// arrives, the even CTA holds the pair a further kPairFallbackNs before the final cluster barrier.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace rdot {

// Shared-memory exchange area, present in both CTAs (only the even CTA's is read). 8-byte aligned.
template <int STAGES>
struct PairExchange {
    uint64_t bar;                 // the odd producer arrives here once (count 1)
    int32_t odd_pos;              // iterations the odd producer issued
    int32_t pad;
    int32_t odd_share[STAGES];    // written by the odd producer: its bytes of its last iteration per stage
    int32_t share[STAGES];        // this CTA's record: the odd CTA's bytes of this CTA's last iteration per stage
};

constexpr uint64_t kPairFallbackNs = 1000000ull;   // 1 ms, far longer than any TMA transfer

// Last iteration below `pos` that used stage s, or -1.
__device__ __forceinline__ int pair_last_iter(int pos, int s, int stages) {
    if (pos <= s) return -1;
    return s + ((pos - 1 - s) / stages) * stages;
}

// The odd producer, after its loop: hand the even CTA its count and shares.
template <int STAGES>
__device__ __forceinline__ void pair_publish(PairExchange<STAGES>* x, int pos) {
    const uint32_t base = mapa_shared(smem_u32(x), 0);
    const uint32_t off_pos = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&x->odd_pos) - reinterpret_cast<uintptr_t>(x));
    const uint32_t off_share =
        static_cast<uint32_t>(reinterpret_cast<uintptr_t>(&x->odd_share[0]) - reinterpret_cast<uintptr_t>(x));
#pragma unroll
    for (int s = 0; s < STAGES; ++s) st_shared_cluster_u32(base + off_share + 4 * s, static_cast<uint32_t>(x->share[s]));
    st_shared_cluster_u32(base + off_pos, static_cast<uint32_t>(pos));
    mbar_arrive_cluster(base);   // the barrier is the first member
}

// The even producer, after its loop: settle every stage (see above). Returns false if the odd
// producer's count never arrived, in which case nothing is known about its loads and the caller
// must not assume they landed.
template <int STAGES>
__device__ __forceinline__ bool pair_settle(PairExchange<STAGES>* x, uint64_t* full, int pos, const WaitGuard& g) {
    int dummy = 0;
    const WaitGuard dg = drain_guard(g, &dummy);
    // the odd producer may still sit in one wait of its own (up to the caller's limit) before it
    // stops and publishes
    const uint64_t publish_limit = g.timeout_ns + kDrainTimeoutNs;
    bool arrived = mbar_try_wait_cluster(&x->bar, 0);
    if (!arrived) {
        const uint64_t t0 = global_timer_ns();
        while (!(arrived = mbar_try_wait_cluster(&x->bar, 0)) && global_timer_ns() - t0 <= publish_limit) {
        }
    }
    if (!arrived) return false;
    const int opos = x->odd_pos;
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        const int L = pair_last_iter(pos, s, STAGES);
        const int O = pair_last_iter(opos, s, STAGES);
        if (L < 0 && O < 0) continue;
        if (L > O) {
            if (x->share[s] > 0) mbar_complete_tx(&full[s], static_cast<uint32_t>(x->share[s]));
        } else if (O > L) {
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(x->odd_share[s]));
        }
        const int last = L > O ? L : O;
        (void)mbar_wait(&full[s], static_cast<uint32_t>((last / STAGES) & 1), dg);
    }
    return true;
}

// Both producers, after their loops: the odd one publishes, the even one settles (falling back to
// a fixed hold if the odd count never arrived).
template <int STAGES>
__device__ __forceinline__ void pair_drain(PairExchange<STAGES>* x, uint64_t* full, int pos, bool leader,
                                           const WaitGuard& g) {
    if (!leader) {
        pair_publish(x, pos);
    } else if (!pair_settle(x, full, pos, g)) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < kPairFallbackNs) {
        }
    }
}

}  // namespace rdot
