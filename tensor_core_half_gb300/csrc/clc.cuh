// clc.cuh -- work ids handed out by cluster launch control (sm_100 family).
//
// A kernel launched with one cluster per work id lets the clusters that are
// running take over the ids of clusters that have not started: one thread
// (the issuer) asks the hardware to cancel the launch of a pending cluster;
// the 16-byte response names it, or says that none was left.  The page
// "tcgen05 for dummies: a B200 GEMM from scratch" (translated), section
// "Persistent kernel", names dynamic scheduling as the step after its static
// scheduler; this is that step on Blackwell.
//
// When to ask: not when an id starts.  Back-to-back launches start their
// clusters a few microseconds apart, as the previous kernel's clusters exit;
// an early cluster that asked at once would cancel clusters that were about
// to start and run their ids after its own, a second wave.  Nor at the very
// end: when all SMs ask at about the same time, answers take microseconds.
// The issuer asks once half of the current id is loaded, or once only
// kClcLeadKBlocks k-blocks are left, whichever comes first.
constexpr int kClcLeadKBlocks = 12;

__device__ __forceinline__ bool clc_time_to_ask(int64_t left, int64_t length) {
  return left <= kClcLeadKBlocks || 2 * left <= length;
}

// Protocol: SLOTS response buffers in shared memory, each with a full barrier
// (one arrival plus 16 transaction bytes) and an empty barrier (one arrival
// per reader).  The issuer asks for the next id as soon as it starts an id;
// every reader waits on the full barrier, decodes the response from its own
// CTA's shared memory, then arrives on the empty barrier of CTA 0 of the
// cluster, after which the slot may take a new request.  After a response
// that names no cluster, no request is issued.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace hg {

template <int CG, int SLOTS>
struct ClcIds {
  uint32_t resp0, full0, empty0;  // slot 0 addresses in this CTA
  bool issuer, warp_wide, arrive;
  int32_t taken = 0;      // responses read
  int32_t requested = 0;  // requests issued (issuer only)

  __device__ ClcIds(uint32_t resp0_, uint32_t full0_, uint32_t empty0_, bool issuer_, bool warp_wide_, bool arrive_)
      : resp0(resp0_), full0(full0_), empty0(empty0_), issuer(issuer_), warp_wide(warp_wide_), arrive(arrive_) {}

  // Barrier set-up, by one thread before the CTA (cluster) synchronises.
  __device__ static void init(uint32_t full0, uint32_t empty0, uint32_t readers) {
    for (int i = 0; i < SLOTS; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, readers);
    }
  }

  // Issuer: ask for the next id.  False if the wait for a free slot gave up.
  __device__ bool request(const WaitCtl& ctl) {
    const int32_t r = requested;
    const uint32_t slot = (uint32_t)(r % SLOTS);
    if (!mbar_wait<CG == 2>(empty0 + 8u * slot, (uint32_t)(((r / SLOTS) & 1) ^ 1), ctl)) return false;
    const uint32_t fb = full0 + 8u * slot;
    mbar_arrive_expect_tx(fb, 16);
    if constexpr (CG == 2) mbar_arrive_expect_tx_cluster(mapa_shared(fb, 1), 16);
    clc_try_cancel<CG>(resp0 + 16u * slot, fb);
    ++requested;
    return true;
  }

  // Every reader: the next response.  1 and *id = the cancelled cluster's
  // index; 0 when no cluster was left; -1 when the wait gave up.
  __device__ int fetch(int64_t* id, const WaitCtl& ctl) {
    const int32_t r = taken;
    const uint32_t slot = (uint32_t)(r % SLOTS);
    if (!mbar_wait<CG == 2>(full0 + 8u * slot, (uint32_t)((r / SLOTS) & 1), ctl)) return -1;
    const int32_t x = clc_first_ctaid_x(resp0 + 16u * slot);
    ++taken;
    if (warp_wide) __syncwarp();
    if (arrive) {
      if constexpr (CG == 1)
        mbar_arrive(empty0 + 8u * slot);
      else
        mbar_arrive_cluster(mapa_shared(empty0 + 8u * slot, 0));
    }
    if (x < 0) return 0;
    *id = x / CG;
    return 1;
  }

  // After giving up: wait for the responses to requests this thread issued
  // and did not read, so that nothing lands in shared memory after exit.
  __device__ bool drain(const WaitCtl& ctl) {
    for (int32_t r = taken; r < requested; ++r) {
      const uint32_t slot = (uint32_t)(r % SLOTS);
      if (!mbar_wait<CG == 2>(full0 + 8u * slot, (uint32_t)((r / SLOTS) & 1), ctl)) return false;
    }
    return true;
  }
};

}  // namespace hg
