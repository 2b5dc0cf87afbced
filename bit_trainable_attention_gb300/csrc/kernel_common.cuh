// Bounded waits shared by the attention kernels.  Every wait on an mbarrier
// gives up after a time limit: it then records SAGEBWD_ERR_TIMEOUT with the
// wait's site id in the caller's status word and raises a CTA-wide abort flag,
// so every other role leaves its loop at its next wait and the CTA tears down
// (copies in flight drained, TMEM freed) instead of hanging.
#pragma once
#include "ptx.cuh"
#include "sagebwd_internal.h"

namespace sagebwd {

struct WaitCtx {
  volatile int* abort;  // shared memory flag, 0 = running
  int* status;          // global status word of this call
  uint64_t limit_ns;
};

__device__ __forceinline__ void record_timeout(const WaitCtx& w, int site) {
  *w.abort = 1;
  atomicCAS(w.status, 0, status_timeout(site));
}

// One thread waits.
__device__ __forceinline__ bool wait1(const WaitCtx& w, uint64_t* bar, uint32_t parity, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (globaltimer_ns() - t0 > w.limit_ns) {
      record_timeout(w, site);
      return false;
    }
  }
}

// All 32 lanes of a warp wait; the outcome is the same on every lane, so the
// warp stays converged for the .sync.aligned tcgen05 instructions that follow.
__device__ __forceinline__ bool waitw(const WaitCtx& w, uint64_t* bar, uint32_t parity, int site) {
  bool done = mbar_try_wait(bar, parity);
  if (__all_sync(0xffffffffu, done)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    done = done || mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    int give_up = 0;
    if ((threadIdx.x & 31) == 0) give_up = (*w.abort != 0) ? 1 : (globaltimer_ns() - t0 > w.limit_ns ? 2 : 0);
    give_up = __shfl_sync(0xffffffffu, give_up, 0);
    if (give_up) {
      if (give_up == 2 && (threadIdx.x & 31) == 0) record_timeout(w, site);
      return false;
    }
  }
}

// Teardown: wait (bounded, ignoring the abort flag) for an asynchronous
// operation this thread started -- a TMA load or the MMAs behind a commit.
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Round to the nearest integer, ties to even, for |x| < 2^22, on the FMA pipe
// (the classic magic-number method): adding 1.5 * 2^23 leaves no fraction bits,
// so the IEEE round-to-nearest-even of the addition is the rounding of x, and
// subtracting the constant again is exact.  Same result as rint(x) there.
__device__ __forceinline__ float rint_small(float x) {
  return __fsub_rn(__fadd_rn(x, 12582912.0f), 12582912.0f);
}
// Two integer-valued floats with |v| <= 256 are exact in BF16, whose bits are
// the upper half of the FP32 bits: pack (lo, hi) into bf16x2 with one byte permute.
__device__ __forceinline__ uint32_t pack_int_bf16x2(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Byte offset of the 16-byte chunk `chunk` (0..15 for 128 BF16 columns) of row
// `row` inside a K-major tile stored as two 128-row x 128-byte sub-tiles with
// the 128-byte swizzle (the layout a TMA load with SWIZZLE_128B produces).
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * 16384 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

}  // namespace sagebwd
