// ra_umma.cuh -- pieces shared by the tcgen05 kernels of libringattn:
// instruction / shared-memory descriptor encoders for kind::f16 MMAs on
// 128-byte-swizzled tiles, and the bounded mbarrier waits every role uses.
#pragma once
#include <cstdint>

#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major,
// B K-major (0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, low word: start address and leading byte
// offset (both in 16-byte units).  A TMA-loaded [128 rows x 64 cols] bf16
// block with 128-byte swizzle is one swizzle atom column; a K-major operand
// steps 32 bytes per K=16 inside a block, an MN-major operand steps 8 rows
// (2048 bytes) per K=16 and finds its second 64-column block LBO bytes on.
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
// high word of a 128-byte-swizzle descriptor: stride byte offset 1024 B
// (8 rows of 128 B), descriptor version 1, swizzle mode 128 B
constexpr uint32_t kDescHiSw128 = ((1024u >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);

// Bounded wait on one mbarrier phase (single thread): sleeps in hardware
// between polls, gives up after `timeout_ns` (or when another role raised
// the CTA's abort flag), and on its own timeout sets the status bit and the
// abort flag.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns, unsigned int* status) {
  // the timeout's reference is read only once a first sleeping wait has
  // returned without the phase: most waits end there, and the timer read
  // would lie on their path
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, 200000u)) return true;
    if (it == 1) t0 = global_timer_ns();
    if ((it & 3u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        if (status) atomicOr(status, kStatusTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait used while tearing down after an abort: never raises the flag
// again and gives up after at most 100 ms.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long t) {
  volatile int never = 0;
  if (!mbar_try_wait(bar, parity))
    wait_slow(bar, parity, &never, t < 100000000ull ? t : 100000000ull, nullptr);
}

}  // namespace ra
