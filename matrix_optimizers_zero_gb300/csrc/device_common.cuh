// Device helpers shared by the kernels: bounded mbarrier waits and bf16
// packing. bf16 -> fp32 widening is exact (the bf16 bits are the upper half of
// the fp32 bits); fp32 -> bf16 uses the CUDA round-to-nearest-even intrinsic.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "mo.h"
#include "ptx.cuh"

namespace mo {

// Default limit of a single device-side wait. A legitimate wait in these
// kernels lasts at most a few hundred microseconds.
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s

// Waits for the phase of `bar` with the given parity. Gives up (returns
// false) when *abort is set by another role, or when the deadline passes, in
// which case it sets *abort and records MO_ERR_DEVICE_TIMEOUT in *status.
// With kCluster the wait acquires at cluster scope (the phase was completed
// by another CTA of the cluster after storing into this CTA's shared memory).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  int* status, uint64_t timeout_ns) {
  auto test = [&] { return kCluster ? ptx::mbar_test_cluster(bar, parity) : ptx::mbar_test(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1; it != 0u; ++it) {
    if (test()) return true;
    if ((it & 127u) == 0u) {
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > timeout_ns) break;
    }
  }
  *abort = 1;
  atomicExch(status, MO_ERR_DEVICE_TIMEOUT);
  return false;
}

// Waits without consulting the abort flag (used while draining in-flight
// copies after an abort). Returns false on expiry.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 0; it != 0xFFFFFFFFu; ++it) {
    if (ptx::mbar_test(bar, parity)) return true;
    if ((it & 127u) == 127u && ptx::globaltimer_ns() - t0 > timeout_ns) return false;
  }
  return false;
}

// 1 - lr wd, rounded once from double with explicit roundings (no
// contraction into a fused multiply-add). Every kernel forms the decoupled
// weight decay this way from lr and wd, whether they arrive by value or from
// device memory, so the two kinds of entry point agree bit for bit.
__device__ __forceinline__ float decay_factor(float lr, float wd) {
  return float(__dsub_rn(1.0, __dmul_rn(double(lr), double(wd))));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return uint32_t(float_to_bf16_bits(lo)) | (uint32_t(float_to_bf16_bits(hi)) << 16);
}

}  // namespace mo
