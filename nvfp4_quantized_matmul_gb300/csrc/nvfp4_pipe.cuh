// mbarrier / TMA helpers for the pipelined kernels, with bounded waits.
//
// Every wait gives up after kWaitLimitNs: it then raises the CTA's abort flag
// and records an error code, so that a stalled pipeline reports instead of
// holding the GPU (the host reads the code with nvfp4_take_device_error).
#pragma once
#include <cuda.h>

#include <cstdint>

namespace nvfp4 {
namespace pipe {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// A waiting thread may be suspended by the hardware for up to this long per
// try (it resumes as soon as the phase completes).
constexpr uint32_t kSuspendHintNs = 1000;

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Arrive with release semantics: this thread's earlier shared-memory writes
// are visible to a thread that observes the completed phase.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive that only signals "done reading": issue is in order and the arrive
// follows every instruction that consumed the buffer's shared loads.
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait by one thread; false once the limit passes (abort flag set,
// `code` recorded in *err) or another warp has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int code, int* err,
                                         uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}

// Bounded wait by all 32 lanes of a warp together: every lane polls (so each
// has acquired the phase) and the decision to stop is taken warp-wide.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int code,
                                              int* err, uint64_t limit_ns = kWaitLimitNs) {
  if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t n = 1;; ++n) {
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    if ((n & 63) == 0) {
      const bool stop = __any_sync(0xffffffffu, *abort_flag != 0 || gtimer() - t0 > limit_ns);
      if (stop) {
        if ((threadIdx.x & 31) == 0) {
          if (!*abort_flag) atomicCAS(err, 0, code);
          *abort_flag = 1;
        }
        return false;
      }
    }
  }
}

// Waits up to the limit for a phase without raising any flag (used to let the
// copies still in flight land before a CTA exits).
__device__ __forceinline__ void wait_bar_quiet(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = gtimer();
  while (!mbar_try(bar, parity) && gtimer() - t0 < kWaitLimitNs) {
  }
}

// 2-D tiled TMA load of the box at (c0, c1) into shared memory; completion is
// counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Box at (c0, c1, c2) of a 3-D tensor map (c0 innermost).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

}  // namespace pipe
}  // namespace nvfp4
