// Shared device/host helpers of the specdec kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specdec.h"

namespace specdec {

// ----------------------------------------------------------------------------------- status

// Record the first nonzero status code; later codes do not overwrite it.
__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------------------------- bf16

// bf16 is the top half of an fp32 bit pattern: widening is a shift, exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_at(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(*p) << 16);
}

// Unpack one 16-byte vector into floats: 8 for bf16, 4 for fp32.
template <typename T> struct Vec;
template <> struct Vec<uint16_t> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* x) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
  }
  __device__ __forceinline__ static float scalar(const uint16_t* p) { return bf16_at(p); }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* x) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static float scalar(const float* p) { return *p; }
};

// Programmatic dependent launch.  A kernel launched with programmatic stream serialization may
// start before the kernel ahead of it on the stream has finished; pdl_wait() blocks until that
// kernel has completed and its memory operations are visible (a no-op for a normal launch).
// pdl_launch_dependents() lets the next such kernel start launching once every CTA of this grid
// has called it or exited (without it, that happens when this grid completes).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Streaming 16-byte load that does not allocate in L1 (each byte is read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// ----------------------------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

// Named CTA barrier `id` (1..15; 0 is __syncthreads) over n threads, a multiple of 32, whole
// warps: sync waits for all n; arrive counts its warp and goes on (a release to the waiters).
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Wait for phase `parity` of the barrier to complete, giving up after `max_tries` polls.
// Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t max_tries) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t it = 0; it < max_tries; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(a), "r"(parity) : "memory");
    if (done) return true;
  }
  return false;
}

// As mbar_wait_bounded, but each poll lets the thread sleep until the phase completes or about
// `sleep_ns` pass (the try_wait suspend-time hint), so waiting warps do not spin on issue slots.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t max_tries,
                                                uint32_t sleep_ns) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t it = 0; it < max_tries; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(a), "r"(parity), "r"(sleep_ns) : "memory");
    if (done) return true;
  }
  return false;
}

// ----------------------------------------------------------------------------------- bulk copy

// global -> shared (this CTA), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// shared -> global, tracked by bulk groups of the issuing thread.
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(gdst), "r"(smem_addr(smem_src)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N> __device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group of this thread has completed (writes visible).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ----------------------------------------------------------------------------------- host

int sm_count();                  // multiprocessors of the current device (cached per device)

// Cluster size for a grid of `rows` clusters of one kernel: the largest C in [c_min, c_max]
// (c_max <= 16) for which all `rows` clusters of C CTAs (threads each, smem dynamic bytes) can
// be resident at once, by cudaOccupancyMaxActiveClusters; c_min when none can.  Results are
// cached per device in `cache` (17 ints per device, 0 = not yet queried).
int cluster_for_one_wave(const void* kernel, int rows, int c_min, int c_max, int threads,
                         size_t smem, int* cache);
int map_cuda_error(cudaError_t); // SPECDEC_OK or SPECDEC_ERR_CUDA (clears non-sticky errors)

inline int elem_size(int dtype) { return dtype == SPECDEC_F32 ? 4 : dtype == SPECDEC_BF16 ? 2 : 0; }

}  // namespace specdec
