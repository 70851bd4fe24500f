// Library-wide entry points (version, status names) and host helpers shared by the kernels.
#include <mutex>

#include "common.cuh"

namespace specdec {

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

int cluster_for_one_wave(const void* kernel, int rows, int c_min, int c_max, int threads,
                         size_t smem, int* cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return c_min;
  int* active = cache + 17 * dev;
  for (int c = c_max; c > c_min; --c) {
    if (active[c] == 0) {
      int n = -1;
      if (c > 8 && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                        1) != cudaSuccess) {
        n = -1;
      } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(c);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = -1;
      }
      (void)cudaGetLastError();
      active[c] = n == 0 ? -1 : n;
    }
    if (active[c] >= rows) return c;
  }
  return c_min;
}

int map_cuda_error(cudaError_t e) {
  if (e == cudaSuccess) return SPECDEC_OK;
  (void)cudaGetLastError();  // clear a non-sticky launch error so later calls start clean
  return SPECDEC_ERR_CUDA;
}

}  // namespace specdec

extern "C" int specdec_version(void) { return SPECDEC_VERSION; }

extern "C" const char* specdec_status_string(int status) {
  switch (status) {
    case SPECDEC_OK: return "ok";
    case SPECDEC_ERR_INVALID_ARG: return "invalid argument";
    case SPECDEC_ERR_UNSUPPORTED: return "unsupported configuration";
    case SPECDEC_ERR_CUDA: return "CUDA launch or attribute call failed";
    case SPECDEC_ERR_CAPACITY: return "destination capacity exceeded";
    case SPECDEC_ERR_INPUT_RANGE: return "input value out of range";
    case SPECDEC_ERR_TIMEOUT: return "bounded wait on an asynchronous copy ran out";
    default: return "unknown status";
  }
}

namespace specdec {
namespace {

// One thread waits, with the bounded wait the streaming kernels use for their copies, on an
// mbarrier that nothing arrives at (no copy is issued, so none can still be in flight when the
// CTA exits); when the wait gives up it records SPECDEC_ERR_TIMEOUT.
__global__ void wait_selftest_kernel(uint32_t polls, uint32_t sleep_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_sleep(&bar, 0, polls, sleep_ns)) set_status(status, SPECDEC_ERR_TIMEOUT);
  }
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_wait_selftest(uint32_t polls, uint32_t sleep_ns, int32_t* dev_status,
                                     void* stream) {
  if (polls < 1 || polls > (1u << 20) || sleep_ns > 1000000u || !dev_status)
    return SPECDEC_ERR_INVALID_ARG;
  specdec::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(polls, sleep_ns,
                                                                                dev_status);
  return specdec::map_cuda_error(cudaGetLastError());
}
