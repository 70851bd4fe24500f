// EXSPEC grouping of a SequencePool by length.
//
// "Batch Speculative Decoding Done Right", section 2.3: keep a pool of active sequences and
// group same-length sequences into batches, which then need no realignment; only the
// mixed-length rows are realigned.
//
// One CTA: a stable counting sort by length.  Per length v with count c_v, the first
// floor(c_v / bs) * bs rows (index order) form uniform batches and the rest are leftovers.  Two
// exclusive scans over the length buckets give each length's start in the uniform section and
// in the leftover section; a row's place is its bucket start plus its rank among earlier rows of
// the same length.  Latency-bound (a few KB in and out), not a roofline kernel.
#include "common.cuh"

namespace specdec {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxN = 4096;
constexpr int kMaxLen = 16383;

__global__ void __launch_bounds__(kThreads)
group_kernel(const int32_t* __restrict__ lengths, int N, int bs, int max_len,
             int32_t* __restrict__ perm, int32_t* __restrict__ offsets,
             uint8_t* __restrict__ uniform, int32_t* __restrict__ num_batches,
             int32_t* __restrict__ num_uniform, int32_t* __restrict__ status) {
  extern __shared__ int sm[];
  const int M = max_len + 1;       // length buckets 0..max_len
  int* ustart = sm;                // [M+1] uniform-section start of each length
  int* lstart = ustart + (M + 1);  // [M+1] leftover-section start of each length
  int* lens = lstart + (M + 1);    // [N]
  __shared__ int s_bad;
  __shared__ int s_part[2][kThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_bad = 0;
  for (int v = tid; v <= M; v += kThreads) ustart[v] = 0;
  __syncthreads();
  for (int i = tid; i < N; i += kThreads) {
    const int v = lengths[i];
    lens[i] = v;
    if (v < 0 || v > max_len) s_bad = 1;
    else atomicAdd(&ustart[v], 1);  // counts for now
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) set_status(status, SPECDEC_ERR_INPUT_RANGE);
    return;
  }

  // Exclusive scans over buckets of u_v = floor(c_v/bs)*bs and l_v = c_v - u_v (thread-contiguous
  // bucket chunks, then a block scan of the chunk totals).
  const int per = (M + kThreads - 1) / kThreads;
  const int v0 = min(M, tid * per), v1 = min(M, v0 + per);
  int su = 0, sl = 0;
  for (int v = v0; v < v1; ++v) {
    const int c = ustart[v];
    const int u = c / bs * bs;
    su += u;
    sl += c - u;
  }
  int iu = su, il = sl;  // inclusive warp scans
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, iu, o);
    const int b = __shfl_up_sync(0xffffffffu, il, o);
    if (lane >= o) { iu += a; il += b; }
  }
  if (lane == 31) { s_part[0][warp] = iu; s_part[1][warp] = il; }
  __syncthreads();
  if (warp == 0) {
    const int pu = s_part[0][lane], pl = s_part[1][lane];  // kThreads / 32 == 32 warps
    int xu = pu, xl = pl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, xu, o);
      const int b = __shfl_up_sync(0xffffffffu, xl, o);
      if (lane >= o) { xu += a; xl += b; }
    }
    s_part[0][lane] = xu - pu;  // exclusive warp offsets
    s_part[1][lane] = xl - pl;
  }
  __syncthreads();
  int ru = s_part[0][warp] + iu - su, rl = s_part[1][warp] + il - sl;
  for (int v = v0; v < v1; ++v) {  // each thread rewrites only its own buckets
    const int c = ustart[v];
    const int u = c / bs * bs;
    ustart[v] = ru;
    lstart[v] = rl;
    ru += u;
    rl += c - u;
  }
  if (tid == kThreads - 1) {  // the last thread's running sums are the totals
    ustart[M] = ru;
    lstart[M] = rl;
  }
  __syncthreads();
  const int TU = ustart[M];

  for (int i = tid; i < N; i += kThreads) {
    const int v = lens[i];
    int rank = 0;
    for (int j = 0; j < i; ++j) rank += (lens[j] == v);
    const int u = ustart[v + 1] - ustart[v];
    perm[rank < u ? ustart[v] + rank : TU + lstart[v] + (rank - u)] = i;
  }
  const int nu = TU / bs;
  const int nm = (N - TU + bs - 1) / bs;
  for (int k = tid; k <= nu + nm; k += kThreads) {
    offsets[k] = k <= nu ? k * bs : min(N, TU + (k - nu) * bs);
    if (k < nu + nm) uniform[k] = k < nu ? 1 : 0;
  }
  if (tid == 0) {
    *num_batches = nu + nm;
    *num_uniform = nu;
  }
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_group_by_length(const int32_t* lengths, int N, int batch_size, int max_len,
                                       int32_t* perm, int32_t* batch_offsets,
                                       uint8_t* batch_uniform, int32_t* num_batches,
                                       int32_t* num_uniform, int32_t* dev_status, void* stream) {
  using namespace specdec;
  if (N < 0 || batch_size < 1 || max_len < 0) return SPECDEC_ERR_INVALID_ARG;
  if (N > kMaxN || max_len > kMaxLen) return SPECDEC_ERR_UNSUPPORTED;
  if ((N > 0 && (!lengths || !perm || !batch_uniform)) || !batch_offsets || !num_batches ||
      !num_uniform || !dev_status)
    return SPECDEC_ERR_INVALID_ARG;
  const size_t smem = (2 * static_cast<size_t>(max_len + 2) + N) * sizeof(int);
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPECDEC_ERR_CUDA;
  if (!attr_set[dev]) {
    const int most = static_cast<int>((2 * static_cast<size_t>(kMaxLen + 2) + kMaxN) * sizeof(int));
    const cudaError_t e =
        cudaFuncSetAttribute(group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return map_cuda_error(e);
    attr_set[dev] = true;
  }
  group_kernel<<<1, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      lengths, N, batch_size, max_len, perm, batch_offsets, batch_uniform, num_batches,
      num_uniform, dev_status);
  return map_cuda_error(cudaGetLastError());
}
