// Greedy verification of D drafts per row against the target's D+1 score rows.
//
// "Inference Engineering: Part 5/8: When Speculative Decoding Backfires":
//   "Exactness Means Different Things For Greedy And Sampled Output" -- the target's choice is the
//   highest-score token; a draft is accepted while it equals that choice;
//   "Draft Possible Tokens, Then Verify Them Together" -- results are read left to right, the
//   first mismatch ends the cycle (later drafts are discarded, the target's choice replaces the
//   rejected draft), and a fully accepted draft earns a bonus token from the last row.
//
// GB300 mapping.  One thread-block cluster of C CTAs per batch row b.  CTA c of the cluster owns
// the vocabulary slice [c*slice, (c+1)*slice) of all D+1 score rows of b, streams it with 16-byte
// loads (8 in flight per lane), and keeps a running (score, index) best per lane.  Warps, then
// the CTA, reduce with the total order "higher score, then lower index", so the result does not
// depend on the reduction order and equals the row's first maximum.  Cluster rank 0 combines the
// C partial results through distributed shared memory, then one warp finds the first mismatch
// with __ballot_sync/__ffs and writes a_b and y_b.  No global scratch, no atomics, no second
// kernel.  The work is HBM-bound: B*(D+1)*V*sizeof(score) bytes are read once.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace specdec {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerLane = 8;
constexpr int kMaxRows = SPECDEC_MAX_DRAFT + 1;

// (v, i) beats (bv, bi): larger score, then lower index.  Index < 0 marks "nothing yet".
__device__ __forceinline__ bool beats(float v, int i, float bv, int bi) {
  if (i < 0) return false;
  if (bi < 0) return true;
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (beats(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Fold one element (index e, visited in ascending order by this lane) into the running best.
// NaN is never taken; the first element of a row is always taken (even -inf).
__device__ __forceinline__ void take(float x, int e, float& bv, int& bi) {
  if (x == x && (bi < 0 || x > bv)) { bv = x; bi = e; }
}

// Fold N consecutive elements starting at index e0.
template <int N>
__device__ __forceinline__ void take_vector(const float* x, int e0, float& bv, int& bi) {
  float m = x[0];
#pragma unroll
  for (int k = 1; k < N; ++k) m = fmaxf(m, x[k]);  // fmaxf drops NaN operands
  if (m == m && (bi < 0 || m > bv)) {
    int k = 0;
#pragma unroll
    for (int q = N - 1; q >= 0; --q)
      if (x[q] == m) k = q;  // first occurrence
    bv = m;
    bi = e0 + k;
  }
}

template <typename T, bool kVec>
__global__ void __launch_bounds__(kThreads)
greedy_kernel(const T* __restrict__ logits, int D, int V, long long row_stride, int C, int slice,
              const int32_t* __restrict__ draft, int32_t* __restrict__ accept_len,
              int32_t* __restrict__ out_token, int32_t* __restrict__ status) {
  __shared__ float s_v[kMaxRows][kWarps];
  __shared__ int s_i[kMaxRows][kWarps];
  __shared__ float c_v[kMaxRows];
  __shared__ int c_i[kMaxRows];

  const int rank = blockIdx.x % C;
  const int b = blockIdx.x / C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = D + 1;
  const int s0 = min(V, rank * slice);
  const int s1 = min(V, s0 + slice);

  for (int k = threadIdx.x; k < kMaxRows * kWarps; k += kThreads) {
    (&s_i[0][0])[k] = -1;
    (&s_v[0][0])[k] = 0.f;
  }
  __syncthreads();

  const T* base = logits + static_cast<long long>(b) * rows * row_stride;
  if constexpr (kVec) {
    constexpr int VN = Vec<T>::N;
    constexpr int UNIT = 32 * kVecPerLane * VN;  // elements of one warp work unit
    const int segs = (s1 - s0 + UNIT - 1) / UNIT;
    const int units = rows * segs;
    int cur = -1;
    float bv = 0.f;
    int bi = -1;
    for (int u = warp; u < units; u += kWarps) {  // warp-uniform trip count
      const int j = u / segs, seg = u - j * segs;
      if (j != cur) {
        if (cur >= 0) {
          warp_argmax(bv, bi);
          if (lane == 0) { s_v[cur][warp] = bv; s_i[cur][warp] = bi; }
        }
        cur = j;
        bv = 0.f;
        bi = -1;
      }
      const T* row = base + static_cast<long long>(j) * row_stride;
      const int e0 = s0 + seg * UNIT;
      uint4 buf[kVecPerLane];
#pragma unroll
      for (int k = 0; k < kVecPerLane; ++k) {
        const int e = e0 + (k * 32 + lane) * VN;
        if (e + VN <= s1) buf[k] = ldg_stream(row + e);
      }
#pragma unroll
      for (int k = 0; k < kVecPerLane; ++k) {
        const int e = e0 + (k * 32 + lane) * VN;
        if (e + VN <= s1) {
          float x[VN];
          Vec<T>::unpack(buf[k], x);
          take_vector<VN>(x, e, bv, bi);
        } else {
          for (int q = e; q < s1 && q < e + VN; ++q) take(Vec<T>::scalar(row + q), q, bv, bi);
        }
      }
    }
    if (cur >= 0) {
      warp_argmax(bv, bi);
      if (lane == 0) { s_v[cur][warp] = bv; s_i[cur][warp] = bi; }
    }
  } else {
    for (int j = 0; j < rows; ++j) {
      const T* row = base + static_cast<long long>(j) * row_stride;
      float bv = 0.f;
      int bi = -1;
      for (int e = s0 + threadIdx.x; e < s1; e += kThreads) take(Vec<T>::scalar(row + e), e, bv, bi);
      warp_argmax(bv, bi);
      if (lane == 0) { s_v[j][warp] = bv; s_i[j][warp] = bi; }
    }
  }
  __syncthreads();

  // CTA result per row.
  for (int j = warp; j < rows; j += kWarps) {
    float v = 0.f;
    int i = -1;
    if (lane < kWarps) { v = s_v[j][lane]; i = s_i[j][lane]; }
    warp_argmax(v, i);
    if (lane == 0) { c_v[j] = v; c_i[j] = i; }
  }
  __syncthreads();

  auto finish = [&](int g) {  // warp 0; lane j holds the target's choice g_j of row j
    const int d = lane < D ? draft[static_cast<long long>(b) * D + lane] : 0;
    const bool bad_draft = lane < D && (d < 0 || d >= V);
    const bool mismatch = lane < D && (bad_draft || g != d);
    const unsigned mm = __ballot_sync(0xffffffffu, mismatch);
    const int a = mm ? __ffs(static_cast<int>(mm)) - 1 : D;
    const int y = __shfl_sync(0xffffffffu, g, a);
    const bool bad = bad_draft || (lane < rows && g < 0);
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, SPECDEC_ERR_INPUT_RANGE);
    if (lane == 0) {
      accept_len[b] = a;
      out_token[b] = y;
    }
  };

  if (C > 1) {
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every CTA's c_v/c_i is final
    if (cluster.block_rank() == 0 && warp == 0) {
      float v = 0.f;
      int i = -1;
      if (lane < rows) {
        for (int r = 0; r < C; ++r) {
          const float ov = cluster.map_shared_rank(c_v, r)[lane];
          const int oi = cluster.map_shared_rank(c_i, r)[lane];
          if (beats(ov, oi, v, i)) { v = ov; i = oi; }
        }
      }
      finish(i);
    }
    cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
  } else if (warp == 0) {
    finish(lane < rows ? c_i[lane] : -1);
  }
}

template <typename K>
int largest_cluster(K kernel, int want, int threads) {
  // Largest power-of-two cluster size <= want that the device can co-schedule (16 needs the
  // non-portable opt-in; fall back to the portable 8).
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] == 0) {
    int best = 8;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 16;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(threads);
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0) best = 16;
    }
    (void)cudaGetLastError();
    cached[dev] = best;
  }
  const int cap = (dev >= 0 && dev < 64) ? cached[dev] : 8;
  int c = 1;
  while (c * 2 <= want && c * 2 <= cap) c *= 2;
  return c;
}

template <typename T, bool kVec>
int launch(const void* logits, int B, int D, int V, long long row_stride, const int32_t* draft,
           int32_t* accept_len, int32_t* out_token, int32_t* status, cudaStream_t stream) {
  auto kernel = greedy_kernel<T, kVec>;
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  // Split the vocabulary while the grid is below two waves and slices stay >= 1024 elements.
  int want = 1;
  while (want < 16 && static_cast<long long>(B) * want < 2LL * sms && V / (2 * want) >= 1024)
    want *= 2;
  const int C = largest_cluster(kernel, want, kThreads);
  constexpr int VN = Vec<T>::N;
  int slice = (V + C - 1) / C;
  slice = (slice + VN - 1) / VN * VN;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(B) * C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<const T*>(logits), D, V,
                                           row_stride, C, slice, draft, accept_len, out_token,
                                           status);
  return map_cuda_error(e);
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_verify_greedy(const void* logits, int dtype, int B, int D, int V,
                                     long long row_stride, const int32_t* draft,
                                     int32_t* accept_len, int32_t* out_token, int32_t* dev_status,
                                     void* stream) {
  using namespace specdec;
  const int es = elem_size(dtype);
  if (es == 0 || B < 0 || D < 1 || V < 1 || row_stride < V) return SPECDEC_ERR_INVALID_ARG;
  if (D > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (!logits || !draft || !accept_len || !out_token || !dev_status) return SPECDEC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % es != 0) return SPECDEC_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * (D + 1) * row_stride > (1LL << 47)) return SPECDEC_ERR_UNSUPPORTED;
  if (B > (1 << 26)) return SPECDEC_ERR_UNSUPPORTED;
  const bool vec = reinterpret_cast<uintptr_t>(logits) % 16 == 0 && (row_stride * es) % 16 == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPECDEC_BF16)
    return vec ? launch<uint16_t, true>(logits, B, D, V, row_stride, draft, accept_len, out_token, dev_status, s)
               : launch<uint16_t, false>(logits, B, D, V, row_stride, draft, accept_len, out_token, dev_status, s);
  return vec ? launch<float, true>(logits, B, D, V, row_stride, draft, accept_len, out_token, dev_status, s)
             : launch<float, false>(logits, B, D, V, row_stride, draft, accept_len, out_token, dev_status, s);
}
