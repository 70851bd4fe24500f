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
// a share of the batch row's D+1 score rows: one contiguous range of them when the rows are
// stored back to back (else its vocabulary slice [c*slice, (c+1)*slice) of every row).  A
// producer thread streams the share through a shared-memory ring in 32 KB cp.async.bulk copies
// (192 KB ring and one CTA per SM when the rows fit on the SMs); 16 consumer warps scan each
// stage row segment by row segment with 16-byte shared loads and keep a
// running (score, index) best per thread.  Warps, then the CTA, reduce with the total order
// "higher score, then lower index", so the result does not depend on the reduction order and
// equals the row's first maximum.  Cluster rank 0 combines the C partial results through
// distributed shared memory (a warp per row, a lane per rank), then one warp finds the first
// mismatch with __ballot_sync/__ffs and writes a_b and y_b.  No global scratch, no atomics, one
// launch.  The work is HBM-bound: B*(D+1)*V*sizeof(score) bytes are read once.
#include <cooperative_groups.h>

#include <algorithm>

#include "stream.cuh"

namespace cg = cooperative_groups;

namespace specdec {
namespace {

constexpr int kWarps = 16;                 // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;  // plus one producer warp
constexpr int kConsumers = kWarps * 32;
constexpr int kRingLarge = 192 * 1024;  // one CTA per SM (B <= SMs)
constexpr int kRingSmall = 96 * 1024;   // two CTAs per SM (more rows than SMs)
constexpr int kChunkBytes = 32768;      // bytes per bulk copy
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
  float t[N];
#pragma unroll
  for (int k = 0; k < N; ++k) t[k] = x[k];
#pragma unroll
  for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
    for (int k = 0; k < w; ++k) t[k] = fmaxf(t[k], t[k + w]);  // fmaxf drops NaN operands
  const float m = t[0];
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
              int ring_bytes, const int32_t* __restrict__ draft, int32_t* __restrict__ accept_len,
              int32_t* __restrict__ out_token, int32_t* __restrict__ status) {
  extern __shared__ __align__(128) char ring[];
  __shared__ float s_v[kMaxRows][kWarps];
  __shared__ int s_i[kMaxRows][kWarps];
  __shared__ float c_v[kMaxRows];
  __shared__ int c_i[kMaxRows];
  __shared__ __align__(8) uint64_t full[kMaxRingStages], empty[kMaxRingStages];
  __shared__ StreamPlan plan;
  __shared__ int s_fail;
  __shared__ int pre_d[kMaxRows];  // draft tokens, fetched while the slice streams

  const int rank = blockIdx.x % C;
  const int b = blockIdx.x / C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = D + 1;
  const int s0 = min(V, rank * slice);
  const int s1 = min(V, s0 + slice);
  constexpr int VN = Vec<T>::N;
  const T* base = logits + static_cast<long long>(b) * rows * row_stride;
  auto row_ptr = [&](int q) { return base + static_cast<long long>(q) * row_stride; };
  // Rows stored back to back: the CTA takes one contiguous range of the batch row's rows*V
  // scores (large bulk copies); otherwise its vocabulary slice of every row.
  const bool contiguous = kVec && row_stride == V && V % VN == 0;
  const int body = (kVec && !contiguous) ? (s1 - s0) / VN * VN : 0;  // per-row streamed part

  for (int k = threadIdx.x; k < kMaxRows * kWarps; k += kThreads) {
    (&s_i[0][0])[k] = -1;
    (&s_v[0][0])[k] = 0.f;
  }
  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int k = 0; k < kMaxRingStages; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], kWarps);
    }
    fence_mbar_init();
    plan.V = V;
    plan.esize = static_cast<int>(sizeof(T));
    plan.nblk = 0;
    if (contiguous) {
      const long long units = static_cast<long long>(rows) * V / VN;
      const long long e0 = units * rank / C * VN, e1 = units * (rank + 1) / C * VN;
      if (e1 > e0) {
        plan.blk[0] = StreamBlock{reinterpret_cast<const char*>(base + e0),
                                  static_cast<int>(e1 - e0), static_cast<int>(e0 / V),
                                  static_cast<int>(e0 % V)};
        plan.nblk = 1;
      }
    } else if (kVec && body > 0) {
      for (int q = 0; q < rows; ++q)
        plan.blk[q] = StreamBlock{reinterpret_cast<const char*>(row_ptr(q) + s0), body, q, s0};
      plan.nblk = rows;
    }
    plan.finish(kChunkBytes / static_cast<int>(sizeof(T)), ring_bytes);
  }
  __syncthreads();

  if constexpr (kVec) {
    if (warp == kWarps) {
      if (lane == 0) {
        if (!stream_produce(plan, ring, full, empty)) s_fail = 1;
      } else if (lane <= D) {
        pre_d[lane - 1] = draft[static_cast<long long>(b) * D + lane - 1];
      }
    } else {
      int cur = -1;
      float bv = 0.f;
      int bi = -1;
      const bool ok = stream_consume(
          plan, ring, full, empty, [&](int q, int v0, int n, const char* data) {
            if (q != cur) {
              if (cur >= 0) {
                warp_argmax(bv, bi);
                if (lane == 0) { s_v[cur][warp] = bv; s_i[cur][warp] = bi; }
              }
              cur = q;
              bv = 0.f;
              bi = -1;
            }
            const uint4* v4 = reinterpret_cast<const uint4*>(data);
            const int nv = n / VN;
            int v = threadIdx.x;  // ascending index order per thread
            for (; v + 3 * kConsumers < nv; v += 4 * kConsumers) {
              uint4 r[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) r[k] = v4[v + k * kConsumers];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float x[VN];
                Vec<T>::unpack(r[k], x);
                take_vector<VN>(x, v0 + (v + k * kConsumers) * VN, bv, bi);
              }
            }
            for (; v < nv; v += kConsumers) {
              float x[VN];
              Vec<T>::unpack(v4[v], x);
              take_vector<VN>(x, v0 + v * VN, bv, bi);
            }
          });
      if (!ok && lane == 0) s_fail = 1;
      if (cur >= 0) {
        warp_argmax(bv, bi);
        if (lane == 0) { s_v[cur][warp] = bv; s_i[cur][warp] = bi; }
      }
    }
  } else if (warp == kWarps) {
    if (lane >= 1 && lane <= D) pre_d[lane - 1] = draft[static_cast<long long>(b) * D + lane - 1];
  } else {
    for (int j = 0; j < rows; ++j) {
      const T* row = row_ptr(j);
      float bv = 0.f;
      int bi = -1;
      for (int e = s0 + threadIdx.x; e < s1; e += kConsumers) take(Vec<T>::scalar(row + e), e, bv, bi);
      warp_argmax(bv, bi);
      if (lane == 0) { s_v[j][warp] = bv; s_i[j][warp] = bi; }
    }
  }
  __syncthreads();
  if (s_fail && threadIdx.x == 0) set_status(status, SPECDEC_ERR_TIMEOUT);

  // CTA result per row, then the few tail elements past the streamed body (higher indices).
  for (int j = warp; j < rows; j += kWarps + 1) {
    float v = 0.f;
    int i = -1;
    if (lane < kWarps) { v = s_v[j][lane]; i = s_i[j][lane]; }
    warp_argmax(v, i);
    if (lane == 0) {
      const T* row = row_ptr(j);
      for (int e = s0 + body; kVec && !contiguous && e < s1; ++e) {
        const float x = Vec<T>::scalar(row + e);
        if (x == x && beats(x, e, v, i)) { v = x; i = e; }
      }
      c_v[j] = v;
      c_i[j] = i;
    }
  }
  __syncthreads();

  __shared__ int g_row[kMaxRows];
  auto finish = [&](int g) {  // warp 0; lane j holds the target's choice g_j of row j
    const int d = lane < D ? pre_d[lane] : 0;
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
    if (cluster.block_rank() == 0) {
      // A warp per row: lane r loads rank r's partial through distributed shared memory (C <= 16),
      // then a warp reduction with the same total order.
      for (int j = warp; j < rows; j += kWarps + 1) {
        float v = 0.f;
        int i = -1;
        if (lane < C) {
          v = cluster.map_shared_rank(c_v, lane)[j];
          i = cluster.map_shared_rank(c_i, lane)[j];
        }
        warp_argmax(v, i);
        if (lane == 0) g_row[j] = i;
      }
      __syncthreads();
      if (warp == 0) finish(lane < rows ? g_row[lane] : -1);
    }
    cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
  } else if (warp == 0) {
    finish(lane < rows ? c_i[lane] : -1);
  }
}

template <typename T, bool kVec>
int launch(const void* logits, int B, int D, int V, long long row_stride, const int32_t* draft,
           int32_t* accept_len, int32_t* out_token, int32_t* status, cudaStream_t stream) {
  auto kernel = greedy_kernel<T, kVec>;
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPECDEC_ERR_CUDA;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kRingLarge);
    if (e != cudaSuccess) return map_cuda_error(e);
    attr_set[dev] = true;
  }
  // Up to as many rows as SMs: one CTA per SM with the large ring, splitting each row over the
  // largest cluster (up to 16 CTAs, slices >= 1024 elements, at most SMs/B CTAs per row) whose B
  // clusters are all resident at once.  More rows: the small ring, two CTAs per SM, one CTA per
  // row where that fits.
  const bool large = B <= sms;
  const int ring = kVec ? (large ? kRingLarge : kRingSmall) : 0;
  static int active_large[64 * 17] = {0}, active_small[64 * 17] = {0};
  const int c_max = large ? std::max(1, std::min(std::min(16, V / 1024), sms / B)) : 1;
  const int C = cluster_for_one_wave(reinterpret_cast<const void*>(kernel), B, 1, c_max, kThreads,
                                     ring, large ? active_large : active_small);
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
  cfg.dynamicSmemBytes = ring;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<const T*>(logits), D, V,
                                           row_stride, C, slice, ring, draft, accept_len, out_token,
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
