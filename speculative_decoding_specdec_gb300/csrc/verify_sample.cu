// Sampled verification (speculative rejection sampling) of D drafts per row.
//
// "Inference Engineering: Part 5/8: When Speculative Decoding Backfires",
//   "Exactness Means Different Things For Greedy And Sampled Output": a draft token x is accepted
//   with probability min(1, p(x)/q(x)) (p: main model, q: draft model, same sampling settings);
//   at a rejection the replacement is drawn from normalize(max(0, p - q));
//   "Draft Possible Tokens, Then Verify Them Together": left to right, the first rejection ends
//   the cycle, and a fully accepted draft earns a bonus token from the distribution after it.
//
// GB300 mapping.  One thread-block cluster of C CTAs per batch row b; CTA c owns the vocabulary
// slice [c*slice, (c+1)*slice).
//  Phase 1  every CTA streams its slice of the 2D+1 score rows (D+1 target, D draft) once with
//           16-byte loads and keeps a per-lane online (max, sum of exp2((x - max) * log2(e)/T));
//           warps and the CTA combine partials, the CTA's in fp64.
//  Phase 2  after a cluster barrier every CTA combines the C partials of every row through
//           distributed shared memory (same order everywhere, so every CTA gets the same bits),
//           and warp 0 computes p_j(d)/q_j(d) for each draft in fp64 from the two scores of d and
//           the normalisers, accepts while u < p/q, and finds the first rejection a with a ballot.
//  Phase 3  each CTA re-reads only row a of both models (L2-warm) or row D of the target (bonus),
//           keeps the residual max(0, p - q) (or p_D) of its slice in shared memory, and takes a
//           block prefix sum.  A second cluster barrier exchanges slice totals; the CTA whose
//           cumulative range holds t = u[b][D] * R finds the token with its block scan.
// No global scratch and no atomics; the score rows are read once (plus the one re-read row).
#include <cooperative_groups.h>

#include <cmath>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace specdec {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerLane = 4;
constexpr int kMaxQ = 2 * SPECDEC_MAX_DRAFT + 1;  // score rows per batch row
constexpr int kMaxSliceBytes = 160 * 1024;        // shared-memory residual slice
constexpr float kLog2e = 1.4426950408889634f;     // log2(e)
constexpr float kNegInf = -INFINITY;

// Slice length: ceil(V / C) rounded up to whole 16-byte vectors.
__host__ __device__ constexpr int V_ceil(int V, int C, int vn) {
  return ((V + C - 1) / C + vn - 1) / vn * vn;
}

// Merge (om, os) into (m, s): sums are relative to their maxima; -inf max means an empty sum.
__device__ __forceinline__ void merge(float& m, float& s, float om, float os, float c2) {
  const float M = fmaxf(m, om);
  const float f1 = (m == kNegInf) ? 0.f : exp2f((m - M) * c2);
  const float f2 = (om == kNegInf) ? 0.f : exp2f((om - M) * c2);
  s = s * f1 + os * f2;
  m = M;
}

__device__ __forceinline__ void warp_merge(float& m, float& s, float c2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    merge(m, s, om, os, c2);
  }
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_fmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <typename T, bool kVec>
__device__ __forceinline__ void load_row_slice(const T* row, int e, int s1, uint4& buf) {
  constexpr int VN = Vec<T>::N;
  if (kVec && e + VN <= s1) buf = ldg_stream(row + e);
}

// The VN values of elements [e, e+VN) (out of range -> -inf), from a preloaded vector if any.
template <typename T, bool kVec>
__device__ __forceinline__ void values(const T* row, int e, int s1, const uint4& buf, float* x) {
  constexpr int VN = Vec<T>::N;
  if (kVec && e + VN <= s1) {
    Vec<T>::unpack(buf, x);
  } else {
#pragma unroll
    for (int i = 0; i < VN; ++i) x[i] = (e + i < s1) ? Vec<T>::scalar(row + e + i) : kNegInf;
  }
}

struct SampleArgs {
  const void* tl;
  const void* dl;
  int D, V;
  long long rs;
  float temperature;
  int C, slice;
  const int32_t* draft;
  const float* uniforms;
  int32_t* accept_len;
  int32_t* out_token;
  float* residual;
  int32_t* status;
};

template <typename T, bool kVec>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleArgs A) {
  extern __shared__ float rbuf[];  // residual of this CTA's slice
  __shared__ float pm[kMaxQ][kWarps];
  __shared__ float ps[kMaxQ][kWarps];
  __shared__ float cm[kMaxQ];   // this CTA's per-row partials, read by the whole cluster
  __shared__ double cs[kMaxQ];
  __shared__ float gm[kMaxQ];   // cluster-combined per-row max and normaliser
  __shared__ double gs[kMaxQ];
  __shared__ float incl[kThreads];
  __shared__ float wtot[kWarps];
  __shared__ double slice_sum[2];  // this CTA's residual total (second slot: fallback to p)
  __shared__ double s_R, s_P;
  __shared__ int s_a, s_bad, s_found, s_y, s_last;

  cg::cluster_group cluster = cg::this_cluster();
  const T* tl = static_cast<const T*>(A.tl);
  const T* dl = static_cast<const T*>(A.dl);
  const int C = A.C, D = A.D, V = A.V;
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Q = 2 * D + 1;
  const int s0 = min(V, rank * A.slice);
  const int s1 = min(V, s0 + A.slice);
  const int len = s1 - s0;
  const float c2 = kLog2e / A.temperature;
  constexpr int VN = Vec<T>::N;

  auto row_ptr = [&](int q) -> const T* {  // q <= D: target row q; q > D: draft row q-D-1
    return q <= D ? tl + (static_cast<long long>(b) * (D + 1) + q) * A.rs
                  : dl + (static_cast<long long>(b) * D + (q - D - 1)) * A.rs;
  };

  for (int k = tid; k < kMaxQ * kWarps; k += kThreads) {
    (&pm[0][0])[k] = kNegInf;
    (&ps[0][0])[k] = 0.f;
  }
  if (tid == 0) { s_bad = 0; s_found = 0; s_last = -1; }
  __syncthreads();

  // ---------------------------------------------------------------- phase 1: normalisers
  {
    constexpr int UNIT = 32 * kVecPerLane * VN;
    const int segs = (len + UNIT - 1) / UNIT;
    const int units = Q * segs;
    int cur = -1;
    float m = kNegInf, s = 0.f;
    for (int u = warp; u < units; u += kWarps) {  // warp-uniform trip count
      const int q = u / segs, seg = u - q * segs;
      if (q != cur) {
        if (cur >= 0) {
          warp_merge(m, s, c2);
          if (lane == 0) { pm[cur][warp] = m; ps[cur][warp] = s; }
        }
        cur = q;
        m = kNegInf;
        s = 0.f;
      }
      const T* row = row_ptr(q);
      const int e0 = s0 + seg * UNIT;
      uint4 buf[kVecPerLane];
#pragma unroll
      for (int k = 0; k < kVecPerLane; ++k)
        load_row_slice<T, kVec>(row, e0 + (k * 32 + lane) * VN, s1, buf[k]);
      float x[kVecPerLane][VN];
      float mu = kNegInf;
#pragma unroll
      for (int k = 0; k < kVecPerLane; ++k) {
        values<T, kVec>(row, e0 + (k * 32 + lane) * VN, s1, buf[k], x[k]);
#pragma unroll
        for (int i = 0; i < VN; ++i) mu = fmaxf(mu, x[k][i]);
      }
      if (mu > m) {  // raise the running maximum (rescale what was summed so far)
        s = (m == kNegInf) ? 0.f : s * exp2f((m - mu) * c2);
        m = mu;
      }
      if (m != kNegInf) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k)
#pragma unroll
          for (int i = 0; i < VN; ++i) acc += exp2f((x[k][i] - m) * c2);
        s += acc;
      }
    }
    if (cur >= 0) {
      warp_merge(m, s, c2);
      if (lane == 0) { pm[cur][warp] = m; ps[cur][warp] = s; }
    }
  }
  __syncthreads();
  for (int q = warp; q < Q; q += kWarps) {  // CTA partial per row, in fp64
    const float m = lane < kWarps ? pm[q][lane] : kNegInf;
    const float s = lane < kWarps ? ps[q][lane] : 0.f;
    const float M = warp_fmax(m);
    const double f = (m == kNegInf) ? 0.0 : static_cast<double>(exp2f((m - M) * c2));
    const double S = warp_sum(static_cast<double>(s) * f);
    if (lane == 0) { cm[q] = M; cs[q] = S; }
  }
  cluster.sync();  // #1: every CTA's partials are final

  // ---------------------------------------------------------------- phase 2: decisions
  if (warp < 2) {
    const int q = warp * 32 + lane;
    if (q < Q) {
      float M = kNegInf;
      for (int r = 0; r < C; ++r) M = fmaxf(M, cluster.map_shared_rank(cm, r)[q]);
      double S = 0.0;
      for (int r = 0; r < C; ++r) {
        const float m = cluster.map_shared_rank(cm, r)[q];
        const double s = cluster.map_shared_rank(cs, r)[q];
        if (m != kNegInf) S += s * static_cast<double>(exp2f((m - M) * c2));
      }
      gm[q] = M;
      gs[q] = S;
    }
  }
  __syncthreads();
  if (warp == 0) {
    bool bad = false;
    for (int q = lane; q < Q; q += 32)
      if (!(gs[q] > 0.0) || !isfinite(gs[q])) bad = true;  // NaN/+inf scores or an empty row
    bool accept = true;
    if (lane < D) {
      const int d = A.draft[static_cast<long long>(b) * D + lane];
      const float u = A.uniforms[static_cast<long long>(b) * (D + 1) + lane];
      if (!(u >= 0.f && u < 1.f)) bad = true;
      if (d < 0 || d >= V) {
        bad = true;
        accept = false;
      } else {
        const double z = static_cast<double>(Vec<T>::scalar(row_ptr(lane) + d));
        const double w = static_cast<double>(Vec<T>::scalar(row_ptr(D + 1 + lane) + d));
        if (w == -INFINITY) {
          accept = true;  // q(d) = 0
        } else {
          const double lr = (z - w - (static_cast<double>(gm[lane]) - gm[D + 1 + lane])) /
                            static_cast<double>(A.temperature);
          const double ratio = exp(lr) * (gs[D + 1 + lane] / gs[lane]);  // p(d) / q(d)
          accept = static_cast<double>(u) < ratio;
        }
      }
    }
    if (lane == 0) {
      const float u = A.uniforms[static_cast<long long>(b) * (D + 1) + D];
      if (!(u >= 0.f && u < 1.f)) bad = true;
    }
    const unsigned rej = __ballot_sync(0xffffffffu, lane < D && !accept);
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_a = rej ? __ffs(static_cast<int>(rej)) - 1 : D;
      s_bad = any_bad ? 1 : 0;
    }
  }
  __syncthreads();
  const int a = s_a;

  // ---------------------------------------------------------------- phase 3: residual draw
  // rbuf[v - s0] = max(0, p_a(v) - q_a(v)) after a rejection, p_D(v) for the bonus.
  auto fill = [&](bool use_p) {
    const int rz = a;                 // target row a (a == D: the bonus row)
    const int rq = D + 1 + a;         // draft row a (a < D only)
    const T* zrow = row_ptr(rz);
    const float Mz = gm[rz];
    const float iz = static_cast<float>(1.0 / gs[rz]);
    const bool resid = (a < D) && !use_p;
    const T* wrow = resid ? row_ptr(rq) : zrow;
    const float Mw = resid ? gm[rq] : 0.f;
    const float iw = resid ? static_cast<float>(1.0 / gs[rq]) : 0.f;
    for (int e = s0 + tid * VN; e < s1; e += kThreads * VN) {
      uint4 bz = make_uint4(0, 0, 0, 0), bw = make_uint4(0, 0, 0, 0);
      load_row_slice<T, kVec>(zrow, e, s1, bz);
      if (resid) load_row_slice<T, kVec>(wrow, e, s1, bw);
      float xz[VN], xw[VN];
      values<T, kVec>(zrow, e, s1, bz, xz);
      if (resid) values<T, kVec>(wrow, e, s1, bw, xw);
#pragma unroll
      for (int i = 0; i < VN; ++i) {
        if (e + i >= s1) break;
        const float p = exp2f((xz[i] - Mz) * c2) * iz;
        float r = p;
        if (resid) r = fmaxf(0.f, p - exp2f((xw[i] - Mw) * c2) * iw);
        rbuf[e + i - s0] = r;
      }
    }
  };
  // Block inclusive scan of per-thread contiguous chunk sums; returns the slice total.
  const int K = (len + kThreads - 1) / kThreads;
  const int c0 = min(len, tid * K), c1 = min(len, c0 + K);
  auto scan = [&]() -> float {
    __syncthreads();
    float own = 0.f;
    for (int i = c0; i < c1; ++i) own += rbuf[i];
    float v = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (lane == 31) wtot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      const float wv = lane < kWarps ? wtot[lane] : 0.f;
      float x = wv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += t;
      }
      if (lane < kWarps) wtot[lane] = x - wv;  // exclusive warp offsets
    }
    __syncthreads();
    incl[tid] = v + wtot[warp];
    __syncthreads();
    return incl[kThreads - 1];
  };
  auto exchange = [&](int slot, float Rc) {  // R over the cluster and this CTA's offset
    if (tid == 0) slice_sum[slot] = static_cast<double>(Rc);
    cluster.sync();
    if (tid == 0) {
      double R = 0.0, P = 0.0;
      for (int r = 0; r < C; ++r) {
        const double x = cluster.map_shared_rank(slice_sum, r)[slot];
        if (r < rank) P += x;
        R += x;
      }
      s_R = R;
      s_P = P;
    }
    __syncthreads();
  };

  fill(false);
  float Rc = scan();
  exchange(0, Rc);  // #2
  if (!(s_R > 0.0) && a < D) {  // residual vanished (p == q): draw from p instead
    fill(true);
    Rc = scan();
    exchange(1, Rc);  // #2b
  }
  const double R = s_R, P = s_P;
  const float u_draw = A.uniforms[static_cast<long long>(b) * (D + 1) + D];
  const double t = static_cast<double>(u_draw) * R;
  const bool valid = (R > 0.0) && isfinite(R) && !s_bad;
  const bool owner = valid && Rc > 0.f && P <= t && t < P + static_cast<double>(Rc);
  if (owner) {
    const float tl_ = static_cast<float>(t - P);
    const float E = tid ? incl[tid - 1] : 0.f;
    if (E <= tl_ && tl_ < incl[tid]) {
      float run = E;
      int y = -1, last = -1;
      for (int i = c0; i < c1; ++i) {
        if (rbuf[i] > 0.f) last = i;
        run += rbuf[i];
        if (run > tl_) { y = i; break; }
      }
      if (y < 0) y = last;  // rounding inside the chunk: its last nonzero entry
      if (y >= 0) { s_y = s0 + y; s_found = 1; }
    }
    __syncthreads();
    if (!s_found) {  // t rounded past this slice's scan: the slice's last nonzero entry
      int last = -1;
      for (int i = c0; i < c1; ++i)
        if (rbuf[i] > 0.f) last = i;
      if (last >= 0) atomicMax(&s_last, last);
      __syncthreads();
      if (tid == 0) s_y = s0 + s_last;
    }
    __syncthreads();
    if (tid == 0) {
      A.accept_len[b] = a;
      A.out_token[b] = s_y;
    }
  }
  if (!valid && rank == 0 && tid == 0) {
    set_status(A.status, SPECDEC_ERR_INPUT_RANGE);
    A.accept_len[b] = a;
    A.out_token[b] = -1;
  }
  if (A.residual != nullptr && valid) {
    const float inv = static_cast<float>(1.0 / R);
    float* out = A.residual + static_cast<long long>(b) * V;
    for (int i = tid; i < len; i += kThreads) out[s0 + i] = rbuf[i] * inv;
  }
  cluster.sync();  // #3: keep shared memory alive until every CTA has read slice_sum
}

template <typename K>
int max_cluster(K kernel, int threads, size_t smem) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 8;
  if (cached[dev] == 0) {
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
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0) best = 16;
    }
    (void)cudaGetLastError();
    cached[dev] = best;
  }
  return cached[dev];
}

template <typename T, bool kVec>
int launch(SampleArgs A, int B, cudaStream_t stream) {
  auto kernel = sample_kernel<T, kVec>;
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPECDEC_ERR_CUDA;
  if (!attr_set[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSliceBytes);
    if (e != cudaSuccess) return map_cuda_error(e);
    attr_set[dev] = true;
  }
  constexpr int VN = Vec<T>::N;
  // Smallest cluster whose slices fit shared memory, then split further while the grid is below
  // two waves and slices stay >= 2048 elements.
  int C = 1;
  while (static_cast<long long>((V_ceil(A.V, C, VN))) * 4 > kMaxSliceBytes) C *= 2;
  const int cap = max_cluster(kernel, kThreads, kMaxSliceBytes);
  if (C > cap) return SPECDEC_ERR_UNSUPPORTED;
  while (C * 2 <= cap && static_cast<long long>(B) * C < 2LL * sms && A.V / (2 * C) >= 2048) C *= 2;
  A.C = C;
  A.slice = V_ceil(A.V, C, VN);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(B) * C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(A.slice) * sizeof(float);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return map_cuda_error(cudaLaunchKernelEx(&cfg, kernel, A));
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_verify_sample(const void* target_logits, const void* draft_logits,
                                     int dtype, int B, int D, int V, long long row_stride,
                                     float temperature, const int32_t* draft,
                                     const float* uniforms, int32_t* accept_len,
                                     int32_t* out_token, float* residual_out, int32_t* dev_status,
                                     void* stream) {
  using namespace specdec;
  const int es = elem_size(dtype);
  if (es == 0 || B < 0 || D < 1 || V < 1 || row_stride < V) return SPECDEC_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SPECDEC_ERR_INVALID_ARG;
  if (D > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (!target_logits || !draft_logits || !draft || !uniforms || !accept_len || !out_token ||
      !dev_status)
    return SPECDEC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(target_logits) % es || reinterpret_cast<uintptr_t>(draft_logits) % es)
    return SPECDEC_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * (D + 1) * row_stride > (1LL << 47) || B > (1 << 26))
    return SPECDEC_ERR_UNSUPPORTED;
  const bool vec = reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(draft_logits) % 16 == 0 && (row_stride * es) % 16 == 0;
  SampleArgs A = {target_logits, draft_logits, D, V, row_stride, temperature, 1, V, draft,
                  uniforms, accept_len, out_token, residual_out, dev_status};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPECDEC_BF16)
    return vec ? launch<uint16_t, true>(A, B, s) : launch<uint16_t, false>(A, B, s);
  return vec ? launch<float, true>(A, B, s) : launch<float, false>(A, B, s);
}
