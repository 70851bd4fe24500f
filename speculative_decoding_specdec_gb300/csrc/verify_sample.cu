// Sampled verification (speculative rejection sampling) of D drafts per row.
//
// "Inference Engineering: Part 5/8: When Speculative Decoding Backfires",
//   "Exactness Means Different Things For Greedy And Sampled Output": a draft token x is accepted
//   with probability min(1, p(x)/q(x)) (p: main model, q: draft model, same sampling settings);
//   at a rejection the replacement is drawn from normalize(max(0, p - q));
//   "Draft Possible Tokens, Then Verify Them Together": left to right, the first rejection ends
//   the cycle, and a fully accepted draft earns a bonus token from the distribution after it.
//
// GB300 mapping.  One thread-block cluster of C CTAs per batch row b (C <= 16, chosen so the grid
// fills one wave of resident CTAs); CTA c owns the vocabulary slice [c*slice, (c+1)*slice).  A
// CTA is either 16 consumer warps with a 192 KB ring (one per SM) or 8 with a 96 KB ring (two per
// SM), whichever lets the B clusters keep more SMs busy (clusters stay inside one GPC, so the
// usable cluster sizes differ between the two).
//  Phase 1  a producer thread streams the slice of the 2D+1 score rows (D+1 target, D draft)
//           through a 192 KB shared-memory ring in 64 KB cp.async.bulk copies (rows stored back
//           to back are read as one contiguous range per CTA; its idle lanes meanwhile fetch
//           the drafts, uniforms and the two scores of every draft); 16 consumer warps keep,
//           per thread and row, a sum s of 2^(x*c2 - o) with c2 = log2(e)/T and an INTEGER offset
//           o.  A new maximum more than 64 binary orders above o moves o; rescaling by 2^(old-new)
//           is then exact, so per score element the work is one FFMA, one ex2.approx and one add.
//           Warps, the CTA (fp64) and the cluster (fp64, through distributed shared memory, one
//           per-row warp reduction) merge (o, s) pairs with the same exact scalings.
//  Phase 2  warp 0 of every CTA computes p_j(d)/q_j(d) in fp64 from the two scores of d and the
//           normalisers, accepts while u < p/q, and finds the first rejection a with a ballot.
//  Phase 3  each CTA stages its slice of row a of both models (or row D of the target for the
//           bonus) in the ring's space with two bulk copies, recomputes the residual
//           max(0, p - q) (or p_D) from it where needed, and takes a block prefix sum.  A cluster
//           barrier exchanges slice totals; the CTA whose cumulative range holds t = u[b][D] * R
//           finds the token with its block scan.
// No global scratch and no atomics; the score rows are read once (plus the one re-read row).
#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>

#include "stream.cuh"

namespace cg = cooperative_groups;

namespace specdec {
namespace {

// Two shapes of CTA: W = 16 consumer warps with a 192 KB ring (one CTA per SM) or W = 8 with a
// 96 KB ring (two per SM).  The launch takes the one whose clusters keep more SMs busy.
template <int W>
struct Cfg {
  static constexpr int kWarps = W;                // consumer warps
  static constexpr int kAllWarps = W + 1;         // plus the producer warp
  static constexpr int kThreads = kAllWarps * 32;
  static constexpr int kConsumers = W * 32;
  static constexpr int kRingBytes = W * 12288;    // W/16 * 192 KB
  static constexpr int kChunkBytes = W * 4096;    // bytes per bulk copy: three ring stages
  static constexpr int kPerSm = 16 / W;           // CTAs per SM
};
constexpr int kMaxQ = 2 * SPECDEC_MAX_DRAFT + 1;  // score rows per batch row
constexpr float kLog2e = 1.4426950408889634f;     // log2(e)
constexpr float kNegInf = -INFINITY;
constexpr float kOffsetNone = -1e30f;             // offset of an empty sum
constexpr float kRescale = 18446744073709551616.f;  // 2^64: a vector sum above it moves o

// Slice length: ceil(V / C) rounded up to whole 16-byte vectors.
__host__ __device__ constexpr int V_ceil(int V, int C, int vn) {
  return ((V + C - 1) / C + vn - 1) / vn * vn;
}

// 2^x by the PTX instruction ex2.approx.ftz.f32 (relative error within 2^-22 by the PTX ISA;
// results below the normal range are flushed to zero, which only drops negligible terms).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Exact 2^k for an integer-valued k <= 0 (offset differences), built from the IEEE-754 fields.
__device__ __forceinline__ float pow2f(float k) {
  if (!(k >= -126.f)) return 0.f;
  return __int_as_float((static_cast<int>(k) + 127) << 23);
}

// Float-float values hi + lo (|lo| <= ulp(hi)/2) summed with Knuth's TwoSum: the cross-block
// totals keep about 44 bits with fp32 instructions only (fp64 throughput is low on this GPU).
// The addition is commutative, so an xor-butterfly leaves the same bits in every lane.
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const float s = a.hi + b.hi;
  const float v = s - a.hi;
  const float e = ((a.hi - (s - v)) + (b.hi - v)) + (a.lo + b.lo);
  const float h = s + e;
  return ff{h, e - (h - s)};
}
__device__ __forceinline__ double ff_to_double(float2 a) {
  return static_cast<double>(a.x) + static_cast<double>(a.y);
}
// Merge per-lane (offset o, sum S) pairs of a warp: the largest offset M and the sum scaled to
// it (power-of-two scalings are exact).
__device__ __forceinline__ void warp_merge_ff(float o, ff S, float& M, ff& T) {
  M = o;
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, k));
  const float sc = pow2f(o - M);
  T = ff{S.hi * sc, S.lo * sc};
#pragma unroll
  for (int k = 16; k > 0; k >>= 1)
    T = ff_add(T, ff{__shfl_xor_sync(0xffffffffu, T.hi, k), __shfl_xor_sync(0xffffffffu, T.lo, k)});
}

// Merge (oo, os) into (o, s): both sums are relative to their integer offsets.
__device__ __forceinline__ void merge(float& o, float& s, float oo, float os) {
  const float M = fmaxf(o, oo);
  s = s * pow2f(o - M) + os * pow2f(oo - M);
  o = M;
}

__device__ __forceinline__ void warp_merge(float& o, float& s) {
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) {
    const float oo = __shfl_xor_sync(0xffffffffu, o, k);
    const float os = __shfl_xor_sync(0xffffffffu, s, k);
    merge(o, s, oo, os);
  }
}

// Fold N values into (o, s).
template <int N>
__device__ __forceinline__ void fold(const float* x, float c2, float& o, float& s) {
  float v = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) v += ex2(fmaf(x[i], c2, -o));
  if (!(v <= kRescale)) {  // first finite values, a much larger maximum, or NaN/+inf
    float mx = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) mx = fmaxf(mx, x[i]);
    const float on = ceilf(mx * c2);
    if (on > o) {
      s *= pow2f(o - on);
      o = on;
    }
    v = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) v += ex2(fmaf(x[i], c2, -o));
  }
  s += v;
}

// Fold four 16-byte vectors: independent tree sums (short dependency chains); if their total
// would need a new offset, fall back to folding them one by one.
template <typename T>
__device__ __forceinline__ void fold4(const uint4* r, float c2, float& o, float& s) {
  constexpr int VN = Vec<T>::N;
  float t[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float x[VN];
    Vec<T>::unpack(r[k], x);
    float e[VN];
#pragma unroll
    for (int i = 0; i < VN; ++i) e[i] = ex2(fmaf(x[i], c2, -o));
#pragma unroll
    for (int w = VN / 2; w > 0; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) e[i] += e[i + w];
    t[k] = e[0];
  }
  const float v = (t[0] + t[1]) + (t[2] + t[3]);
  if (v <= kRescale) {
    s += v;
  } else {  // first finite values, a much larger maximum, or NaN/+inf
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float x[VN];
      Vec<T>::unpack(r[k], x);
      fold<VN>(x, c2, o, s);
    }
  }
}

// fold4 for four vectors already unpacked (and masked) into floats.
template <int VN>
__device__ __forceinline__ void fold4f(const float (&x)[4][VN], float c2, float& o, float& s) {
  float t[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float e[VN];
#pragma unroll
    for (int i = 0; i < VN; ++i) e[i] = ex2(fmaf(x[k][i], c2, -o));
#pragma unroll
    for (int w = VN / 2; w > 0; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) e[i] += e[i + w];
    t[k] = e[0];
  }
  const float v = (t[0] + t[1]) + (t[2] + t[3]);
  if (v <= kRescale) {
    s += v;
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) fold<VN>(x[k], c2, o, s);
  }
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
  const uint2* keep;  // [B][2D+1] keep bounds of the sampling settings, or NULL (keep all)
  int32_t* status;
  unsigned long long seed, offset;  // uniforms == NULL: drawn in-kernel (philox_uniform)
};

// Philox4x32-10 ("Parallel Random Numbers: As Easy as 1, 2, 3", SC11): ten rounds of
// (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2, c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0), with
// the key advanced by the Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k.x += kW0;
      k.y += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, c.x), lo0 = kM0 * c.x;
    const uint32_t hi1 = __umulhi(kM1, c.z), lo1 = kM1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// The uniform u[b][j] of a round drawn from (seed, offset): word j mod 4 of Philox4x32-10 at
// counter (j div 4, b, offset lo, offset hi) and key (seed lo, seed hi), as a 24-bit value in
// [0, 1) (exact in fp32).
__device__ __forceinline__ float philox_uniform(unsigned long long seed, unsigned long long offset,
                                                int b, int j) {
  const uint4 x = philox4x32_10(
      make_uint4(static_cast<uint32_t>(j >> 2), static_cast<uint32_t>(b),
                 static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32)),
      make_uint2(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)));
  const uint32_t w = (j & 3) == 0 ? x.x : (j & 3) == 1 ? x.y : (j & 3) == 2 ? x.z : x.w;
  return static_cast<float>(w >> 8) * (1.0f / 16777216.0f);
}

// A row's keep bound (order-preserving 32-bit key of the last kept score, its index) as a float
// threshold: a token with score x at index v is kept iff x > t, or x == t and v <= ti.  Keys at
// or below the key of -inf (-inf itself, negative NaN patterns) give t = -inf.  The test keeps
// NaN (it is never below t), so a NaN score still makes its row invalid.
struct KeepF {
  float t;
  int ti;
};
__device__ __forceinline__ KeepF keep_threshold(uint2 bd) {
  constexpr uint32_t kNegInfKey = 0x007fffffu;  // key of -inf: ~0xff800000
  if (bd.x < kNegInfKey) return {kNegInf, 0x7fffffff};
  if (bd.x == kNegInfKey) return {kNegInf, static_cast<int>(bd.y)};
  const uint32_t u = (bd.x & 0x80000000u) ? (bd.x & 0x7fffffffu) : ~bd.x;
  return {__uint_as_float(u), static_cast<int>(bd.y)};
}
__device__ __forceinline__ float masked(const KeepF& k, float x, int v) {
  return (!(x < k.t) && (x != k.t || v <= k.ti)) ? x : kNegInf;
}

template <typename T, bool kVec, int W>
__global__ void __launch_bounds__(Cfg<W>::kThreads, Cfg<W>::kPerSm) sample_kernel(const SampleArgs A) {
  constexpr int kWarps = Cfg<W>::kWarps, kAllWarps = Cfg<W>::kAllWarps;
  constexpr int kThreads = Cfg<W>::kThreads, kConsumers = Cfg<W>::kConsumers;
  constexpr int kRingBytes = Cfg<W>::kRingBytes;
  extern __shared__ __align__(128) char dyn[];  // phase 1: the ring; phase 3: two staged rows
  pdl_launch_dependents();  // a realignment launched after this may start its launch now
  __shared__ float po[kMaxQ][kWarps];
  __shared__ float ps[kMaxQ][kWarps];
  __shared__ float co[kMaxQ];   // this CTA's per-row partials, read by the whole cluster
  __shared__ float2 cs[kMaxQ];  // (hi, lo)
  __shared__ float go[kMaxQ];   // cluster-combined per-row offset and normaliser
  __shared__ float2 gs[kMaxQ];
  __shared__ float incl[kThreads];
  __shared__ float wtot[32];
  __shared__ float slice_sum[2];  // this CTA's residual total (second slot: fallback to p)
  __shared__ int slice_fail[2];   // this CTA gave up a bounded wait (read by the whole cluster)
  __shared__ double s_R, s_P;
  __shared__ float s_tl, s_inv, s_iz, s_iw;
  __shared__ int s_owner, s_valid, s_chunk;
  __shared__ int s_a, s_bad, s_found, s_y, s_last, s_fail, s_cfail;
  __shared__ __align__(8) uint64_t full[kMaxRingStages], empty[kMaxRingStages], pbar;
  __shared__ StreamPlan plan;
  __shared__ KeepF s_keep[kMaxQ];            // the rows' keep thresholds (sampling settings)
  __shared__ int pre_d[SPECDEC_MAX_DRAFT];   // fetched while the slice streams
  __shared__ float pre_u[SPECDEC_MAX_DRAFT + 1], pre_z[SPECDEC_MAX_DRAFT], pre_w[SPECDEC_MAX_DRAFT];

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
  const int body = kVec ? len / VN * VN : 0;  // vector-aligned part of the slice
  // Rows stored back to back: phase 1 takes one contiguous range of the batch row's (2D+1)*V
  // scores (target rows, then draft rows; large bulk copies); otherwise the vocabulary slice of
  // every row, whose sub-vector tail is folded separately.
  const bool contiguous = kVec && A.rs == V && V % VN == 0;
  const int tail_from = contiguous ? s1 : s0 + body;

  auto row_ptr = [&](int q) -> const T* {  // q <= D: target row q; q > D: draft row q-D-1
    return q <= D ? tl + (static_cast<long long>(b) * (D + 1) + q) * A.rs
                  : dl + (static_cast<long long>(b) * D + (q - D - 1)) * A.rs;
  };

  // Draft tokens, uniforms and the two scores of each draft: fetched by the producer warp's idle
  // lanes 1..31 while the slice streams (item j = lane - 1, lane + 30, ...; D+1 uniforms).
  auto prefetch = [&](int j) {
    if (j <= D)
      pre_u[j] = A.uniforms ? A.uniforms[static_cast<long long>(b) * (D + 1) + j]
                            : philox_uniform(A.seed, A.offset, b, j);
    if (j < D) {
      const int d = A.draft[static_cast<long long>(b) * D + j];
      pre_d[j] = d;
      if (d >= 0 && d < V) {
        pre_z[j] = Vec<T>::scalar(row_ptr(j) + d);
        pre_w[j] = Vec<T>::scalar(row_ptr(D + 1 + j) + d);
      }
    }
  };

  // The producer warp sets up the ring's barriers and the stream plan and goes straight on to
  // its copies; the consumers clear the partials, read the keep bounds and wait (named barrier
  // 1) until the barriers and the plan exist.
  const bool filter = A.keep != nullptr;
  if (warp != kWarps) {
    for (int k = tid; k < kMaxQ * kWarps; k += kConsumers) {
      (&po[0][0])[k] = kOffsetNone;
      (&ps[0][0])[k] = 0.f;
    }
    for (int k = tid; k < Q; k += kConsumers)
      s_keep[k] = keep_threshold(filter ? A.keep[static_cast<long long>(b) * Q + k]
                                        : make_uint2(0u, 0x7fffffffu));
    named_bar_sync(1, kThreads);
  } else if (lane == 0) {
    s_bad = 0;
    s_found = 0;
    s_chunk = -1;
    s_last = -1;
    s_fail = 0;
    for (int k = 0; k < kMaxRingStages; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], kWarps);
    }
    mbar_init(&pbar, 1);
    fence_mbar_init();
    plan.V = V;
    plan.esize = static_cast<int>(sizeof(T));
    plan.nblk = 0;
    if (contiguous) {
      const long long nt = static_cast<long long>(D + 1) * V;  // target scores of this row
      const long long units = (nt + static_cast<long long>(D) * V) / VN;
      // 32-bit quotients where they fit (a 64-bit division is a long dependent sequence, and
      // these precede this CTA's first copy)
      const bool narrow = units * C < (1LL << 32) && nt + static_cast<long long>(D) * V < (1LL << 32);
      auto qd = [&](long long a, long long d) -> long long {
        return narrow ? static_cast<long long>(static_cast<unsigned>(a) / static_cast<unsigned>(d))
                      : a / d;
      };
      const long long e0 = qd(units * rank, C) * VN, e1 = qd(units * (rank + 1), C) * VN;
      if (e0 < nt) {  // the target part of the range
        const long long hi = min(e1, nt);
        const long long r0 = qd(e0, V);
        plan.blk[plan.nblk++] = StreamBlock{reinterpret_cast<const char*>(row_ptr(0) + e0),
                                            static_cast<int>(hi - e0), static_cast<int>(r0),
                                            static_cast<int>(e0 - r0 * V)};
      }
      if (e1 > nt) {  // the draft part
        const long long lo = max(e0, nt) - nt, hi = e1 - nt;
        const long long r0 = qd(lo, V);
        plan.blk[plan.nblk++] = StreamBlock{reinterpret_cast<const char*>(row_ptr(D + 1) + lo),
                                            static_cast<int>(hi - lo),
                                            D + 1 + static_cast<int>(r0),
                                            static_cast<int>(lo - r0 * V)};
      }
    } else if (kVec && body > 0) {
      for (int q = 0; q < Q; ++q)
        plan.blk[plan.nblk++] =
            StreamBlock{reinterpret_cast<const char*>(row_ptr(q) + s0), body, q, s0};
    }
    plan.finish(Cfg<W>::kChunkBytes / static_cast<int>(sizeof(T)), kRingBytes);
  }
  if (warp == kWarps) {
    __syncwarp();
    named_bar_arrive(1, kThreads);
  }

  // ---------------------------------------------------------------- phase 1: normalisers
  if (kVec) {
    if (warp == kWarps) {
      if (lane == 0) {
        if (!stream_produce(plan, dyn, full, empty)) s_fail = 1;
      } else {
        for (int j = lane - 1; j <= D; j += 31) prefetch(j);
      }
    } else {
      int cur = -1;
      float o = kOffsetNone, s = 0.f;
      const bool ok = stream_consume(
          plan, dyn, full, empty, [&](int q, int v0, int n, const char* stage) {  // row segment
            if (q != cur) {
              if (cur >= 0) {
                warp_merge(o, s);
                if (lane == 0) { po[cur][warp] = o; ps[cur][warp] = s; }
              }
              cur = q;
              o = kOffsetNone;
              s = 0.f;
            }
            const uint4* v4 = reinterpret_cast<const uint4*>(stage);
            const int nv = n / VN;
            int v = tid;
            if (filter) {  // sampling settings: tokens outside the row's kept set weigh 0
              // Four vectors whose largest score is below the keep threshold hold no kept token
              // and are skipped whole (a NaN is never below it, so it still reaches the fold).
              const KeepF kf = s_keep[q];
              for (; v + 3 * kConsumers < nv; v += 4 * kConsumers) {
                uint4 r[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) r[k] = v4[v + k * kConsumers];
                float x[4][VN];
                float m = kNegInf;
                if constexpr (sizeof(T) == 2) {
                  // bf16: a half is NaN iff its magnitude bits exceed 0x7f80, which one add shows
                  // for both halves of a word (no carry crosses them); the maximum of the rest
                  // decides the skip
                  uint32_t nan_bits = 0;
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    Vec<T>::unpack(r[k], x[k]);
                    const uint32_t w4[4] = {r[k].x, r[k].y, r[k].z, r[k].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) nan_bits |= (w4[j] & 0x7fff7fffu) + 0x007f007fu;
#pragma unroll
                    for (int i = 0; i < VN; ++i) m = fmaxf(m, x[k][i]);
                  }
                  if (!(nan_bits & 0x80008000u) && m < kf.t) continue;
                } else {
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    Vec<T>::unpack(r[k], x[k]);
#pragma unroll
                    for (int i = 0; i < VN; ++i) m = (x[k][i] > m || x[k][i] != x[k][i]) ? x[k][i] : m;
                  }
                  if (m < kf.t) continue;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int e0 = v0 + (v + k * kConsumers) * VN;
#pragma unroll
                  for (int i = 0; i < VN; ++i) x[k][i] = masked(kf, x[k][i], e0 + i);
                }
                fold4f<VN>(x, c2, o, s);
              }
              for (; v < nv; v += kConsumers) {
                float x[VN];
                Vec<T>::unpack(v4[v], x);
#pragma unroll
                for (int i = 0; i < VN; ++i) x[i] = masked(kf, x[i], v0 + v * VN + i);
                fold<VN>(x, c2, o, s);
              }
              return;
            }
            for (; v + 3 * kConsumers < nv; v += 4 * kConsumers) {
              uint4 r[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) r[k] = v4[v + k * kConsumers];
              fold4<T>(r, c2, o, s);
            }
            for (; v < nv; v += kConsumers) {
              float x[VN];
              Vec<T>::unpack(v4[v], x);
              fold<VN>(x, c2, o, s);
            }
          });
      if (!ok && lane == 0) s_fail = 1;
      if (cur >= 0) {
        warp_merge(o, s);
        if (lane == 0) { po[cur][warp] = o; ps[cur][warp] = s; }
      }
    }
  } else if (warp == kWarps) {
    if (lane >= 1)
      for (int j = lane - 1; j <= D; j += 31) prefetch(j);
  } else {  // rows not 16-byte aligned: plain loads
    for (int q = 0; q < Q; ++q) {
      const T* row = row_ptr(q);
      float o = kOffsetNone, s = 0.f;
      for (int e = s0 + tid; e < s1; e += kConsumers) {
        float x = masked(s_keep[q], Vec<T>::scalar(row + e), e);
        fold<1>(&x, c2, o, s);
      }
      warp_merge(o, s);
      if (lane == 0) { po[q][warp] = o; ps[q][warp] = s; }
    }
  }
  __syncthreads();
  if (s_fail && tid == 0) set_status(A.status, SPECDEC_ERR_TIMEOUT);
  for (int q = warp; q < Q; q += kAllWarps) {  // CTA partial per row, plus the tail
    float o = lane < kWarps ? po[q][lane] : kOffsetNone;
    float s = lane < kWarps ? ps[q][lane] : 0.f;
    if (lane == kWarps && kVec) {  // elements past the streamed body (fewer than one vector)
      const T* row = row_ptr(q);
      for (int e = tail_from; e < s1; ++e) {
        float x = masked(s_keep[q], Vec<T>::scalar(row + e), e);
        fold<1>(&x, c2, o, s);
      }
    }
    float M;
    ff S;
    warp_merge_ff(o, ff{s, 0.f}, M, S);
    if (lane == 0) { co[q] = M; cs[q] = make_float2(S.hi, S.lo); }
  }
  cluster.sync();  // #1: every CTA's partials are final

  // ---------------------------------------------------------------- phase 2: decisions
  // Every CTA combines the C partials of every row: a warp per row, lane r loading rank r's
  // partial through distributed shared memory (C <= 16), then a warp reduction.
  for (int q = warp; q < Q; q += kAllWarps) {
    const float o = lane < C ? cluster.map_shared_rank(co, lane)[q] : kOffsetNone;
    const float2 sp = lane < C ? cluster.map_shared_rank(cs, lane)[q] : make_float2(0.f, 0.f);
    float M;
    ff S;
    warp_merge_ff(o, ff{sp.x, sp.y}, M, S);
    if (lane == 0) {
      go[q] = M;
      gs[q] = make_float2(S.hi, S.lo);
    }
  }
  __syncthreads();
  if (warp == 0) {
    bool bad = false;
    for (int q = lane; q < Q; q += 32)  // NaN/+inf scores or an empty row
      if (!(gs[q].x > 0.f) || !isfinite(gs[q].x) || !isfinite(gs[q].y)) bad = true;
    bool accept = true;
    if (lane < D) {
      const int d = pre_d[lane];
      const float u = pre_u[lane];
      if (!(u >= 0.f && u < 1.f)) bad = true;
      if (d < 0 || d >= V) {
        bad = true;
        accept = false;
      } else {
        // A draft outside a row's kept set (or with score -inf) has probability 0 there.  With
        // q(d) = 0 the draft is accepted iff p(d) > 0: a token the target cannot emit is never
        // committed.
        const float z = masked(s_keep[lane], pre_z[lane], d);
        const float w = masked(s_keep[D + 1 + lane], pre_w[lane], d);
        if (w == kNegInf) {
          accept = z != kNegInf;
        } else if (z == kNegInf) {
          accept = false;  // p(d) = 0 < q(d)
        } else {
          // p(d)/q(d) = 2^e * S_q / S_p with e = (z - w)*c2 - (o_p - o_q).  Estimate it in fp32:
          // e as an exact float-float (TwoProd by fmaf, TwoSum), 2^e by ex2.approx of its
          // fraction (relative error below 1e-6 in all).  Decide from the estimate when it is
          // clear by a margin of 4e-6 (relative), otherwise in fp64.
          const float op = go[lane], oq = go[D + 1 + lane];
          const float dz = z - w;
          const float ph = dz * c2, pl = fmaf(dz, c2, -ph);
          const ff e = ff_add(ff{ph, pl}, ff{oq - op, 0.f});
          const float n = rintf(e.hi);
          const float f = (e.hi - n) + e.lo;
          const float r = ldexpf(ex2(f), static_cast<int>(n)) * (gs[D + 1 + lane].x / gs[lane].x);
          const bool exact_in = fabsf(op) < 4.0e6f && fabsf(oq) < 4.0e6f && isfinite(dz);
          if (exact_in && r > 1.00001f) {
            accept = true;  // ratio above 1: every u in [0, 1) accepts
          } else if (exact_in && r < 1e-30f && u > 1e-29f) {
            accept = false;  // ratio below 1e-30 and u above twice its bound
          } else if (exact_in && r >= 1e-30f && fabsf(u - r) > 4e-6f * r) {
            accept = u < r;
          } else {
            const double ed = (static_cast<double>(z) - static_cast<double>(w)) * static_cast<double>(c2) -
                              (static_cast<double>(op) - static_cast<double>(oq));
            accept = static_cast<double>(u) <
                     exp2(ed) * (ff_to_double(gs[D + 1 + lane]) / ff_to_double(gs[lane]));
          }
        }
      }
    }
    if (lane == 0) {
      const float u = pre_u[D];
      if (!(u >= 0.f && u < 1.f)) bad = true;
    }
    const unsigned rej = __ballot_sync(0xffffffffu, lane < D && !accept);
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      const int a = rej ? __ffs(static_cast<int>(rej)) - 1 : D;
      s_a = a;
      s_bad = any_bad ? 1 : 0;
      s_iz = 1.f / (gs[a].x + gs[a].y);
      s_iw = a < D ? 1.f / (gs[D + 1 + a].x + gs[D + 1 + a].y) : 0.f;
    }
  }
  __syncthreads();
  const int a = s_a;

  // ---------------------------------------------------------------- phase 3: residual draw
  // The slice of target row a (and draft row a after a rejection) is staged in shared memory
  // (the ring's space, free again): one bulk copy each, the sub-vector tail by plain loads.  The
  // residual r(i) = max(0, p_a - q_a) (or p, for the bonus and the p-fallback) is recomputed from
  // the staged scores wherever it is needed, so it needs no storage of its own.
  const bool resid = a < D;
  const T* zrow = row_ptr(a);
  const T* wrow = row_ptr(resid ? D + 1 + a : a);
  const int stage_elems = ((len * static_cast<int>(sizeof(T)) + 127) / 128 * 128) /
                          static_cast<int>(sizeof(T));
  T* zs = reinterpret_cast<T*>(dyn);
  T* ws = zs + stage_elems;
  if (kVec && body > 0 && tid == kWarps * 32) {
    const uint32_t bytes = static_cast<uint32_t>(body) * sizeof(T);
    mbar_arrive_expect_tx(&pbar, resid ? 2 * bytes : bytes);
    bulk_g2s(zs, zrow + s0, bytes, &pbar);
    if (resid) bulk_g2s(ws, wrow + s0, bytes, &pbar);
  }
  for (int i = (kVec ? body : 0) + tid; i < len; i += kThreads) {  // tail / unaligned rows
    zs[i] = zrow[s0 + i];
    if (resid) ws[i] = wrow[s0 + i];
  }
  if (kVec && body > 0) {
    const bool got = mbar_wait_sleep(&pbar, 0, kSleepTries, kSleepNs);
    if (!got) s_fail = 1;
  }
  __syncthreads();
  if (s_fail && tid == 0) set_status(A.status, SPECDEC_ERR_TIMEOUT);
  const float oz = go[a];
  const float iz = s_iz;
  const float ow = resid ? go[D + 1 + a] : 0.f;
  const float iw = s_iw;
  bool use_p = !resid;
  const KeepF kz = s_keep[a], kw = s_keep[resid ? D + 1 + a : a];
  auto zmask = [&](float x, int i) { return masked(kz, x, s0 + i); };
  auto wmask = [&](float x, int i) { return masked(kw, x, s0 + i); };
  auto r_at = [&](int i) -> float {
    const float p = ex2(fmaf(zmask(Vec<T>::scalar(zs + i), i), c2, -oz)) * iz;
    if (use_p) return p;
    return fmaxf(0.f, p - ex2(fmaf(wmask(Vec<T>::scalar(ws + i), i), c2, -ow)) * iw);
  };
  // The VN residual values of elements [i, i + VN) (i a multiple of VN, inside the slice).
  auto r_vec = [&](int i, float* r) {
    float z[VN];
    Vec<T>::unpack(*reinterpret_cast<const uint4*>(zs + i), z);
    if (filter) {
      // with sampling settings most vectors hold no kept token of row a: then every residual
      // entry is zero (p = 0 there), and no exponential is needed (a NaN is never below the
      // threshold, so a NaN row still goes through the arithmetic)
      float zm = kNegInf;
#pragma unroll
      for (int k = 0; k < VN; ++k) zm = (z[k] > zm || z[k] != z[k]) ? z[k] : zm;
      if (zm < kz.t) {
#pragma unroll
        for (int k = 0; k < VN; ++k) r[k] = 0.f;
        return;
      }
#pragma unroll
      for (int k = 0; k < VN; ++k) z[k] = zmask(z[k], i + k);
    }
#pragma unroll
    for (int k = 0; k < VN; ++k) r[k] = ex2(fmaf(z[k], c2, -oz)) * iz;
    if (!use_p) {
      float w[VN];
      Vec<T>::unpack(*reinterpret_cast<const uint4*>(ws + i), w);
      if (filter) {
#pragma unroll
        for (int k = 0; k < VN; ++k) w[k] = wmask(w[k], i + k);
      }
#pragma unroll
      for (int k = 0; k < VN; ++k) r[k] = fmaxf(0.f, r[k] - ex2(fmaf(w[k], c2, -ow)) * iw);
    }
  };
  // Block inclusive scan of per-thread contiguous chunk sums; returns the slice total.  Chunks
  // start at multiples of VN so the staged scores are read 16 bytes at a time.
  const int K = ((len + kThreads - 1) / kThreads + VN - 1) / VN * VN;
  const int c0 = min(len, tid * K), c1 = min(len, c0 + K);
  const int cv = c0 + (c1 - c0) / VN * VN;  // end of this chunk's whole vectors
  auto scan = [&]() -> float {
    float acc[VN];
#pragma unroll
    for (int k = 0; k < VN; ++k) acc[k] = 0.f;
    for (int i = c0; i < cv; i += VN) {
      float r[VN];
      r_vec(i, r);
#pragma unroll
      for (int k = 0; k < VN; ++k) acc[k] += r[k];
    }
    for (int i = cv; i < c1; ++i) acc[0] += r_at(i);
#pragma unroll
    for (int w = VN / 2; w > 0; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) acc[k] += acc[k + w];
    const float own = acc[0];
    float v = own;
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, v, k);
      if (lane >= k) v += t;
    }
    if (lane == 31) wtot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      const float wv = lane < kAllWarps ? wtot[lane] : 0.f;
      float x = wv;
#pragma unroll
      for (int k = 1; k < 32; k <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, x, k);
        if (lane >= k) x += t;
      }
      if (lane < kAllWarps) wtot[lane] = x - wv;  // exclusive warp offsets
    }
    __syncthreads();
    incl[tid] = v + wtot[warp];
    __syncthreads();
    return incl[kThreads - 1];
  };
  // R over the cluster and this CTA's offset; s_cfail: some CTA of the cluster gave up a wait
  // (its partials or staged rows are incomplete), so the row's outputs are not written.
  auto exchange = [&](int slot, float Rc) {
    if (tid == 0) {
      slice_sum[slot] = Rc;
      slice_fail[slot] = s_fail;
    }
    cluster.sync();
    if (warp == 0) {
      const float x = lane < C ? cluster.map_shared_rank(slice_sum, lane)[slot] : 0.f;
      const int f = lane < C ? cluster.map_shared_rank(slice_fail, lane)[slot] : 0;
      const bool any_fail = __any_sync(0xffffffffu, f != 0);
      if (lane == 0) s_cfail = any_fail ? 1 : 0;
      ff R{0.f, 0.f}, P{0.f, 0.f};  // rank order in every CTA: P_c + Rc_c == P_{c+1} bit for bit
      for (int r = 0; r < C; ++r) {
        const float xr = __shfl_sync(0xffffffffu, x, r);
        if (r == rank) P = R;
        R = ff_add(R, ff{xr, 0.f});
      }
      if (lane == 0) {
        s_R = ff_to_double(make_float2(R.hi, R.lo));
        s_P = ff_to_double(make_float2(P.hi, P.lo));
      }
    }
    __syncthreads();
  };

  float Rc = scan();
  exchange(0, Rc);  // #2
  if (!(s_R > 0.0) && a < D) {  // residual vanished (p == q): draw from p instead
    use_p = true;
    Rc = scan();
    exchange(1, Rc);  // #2b
  }
  if (tid == 0) {  // the draw's scalar arithmetic in fp64, on one thread
    const double R = s_R, P = s_P;
    const double t = static_cast<double>(pre_u[D]) * R;
    const bool ok = (R > 0.0) && isfinite(R) && !s_bad && !s_cfail;
    s_valid = ok ? 1 : 0;
    s_owner = (ok && Rc > 0.f && P <= t && t < P + static_cast<double>(Rc)) ? 1 : 0;
    s_tl = static_cast<float>(t - P);
    s_inv = ok ? static_cast<float>(1.0 / R) : 0.f;
  }
  __syncthreads();
  const bool valid = s_valid != 0;
  if (s_owner) {
    const float tl_ = s_tl;
    {
      const float E = tid ? incl[tid - 1] : 0.f;
      if (E <= tl_ && tl_ < incl[tid]) s_chunk = tid;  // the thread chunk that holds t
    }
    __syncthreads();
    const int oc = s_chunk;
    if (oc >= 0 && warp == oc / 32) {
      // The owning chunk [o0, o1) is searched by the whole warp: lane l sums its m entries, a
      // warp scan places the lanes, and the lane whose entries hold t walks them in order.
      const int o0 = min(len, oc * K), o1 = min(len, o0 + K);
      const int m = (o1 - o0 + 31) / 32;
      const int l0 = min(o1, o0 + lane * m), l1 = min(o1, l0 + m);
      float part = 0.f;
      int last = -1;
      for (int i = l0; i < l1; ++i) {
        const float r = r_at(i);
        part += r;
        if (r > 0.f) last = i;
      }
      float inc = part;
#pragma unroll
      for (int k = 1; k < 32; k <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, inc, k);
        if (lane >= k) inc += t;
      }
      const float E = oc ? incl[oc - 1] : 0.f;
      const unsigned hit = __ballot_sync(0xffffffffu, E + inc > tl_);
      int y = -1;
      if (hit) {
        const int hl = __ffs(static_cast<int>(hit)) - 1;
        if (lane == hl) {
          float run = E + (inc - part);
          for (int i = l0; i < l1 && y < 0; ++i) {
            run += r_at(i);
            if (run > tl_) y = i;
          }
          if (y < 0) y = last;  // rounding inside the lane's entries: its last nonzero one
        }
        y = __shfl_sync(0xffffffffu, y, hl);
      }
      if (y < 0) {  // rounding past the chunk's end: the chunk's last nonzero entry
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, k));
        y = last;
      }
      if (lane == 0 && y >= 0) { s_y = s0 + y; s_found = 1; }
    }
    __syncthreads();
    if (!s_found) {  // t rounded past this slice's scan: the slice's last nonzero entry
      int last = -1;
      for (int i = c0; i < c1; ++i)
        if (r_at(i) > 0.f) last = i;
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
  if (!valid && !s_cfail && rank == 0 && tid == 0) {
    set_status(A.status, SPECDEC_ERR_INPUT_RANGE);
    A.accept_len[b] = a;
    A.out_token[b] = -1;
  }
  if (A.residual != nullptr && valid) {
    const float inv = s_inv;
    float* out = A.residual + static_cast<long long>(b) * V;
    for (int i = tid; i < len; i += kThreads) out[s0 + i] = r_at(i) * inv;
  }
  cluster.sync();  // #3: keep shared memory alive until every CTA has read slice_sum
}

// The cluster size configuration W would use for this shape, and how many SMs it keeps busy.
struct Choice {
  int C = 0;
  double sms_busy = -1.0;
};

template <typename T, bool kVec, int W>
int prepare(const SampleArgs& A, int B, Choice* ch) {
  auto kernel = sample_kernel<T, kVec, W>;
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  static bool attr_set[64] = {false};
  static int active[64 * 17] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPECDEC_ERR_CUDA;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<W>::kRingBytes);
    if (e != cudaSuccess) return map_cuda_error(e);
    attr_set[dev] = true;
  }
  constexpr int VN = Vec<T>::N;
  // The largest cluster (up to 16 CTAs, slices >= 2048 elements, at most kPerSm CTAs per SM) for
  // which the B clusters are all resident at once, but at least the smallest one whose two
  // staged rows fit the ring.
  auto staged_bytes = [&](int c) {
    return 2LL * ((static_cast<long long>(V_ceil(A.V, c, VN)) * sizeof(T) + 127) / 128 * 128);
  };
  int c_min = 1;
  while (c_min <= 16 && staged_bytes(c_min) > Cfg<W>::kRingBytes) ++c_min;
  if (c_min > 16) return SPECDEC_OK;  // not possible with this configuration
  const int slots = sms * Cfg<W>::kPerSm;
  const int c_max = max(c_min, std::min(std::min(16, A.V / 2048), slots / max(B, 1)));
  const int C = cluster_for_one_wave(reinterpret_cast<const void*>(kernel), B, c_min, c_max,
                                     Cfg<W>::kThreads, Cfg<W>::kRingBytes, active);
  const long long ctas = static_cast<long long>(B) * C;
  const long long waves = (ctas + slots - 1) / slots;
  ch->C = C;
  ch->sms_busy = static_cast<double>(ctas) / Cfg<W>::kPerSm / static_cast<double>(waves);
  return SPECDEC_OK;
}

template <typename T, bool kVec, int W>
int launch(SampleArgs A, int B, int C, cudaStream_t stream) {
  auto kernel = sample_kernel<T, kVec, W>;
  constexpr int VN = Vec<T>::N;
  A.C = C;
  A.slice = V_ceil(A.V, C, VN);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(B) * C);
  cfg.blockDim = dim3(Cfg<W>::kThreads);
  cfg.dynamicSmemBytes = Cfg<W>::kRingBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return map_cuda_error(cudaLaunchKernelEx(&cfg, kernel, A));
}

template <typename T, bool kVec>
int launch(SampleArgs A, int B, cudaStream_t stream) {
  Choice one, two;  // W = 16 (one CTA per SM) and W = 8 (two per SM)
  int rc = prepare<T, kVec, 16>(A, B, &one);
  if (rc != SPECDEC_OK) return rc;
  rc = prepare<T, kVec, 8>(A, B, &two);
  if (rc != SPECDEC_OK) return rc;
  if (one.C == 0 && two.C == 0) return SPECDEC_ERR_UNSUPPORTED;
  if (two.C != 0 && two.sms_busy > one.sms_busy * 1.05)
    return launch<T, kVec, 8>(A, B, two.C, stream);
  return launch<T, kVec, 16>(A, B, one.C, stream);
}

}  // namespace
}  // namespace specdec

namespace specdec {
namespace {

__global__ void __launch_bounds__(256) philox_uniforms_kernel(unsigned long long seed,
                                                              unsigned long long offset, int B,
                                                              int D, float* out) {
  const long long n = static_cast<long long>(B) * (D + 1);
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += gridDim.x * 256LL)
    out[i] = philox_uniform(seed, offset, static_cast<int>(i / (D + 1)), static_cast<int>(i % (D + 1)));
}

int verify_sample_common(const void* target_logits, const void* draft_logits, int dtype, int B,
                         int D, int V, long long row_stride, float temperature,
                         const int32_t* draft, const float* uniforms, bool philox,
                         unsigned long long seed, unsigned long long offset,
                         int32_t* accept_len, int32_t* out_token,
                         float* residual_out, const void* keep_bounds, int32_t* dev_status,
                         void* stream) {
  const int es = elem_size(dtype);
  if (es == 0 || B < 0 || D < 1 || V < 1 || row_stride < V) return SPECDEC_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SPECDEC_ERR_INVALID_ARG;
  if (D > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (!target_logits || !draft_logits || !draft || !accept_len || !out_token || !dev_status ||
      (!philox && !uniforms))
    return SPECDEC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(target_logits) % es ||
      reinterpret_cast<uintptr_t>(draft_logits) % es)
    return SPECDEC_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * (D + 1) * row_stride > (1LL << 47) || B > (1 << 26))
    return SPECDEC_ERR_UNSUPPORTED;
  const bool vec = reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(draft_logits) % 16 == 0 &&
                   (row_stride * es) % 16 == 0;
  if (reinterpret_cast<uintptr_t>(keep_bounds) % 8) return SPECDEC_ERR_INVALID_ARG;
  SampleArgs A = {target_logits, draft_logits, D, V, row_stride, temperature, 1, V, draft,
                  uniforms, accept_len, out_token, residual_out,
                  static_cast<const uint2*>(keep_bounds), dev_status, seed, offset};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPECDEC_BF16)
    return vec ? launch<uint16_t, true>(A, B, s) : launch<uint16_t, false>(A, B, s);
  return vec ? launch<float, true>(A, B, s) : launch<float, false>(A, B, s);
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_verify_sample(const void* target_logits, const void* draft_logits,
                                     int dtype, int B, int D, int V, long long row_stride,
                                     float temperature, const int32_t* draft,
                                     const float* uniforms, int32_t* accept_len,
                                     int32_t* out_token, float* residual_out,
                                     const void* keep_bounds, int32_t* dev_status, void* stream) {
  return specdec::verify_sample_common(target_logits, draft_logits, dtype, B, D, V, row_stride,
                                       temperature, draft, uniforms, false, 0ull, 0ull, accept_len,
                                       out_token, residual_out, keep_bounds, dev_status, stream);
}

extern "C" int specdec_verify_sample_philox(const void* target_logits, const void* draft_logits,
                                            int dtype, int B, int D, int V, long long row_stride,
                                            float temperature, const int32_t* draft,
                                            uint64_t seed, uint64_t offset, int32_t* accept_len,
                                            int32_t* out_token, float* residual_out,
                                            const void* keep_bounds, int32_t* dev_status,
                                            void* stream) {
  return specdec::verify_sample_common(target_logits, draft_logits, dtype, B, D, V, row_stride,
                                       temperature, draft, nullptr, true, seed, offset, accept_len,
                                       out_token, residual_out, keep_bounds, dev_status, stream);
}

extern "C" int specdec_philox_uniforms(uint64_t seed, uint64_t offset, int B, int D, float* out,
                                       void* stream) {
  using namespace specdec;
  if (B < 0 || D < 1) return SPECDEC_ERR_INVALID_ARG;
  if (D > SPECDEC_MAX_DRAFT || B > (1 << 26)) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (!out) return SPECDEC_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(B) * (D + 1);
  const int grid = static_cast<int>(std::min<long long>((n + 255) / 256, 4096));
  philox_uniforms_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(seed, offset, B, D,
                                                                               out);
  return map_cuda_error(cudaGetLastError());
}
