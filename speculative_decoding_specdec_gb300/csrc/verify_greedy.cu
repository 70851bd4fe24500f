// Greedy verification of D drafts per row against the target's D+1 score rows.
//
// "Inference Engineering: Part 5/8: When Speculative Decoding Backfires":
//   "Exactness Means Different Things For Greedy And Sampled Output" -- the target's choice is the
//   highest-score token; a draft is accepted while it equals that choice;
//   "Draft Possible Tokens, Then Verify Them Together" -- results are read left to right, the
//   first mismatch ends the cycle (later drafts are discarded, the target's choice replaces the
//   rejected draft), and a fully accepted draft earns a bonus token from the last row.
//
// GB300 mapping.  The B*(D+1) score rows form one virtual sequence of 16-byte units (each row
// padded to whole units); the grid splits it into equal contiguous shares, so every SM streams
// the same number of bytes whatever B, D and V are.  Rows stored back to back are streamed by one
// CTA per SM through a shared-memory ring of bulk copies (greedy_ring_kernel: the whole share is
// in flight at once); other layouts by up to two CTAs per SM with 16-byte loads, where each
// thread walks its units (one every kThreads) with a cursor that only adds, keeps 8 loads in
// flight across row boundaries, and folds elements into a running best.  A best is a 64-bit key
// (order-preserving score bits above the complemented index), so "higher score, then lower index"
// is a plain integer maximum and the result is the row's first maximum whatever the order of
// reduction.  On a row change a thread merges its key into a shared-memory slot of that row
// (atomicMax); after one barrier the CTA merges its slots into the per-row keys of the workspace
// (red.max at GPU scope) and takes a ticket on each batch row it touched.  The CTA that takes a
// batch row's last ticket reads that row's D+1 keys at once, finds the first mismatch with
// __ballot_sync/__ffs, writes a_b and y_b, and sets the keys and the ticket back to zero.  One
// launch, no waiting between CTAs; the work is B*(D+1)*V*sizeof(score) bytes of HBM, read once.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "stream.cuh"

namespace specdec {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 8;          // 16-byte loads in flight per thread
constexpr int kMinUnits = 512;      // fewest units a CTA is given
constexpr int kMaxSegs = 1024;      // row segments one CTA may touch (shared-memory key slots)
constexpr long long kMaxShare = 1LL << 30;  // units per CTA, at most (32-bit local offsets)

// Score -> unsigned integer with the same order (-0 counted as +0).  NaN is never encoded.
__device__ __forceinline__ uint32_t order_bits(float f) {
  const uint32_t u = (f == 0.f) ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Key of (score, index): larger score first, then lower index.  0 means "no element".
__device__ __forceinline__ unsigned long long make_key(float v, int i) {
  return (static_cast<unsigned long long>(order_bits(v)) << 32) | static_cast<uint32_t>(~i);
}

// Fold one element (indices visited in ascending order by this thread) into the running best.
// NaN is never taken; the first non-NaN element of a row is always taken (even -inf).
__device__ __forceinline__ void take(float x, int e, float& bv, int& bi) {
  if (x == x && (bi < 0 || x > bv)) { bv = x; bi = e; }
}

// Fold N consecutive elements starting at index e0 (max tree, first occurrence).
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

__device__ __forceinline__ void red_max_gpu(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Equal contiguous shares of `units` units over G CTAs (G <= units, so no share is empty).
// narrow: units * G < 2^32, so every product and quotient below fits 32-bit unsigned arithmetic
// (a 64-bit division is a long dependent instruction sequence on the GPU; these sit on the
// critical path of a launch's start and of its per-row merge).
struct Split {
  long long units;
  int G;
  int narrow;
  __device__ __host__ long long start(int c) const {
    if (narrow)
      return static_cast<long long>(static_cast<unsigned>(units) * static_cast<unsigned>(c) /
                                    static_cast<unsigned>(G));
    return units * c / G;
  }
  // The CTA whose share holds unit u: the largest c with start(c) <= u.
  __device__ int owner(long long u) const {
    if (narrow)
      return static_cast<int>((static_cast<unsigned>(u + 1) * static_cast<unsigned>(G) - 1u) /
                              static_cast<unsigned>(units));
    return static_cast<int>(((u + 1) * G - 1) / units);
  }
  // u / d for 0 <= u <= units and d >= 1.
  __device__ long long div(long long u, int d) const {
    if (narrow) return static_cast<long long>(static_cast<unsigned>(u) / static_cast<unsigned>(d));
    return u / d;
  }
};

struct GreedyArgs {
  const void* logits;
  int B, D, V;
  int RU;                   // units per row (row padded to whole units)
  int RUfull;               // whole units inside [0, V)
  int step_rows, step_off;  // kThreads units = step_rows rows + step_off units
  long long row_stride;     // elements
  Split split;
  const int32_t* draft;
  int32_t* accept_len;
  int32_t* out_token;
  int32_t* status;
  unsigned long long* key;  // [B*(D+1)], zero between calls
  unsigned* ticket;         // [B], zero between calls
};

// Position of one unit: row (relative to the CTA's first row) and unit within the row.
struct Cursor {
  int row, off;
  __device__ __forceinline__ void init(const GreedyArgs& A, int lu) {
    row = lu / A.RU;
    off = lu - row * A.RU;
  }
  __device__ __forceinline__ bool advance(const GreedyArgs& A) {  // by kThreads units
    row += A.step_rows;
    off += A.step_off;
    const bool wrap = off >= A.RU;
    if (wrap) {
      off -= A.RU;
      ++row;
    }
    return wrap;
  }
};

// A CTA whose bounded wait ran out adds this to each ticket it takes besides its count of one,
// so that the CTA taking the last ticket knows a contributing CTA's keys are incomplete.  The
// count stays below it: a batch row is touched by at most 2 CTAs per SM.
constexpr unsigned kTicketFail = 1u << 20;

// After a CTA's row segments are final in s_key: merge them into the per-row keys of the
// workspace, take one ticket per batch row touched, and decide the batch rows whose last ticket
// this CTA took.  `failed`: this CTA's stream gave up (SPECDEC_ERR_TIMEOUT is already set); a
// batch row with such a contributor gets no accept length or token, but its keys and ticket are
// still reset for the next call.  NT = threads of the CTA.
template <int NT>
__device__ void merge_and_decide(const GreedyArgs& A, const unsigned long long* s_key,
                                 unsigned char* s_last, long long g0, long long g1, int nseg,
                                 bool failed) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Q = A.D + 1;
  // Merge this CTA's row segments into the per-row keys, then take one ticket per batch row.
  for (int s = tid; s < nseg; s += NT) {
    if (s_key[s] != 0ull) red_max_gpu(&A.key[g0 + s], s_key[s]);
    fence_acq_rel_gpu();
  }
  __syncthreads();
  const long long b0 = A.split.div(g0, Q), b1 = A.split.div(g1, Q);
  const int nb = static_cast<int>(b1 - b0 + 1);
  for (int k = tid; k < nb; k += NT) {
    const long long b = b0 + k;
    const long long r0 = b * Q * A.RU, r1 = (b + 1) * Q * A.RU - 1;  // its units
    const unsigned expected =
        static_cast<unsigned>(A.split.owner(r1) - A.split.owner(r0) + 1);
    const unsigned inc = failed ? 1u + kTicketFail : 1u;
    const unsigned old = atom_add_acq_rel_gpu(&A.ticket[b], inc);
    s_last[k] = (old & (kTicketFail - 1u)) != expected - 1u ? 0 : (old + inc >= kTicketFail ? 2 : 1);
  }
  __syncthreads();
  for (int k = warp; k < nb; k += NT / 32) {
    if (!s_last[k]) continue;
    const long long b = b0 + k;
    int g = -1;  // lane j: the target's choice of row j of batch row b
    if (lane < Q) {
      const unsigned long long key = ld_relaxed_gpu(&A.key[b * Q + lane]);
      if (key != 0ull) g = static_cast<int>(~static_cast<uint32_t>(key));
    }
    const int D = A.D;
    const int d = lane < D ? A.draft[b * D + lane] : 0;
    const bool bad_draft = lane < D && (d < 0 || d >= A.V);
    const bool mismatch = lane < D && (bad_draft || g != d);
    const unsigned mm = __ballot_sync(0xffffffffu, mismatch);
    const int a = mm ? __ffs(static_cast<int>(mm)) - 1 : D;
    const int y = __shfl_sync(0xffffffffu, g, a);
    const bool bad = bad_draft || (lane < Q && g < 0);
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(A.status, SPECDEC_ERR_INPUT_RANGE);
    if (lane < Q) A.key[b * Q + lane] = 0ull;  // ready for the next call
    if (lane == 0) {
      if (s_last[k] == 1) {  // 2: a contributing CTA's stream gave up, its keys are incomplete
        A.accept_len[b] = a;
        A.out_token[b] = y;
      }
      A.ticket[b] = 0u;
    }
  }
}

template <typename T, bool kVec>
__global__ void __launch_bounds__(kThreads, 2) greedy_kernel(const GreedyArgs A) {
  __shared__ unsigned long long s_key[kMaxSegs];
  __shared__ unsigned char s_last[kMaxSegs];
  pdl_launch_dependents();  // a realignment launched after this may start its launch now

  constexpr int VN = kVec ? Vec<T>::N : 1;
  const int c = blockIdx.x;
  const int tid = threadIdx.x;
  const long long u0 = A.split.start(c), u1 = A.split.start(c + 1);
  const long long g0 = A.split.div(u0, A.RU), g1 = A.split.div(u1 - 1, A.RU);  // rows touched
  const int nseg = static_cast<int>(g1 - g0 + 1);
  if (nseg > kMaxSegs) {  // excluded by the launch geometry
    if (tid == 0) set_status(A.status, SPECDEC_ERR_UNSUPPORTED);
    return;
  }
  for (int s = tid; s < nseg; s += kThreads) s_key[s] = 0ull;
  __syncthreads();

  const T* base = static_cast<const T*>(A.logits) + g0 * A.row_stride;
  const int lu0 = static_cast<int>(u0 - g0 * A.RU), lu1 = static_cast<int>(u1 - g0 * A.RU);
  float bv = 0.f;
  int bi = -1, prow = 0;
  auto flush = [&](int row) {
    if (bi >= 0) atomicMax(&s_key[row], make_key(bv, bi));
    bi = -1;
  };
  // Load and fold cursors walk the same units, the fold cursor kUnroll units behind.  The load
  // cursor also carries the unit's address.
  Cursor L, P;
  L.init(A, lu0 + tid);
  P = L;
  prow = P.row;
  const T* lp = base + L.row * A.row_stride + static_cast<long long>(L.off) * VN;
  const long long jump = A.step_rows * A.row_stride + static_cast<long long>(A.step_off) * VN;
  const long long wrap = A.row_stride - static_cast<long long>(A.RU) * VN;
  for (int lu = lu0 + tid; lu < lu1; lu += kThreads * kUnroll) {
    if constexpr (kVec) {
      uint4 r[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (lu + k * kThreads < lu1 && L.off < A.RUfull) r[k] = ldg_stream(lp);
        lp += jump;
        if (L.advance(A)) lp += wrap;
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (lu + k * kThreads < lu1) {
          if (P.row != prow) { flush(prow); prow = P.row; }
          const int e = P.off * VN;
          if (P.off < A.RUfull) {
            float x[VN];
            Vec<T>::unpack(r[k], x);
            take_vector<VN>(x, e, bv, bi);
          } else {  // the row's last, partial unit: only its elements below V exist
            const T* row = base + P.row * A.row_stride;
            for (int j = e; j < A.V; ++j) take(Vec<T>::scalar(row + j), j, bv, bi);
          }
        }
        P.advance(A);
      }
    } else {
      float r[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (lu + k * kThreads < lu1) r[k] = Vec<T>::scalar(lp);
        lp += jump;
        if (L.advance(A)) lp += wrap;
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        if (lu + k * kThreads < lu1) {
          if (P.row != prow) { flush(prow); prow = P.row; }
          take(r[k], P.off, bv, bi);
        }
        P.advance(A);
      }
    }
  }
  flush(prow);
  __syncthreads();

  merge_and_decide<kThreads>(A, s_key, s_last, g0, g1, nseg, false);  // no waits in this kernel
}


// Rows stored back to back (row_stride == V, V a multiple of the vector width, 16-byte aligned):
// one CTA per SM streams its share through a 192 KB shared-memory ring with cp.async.bulk copies
// of up to 32 KB (cut at row ends) issued by one thread, so a whole share of up to ~190 KB is in
// flight at once; 16 consumer warps fold the landed chunks.  Same keys, tickets and workspace.
constexpr int kRingWarps = 16;
constexpr int kRingThreads = (kRingWarps + 1) * 32;
constexpr int kRingConsumers = kRingWarps * 32;
constexpr int kRingChunk = 32768;
constexpr int kRingStages = 6;
constexpr int kRingBytes = kRingStages * kRingChunk;
constexpr int kRingChunkUnits = kRingChunk / 16;

template <typename T>
__global__ void __launch_bounds__(kRingThreads, 1) greedy_ring_kernel(const GreedyArgs A) {
  pdl_launch_dependents();  // a realignment launched after this may start its launch now
  extern __shared__ __align__(128) char ring[];
  __shared__ unsigned long long s_key[kMaxSegs];
  __shared__ unsigned char s_last[kMaxSegs];
  __shared__ __align__(8) uint64_t full[kRingStages], empty[kRingStages];
  __shared__ int s_fail;

  constexpr int VN = Vec<T>::N;
  const int c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int RU = A.RU;
  const long long u0 = A.split.start(c), u1 = A.split.start(c + 1);
  const long long g0 = A.split.div(u0, RU), g1 = A.split.div(u1 - 1, RU);  // rows touched
  const int nseg = static_cast<int>(g1 - g0 + 1);
  if (nseg > kMaxSegs) {  // excluded by the launch geometry
    if (tid == 0) set_status(A.status, SPECDEC_ERR_UNSUPPORTED);
    return;
  }
  // The producer warp sets up the ring's barriers and goes straight on to its copies; the
  // consumers clear the row keys and wait (named barrier 1) until the barriers exist.
  if (warp == kRingWarps) {
    if (lane == 0) {
      s_fail = 0;
      for (int k = 0; k < kRingStages; ++k) {
        mbar_init(&full[k], 1);
        mbar_init(&empty[k], kRingWarps);
      }
      fence_mbar_init();
    }
    __syncwarp();
    named_bar_arrive(1, kRingThreads);
  } else {
    for (int s = tid; s < nseg; s += kRingConsumers) s_key[s] = 0ull;
    named_bar_sync(1, kRingThreads);
  }
  const char* base = static_cast<const char*>(A.logits);  // unit u at base + 16 u
  // Segment k: units [lo, hi) of row g0 + k.
  auto seg_lo = [&](int k) { return static_cast<int>(max(u0, (g0 + k) * RU) - (g0 + k) * RU); };
  auto seg_hi = [&](int k) { return static_cast<int>(min(u1, (g0 + k + 1) * RU) - (g0 + k) * RU); };

  if (warp == kRingWarps) {
    if (lane == 0) {  // producer: every segment's chunks, in order, through the ring
      int n = 0;
      bool ok = true;
      for (int k = 0; k < nseg && ok; ++k) {
        const int lo = seg_lo(k), hi = seg_hi(k);
        const char* src = base + ((g0 + k) * RU + lo) * 16;
        for (int off = 0; off < hi - lo; off += kRingChunkUnits, ++n) {
          const int st = n % kRingStages, r = n / kRingStages;
          if (r > 0 && !mbar_wait_sleep(&empty[st], static_cast<uint32_t>((r - 1) & 1), kSleepTries,
                                        kSleepNs)) {
            ok = false;
            break;
          }
          const uint32_t bytes = static_cast<uint32_t>(min(kRingChunkUnits, hi - lo - off)) * 16u;
          mbar_arrive_expect_tx(&full[st], bytes);
          bulk_g2s(ring + st * kRingChunk, src + static_cast<long long>(off) * 16, bytes, &full[st]);
        }
      }
      if (!ok) s_fail = 1;
      for (int m = max(0, n - kRingStages); m < n; ++m)  // no copy outlives the kernel
        (void)mbar_wait_sleep(&full[m % kRingStages], static_cast<uint32_t>((m / kRingStages) & 1),
                              kSleepTries, kSleepNs);
    }
  } else {
    int n = 0;
    bool ok = true;
    for (int k = 0; k < nseg && ok; ++k) {
      const int lo = seg_lo(k), hi = seg_hi(k);
      float bv = 0.f;
      int bi = -1;
      for (int off = 0; off < hi - lo; off += kRingChunkUnits, ++n) {
        const int st = n % kRingStages, r = n / kRingStages;
        const bool got =
            mbar_wait_sleep(&full[st], static_cast<uint32_t>(r & 1), kSleepTries, kSleepNs);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const int cu = min(kRingChunkUnits, hi - lo - off);
        const uint4* v4 = reinterpret_cast<const uint4*>(ring + st * kRingChunk);
        const int e0 = (lo + off) * VN;  // vocabulary index of the chunk's first element
#pragma unroll 4
        for (int v = tid; v < cu; v += kRingConsumers) {
          float x[VN];
          Vec<T>::unpack(v4[v], x);
          take_vector<VN>(x, e0 + v * VN, bv, bi);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      if (bi >= 0) atomicMax(&s_key[k], make_key(bv, bi));
    }
    if (!ok && lane == 0) s_fail = 1;
  }
  __syncthreads();
  if (s_fail && tid == 0) set_status(A.status, SPECDEC_ERR_TIMEOUT);
  merge_and_decide<kRingThreads>(A, s_key, s_last, g0, g1, nseg, s_fail != 0);
}

struct Geometry {
  int G, RU;
  long long units;
};

Geometry geometry(int B, int D, int V, int vn, int sms) {
  Geometry g;
  g.RU = (V + vn - 1) / vn;
  g.units = static_cast<long long>(B) * (D + 1) * g.RU;
  long long G = std::min(2LL * sms, (g.units + kMinUnits - 1) / kMinUnits);
  // A share of at most (kMaxSegs - 2) rows' units touches at most kMaxSegs - 1 rows.
  G = std::max(G, (g.units + static_cast<long long>(kMaxSegs - 2) * g.RU - 1) /
                      (static_cast<long long>(kMaxSegs - 2) * g.RU));
  G = std::max(G, (g.units + kMaxShare - 1) / kMaxShare);
  g.G = static_cast<int>(std::max(1LL, std::min(G, g.units)));
  return g;
}

// The ring kernel's grid: at most one CTA per SM, at least 1024 units (16 KB) per CTA.
Geometry geometry_ring(int B, int D, int V, int vn, int sms) {
  Geometry g;
  g.RU = V / vn;
  g.units = static_cast<long long>(B) * (D + 1) * g.RU;
  long long G = std::min<long long>(sms, (g.units + 1023) / 1024);
  G = std::max(G, (g.units + static_cast<long long>(kMaxSegs - 2) * g.RU - 1) /
                      (static_cast<long long>(kMaxSegs - 2) * g.RU));
  G = std::max(G, (g.units + kMaxShare - 1) / kMaxShare);
  g.G = static_cast<int>(std::max(1LL, std::min(G, g.units)));
  return g;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

size_t workspace_bytes(int B, int D) {
  return round256(static_cast<size_t>(B) * (D + 1) * sizeof(unsigned long long)) +
         round256(static_cast<size_t>(B) * sizeof(unsigned));
}

template <typename T, bool kVec>
int launch(const void* logits, int B, int D, int V, long long row_stride, const int32_t* draft,
           int32_t* accept_len, int32_t* out_token, int32_t* status, void* ws,
           cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  constexpr int VN = kVec ? Vec<T>::N : 1;
  // Rows back to back, whole 16-byte vectors: the bulk-copy ring kernel.
  const bool use_ring = kVec && row_stride == V && V % VN == 0;
  if (use_ring) {
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPECDEC_ERR_CUDA;
    if (!attr_set[dev]) {
      const cudaError_t e = cudaFuncSetAttribute(
          greedy_ring_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
      if (e != cudaSuccess) return map_cuda_error(e);
      attr_set[dev] = true;
    }
  }
  const Geometry g = use_ring ? geometry_ring(B, D, V, VN, sms) : geometry(B, D, V, VN, sms);
  char* p = static_cast<char*>(ws);
  GreedyArgs A;
  A.logits = logits;
  A.B = B;
  A.D = D;
  A.V = V;
  A.RU = g.RU;
  A.RUfull = V / VN;
  A.step_rows = kThreads / g.RU;
  A.step_off = kThreads % g.RU;
  A.row_stride = row_stride;
  A.split = Split{g.units, g.G, g.units * g.G < (1LL << 32) ? 1 : 0};
  A.draft = draft;
  A.accept_len = accept_len;
  A.out_token = out_token;
  A.status = status;
  A.key = reinterpret_cast<unsigned long long*>(p);
  A.ticket = reinterpret_cast<unsigned*>(
      p + round256(static_cast<size_t>(B) * (D + 1) * sizeof(unsigned long long)));
  if (use_ring)
    greedy_ring_kernel<T><<<g.G, kRingThreads, kRingBytes, stream>>>(A);
  else
    greedy_kernel<T, kVec><<<g.G, kThreads, 0, stream>>>(A);
  return map_cuda_error(cudaGetLastError());
}

}  // namespace
}  // namespace specdec

extern "C" size_t specdec_verify_greedy_workspace(int B, int D) {
  if (B < 1 || D < 1 || D > SPECDEC_MAX_DRAFT) return 0;
  return specdec::workspace_bytes(B, D);
}

namespace specdec {
namespace {

// The checks of greedy verification's arguments other than the workspace, in the order both
// entry points apply them: sizes and dtype, then (for B > 0) pointers and alignment.
int check_greedy_args(const void* logits, int dtype, int B, int D, int V, long long row_stride,
                      const int32_t* draft, const int32_t* accept_len, const int32_t* out_token,
                      const int32_t* dev_status) {
  const int es = elem_size(dtype);
  if (es == 0 || B < 0 || D < 1 || V < 1 || row_stride < V) return SPECDEC_ERR_INVALID_ARG;
  if (D > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (!logits || !draft || !accept_len || !out_token || !dev_status) return SPECDEC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % es != 0) return SPECDEC_ERR_INVALID_ARG;
  return SPECDEC_OK;
}

// Scores beyond 2^40 bytes are outside the library's limits.
bool greedy_too_large(int dtype, int B, int D, long long row_stride) {
  return static_cast<long long>(B) * (D + 1) * row_stride * elem_size(dtype) > (1LL << 40);
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_verify_greedy(const void* logits, int dtype, int B, int D, int V,
                                     long long row_stride, const int32_t* draft,
                                     int32_t* accept_len, int32_t* out_token, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_status, void* stream) {
  using namespace specdec;
  const int rc = check_greedy_args(logits, dtype, B, D, V, row_stride, draft, accept_len,
                                   out_token, dev_status);
  if (rc != SPECDEC_OK || B == 0) return rc;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
      workspace_bytes < specdec::workspace_bytes(B, D))
    return SPECDEC_ERR_INVALID_ARG;
  if (greedy_too_large(dtype, B, D, row_stride)) return SPECDEC_ERR_UNSUPPORTED;
  const int es = elem_size(dtype);
  const bool vec = reinterpret_cast<uintptr_t>(logits) % 16 == 0 && (row_stride * es) % 16 == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPECDEC_BF16)
    return vec ? launch<uint16_t, true>(logits, B, D, V, row_stride, draft, accept_len, out_token,
                                        dev_status, workspace, s)
               : launch<uint16_t, false>(logits, B, D, V, row_stride, draft, accept_len, out_token,
                                         dev_status, workspace, s);
  return vec ? launch<float, true>(logits, B, D, V, row_stride, draft, accept_len, out_token,
                                   dev_status, workspace, s)
             : launch<float, false>(logits, B, D, V, row_stride, draft, accept_len, out_token,
                                    dev_status, workspace, s);
}

// ------------------------------------------------------------------ variant without a workspace
// The same launch on a static per-device scratch array instead of a caller workspace.  Static
// device memory is zero when the module loads, and every greedy call leaves its workspace zero.
namespace specdec {
namespace {

constexpr int kMaxDevices = 64;
static __device__ __align__(256) unsigned char g_greedy_scratch[SPECDEC_GREEDY_SCRATCH_BYTES];
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];  // the array's address on each device, looked up once

int greedy_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return map_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return SPECDEC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_greedy_scratch);  // with device `dev` current
    if (e != cudaSuccess) return map_cuda_error(e);
    if (p == nullptr) return SPECDEC_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SPECDEC_OK;
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_verify_greedy_noalloc(const void* logits, int dtype, int B, int D, int V,
                                             long long row_stride, const int32_t* draft,
                                             int32_t* accept_len, int32_t* out_token,
                                             int32_t* dev_status, void* stream) {
  // The workspace entry point's own checks first (same codes for the same mistakes), then the
  // limit of the static scratch.
  const int rc0 = specdec::check_greedy_args(logits, dtype, B, D, V, row_stride, draft,
                                             accept_len, out_token, dev_status);
  if (rc0 != SPECDEC_OK || B == 0) return rc0;
  if (specdec::greedy_too_large(dtype, B, D, row_stride) ||
      specdec::workspace_bytes(B, D) > SPECDEC_GREEDY_SCRATCH_BYTES)
    return SPECDEC_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int rc = specdec::greedy_scratch(&scratch);
  if (rc != SPECDEC_OK) return rc;
  return specdec_verify_greedy(logits, dtype, B, D, V, row_stride, draft, accept_len, out_token,
                               scratch, SPECDEC_GREEDY_SCRATCH_BYTES, dev_status, stream);
}
