// Top-k / top-p keep bounds of every score row (the sampling settings of sampled verification).
//
// "Inference Engineering: Part 5/8: When Speculative Decoding Backfires": sampling "can choose
// among several likely tokens using settings such as temperature and top-p" (section "Draft
// Possible Tokens, Then Verify Them Together"), and both models must use the same sampling
// settings ("Exactness Means Different Things For Greedy And Sampled Output").
//
// Reading.  A row's tokens are ordered by score, highest first, ties by lower token index.  Top-k
// (1 <= k < V) keeps the first k; top-p (0 < top_p < 1) then keeps, in the same order, every token
// whose preceding probability mass within the kept set is below top_p.  The kept set is always a
// prefix of that order, so it is described by its last token: a bound (key, index) such that a
// token with score x at index v is kept iff key(x) > bound.key, or key(x) == bound.key and
// v <= bound.index, where key is the order-preserving 32-bit code of the score.
//
// GB300 mapping.  One CTA of 512 threads per row at a time (one CTA per SM walks the rows).
//
// bf16 rows: a bf16 score has only 65536 possible values, so one read of the row from HBM builds
// a count per value in shared memory (16-bit counters, two to a 32-bit word, 128 KB; shared
// atomics without return).  The highest score, the top-k cut (counts from the top) and the top-p
// cut (count x per-value weight, from the top) then come from block scans over that histogram,
// and one more pass (from L2) finds the index of the last kept token among the tokens of the cut
// value; that pass is skipped when the cut keeps every token of its value (the bound's index is
// then INT_MAX).  The key code of two bf16 scores is computed in one 32-bit word, and the tie
// search counts equal keys two per word.  If the counts do not add up to V (a counter passed
// 65535: more than 65535 equal scores) the row takes the radix path instead.
//
// fp32 rows: radix selection over the order-preserving key of the score (11 + 11 + 10 bits),
// highest level first: a shared-memory histogram per level (2048 bins at the first level, since
// score keys crowd into few exponent values and narrower histograms serialise their atomics),
// counts for top-k and masses for top-p; one warp picks the bin where the running total from the
// top reaches the target, and the next level looks only inside it.  Ties on the final key are
// resolved by index from per-step match counts.
//
// Masses are 2^(x*c2 - o) (c2 = log2(e)/T, o the row's integer offset) in 2^44 fixed point, so
// every sum is an exact integer sum and no result depends on the order of the atomics.
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kFThreads = 512;
constexpr float kFixedScale = 17592186044416.f;  // 2^44: masses in (0, 1] as integers

// 2^x by the PTX instruction ex2.approx.ftz.f32.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving code of a float score (-0 counted as +0).
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = (f == 0.f) ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <typename T> struct Bits;
template <> struct Bits<uint16_t> {  // bf16
  static constexpr int K = 16, VN = 8;
  __device__ static uint32_t raw(const uint16_t* p) { return *p; }
  __device__ static float value(uint32_t raw) { return __uint_as_float(raw << 16); }
  __device__ static uint32_t lane(const uint4& v, int i) {  // element i of a 16-byte vector
    const uint32_t w = (&v.x)[i >> 1];
    return (i & 1) ? (w >> 16) : (w & 0xffffu);
  }
};
template <> struct Bits<float> {
  static constexpr int K = 32, VN = 4;
  __device__ static uint32_t raw(const float* p) { return __float_as_uint(*p); }
  __device__ static float value(uint32_t raw) { return __uint_as_float(raw); }
  __device__ static uint32_t lane(const uint4& v, int i) { return (&v.x)[i]; }
};

// Calls fn(i, raw) for every element of a row of V scores, all threads of the CTA together:
// 16-byte vectors, kFly in flight per thread, when the row is 16-byte aligned; then the tail.
template <typename T, int kFly = 4, typename Fn>
__device__ __forceinline__ void visit_row(const T* x, int V, bool vec, Fn fn) {
  constexpr int VN = Bits<T>::VN;
  int done = 0;
  if (vec) {
    const uint4* v4 = reinterpret_cast<const uint4*>(x);
    const int nv = V / VN;
    for (int base = threadIdx.x; base < nv; base += kFly * kFThreads) {
      uint4 r[kFly];
#pragma unroll
      for (int k = 0; k < kFly; ++k)
        if (base + k * kFThreads < nv) r[k] = v4[base + k * kFThreads];
#pragma unroll
      for (int k = 0; k < kFly; ++k) {
        const int u = base + k * kFThreads;
        if (u < nv) {
#pragma unroll
          for (int i = 0; i < VN; ++i) fn(u * VN + i, Bits<T>::lane(r[k], i));
        }
      }
    }
    done = nv * VN;
  }
  for (int i = done + static_cast<int>(threadIdx.x); i < V; i += kFThreads) fn(i, Bits<T>::raw(x + i));
}

// Order-preserving code of the score's own K bits, and its inverse.
template <typename T>
__device__ __forceinline__ uint32_t nkey(uint32_t raw) {
  constexpr uint32_t sign = 1u << (Bits<T>::K - 1);
  constexpr uint32_t mask = Bits<T>::K == 32 ? 0xffffffffu : ((1u << Bits<T>::K) - 1u);
  if (raw == sign) raw = 0;  // -0 as +0
  return (raw & sign) ? (~raw & mask) : (raw | sign);
}
template <typename T>
__device__ __forceinline__ uint32_t nraw(uint32_t key) {
  constexpr uint32_t sign = 1u << (Bits<T>::K - 1);
  constexpr uint32_t mask = Bits<T>::K == 32 ? 0xffffffffu : ((1u << Bits<T>::K) - 1u);
  return (key & sign) ? (key & ~sign) : (~key & mask);
}

// nkey for the two bf16 scores of one 32-bit word at once (element 2i in the low half): a half
// whose magnitude bits are zero (-0 or +0) is first made +0, then a negative half is inverted
// and a positive one gets its top bit set.  (mag + 0x7fff) stays below 2^16 in each half, so no
// carry crosses halves.
__device__ __forceinline__ uint32_t nkey2(uint32_t w) {
  const uint32_t nonzero = ((w & 0x7fff7fffu) + 0x7fff7fffu) & 0x80008000u;
  w &= nonzero | 0x7fff7fffu;
  const uint32_t neg = (w >> 15) & 0x00010001u;
  return w ^ (neg * 0xffffu | 0x80008000u);
}

// How many of the two bf16 halves of w have the key of the pair pattern (pat, m) from
// key_pattern: the halves of (w & m) ^ pat that are zero, counted by their top bit.
__device__ __forceinline__ uint32_t count_key2(uint32_t w, uint32_t pat, uint32_t m) {
  const uint32_t d = (w & m) ^ pat;
  const uint32_t z = ~((((d & 0x7fff7fffu) + 0x7fff7fffu) | d)) & 0x80008000u;
  return static_cast<uint32_t>(__popc(z));
}
// The raw bf16 patterns with 16-bit key `key`, for count_key2: one pattern in both halves, and a
// mask that ignores the sign bit for the key of zero (raw +0 and -0 share it).
__device__ __forceinline__ void key_pattern(uint32_t key, uint32_t& pat, uint32_t& m) {
  const uint32_t raw = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
  m = key == 0x8000u ? 0x7fff7fffu : 0xffffffffu;
  pat = (raw | (raw << 16)) & m;
}

struct FilterArgs {
  const void* tl;
  const void* dl;
  int B, D, V;
  long long rs;
  float c2;
  int top_k;      // 0: off
  float top_p;    // 1: off
  uint2* bounds;  // [B][2D+1]: (key, index)
  int32_t* status;
};

constexpr int kWarpsF = kFThreads / 32;
constexpr int kBins = 2048;  // widest radix level: 11 key bits
constexpr int kParts = 4;    // a mass (<= 2^44) as 11-bit parts, each summed in 32 bits
constexpr int kHistWords = 65536 / 2;  // bf16 value histogram: two 16-bit counters per word

struct Shared {  // dynamic shared memory
  uint32_t cnt[kBins];
  uint32_t part[kParts][kBins];
  uint32_t steps[4096];                         // matches per step of the tie search
  unsigned long long ctot[kFThreads];           // per-thread chunk totals of the bf16 histogram
  uint32_t wcnt[kWarpsF];
  unsigned long long wmass[kWarpsF];
  int ovf;
  uint32_t r_u[4];
  unsigned long long r_m[2];
};

// The bf16 histogram follows Shared in dynamic shared memory, 128-byte aligned (it is cleared
// with 16-byte stores).
constexpr size_t kHistOffset = (sizeof(Shared) + 127) & ~static_cast<size_t>(127);
static_assert(kHistOffset % 16 == 0, "histogram must be 16-byte aligned");

// Block-wide max of one value per thread.
__device__ uint32_t block_max(uint32_t v, Shared& s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) s.wcnt[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t x = lane < kWarpsF ? s.wcnt[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) s.r_u[0] = x;
  }
  __syncthreads();
  const uint32_t r = s.r_u[0];
  __syncthreads();
  return r;
}

// Warp 0 walks `nb` totals in the given direction (from entry nb-1 down, or from 0 up) and finds
// the entry where the running total first reaches `target` (1 <= target <= total); writes the
// entry to r_u[1] and the total before it to r_m[0].  `vals(e)` gives entry e's total.
template <typename Vals>
__device__ void pick(Shared& s, int nb, bool top_down, unsigned long long target, Vals vals) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int per = (nb + 31) / 32;  // entries per lane, lane 0 first in walking order
  auto entry = [&](int k) { return top_down ? nb - 1 - k : k; };
  auto val = [&](int k) -> unsigned long long { return k < nb ? vals(entry(k)) : 0ull; };
  unsigned long long tot = 0;
  for (int k = lane * per; k < (lane + 1) * per; ++k) tot += val(k);
  unsigned long long incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned long long above = incl - tot;
  const unsigned mine = __ballot_sync(0xffffffffu, above < target && target <= incl);
  const int owner = mine ? __ffs(static_cast<int>(mine)) - 1 : 31;
  if (lane == owner) {
    unsigned long long run = above;
    int k = lane * per;
    const int last = max(k, min(nb, (lane + 1) * per) - 1);
    for (; k < last; ++k) {
      const unsigned long long v = val(k);
      if (run + v >= target) break;
      run += v;
    }
    s.r_u[1] = static_cast<uint32_t>(entry(k));
    s.r_m[0] = run;
  }
}

// The need-th (1-based) token in index order among those with key == tkey passing `pred`:
// every warp counts the matches of whole steps of 32*VN consecutive elements (16-byte loads,
// four steps in flight), a prefix over the steps picks one, and warp 0 finds the token in it.
template <typename T, bool kAllKept = false, typename Pred>
__device__ __forceinline__ int nth_index(const T* x, int V, bool vec, Shared& s, uint32_t tkey,
                                         unsigned long long need, Pred pred) {
  constexpr int VN = Bits<T>::VN;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int step = 32 * VN;
  const int nst = (V + step - 1) / step;
  // bf16 with every token eligible: compare the raw halves of each word to the key's pattern
  uint32_t pat = 0, pm = 0;
  if constexpr (kAllKept && Bits<T>::K == 16) key_pattern(tkey, pat, pm);
  // Matches among the lane's VN elements of step st (from its vector when the step is whole and
  // the row aligned, else element by element).
  auto count_lane = [&](int st, const uint4& r) {
    const int e0 = st * step + lane * VN;
    unsigned n = 0;
    if constexpr (kAllKept && Bits<T>::K == 16) {
      if (vec && e0 + VN <= V)
        return count_key2(r.x, pat, pm) + count_key2(r.y, pat, pm) + count_key2(r.z, pat, pm) +
               count_key2(r.w, pat, pm);
    }
    if (vec && e0 + VN <= V) {
#pragma unroll
      for (int i = 0; i < VN; ++i) {
        const uint32_t key = nkey<T>(Bits<T>::lane(r, i));
        n += (key == tkey && pred(key, e0 + i)) ? 1u : 0u;
      }
    } else {
#pragma unroll 1
      for (int i = 0; i < VN; ++i) {
        if (e0 + i >= V) break;
        const uint32_t key = nkey<T>(Bits<T>::raw(x + e0 + i));
        n += (key == tkey && pred(key, e0 + i)) ? 1u : 0u;
      }
    }
    return n;
  };
  auto load_lane = [&](int st) -> uint4 {
    const int e0 = st * step + lane * VN;
    if (vec && e0 + VN <= V) return *reinterpret_cast<const uint4*>(x + e0);
    return make_uint4(0u, 0u, 0u, 0u);
  };
  if (tid == 0) s.r_u[2] = static_cast<uint32_t>(V - 1);  // (never used: need <= matches)
  constexpr int kSteps = kAllKept ? 8 : 4;  // steps in flight per warp
  for (int st0 = warp; st0 < nst; st0 += kSteps * kWarpsF) {
    uint4 r[kSteps];
#pragma unroll
    for (int u = 0; u < kSteps; ++u)
      r[u] = st0 + u * kWarpsF < nst ? load_lane(st0 + u * kWarpsF) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const int st = st0 + u * kWarpsF;
      if (st < nst) {  // warp-uniform
        const unsigned n = __reduce_add_sync(0xffffffffu, count_lane(st, r[u]));
        if (lane == 0) s.steps[st] = n;
      }
    }
  }
  __syncthreads();
  pick(s, nst, false, need, [&](int e) -> unsigned long long { return s.steps[e]; });
  __syncthreads();
  if (warp == 0) {  // the token inside the picked step
    const int st = static_cast<int>(s.r_u[1]);
    const int e0 = st * step + lane * VN;
    const uint4 rv = load_lane(st);
    const unsigned n = count_lane(st, rv);
    unsigned incl = n;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
      const unsigned t = __shfl_up_sync(0xffffffffu, incl, o2);
      if (lane >= o2) incl += t;
    }
    const unsigned long long before = s.r_m[0] + (incl - n);
    if (n > 0 && before < need && need <= before + n) {
      unsigned long long r = before;
      for (int i = 0; i < VN && e0 + i < V; ++i) {
        const uint32_t raw = (vec && e0 + VN <= V) ? Bits<T>::lane(rv, i) : Bits<T>::raw(x + e0 + i);
        const uint32_t key = nkey<T>(raw);
        if (key == tkey && pred(key, e0 + i) && ++r == need) {
          s.r_u[2] = static_cast<uint32_t>(e0 + i);
          break;
        }
      }
    }
  }
  __syncthreads();
  const int idx = static_cast<int>(s.r_u[2]);
  __syncthreads();
  return idx;
}

// Radix selection path (fp32 rows, and bf16 rows whose value histogram would overflow): the
// row's keep bound, returned to every thread.  Kept out of line so that its register pressure
// does not spill into the histogram path.
template <typename T>
__device__ __noinline__ uint2 radix_bound(const T* x, int V, bool vec, Shared& s, float c2,
                                          int top_k, float top_p, bool use_k, bool use_p) {
  constexpr int KB = Bits<T>::K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto all = [](uint32_t, int) { return true; };
  // Highest score: the offset of the masses; a NaN or +inf row keeps everything (verification
  // reports such rows as invalid).
  uint32_t km = 0;
  visit_row(x, V, vec, [&](int, uint32_t raw) { km = max(km, nkey<T>(raw)); });
  km = block_max(km, s);
  const float vmax = Bits<T>::value(nraw<T>(km));
  const bool finite_max = vmax == vmax && vmax != INFINITY && vmax != -INFINITY;
  if (!finite_max) return make_uint2(0u, static_cast<uint32_t>(INT_MAX));  // keep all
  const float o = ceilf(vmax * c2);
  auto weight = [&](uint32_t raw) -> unsigned long long {
    const float w = ex2(fmaf(Bits<T>::value(raw), c2, -o));
    return __float2ull_rz(w * kFixedScale);
  };

  uint32_t kkey = 0;
  int kidx = INT_MAX;
  auto in_k = [&](uint32_t key, int v) { return key > kkey || (key == kkey && v <= kidx); };

  // Radix selection over the keys passing `pred`, by counts or masses, from the top: bf16 keys
  // in levels of 11 and 5 bits, fp32 keys 11 + 11 + 10.  Counts and the four 11-bit parts of
  // the masses go to the shared histogram with 32-bit atomics (integer sums: the result does
  // not depend on their order).  With `p_of_total` the target is that fraction of the first
  // level's total (top-p).  Returns the final key; `rest` receives the target left for the ties
  // on that key.
  auto select = [&](bool mass, unsigned long long target, float p_of_total, auto pred,
                    unsigned long long& rest) {
    uint32_t pre = 0;
    int done = 0;  // key bits fixed so far
    for (int l = 0; l < (KB == 16 ? 2 : 3); ++l) {
      const int bits = KB == 16 ? (l == 0 ? 11 : 5) : (l == 2 ? 10 : 11);
      const int nb = 1 << bits, sh = KB - done - bits;
      for (int i = tid; i < nb; i += kFThreads) {
        s.cnt[i] = 0u;
#pragma unroll
        for (int k = 0; k < kParts; ++k) s.part[k][i] = 0u;
      }
      __syncthreads();
      visit_row(x, V, vec, [&](int i, uint32_t raw) {
        const uint32_t key = nkey<T>(raw);
        if ((done == 0 || (key >> (sh + bits)) == pre) && pred(key, i)) {
          const int bin = static_cast<int>((key >> sh) & static_cast<uint32_t>(nb - 1));
          if (mass) {
            const unsigned long long w = weight(raw);
#pragma unroll
            for (int k = 0; k < kParts; ++k) {
              // the top part also holds bit 44 (a mass of exactly 1): at most 2^11 per token
              const uint32_t pk = static_cast<uint32_t>(k == kParts - 1 ? (w >> (11 * k)) : ((w >> (11 * k)) & 0x7ffull));
              if (pk) atomicAdd(&s.part[k][bin], pk);
            }
          } else {
            atomicAdd(&s.cnt[bin], 1u);
          }
        }
      });
      __syncthreads();
      auto bin_mass = [&](int e) -> unsigned long long {
        unsigned long long m = 0;
#pragma unroll
        for (int k = 0; k < kParts; ++k) m += static_cast<unsigned long long>(s.part[k][e]) << (11 * k);
        return m;
      };
      if (l == 0 && p_of_total < 1.f) {  // top-p: keep while mass before < ceil(p * total)
        unsigned long long t = 0;
        for (int i = tid; i < nb; i += kFThreads) t += bin_mass(i);
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o2);
        if (lane == 0) s.wmass[warp] = t;
        __syncthreads();
        if (tid == 0) {
          unsigned long long tt = 0;
          for (int w = 0; w < kWarpsF; ++w) tt += s.wmass[w];
          const unsigned long long tg =
              static_cast<unsigned long long>(ceil(static_cast<double>(p_of_total) * static_cast<double>(tt)));
          s.r_m[1] = tg == 0 ? 1 : tg;
        }
        __syncthreads();
        target = s.r_m[1];
      }
      pick(s, nb, true, target, [&](int e) -> unsigned long long {
        return mass ? bin_mass(e) : static_cast<unsigned long long>(s.cnt[e]);
      });
      __syncthreads();
      pre = (pre << bits) | s.r_u[1];
      target -= s.r_m[0];
      done += bits;
      __syncthreads();
    }
    rest = target;
    return pre;
  };

  if (use_k) {
    unsigned long long rest = 0;
    const uint32_t key = select(false, static_cast<unsigned long long>(top_k), 1.f, all, rest);
    kidx = nth_index<T>(x, V, vec, s, key, rest, all);
    kkey = key;
  }
  uint32_t fkey = kkey;
  int fidx = kidx;
  if (use_p) {
    // The token where the mass before it (within the top-k set, or the row) stops being below
    // top_p of that set's total.
    unsigned long long rest = 0;
    const uint32_t key = select(true, 1ull, top_p, in_k, rest);
    // Inside the final key every kept token weighs the same w: the m-th one (index order) is
    // the last kept, m = ceil(rest / w).
    const unsigned long long w = weight(nraw<T>(key));
    const unsigned long long m = w > 0 ? (rest + w - 1) / w : 1;
    fidx = nth_index<T>(x, V, vec, s, key, m < 1 ? 1 : m, in_k);
    fkey = key;
  }
  return make_uint2(score_key(Bits<T>::value(nraw<T>(fkey))), static_cast<uint32_t>(fidx));
}

template <typename T>
__global__ void __launch_bounds__(kFThreads, 1) filter_kernel(const FilterArgs A) {
  extern __shared__ __align__(128) char smem_raw[];
  Shared& s = *reinterpret_cast<Shared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Q = 2 * A.D + 1, V = A.V;
  const long long rows = static_cast<long long>(A.B) * Q;
  const bool use_k = A.top_k >= 1 && A.top_k < V;
  const bool use_p = A.top_p < 1.f;

  auto row_ptr = [&](long long row) -> const T* {
    const int b = static_cast<int>(row / Q), q = static_cast<int>(row % Q);
    return q <= A.D ? static_cast<const T*>(A.tl) + (static_cast<long long>(b) * (A.D + 1) + q) * A.rs
                    : static_cast<const T*>(A.dl) + (static_cast<long long>(b) * A.D + (q - A.D - 1)) * A.rs;
  };
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const T* x = row_ptr(row);
    uint2 bound = make_uint2(0u, static_cast<uint32_t>(INT_MAX));  // keep all
    if (!use_k && !use_p) {
      if (tid == 0) A.bounds[row] = bound;
      continue;
    }
    const bool vec = (reinterpret_cast<uintptr_t>(x) % 16) == 0;
    auto all = [](uint32_t, int) { return true; };

    if constexpr (Bits<T>::K == 16) {
      // bf16: a count per score value (65536 of them, 16-bit counters two to a word) from one
      // read of the row; the highest score, the top-k cut and the top-p cut follow from the
      // counts and the per-value weights, exactly as from the tokens themselves.  A counter that
      // would pass 65535 sends the row to the radix selection below.
      uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw + kHistOffset);
      uint4* h4 = reinterpret_cast<uint4*>(hist);
      for (int i = tid; i < kHistWords / 4; i += kFThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      auto count_key = [&](uint32_t key) { atomicAdd(&hist[key >> 1], 1u << ((key & 1u) << 4)); };
      int done_v = 0;
      if (vec) {  // two keys per 32-bit word; five 16-byte vectors per batch per thread, the next
                  // batch's loads issued before this batch is counted
        constexpr int kFlyH = 5;
        const uint4* v4 = reinterpret_cast<const uint4*>(x);
        const int nv = V / 8;
        uint4 nx[kFlyH];
#pragma unroll
        for (int k = 0; k < kFlyH; ++k)
          if (tid + k * kFThreads < nv) nx[k] = v4[tid + k * kFThreads];
        for (int base = tid; base < nv; base += kFlyH * kFThreads) {
          uint4 r[kFlyH];
#pragma unroll
          for (int k = 0; k < kFlyH; ++k) r[k] = nx[k];
          const int nb = base + kFlyH * kFThreads;
#pragma unroll
          for (int k = 0; k < kFlyH; ++k)
            if (nb + k * kFThreads < nv) nx[k] = v4[nb + k * kFThreads];
#pragma unroll
          for (int k = 0; k < kFlyH; ++k) {
            if (base + k * kFThreads < nv) {
              const uint32_t w4[4] = {r[k].x, r[k].y, r[k].z, r[k].w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t k2 = nkey2(w4[j]);
                count_key(k2 & 0xffffu);
                count_key(k2 >> 16);
              }
            }
          }
        }
        done_v = nv * 8;
      }
      for (int i = done_v + tid; i < V; i += kFThreads) count_key(nkey<T>(Bits<T>::raw(x + i)));
      __syncthreads();
      auto cnt = [&](uint32_t key) -> uint32_t {
        return (hist[key >> 1] >> ((key & 1u) << 4)) & 0xffffu;
      };
      // The 65536 keys in kFThreads chunks of kChunk, totals in s.ctot (key order).  For masses
      // (an exp2 per populated key) chunk c is summed by warp c mod kWarpsF, its lanes on
      // consecutive words, so the few chunks that hold the row's values are spread over all warps;
      // chunks whose count is zero are skipped.
      constexpr int kChunk = 65536 / kFThreads;
      auto chunk_totals = [&](auto val_pair) {
        for (int c = warp; c < kFThreads; c += kWarpsF) {
          // s.ctot still holds the chunk's count here: a chunk no token falls in has total 0
          if (s.ctot[c] == 0ull) continue;
          unsigned long long t = 0;
#pragma unroll
          for (int h = 0; h < kChunk / 64; ++h) {
            const uint32_t w = static_cast<uint32_t>(c * (kChunk / 2) + h * 32 + lane);
            t += val_pair(w);
          }
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o2);
          if (lane == 0) s.ctot[c] = t;
        }
      };
      // Counts (cheap) per thread over its own chunk, 16 bytes at a time from vector
      // (lane + i) mod 16, so that each quarter of a warp reads 32 different banks; the highest
      // populated key comes from the highest nonzero word.
      uint32_t km = 0;
      unsigned long long tc = 0;
      {
        const uint32_t k0 = static_cast<uint32_t>(tid) * kChunk;
        const uint32_t* hw = hist + (k0 >> 1);
        const uint4* hw4 = reinterpret_cast<const uint4*>(hw);
        uint32_t lo = 0, hi = 0;
        int wm = -1;  // highest nonzero word of the chunk
#pragma unroll 4
        for (int i = 0; i < kChunk / 8; ++i) {
          const int qv = (i + lane) & (kChunk / 8 - 1);
          const uint4 v = hw4[qv];
          lo += (v.x & 0xffffu) + (v.y & 0xffffu) + (v.z & 0xffffu) + (v.w & 0xffffu);
          hi += (v.x >> 16) + (v.y >> 16) + (v.z >> 16) + (v.w >> 16);
          const int top = v.w ? 3 : v.z ? 2 : v.y ? 1 : v.x ? 0 : -1;
          if (top >= 0) wm = max(wm, 4 * qv + top);
        }
        tc = static_cast<unsigned long long>(lo) + hi;
        if (wm >= 0) km = k0 + 2u * static_cast<uint32_t>(wm) + ((hw[wm] >> 16) ? 1u : 0u);
        s.ctot[tid] = tc;
      }
      // A counter that passed 65535 lost 65535 (or, carried out of its word, 65536) counts, so
      // the counts add up to V exactly when none overflowed.
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) tc += __shfl_xor_sync(0xffffffffu, tc, o2);
      if (lane == 0) s.wmass[warp] = tc;
      __syncthreads();
      if (tid == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < kWarpsF; ++w) t += s.wmass[w];
        s.ovf = t != static_cast<unsigned long long>(V);
      }
      km = block_max(km, s);  // (its barriers also publish s.ovf)
      if (!s.ovf) {
        const float vmax = Bits<T>::value(nraw<T>(km));
        if (!(vmax == vmax && vmax != INFINITY && vmax != -INFINITY)) {
          if (tid == 0) A.bounds[row] = bound;  // keep all (verification reports the row)
          __syncthreads();
          continue;
        }
        const float o = ceilf(vmax * A.c2);
        auto wgt = [&](uint32_t key) -> unsigned long long {
          const float w = ex2(fmaf(Bits<T>::value(nraw<T>(key)), A.c2, -o));
          return __float2ull_rz(w * kFixedScale);
        };
        // Warp 0 walks chunk e from its highest key down, starting with `run` above it, to the
        // key where the running total reaches `target`; r_u[2] = that key, r_m[1] = the target
        // left for it.
        auto walk = [&](int e, unsigned long long run, unsigned long long target, auto val) {
          if (warp == 0) {
            unsigned long long v[kChunk / 32], t = 0;
#pragma unroll
            for (int i = 0; i < kChunk / 32; ++i) {
              v[i] = val(static_cast<uint32_t>(e * kChunk + kChunk - 1 - (lane * (kChunk / 32) + i)));
              t += v[i];
            }
            unsigned long long incl = t;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
              const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o2);
              if (lane >= o2) incl += y;
            }
            const unsigned long long before = run + incl - t;
            const unsigned mine = __ballot_sync(0xffffffffu, before < target && target <= run + incl);
            const int owner = mine ? __ffs(static_cast<int>(mine)) - 1 : 31;
            if (lane == owner) {
              unsigned long long r = before;
              int i = 0;
              for (; i < kChunk / 32 - 1; ++i) {
                if (r + v[i] >= target) break;
                r += v[i];
              }
              s.r_u[2] = static_cast<uint32_t>(e * kChunk + kChunk - 1 - (lane * (kChunk / 32) + i));
              s.r_m[1] = target - r;
            }
          }
          __syncthreads();
        };
        uint32_t K = 0, kk = 0;
        unsigned long long need = 1, krest = 0;
        if (use_k) {
          pick(s, kFThreads, true, static_cast<unsigned long long>(A.top_k),
               [&](int e) -> unsigned long long { return s.ctot[e]; });
          __syncthreads();
          walk(static_cast<int>(s.r_u[1]), s.r_m[0], static_cast<unsigned long long>(A.top_k),
               [&](uint32_t key) -> unsigned long long { return cnt(key); });
          kk = s.r_u[2];
          krest = s.r_m[1];
          K = kk;
          need = krest;
          __syncthreads();
        }
        if (use_p) {
          // masses within the top-k set: of the boundary key only its first krest tokens count
          auto mass_of = [&](uint32_t key) -> unsigned long long {
            unsigned long long c = cnt(key);
            if (use_k) {
              if (key < kk) return 0ull;
              if (key == kk) c = krest;
            }
            return c ? c * wgt(key) : 0ull;
          };
          chunk_totals([&](uint32_t w) -> unsigned long long {
            const uint32_t v = hist[w];
            if (v == 0u) return 0ull;  // neither value of the word occurs
            return mass_of(2 * w) + mass_of(2 * w + 1);
          });
          __syncthreads();
          if (warp == 0) {
            unsigned long long t = 0;
            for (int e = lane; e < kFThreads; e += 32) t += s.ctot[e];
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o2);
            if (lane == 0) {
              const unsigned long long tg = static_cast<unsigned long long>(
                  ceil(static_cast<double>(A.top_p) * static_cast<double>(t)));
              s.r_m[1] = tg == 0 ? 1 : tg;
            }
          }
          __syncthreads();
          const unsigned long long target = s.r_m[1];
          __syncthreads();
          pick(s, kFThreads, true, target, [&](int e) -> unsigned long long { return s.ctot[e]; });
          __syncthreads();
          walk(static_cast<int>(s.r_u[1]), s.r_m[0], target, mass_of);
          K = s.r_u[2];
          const unsigned long long rest = s.r_m[1];
          __syncthreads();
          // inside key K every token weighs the same w: the m-th one (index order) is the last
          const unsigned long long w = wgt(K);
          const unsigned long long mm = w > 0 ? (rest + w - 1) / w : 1;
          need = mm < 1 ? 1 : mm;
        }
        // The tie search is needed only where the cut splits the tokens of score K: when every
        // one of them is kept (all of K's tokens within the top-k set, where that applies), the
        // bound's index is INT_MAX.
        const unsigned long long eligible = (use_k && K == kk) ? krest : cnt(K);
        const bool all_of_k = need >= eligible && (!use_k || K != kk || krest == cnt(K));
        const int idx = all_of_k ? INT_MAX : nth_index<T, true>(x, V, vec, s, K, need, all);
        bound = make_uint2(score_key(Bits<T>::value(nraw<T>(K))), static_cast<uint32_t>(idx));
        if (tid == 0) A.bounds[row] = bound;
        __syncthreads();
        continue;
      }
    }
    bound = radix_bound<T>(x, V, vec, s, A.c2, A.top_k, A.top_p, use_k, use_p);
    if (tid == 0) A.bounds[row] = bound;
    __syncthreads();
  }
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_sampling_filter(const void* target_logits, const void* draft_logits,
                                       int dtype, int B, int D, int V, long long row_stride,
                                       float temperature, int top_k, float top_p,
                                       void* keep_bounds, int32_t* dev_status, void* stream) {
  using namespace specdec;
  const int es = elem_size(dtype);
  if (es == 0 || B < 0 || D < 1 || V < 1 || row_stride < V) return SPECDEC_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return SPECDEC_ERR_INVALID_ARG;
  if (!(top_p > 0.f && top_p <= 1.f) || top_k < 0) return SPECDEC_ERR_INVALID_ARG;
  if (D > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0) return SPECDEC_OK;
  if (!target_logits || !draft_logits || !keep_bounds || !dev_status) return SPECDEC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(target_logits) % es ||
      reinterpret_cast<uintptr_t>(draft_logits) % es ||
      reinterpret_cast<uintptr_t>(keep_bounds) % 8)
    return SPECDEC_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * (2 * D + 1) > (1LL << 31)) return SPECDEC_ERR_UNSUPPORTED;
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  FilterArgs A;
  A.tl = target_logits;
  A.dl = draft_logits;
  A.B = B;
  A.D = D;
  A.V = V;
  A.rs = row_stride;
  A.c2 = 1.4426950408889634f / temperature;
  A.top_k = top_k;
  A.top_p = top_p;
  A.bounds = static_cast<uint2*>(keep_bounds);
  A.status = dev_status;
  const long long rows = static_cast<long long>(B) * (2 * D + 1);
  const int grid = static_cast<int>(std::min<long long>(rows, sms));
  const int smem = dtype == SPECDEC_BF16
                       ? static_cast<int>(kHistOffset) + kHistWords * static_cast<int>(sizeof(uint32_t))
                       : static_cast<int>(sizeof(Shared));
  static bool attr_set[2][64] = {{false}};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPECDEC_ERR_CUDA;
  const int which = dtype == SPECDEC_BF16 ? 0 : 1;
  if (!attr_set[which][dev]) {
    const cudaError_t e = which == 0
        ? cudaFuncSetAttribute(filter_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
        : cudaFuncSetAttribute(filter_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return map_cuda_error(e);
    attr_set[which][dev] = true;
  }
  if (V > 4096 * 32 * (16 / es)) return SPECDEC_ERR_UNSUPPORTED;  // steps of the tie search
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (which == 0)
    filter_kernel<uint16_t><<<grid, kFThreads, smem, s>>>(A);
  else
    filter_kernel<float><<<grid, kFThreads, smem, s>>>(A);
  return map_cuda_error(cudaGetLastError());
}
