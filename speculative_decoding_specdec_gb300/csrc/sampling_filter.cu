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
// GB300 mapping.  One CTA per row at a time (a grid of up to two CTAs per SM walks the rows).  The
// bound is found by radix selection over the order-preserving key of the score's own bits (16 for
// bf16, 32 for fp32), 8 bits per level, highest first: a 256-bin histogram in shared memory per
// level (counts for top-k, masses for top-p), one warp picks the bin where the running total from
// the top reaches the target, and the next level looks only inside it.  Ties on the final key are
// resolved by index with a block scan.  Masses are 2^(x*c2 - o) (c2 = log2(e)/T, o the row's
// integer offset) in 64-bit fixed point, so every sum is an exact integer sum and the result does
// not depend on the order of the atomics.  The row is read once from HBM; the later passes hit L2.
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
  static constexpr int K = 16;
  __device__ static uint32_t raw(const uint16_t* p) { return *p; }
  __device__ static float value(uint32_t raw) { return __uint_as_float(raw << 16); }
};
template <> struct Bits<float> {
  static constexpr int K = 32;
  __device__ static uint32_t raw(const float* p) { return __float_as_uint(*p); }
  __device__ static float value(uint32_t raw) { return __uint_as_float(raw); }
};

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

struct Shared {
  uint32_t cnt[256];
  unsigned long long mass[256];
  uint32_t wcnt[kFThreads / 32];
  unsigned long long wmass[kFThreads / 32];
  uint32_t r_u[4];
  unsigned long long r_m[2];
};

// Block-wide max of one value per thread.
__device__ uint32_t block_max(uint32_t v, Shared& s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) s.wcnt[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t x = lane < kFThreads / 32 ? s.wcnt[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) s.r_u[0] = x;
  }
  __syncthreads();
  const uint32_t r = s.r_u[0];
  __syncthreads();
  return r;
}

// Warp 0 picks, from the 256 bins of this level (bin 255 first), the bin where the running total
// from the top first reaches `target` (1 <= target <= total); writes the bin and the total of the
// bins above it.  `use_mass` selects the mass histogram, else the counts.
__device__ void pick_bin(Shared& s, bool use_mass, unsigned long long target) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  unsigned long long v[8], tot = 0;  // lane l holds bins 255-8l .. 248-8l, top first
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int b = 255 - 8 * lane - i;
    v[i] = use_mass ? s.mass[b] : s.cnt[b];
    tot += v[i];
  }
  unsigned long long incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned long long above = incl - tot;  // bins of the lanes before this one
  const bool here = above < target && target <= incl;
  const unsigned mine = __ballot_sync(0xffffffffu, here);
  const int owner = mine ? __ffs(static_cast<int>(mine)) - 1 : 31;
  if (lane == owner) {
    unsigned long long run = above;
    int bin = 255 - 8 * lane - 7;
    for (int i = 0; i < 8; ++i) {
      if (run + v[i] >= target || i == 7) {
        bin = 255 - 8 * lane - i;
        break;
      }
      run += v[i];
    }
    s.r_u[1] = static_cast<uint32_t>(bin);
    s.r_m[0] = run;  // total of the bins above the chosen one
  }
}

template <typename T>
__global__ void __launch_bounds__(kFThreads) filter_kernel(const FilterArgs A) {
  __shared__ Shared s;
  constexpr int KB = Bits<T>::K, LV = KB / 8;
  const int tid = threadIdx.x;
  const int Q = 2 * A.D + 1, V = A.V;
  const long long rows = static_cast<long long>(A.B) * Q;
  const bool use_k = A.top_k >= 1 && A.top_k < V;
  const bool use_p = A.top_p < 1.f;

  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int b = static_cast<int>(row / Q), q = static_cast<int>(row % Q);
    const T* x = q <= A.D ? static_cast<const T*>(A.tl) + (static_cast<long long>(b) * (A.D + 1) + q) * A.rs
                          : static_cast<const T*>(A.dl) + (static_cast<long long>(b) * A.D + (q - A.D - 1)) * A.rs;
    uint2 bound = make_uint2(0u, static_cast<uint32_t>(INT_MAX));  // keep all
    if (!use_k && !use_p) {
      if (tid == 0) A.bounds[row] = bound;
      continue;
    }
    // Highest score: the offset of the masses; a NaN or +inf row keeps everything (verification
    // reports such rows as invalid).
    uint32_t km = 0;
    for (int i = tid; i < V; i += kFThreads) km = max(km, nkey<T>(Bits<T>::raw(x + i)));
    km = block_max(km, s);
    const float vmax = Bits<T>::value(nraw<T>(km));
    const bool finite_max = vmax == vmax && vmax != INFINITY && vmax != -INFINITY;
    const float o = finite_max ? ceilf(vmax * A.c2) : 0.f;
    auto weight = [&](uint32_t raw) -> unsigned long long {
      const float w = ex2(fmaf(Bits<T>::value(raw), A.c2, -o));
      return __float2ull_rz(w * kFixedScale);
    };

    // Top-k: the k-th token of the order, by counts.  K-set = key > kkey or (== kkey and v <= kidx).
    uint32_t kkey = 0;
    int kidx = INT_MAX;
    auto in_k = [&](uint32_t key, int v) { return key > kkey || (key == kkey && v <= kidx); };
    // Radix selection over the keys of the tokens that pass `pred`, by counts (mass = false) or
    // masses; returns the final key and, through `rest`, the target left for its ties.
    auto select = [&](bool mass, unsigned long long target, auto pred, unsigned long long& rest) {
      uint32_t pre = 0;
      for (int L = LV - 1; L >= 0; --L) {
        for (int i = tid; i < 256; i += kFThreads) {
          s.cnt[i] = 0u;
          s.mass[i] = 0ull;
        }
        __syncthreads();
        const int sh = 8 * L;
        for (int i = tid; i < V; i += kFThreads) {
          const uint32_t raw = Bits<T>::raw(x + i);
          const uint32_t key = nkey<T>(raw);
          if ((L == LV - 1 || (key >> (sh + 8)) == pre) && pred(key, i)) {
            const int bin = (key >> sh) & 255;
            if (mass) atomicAdd(&s.mass[bin], weight(raw));
            else atomicAdd(&s.cnt[bin], 1u);
          }
        }
        __syncthreads();
        pick_bin(s, mass, target);
        __syncthreads();
        pre = (pre << 8) | s.r_u[1];
        target -= s.r_m[0];
        __syncthreads();
      }
      rest = target;
      return pre;
    };
    // The need-th (1-based) token in index order among those with key == tkey passing `pred`.
    auto nth_index = [&](uint32_t tkey, unsigned long long need, auto pred) {
      const int chunk = (V + kFThreads - 1) / kFThreads;
      const int c0 = min(V, tid * chunk), c1 = min(V, c0 + chunk);
      uint32_t c = 0;
      for (int i = c0; i < c1; ++i) {
        const uint32_t key = nkey<T>(Bits<T>::raw(x + i));
        if (key == tkey && pred(key, i)) ++c;
      }
      const int lane = tid & 31, warp = tid >> 5;
      uint32_t incl = c;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o2);
        if (lane >= o2) incl += t;
      }
      if (lane == 31) s.wcnt[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        const uint32_t wv = lane < kFThreads / 32 ? s.wcnt[lane] : 0u;
        uint32_t xx = wv;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const uint32_t t = __shfl_up_sync(0xffffffffu, xx, o2);
          if (lane >= o2) xx += t;
        }
        if (lane < kFThreads / 32) s.wcnt[lane] = xx - wv;
      }
      __syncthreads();
      const unsigned long long before = (incl - c) + s.wcnt[warp];
      if (before < need && need <= before + c) {
        unsigned long long run = before;
        for (int i = c0; i < c1; ++i) {
          const uint32_t key = nkey<T>(Bits<T>::raw(x + i));
          if (key == tkey && pred(key, i) && ++run == need) {
            s.r_u[2] = static_cast<uint32_t>(i);
            break;
          }
        }
      }
      __syncthreads();
      const int idx = static_cast<int>(s.r_u[2]);
      __syncthreads();
      return idx;
    };
    auto all = [](uint32_t, int) { return true; };

    if (!finite_max) {
      if (tid == 0) A.bounds[row] = bound;
      continue;
    }
    if (use_k) {
      unsigned long long rest = 0;
      const uint32_t key = select(false, static_cast<unsigned long long>(A.top_k), all, rest);
      kidx = nth_index(key, rest, all);
      kkey = key;
    }
    uint32_t fkey = kkey;
    int fidx = kidx;
    if (use_p) {
      // Mass of the top-k set (or of the row), then the token where the mass before it stops
      // being below top_p of that total.
      unsigned long long mk = 0;
      for (int i = tid; i < V; i += kFThreads) {
        const uint32_t raw = Bits<T>::raw(x + i);
        if (in_k(nkey<T>(raw), i)) mk += weight(raw);
      }
      const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) mk += __shfl_xor_sync(0xffffffffu, mk, o2);
      if (lane == 0) s.wmass[warp] = mk;
      __syncthreads();
      if (tid == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < kFThreads / 32; ++w) t += s.wmass[w];
        // Keep a token iff (mass before it) < top_p * total, i.e. (mass before) < ceil(...).
        const double tau = static_cast<double>(A.top_p) * static_cast<double>(t);
        unsigned long long target = static_cast<unsigned long long>(ceil(tau));
        if (target == 0) target = 1;
        s.r_m[1] = target;
      }
      __syncthreads();
      const unsigned long long target = s.r_m[1];
      __syncthreads();
      unsigned long long rest = 0;
      const uint32_t key = select(true, target, in_k, rest);
      // Inside the final key every kept token weighs the same w: the m-th one (index order) is
      // the last kept, m = ceil(rest / w).
      const unsigned long long w = weight(nraw<T>(key));
      const unsigned long long m = w > 0 ? (rest + w - 1) / w : 1;
      fidx = nth_index(key, m < 1 ? 1 : m, in_k);
      fkey = key;
    }
    bound = make_uint2(score_key(Bits<T>::value(nraw<T>(fkey))), static_cast<uint32_t>(fidx));
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
  const int grid = static_cast<int>(std::min<long long>(rows, 2LL * sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SPECDEC_BF16)
    filter_kernel<uint16_t><<<grid, kFThreads, 0, s>>>(A);
  else
    filter_kernel<float><<<grid, kFThreads, 0, s>>>(A);
  return map_cuda_error(cudaGetLastError());
}
