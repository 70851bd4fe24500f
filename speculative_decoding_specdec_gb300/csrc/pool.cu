// SequencePool lifecycle on the device: the per-round schedule and the admission of prompts.
//
// "Batch Speculative Decoding Done Right", section 2.3: EXSPEC keeps a pool of active sequences
// and groups same-length sequences into batches, which need no realignment; only the
// mixed-length ones are realigned.
//
// Schedule (one CTA, latency-bound: a few KB in and out).  The ACTIVE slots are sorted by the
// unique key (length << 12 | slot) with a bitonic sort in shared memory.  The window rule walks
// the sorted rows: at position i the next bs rows form a batch if they span at most w in length
// (feasible(i)), and the walk jumps to i + bs; otherwise row i is a leftover and the walk moves to
// i + 1.  That walk is a chain through next(i); instead of following it one step at a time, the
// positions it visits are found by pointer doubling (log2 of the pool size rounds of parallel
// composition).  Two block scans then give each windowed batch and each leftover its place.
// Finished slots are listed by a third scan and set FREE.
//
// Admission (two launches on the caller's stream).  A one-CTA launch checks every entry (slot
// free and named once, prompt length, limit and arena range); a second launch copies the prompts
// and writes the slot metadata only if dev_status is still zero.  Splitting the two removes any
// race between a CTA that marks a slot ACTIVE and another that is still checking it is FREE.
#include <algorithm>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kSThreads = 1024;
constexpr int kMaxSlots = 4096;   // slots of one pool (12 bits of the sort key)
constexpr int kLenLimit = 1 << 20;  // lengths below 2^20 (the other 20 bits of the key)

// Exclusive block scan of two counters given as per-thread totals; returns both prefixes and
// writes the block totals to tot[0..1].
__device__ void scan2(int a, int b, int& pa, int& pb, int* tmp, int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, ia, o);
    const int y = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += x; ib += y; }
  }
  if (lane == 31) { tmp[warp] = ia; tmp[32 + warp] = ib; }
  __syncthreads();
  if (warp == 0) {
    const int va = tmp[lane], vb = tmp[32 + lane];  // kSThreads / 32 == 32 warps
    int xa = va, xb = vb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, xa, o);
      const int y = __shfl_up_sync(0xffffffffu, xb, o);
      if (lane >= o) { xa += x; xb += y; }
    }
    tmp[64 + lane] = xa - va;
    tmp[96 + lane] = xb - vb;
    if (lane == 31) { tot[0] = xa; tot[1] = xb; }
  }
  __syncthreads();
  pa = tmp[64 + warp] + ia - a;
  pb = tmp[96 + warp] + ib - b;
  __syncthreads();
}

struct SchedArgs {
  int S, bs, window;
  uint8_t* state;
  const int32_t* len;
  int32_t* perm;
  int32_t* offsets;
  uint8_t* uniform;
  int32_t* finished;
  uint8_t* reason;
  int32_t* counts;
  int32_t* status;
};

__global__ void __launch_bounds__(kSThreads) schedule_kernel(const SchedArgs A) {
  __shared__ uint32_t keys[kMaxSlots];
  __shared__ int16_t jump_a[kMaxSlots + 1], jump_b[kMaxSlots + 1], chain[kMaxSlots + 1];
  __shared__ int tmp[128], tot[2];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  const int S = A.S, bs = A.bs;
  int P = 1;
  while (P < S) P <<= 1;

  // Validate and load: active slots get their key, all others sort to the end.
  if (tid == 0) s_bad = 0;
  __syncthreads();
  int act = 0, fin = 0;
  constexpr int kPer = kMaxSlots / kSThreads;  // slots per thread, contiguous
  for (int k = 0; k < kPer; ++k) {
    const int s = tid * kPer + k;
    if (s >= P) break;
    uint32_t key = 0xffffffffu;
    if (s < S) {
      const int st = A.state[s];
      if (st > SPECDEC_SLOT_FINISHED_LENGTH) s_bad = 1;
      if (st == SPECDEC_SLOT_ACTIVE) {
        const int n = A.len[s];
        if (n < 1 || n >= kLenLimit) s_bad = 1;
        key = (static_cast<uint32_t>(n) << 12) | static_cast<uint32_t>(s);
        ++act;
      } else if (st >= SPECDEC_SLOT_FINISHED_EOS) {
        ++fin;
      }
    }
    keys[s] = key;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) set_status(A.status, SPECDEC_ERR_INPUT_RANGE);
    return;
  }
  int pa, pf;
  scan2(act, fin, pa, pf, tmp, tot);
  const int n = tot[0], nfin = tot[1];

  // Finished slots, in slot order: report and free.
  for (int k = 0; k < kPer; ++k) {
    const int s = tid * kPer + k;
    if (s >= S) break;
    const int st = A.state[s];
    if (st >= SPECDEC_SLOT_FINISHED_EOS) {
      A.finished[pf] = s;
      A.reason[pf] = static_cast<uint8_t>(st);
      A.state[s] = SPECDEC_SLOT_FREE;
      ++pf;
    }
  }

  // Bitonic sort of the P keys (ascending).
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += kSThreads) {
        const int l = i ^ j;
        if (l > i) {
          const uint32_t x = keys[i], y = keys[l];
          if (((i & k) == 0) == (x > y)) { keys[i] = y; keys[l] = x; }
        }
      }
      __syncthreads();
    }
  }

  // The walk: next(i) = i + bs where feasible, else i + 1; position n is its end.
  auto len_at = [&](int i) { return static_cast<int>(keys[i] >> 12); };
  auto feasible = [&](int i) {
    return i + bs <= n && len_at(i + bs - 1) - len_at(i) <= A.window;
  };
  for (int i = tid; i <= n; i += kSThreads)
    jump_a[i] = static_cast<int16_t>(i == n ? n : (feasible(i) ? i + bs : i + 1));
  if (tid == 0) chain[0] = 0;
  __syncthreads();
  int16_t* jf = jump_a;  // next^known
  int16_t* jt = jump_b;
  for (int known = 1; known <= n; known <<= 1) {
    for (int j = known + tid; j < 2 * known && j <= n; j += kSThreads) chain[j] = jf[chain[j - known]];
    for (int i = tid; i <= n; i += kSThreads) jt[i] = jf[jf[i]];
    __syncthreads();
    int16_t* t = jf; jf = jt; jt = t;
  }
  // Visited positions (the chain is increasing and ends at n): reuse jt as flags.
  for (int i = tid; i <= n; i += kSThreads) jt[i] = 0;
  __syncthreads();
  for (int j = tid; j <= n; j += kSThreads)
    if (chain[j] < n) jt[chain[j]] = 1;
  __syncthreads();

  // Windowed batches and leftovers, each in walk order.
  const int per = (n + kSThreads - 1) / kSThreads;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  int cw = 0, cl = 0;
  for (int i = i0; i < i1; ++i)
    if (jt[i]) { if (feasible(i)) ++cw; else ++cl; }
  int pw, pl;
  scan2(cw, cl, pw, pl, tmp, tot);
  const int nw = tot[0], nl = tot[1];
  for (int i = i0; i < i1; ++i) {
    if (!jt[i]) continue;
    if (feasible(i)) {
      for (int t = 0; t < bs; ++t) A.perm[pw * bs + t] = static_cast<int32_t>(keys[i + t] & 0xfffu);
      A.uniform[pw] = len_at(i) == len_at(i + bs - 1) ? 1 : 0;
      ++pw;
    } else {
      A.perm[nw * bs + pl] = static_cast<int32_t>(keys[i] & 0xfffu);
      ++pl;
    }
  }
  const int nm = (nl + bs - 1) / bs;
  for (int k = tid; k <= nw + nm; k += kSThreads) {
    A.offsets[k] = k <= nw ? k * bs : min(n, nw * bs + (k - nw) * bs);
    if (k >= nw && k < nw + nm) A.uniform[k] = 0;
  }
  if (tid == 0) {
    A.counts[0] = nw + nm;
    A.counts[1] = nw;
    A.counts[2] = n;
    A.counts[3] = nfin;
  }
}

// ------------------------------------------------------------------------------ admission

struct AdmitArgs {
  int n, S, D, ids_cap;
  long long arena_cols;
  const int32_t* slots;
  const int32_t* cols;
  const int32_t* caps;
  const int32_t* limits;
  const int32_t* prompt_ids;
  const int32_t* prompt_off;
  uint8_t* state;
  int32_t* slot_col;
  int32_t* slot_cap;
  int32_t* slot_len;
  int32_t* slot_limit;
  int32_t* pool_ids;
  int32_t* status;
};

constexpr int kAdmitThreads = 1024;
constexpr int kMaxAdmit = 1024;

__global__ void __launch_bounds__(kAdmitThreads) admit_check_kernel(const AdmitArgs A) {
  __shared__ uint32_t seen[kMaxSlots / 32];
  __shared__ int s_bad;  // bit 0: range, bit 1: capacity
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  for (int k = tid; k < kMaxSlots / 32; k += kAdmitThreads) seen[k] = 0u;
  __syncthreads();
  int bad = 0;
  for (int i = tid; i < A.n; i += kAdmitThreads) {
    const int s = A.slots[i];
    const int o0 = A.prompt_off[i], o1 = A.prompt_off[i + 1];
    const int len = o1 - o0, lim = A.limits[i], c0 = A.cols[i], cap = A.caps[i];
    if (s < 0 || s >= A.S || o0 < 0 || len < 1 || len >= lim || c0 < 0 || cap < 1 ||
        static_cast<long long>(c0) + cap > A.arena_cols) {
      bad |= 1;
      continue;
    }
    if (A.state[s] != SPECDEC_SLOT_FREE) bad |= 1;
    const uint32_t bit = 1u << (s & 31);
    if (atomicOr(&seen[s >> 5], bit) & bit) bad |= 1;  // named twice
    if (static_cast<long long>(lim) + A.D - 1 > cap || static_cast<long long>(lim) + A.D > A.ids_cap)
      bad |= 2;
  }
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  if (tid == 0 && s_bad)
    set_status(A.status, (s_bad & 1) ? SPECDEC_ERR_INPUT_RANGE : SPECDEC_ERR_CAPACITY);
}

// One CTA per admitted sequence at a time; nothing is written unless dev_status is zero.
__global__ void __launch_bounds__(256) admit_write_kernel(const AdmitArgs A) {
  if (*reinterpret_cast<volatile int32_t*>(A.status) != 0) return;
  for (int i = blockIdx.x; i < A.n; i += gridDim.x) {
    const int s = A.slots[i];
    const int o0 = A.prompt_off[i], len = A.prompt_off[i + 1] - o0;
    int32_t* dst = A.pool_ids + static_cast<long long>(s) * A.ids_cap;
    for (int q = threadIdx.x; q < len; q += blockDim.x) dst[q] = A.prompt_ids[o0 + q];
    if (threadIdx.x == 0) {
      A.slot_col[s] = A.cols[i];
      A.slot_cap[s] = A.caps[i];
      A.slot_len[s] = len;
      A.slot_limit[s] = A.limits[i];
      A.state[s] = SPECDEC_SLOT_ACTIVE;
    }
  }
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_pool_schedule(const specdec_schedule_args* a, void* stream) {
  using namespace specdec;
  if (!a) return SPECDEC_ERR_INVALID_ARG;
  if (a->S < 0 || a->batch_size < 1 || a->window < 0) return SPECDEC_ERR_INVALID_ARG;
  if (a->S > kMaxSlots || a->batch_size > kMaxSlots) return SPECDEC_ERR_UNSUPPORTED;
  if (!a->batch_offsets || !a->counts || !a->dev_status) return SPECDEC_ERR_INVALID_ARG;
  if (a->S > 0 && (!a->slot_state || !a->slot_len || !a->perm || !a->batch_uniform ||
                   !a->finished || !a->finished_reason))
    return SPECDEC_ERR_INVALID_ARG;
  SchedArgs A;
  A.S = a->S;
  A.bs = a->batch_size;
  A.window = a->window;
  A.state = a->slot_state;
  A.len = a->slot_len;
  A.perm = a->perm;
  A.offsets = a->batch_offsets;
  A.uniform = a->batch_uniform;
  A.finished = a->finished;
  A.reason = a->finished_reason;
  A.counts = a->counts;
  A.status = a->dev_status;
  schedule_kernel<<<1, kSThreads, 0, static_cast<cudaStream_t>(stream)>>>(A);
  return map_cuda_error(cudaGetLastError());
}

extern "C" int specdec_pool_admit(const specdec_admit_args* a, void* stream) {
  using namespace specdec;
  if (!a) return SPECDEC_ERR_INVALID_ARG;
  if (a->n < 0 || a->S < 0 || a->D < 1 || a->ids_cap < 1 || a->arena_cols < 0)
    return SPECDEC_ERR_INVALID_ARG;
  if (a->n > kMaxAdmit || a->S > kMaxSlots || a->D > SPECDEC_MAX_DRAFT) return SPECDEC_ERR_UNSUPPORTED;
  if (a->n == 0) return SPECDEC_OK;
  if (!a->slots || !a->cols || !a->caps || !a->limits || !a->prompt_ids || !a->prompt_off ||
      !a->slot_state || !a->slot_col || !a->slot_cap || !a->slot_len || !a->slot_limit ||
      !a->pool_ids || !a->dev_status)
    return SPECDEC_ERR_INVALID_ARG;
  AdmitArgs A;
  A.n = a->n;
  A.S = a->S;
  A.D = a->D;
  A.ids_cap = a->ids_cap;
  A.arena_cols = a->arena_cols;
  A.slots = a->slots;
  A.cols = a->cols;
  A.caps = a->caps;
  A.limits = a->limits;
  A.prompt_ids = a->prompt_ids;
  A.prompt_off = a->prompt_off;
  A.state = a->slot_state;
  A.slot_col = a->slot_col;
  A.slot_cap = a->slot_cap;
  A.slot_len = a->slot_len;
  A.slot_limit = a->slot_limit;
  A.pool_ids = a->pool_ids;
  A.status = a->dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  admit_check_kernel<<<1, kAdmitThreads, 0, s>>>(A);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return map_cuda_error(e);
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  admit_write_kernel<<<std::min(a->n, 2 * sms), 256, 0, s>>>(A);
  return map_cuda_error(cudaGetLastError());
}
