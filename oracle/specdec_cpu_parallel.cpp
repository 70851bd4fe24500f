// Row-parallel CPU baseline of the greedy round: greedy verification and EQSPEC realignment on
// the host cores, one std::thread per core over score rows and K/V runs.
//
// TEST AND BASELINE INFRASTRUCTURE ONLY, like the oracle beside it: bench.py times it as a fair
// multi-core CPU baseline (reported next to the single-threaded oracle, never as a target) and
// tests/ check it against the oracle.  The product path (the CUDA library and its binding) never
// loads it, and it shares no code with that path.
//
// What it computes is the oracle's definition, restated in plain C++ (see specdec_oracle.py for
// the readings of the pages; sources cited by page title and section):
//  * greedy verification [IE5, "One Verification Pass Can Commit Several Tokens" and "Exactness
//    Means Different Things For Greedy And Sampled Output"]: per score row the highest score,
//    lowest token index on ties (a NaN score is an error); a_b = number of leading drafts equal
//    to the target's choice, y_b = the choice at row a_b;
//  * realignment [BSDDR sections 2.1, 2.2]: N'_b = N_b + a_b + 1, W' = max N'_b; the surviving
//    columns [W - N_b, W + a_b) of every (layer, k/v, head) of row b move to [W' - N'_b, W' - 1)
//    of the destination (other columns of the destination are left as they were); ids are the
//    old committed tokens, the accepted drafts and y_b ending at W' - 1, mask 1 on the content,
//    position IDs 0..N'_b - 1 there, 0 and pad_id elsewhere.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

enum { kOk = 0, kErrRange = 1, kErrCapacity = 2, kErrArg = 3 };

float to_float(const void* row, int dtype, long long i) {
  if (dtype == 0) return static_cast<const float*>(row)[i];
  const uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(row)[i]) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);  // a bfloat16 is the high half of the float's bits
  return f;
}

// Run fn(t, lo, hi) over [0, n) split into `threads` contiguous parts, one std::thread each
// (t = the part's index, below the returned part count).
template <class Fn>
int parallel_for(long long n, int threads, Fn fn) {
  if (threads < 1) threads = 1;
  if (n < threads) threads = static_cast<int>(n > 0 ? n : 1);
  std::vector<std::thread> pool;
  pool.reserve(threads);
  for (int t = 0; t < threads; ++t) {
    const long long lo = n * t / threads, hi = n * (t + 1) / threads;
    pool.emplace_back([=] { fn(t, lo, hi); });
  }
  for (auto& th : pool) th.join();
  return threads;
}

}  // namespace

extern "C" {

// logits [B][D+1][V] (dtype 0: float32, 1: bfloat16), draft [B][D] -> accept[B], token[B].
// Returns 0, or 1 for a NaN score or a draft outside [0, V) (outputs then unspecified).
int cpu_verify_greedy(const void* logits, int dtype, int B, int D, int V, const int32_t* draft,
                      int32_t* accept, int32_t* token, int threads) {
  if (B < 0 || D < 1 || V < 1 || (dtype != 0 && dtype != 1)) return kErrArg;
  const long long rows = static_cast<long long>(B) * (D + 1);
  std::vector<int32_t> choice(static_cast<size_t>(rows));
  std::vector<int> bad(threads > 0 ? threads : 1, 0);  // one flag per part
  const size_t esize = dtype == 0 ? 4 : 2;
  parallel_for(rows, threads, [&](int t, long long lo, long long hi) {
    for (long long r = lo; r < hi; ++r) {
      const char* row = static_cast<const char*>(logits) + r * V * static_cast<long long>(esize);
      float best = 0.f;
      int arg = -1;
      for (int v = 0; v < V; ++v) {
        const float x = to_float(row, dtype, v);
        if (std::isnan(x)) {
          bad[static_cast<size_t>(t)] = 1;
          arg = -1;
          break;
        }
        if (arg < 0 || x > best) {  // strict: the lowest index keeps a tie
          best = x;
          arg = v;
        }
      }
      choice[static_cast<size_t>(r)] = arg;
    }
  });
  for (int f : bad)
    if (f) return kErrRange;
  for (int b = 0; b < B; ++b) {
    const int32_t* g = &choice[static_cast<size_t>(b) * (D + 1)];
    int a = D;
    for (int j = 0; j < D; ++j) {
      const int d = draft[static_cast<long long>(b) * D + j];
      if (d < 0 || d >= V) return kErrRange;
      if (g[j] != d) {
        a = j;
        break;
      }
    }
    for (int j = a + 1; j < D; ++j) {  // later drafts are discarded but must still be in range
      const int d = draft[static_cast<long long>(b) * D + j];
      if (d < 0 || d >= V) return kErrRange;
    }
    if (g[a] < 0) return kErrRange;
    accept[b] = a;
    token[b] = g[a];
  }
  return kOk;
}

// Sampled verification (speculative rejection sampling) [IE5, "Exactness Means Different Things
// For Greedy And Sampled Output"]: p = softmax(z / T), q = softmax(w / T) per position, in double;
// d_{j+1} is accepted iff u[b][j] < p_j(d) / q_j(d), left to right; at the first rejection a the
// token is drawn from max(0, p_a - q_a) (from p_a if that is all zero), after D acceptances from
// p_D, by inverse CDF with u[b][D] over ascending token ids (the first k whose running sum exceeds
// u * total; if rounding leaves none, the last k with nonzero weight).  target [B][D+1][V], drafts'
// scores [B][D][V] (dtype 0: float32, 1: bfloat16), draft [B][D], uniforms [B][D+1].  Batch rows
// are split over the threads.  Returns 0, 1 (a draft outside [0, V)) or 3 (bad arguments).
int cpu_verify_sample(const void* target, const void* draft_scores, int dtype, int B, int D,
                      int V, const int32_t* draft, const float* uniforms, double temperature,
                      int32_t* accept, int32_t* token, int threads) {
  if (B < 0 || D < 1 || V < 1 || (dtype != 0 && dtype != 1) || !(temperature > 0.0))
    return kErrArg;
  for (long long i = 0; i < static_cast<long long>(B) * D; ++i)
    if (draft[i] < 0 || draft[i] >= V) return kErrRange;
  const size_t esize = dtype == 0 ? 4 : 2;
  const double T = temperature;
  parallel_for(B, threads, [&](int, long long lo, long long hi) {
    std::vector<double> p(static_cast<size_t>(V)), q(static_cast<size_t>(V));
    // softmax of one score row at T, into out (normalised)
    auto softmax = [&](const void* rows, long long row, std::vector<double>& out) {
      const char* base = static_cast<const char*>(rows) + row * V * static_cast<long long>(esize);
      double m = -INFINITY;
      for (int v = 0; v < V; ++v) {
        out[v] = static_cast<double>(to_float(base, dtype, v)) / T;
        if (out[v] > m) m = out[v];
      }
      double sum = 0.0;
      for (int v = 0; v < V; ++v) {
        out[v] = std::exp(out[v] - m);
        sum += out[v];
      }
      for (int v = 0; v < V; ++v) out[v] /= sum;
    };
    for (long long b = lo; b < hi; ++b) {
      const float* u = uniforms + b * (D + 1);
      int a = D;
      for (int j = 0; j < D; ++j) {
        softmax(target, b * (D + 1) + j, p);
        softmax(draft_scores, b * D + j, q);
        const int x = draft[b * D + j];
        // q(x) = 0 < p(x) accepts; p(x) = 0 rejects whatever q(x) is
        const double r = q[x] > 0.0 ? p[x] / q[x] : (p[x] > 0.0 ? INFINITY : 0.0);
        if (!(static_cast<double>(u[j]) < r)) {
          a = j;
          break;
        }
      }
      // weights of the draw, in p
      if (a < D) {  // p and q still hold row a
        bool any = false;
        for (int v = 0; v < V; ++v) {
          const double w = p[v] - q[v];
          q[v] = w > 0.0 ? w : 0.0;
          any = any || q[v] > 0.0;
        }
        if (any) p.swap(q);
      } else {
        softmax(target, b * (D + 1) + D, p);
      }
      double total = 0.0;
      for (int v = 0; v < V; ++v) total += p[v];
      const double t = static_cast<double>(u[D]) * total;
      double run = 0.0;
      int k = -1, last = -1;
      for (int v = 0; v < V; ++v) {
        if (p[v] > 0.0) last = v;
        run += p[v];
        if (k < 0 && run > t) k = v;
      }
      accept[b] = a;
      token[b] = k >= 0 ? k : last;
    }
  });
  return kOk;
}

// Out-of-place realignment of caches laid out [L][2][B][H][S][col_bytes] (S = s_src or s_dst
// columns).  n[B], width, accept[B], token[B], draft[B][D], ids_src[B][s_src] in; dst, ids_dst,
// mask_dst, pos_dst ([B][s_dst]), n_out[B], *w_out out.  Returns 0, 1 (a length or accept length
// out of range, W + D > s_src) or 2 (W' + D > s_dst); nothing is written on an error.
int cpu_realign(const void* src, void* dst, int L, int B, int H, int s_src, int s_dst,
                int col_bytes, int D, const int32_t* n, int width, const int32_t* accept,
                const int32_t* token, const int32_t* draft, const int32_t* ids_src,
                int32_t* ids_dst, uint8_t* mask_dst, int32_t* pos_dst, int32_t* n_out,
                int32_t* w_out, int32_t pad_id, int threads) {
  if (L < 1 || B < 0 || H < 1 || s_src < 1 || s_dst < 1 || col_bytes < 1 || D < 1) return kErrArg;
  if (width + D > s_src) return kErrRange;
  int w_new = 0;
  for (int b = 0; b < B; ++b) {
    if (n[b] < 1 || n[b] > width || accept[b] < 0 || accept[b] > D) return kErrRange;
    const int nn = n[b] + accept[b] + 1;
    if (nn > w_new) w_new = nn;
  }
  if (w_new + D > s_dst) return kErrCapacity;
  const long long src_head = static_cast<long long>(s_src) * col_bytes;
  const long long dst_head = static_cast<long long>(s_dst) * col_bytes;
  // Runs (l, kv, b, h): the K/V moves, split over the threads.
  const long long runs = static_cast<long long>(L) * 2 * B * H;
  parallel_for(runs, threads, [&](int, long long lo, long long hi) {
    for (long long k = lo; k < hi; ++k) {
      const long long lkv = k / (static_cast<long long>(B) * H);
      const int b = static_cast<int>((k / H) % B);
      const long long row = lkv * B + b;  // (l, kv, b)
      const int h = static_cast<int>(k % H);
      const int keep = n[b] + accept[b];
      const int s_lo = width - n[b];
      const int d_lo = w_new - (n[b] + accept[b] + 1);
      const char* s = static_cast<const char*>(src) + (row * H + h) * src_head +
                      static_cast<long long>(s_lo) * col_bytes;
      char* d = static_cast<char*>(dst) + (row * H + h) * dst_head +
                static_cast<long long>(d_lo) * col_bytes;
      std::memcpy(d, s, static_cast<size_t>(keep) * col_bytes);
    }
  });
  // The per-row metadata, split over the threads by row.
  parallel_for(B, threads, [&](int, long long lo, long long hi) {
    for (long long b = lo; b < hi; ++b) {
      const int N = n[b], a = accept[b], nn = N + a + 1;
      const int d_lo = w_new - nn;
      int32_t* ids = ids_dst + b * s_dst;
      uint8_t* mask = mask_dst + b * s_dst;
      int32_t* pos = pos_dst + b * s_dst;
      for (int c = 0; c < s_dst; ++c) {
        ids[c] = pad_id;
        mask[c] = 0;
        pos[c] = 0;
      }
      for (int q = 0; q < nn; ++q) {
        int32_t id;
        if (q < N) id = ids_src[b * s_src + (width - N) + q];
        else if (q < N + a) id = draft[b * D + (q - N)];
        else id = token[b];
        ids[d_lo + q] = id;
        mask[d_lo + q] = 1;
        pos[d_lo + q] = q;
      }
      n_out[b] = nn;
    }
  });
  *w_out = w_new;
  return kOk;
}

}  // extern "C"
