// Realignment of a left-padded speculative batch (EQSPEC unpad-append-repad) and the pool moves
// of EXSPEC's mixed leftovers.
//
// "Batch Speculative Decoding Done Right", section 2.2: unpad every row, append the accepted
// tokens and the bonus/replacement token, re-left-pad to the longest row, recompute position
// IDs and shift the KV cache; section 2.1: afterwards pad + content is equal for every row
// (rectangular alignment) and position IDs run from 0 over the content (contiguity); section
// 2.3: in a pool only mixed-length rows are realigned.  "Correctness Forensics for Batch
// Speculative Decoding", Abstract: under contiguous layouts this realignment is the cost that
// grows superlinearly with batch size.  "Inference Engineering: Part 5/8", "Acceptance changes
// across the workload": committed K/V is kept, speculative K/V after the first rejection is
// discarded (here: never copied).
//
// GB300 mapping.  The work is a set of contiguous byte runs, one per (layer, k/v, row, head):
// run (l, kv, r, h) moves ncols_r columns of col_bytes from src column src_col_r to dst column
// dst_col_r.  Every CTA recomputes the per-row plan from a few device ints (so no host
// synchronisation is needed) and cuts every run into tiles of at most `tile` bytes.  The tiles
// are numbered (l, kv, row, head, chunk) -- memory order -- and the CTAs of a persistent grid
// (a multiple of the SM count) share them out (see Scheduling).  One elected thread streams
// its tiles through a ring of shared-memory stages with cp.async.bulk global->shared
// (completion on an mbarrier) and cp.async.bulk shared->global (bulk groups), keeping
// stages-1 loads in flight; the other warps meanwhile write the ids, mask and position IDs.
// Bytes moved = read + write of every surviving column, nothing else.
//
// Scheduling.  With a caller-owned schedule (two 32-bit words), the tiles are cut into work
// items -- a few tiles, or one whole run in place, longest runs first -- and every CTA's elected
// thread takes the next item from a counter as its ring frees up, keeping one item taken
// ahead.  Measured on GB300, the SMs of one launch stream at unequal rates (the first CTA of an
// equal split finishes ~20 % before the last), so a fixed split leaves SMs idle at the end while
// items from a counter keep them all busy to the last item.  The last CTA to finish sets the
// words back to zero.  Without a schedule every CTA takes one fixed, contiguous share of the
// tiles (in place: ending at the nearest run boundary).
//
// In place (EQSPEC, one K/V buffer): a run moves within its own head row by the row's shift
// s = dst_col - src_col.  Every run is handled by one CTA, which takes its tiles in ascending
// column order when s < 0 and descending when s > 0;
// since a tile is stored only after its own load and every earlier load has landed, no store
// reaches source bytes that are still to be read.  Rows with s = 0 move nothing.
#include <climits>

#include "common.cuh"

#ifndef SPECDEC_REALIGN_TILE
#define SPECDEC_REALIGN_TILE 65536
#endif
#ifndef SPECDEC_REALIGN_STAGES
#define SPECDEC_REALIGN_STAGES 3
#endif
#ifndef SPECDEC_REALIGN_CTAS_PER_SM
#define SPECDEC_REALIGN_CTAS_PER_SM 1
#endif
#ifndef SPECDEC_APPEND_CTAS_PER_SM
#define SPECDEC_APPEND_CTAS_PER_SM 4
#endif

namespace specdec {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxRows = 1024;
constexpr int kMaxStages = 8;
constexpr uint32_t kWaitTries = 1u << 22;
constexpr int kVecUnroll = 8;
constexpr int kLptRows = 256;  // scheduled in place: longest-first item order up to this many rows

enum Mode { kEqspec = 0, kPoolGather = 1, kPoolAppend = 2 };

struct ByteView {
  char* base;
  long long sl, skv, srow, shead;  // bytes
};

struct Params {
  ByteView src, dst;
  int mode, R, D, L, H, col_bytes, tile, stages, copy_engine, in_place, by_slot;
  int kv_in_place;  // EQSPEC: src and dst are one K/V buffer
  int pdl;          // launch with programmatic stream serialization
  int32_t pad_id;
  // EQSPEC
  const int32_t* n_committed;
  const int32_t* width;
  const int32_t* accept_len;
  const int32_t* out_token;
  const int32_t* draft;
  const int32_t* ids_src;
  int src_cap, dst_cap;
  int32_t* ids_dst;
  uint8_t* mask_dst;
  int32_t* pos_dst;
  int32_t* n_dst;
  int32_t* width_dst;
  // pool
  const int32_t* rows;
  const int32_t* slot_col;
  const int32_t* slot_cap;
  int32_t* slot_len;
  int32_t* pool_ids;
  int ids_cap;
  int32_t* batch_len;
  int32_t* bwidth;
  int32_t* s_ids;
  uint8_t* s_mask;
  int32_t* s_pos;
  int scratch_cap, arena_cap;
  uint8_t* slot_state;  // append: retirement when set
  const int32_t* slot_limit;
  int32_t eos_id;
  int32_t* status;
  unsigned* sched;  // [2] next work item, finished CTAs (zero between calls); null: fixed shares
};

struct Plan {  // per-row plan, arrays in dynamic shared memory (8 ints per row)
  int *src_col, *dst_col, *ncols, *tiles, *prefix;
  int* order;  // scheduled, in place: the rows that move, longest first (runs_per_group / H)
  int* aux;  // EQSPEC: N_b; pool: N_s
  int* acc;  // EQSPEC / append: a
  int W, Wp, per_group;
  int runs_per_group;  // runs with at least one tile in one (layer, k/v) group
};

__host__ __device__ constexpr size_t plan_bytes(int rows) {
  return static_cast<size_t>(rows) * 8 * sizeof(int);
}

__device__ __forceinline__ int src_row_of(int mode, int r) { return mode == kPoolGather ? 0 : r; }
__device__ __forceinline__ int dst_row_of(int mode, int r) { return mode == kPoolAppend ? 0 : r; }

__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide max and or of one int per thread (results broadcast through shared memory).
__device__ void block_max_or(int& mx, int& orv, int* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  mx = warp_max(mx);
  orv = warp_or(orv);
  __syncthreads();
  if (lane == 0) { red[warp] = mx; red[32 + warp] = orv; }
  __syncthreads();
  if (warp == 0) {
    int m = lane < kThreads / 32 ? red[lane] : INT_MIN;
    int o = lane < kThreads / 32 ? red[32 + lane] : 0;
    m = warp_max(m);
    o = warp_or(o);
    if (lane == 0) { red[64] = m; red[65] = o; }
  }
  __syncthreads();
  mx = red[64];
  orv = red[65];
  __syncthreads();
}

// Build the per-row plan; returns false (after recording a status) when nothing may be written.
// Every CTA computes the same plan from the same inputs, so every CTA takes the same branch.
__device__ bool build_plan(const Params& p, Plan& s, int* red) {
  const int R = p.R, D = p.D;
  int mx = INT_MIN, bad = 0;  // bad: bit0 range error, bit1 capacity
  if (p.mode == kEqspec) {
    const int W = *p.width;
    for (int r = threadIdx.x; r < R; r += kThreads) {
      const int N = p.n_committed[r], a = p.accept_len[r];
      if (N < 1 || N > W || a < 0 || a > D) bad |= 1;
      s.aux[r] = N;
      s.acc[r] = a;
      mx = max(mx, N + a + 1);
    }
    if (W < 1 || W + D > p.src_cap) bad |= 1;
    block_max_or(mx, bad, red);
    if (!(bad & 1) && mx + D > p.dst_cap) bad |= 2;
    if (threadIdx.x == 0) { s.W = W; s.Wp = mx; }
    for (int r = threadIdx.x; r < R; r += kThreads) {
      const int N = s.aux[r], a = s.acc[r];
      s.src_col[r] = W - N;
      s.dst_col[r] = mx - (N + a + 1);
      s.ncols[r] = (p.kv_in_place && s.src_col[r] == s.dst_col[r]) ? 0 : N + a;
    }
  } else if (p.mode == kPoolGather) {
    for (int r = threadIdx.x; r < R; r += kThreads) {
      const int sl = p.rows[r];
      const int N = p.slot_len[sl], cap = p.slot_cap[sl], c0 = p.slot_col[sl];
      if (N < 1 || N > cap || N > p.ids_cap || c0 < 0 || cap > p.arena_cap - c0) bad |= 1;
      else if (N + D > cap) bad |= 2;
      s.aux[r] = N;
      mx = max(mx, N);
    }
    block_max_or(mx, bad, red);
    if (!(bad & 1) && !p.in_place && mx + D > p.scratch_cap) bad |= 2;
    if (threadIdx.x == 0) { s.W = mx; s.Wp = mx; }
    for (int r = threadIdx.x; r < R; r += kThreads) {
      const int N = s.aux[r];
      s.src_col[r] = p.slot_col[p.rows[r]];
      s.dst_col[r] = mx - N;
      s.ncols[r] = p.in_place ? 0 : N - 1;
    }
  } else {  // kPoolAppend
    const int W = *p.bwidth;
    for (int r = threadIdx.x; r < R; r += kThreads) {
      const int sl = p.rows[r], c0 = p.slot_col[sl], cap = p.slot_cap[sl];
      const int N = p.batch_len[r], a = p.accept_len[p.by_slot ? sl : r];
      if (a < 0 || a > D || N < 1 || N > W || c0 < 0 || cap > p.arena_cap - c0) bad |= 1;
      else if (N + a + 1 > p.ids_cap || N + a > cap) bad |= 2;
      s.aux[r] = N;
      s.acc[r] = a;
    }
    if (!p.in_place && (W < 1 || W + D > p.scratch_cap)) bad |= 1;
    block_max_or(mx, bad, red);
    if (threadIdx.x == 0) { s.W = W; s.Wp = W; }
    for (int r = threadIdx.x; r < R; r += kThreads) {
      const int N = s.aux[r], a = s.acc[r];
      s.src_col[r] = W - 1;
      s.dst_col[r] = p.slot_col[p.rows[r]] + N - 1;
      s.ncols[r] = p.in_place ? 0 : a + 1;
    }
  }
  if (bad) {
    if (threadIdx.x == 0)
      set_status(p.status, (bad & 1) ? SPECDEC_ERR_INPUT_RANGE : SPECDEC_ERR_CAPACITY);
    return false;
  }
  // Tiles per head run and their prefix over rows (warp 0, lane-contiguous row blocks).
  for (int r = threadIdx.x; r < R; r += kThreads) {
    const long long bytes = static_cast<long long>(s.ncols[r]) * p.col_bytes;
    s.tiles[r] = static_cast<int>((bytes + p.tile - 1) / p.tile);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (R + 31) / 32;
    const int r0 = min(R, lane * per), r1 = min(R, r0 + per);
    int local = 0, runs = 0;
    for (int r = r0; r < r1; ++r) {
      local += s.tiles[r] * p.H;
      runs += s.tiles[r] > 0 ? p.H : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) runs += __shfl_xor_sync(0xffffffffu, runs, o);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int r = r0; r < r1; ++r) {
      s.prefix[r] = run;
      run += s.tiles[r] * p.H;
    }
    if (lane == 31) {
      s.per_group = incl;
      s.runs_per_group = runs;
    }
    if (p.sched && p.kv_in_place && R > kLptRows) {  // the moving rows in index order
      int nz = 0;
      for (int r = r0; r < r1; ++r) nz += s.tiles[r] > 0;
      int nz_incl = nz;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, nz_incl, o);
        if (lane >= o) nz_incl += v;
      }
      int k = nz_incl - nz;
      for (int r = r0; r < r1; ++r)
        if (s.tiles[r] > 0) s.order[k++] = r;
    }
  }
  if (p.sched && p.kv_in_place && R <= kLptRows) {
    // The moving rows, longest runs first (ties: lower row first), so that the last work items
    // a scheduled launch hands out are its shortest runs.
    for (int r = threadIdx.x; r < R; r += kThreads) {
      const int tr = s.tiles[r];
      if (tr == 0) continue;
      int rank = 0;
      for (int q = 0; q < R; ++q) {
        const int tq = s.tiles[q];
        rank += (tq > tr) || (tq == tr && q < r);
      }
      s.order[rank] = r;
    }
  }
  __syncthreads();
  return true;
}

struct Tile {
  const char* src;
  char* dst;
  uint32_t bytes;
};

__device__ __forceinline__ Tile decode(const Params& p, const Plan& s, long long t) {
  const int per = s.per_group;
  const long long g = t / per;  // (layer, kv) group
  const int in = static_cast<int>(t - g * per);
  // Largest row r with prefix[r] <= in (rows with no tiles share their successor's prefix).
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.prefix[mid] <= in) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const int within = in - s.prefix[r];
  const int c = s.tiles[r];
  const int h = within / c;
  int chunk = within - h * c;
  if (p.kv_in_place && s.dst_col[r] > s.src_col[r]) chunk = c - 1 - chunk;  // right shift: last first
  const long long off = static_cast<long long>(chunk) * p.tile;
  const long long run = static_cast<long long>(s.ncols[r]) * p.col_bytes;
  const long long l = g >> 1, kv = g & 1;
  Tile tl;
  tl.src = p.src.base + l * p.src.sl + kv * p.src.skv + src_row_of(p.mode, r) * p.src.srow +
           h * p.src.shead + static_cast<long long>(s.src_col[r]) * p.col_bytes + off;
  tl.dst = p.dst.base + l * p.dst.sl + kv * p.dst.skv + dst_row_of(p.mode, r) * p.dst.srow +
           h * p.dst.shead + static_cast<long long>(s.dst_col[r]) * p.col_bytes + off;
  tl.bytes = static_cast<uint32_t>(min(static_cast<long long>(p.tile), run - off));
  return tl;
}

// The run boundary nearest to tile t: the first tile of the run that holds t, or the first tile
// after that run, whichever is closer (t == total: total).  Monotone in t, so boundaries taken
// from increasing t still partition the tiles.
__device__ long long run_boundary(const Params& p, const Plan& s, long long t, long long total) {
  if (t >= total) return total;
  const int per = s.per_group;
  const long long g = t / per;
  const int in = static_cast<int>(t - g * per);
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.prefix[mid] <= in) lo = mid; else hi = mid - 1;
  }
  const int c = s.tiles[lo];
  const int chunk = (in - s.prefix[lo]) % c;
  return 2 * chunk > c ? t - chunk + c : t - chunk;
}

// One elected thread moves the tiles that next_tile() hands out, in that order, through
// `stages` shared-memory buffers: stages - 1 loads stay in flight behind each store.
template <class NextTile>
__device__ void copy_bulk(const Params& p, const Plan& s, NextTile&& next_tile, char* ring,
                          uint64_t* bars, char** ring_dst, uint32_t* ring_bytes) {
  const int S = p.stages;
  long long issued = 0, t = 0;
  bool more = true;
  for (int k = 0; k < S; ++k) {
    if (!next_tile(t)) {
      more = false;
      break;
    }
    const Tile tl = decode(p, s, t);
    ring_dst[k] = tl.dst;
    ring_bytes[k] = tl.bytes;
    mbar_arrive_expect_tx(&bars[k], tl.bytes);
    bulk_g2s(ring + static_cast<long long>(k) * p.tile, tl.src, tl.bytes, &bars[k]);
    ++issued;
  }
  for (long long i = 0; i < issued; ++i) {
    const int st = static_cast<int>(i % S);
    const uint32_t parity = static_cast<uint32_t>((i / S) & 1);
    if (!mbar_wait_bounded(&bars[st], parity, kWaitTries)) {
      set_status(p.status, SPECDEC_ERR_TIMEOUT);
      // Give the loads still in flight a bounded chance to land before the CTA exits.
      for (long long k = i + 1; k < issued; ++k)
        (void)mbar_wait_bounded(&bars[k % S], static_cast<uint32_t>((k / S) & 1), kWaitTries);
      break;
    }
    bulk_s2g(ring_dst[st], ring + static_cast<long long>(st) * p.tile, ring_bytes[st]);
    bulk_commit();
    if (i >= 1 && more) {
      // Refill the stage of tile i-1 (its store must have read shared memory) with tile
      // number i-1+S.
      bulk_wait_read<1>();
      if (!next_tile(t)) {
        more = false;
        continue;
      }
      const int rs = static_cast<int>((i - 1) % S);
      const Tile tl = decode(p, s, t);
      ring_dst[rs] = tl.dst;
      ring_bytes[rs] = tl.bytes;
      mbar_arrive_expect_tx(&bars[rs], tl.bytes);
      bulk_g2s(ring + static_cast<long long>(rs) * p.tile, tl.src, tl.bytes, &bars[rs]);
      ++issued;
    }
  }
  bulk_wait_all();
}

// Work items for the counter.  Out of place: kItemTiles consecutive tiles (runs may be cut).
// In place: one run each (a run is moved by one CTA), the longest rows' runs first, so that the
// items handed out last -- the ones that decide when the launch ends -- are the shortest.  The
// first item of every CTA is its own index; later ones come from the counter, offset by the grid
// size, so the launch does not start with every CTA on one atomic.
constexpr long long kItemTiles = 4;

__device__ void copy_bulk_scheduled(const Params& p, const Plan& s, long long total, char* ring,
                                    uint64_t* bars, char** ring_dst, uint32_t* ring_bytes) {
  const long long row_runs = 2LL * p.L * p.H;  // runs of one row (every (layer, k/v, head))
  const long long items =
      p.kv_in_place ? static_cast<long long>(s.runs_per_group / p.H) * row_runs
                    : (total + kItemTiles - 1) / kItemTiles;
  long long cur = 0, end = 0;
  long long ahead = blockIdx.x;  // the next item
  copy_bulk(p, s, [&](long long& t) -> bool {
    while (cur >= end) {
      if (ahead >= items) return false;
      if (p.kv_in_place) {
        const long long q = ahead / row_runs, rem = ahead - q * row_runs;
        const long long g = rem / p.H, h = rem - g * p.H;
        const int r = s.order[q];
        cur = g * s.per_group + s.prefix[r] + h * s.tiles[r];
        end = cur + s.tiles[r];
      } else {
        cur = ahead * kItemTiles;
        end = cur + kItemTiles < total ? cur + kItemTiles : total;
      }
      ahead = static_cast<long long>(atomicAdd(&p.sched[0], 1u)) + gridDim.x;
    }
    t = cur++;
    return true;
  }, ring, bars, ring_dst, ring_bytes);
  // Every CTA has taken its last item once all have passed here: the last one clears the words.
  __threadfence();
  if (atomicAdd(&p.sched[1], 1u) == gridDim.x - 1) {
    p.sched[0] = 0u;
    p.sched[1] = 0u;
    __threadfence();
  }
}

// A coherent 16-byte global load.  In place the kernel writes bytes that other threads of the
// CTA load, so the non-coherent read-only path is not allowed there: its loads are outside the
// memory model, and a block barrier does not keep another thread's later store from reaching a
// load still in flight.  A plain load is ordered before the stores behind the barrier.
__device__ __forceinline__ uint4 ldg_coherent(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
  return r;
}

// All threads of the CTA move tiles [t0, t1) with 16-byte loads/stores (streaming read-only
// loads out of place, coherent loads in place).
__device__ void copy_vec(const Params& p, const Plan& s, long long t0, long long t1) {
  for (long long t = t0; t < t1; ++t) {
    const Tile tl = decode(p, s, t);
    const uint4* src = reinterpret_cast<const uint4*>(tl.src);
    uint4* dst = reinterpret_cast<uint4*>(tl.dst);
    const int nv = static_cast<int>(tl.bytes / 16);
    for (int base = 0; base < nv; base += kThreads * kVecUnroll) {
      uint4 buf[kVecUnroll];
#pragma unroll
      for (int k = 0; k < kVecUnroll; ++k) {
        const int v = base + k * kThreads + threadIdx.x;
        if (v < nv) buf[k] = p.kv_in_place ? ldg_coherent(src + v) : ldg_stream(src + v);
      }
      // In place a tile's destination may overlap its own source: every thread has loaded its
      // part (tiles are at most kThreads * kVecUnroll vectors) before any thread stores.
      if (p.kv_in_place) __syncthreads();
#pragma unroll
      for (int k = 0; k < kVecUnroll; ++k) {
        const int v = base + k * kThreads + threadIdx.x;
        if (v < nv) dst[v] = buf[k];
      }
    }
  }
}

// Metadata: grid-wide items through (gt, gn); the small per-row outputs in CTA 0 through (lt, ln).
__device__ void write_metadata(const Params& p, const Plan& s, long long gt, long long gn, int lt,
                               int ln) {
  if (p.mode == kEqspec) {
    const long long items = static_cast<long long>(p.R) * p.dst_cap;
    const int W = s.W, Wp = s.Wp;
    for (long long k = gt; k < items; k += gn) {
      const int r = static_cast<int>(k / p.dst_cap);
      const int c = static_cast<int>(k - static_cast<long long>(r) * p.dst_cap);
      const int N = s.aux[r], a = s.acc[r];
      const int lo = Wp - (N + a + 1);
      int id = p.pad_id, pos = 0;
      uint8_t m = 0;
      if (c >= lo && c < Wp) {
        const int q = c - lo;
        pos = q;
        m = 1;
        if (q < N) id = p.ids_src[static_cast<long long>(r) * p.src_cap + (W - N) + q];
        else if (q < N + a) id = p.draft[static_cast<long long>(r) * p.D + (q - N)];
        else id = p.out_token[r];
      }
      p.ids_dst[k] = id;
      p.mask_dst[k] = m;
      p.pos_dst[k] = pos;
    }
    if (blockIdx.x == 0) {
      for (int r = lt; r < p.R; r += ln) p.n_dst[r] = s.aux[r] + s.acc[r] + 1;
      if (lt == 0) *p.width_dst = Wp;
    }
  } else if (p.mode == kPoolGather) {
    if (!p.in_place) {
      const long long items = static_cast<long long>(p.R) * p.scratch_cap;
      const int W = s.W;
      for (long long k = gt; k < items; k += gn) {
        const int r = static_cast<int>(k / p.scratch_cap);
        const int c = static_cast<int>(k - static_cast<long long>(r) * p.scratch_cap);
        const int N = s.aux[r];
        const int lo = W - N;
        int id = p.pad_id, pos = 0;
        uint8_t m = 0;
        if (c >= lo && c < W) {
          pos = c - lo;
          m = 1;
          id = p.pool_ids[static_cast<long long>(p.rows[r]) * p.ids_cap + pos];
        }
        p.s_ids[k] = id;
        p.s_mask[k] = m;
        p.s_pos[k] = pos;
      }
    }
    if (blockIdx.x == 0) {
      for (int r = lt; r < p.R; r += ln) p.batch_len[r] = s.aux[r];
      if (lt == 0) *p.bwidth = s.W;
    }
  } else if (blockIdx.x == 0) {  // kPoolAppend: tiny, one CTA
    for (int r = lt; r < p.R; r += ln) {
      const int sl = p.rows[r];
      const int N = s.aux[r], a = s.acc[r];
      const int src = p.by_slot ? sl : r;  // row of accept_len / out_token / draft
      if (p.slot_state && p.slot_state[sl] != SPECDEC_SLOT_ACTIVE) {
        set_status(p.status, SPECDEC_ERR_INPUT_RANGE);
        continue;
      }
      int32_t* ids = p.pool_ids + static_cast<long long>(sl) * p.ids_cap;
      for (int q = 0; q < a; ++q) ids[N + q] = p.draft[static_cast<long long>(src) * p.D + q];
      ids[N + a] = p.out_token[src];
      int len = N + a + 1;
      if (p.slot_state) {  // retirement: first end-of-sequence token or the length limit
        const int lim = p.slot_limit[sl];
        for (int q = N; q <= N + a; ++q) {
          if (ids[q] == p.eos_id) {
            len = q + 1;
            p.slot_state[sl] = SPECDEC_SLOT_FINISHED_EOS;
            break;
          }
          if (q + 1 >= lim) {
            len = q + 1;
            p.slot_state[sl] = SPECDEC_SLOT_FINISHED_LENGTH;
            break;
          }
        }
      }
      p.slot_len[sl] = len;
    }
  }
}

__global__ void __launch_bounds__(kThreads) realign_kernel(const Params p) {
  // Launched with programmatic serialization, this grid may be resident before the verification
  // ahead of it has finished: wait for it before reading anything it wrote.
  pdl_wait();
  extern __shared__ __align__(128) char dyn[];
  __shared__ Plan s;
  __shared__ int red[72];
  __shared__ __align__(8) uint64_t bars[kMaxStages];
  __shared__ char* ring_dst[kMaxStages];
  __shared__ uint32_t ring_bytes[kMaxStages];

  const size_t ring_total = p.copy_engine == 0 ? static_cast<size_t>(p.tile) * p.stages : 0;
  char* ring = dyn;
  if (threadIdx.x == 0) {
    int* a = reinterpret_cast<int*>(dyn + ring_total);
    s.src_col = a;
    s.dst_col = a + p.R;
    s.ncols = a + 2 * p.R;
    s.tiles = a + 3 * p.R;
    s.prefix = a + 4 * p.R;
    s.aux = a + 5 * p.R;
    s.acc = a + 6 * p.R;
    s.order = a + 7 * p.R;
  }
  __syncthreads();
  if (!build_plan(p, s, red)) return;

  const long long total = 2LL * p.L * s.per_group;
  const long long G = gridDim.x;
  long long t0 = total * blockIdx.x / G;
  long long t1 = total * (blockIdx.x + 1) / G;
  if (p.kv_in_place) {  // whole runs per CTA: move both ends to the nearest run boundary
    t0 = run_boundary(p, s, t0, total);
    t1 = run_boundary(p, s, t1, total);
  }

  if (p.copy_engine == 0) {
    if (threadIdx.x == 0) {
      for (int k = 0; k < p.stages; ++k) mbar_init(&bars[k], 1);
      fence_mbar_init();
      if (p.sched) {
        copy_bulk_scheduled(p, s, total, ring, bars, ring_dst, ring_bytes);
      } else {
        long long next = t0;
        copy_bulk(p, s, [&](long long& t) -> bool {
          if (next >= t1) return false;
          t = next++;
          return true;
        }, ring, bars, ring_dst, ring_bytes);
      }
    } else if (threadIdx.x >= 32) {
      const int per_cta = kThreads - 32;
      const int lt = threadIdx.x - 32;
      write_metadata(p, s, static_cast<long long>(blockIdx.x) * per_cta + lt, G * per_cta, lt,
                     per_cta);
    }
  } else {
    copy_vec(p, s, t0, t1);
    write_metadata(p, s, static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x,
                   G * kThreads, threadIdx.x, kThreads);
  }
}

int check_view(const specdec_kv_view& v, int es_expect) {
  const int es = elem_size(v.dtype);
  if (es == 0 || !v.base) return SPECDEC_ERR_INVALID_ARG;
  if (es_expect && es != es_expect) return SPECDEC_ERR_INVALID_ARG;
  if (v.layers < 1 || v.rows < 1 || v.heads < 1 || v.head_dim < 1 || v.cap_cols < 1)
    return SPECDEC_ERR_INVALID_ARG;
  if (v.stride_layer < 0 || v.stride_kv < 0 || v.stride_row < 0 || v.stride_head < 0)
    return SPECDEC_ERR_INVALID_ARG;
  const long long cb = static_cast<long long>(v.head_dim) * es;
  if (cb % 16 || reinterpret_cast<uintptr_t>(v.base) % 16 || (v.stride_layer * es) % 16 ||
      (v.stride_kv * es) % 16 || (v.stride_row * es) % 16 || (v.stride_head * es) % 16)
    return SPECDEC_ERR_UNSUPPORTED;
  if (static_cast<long long>(v.cap_cols) * cb > (1LL << 40)) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}

// Byte span [lo, hi) a view can address (for overlap checks).
void view_span(const specdec_kv_view& v, uintptr_t& lo, uintptr_t& hi) {
  const long long es = elem_size(v.dtype);
  const long long last = (v.layers - 1) * v.stride_layer + v.stride_kv +
                         (v.rows - 1) * v.stride_row + (v.heads - 1) * v.stride_head +
                         static_cast<long long>(v.cap_cols) * v.head_dim;
  lo = reinterpret_cast<uintptr_t>(v.base);
  hi = lo + static_cast<uintptr_t>(last * es);
}

ByteView to_bytes(const specdec_kv_view& v) {
  const long long es = elem_size(v.dtype);
  return ByteView{static_cast<char*>(v.base), v.stride_layer * es, v.stride_kv * es,
                  v.stride_row * es, v.stride_head * es};
}

int launch(Params& p, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return SPECDEC_ERR_CUDA;
  static_assert(SPECDEC_REALIGN_TILE % 16 == 0, "tile must be a multiple of 16 bytes");
  static_assert(SPECDEC_REALIGN_TILE < (1 << 20), "a tile must fit one mbarrier transaction count");
  static_assert(SPECDEC_REALIGN_STAGES >= 2 && SPECDEC_REALIGN_STAGES <= kMaxStages, "stages");
  // The vector engine loads a whole tile before storing it (in place, its destination may
  // overlap its source): its tiles are one pass of kThreads * kVecUnroll vectors at most.
  constexpr int kVecTile = SPECDEC_REALIGN_TILE < kThreads * kVecUnroll * 16
                               ? SPECDEC_REALIGN_TILE : kThreads * kVecUnroll * 16;
  p.tile = p.copy_engine == 0 ? SPECDEC_REALIGN_TILE : kVecTile;
  p.stages = SPECDEC_REALIGN_STAGES;
  int ctas_per_sm = SPECDEC_REALIGN_CTAS_PER_SM;
  if (p.mode == kPoolAppend && p.copy_engine == 0) {
    // An append moves at most D + 1 columns per run: one small tile per run, and more CTAs per
    // SM issuing copies (the number of copies in flight, not their size, bounds these launches).
    const long long run = static_cast<long long>(p.D + 1) * p.col_bytes;  // a multiple of 16
    if (run < p.tile) p.tile = static_cast<int>(run);
    ctas_per_sm = SPECDEC_APPEND_CTAS_PER_SM;
  }
  const size_t ring = p.copy_engine == 0 ? static_cast<size_t>(p.tile) * p.stages : 0;
  const size_t smem = ring + plan_bytes(p.R);
  constexpr size_t kMaxSmem =
      static_cast<size_t>(SPECDEC_REALIGN_TILE) * SPECDEC_REALIGN_STAGES + plan_bytes(kMaxRows);
  static bool attr_set[64] = {false};  // the attribute is per function and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPECDEC_ERR_CUDA;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        realign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxSmem));
    if (e != cudaSuccess) return map_cuda_error(e);
    attr_set[dev] = true;
  }
  const int grid = sms * ctas_per_sm;
  if (p.pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return map_cuda_error(cudaLaunchKernelEx(&cfg, realign_kernel, p));
  }
  realign_kernel<<<grid, kThreads, smem, stream>>>(p);
  return map_cuda_error(cudaGetLastError());
}

int pool_common(const specdec_pool_args* a, Params& p, bool append) {
  if (!a) return SPECDEC_ERR_INVALID_ARG;
  if (a->n_rows < 1 || a->D < 1 || a->ids_cap < 1) return SPECDEC_ERR_INVALID_ARG;
  if (a->D > SPECDEC_MAX_DRAFT || a->n_rows > kMaxRows) return SPECDEC_ERR_UNSUPPORTED;
  int st = check_view(a->arena, 0);
  if (st) return st;
  st = check_view(a->scratch, elem_size(a->arena.dtype));
  if (st) return st;
  const specdec_kv_view &ar = a->arena, &sc = a->scratch;
  if (ar.rows != 1 || ar.layers != sc.layers || ar.heads != sc.heads ||
      ar.head_dim != sc.head_dim || a->n_rows > sc.rows)
    return SPECDEC_ERR_INVALID_ARG;
  if (!a->rows || !a->slot_col || !a->slot_cap || !a->slot_len || !a->pool_ids ||
      !a->batch_len || !a->width || !a->dev_status)
    return SPECDEC_ERR_INVALID_ARG;
  if (!append && !a->in_place && (!a->scratch_ids || !a->scratch_mask || !a->scratch_pos))
    return SPECDEC_ERR_INVALID_ARG;
  if (append && (!a->accept_len || !a->out_token || !a->draft)) return SPECDEC_ERR_INVALID_ARG;
  if (append && a->slot_state && !a->slot_limit) return SPECDEC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a->schedule) % alignof(uint32_t)) return SPECDEC_ERR_INVALID_ARG;
  uintptr_t alo, ahi, slo, shi;
  view_span(ar, alo, ahi);
  view_span(sc, slo, shi);
  if (!a->in_place && alo < shi && slo < ahi) return SPECDEC_ERR_INVALID_ARG;
  p = Params{};
  p.src = append ? to_bytes(sc) : to_bytes(ar);
  p.dst = append ? to_bytes(ar) : to_bytes(sc);
  p.mode = append ? kPoolAppend : kPoolGather;
  p.R = a->n_rows;
  p.D = a->D;
  p.L = ar.layers;
  p.H = ar.heads;
  p.col_bytes = ar.head_dim * elem_size(ar.dtype);
  p.copy_engine = 0;
  p.in_place = a->in_place ? 1 : 0;
  p.by_slot = a->by_slot ? 1 : 0;
  p.pad_id = a->pad_id;
  p.accept_len = a->accept_len;
  p.out_token = a->out_token;
  p.draft = a->draft;
  p.rows = a->rows;
  p.slot_col = a->slot_col;
  p.slot_cap = a->slot_cap;
  p.slot_len = a->slot_len;
  p.pool_ids = a->pool_ids;
  p.ids_cap = a->ids_cap;
  p.batch_len = a->batch_len;
  p.bwidth = a->width;
  p.s_ids = a->scratch_ids;
  p.s_mask = a->scratch_mask;
  p.s_pos = a->scratch_pos;
  p.scratch_cap = sc.cap_cols;
  p.arena_cap = ar.cap_cols;
  p.slot_state = append ? a->slot_state : nullptr;
  p.slot_limit = a->slot_limit;
  p.eos_id = a->eos_id;
  p.status = a->dev_status;
  p.sched = reinterpret_cast<unsigned*>(a->schedule);
  return SPECDEC_OK;
}

}  // namespace
}  // namespace specdec

namespace specdec {
namespace {

int realign_common(const specdec_realign_args* a, bool in_place, void* stream) {
  if (!a) return SPECDEC_ERR_INVALID_ARG;
  if (a->B < 0 || a->D < 1) return SPECDEC_ERR_INVALID_ARG;
  if (a->D > SPECDEC_MAX_DRAFT || a->B > kMaxRows) return SPECDEC_ERR_UNSUPPORTED;
  if (a->copy_engine != 0 && a->copy_engine != 1) return SPECDEC_ERR_INVALID_ARG;
  if (a->flags & ~SPECDEC_REALIGN_PDL) return SPECDEC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a->schedule) % alignof(uint32_t)) return SPECDEC_ERR_INVALID_ARG;
  if (a->B == 0) return SPECDEC_OK;
  int st = check_view(a->src, 0);
  if (st) return st;
  st = check_view(a->dst, elem_size(a->src.dtype));
  if (st) return st;
  const specdec_kv_view &s = a->src, &d = a->dst;
  if (s.layers != d.layers || s.heads != d.heads || s.head_dim != d.head_dim || s.rows != a->B ||
      d.rows != a->B)
    return SPECDEC_ERR_INVALID_ARG;
  if (in_place) {  // one K/V buffer: the destination view must be the source view
    if (d.base != s.base || d.stride_layer != s.stride_layer || d.stride_kv != s.stride_kv ||
        d.stride_row != s.stride_row || d.stride_head != s.stride_head || d.dtype != s.dtype ||
        d.cap_cols != s.cap_cols)
      return SPECDEC_ERR_INVALID_ARG;
  } else {
    uintptr_t slo, shi, dlo, dhi;
    view_span(s, slo, shi);
    view_span(d, dlo, dhi);
    if (slo < dhi && dlo < shi) return SPECDEC_ERR_INVALID_ARG;  // out of place: no overlap
  }
  if (!a->n_committed || !a->width || !a->accept_len || !a->out_token || !a->draft ||
      !a->ids_src || !a->ids_dst || !a->mask_dst || !a->pos_dst || !a->n_committed_dst ||
      !a->width_dst || !a->dev_status)
    return SPECDEC_ERR_INVALID_ARG;
  if (a->n_committed == a->n_committed_dst || a->width == a->width_dst ||
      a->ids_src == a->ids_dst)
    return SPECDEC_ERR_INVALID_ARG;
  Params p = {};
  p.src = to_bytes(s);
  p.dst = to_bytes(d);
  p.mode = kEqspec;
  p.R = a->B;
  p.D = a->D;
  p.L = s.layers;
  p.H = s.heads;
  p.col_bytes = s.head_dim * elem_size(s.dtype);
  p.copy_engine = a->copy_engine;
  p.pad_id = a->pad_id;
  p.n_committed = a->n_committed;
  p.width = a->width;
  p.accept_len = a->accept_len;
  p.out_token = a->out_token;
  p.draft = a->draft;
  p.ids_src = a->ids_src;
  p.src_cap = s.cap_cols;
  p.dst_cap = d.cap_cols;
  p.ids_dst = a->ids_dst;
  p.mask_dst = a->mask_dst;
  p.pos_dst = a->pos_dst;
  p.n_dst = a->n_committed_dst;
  p.width_dst = a->width_dst;
  p.status = a->dev_status;
  p.kv_in_place = in_place ? 1 : 0;
  p.pdl = (a->flags & SPECDEC_REALIGN_PDL) ? 1 : 0;
  p.sched = a->copy_engine == 0 ? reinterpret_cast<unsigned*>(a->schedule) : nullptr;
  return launch(p, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace specdec

extern "C" int specdec_realign(const specdec_realign_args* a, void* stream) {
  return specdec::realign_common(a, false, stream);
}

extern "C" int specdec_realign_inplace(const specdec_realign_args* a, void* stream) {
  return specdec::realign_common(a, true, stream);
}

extern "C" int specdec_pool_gather(const specdec_pool_args* a, void* stream) {
  specdec::Params p;
  const int st = specdec::pool_common(a, p, false);
  if (st) return st;
  return specdec::launch(p, static_cast<cudaStream_t>(stream));
}

extern "C" int specdec_pool_append(const specdec_pool_args* a, void* stream) {
  specdec::Params p;
  const int st = specdec::pool_common(a, p, true);
  if (st) return st;
  return specdec::launch(p, static_cast<cudaStream_t>(stream));
}
