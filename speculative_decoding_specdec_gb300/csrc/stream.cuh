// Streaming score elements through a shared-memory ring with bulk async copies (sm_103a).
//
// A CTA's share of score elements is a list of contiguous blocks in global memory.  Each block
// knows the (row, vocabulary index) of its first element; rows are V elements long and follow
// each other inside a block (score rows stored back to back), so a block may cross row
// boundaries.  One producer thread cuts the blocks into chunks of at most `chunk` elements and
// copies each with one cp.async.bulk global->shared into a ring stage; consumer warps wait on
// the stage's "full" mbarrier, process the chunk row segment by row segment, and release the
// stage on its "empty" mbarrier (one arrival per consumer warp).
//
// Large copies matter: a bulk copy costs a roughly fixed issue time, so 32 KB copies move data
// several times faster per CTA than 4 KB ones.  Every wait is bounded; a consumer warp that gives
// up reports failure warp-uniformly.
#pragma once

#include "common.cuh"

namespace specdec {

constexpr uint32_t kStreamWaitTries = 1u << 22;
constexpr uint32_t kSleepTries = 1u << 17;  // consumer polls of at most kSleepNs each (~2.6 s)
constexpr uint32_t kSleepNs = 20000;
constexpr int kMaxBlocks = 2 * SPECDEC_MAX_DRAFT + 2;
constexpr int kMaxRingStages = 8;

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

struct StreamBlock {
  const char* ptr;   // global address of the block's first element (16-byte aligned)
  int len;           // elements (a multiple of 16 bytes' worth)
  int row0, v0;      // row and vocabulary index of the first element
};

// The plan lives in shared memory; thread 0 builds it.
struct StreamPlan {
  StreamBlock blk[kMaxBlocks];
  int nblk, chunk, stages, stage_bytes, total, V, esize;

  __device__ void finish(int chunk_elems, int ring_bytes) {
    chunk = chunk_elems;
    stage_bytes = chunk_elems * esize;
    stages = min(kMaxRingStages, ring_bytes / stage_bytes);
    int c = 0;
    for (int k = 0; k < nblk; ++k) c += (blk[k].len + chunk - 1) / chunk;
    total = c;
  }
};

// Walks the chunks of a plan in order with additions only (no division per chunk).
struct ChunkCursor {
  int k = 0, off = 0;  // block and element offset within it
  int q = 0, v = 0;    // row and vocabulary index of the chunk's first element

  __device__ void start(const StreamPlan& p) {
    k = 0;
    off = 0;
    if (p.nblk > 0) { q = p.blk[0].row0; v = p.blk[0].v0; }
  }
  __device__ int size(const StreamPlan& p) const { return min(p.chunk, p.blk[k].len - off); }
  __device__ void next(const StreamPlan& p, int n) {
    off += n;
    if (off >= p.blk[k].len && k + 1 < p.nblk) {
      ++k;
      off = 0;
      q = p.blk[k].row0;
      v = p.blk[k].v0;
    } else {
      v += n;
      while (v >= p.V) { v -= p.V; ++q; }
    }
  }
};

// Producer (a single thread).  Before returning it waits (bounded) until the last chunks it
// issued have landed, so no copy outlives the CTA.
__device__ inline bool stream_produce(const StreamPlan& plan, char* ring, uint64_t* full,
                                      uint64_t* empty) {
  const int S = plan.stages;
  bool ok = true;
  int issued = 0;
  ChunkCursor cur;
  cur.start(plan);
  for (int i = 0; i < plan.total; ++i) {
    const int st = i % S, k = i / S;
    if (k > 0 && !mbar_wait_sleep(&empty[st], static_cast<uint32_t>((k - 1) & 1), kSleepTries,
                                   kSleepNs)) {
      ok = false;
      break;
    }
    const int n = cur.size(plan);
    const uint32_t bytes = static_cast<uint32_t>(n) * plan.esize;
    mbar_arrive_expect_tx(&full[st], bytes);
    bulk_g2s(ring + st * plan.stage_bytes,
             plan.blk[cur.k].ptr + static_cast<long long>(cur.off) * plan.esize, bytes, &full[st]);
    cur.next(plan, n);
    issued = i + 1;
  }
  for (int i = max(0, issued - S); i < issued; ++i)
    (void)mbar_wait_sleep(&full[i % S], static_cast<uint32_t>((i / S) & 1), kSleepTries, kSleepNs);
  return ok;
}

// Consumer warps.  seg(q, v0, n, data) processes the n elements of row q starting at vocabulary
// index v0, found at `data` in shared memory; every lane of every consumer warp sees the same
// segment sequence (rows in the order the blocks list them).
template <typename Fn>
__device__ bool stream_consume(const StreamPlan& plan, const char* ring, uint64_t* full,
                               uint64_t* empty, Fn seg) {
  const int lane = threadIdx.x & 31;
  const int S = plan.stages;
  ChunkCursor cur;
  cur.start(plan);
  for (int i = 0; i < plan.total; ++i) {
    const int st = i % S, k = i / S;
    const bool got =
        mbar_wait_sleep(&full[st], static_cast<uint32_t>(k & 1), kSleepTries, kSleepNs);
    if (!__all_sync(0xffffffffu, got)) return false;
    const int n = cur.size(plan);
    const char* data = ring + st * plan.stage_bytes;
    int q = cur.q, v = cur.v, done = 0;
    while (done < n) {  // split the chunk at row boundaries
      const int m = min(n - done, plan.V - v);
      seg(q, v, m, data + done * plan.esize);
      done += m;
      v = 0;
      ++q;
    }
    cur.next(plan, n);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  return true;
}

}  // namespace specdec
