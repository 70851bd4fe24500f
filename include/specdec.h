/*
 * specdec.h -- C ABI of the GB300 (sm_103a) hot path of batch speculative decoding.
 *
 * One verification round of batched speculative decoding is:
 *   1. verification of D draft tokens per sequence against the target's scores
 *      (specdec_verify_greedy or specdec_verify_sample), giving an accept length a_b in [0, D]
 *      and one replacement-or-bonus token y_b per row, and
 *   2. realignment of the left-padded batch (specdec_realign): unpad every row, append the
 *      a_b accepted drafts and y_b, re-left-pad to the longest row, rebuild the attention mask and
 *      position IDs, and move every layer's surviving K/V columns, so that rectangular alignment
 *      and position-ID contiguity hold again.
 * For a pool of sequences, specdec_group_by_length forms batches of equal-length rows (which
 * need no realignment) and batches of mixed leftovers, and specdec_pool_gather /
 * specdec_pool_append move a mixed batch between the pool and a padded batch buffer.  The pool's
 * lifecycle (specdec_pool_admit, retirement inside specdec_pool_append, specdec_pool_schedule,
 * and the host allocator of arena columns specdec_arena_*) lets sequences join and leave it.
 *
 * Sources (page title, section):
 *   [IE5]   "Inference Engineering: Part 5/8: When Speculative Decoding Backfires"
 *   [BSDDR] "Batch Speculative Decoding Done Right" (technical summary of arXiv 2510.22876)
 *   [CF]    "Correctness Forensics for Batch Speculative Decoding: Diagnosing the Ragged Tensor
 *           Problem", Abstract
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller.  The library allocates no
 *     device memory and keeps no state between calls (the host arena allocator objects, which
 *     the caller creates and destroys, and the static scratch of specdec_verify_greedy_noalloc,
 *     are the exceptions).  Greedy verification also takes a caller-owned device WORKSPACE (size
 *     from specdec_verify_greedy_workspace, 256-byte aligned) through which its CTAs exchange
 *     per-row results, and the realignment and pool moves may take two caller-owned SCHEDULING
 *     WORDS (specdec_realign_args.schedule) from which their CTAs take work items.  Zero-fill
 *     either once before its first use: every call leaves it all zero again (also when it reports
 *     an out-of-range input through dev_status), so it is reused as is, for any shape it is large
 *     enough for.  Calls that may overlap on the GPU need separate ones (one per stream).
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *     default stream).  The return value reports host-detected problems only: an invalid
 *     argument, an unsupported configuration, or a failed launch.  It does not wait for the GPU.
 *   - Problems that only the GPU can see (a length, token or accept value out of range, a cache
 *     too small for the new width) are reported through `dev_status`, a device int32 that the
 *     caller zeroes beforehand: the kernel writes the first nonzero specdec_status it meets and
 *     then writes no further outputs that depend on the bad value.  Kernels never trap, assert or
 *     spin without bound; every wait has an iteration limit (SPECDEC_ERR_TIMEOUT).
 *   - Integer outputs are bit-exact and deterministic.  Floating-point work is done in fp32 with
 *     fp64 for the few cross-block combinations stated below.
 *   - Beyond the plainest form of each operation (its inputs, outputs, dev_status and stream),
 *     four entry points take more, each for a stated reason: specdec_verify_greedy takes
 *     `workspace` and `workspace_bytes` after out_token (its CTAs merge per-row results through
 *     device memory, and the library allocates none); specdec_verify_sample takes `keep_bounds`
 *     before dev_status (NULL: no top-k / top-p); specdec_realign_args carries `pad_id`,
 *     `copy_engine`, `schedule` (NULL: fixed work shares) and `flags` (0, or
 *     SPECDEC_REALIGN_PDL); specdec_realign_args and specdec_pool_args name the K/V caches by
 *     specdec_kv_view (base pointer, element strides and sizes) rather than by a fixed layout.
 */
#ifndef SPECDEC_H
#define SPECDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPECDEC_VERSION 100  /* 1.0.0 */
#define SPECDEC_MAX_DRAFT 31 /* D <= 31: D+1 rows fit one warp ballot */
#define SPECDEC_GREEDY_SCRATCH_BYTES 73728 /* static scratch of specdec_verify_greedy_noalloc */

typedef enum {
  SPECDEC_OK = 0,
  SPECDEC_ERR_INVALID_ARG = 1, /* host: NULL pointer, negative or inconsistent size, aliasing */
  SPECDEC_ERR_UNSUPPORTED = 2, /* host: valid but outside the library's limits (sizes, alignment) */
  SPECDEC_ERR_CUDA = 3,        /* host: a CUDA launch or attribute call failed */
  SPECDEC_ERR_CAPACITY = 4,    /* device: the new width (+ D columns for the next pass) does not
                                  fit the destination; nothing was moved */
  SPECDEC_ERR_INPUT_RANGE = 5, /* device: a length, accept value, token id or uniform out of
                                  range, or a score row with no comparable value (all NaN) */
  SPECDEC_ERR_TIMEOUT = 6      /* device: a bounded wait on an asynchronous copy ran out */
} specdec_status;

typedef enum { SPECDEC_F32 = 0, SPECDEC_BF16 = 1 } specdec_dtype;

/* Library version (SPECDEC_VERSION of the build). */
int specdec_version(void);

/* Static, human-readable name of a specdec_status value ("unknown status" otherwise). */
const char* specdec_status_string(int status);

/*
 * Self-test of the device-side failure reporting.  The pages have no counterpart: this is a
 * diagnostic of the library, not part of the method.  One thread of one CTA waits, with the same
 * bounded mbarrier wait the streaming kernels use for their bulk copies, on a barrier that nothing
 * completes: at most `polls` polls, each suspending for at most about `sleep_ns` nanoseconds.  It
 * then writes SPECDEC_ERR_TIMEOUT to *dev_status (a device int32; the first nonzero code written
 * stays) and exits.  No copy is issued, so nothing is in flight when it exits and the context
 * stays usable.  Limits: 1 <= polls <= 2^20, sleep_ns <= 10^6 (so the wait ends within about a
 * second); otherwise, or with a NULL dev_status, SPECDEC_ERR_INVALID_ARG.
 */
int specdec_wait_selftest(uint32_t polls, uint32_t sleep_ns, int32_t* dev_status, void* stream);

/*
 * Greedy verification.  [IE5, "Exactness Means Different Things For Greedy And Sampled Output"
 * (greedy: accept while the draft equals the main model's highest-score token, replace the first
 * mismatch with the main model's choice); "Draft Possible Tokens, Then Verify Them Together"
 * (read left to right, discard everything after the first rejection, bonus token after a fully
 * accepted draft); "One Verification Pass Can Commit Several Tokens" (worked example).]
 *
 *   logits     [B][D+1][row_stride] scores of the target (dtype F32 or BF16); row (b, j) holds
 *              the scores of the token after draft j of row b (j = 0: after the last committed
 *              token).  Only the first V elements of each row are read.  Element-aligned.
 *   draft      [B][D] int32 draft tokens d_1..d_D.
 *   accept_len [B] int32 out: a_b = number of leading drafts equal to the target's choice.
 *   out_token  [B] int32 out: y_b = the target's choice at row a_b (the replacement when a_b < D,
 *              the bonus token when a_b == D).  The cycle commits a_b + 1 tokens.
 *   workspace  device buffer of at least specdec_verify_greedy_workspace(B, D) bytes, all zero
 *              (see the conventions above).
 * The target's choice of a row is its maximum score, lowest token index on ties; NaN scores are
 * never chosen (a row of only NaN sets SPECDEC_ERR_INPUT_RANGE).  A draft id outside [0, V) sets
 * SPECDEC_ERR_INPUT_RANGE and counts as a mismatch.
 * Limits: B >= 0, 1 <= D <= 31, 1 <= V, row_stride >= V; a NULL, unaligned or too small
 * workspace is SPECDEC_ERR_INVALID_ARG; more than 2^40 bytes of scores is
 * SPECDEC_ERR_UNSUPPORTED.
 */
int specdec_verify_greedy(const void* logits, int dtype, int B, int D, int V,
                          long long row_stride, const int32_t* draft, int32_t* accept_len,
                          int32_t* out_token, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream);

/* Workspace bytes specdec_verify_greedy needs for B rows of D drafts (0 for an invalid shape):
 * one 64-bit key per score row and one 32-bit counter per batch row, each array 256-byte
 * aligned. */
size_t specdec_verify_greedy_workspace(int B, int D);

/*
 * Greedy verification without a caller workspace.  The pages have no counterpart: this is an
 * interface convenience, not part of the method.  It computes exactly what specdec_verify_greedy
 * computes (same arguments minus the workspace, same results, limits and status codes) for
 * callers that cannot allocate device memory or keep a buffer alive between calls: a host that
 * links this C library alone and has no device allocator of its own, or a plugin that a serving
 * framework hands raw device pointers while keeping every allocation to itself.
 *
 * Scratch: one static device array of SPECDEC_GREEDY_SCRATCH_BYTES per device, inside this
 * library.  It is zero when the library is loaded, and every call leaves it zero again, which is
 * the state the next call needs.  The first call on a device looks up the array's address
 * (cudaGetSymbolAddress, with that device current on the calling thread) and keeps it; make that
 * first call before any stream capture.  Later calls use the device current on the calling thread.
 * A shape whose workspace, specdec_verify_greedy_workspace(B, D), exceeds
 * SPECDEC_GREEDY_SCRATCH_BYTES is SPECDEC_ERR_UNSUPPORTED (for example B = 1024 with D = 7 fits; B = 4096
 * with D = 5 does not).  Calls that may overlap on one device (other streams, other
 * host threads) share the array and race: run them on one stream, or use specdec_verify_greedy
 * with one workspace per stream.  Returns SPECDEC_ERR_CUDA if the address lookup fails.
 */
int specdec_verify_greedy_noalloc(const void* logits, int dtype, int B, int D, int V,
                                  long long row_stride, const int32_t* draft, int32_t* accept_len,
                                  int32_t* out_token, int32_t* dev_status, void* stream);

/*
 * Sampled verification (speculative rejection sampling).  [IE5, "Exactness Means Different
 * Things For Greedy And Sampled Output": accept a draft x with probability min(1, p(x)/q(x)); at
 * a rejection draw the replacement from normalize(max(0, p - q)); both models use the same
 * sampling settings.  "Draft Possible Tokens, Then Verify Them Together": left to right, the
 * first rejection ends the cycle, the bonus comes from the distribution after the full draft.]
 *
 *   target_logits [B][D+1][row_stride] target scores; p_j = softmax(target row j / T).
 *   draft_logits  [B][D][row_stride] draft-model scores; q_j = softmax(draft row j / T).
 *   draft         [B][D] draft tokens (drawn from q by the draft model).
 *   uniforms      [B][D+1] float32 in [0, 1): u[b][j] (j < D) decides draft j+1: accepted iff
 *                 u < p_j(d)/q_j(d); u[b][D] drives the replacement / bonus draw.
 *   accept_len, out_token  as for greedy verification.
 *   residual_out  [B][V] float32 out, may be NULL: the normalised distribution y_b was drawn from
 *                 (normalize(max(0, p_a - q_a)) after a rejection at a = a_b < D, p_D when all
 *                 drafts were accepted).
 *   keep_bounds   [B][2D+1] specdec_keep_bound from specdec_sampling_filter (rows 0..D the
 *                 target's, D+1..2D the draft's), or NULL for no top-k / top-p: p_j and q_j are
 *                 then the softmax restricted to each row's kept tokens and renormalised.
 * A draft the target cannot emit (outside p's kept set, or a score of -inf: p(d) = 0) is rejected
 * whatever q(d) is; one with q(d) = 0 < p(d) is accepted.
 * The draw is an inverse CDF over ascending token ids: the first k whose running sum exceeds
 * u[b][D] * (total).  If max(0, p - q) is zero everywhere the draw uses p instead.
 * Precision: exponentials and per-element probabilities in fp32; the acceptance ratio p(d)/q(d)
 * and the cross-block normalisers in fp64.  Limits: B >= 0, 1 <= D <= 31, 1 <= V,
 * row_stride >= V, temperature > 0 and finite.  Uniforms outside [0, 1) set
 * SPECDEC_ERR_INPUT_RANGE.
 */
int specdec_verify_sample(const void* target_logits, const void* draft_logits, int dtype, int B,
                          int D, int V, long long row_stride, float temperature,
                          const int32_t* draft, const float* uniforms, int32_t* accept_len,
                          int32_t* out_token, float* residual_out, const void* keep_bounds,
                          int32_t* dev_status, void* stream);

/*
 * Sampled verification with the uniforms drawn in-kernel (the fused round needs no uniform
 * buffer).  [Counter-based generator: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 * Easy as 1, 2, 3" (SC11), Philox4x32-10.]  As specdec_verify_sample, with u[b][j] (j = 0..D)
 * = (x >> 8) * 2^-24, where x is word j mod 4 of Philox4x32-10 at counter
 * (j div 4, b, offset mod 2^32, offset div 2^32) and key (seed mod 2^32, seed div 2^32): 24-bit
 * uniforms in [0, 1), the same in fp32 and fp64.  The caller advances `offset` every round (any
 * (seed, offset) pair gives an independent stream of B * 8 blocks).
 */
int specdec_verify_sample_philox(const void* target_logits, const void* draft_logits, int dtype,
                                 int B, int D, int V, long long row_stride, float temperature,
                                 const int32_t* draft, uint64_t seed, uint64_t offset,
                                 int32_t* accept_len, int32_t* out_token, float* residual_out,
                                 const void* keep_bounds, int32_t* dev_status, void* stream);

/*
 * The uniforms u[B][D+1] (fp32, row-major, device memory) that specdec_verify_sample_philox draws
 * for (seed, offset): to log or replay a round through specdec_verify_sample.  Limits: B >= 0,
 * 1 <= D <= 31.
 */
int specdec_philox_uniforms(uint64_t seed, uint64_t offset, int B, int D, float* out,
                            void* stream);

/*
 * The kept set of one score row under the sampling settings, as its last token in the settings'
 * order.  A token with score x at index v is kept iff key(x) > key, or key(x) == key and
 * v <= index, where key(x) is the order-preserving code of the score as a float: its IEEE bits
 * with -0 taken as +0, the sign bit set for x >= 0 and all bits inverted for x < 0.  `index` is
 * the index of the last kept token of score `key`, or INT32_MAX when every token with that score
 * is kept (bf16 rows; fp32 rows always give the token's index).
 */
typedef struct {
  uint32_t key;
  int32_t index;
} specdec_keep_bound;

/*
 * Top-k / top-p keep bounds of every score row, for specdec_verify_sample.  [IE5, "Draft Possible
 * Tokens, Then Verify Them Together": sampling settings "such as temperature and top-p";
 * "Exactness Means Different Things For Greedy And Sampled Output": both models use the same
 * sampling settings.]
 *
 * Reading: a row's tokens are ordered by score, highest first, ties by lower token index.
 * top_k (1 <= top_k < V; 0 or >= V is off) keeps the first top_k tokens; top_p (0 < top_p < 1;
 * 1 is off) then keeps, in the same order, every token whose preceding probability mass (softmax
 * at T within the kept set) is below top_p, so the token that reaches top_p is kept.
 *   target_logits, draft_logits, dtype, B, D, V, row_stride, temperature  as for
 *                 specdec_verify_sample.
 *   keep_bounds   [B][2D+1] specdec_keep_bound out (8-byte aligned device memory).
 * Top-k is exact.  Top-p sums the masses 2^(x*log2(e)/T - o) in 64-bit fixed point (2^-44 of the
 * row's largest mass, from an exp2 with relative error below 2^-21): its cut can differ from an
 * exact one only where top_p lies within about 1e-6 of a cumulative mass of the order.  Rows with
 * NaN or +inf scores keep every token (verification reports them).  Limits: as for
 * specdec_verify_sample; top_k >= 0, 0 < top_p <= 1.
 */
int specdec_sampling_filter(const void* target_logits, const void* draft_logits, int dtype, int B,
                            int D, int V, long long row_stride, float temperature, int top_k,
                            float top_p, void* keep_bounds, int32_t* dev_status, void* stream);

/*
 * A view of a K/V cache in device memory.  Element (layer l, k-or-v kv, row r, head h,
 * column c, e) lives at  base + l*stride_layer + kv*stride_kv + r*stride_row + h*stride_head
 *                        + c*head_dim + e          (strides in elements).
 * One column of one head (head_dim elements) is contiguous, and the columns of one
 * (l, kv, r, h) are contiguous.  The natural layout [L][2][rows][H][cap_cols][head_dim] has
 * stride_head = cap_cols*head_dim, stride_row = H*stride_head, stride_kv = rows*stride_row,
 * stride_layer = 2*stride_kv.  `base` and head_dim*element size must be multiples of 16 bytes,
 * and so must every stride times the element size.
 */
typedef struct {
  void* base;
  long long stride_layer, stride_kv, stride_row, stride_head;
  int dtype; /* specdec_dtype of the elements (only the size matters: values are moved) */
  int layers, rows, heads, head_dim, cap_cols;
} specdec_kv_view;

/*
 * EQSPEC realignment (unpad, append, repad), out of place.  [BSDDR section 2.2 (unpad each row,
 * append accepted and bonus tokens, left-pad to the longest row, recompute position IDs, shift
 * the KV cache); section 2.1 (rectangular alignment: pad + content equal across the batch;
 * position-ID contiguity: IDs from 0, contiguous over the mask's content); CF Abstract (the
 * ragged tensor problem under contiguous layouts); IE5 "Acceptance changes across the workload"
 * (keep committed K/V, discard speculative entries after the first rejection).]
 *
 * State before (width W = *width, N_b = n_committed[b] in [1, W]):
 *   ids_src row b holds the N_b committed tokens at columns [W - N_b, W); src holds K/V for
 *   columns [W - N_b, W - 1) (all committed tokens but the last, "pending" one) and for the D+1
 *   columns [W - 1, W + D) the verification pass wrote for [pending, d_1 .. d_D].
 * State after (N'_b = N_b + a_b + 1, W' = max_b N'_b):
 *   dst columns [W' - N'_b, W' - 1) of every (layer, kv, head) of row b = src columns
 *   [W - N_b, W + a_b) (the rejected drafts' columns [W + a_b, W + D) are not copied);
 *   ids_dst row b = pad_id at [0, W' - N'_b), then the old committed tokens, d_1..d_{a_b} and
 *   y_b ending at column W' - 1, pad_id again from W' on; mask_dst = 1 exactly on
 *   [W' - N'_b, W'); pos_dst = 0, 1, .., N'_b - 1 there and 0 elsewhere; n_committed_dst = N';
 *   *width_dst = W'.  dst pad columns are left as they were (unspecified).
 * All per-row values are read on the device: no host synchronisation is needed between
 * verification and realignment, and the call can be captured in a CUDA graph.
 * Device-detected errors (no output is written): N_b outside [1, W] or a_b outside [0, D]
 * (SPECDEC_ERR_INPUT_RANGE); W + D > src.cap_cols (SPECDEC_ERR_INPUT_RANGE); W' + D > dst.cap_cols
 * (SPECDEC_ERR_CAPACITY: the next verification pass could not be written).
 * src and dst must be distinct, non-overlapping buffers of equal geometry except cap_cols; the
 * metadata outputs must not alias their inputs.  Limits: 0 <= B <= 1024 (B == src.rows ==
 * dst.rows), 1 <= D <= 31.
 */
typedef struct {
  specdec_kv_view src, dst;
  int B, D;
  int32_t pad_id;
  int copy_engine;                /* 0: TMA bulk copies (default); 1: 16-byte vector loads */
  const int32_t* n_committed;     /* [B]  N_b */
  const int32_t* width;           /* [1]  W */
  const int32_t* accept_len;      /* [B]  a_b */
  const int32_t* out_token;       /* [B]  y_b */
  const int32_t* draft;           /* [B][D] */
  const int32_t* ids_src;         /* [B][src.cap_cols] */
  int32_t* ids_dst;               /* [B][dst.cap_cols] */
  uint8_t* mask_dst;              /* [B][dst.cap_cols] */
  int32_t* pos_dst;               /* [B][dst.cap_cols] */
  int32_t* n_committed_dst;       /* [B]  N'_b */
  int32_t* width_dst;             /* [1]  W' */
  int32_t* dev_status;            /* [1] */
  int flags;                      /* 0, or SPECDEC_REALIGN_PDL */
  uint32_t* schedule;             /* NULL, or [2] caller-owned scheduling words (below) */
} specdec_realign_args;

/*
 * schedule (optional, device memory, not in the pages: a launch detail).  NULL: every CTA of the
 * launch moves one fixed, equal, contiguous share of the tiles.  Non-NULL: two uint32 words that
 * are zero before the first call; the CTAs take work items (a few tiles; whole runs in place)
 * from a counter in schedule[0] as they free up, so SMs that stream faster take more, and the
 * last CTA to finish sets both words back to zero -- one pair serves every later call, in a CUDA
 * graph too.  Calls that may run at the same time (other streams) need their own pair; calls in
 * order on one stream may share one.  Results are the same either way.  Ignored with
 * copy_engine 1.  A pointer that is not 4-byte aligned is SPECDEC_ERR_INVALID_ARG.
 */

/*
 * SPECDEC_REALIGN_PDL: launch the realignment with programmatic stream serialization, so that it
 * may be launched while the kernel ahead of it on the stream (normally the verification, which
 * signals its dependents as it starts) is still running; the realignment waits for that kernel to
 * complete, and for its writes to be visible, before it reads or writes anything.  The result is
 * the same; the launch latency between the two kernels is hidden.
 */
#define SPECDEC_REALIGN_PDL 1

int specdec_realign(const specdec_realign_args* args, void* stream);

/*
 * EQSPEC realignment with the K/V cache moved in place: one cache buffer instead of two, which
 * halves the cache memory.  [BSDDR section 2.2, "shift the KV cache", as an in-place shift.]
 * Same arguments, results and errors as specdec_realign, except:
 *   - args->dst must be the same view as args->src (same base, strides, dtype and cap_cols);
 *     the metadata (ids/mask/pos, lengths, width) is still written to separate outputs;
 *   - after the call the buffer's columns [W' - N'_b, W' - 1) of row b hold the surviving K/V as
 *     above; every other column keeps whatever it held before (the old values of columns that
 *     were not overwritten);
 *   - rows whose columns do not move (W' - N'_b == W - N_b) are not copied at all.
 * Each (layer, kv, row, head) run is moved by one CTA in the direction that never overwrites a
 * source byte before it has been read.
 */
int specdec_realign_inplace(const specdec_realign_args* args, void* stream);

/*
 * EXSPEC grouping of a SequencePool by length.  [BSDDR section 2.3: keep a pool of active
 * sequences; group same-length sequences so they need no realignment; only mixed-length ones are
 * realigned.]
 *
 *   lengths       [N] int32 in [0, max_len]: committed length of each pool row.
 *   perm          [N] int32 out: pool rows in batch order.
 *   batch_offsets [N+1] int32 out: batch k is perm[batch_offsets[k] .. batch_offsets[k+1]).
 *   batch_uniform [N] uint8 out: 1 for a uniform batch (batch_size rows of one length).
 *   num_batches, num_uniform  [1] int32 out.
 * Rule: a stable counting sort by length; rows of one length, in index order, fill whole batches
 * of batch_size first (uniform batches, ascending length); the remaining rows of every length,
 * in (length, index) order, are cut into mixed batches of batch_size rows (the last may be
 * shorter).  Uniform batches come first.  Entries past num_batches are not written.
 * Limits: 0 <= N <= 4096, batch_size >= 1, 0 <= max_len <= 16383.  A length outside
 * [0, max_len] sets SPECDEC_ERR_INPUT_RANGE (no output written).
 */
int specdec_group_by_length(const int32_t* lengths, int N, int batch_size, int max_len,
                            int32_t* perm, int32_t* batch_offsets, uint8_t* batch_uniform,
                            int32_t* num_batches, int32_t* num_uniform, int32_t* dev_status,
                            void* stream);

/*
 * Pool <-> padded-batch moves for EXSPEC's mixed leftovers.  [BSDDR section 2.3 (only
 * mixed-length sequences are realigned) with the unpad-append-repad of section 2.2.]
 *
 * The pool is unpadded at rest: slot s owns arena columns [slot_col[s], slot_col[s] +
 * slot_cap[s]) of row 0 of `arena`, and holds K/V for its first N_s - 1 tokens (all but the
 * pending one) at the start of that range; pool_ids[s][0 .. N_s) are its tokens.
 *
 * specdec_pool_gather (repad): for the k = n_rows slots rows[0..k) with W = max N_s:
 *   scratch row i columns [W - N_s, W - 1) = the slot's K/V columns [0, N_s - 1);
 *   scratch_ids / scratch_mask / scratch_pos row i = the left-padded batch of width W (as
 *   specdec_realign writes them); batch_len[i] = N_s; *width = W.
 *   in_place != 0 (a uniform batch, all N_s equal): no K/V or metadata is moved; only batch_len
 *   and *width are written (the verification pass can work on the slots directly).
 *   Errors: N_s < 1, N_s > slot_cap[s], or a slot range outside the arena (INPUT_RANGE);
 *   W + D > scratch.cap_cols, or N_s + D > slot_cap[s] (CAPACITY).
 * specdec_pool_append (append): after the verification pass wrote columns [W - 1, W + D) of
 *   every scratch row (or, in place, slot columns [N_s - 1, N_s + D)) and verification gave
 *   accept_len[i], out_token[i] in batch-row order:
 *   slot columns [N_s - 1, N_s + a_i) = scratch row i columns [W - 1, W + a_i) (not copied in
 *   place); pool_ids[s][N_s .. N_s + a_i) = d_1..d_{a_i}, pool_ids[s][N_s + a_i] = y_i;
 *   slot_len[s] = N_s + a_i + 1, with N_s = batch_len[i] as the gather recorded it.
 *   by_slot != 0: accept_len, out_token and draft are pool-wide arrays indexed by slot s =
 *   rows[i] (e.g. one verification call over the whole pool) instead of by batch row i.
 *   Errors: a_i outside [0, D], a recorded width/length out of range (INPUT_RANGE; nothing
 *   written).
 * Limits: 1 <= n_rows <= min(1024, scratch.rows), 1 <= D <= 31, arena.rows == 1, arena and
 * scratch of equal layers, heads, head_dim and element size.  Rows must name distinct slots.
 */
typedef struct {
  specdec_kv_view arena;        /* the pool's K/V (rows == 1) */
  specdec_kv_view scratch;      /* padded batch buffer [L][2][R][H][Sc][hd] */
  int n_rows, D;
  int32_t pad_id;
  int in_place;                 /* uniform batch: verification works on the slots directly */
  const int32_t* rows;          /* [n_rows] slot of each batch row */
  const int32_t* slot_col;      /* [S] first arena column of each slot */
  const int32_t* slot_cap;      /* [S] arena columns owned by each slot */
  int32_t* slot_len;            /* [S] N_s (read by gather; advanced by append) */
  int32_t* pool_ids;            /* [S][ids_cap] tokens of each slot */
  int ids_cap;
  int32_t* batch_len;           /* [n_rows] N_s recorded by gather, read by append */
  int32_t* width;               /* [1] W written by gather, read by append */
  int32_t* scratch_ids;         /* [R][Sc] written by gather (may be NULL when in_place) */
  uint8_t* scratch_mask;        /* [R][Sc] */
  int32_t* scratch_pos;         /* [R][Sc] */
  const int32_t* accept_len;    /* [n_rows] (or [S] with by_slot) append only */
  const int32_t* out_token;     /* [n_rows] (or [S] with by_slot) append only */
  const int32_t* draft;         /* [n_rows][D] (or [S][D] with by_slot) append only */
  int by_slot;                  /* append: index the three arrays above by slot */
  int32_t* dev_status;          /* [1] */
  /* Retirement (append only; slot_state NULL: none).  See "SequencePool lifecycle" below. */
  uint8_t* slot_state;          /* [S] specdec_slot_state of each slot */
  const int32_t* slot_limit;    /* [S] length limit of each slot */
  int32_t eos_id;               /* end-of-sequence token id (< 0: length limit only) */
  uint32_t* schedule;           /* NULL, or [2] scheduling words, as in specdec_realign_args */
} specdec_pool_args;

int specdec_pool_gather(const specdec_pool_args* args, void* stream);
int specdec_pool_append(const specdec_pool_args* args, void* stream);

/*
 * SequencePool lifecycle.  [BSDDR section 2.3: the pool holds the *active* sequences; those of one
 * length are batched without realignment and only mixed-length ones are realigned.]
 *
 * Each slot s has a state byte slot_state[s]:
 *     FREE --specdec_pool_admit--> ACTIVE --retirement in specdec_pool_append--> FINISHED_*
 *     FINISHED_* --specdec_pool_schedule (reported once)--> FREE
 * Only ACTIVE slots are scheduled.  A finished slot keeps its tokens (pool_ids[s][0 .. slot_len[s]))
 * and K/V until it is admitted again.
 *
 * Retirement (specdec_pool_append with slot_state != NULL and slot_limit != NULL): after the
 *   append of batch row i (slot s, old length N = batch_len[i], new length N + a_i + 1), the
 *   committed positions q = N .. N + a_i are scanned in order; at the first q whose token is
 *   eos_id the slot becomes FINISHED_EOS, else at the first q with q + 1 == slot_limit[s] it
 *   becomes FINISHED_LENGTH; either way slot_len[s] = q + 1 (later tokens of the round are
 *   dropped).  A row whose slot is not ACTIVE sets SPECDEC_ERR_INPUT_RANGE and its length, ids
 *   and state are left alone (its K/V columns past N - 1 may still be written: name ACTIVE slots).
 *
 * specdec_pool_schedule: groups the ACTIVE slots by length window and lists the finished ones.
 *   Rule: walk the ACTIVE slots in (slot_len, slot) order; where the next batch_size of them span
 *   at most `window` in length they form a windowed batch and the walk moves past them, else the
 *   slot is a leftover and the walk moves on by one.  Windowed batches come first, then the
 *   leftovers, in (length, slot) order, cut into mixed batches of batch_size (the last may be
 *   shorter).  window = 0 is the exact-length rule of specdec_group_by_length (over the ACTIVE
 *   slots).  batch_uniform[k] = 1 only for a windowed batch of one length.
 *   Outputs: perm[0 .. num_active) slots in batch order; batch k is perm[batch_offsets[k] ..
 *   batch_offsets[k+1]); finished[0 .. num_finished) the FINISHED slots in slot order with their
 *   state in finished_reason, and those slots are set FREE; counts = {num_batches, num_windowed,
 *   num_active, num_finished}.  Entries past the counts are not written.
 *   Limits: 0 <= S <= 4096, 1 <= batch_size <= 4096, window >= 0; ACTIVE lengths in [1, 2^20).
 *   A state above FINISHED_LENGTH or an ACTIVE length out of range sets SPECDEC_ERR_INPUT_RANGE
 *   and nothing is written.  One CTA; latency-bound.
 */
typedef enum {
  SPECDEC_SLOT_FREE = 0,
  SPECDEC_SLOT_ACTIVE = 1,
  SPECDEC_SLOT_FINISHED_EOS = 2,
  SPECDEC_SLOT_FINISHED_LENGTH = 3
} specdec_slot_state;

typedef struct {
  int S, batch_size, window;
  uint8_t* slot_state;          /* [S] read; FINISHED slots set FREE */
  const int32_t* slot_len;      /* [S] */
  int32_t* perm;                /* [S] out */
  int32_t* batch_offsets;       /* [S+1] out */
  uint8_t* batch_uniform;       /* [S] out */
  int32_t* finished;            /* [S] out */
  uint8_t* finished_reason;     /* [S] out */
  int32_t* counts;              /* [4] out */
  int32_t* dev_status;          /* [1] */
} specdec_schedule_args;

int specdec_pool_schedule(const specdec_schedule_args* args, void* stream);

/*
 * specdec_pool_admit: put n prompts into FREE slots.  Entry i: slot slots[i] gets arena columns
 *   [cols[i], cols[i] + caps[i]), length limit limits[i], slot_len = its prompt length, pool_ids
 *   row = the prompt (prompt_ids[prompt_off[i] .. prompt_off[i+1])), and becomes ACTIVE.  The
 *   prompt's K/V is the caller's (the target's prefill writes it).
 *   Every entry is checked first: slot in [0, S), FREE and named once; prompt length >= 1 and
 *   below its limit; arena range inside [0, arena_cols) (else SPECDEC_ERR_INPUT_RANGE);
 *   limit + D - 1 <= caps[i] and limit + D <= ids_cap, so that every round until the limit has
 *   room (else SPECDEC_ERR_CAPACITY).  On any error nothing is written.  The writes are also
 *   skipped when dev_status is nonzero on entry.  Arena ranges of different slots must not
 *   overlap (not checked: the arena allocator below hands out disjoint runs); the prompt buffer
 *   must hold prompt_off[n] tokens.
 *   Limits: 0 <= n <= 1024, 0 <= S <= 4096, 1 <= D <= 31.  Two launches (check, then write).
 */
typedef struct {
  int n, S, D, ids_cap;
  int64_t arena_cols;
  const int32_t* slots;         /* [n] */
  const int32_t* cols;          /* [n] first arena column */
  const int32_t* caps;          /* [n] arena columns */
  const int32_t* limits;        /* [n] length limit */
  const int32_t* prompt_ids;    /* [prompt_off[n]] */
  const int32_t* prompt_off;    /* [n+1] */
  uint8_t* slot_state;          /* [S] */
  int32_t* slot_col;            /* [S] */
  int32_t* slot_cap;            /* [S] */
  int32_t* slot_len;            /* [S] */
  int32_t* slot_limit;          /* [S] */
  int32_t* pool_ids;            /* [S][ids_cap] */
  int32_t* dev_status;          /* [1] */
} specdec_admit_args;

int specdec_pool_admit(const specdec_admit_args* args, void* stream);

/*
 * Arena allocator (HOST only, thread safe).  Columns [0, cols) of the pool's K/V arena are handed
 * out first fit: specdec_arena_alloc returns the lowest column c with [c, c + ncols) free
 * (SPECDEC_ERR_CAPACITY if there is none); specdec_arena_free takes the start of an allocation
 * (SPECDEC_ERR_INVALID_ARG otherwise) and merges the run with free neighbours.  The arena object
 * is created and destroyed by the caller; no GPU is touched.
 */
typedef struct specdec_arena specdec_arena;
int specdec_arena_create(int64_t cols, specdec_arena** out);
void specdec_arena_destroy(specdec_arena* arena);
int specdec_arena_alloc(specdec_arena* arena, int64_t ncols, int64_t* col);
int specdec_arena_free(specdec_arena* arena, int64_t col);
int specdec_arena_stats(specdec_arena* arena, int64_t* free_cols, int64_t* largest_free,
                        int64_t* allocations);

#ifdef __cplusplus
}
#endif
#endif /* SPECDEC_H */
