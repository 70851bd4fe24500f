"""CPU oracle for the per-round hot path of batch speculative decoding.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` may import this module.  The product path (the CUDA library and its
Python binding) never imports, calls or links it, and it shares no code with that path: no helper,
table or constant.  Inputs come from the seeded generators in
``speculative_decoding_specdec_gb300.synth`` (which hold none of the method's arithmetic) or from
hand-written fixtures.

Everything here is plain numpy in float64, written for a reader to check against the pages by eye.
Sources, cited by page title and section:

* [IE5]   "Inference Engineering: Part 5/8: When Speculative Decoding Backfires"
          - "Draft Possible Tokens, Then Verify Them Together"      (left-to-right acceptance, bonus)
          - "One Verification Pass Can Commit Several Tokens"       (greedy worked example)
          - "Exactness Means Different Things For Greedy And Sampled Output"
                                                                     (min(1, p/q), normalize(max(0, p-q)))
          - "Acceptance changes across the workload"                (discard after first rejection;
                                                                     speculative KV commit/discard)
* [BSDDR] "Batch Speculative Decoding Done Right" (technical summary of arXiv 2510.22876)
          - section 2.1 (synchronisation invariants: rectangular alignment, position-ID contiguity)
          - section 2.2 (EQSPEC unpad-append-repad)
          - section 2.3 (EXSPEC SequencePool, grouping of same-length sequences)
* [CF]    "Correctness Forensics for Batch Speculative Decoding: Diagnosing the Ragged Tensor
          Problem", Abstract (ragged tensor problem, contiguous-layout realignment).

Readings where the pages leave a step open (the pages are silent or ambiguous on each):

* The target produces D+1 score rows per sequence; row j scores the token after the j-th draft
  (row 0 after the last committed token).  The bonus needs the distribution "after the complete
  draft" [IE5, Draft Possible Tokens], which is row D.
* Greedy ties go to the lowest token index.  The pages are silent.
* A draft x is accepted iff u < p(x)/q(x) with u uniform in [0, 1); this is the min(1, p/q) rule
  with the min implicit.  u == p/q rejects.
* Temperature T divides the scores of both models ("same sampling settings" [IE5, Exactness]).
* Top-k / top-p, the other sampling settings the pages name ("temperature and top-p" [IE5, Draft
  Possible Tokens]), apply to both models' rows alike.  A row's tokens are ordered by score,
  highest first, ties by lower token index.  Top-k (1 <= k < V; otherwise off) keeps the first k.
  Top-p (0 < top_p < 1; 1 is off) then keeps, in the same order, every token whose preceding
  probability mass within the kept set (renormalised) is below top_p, so the token that reaches
  top_p is kept.  p and q are the softmax at T restricted to their kept sets and renormalised;
  acceptance, residual and bonus use them as they are.
* The replacement or bonus token is an inverse-CDF draw with the row's last uniform u[b][D], over
  token ids in ascending order, first k whose running sum exceeds u * (total).  If the residual
  max(0, p - q) is all zero the draw falls back to p.
* K/V state model: at round start row b holds N_b committed tokens right-aligned in width W; the
  cache holds K/V for all of them but the last (the "pending" token, not yet run through the
  target).  The verification pass writes K/V for [pending, d_1..d_D] at columns [W-1, W+D).
  After acceptance a_b the surviving K/V columns are [W-N_b, W+a_b); the new pending token is the
  replacement/bonus y_b.  The new width is W' = max_b (N_b + a_b + 1) (minimal padding).
* Pad token ids are a caller-chosen ``pad_id``; pad position IDs are 0; pad K/V columns of the
  destination are unspecified (left as they were).
* Length grouping: within one length, rows in index order fill whole batches of ``bs`` first; the
  remaining rows of every length, in (length, index) order, are chunked into mixed batches.
  Uniform batches come first (ascending length), then mixed batches.
* Length-window grouping (window w >= 0): walk the rows in (length, index) order; where the next
  ``bs`` rows span at most w in length they form a windowed batch, otherwise the row becomes a
  leftover.  w = 0 is the exact-length rule above.  Windowed batches come first, then the
  leftovers in (length, index) order cut into mixed batches.  Only a windowed batch of one length
  is flagged uniform (verified in place).
* In-kernel uniforms (the fused round): u[b][j] for batch row b and j = 0..D is word j mod 4 of
  Philox4x32-10 [Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
  SC11] at counter (j div 4, b, offset mod 2^32, offset div 2^32) and key (seed mod 2^32,
  seed div 2^32), as (x >> 8) * 2^-24 (24 bits: exact in fp32 and fp64, in [0, 1)).  The caller
  advances ``offset`` per round.
* SequencePool lifecycle: a slot is FREE, ACTIVE, or FINISHED (by end-of-sequence token or by its
  length limit).  Only ACTIVE slots are grouped ("a pool of active sequences").  A sequence
  finishes at the first newly committed position q with token == eos_id or q + 1 == its length
  limit (the end-of-sequence token wins at the same position); its length becomes q + 1 and the
  later tokens of that round are dropped.  A schedule reports each FINISHED slot once and frees
  it.  Admission puts a prompt (N >= 1 tokens, N < limit) into a FREE slot with arena range
  [col, col + cap), where limit + D - 1 <= cap and limit + D <= ids_cap, so that every round of
  an unfinished sequence has room.  Arena ranges are given first fit: the lowest column where
  enough consecutive columns are free.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "OracleError",
    "greedy_choice",
    "verify_greedy",
    "softmax",
    "sampling_keep",
    "filtered_softmax",
    "top_p_margin",
    "verify_sample",
    "realign_plan",
    "realign",
    "check_invariants",
    "group_by_length",
    "pool_gather",
    "pool_append",
    "FREE", "ACTIVE", "FINISHED_EOS", "FINISHED_LENGTH",
    "group_by_window",
    "pool_schedule",
    "retire",
    "pool_admit",
    "FirstFitArena",
    "philox",
    "philox_uniforms",
]


class OracleError(ValueError):
    """Raised for inputs the method does not define (the GPU path reports these as a status)."""


# --------------------------------------------------------------------------------------------
# Greedy verification  [IE5, "Exactness Means Different Things..." (greedy paragraph);
#                       "Draft Possible Tokens, Then Verify Them Together"]
# --------------------------------------------------------------------------------------------

def greedy_choice(scores) -> int:
    """The target's greedy choice for one score row: the highest score, lowest index on ties.

    Greedy decoding "picks the token with the highest score" [IE5, opening section].  np.argmax
    returns the first index of the maximum, which is the lowest-index tie rule.
    """
    row = np.asarray(scores, dtype=np.float64)
    if np.isnan(row).any():
        raise OracleError("NaN score")
    return int(np.argmax(row))


def verify_greedy(logits, draft):
    """Greedy verification of a batch.

    logits: [B, D+1, V] target scores; row j scores the token after draft j (row 0: after the
            last committed token).
    draft:  [B, D] draft token ids d_1..d_D.
    Returns (accept_len[B], out_token[B]) as int32 arrays:
      a_b = number of leading drafts equal to the target's choice (first mismatch stops the scan;
            every later draft is discarded);
      y_b = the target's choice at row a_b: the replacement for the rejected draft when a_b < D,
            the bonus token when a_b == D.
    """
    logits = np.asarray(logits, dtype=np.float64)
    draft = np.asarray(draft)
    B, Dp1, V = logits.shape
    D = Dp1 - 1
    if draft.shape != (B, D):
        raise OracleError("draft shape")
    if ((draft < 0) | (draft >= V)).any():
        raise OracleError("draft token out of range")
    accept_len = np.zeros(B, dtype=np.int32)
    out_token = np.zeros(B, dtype=np.int32)
    for b in range(B):
        choices = [greedy_choice(logits[b, j]) for j in range(D + 1)]
        a = D
        for j in range(D):               # read left to right, stop at the first rejection
            if choices[j] != int(draft[b, j]):
                a = j
                break
        accept_len[b] = a
        out_token[b] = choices[a]        # replacement (a < D) or bonus (a == D)
    return accept_len, out_token


# --------------------------------------------------------------------------------------------
# Sampled verification  [IE5, "Exactness Means Different Things For Greedy And Sampled Output"]
# --------------------------------------------------------------------------------------------

def softmax(scores, temperature: float):
    """Probabilities of one score row at temperature T, in float64."""
    x = np.asarray(scores, dtype=np.float64) / float(temperature)
    e = np.exp(x - x.max())
    return e / e.sum()


def _sort_order(z):
    """Token order of the sampling settings: score descending, lower index first on ties."""
    return np.lexsort((np.arange(len(z)), -z))


def sampling_keep(scores, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """Boolean mask of the tokens one score row keeps under top-k and top-p (module readings)."""
    z = np.asarray(scores, dtype=np.float64)
    V = len(z)
    if not 0.0 < top_p <= 1.0:
        raise OracleError("top_p")
    order = _sort_order(z)
    k = V if (top_k <= 0 or top_k >= V) else int(top_k)
    kept = order[:k]
    if top_p < 1.0:
        p = softmax(z[kept], temperature)              # renormalised over the top-k set
        before = np.concatenate(([0.0], np.cumsum(p)[:-1]))
        kept = kept[before < top_p]
    keep = np.zeros(V, dtype=bool)
    keep[kept] = True
    return keep


def filtered_softmax(scores, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """Softmax at T restricted to the kept tokens and renormalised (plain softmax when both
    settings are off)."""
    z = np.asarray(scores, dtype=np.float64)
    if (top_k <= 0 or top_k >= len(z)) and top_p >= 1.0:
        return softmax(z, temperature)
    p = softmax(z, temperature) * sampling_keep(z, temperature, top_k, top_p)
    return p / p.sum()


def top_p_margin(scores, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """How far top_p lies from the nearest cumulative mass at which the top-p cut would move
    (the preceding mass of the last kept and of the first dropped token); inf when top-p is off.
    A top-p cut computed in lower precision can differ from this oracle's only where this margin
    is below that precision."""
    z = np.asarray(scores, dtype=np.float64)
    if top_p >= 1.0:
        return np.inf
    order = _sort_order(z)
    V = len(z)
    k = V if (top_k <= 0 or top_k >= V) else int(top_k)
    p = softmax(z[order[:k]], temperature)
    before = np.concatenate(([0.0], np.cumsum(p)[:-1]))
    return float(np.min(np.abs(before - top_p)))


def _inverse_cdf(weights, u: float):
    """First k (ascending token id) whose running sum exceeds u * total; the running sum is
    sequential.  If rounding leaves no such k, the last k with a nonzero weight."""
    cdf = np.cumsum(weights)
    total = cdf[-1]
    t = u * total
    k = int(np.searchsorted(cdf, t, side="right"))
    if k >= len(weights):
        k = int(np.nonzero(weights > 0)[0][-1])
    lo = cdf[k - 1] if k > 0 else 0.0
    return k, t, total, lo, cdf[k]


def verify_sample(target_logits, draft_logits, draft, uniforms, temperature: float,
                  top_k: int = 0, top_p: float = 1.0):
    """Speculative rejection sampling over a batch.

    target_logits: [B, D+1, V] scores of the main model (p after softmax at T).
    draft_logits:  [B, D, V]   scores of the draft model (q after softmax at T).
    draft:         [B, D]      the draft tokens (drawn from q by the draft model).
    uniforms:      [B, D+1]    u[b][j], j < D decide the accept tests; u[b][D] drives the
                               replacement/bonus draw.
    For j = 0..D-1 (left to right): accept d_{j+1} iff u[b][j] < p_j(d)/q_j(d), i.e. with
    probability min(1, p/q).  At the first rejection j*: draw y from normalize(max(0, p_j* - q_j*)).
    If every draft is accepted: draw the bonus y from p_D.
    With top_k / top_p set, p and q are the filtered, renormalised distributions of every row
    (filtered_softmax); a draft the target cannot emit (p(d) = 0) is rejected whatever q(d) is,
    and one outside q's kept set only (q(d) = 0 < p(d)) is accepted.

    Returns (accept_len[B], out_token[B], residual[B, V], trace) where residual[b] is the
    normalised distribution y_b was drawn from, and trace holds float64 diagnostics for the
    parity tolerance: ratio[B, D] (p/q of each evaluated test, NaN where not evaluated), and for
    the draw t = u*R, R, and the running sums just below and at y.
    """
    tl = np.asarray(target_logits, dtype=np.float64)
    dl = np.asarray(draft_logits, dtype=np.float64)
    draft = np.asarray(draft)
    u = np.asarray(uniforms, dtype=np.float64)
    B, Dp1, V = tl.shape
    D = Dp1 - 1
    if dl.shape != (B, D, V) or draft.shape != (B, D) or u.shape != (B, D + 1):
        raise OracleError("shape")
    if not temperature > 0:
        raise OracleError("temperature")
    if ((draft < 0) | (draft >= V)).any():
        raise OracleError("draft token out of range")
    accept_len = np.zeros(B, dtype=np.int32)
    out_token = np.zeros(B, dtype=np.int32)
    residual = np.zeros((B, V), dtype=np.float64)
    ratio = np.full((B, D), np.nan)
    t_draw = np.zeros(B)
    r_total = np.zeros(B)
    cdf_lo = np.zeros(B)
    cdf_hi = np.zeros(B)
    for b in range(B):
        a = D
        for j in range(D):
            p = filtered_softmax(tl[b, j], temperature, top_k, top_p)
            q = filtered_softmax(dl[b, j], temperature, top_k, top_p)
            x = int(draft[b, j])
            # min(1, p/q): q(x) = 0 < p(x) accepts; p(x) = 0 rejects whatever q(x) is
            r = p[x] / q[x] if q[x] > 0 else (np.inf if p[x] > 0 else 0.0)
            ratio[b, j] = r
            if not (u[b, j] < r):        # reject: stop here, later drafts are discarded
                a = j
                break
        if a < D:
            p = filtered_softmax(tl[b, a], temperature, top_k, top_p)
            q = filtered_softmax(dl[b, a], temperature, top_k, top_p)
            w = np.maximum(0.0, p - q)   # the probability still missing for each token
            if not (w > 0).any():
                w = p                    # unreachable unless p == q exactly
        else:
            w = filtered_softmax(tl[b, D], temperature, top_k, top_p)  # bonus: after the full draft
        k, t, total, lo, hi = _inverse_cdf(w, u[b, D])
        accept_len[b] = a
        out_token[b] = k
        residual[b] = w / total
        t_draw[b], r_total[b], cdf_lo[b], cdf_hi[b] = t, total, lo, hi
    trace = {"ratio": ratio, "t": t_draw, "R": r_total, "cdf_lo": cdf_lo, "cdf_hi": cdf_hi}
    return accept_len, out_token, residual, trace


# --------------------------------------------------------------------------------------------
# Realignment (EQSPEC unpad-append-repad)  [BSDDR 2.1, 2.2; CF Abstract; IE5 "Acceptance
# changes across the workload" (commit accepted KV, discard speculative KV)]
# --------------------------------------------------------------------------------------------

def realign_plan(n_committed, width: int, accept_len, draft_len: int):
    """Per-row column plan of one realignment.

    Returns (n_new[B], W_new, src_lo[B], dst_lo[B], keep[B]):
      N'_b  = N_b + a_b + 1                 (accepted drafts plus the replacement/bonus)
      W'    = max_b N'_b                    (re-left-pad to the longest row)
      keep_b = N'_b - 1 = N_b + a_b         (surviving K/V columns: committed, pending, accepted)
      src_lo_b = W - N_b,  dst_lo_b = W' - N'_b
    """
    n = np.asarray(n_committed, dtype=np.int64)
    a = np.asarray(accept_len, dtype=np.int64)
    if (a < 0).any() or (a > draft_len).any():
        raise OracleError("accept length out of range")
    if (n < 1).any() or (n > width).any():
        raise OracleError("committed length out of range")
    n_new = n + a + 1
    w_new = int(n_new.max()) if len(n_new) else 0
    return n_new, w_new, width - n, w_new - n_new, n + a


def realign(kv_src, kv_dst, n_committed, width: int, accept_len, out_token, draft, ids_src,
            pad_id: int = 0):
    """One EQSPEC realignment, out of place.

    kv_src, kv_dst: [L, 2, B, H, S, hd] caches (any dtype; values are only moved).  kv_src holds
                    K/V for columns [W-N_b, W+D) of row b (committed but pending, then the D+1
                    columns the verification pass wrote).  kv_dst is the other buffer of the
                    ping-pong pair; its pad columns are left as they were.
    ids_src:        [B, S_src] token ids, row b's committed tokens at [W-N_b, W).
    Returns (kv_out, ids[B, S_dst], mask[B, S_dst] uint8, pos[B, S_dst] int32, n_new[B], W').

    Unpad each row, append the accepted drafts and the replacement/bonus token, re-left-pad to the
    longest row, recompute position IDs from 0 over the content, and shift the surviving K/V
    columns; the rejected drafts' columns [W+a_b, W+D) are discarded (never copied).
    """
    draft = np.asarray(draft)
    B, D = draft.shape
    S_src = kv_src.shape[4]
    S_dst = kv_dst.shape[4]
    if width + D > S_src:
        raise OracleError("source capacity")
    n_new, w_new, src_lo, dst_lo, keep = realign_plan(n_committed, width, accept_len, D)
    if w_new + D > S_dst:
        raise OracleError("capacity")   # the next verification pass could not be written
    kv_out = np.array(kv_dst, copy=True)
    ids = np.full((B, S_dst), pad_id, dtype=np.int32)
    mask = np.zeros((B, S_dst), dtype=np.uint8)
    pos = np.zeros((B, S_dst), dtype=np.int32)
    n = np.asarray(n_committed, dtype=np.int64)
    a = np.asarray(accept_len, dtype=np.int64)
    for b in range(B):
        s, d, k = int(src_lo[b]), int(dst_lo[b]), int(keep[b])
        kv_out[:, :, b, :, d:d + k, :] = kv_src[:, :, b, :, s:s + k, :]
        tokens = (list(np.asarray(ids_src[b, width - n[b]:width]))
                  + list(draft[b, :a[b]]) + [int(out_token[b])])
        ids[b, d:w_new] = tokens
        mask[b, d:w_new] = 1
        pos[b, d:w_new] = np.arange(n_new[b])
    return kv_out, ids, mask, pos, n_new.astype(np.int32), w_new


def check_invariants(mask, pos, n_committed, width: int):
    """The two synchronisation invariants of [BSDDR 2.1] for a left-padded batch of width W.

    (1) rectangular alignment: every row has pad + content == W (content right-aligned, ending
        at column W-1, and nothing at or beyond W);
    (2) position-ID contiguity: position IDs run 0, 1, ..., N_b-1 over the content columns that
        the mask marks.
    Returns a list of violation strings (empty when both hold).
    """
    bad = []
    mask = np.asarray(mask)
    pos = np.asarray(pos)
    for b, nb in enumerate(np.asarray(n_committed)):
        nb = int(nb)
        row_m = mask[b]
        content = np.nonzero(row_m)[0]
        if len(content) != nb:
            bad.append(f"row {b}: {len(content)} content columns, expected {nb}")
            continue
        if nb and (content[0] != width - nb or content[-1] != width - 1):
            bad.append(f"row {b}: content not right-aligned at width {width}")
        if (np.diff(content) != 1).any():
            bad.append(f"row {b}: content not contiguous")
        if (pos[b, content] != np.arange(nb)).any():
            bad.append(f"row {b}: position IDs not 0..N-1 over content")
    return bad


# --------------------------------------------------------------------------------------------
# EXSPEC grouping  [BSDDR 2.3: SequencePool, cross-batch grouping of same-length sequences]
# --------------------------------------------------------------------------------------------

def group_by_length(lengths, batch_size: int):
    """Group pool rows into batches.

    Rows of equal length, in index order, fill whole batches of ``batch_size`` (uniform batches:
    no realignment needed).  What is left of every length, in (length, index) order, is cut into
    mixed batches of at most ``batch_size`` rows (these are realigned).
    Returns (perm[N], batch_offsets[nb+1], batch_uniform[nb], num_uniform).
    """
    lengths = [int(x) for x in lengths]
    if batch_size < 1:
        raise OracleError("batch size")
    by_len = {}
    for i in sorted(range(len(lengths)), key=lambda i: (lengths[i], i)):
        by_len.setdefault(lengths[i], []).append(i)
    batches, uniform, leftover = [], [], []
    for length in sorted(by_len):
        rows = by_len[length]
        whole = len(rows) // batch_size * batch_size
        for k in range(0, whole, batch_size):
            batches.append(rows[k:k + batch_size])
            uniform.append(1)
        leftover.extend(rows[whole:])
    num_uniform = len(batches)
    for k in range(0, len(leftover), batch_size):
        batches.append(leftover[k:k + batch_size])
        uniform.append(0)
    perm = np.array([i for bt in batches for i in bt], dtype=np.int32)
    offsets = np.zeros(len(batches) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum([len(bt) for bt in batches])
    return perm, offsets, np.array(uniform, dtype=np.uint8), num_uniform


def pool_gather(arena, slot_cols, slot_len, rows, scratch, pad_id: int = 0, pool_ids=None):
    """Gather mixed-length pool rows into a left-padded batch (the "repad" of [BSDDR 2.2]
    applied to EXSPEC's leftovers [BSDDR 2.3]).

    arena:     [L, 2, H, C, hd]  the pool's K/V, unpadded at rest: slot s owns columns
               [slot_cols[s], slot_cols[s] + capacity) and holds K/V of its first N_s - 1 tokens.
    slot_len:  [S] committed length N_s per slot.
    rows:      the batch's slots, in batch order.
    scratch:   [L, 2, R, H, Sc, hd] padded batch buffer (R >= len(rows)).
    Row i of the batch gets width W = max N_s over the batch; its K/V columns [0, N_s - 1) move to
    scratch columns [W - N_s, W - 1).  Returns (scratch_out, W, ids, mask, pos) where ids is only
    filled when ``pool_ids`` ([S, cap]) is given.
    """
    n = np.array([int(slot_len[s]) for s in rows], dtype=np.int64)
    if (n < 1).any():
        raise OracleError("empty sequence")
    width = int(n.max())
    out = np.array(scratch, copy=True)
    Sc = scratch.shape[4]
    ids = np.full((len(rows), Sc), pad_id, dtype=np.int32)
    mask = np.zeros((len(rows), Sc), dtype=np.uint8)
    pos = np.zeros((len(rows), Sc), dtype=np.int32)
    for i, s in enumerate(rows):
        c0 = int(slot_cols[s])
        k = int(n[i]) - 1
        d = width - int(n[i])
        out[:, :, i, :, d:d + k, :] = arena[:, :, :, c0:c0 + k, :]
        mask[i, d:width] = 1
        pos[i, d:width] = np.arange(n[i])
        if pool_ids is not None:
            ids[i, d:width] = np.asarray(pool_ids[s, :n[i]])
    return out, width, ids, mask, pos


def pool_append(arena, slot_cols, slot_len, rows, scratch, width: int, accept_len, out_token,
                draft, pool_ids=None):
    """Append a verified batch back to its slots (the "append" of [BSDDR 2.2] for the pool).

    Batch row i (slot s) keeps scratch columns [W - 1, W + a_i) (its pending token and accepted
    drafts) which move to slot columns [N_s - 1, N_s + a_i); N_s grows by a_i + 1, and when
    ``pool_ids`` is given the accepted drafts and the replacement/bonus token are appended to the
    slot's ids.  Returns (arena_out, slot_len_out, pool_ids_out).
    """
    out = np.array(arena, copy=True)
    new_len = np.array(slot_len, copy=True)
    ids_out = None if pool_ids is None else np.array(pool_ids, copy=True)
    for i, s in enumerate(rows):
        a = int(accept_len[i])
        nb = int(slot_len[s])
        c0 = int(slot_cols[s])
        out[:, :, :, c0 + nb - 1:c0 + nb + a, :] = scratch[:, :, i, :, width - 1:width + a, :]
        new_len[s] = nb + a + 1
        if ids_out is not None:
            ids_out[s, nb:nb + a] = np.asarray(draft[i, :a])
            ids_out[s, nb + a] = int(out_token[i])
    return out, new_len, ids_out


# --------------------------------------------------------------------------------------------
# SequencePool lifecycle  [BSDDR 2.3: "a pool of active sequences" grouped by length; only the
# mixed-length ones are realigned]
# --------------------------------------------------------------------------------------------

FREE, ACTIVE, FINISHED_EOS, FINISHED_LENGTH = 0, 1, 2, 3


def group_by_window(lengths, batch_size: int, window: int):
    """Group rows into batches by a length window.

    Walk the rows in (length, index) order.  At row position i, if the ``batch_size`` rows
    i .. i + batch_size - 1 span at most ``window`` in length, they form a windowed batch and the
    walk moves past them; otherwise row i is a leftover and the walk moves on by one.  The
    leftovers, in (length, index) order, are cut into mixed batches of at most ``batch_size``.
    With window 0 this is the exact-length rule of ``group_by_length``.
    Returns (perm[N], batch_offsets[nb+1], batch_uniform[nb], num_windowed); a windowed batch is
    flagged uniform iff all its rows have one length, a mixed batch never.
    """
    lengths = [int(x) for x in lengths]
    if batch_size < 1 or window < 0:
        raise OracleError("batch size / window")
    order = sorted(range(len(lengths)), key=lambda i: (lengths[i], i))
    sl = [lengths[i] for i in order]
    n = len(order)
    batches, uniform, leftover = [], [], []
    i = 0
    while i < n:
        last = i + batch_size - 1
        if last < n and sl[last] - sl[i] <= window:
            batches.append(order[i:last + 1])
            uniform.append(1 if sl[last] == sl[i] else 0)
            i = last + 1
        else:
            leftover.append(order[i])
            i += 1
    num_windowed = len(batches)
    for k in range(0, len(leftover), batch_size):
        batches.append(leftover[k:k + batch_size])
        uniform.append(0)
    perm = np.array([r for bt in batches for r in bt], dtype=np.int32)
    offsets = np.zeros(len(batches) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum([len(bt) for bt in batches])
    return perm, offsets, np.array(uniform, dtype=np.uint8), num_windowed


def pool_schedule(state, slot_len, batch_size: int, window: int = 0):
    """One scheduling step of the pool.

    The ACTIVE slots (in slot order) are grouped by ``group_by_window``; perm lists slots.  Every
    FINISHED slot is reported once, in slot order, with its state as the reason, and becomes FREE.
    Returns a dict with perm, offsets, uniform, num_windowed, num_active, finished, reason and
    the new state.
    """
    state = np.asarray(state, dtype=np.uint8)
    slot_len = np.asarray(slot_len)
    if (state > FINISHED_LENGTH).any():
        raise OracleError("slot state")
    active = [s for s in range(len(state)) if state[s] == ACTIVE]
    if any(int(slot_len[s]) < 1 for s in active):
        raise OracleError("empty sequence")
    perm, offsets, uniform, nw = group_by_window([int(slot_len[s]) for s in active], batch_size,
                                                 window)
    finished = [s for s in range(len(state)) if state[s] in (FINISHED_EOS, FINISHED_LENGTH)]
    new_state = state.copy()
    new_state[finished] = FREE
    return {"perm": np.array([active[i] for i in perm], dtype=np.int32), "offsets": offsets,
            "uniform": uniform, "num_windowed": nw, "num_active": len(active),
            "finished": np.array(finished, dtype=np.int32),
            "reason": state[finished].astype(np.uint8), "state": new_state}


def retire(len_before, len_after, pool_ids, rows, slot_limit, eos_id: int, state):
    """Retirement after an append: for each slot s in ``rows``, scan the tokens committed this
    round, positions q = len_before[s] .. len_after[s] - 1 in order.  At the first q whose token
    is ``eos_id`` the sequence finishes by end of sequence; else at the first q with q + 1 ==
    slot_limit[s] it finishes by length.  Either way its length becomes q + 1.
    Returns (slot_len_out, state_out)."""
    new_len = np.array(len_after, copy=True)
    new_state = np.array(state, dtype=np.uint8, copy=True)
    for s in rows:
        for q in range(int(len_before[s]), int(len_after[s])):
            if int(pool_ids[s][q]) == eos_id:
                new_len[s], new_state[s] = q + 1, FINISHED_EOS
                break
            if q + 1 >= int(slot_limit[s]):
                new_len[s], new_state[s] = q + 1, FINISHED_LENGTH
                break
    return new_len, new_state


def pool_admit(state, slot_col, slot_cap, slot_len, slot_limit, pool_ids, slots, cols, caps,
               limits, prompts, D: int, arena_cols: int):
    """Admit prompts into FREE slots: slot s = slots[i] gets arena columns [cols[i], cols[i] +
    caps[i]), limit limits[i], length len(prompts[i]) and the prompt as its first tokens; it
    becomes ACTIVE.  Nothing changes if any entry is invalid: a slot out of range, not FREE or
    named twice, an empty prompt, a prompt not shorter than its limit, or a range outside the
    arena (OracleError "range"); limit + D - 1 > cap or limit + D > ids_cap (OracleError
    "capacity").  Returns the new (state, slot_col, slot_cap, slot_len, slot_limit, pool_ids)."""
    S, ids_cap = np.asarray(pool_ids).shape
    if len(set(int(x) for x in slots)) != len(slots):
        raise OracleError("range")
    for i, s in enumerate(slots):
        s, n, lim, c0, cap = int(s), len(prompts[i]), int(limits[i]), int(cols[i]), int(caps[i])
        if not (0 <= s < S) or state[s] != FREE or n < 1 or n >= lim or c0 < 0 or cap < 1 \
                or c0 + cap > arena_cols:
            raise OracleError("range")
        if lim + D - 1 > cap or lim + D > ids_cap:
            raise OracleError("capacity")
    out = [np.array(x, copy=True) for x in (state, slot_col, slot_cap, slot_len, slot_limit,
                                            pool_ids)]
    st, col, cap, ln, lim, ids = out
    for i, s in enumerate(slots):
        s = int(s)
        st[s], col[s], cap[s] = ACTIVE, int(cols[i]), int(caps[i])
        ln[s], lim[s] = len(prompts[i]), int(limits[i])
        ids[s, :len(prompts[i])] = np.asarray(prompts[i])
    return st, col, cap, ln, lim, ids


class FirstFitArena:
    """Arena columns [0, cols) handed out first fit: an allocation of n columns takes the lowest
    column c with [c, c + n) all free.  Kept as a plain occupancy bitmap."""

    def __init__(self, cols: int):
        if cols < 1:
            raise OracleError("arena size")
        self.used = np.zeros(cols, dtype=bool)
        self.blocks = {}

    def alloc(self, n: int) -> int:
        if n < 1:
            raise OracleError("size")
        cols = len(self.used)
        for c in range(cols - n + 1):
            if not self.used[c:c + n].any():
                self.used[c:c + n] = True
                self.blocks[c] = n
                return c
        raise OracleError("capacity")

    def free(self, c: int) -> None:
        if c not in self.blocks:
            raise OracleError("not an allocation")
        self.used[c:c + self.blocks.pop(c)] = False

    def free_cols(self) -> int:
        return int((~self.used).sum())

    def largest_free(self) -> int:
        best = run = 0
        for u in self.used:
            run = 0 if u else run + 1
            best = max(best, run)
        return best


# --------------------------------------------------------------------------------------------
# Counter-based uniforms for the fused round  [Philox, SC11 "Parallel Random Numbers: As Easy as
# 1, 2, 3"; the uniforms u[b][j] of IE5 "Exactness Means Different Things..." drawn in-kernel]
# --------------------------------------------------------------------------------------------

# The paper's multipliers (M0, M1) and Weyl key increments (W0, W1) for each word size.
PHILOX_CONSTANTS = {
    32: ((0xD2511F53, 0xCD9E8D57), (0x9E3779B9, 0xBB67AE85)),
    64: ((0xD2E7470EE14C6C93, 0xCA5A826395121157), (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)),
}


def philox(ctr, key, bits: int = 32, rounds: int = 10):
    """PhiloxNx W-R with N = 4 words of ``bits`` (32 or 64) bits: ``rounds`` rounds of
    (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2, c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),
    the key bumped by the Weyl constants (W0, W1) between rounds."""
    mask = (1 << bits) - 1
    if bits not in PHILOX_CONSTANTS:
        raise OracleError("word size")
    M, W = PHILOX_CONSTANTS[bits]
    c = [int(x) & mask for x in ctr]
    k = [int(x) & mask for x in key]
    for r in range(rounds):
        if r:
            k = [(k[0] + W[0]) & mask, (k[1] + W[1]) & mask]
        p0 = M[0] * c[0]
        p1 = M[1] * c[2]
        c = [(p1 >> bits) ^ c[1] ^ k[0], p1 & mask, (p0 >> bits) ^ c[3] ^ k[1], p0 & mask]
    return c


def philox_uniforms(seed: int, offset: int, B: int, D: int):
    """The uniforms u[B, D+1] of one round drawn from (seed, offset) as the fused round draws
    them: u[b][j] = (x >> 8) * 2^-24, x = word j mod 4 of Philox4x32-10 at counter
    (j div 4, b, offset mod 2^32, offset div 2^32), key (seed mod 2^32, seed div 2^32)."""
    u = np.zeros((B, D + 1), dtype=np.float64)
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    for b in range(B):
        for j in range(D + 1):
            x = philox((j // 4, b, offset & 0xFFFFFFFF, (offset >> 32) & 0xFFFFFFFF), key)[j % 4]
            u[b, j] = (x >> 8) / float(1 << 24)
    return u
