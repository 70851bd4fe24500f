"""Caller-side state of a left-padded speculative batch: ping-pong K/V caches and metadata.

The library itself keeps no state; this class owns the device buffers one EQSPEC batch needs and
calls the C ABI in the order of a round: verification, then realignment from the current cache
into the other one.  Committed lengths and widths are kept per round in a history tensor (round r
reads row r and writes row r+1), so a sequence of rounds needs no host synchronisation and can be
examined afterwards.
"""
from __future__ import annotations

import torch

from . import specdec


class Workspaces:
    """Zero-filled verification workspaces, one per kind, grown on demand (a workspace is left
    zero-filled by every call, so one buffer serves every shape it is large enough for)."""

    def __init__(self, device):
        self.device = device
        self._ws = {}

    def get(self, kind, nbytes):
        ws = self._ws.get(kind)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            self._ws[kind] = ws
        return ws

    def greedy(self, logits, draft):
        B, D = draft.shape
        return self.get("greedy", specdec.greedy_workspace_bytes(B, D))

    def bounds(self, draft):
        """Keep-bound buffer [B, 2D+1, 2] int32 for the sampling settings."""
        B, D = draft.shape
        key = ("bounds", B, D)
        t = self._ws.get(key)
        if t is None:
            t = torch.zeros((B, 2 * D + 1, 2), dtype=torch.int32, device=self.device)
            self._ws[key] = t
        return t


class EqspecBatch:
    """``in_place=True`` keeps one K/V cache and realigns it in place (half the cache memory);
    ids, mask and positions stay double-buffered.  ``scheduled=True`` (default) gives the
    realignment its two scheduling words, so its CTAs take work items from a counter; False
    gives every CTA a fixed share."""

    def __init__(self, layers, heads, head_dim, kv_dtype, B, D, cap, max_rounds, device="cuda",
                 pad_id=0, in_place=False, pdl=False, scheduled=True):
        self.L, self.H, self.hd, self.B, self.D, self.cap = layers, heads, head_dim, B, D, cap
        self.max_rounds = max_rounds
        self.pad_id = pad_id
        dev = torch.device(device)
        self.in_place = in_place
        self.pdl = pdl
        self.kv = [torch.empty((layers, 2, B, heads, cap, head_dim), dtype=kv_dtype, device=dev)
                   for _ in range(1 if in_place else 2)]
        self.ids = [torch.full((B, cap), pad_id, dtype=torch.int32, device=dev) for _ in range(2)]
        self.mask = [torch.zeros((B, cap), dtype=torch.uint8, device=dev) for _ in range(2)]
        self.pos = [torch.zeros((B, cap), dtype=torch.int32, device=dev) for _ in range(2)]
        # Per-round history, row r = [N (B), W, accept lengths (B), tokens (B)]: N and W at the
        # start of round r, round r's verification results.  Round r's results and the lengths
        # and width they produce (row r + 1) are one contiguous span of 3B + 1 ints.
        self.hist = torch.zeros((max_rounds + 1, 3 * B + 1), dtype=torch.int32, device=dev)
        self.n_hist = self.hist[:, :B]
        self.w_hist = self.hist[:, B:B + 1]
        self.accept_len = self.hist[0, B + 1:2 * B + 1]
        self.out_token = self.hist[0, 2 * B + 1:]
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.sched_words = torch.zeros(2, dtype=torch.int32, device=dev) if scheduled else None
        self.workspaces = Workspaces(dev)
        self.round = 0
        self.cur = 0

    # ------------------------------------------------------------------ set-up (not the hot path)
    def start(self, prompts):
        """Right-align the prompts (lists of token ids, each non-empty) in the current buffers."""
        B = self.B
        n = torch.tensor([len(p) for p in prompts], dtype=torch.int32)
        if len(prompts) != B or (n < 1).any():
            raise ValueError("need B non-empty prompts")
        W = int(n.max())
        if W + self.D > self.cap:
            raise ValueError("cache too small for the prompts")
        ids = torch.full((B, self.cap), self.pad_id, dtype=torch.int32)
        mask = torch.zeros((B, self.cap), dtype=torch.uint8)
        pos = torch.zeros((B, self.cap), dtype=torch.int32)
        for b, p in enumerate(prompts):
            lo = W - len(p)
            ids[b, lo:W] = torch.as_tensor(p, dtype=torch.int32)
            mask[b, lo:W] = 1
            pos[b, lo:W] = torch.arange(len(p), dtype=torch.int32)
        self.round, self.cur = 0, 0
        self.accept_len = self.hist[0, B + 1:2 * B + 1]
        self.out_token = self.hist[0, 2 * B + 1:]
        self.ids[0].copy_(ids)
        self.mask[0].copy_(mask)
        self.pos[0].copy_(pos)
        self.n_hist[0].copy_(n)
        self.w_hist[0].fill_(W)
        self.status.zero_()
        return W

    # ------------------------------------------------------------------ current state
    @property
    def cache(self):
        return self.kv[0 if self.in_place else self.cur]

    @property
    def n_committed(self):
        return self.n_hist[self.round]

    @property
    def width(self):
        return self.w_hist[self.round]

    # ------------------------------------------------------------------ one round
    def _results_row(self):
        """Point accept_len / out_token at this round's row of the history."""
        r, B = self.round, self.B
        if r >= self.max_rounds:
            raise RuntimeError("round history is full")
        self.accept_len = self.hist[r, B + 1:2 * B + 1]
        self.out_token = self.hist[r, 2 * B + 1:]

    def results_span(self, r):
        """Round r's results as one contiguous int32 view [accept lengths (B), tokens (B),
        committed lengths after the round (B), width after the round]."""
        n = 3 * self.B + 1
        return self.hist.view(-1)[r * n + self.B + 1:(r + 1) * n + self.B + 1]

    def verify_greedy(self, logits, draft, stream=None):
        self._results_row()
        specdec.verify_greedy(logits, draft, self.accept_len, self.out_token, self.status,
                              self.workspaces.greedy(logits, draft), stream)

    def verify_sample(self, target_logits, draft_logits, draft, uniforms, temperature,
                      residual=None, stream=None, top_k=0, top_p=1.0, seed=None):
        """Sampled verification; with top_k / top_p the rows' keep bounds are computed first
        (specdec_sampling_filter) into a buffer this batch keeps.  ``uniforms`` None: they are
        drawn in-kernel from ``seed`` with this round's index as the Philox offset."""
        self._results_row()
        bounds = None
        if (0 < top_k < target_logits.shape[-1]) or top_p < 1.0:
            bounds = self.workspaces.bounds(draft)
            specdec.sampling_filter(target_logits, draft_logits, temperature, top_k, top_p,
                                    bounds, self.status, stream)
        if uniforms is None:
            if seed is None:
                raise ValueError("in-kernel uniforms need a seed")
            specdec.verify_sample_philox(target_logits, draft_logits, draft, seed, self.round,
                                         temperature, self.accept_len, self.out_token,
                                         self.status, residual, stream, keep_bounds=bounds)
            return
        specdec.verify_sample(target_logits, draft_logits, draft, uniforms, temperature,
                              self.accept_len, self.out_token, self.status, residual, stream,
                              keep_bounds=bounds)

    def realign(self, draft, copy_engine=0, stream=None):
        """Realign after this round's verification; with ``pdl`` (constructor) the realignment
        is launched as a programmatic dependent of the verification kernel ahead of it."""
        r = self.round
        if r >= self.max_rounds:
            raise RuntimeError("round history is full")
        s, d = self.cur, 1 - self.cur
        ks, kd = (self.kv[0], self.kv[0]) if self.in_place else (self.kv[s], self.kv[d])
        specdec.realign(ks, kd, self.n_hist[r], self.w_hist[r], self.accept_len,
                        self.out_token, draft, self.ids[s], self.ids[d], self.mask[d],
                        self.pos[d], self.n_hist[r + 1], self.w_hist[r + 1], self.status,
                        pad_id=self.pad_id, copy_engine=copy_engine, pdl=self.pdl, stream=stream,
                        schedule=self.sched_words)
        self.cur = d
        self.round = r + 1


class HostRounds:
    """Rounds of one ``EqspecBatch`` fed from pinned host memory.

    Each round's inputs are pinned host tensors (for instance ``logits`` and ``draft``, plus
    ``draft_logits`` and ``uniforms`` for sampled rounds).  They are copied into one of ``depth``
    device staging sets on a copy stream while earlier rounds run on the compute stream: round j
    goes to set j mod depth, so the copy stream may run up to depth - 1 rounds ahead of the
    verification and realignment, and a copy that the host link delays is hidden as long as that
    lead lasts.  A staging set is refilled only once the realignment that last read it has
    finished.  After each realignment the
    round's results (accept lengths, tokens, committed lengths and the width: 3B + 1 int32, one
    contiguous span of the batch's history) are copied into a row of a pinned host tensor on a
    third stream, so no round waits for the copy-back of the one before.
    """

    def __init__(self, batch: EqspecBatch, like: dict, stream=None, timed=False, depth=2):
        dev = batch.status.device
        if int(depth) < 1:
            raise ValueError("depth must be at least 1")
        self.batch = batch
        self.depth = int(depth)
        self.timed = timed          # record events around every input copy (copy_ms)
        self._copy_events = []
        self.stream = stream or torch.cuda.current_stream(dev)
        self.copy_stream = torch.cuda.Stream(dev)
        self.slots = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in like.items()}
                      for _ in range(self.depth)]
        self.d2h_stream = torch.cuda.Stream(dev)
        self.copied = [torch.cuda.Event() for _ in range(self.depth)]
        self.freed = [torch.cuda.Event() for _ in range(self.depth)]
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in like.values())
        self.d2h_bytes = (3 * batch.B + 1) * 4

    def _stage(self, k, host, wait_freed):
        if wait_freed:
            self.copy_stream.wait_event(self.freed[k])
        if self.timed:
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(self.copy_stream)
        with torch.cuda.stream(self.copy_stream):
            for name, t in host.items():
                self.slots[k][name].copy_(t, non_blocking=True)
        self.copied[k].record(self.copy_stream)
        if self.timed:
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(self.copy_stream)
            self._copy_events.append((e0, e1))

    def copy_ms(self):
        """Milliseconds of every input copy staged so far (timed=True; synchronise first)."""
        return [e0.elapsed_time(e1) for e0, e1 in self._copy_events]

    def run(self, host_rounds, step, out):
        """Run ``len(host_rounds)`` rounds.  ``host_rounds[i]`` maps input names to pinned host
        tensors; ``step(inputs)`` launches round i's verification on the batch given the device
        copies (the realignment, with ``inputs["draft"]``, follows here); ``out`` is a pinned int32
        tensor [len(host_rounds), 3B + 1].  Asynchronous: synchronise the stream before reading
        ``out``."""
        n = len(host_rounds)
        if n == 0:
            return
        B = self.batch.B
        if (out.dtype != torch.int32 or out.dim() != 2 or out.shape[0] < n
                or out.shape[1] != 3 * B + 1 or not out.is_pinned()):
            raise ValueError("out must be a pinned int32 tensor [rounds, 3B + 1]")
        P = self.depth
        start = torch.cuda.Event()
        start.record(self.stream)
        self.copy_stream.wait_event(start)   # no copy starts before the work issued so far
        for j in range(min(P - 1, n)):       # fill: every set but one, nothing to wait for
            self._stage(j, host_rounds[j], False)
        for i in range(n):
            j = i + P - 1                    # its set was last read by round i - 1
            if j < n:
                self._stage(j % P, host_rounds[j], i >= 1)
            k = i % P
            self.stream.wait_event(self.copied[k])
            inp = self.slots[k]
            with torch.cuda.stream(self.stream):
                r = self.batch.round
                step(inp)
                self.batch.realign(inp["draft"])
                self.freed[k].record(self.stream)
            # The result copy waits for the round on its own stream: the next round's kernels
            # do not wait for it (each round's results have their own row of the history).
            self.d2h_stream.wait_event(self.freed[k])
            with torch.cuda.stream(self.d2h_stream):
                out[i].copy_(self.batch.results_span(r), non_blocking=True)
        self.stream.wait_stream(self.copy_stream)
        self.stream.wait_stream(self.d2h_stream)


class ExspecPool:
    """Caller-side state of an EXSPEC SequencePool (one GPU).

    Slots are unpadded at rest in one arena [L, 2, 1, H, sum(cap_s), hd]: slot s owns columns
    [slot_col[s], slot_col[s] + cap_s) and holds the K/V of its first N_s - 1 tokens.  A round
    groups the slots by length (uniform batches of ``batch_size`` equal-length rows first, then
    mixed leftovers), verifies every slot's drafts in one call, and then per batch either commits
    in place (uniform batch) or gathers the rows into the padded batch buffer and appends the
    accepted columns back (mixed batch).  The schedule is read back to the host once per round:
    it decides which calls follow.
    """

    def __init__(self, layers, heads, head_dim, kv_dtype, prompts, D, rounds, batch_size=8,
                 device="cuda", pad_id=0, scheduled=True):
        dev = torch.device(device)
        self.S = len(prompts)
        self.D, self.bs, self.pad_id = D, batch_size, pad_id
        n0 = [len(p) for p in prompts]
        if min(n0) < 1:
            raise ValueError("empty prompt")
        grow = rounds * (D + 1) + D + 1
        caps = [n + grow for n in n0]
        cols = [0]
        for c in caps[:-1]:
            cols.append(cols[-1] + c)
        self.max_len = max(caps)
        self.arena = torch.empty((layers, 2, 1, heads, sum(caps), head_dim), dtype=kv_dtype,
                                 device=dev)
        sc_cap = max(n0) + grow
        self.scratch = torch.empty((layers, 2, batch_size, heads, sc_cap, head_dim), dtype=kv_dtype,
                                   device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        self.slot_col = torch.tensor(cols, **i32)
        self.slot_cap = torch.tensor(caps, **i32)
        self.slot_len = torch.tensor(n0, **i32)
        self.pool_ids = torch.full((self.S, self.max_len), pad_id, **i32)
        for s, p in enumerate(prompts):
            self.pool_ids[s, :len(p)] = torch.as_tensor(p, dtype=torch.int32)
        self.scratch_ids = torch.zeros((batch_size, sc_cap), **i32)
        self.scratch_mask = torch.zeros((batch_size, sc_cap), dtype=torch.uint8, device=dev)
        self.scratch_pos = torch.zeros((batch_size, sc_cap), **i32)
        self.batch_len = torch.zeros(batch_size, **i32)
        self.width = torch.zeros(1, **i32)
        self.perm = torch.zeros(self.S, **i32)
        self.offsets = torch.zeros(self.S + 1, **i32)
        self.uniform = torch.zeros(self.S, dtype=torch.uint8, device=dev)
        self.counts = torch.zeros(2, **i32)  # num_batches, num_uniform
        self.accept_len = torch.zeros(self.S, **i32)
        self.out_token = torch.zeros(self.S, **i32)
        self.status = torch.zeros(1, **i32)
        self.sched_words = torch.zeros(2, **i32) if scheduled else None  # gather/append work items
        self.workspaces = Workspaces(dev)
        self._host = torch.zeros(2 + (self.S + 1) + self.S, dtype=torch.int32).pin_memory()

    def schedule(self, stream=None):
        """Group the slots by length on the device; returns the batches as (offset, rows, uniform)
        after one small device-to-host copy."""
        specdec.group_by_length(self.slot_len, self.bs, self.max_len, self.perm, self.offsets,
                                self.uniform, self.counts[0:1], self.counts[1:2], self.status,
                                stream)
        h = self._host
        S = self.S
        h[0:2].copy_(self.counts, non_blocking=True)
        h[2:3 + S].copy_(self.offsets, non_blocking=True)
        h[3 + S:].copy_(self.uniform.to(torch.int32), non_blocking=True)
        (stream or torch.cuda.current_stream()).synchronize()
        nb = int(h[0])
        off = h[2:3 + S].tolist()
        uni = h[3 + S:].tolist()
        return [(off[k], off[k + 1] - off[k], bool(uni[k])) for k in range(nb)]

    def verify_greedy(self, logits, draft, stream=None):
        """Greedy verification of every slot: logits [S, D+1, V], draft [S, D] in slot order."""
        specdec.verify_greedy(logits, draft, self.accept_len, self.out_token, self.status,
                              self.workspaces.greedy(logits, draft), stream)

    def verify_sample(self, target_logits, draft_logits, draft, uniforms, temperature,
                      stream=None):
        specdec.verify_sample(target_logits, draft_logits, draft, uniforms, temperature,
                              self.accept_len, self.out_token, self.status, None, stream)

    def gather(self, off, n, uniform, stream=None):
        """Repad batch perm[off:off+n] into the batch buffer (uniform batches: lengths only)."""
        rows = self.perm[off:off + n]
        specdec.pool_gather(self.arena, self.scratch, rows, self.D, self.slot_col, self.slot_cap,
                            self.slot_len, self.pool_ids, self.batch_len[:n], self.width,
                            self.status, self.scratch_ids, self.scratch_mask, self.scratch_pos,
                            pad_id=self.pad_id, in_place=uniform, stream=stream,
                            schedule=self.sched_words)

    def append(self, off, n, uniform, draft, stream=None):
        """Commit batch perm[off:off+n] back to its slots (pool-wide accept lengths and tokens)."""
        rows = self.perm[off:off + n]
        specdec.pool_append(self.arena, self.scratch, rows, self.D, self.slot_col, self.slot_cap,
                            self.slot_len, self.pool_ids, self.batch_len[:n], self.width,
                            self.accept_len, self.out_token, draft, self.status,
                            in_place=uniform, by_slot=True, stream=stream,
                            schedule=self.sched_words)


class SequencePool:
    """EXSPEC SequencePool with its lifecycle (one GPU): sequences are admitted into free slots,
    scheduled each round in batches by length window, verified, committed, and retired by the
    end-of-sequence token or their length limit.

    Device state: slot_state / slot_col / slot_cap / slot_len / slot_limit [S] and pool_ids
    [S, ids_cap]; K/V in one arena [L, 2, 1, H, arena_cols, hd] whose column runs are handed out
    by the host first-fit allocator (``specdec.Arena``).  The host keeps which slots are taken
    (admitted and not yet reported finished) and which run each one holds; it learns of finished
    sequences from the schedule's readback, the one device-to-host copy of a round, which also
    decides the calls that follow.

    A round: ``schedule()`` -> [admit()] -> verify (all slots, by slot) -> per batch
    ``gather()`` / (the target's verification pass writes K/V) / ``append()``.  Uniform batches are
    verified in place in their slots (no K/V is moved); windowed and mixed ones go through the
    padded batch buffer.
    """

    def __init__(self, layers, heads, head_dim, kv_dtype, S, arena_cols, D, max_len,
                 batch_size=8, window=0, eos_id=-1, device="cuda", pad_id=0, scheduled=True):
        dev = torch.device(device)
        self.S, self.D, self.bs, self.window = S, D, batch_size, window
        self.eos_id, self.pad_id, self.max_len = eos_id, pad_id, max_len
        self.arena_cols = arena_cols
        self.arena = torch.empty((layers, 2, 1, heads, arena_cols, head_dim), dtype=kv_dtype,
                                 device=dev)
        self.alloc = specdec.Arena(arena_cols)
        i32 = dict(dtype=torch.int32, device=dev)
        u8 = dict(dtype=torch.uint8, device=dev)
        self.slot_state = torch.zeros(S, **u8)
        self.slot_col = torch.zeros(S, **i32)
        self.slot_cap = torch.zeros(S, **i32)
        self.slot_len = torch.zeros(S, **i32)
        self.slot_limit = torch.zeros(S, **i32)
        self.ids_cap = max_len + D + 1
        self.pool_ids = torch.full((S, self.ids_cap), pad_id, **i32)
        sc_cap = max_len + D + 1
        self.scratch = torch.empty((layers, 2, batch_size, heads, sc_cap, head_dim),
                                   dtype=kv_dtype, device=dev)
        self.scratch_ids = torch.zeros((batch_size, sc_cap), **i32)
        self.scratch_mask = torch.zeros((batch_size, sc_cap), **u8)
        self.scratch_pos = torch.zeros((batch_size, sc_cap), **i32)
        self.batch_len = torch.zeros(batch_size, **i32)
        self.width = torch.zeros(1, **i32)
        self.perm = torch.zeros(S, **i32)
        self.offsets = torch.zeros(S + 1, **i32)
        self.uniform = torch.zeros(S, **u8)
        self.finished = torch.zeros(S, **i32)
        self.reason = torch.zeros(S, **u8)
        self.counts = torch.zeros(4, **i32)
        self.accept_len = torch.zeros(S, **i32)
        self.out_token = torch.zeros(S, **i32)
        self.status = torch.zeros(1, **i32)
        self.sched_words = torch.zeros(2, **i32) if scheduled else None  # gather/append work items
        self.workspaces = Workspaces(dev)
        # schedule readback: counts | offsets | uniform | finished | reason | slot_len | perm
        self._host = torch.zeros(4 + (S + 1) + 5 * S, dtype=torch.int32).pin_memory()
        self._dev_rb = torch.zeros_like(self._host, device=dev)
        self.host_len = [0] * S           # slot lengths as of the last schedule
        self.host_perm = []               # the last schedule's slots in batch order
        self.taken = [False] * S          # admitted and not yet reported finished
        self.run_of = [None] * S          # arena run of each taken slot

    # -------------------------------------------------------------- admission
    def admit(self, prompts, limits, stream=None):
        """Admit as many of ``prompts`` (token lists, in order) as there are free slots and arena
        room for; returns their slots (a prefix of the prompts is admitted).  Each needs
        limit + D - 1 arena columns.  The prompt's K/V is the caller's to write (prefill) at
        columns [slot_col, slot_col + len - 1) of the arena."""
        slots, cols, caps = [], [], []
        free = [s for s in range(self.S) if not self.taken[s]]
        for p, lim in zip(prompts, limits):
            if not free:
                break
            if lim > self.max_len or len(p) < 1 or len(p) >= lim:
                raise ValueError("prompt length / limit out of range")
            need = lim + self.D - 1
            c = self.alloc.alloc(need)
            if c is None:
                break
            s = free.pop(0)
            slots.append(s)
            cols.append(c)
            caps.append(need)
        n = len(slots)
        if n == 0:
            return []
        lens = [len(p) for p in prompts[:n]]
        off = [0]
        for x in lens:
            off.append(off[-1] + x)
        flat = [t for p in prompts[:n] for t in p]
        host = torch.tensor(slots + cols + caps + list(limits[:n]) + off + flat,
                            dtype=torch.int32).pin_memory()
        st = stream or torch.cuda.current_stream()
        with torch.cuda.stream(st):       # one copy of every argument, then the two launches
            dev = host.to(self.slot_len.device, non_blocking=True)
            v = [dev[k * n:(k + 1) * n] for k in range(4)]
            specdec.pool_admit(v[0], v[1], v[2], v[3], dev[5 * n + 1:], dev[4 * n:5 * n + 1],
                               self.D, self.arena_cols, self.slot_state, self.slot_col,
                               self.slot_cap, self.slot_len, self.slot_limit, self.pool_ids,
                               self.status, st)
        for s, c in zip(slots, cols):
            self.taken[s] = True
            self.run_of[s] = c
        return slots

    # -------------------------------------------------------------- schedule
    def schedule(self, stream=None):
        """Schedule the round on the device and read it back once.  Returns (batches, finished):
        batches as (offset, rows, uniform) into ``perm``; finished as (slot, reason) -- those
        slots' tokens stay readable (``tokens``) until they are admitted again, and their arena
        runs are returned to the allocator now.  ``host_len`` receives every slot's length and
        ``host_perm`` the scheduled slots in batch order."""
        specdec.pool_schedule(self.slot_state, self.slot_len, self.bs, self.window, self.perm,
                              self.offsets, self.uniform, self.finished, self.reason, self.counts,
                              self.status, stream)
        S, rb = self.S, self._dev_rb
        rb[0:4].copy_(self.counts, non_blocking=True)
        rb[4:5 + S].copy_(self.offsets, non_blocking=True)
        rb[5 + S:5 + 2 * S].copy_(self.uniform, non_blocking=True)
        rb[5 + 2 * S:5 + 3 * S].copy_(self.finished, non_blocking=True)
        rb[5 + 3 * S:5 + 4 * S].copy_(self.reason, non_blocking=True)
        rb[5 + 4 * S:5 + 5 * S].copy_(self.slot_len, non_blocking=True)
        rb[5 + 5 * S:5 + 6 * S].copy_(self.perm, non_blocking=True)
        self._host.copy_(rb, non_blocking=True)
        (stream or torch.cuda.current_stream()).synchronize()
        h = self._host.tolist()
        nb, nf = h[0], h[3]
        off = h[4:5 + S]
        uni = h[5 + S:5 + 2 * S]
        fin = list(zip(h[5 + 2 * S:5 + 2 * S + nf], h[5 + 3 * S:5 + 3 * S + nf]))
        self.host_len = h[5 + 4 * S:5 + 5 * S]
        self.host_perm = h[5 + 5 * S:5 + 5 * S + h[2]]
        for s, _ in fin:
            self.alloc.free(self.run_of[s])
            self.taken[s] = False
            self.run_of[s] = None
        return [(off[k], off[k + 1] - off[k], bool(uni[k])) for k in range(nb)], fin

    def tokens(self, slot):
        """Committed tokens of a slot (a device-to-host copy)."""
        n = int(self.slot_len[slot].item())
        return self.pool_ids[slot, :n].tolist()

    # -------------------------------------------------------------- one round's calls
    def verify_greedy(self, logits, draft, stream=None):
        """Greedy verification of every slot: logits [S, D+1, V], draft [S, D] in slot order
        (rows of slots that are not scheduled are ignored)."""
        specdec.verify_greedy(logits, draft, self.accept_len, self.out_token, self.status,
                              self.workspaces.greedy(logits, draft), stream)

    def gather(self, off, n, uniform, stream=None):
        """Repad batch perm[off:off+n] into the batch buffer (uniform batches: lengths only)."""
        specdec.pool_gather(self.arena, self.scratch, self.perm[off:off + n], self.D,
                            self.slot_col, self.slot_cap, self.slot_len, self.pool_ids,
                            self.batch_len[:n], self.width, self.status, self.scratch_ids,
                            self.scratch_mask, self.scratch_pos, pad_id=self.pad_id,
                            in_place=uniform, stream=stream, schedule=self.sched_words)

    def append(self, off, n, uniform, draft, stream=None):
        """Commit batch perm[off:off+n] back to its slots and retire finished sequences."""
        specdec.pool_append(self.arena, self.scratch, self.perm[off:off + n], self.D,
                            self.slot_col, self.slot_cap, self.slot_len, self.pool_ids,
                            self.batch_len[:n], self.width, self.accept_len, self.out_token,
                            draft, self.status, in_place=uniform, by_slot=True,
                            slot_state=self.slot_state, slot_limit=self.slot_limit,
                            eos_id=self.eos_id, stream=stream, schedule=self.sched_words)
