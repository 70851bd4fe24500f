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


class EqspecBatch:
    def __init__(self, layers, heads, head_dim, kv_dtype, B, D, cap, max_rounds, device="cuda",
                 pad_id=0):
        self.L, self.H, self.hd, self.B, self.D, self.cap = layers, heads, head_dim, B, D, cap
        self.max_rounds = max_rounds
        self.pad_id = pad_id
        dev = torch.device(device)
        self.kv = [torch.empty((layers, 2, B, heads, cap, head_dim), dtype=kv_dtype, device=dev)
                   for _ in range(2)]
        self.ids = [torch.full((B, cap), pad_id, dtype=torch.int32, device=dev) for _ in range(2)]
        self.mask = [torch.zeros((B, cap), dtype=torch.uint8, device=dev) for _ in range(2)]
        self.pos = [torch.zeros((B, cap), dtype=torch.int32, device=dev) for _ in range(2)]
        self.n_hist = torch.zeros((max_rounds + 1, B), dtype=torch.int32, device=dev)
        self.w_hist = torch.zeros((max_rounds + 1, 1), dtype=torch.int32, device=dev)
        self.accept_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.out_token = torch.zeros(B, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
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
        return self.kv[self.cur]

    @property
    def n_committed(self):
        return self.n_hist[self.round]

    @property
    def width(self):
        return self.w_hist[self.round]

    # ------------------------------------------------------------------ one round
    def verify_greedy(self, logits, draft, stream=None):
        specdec.verify_greedy(logits, draft, self.accept_len, self.out_token, self.status, stream)

    def verify_sample(self, target_logits, draft_logits, draft, uniforms, temperature,
                      residual=None, stream=None):
        specdec.verify_sample(target_logits, draft_logits, draft, uniforms, temperature,
                              self.accept_len, self.out_token, self.status, residual, stream)

    def realign(self, draft, copy_engine=0, stream=None):
        r = self.round
        if r >= self.max_rounds:
            raise RuntimeError("round history is full")
        s, d = self.cur, 1 - self.cur
        specdec.realign(self.kv[s], self.kv[d], self.n_hist[r], self.w_hist[r], self.accept_len,
                        self.out_token, draft, self.ids[s], self.ids[d], self.mask[d],
                        self.pos[d], self.n_hist[r + 1], self.w_hist[r + 1], self.status,
                        pad_id=self.pad_id, copy_engine=copy_engine, stream=stream)
        self.cur = d
        self.round = r + 1
