"""Seeded synthetic inputs for the verify + realign hot path.

This module only draws inputs; it holds none of the method's arithmetic (no acceptance test, no
argmax over a verified row, no realignment).  Both the CUDA path's tests/bench and the CPU oracle
consume what it produces.  Everything is plain torch on whatever device is asked for; a
``torch.Generator`` on that device makes it reproducible.

Shapes and distributions follow the model-shaped workloads:
* scores N(0, 1); for greedy rounds each draft position j < D, with probability alpha, gets its
  draft token's score raised to the row maximum + 1 (in fp32, then rounded to the storage dtype),
  so that acceptance is geometric in alpha; other drafts are uniform token ids;
* for sampled rounds, draft-model scores are target scores + N(0, sigma^2) and the drafts are
  drawn from the draft model's softmax at the sampling temperature (that is the draft model's
  job, not verification's);
* K/V values are either N(0, 1) (timing) or a *tag*: an exact function of
  (sequence, layer, k/v, head, position, token, dim) with values k/64, k in [-128, 128), exactly
  representable in bf16 and fp32, so a cache can be rebuilt from each sequence's tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

MASK32 = 0xFFFFFFFF


def make_gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


# ---------------------------------------------------------------------------- prompt lengths

def lengths_uniform(gen, n, lo, hi, device="cpu"):
    """Integers uniform in [lo, hi]."""
    return torch.randint(lo, hi + 1, (n,), generator=gen, device=device, dtype=torch.int64)


def lengths_lognormal(gen, n, median, sigma, lo, hi, device="cpu"):
    """exp(N(log median, sigma^2)) rounded and clipped to [lo, hi]."""
    z = torch.randn(n, generator=gen, device=device, dtype=torch.float64)
    x = torch.exp(math.log(median) + sigma * z).round()
    return x.clamp(lo, hi).to(torch.int64)


def lengths_discrete(gen, n, values, device="cpu"):
    """Each length drawn uniformly from ``values``."""
    v = torch.as_tensor(values, dtype=torch.int64, device=device)
    idx = torch.randint(0, len(values), (n,), generator=gen, device=device)
    return v[idx]


# ---------------------------------------------------------------------------- score rows

def greedy_round(gen, B, D, V, alpha, dtype=torch.bfloat16, device="cpu", row_stride=None):
    """Target scores [B, D+1, V] (stored with ``row_stride`` >= V elements per row) and drafts
    [B, D] int32, with planted agreement of probability ``alpha`` (scalar or per-row tensor)."""
    z = torch.randn(B, D + 1, V, generator=gen, device=device, dtype=torch.float32)
    draft = torch.randint(0, V, (B, D), generator=gen, device=device, dtype=torch.int64)
    u = torch.rand(B, D, generator=gen, device=device, dtype=torch.float32)
    a = torch.as_tensor(alpha, dtype=torch.float32, device=device)
    if a.dim() == 1:
        a = a[:, None]
    plant = u < a
    raised = z[:, :D, :].amax(dim=-1) + 1.0
    old = z[:, :D, :].gather(-1, draft[..., None])[..., 0]
    z[:, :D, :].scatter_(-1, draft[..., None], torch.where(plant, raised, old)[..., None])
    return _strided(z.to(dtype), row_stride), draft.to(torch.int32)


def sampled_round(gen, B, D, V, temperature, sigma=0.5, dtype=torch.bfloat16, device="cpu",
                  row_stride=None, draft_candidates=0):
    """Target scores [B, D+1, V], draft-model scores [B, D, V] = target + N(0, sigma^2), drafts
    drawn from the draft model's softmax at ``temperature``, and uniforms [B, D+1] in [0, 1).
    With ``draft_candidates`` = k (0 < k < V) the draft model samples among its k highest scores
    only, as a draft model run with a top-k setting does."""
    z = torch.randn(B, D + 1, V, generator=gen, device=device, dtype=torch.float32)
    w = z[:, :D, :] + sigma * torch.randn(B, D, V, generator=gen, device=device,
                                          dtype=torch.float32)
    z = z.to(dtype)
    w = w.to(dtype)
    if 0 < draft_candidates < V:
        val, idx = torch.topk(w.to(torch.float64), draft_candidates, dim=-1)
        qk = torch.softmax(val / temperature, dim=-1)
        pick = torch.multinomial(qk.reshape(B * D, -1), 1, generator=gen).reshape(B, D)
        draft = idx.gather(-1, pick[..., None])[..., 0]
    else:
        q = torch.softmax(w.to(torch.float64) / temperature, dim=-1)
        draft = torch.multinomial(q.reshape(B * D, V), 1, generator=gen).reshape(B, D)
    uniforms = torch.rand(B, D + 1, generator=gen, device=device, dtype=torch.float32)
    return (_strided(z, row_stride), _strided(w, row_stride), draft.to(torch.int32), uniforms)


def _strided(x, row_stride):
    """Return ``x`` [.., V] viewed inside a buffer whose rows are ``row_stride`` elements apart."""
    V = x.shape[-1]
    if row_stride is None or row_stride == V:
        return x.contiguous()
    buf = torch.zeros(*x.shape[:-1], row_stride, dtype=x.dtype, device=x.device)
    buf[..., :V] = x
    return buf[..., :V]


# ---------------------------------------------------------------------------- K/V tags

def _mix(x):
    x = x & MASK32
    x = ((x >> 16) ^ x) * 0x45D9F3B & MASK32
    x = ((x >> 16) ^ x) * 0x45D9F3B & MASK32
    return (x >> 16) ^ x


def kv_tag(seq, layer, kv, head, position, token, head_dim, dtype, device="cpu"):
    """Tag values [..., head_dim] for broadcastable int64 index tensors.  Value = k/64 with
    k in [-128, 128) from an integer hash, exact in bf16 and fp32."""
    def t(v):
        return torch.as_tensor(v, dtype=torch.int64, device=device)
    h = _mix(t(seq) * 0x9E3779B1 + 0x1234567)
    h = _mix(h ^ (t(layer) * 0x85EBCA6B))
    h = _mix(h ^ (t(kv) * 0xC2B2AE35 + 7))
    h = _mix(h ^ (t(head) * 0x27D4EB2F))
    h = _mix(h ^ (t(position) * 0x165667B1))
    h = _mix(h ^ ((t(token) + 1) * 0x61C88647))
    e = torch.arange(head_dim, dtype=torch.int64, device=device)
    h = _mix(h[..., None] ^ (e * 0x2C1B3C6D + 0x9E37))
    k = ((h >> 8) & 0xFF) - 128
    return (k.to(torch.float32) / 64.0).to(dtype)


def write_tagged_columns(cache, row, col0, seq, positions, tokens):
    """Write tag values into ``cache`` [L, 2, B, H, S, hd] for one batch row: column col0 + i
    gets the K/V of (seq, positions[i], tokens[i]) for every layer, k/v and head."""
    L, _, _, H, _, hd = cache.shape
    n = len(positions)
    if n == 0:
        return
    dev = cache.device
    li = torch.arange(L, device=dev)[:, None, None, None]
    kv = torch.arange(2, device=dev)[None, :, None, None]
    hh = torch.arange(H, device=dev)[None, None, :, None]
    p = torch.as_tensor(positions, dtype=torch.int64, device=dev)[None, None, None, :]
    tk = torch.as_tensor(tokens, dtype=torch.int64, device=dev)[None, None, None, :]
    vals = kv_tag(seq, li, kv, hh, p, tk, hd, cache.dtype, device=dev)
    cache[:, :, row, :, col0:col0 + n, :] = vals


# ---------------------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    """One model-shaped workload: cache geometry, batch, draft length, vocabulary and rounds."""
    name: str
    layers: int
    heads: int
    head_dim: int
    kv_dtype: torch.dtype
    B: int
    D: int
    V: int
    logit_dtype: torch.dtype
    rounds: int
    mode: str                 # "greedy" | "sampled" | "pool"
    alpha: float = 0.7
    temperature: float = 1.0
    prompt: tuple = ("uniform", 5, 20)
    seed: int = 0

    @property
    def col_bytes(self):
        return self.head_dim * torch.tensor([], dtype=self.kv_dtype).element_size()

    @property
    def token_bytes(self):
        """K/V bytes of one token over all layers and heads (P_tok)."""
        return self.layers * 2 * self.heads * self.col_bytes

    def prompt_lengths(self, gen, device="cpu"):
        kind = self.prompt[0]
        if kind == "uniform":
            return lengths_uniform(gen, self.B, self.prompt[1], self.prompt[2], device)
        if kind == "lognormal":
            _, median, sigma, lo, hi = self.prompt
            return lengths_lognormal(gen, self.B, median, sigma, lo, hi, device)
        if kind == "discrete":
            return lengths_discrete(gen, self.B, self.prompt[1], device)
        raise ValueError(kind)

    def capacity(self, max_prompt, rounds=None):
        """Columns a cache needs for ``rounds`` rounds from prompts of at most ``max_prompt``."""
        r = self.rounds if rounds is None else rounds
        return int(max_prompt) + r * (self.D + 1) + self.D + 1


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 64, torch.float32, B=2, D=4, V=1000,
                     logit_dtype=torch.float32, rounds=3, mode="greedy", alpha=0.7,
                     prompt=("uniform", 5, 20), seed=0),
    "vicuna7b": Workload("vicuna7b", 32, 32, 128, torch.bfloat16, B=8, D=5, V=32000,
                         logit_dtype=torch.bfloat16, rounds=64, mode="greedy", alpha=0.7,
                         prompt=("uniform", 128, 1024), seed=1),
    "qwen3_8b": Workload("qwen3_8b", 36, 8, 128, torch.bfloat16, B=16, D=4, V=151936,
                         logit_dtype=torch.bfloat16, rounds=64, mode="greedy", alpha=0.6,
                         prompt=("lognormal", 512, 1.0, 32, 4096), seed=2),
    "glm4_9b": Workload("glm4_9b", 40, 2, 128, torch.bfloat16, B=32, D=6, V=151552,
                        logit_dtype=torch.bfloat16, rounds=32, mode="sampled",
                        temperature=0.7, prompt=("uniform", 1024, 8192), seed=3),
    "exspec_pool": Workload("exspec_pool", 32, 32, 128, torch.bfloat16, B=256, D=5, V=32000,
                            logit_dtype=torch.bfloat16, rounds=128, mode="pool",
                            prompt=("discrete", tuple(range(256, 2049, 256))), seed=4),
}
