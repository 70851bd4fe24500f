"""Side-by-side round runner for the GPU path and the CPU oracle (test infrastructure)."""
import numpy as np
import torch

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth


def host_bits(t):
    """Host copy of a cache tensor; bf16 as its int16 bit patterns (values are only moved)."""
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).cpu().numpy()


def eqspec_rounds(L, H, hd, kv_dtype, B, D, V, rounds, prompt_lo, prompt_hi, seed,
                  copy_engine=0, alpha=0.6, logit_dtype=torch.float32, cap_extra=0,
                  check_full_dst=True, in_place=False, pdl=False, scheduled=True):
    """Greedy verify + realign for ``rounds`` rounds with tagged K/V; every round is compared
    with the oracle: accept lengths, tokens, lengths, width, ids, mask, position IDs, and the
    whole destination cache (the oracle leaves pad columns as they were, and so must the
    kernel).  With ``in_place`` the cache is one buffer realigned in place: the expected result
    is the oracle's realignment into a copy of the source.  ``scheduled``: the realignment takes
    work items from its scheduling words (checked back at zero after every call), else every
    CTA a fixed share.  Returns the per-round accept lengths."""
    from speculative_decoding_specdec_gb300.engine import EqspecBatch
    gen = synth.make_gen(seed)
    n0 = synth.lengths_uniform(gen, B, prompt_lo, prompt_hi)
    prompts = [torch.randint(0, V, (int(n),), generator=gen).tolist() for n in n0]
    cap = int(n0.max()) + rounds * (D + 1) + D + 1 + cap_extra
    eng = EqspecBatch(L, H, hd, kv_dtype, B, D, cap, rounds, in_place=in_place, pdl=pdl,
                      scheduled=scheduled)
    W = eng.start(prompts)
    eng.kv[0].fill_(-3.0)
    if not in_place:
        eng.kv[1].fill_(-5.0)
    toks = [list(p) for p in prompts]
    for b in range(B):
        synth.write_tagged_columns(eng.cache, b, W - len(toks[b]), b,
                                   list(range(len(toks[b]) - 1)), toks[b][:-1])
    ids = eng.ids[0].cpu().numpy()
    n = np.array([len(t) for t in toks])
    history = []
    for _ in range(rounds):
        logits, draft = synth.greedy_round(gen, B, D, V, alpha, dtype=logit_dtype)
        for b in range(B):
            synth.write_tagged_columns(eng.cache, b, W - 1, b,
                                       list(range(len(toks[b]) - 1, len(toks[b]) + D)),
                                       [toks[b][-1]] + draft[b].tolist())
        src = host_bits(eng.cache)
        dst_before = src.copy() if in_place else host_bits(eng.kv[1 - eng.cur])
        dd = draft.cuda()
        eng.verify_greedy(logits.cuda(), dd)
        eng.realign(dd, copy_engine=copy_engine)
        torch.cuda.synchronize()
        assert int(eng.status.item()) == 0
        if scheduled:
            assert eng.sched_words.tolist() == [0, 0]
        a, y = O.verify_greedy(logits.double().numpy(), draft.numpy())
        kv, ids, mask, pos, n, W = O.realign(src, dst_before, n, W, a, y, draft.numpy(), ids, 0)
        np.testing.assert_array_equal(eng.accept_len.cpu().numpy(), a)
        np.testing.assert_array_equal(eng.out_token.cpu().numpy(), y)
        assert int(eng.width.item()) == W
        np.testing.assert_array_equal(eng.n_committed.cpu().numpy(), n)
        np.testing.assert_array_equal(eng.ids[eng.cur].cpu().numpy(), ids)
        np.testing.assert_array_equal(eng.mask[eng.cur].cpu().numpy(), mask)
        np.testing.assert_array_equal(eng.pos[eng.cur].cpu().numpy(), pos)
        assert O.check_invariants(eng.mask[eng.cur].cpu().numpy(), eng.pos[eng.cur].cpu().numpy(),
                                  n, W) == []
        got = host_bits(eng.cache)
        if check_full_dst:
            np.testing.assert_array_equal(got, kv)
        else:
            for b in range(B):
                lo = W - int(n[b])
                np.testing.assert_array_equal(got[:, :, b, :, lo:W - 1], kv[:, :, b, :, lo:W - 1])
        for b in range(B):
            toks[b] += draft[b, :a[b]].tolist() + [int(y[b])]
        history.append(a)
    return history


# ------------------------------------------------------------------ SequencePool lifecycle runs

D, V, EOS = 3, 24, 0   # draft length, vocabulary and end-of-sequence token of the lifecycle runs


def round_scores(seq, r):
    """The fp32 scores [D+1, V] and draft [D] of round r of sequence seq: the same whether the
    sequence runs in a pool or alone."""
    logits, draft = synth.greedy_round(synth.make_gen(7919 * seq + r), 1, D, V, 0.7,
                                       dtype=torch.float32)
    return logits[0], draft[0]


def alone(prompt, limit, seq):
    """The tokens a sequence commits when it runs by itself, and why it stops (oracle only)."""
    toks, r = list(prompt), 0
    while True:
        logits, draft = round_scores(seq, r)
        a, y = O.verify_greedy(logits.double().numpy()[None], draft.numpy()[None])
        for t in draft[:a[0]].tolist() + [int(y[0])]:
            toks.append(int(t))
            if t == EOS or len(toks) >= limit:
                return toks, (O.FINISHED_EOS if t == EOS else O.FINISHED_LENGTH)
        r += 1
