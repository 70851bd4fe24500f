"""Pins for the CPU oracle: what the pages and the mathematics fix, independent of the oracle.

Sources: "Inference Engineering: Part 5/8: When Speculative Decoding Backfires" (worked greedy
example, 40/60 sampling example, bonus token and 1..D+1 range, discard after the first rejection);
"Batch Speculative Decoding Done Right" section 2.1 (invariants), 2.2 (EQSPEC), 2.3 (EXSPEC).
"""
import json
import os

import numpy as np
import pytest
import torch
from scipy import stats

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def onehot_scores(choices, V, rng=None):
    """Score rows whose unique maximum is at each of ``choices``."""
    s = np.zeros((len(choices), V)) if rng is None else rng.normal(size=(len(choices), V))
    for j, c in enumerate(choices):
        s[j, c] = s[j].max() + 1.0
    return s


# ------------------------------------------------------------------------------------- greedy

def test_greedy_worked_example():
    g = golden("greedy_worked_example.json")
    tok = {w: i for i, w in enumerate(g["vocab"])}
    V = len(g["vocab"])
    draft = np.array([[tok[w] for w in g["draft"]]])
    logits = onehot_scores([tok[w] for w in g["target_choice"]], V)[None]
    a, y = O.verify_greedy(logits, draft)
    assert a[0] == g["expect_accept_len"]
    assert y[0] == tok[g["expect_out_token"]]
    assert a[0] + 1 == g["expect_committed_this_cycle"]


@pytest.mark.parametrize("case", golden("cycle_counts.json")["cases"])
def test_cycle_counts(case):
    D = case["D"]
    V = 50
    rng = np.random.default_rng(1)
    draft = rng.integers(0, V, size=D)
    fr = case["first_rejection"]           # 1-based position of the first rejection, or None
    choices = list(draft) + [7]
    if fr is not None:
        choices[fr - 1] = (draft[fr - 1] + 1) % V
        # later positions agree with the draft again: they must still be discarded
    logits = onehot_scores(choices, V, rng)[None]
    a, y = O.verify_greedy(logits, draft[None])
    assert a[0] == case["expect_accepted"]
    assert a[0] + 1 == case["expect_added"]
    assert y[0] == choices[a[0]]


def _greedy_brute(logits, draft):
    """Independent restatement: strict '>' scan for the choice, explicit leading-match count."""
    B, Dp1, V = logits.shape
    out_a, out_y = [], []
    for b in range(B):
        ch = []
        for j in range(Dp1):
            best_v, best_i = None, None
            for v in range(V):
                s = float(logits[b, j, v])
                if best_v is None or s > best_v:
                    best_v, best_i = s, v
            ch.append(best_i)
        k = 0
        while k < Dp1 - 1 and ch[k] == draft[b][k]:
            k += 1
        out_a.append(k)
        out_y.append(ch[k])
    return out_a, out_y


def test_greedy_brute_force_with_ties():
    rng = np.random.default_rng(2)
    B, D, V = 300, 3, 6
    logits = rng.integers(0, 3, size=(B, D + 1, V)).astype(np.float64)   # many ties
    draft = rng.integers(0, V, size=(B, D))
    # make leading agreement common
    for b in range(B):
        for j in range(D):
            if rng.random() < 0.6:
                draft[b, j] = int(np.argmax(logits[b, j]))
    a, y = O.verify_greedy(logits, draft)
    ba, by = _greedy_brute(logits, draft)
    assert list(a) == ba and list(y) == by


def test_greedy_cycle_invariants_and_discard():
    gen = synth.make_gen(3)
    B, D, V = 64, 5, 97
    logits, draft = synth.greedy_round(gen, B, D, V, 0.6, dtype=torch.float32)
    L = logits.double().numpy()
    dr = draft.numpy()
    a, y = O.verify_greedy(L, dr)
    assert ((a >= 0) & (a <= D)).all()              # commits 1..D+1 tokens
    for b in range(B):
        if a[b] < D:
            assert y[b] != dr[b, a[b]]               # replacement differs from the rejected draft
        assert y[b] == int(np.argmax(L[b, a[b]]))    # bonus iff all accepted: row D
    # drafts after the first rejection do not change anything
    dr2 = dr.copy()
    for b in range(B):
        if a[b] + 1 < D:
            dr2[b, a[b] + 1:] = (dr2[b, a[b] + 1:] + 1) % V
    a2, y2 = O.verify_greedy(L, dr2)
    assert (a2 == a).all() and (y2 == y).all()


def test_greedy_planted_acceptance_geometric():
    gen = synth.make_gen(4)
    B, D, V = 4000, 4, 64
    logits, draft = synth.greedy_round(gen, B, D, V, 0.7, dtype=torch.float32)
    a, _ = O.verify_greedy(logits.double().numpy(), draft.numpy())
    # P(a >= k) = P(first k planted or draft hits the argmax) ~ (0.7 + 0.3/64)^k
    for k in range(1, D + 1):
        p = (0.7 + 0.3 / V) ** k
        frac = (a >= k).mean()
        assert abs(frac - p) < 4 * np.sqrt(p * (1 - p) / B) + 1e-3


# ------------------------------------------------------------------------------------ sampled

def test_sampling_40_60_example():
    g = golden("sampling_40_60.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    T = 0.5
    tl = np.stack([T * np.log(p), T * np.log(p)])[None]      # softmax(scores / T) == p
    dl = (T * np.log(q))[None, None]
    for x in (0, 1):
        _, _, _, tr = O.verify_sample(tl, dl, np.array([[x]]), np.array([[0.999, 0.5]]), T)
        assert min(1.0, tr["ratio"][0, 0]) == pytest.approx(g["expect_accept_prob"][x], abs=1e-12)
    a, y, res, _ = O.verify_sample(tl, dl, np.array([[0]]), np.array([[0.7, 0.01]]), T)
    assert a[0] == 0 and y[0] == 1                          # every replacement is 'life'
    np.testing.assert_allclose(res[0], g["expect_residual"], atol=1e-12)
    a, _, _, _ = O.verify_sample(tl, dl, np.array([[0]]), np.array([[0.3, 0.5]]), T)
    assert a[0] == 1


def _sample_trials(p_rows, q_rows, n, T, seed):
    """Run n independent one-row verifications with drafts drawn from q (test-side sampling)."""
    rng = np.random.default_rng(seed)
    D = len(q_rows)
    V = len(p_rows[0])
    tl = np.stack([T * np.log(r) for r in p_rows])
    dl = np.stack([T * np.log(r) for r in q_rows])
    draft = np.stack([rng.choice(V, size=n, p=q_rows[j]) for j in range(D)], axis=1)
    u = rng.random((n, D + 1))
    a, y, _, _ = O.verify_sample(np.broadcast_to(tl, (n,) + tl.shape),
                                 np.broadcast_to(dl, (n,) + dl.shape), draft, u, T)
    first = np.where(a >= 1, draft[:, 0], y)
    return a, y, draft, first


def test_sampling_40_60_split():
    g = golden("sampling_40_60.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    n = 20000
    a, y, draft, first = _sample_trials([p, p], [q], n, 1.0, 5)
    frac = (first == 1).mean()
    assert abs(frac - g["expect_output_split"][1]) < 4 * np.sqrt(0.24 / n)
    acc = (a >= 1)
    assert abs(acc[draft[:, 0] == 0].mean() - 0.5) < 4 * np.sqrt(0.25 / (draft[:, 0] == 0).sum())
    assert acc[draft[:, 0] == 1].all()


def test_distribution_preservation_chi_square():
    rng = np.random.default_rng(6)
    V, n, T = 8, 30000, 0.7
    p0 = rng.dirichlet(np.ones(V))
    p1 = rng.dirichlet(np.ones(V))
    q0 = rng.dirichlet(np.ones(V))
    a, y, draft, first = _sample_trials([p0, p1], [q0], n, T, 7)
    counts = np.bincount(first, minlength=V)
    assert stats.chisquare(counts, p0 * n).pvalue > 1e-3
    bonus = y[a == 1]                                   # all (D=1) accepted: bonus ~ p_D
    assert stats.chisquare(np.bincount(bonus, minlength=V), p1 * len(bonus)).pvalue > 1e-3
    # closed form: P(accept) = sum_x q(x) min(1, p/q) = sum_x min(p, q)
    pacc = np.minimum(p0, q0).sum()
    assert abs((a == 1).mean() - pacc) < 4 * np.sqrt(pacc * (1 - pacc) / n)


def test_q_equal_p_always_accepts():
    gen = synth.make_gen(8)
    B, D, V = 50, 4, 33
    z = torch.randn(B, D + 1, V, generator=gen, dtype=torch.float64).numpy()
    draft = np.random.default_rng(9).integers(0, V, size=(B, D))
    u = np.random.default_rng(10).random((B, D + 1))
    a, y, res, tr = O.verify_sample(z, z[:, :D], draft, u, 0.9)
    assert (a == D).all()
    np.testing.assert_allclose(tr["ratio"], 1.0, rtol=0, atol=1e-15)


def test_residual_is_normalised_positive_part():
    gen = synth.make_gen(11)
    tl, dl, draft, u = synth.sampled_round(gen, 40, 3, 50, 0.7, dtype=torch.float32)
    tl, dl = tl.double().numpy(), dl.double().numpy()
    a, y, res, tr = O.verify_sample(tl, dl, draft.numpy(), u.double().numpy(), 0.7)
    assert (res >= 0).all()
    np.testing.assert_allclose(res.sum(1), 1.0, atol=1e-12)
    for b in range(40):
        if a[b] < 3:
            p = np.exp(tl[b, a[b]] / 0.7); p /= p.sum()
            q = np.exp(dl[b, a[b]] / 0.7); q /= q.sum()
            assert (res[b][p <= q] == 0).all()          # no mass where nothing is missing
            assert res[b, y[b]] > 0
        assert tr["cdf_lo"][b] <= tr["t"][b] < tr["cdf_hi"][b]


# ------------------------------------------------------------------------------------ realign

def _round_state(B, D, L, H, hd, S, gen, V=40, dtype=torch.float32):
    """Prompts of random length, tagged cache, and the per-sequence token lists."""
    n = synth.lengths_uniform(gen, B, 1, 6).numpy()
    W = int(n.max())
    toks = [list(torch.randint(0, V, (int(n[b]),), generator=gen).numpy()) for b in range(B)]
    cache = torch.zeros(L, 2, B, H, S, hd, dtype=dtype)
    ids = np.zeros((B, S), dtype=np.int32)
    for b in range(B):
        c0 = W - int(n[b])
        ids[b, c0:W] = toks[b]
        synth.write_tagged_columns(cache, b, c0, b, list(range(int(n[b]) - 1)), toks[b][:-1])
    return n, W, toks, cache.numpy(), ids


def _simulate(rounds, B=4, D=3, L=2, H=2, hd=8, V=40, seed=12, plan_hook=None):
    gen = synth.make_gen(seed)
    S = 6 + rounds * (D + 1) + D + 1
    n, W, toks, A, ids = _round_state(B, D, L, H, hd, S, gen, V)
    Bbuf = np.full_like(A, 99.0)
    for r in range(rounds):
        logits, draft = synth.greedy_round(gen, B, D, V, 0.6, dtype=torch.float32)
        dr = draft.numpy()
        # synthetic verification pass: K/V of [pending, d_1..d_D] at [W-1, W+D)
        At = torch.from_numpy(A)
        for b in range(B):
            pend = toks[b][-1]
            synth.write_tagged_columns(At, b, W - 1, b, list(range(int(n[b]) - 1, int(n[b]) + D)),
                                       [pend] + list(dr[b]))
        a, y = O.verify_greedy(logits.double().numpy(), dr)
        kv, ids, mask, pos, n2, W2 = O.realign(A, Bbuf, n, W, a, y, dr, ids, pad_id=0)
        for b in range(B):
            toks[b] = toks[b] + list(dr[b, :a[b]]) + [int(y[b])]
        assert O.check_invariants(mask, pos, n2, W2) == []
        yield dict(kv=kv, ids=ids, mask=mask, pos=pos, n=n2, W=W2, toks=toks, a=a, L=L, H=H,
                   hd=hd, B=B)
        A, Bbuf, n, W = kv, A, n2, W2


def _rebuild(st):
    """From-scratch cache content of every row: K/V of each committed token but the last."""
    for b in range(st["B"]):
        t = st["toks"][b]
        assert len(t) == st["n"][b]
        ref = torch.zeros(st["L"], 2, 1, st["H"], len(t) - 1, st["hd"])
        synth.write_tagged_columns(ref, 0, 0, b, list(range(len(t) - 1)), t[:-1])
        c0 = st["W"] - len(t)
        got = st["kv"][:, :, b, :, c0:st["W"] - 1, :]
        np.testing.assert_array_equal(got, ref[:, :, 0].numpy())
        np.testing.assert_array_equal(st["ids"][b, c0:st["W"]], t)


def test_realign_rebuild_from_scratch():
    for st in _simulate(8):
        _rebuild(st)


def test_realign_worked_example_text():
    g = golden("greedy_worked_example.json")
    tok = {w: i for i, w in enumerate(g["vocab"])}
    V = len(g["vocab"])
    prompt = [tok[w] for w in g["committed"]]
    other = [tok["For"], tok["college"]]                   # a second, shorter row
    B, D, S = 2, 4, 16
    n = np.array([len(prompt), len(other)])
    W = 4
    ids = np.zeros((B, S), dtype=np.int32)
    ids[0, 0:4] = prompt
    ids[1, 2:4] = other
    draft = np.array([[tok[w] for w in g["draft"]], [tok["x"]] * 4])
    logits = np.stack([onehot_scores([tok[w] for w in g["target_choice"]], V),
                       onehot_scores([tok["and"]] * 5, V)])
    a, y = O.verify_greedy(logits, draft)
    kv = np.zeros((1, 2, B, 1, S, 2))
    _, ids2, mask, pos, n2, W2 = O.realign(kv, kv, n, W, a, y, draft, ids, pad_id=0)
    assert list(n2) == [7, 3] and W2 == 7
    assert list(ids2[0, :7]) == [tok[w] for w in g["expect_text_after"]]
    assert list(ids2[1, :7]) == [0, 0, 0, 0, tok["For"], tok["college"], tok["and"]]
    assert list(pos[1, :7]) == [0, 0, 0, 0, 0, 1, 2]
    assert O.check_invariants(mask, pos, n2, W2) == []


def test_realign_capacity_and_range_errors():
    kv = np.zeros((1, 2, 2, 1, 10, 2))
    small = np.zeros((1, 2, 2, 1, 8, 2))
    args = dict(n_committed=np.array([3, 2]), width=3, accept_len=np.array([2, 0]),
                out_token=np.array([1, 1]), draft=np.zeros((2, 3), int),
                ids_src=np.zeros((2, 10), np.int32))
    O.realign(kv, kv, **args)
    with pytest.raises(O.OracleError):
        O.realign(kv, small, **args)                       # W' + D = 6 + 3 > 8
    with pytest.raises(O.OracleError):
        O.realign(kv, kv, **{**args, "accept_len": np.array([4, 0])})


def test_invariant_checker_catches_violations():
    mask = np.array([[0, 1, 1], [1, 1, 1]], np.uint8)
    pos = np.array([[0, 0, 1], [0, 1, 2]])
    assert O.check_invariants(mask, pos, [2, 3], 3) == []
    assert O.check_invariants(mask, np.array([[0, 1, 2], [0, 1, 2]]), [2, 3], 3)   # pos from 1
    assert O.check_invariants(np.array([[1, 1, 0], [1, 1, 1]]), pos, [2, 3], 3)    # not right-aligned


# ------------------------------------------------------------------------------- planted mistakes

def test_planted_shift_error_is_caught(monkeypatch):
    real = O.realign_plan

    def off_by_one(*a, **k):
        n_new, w_new, src_lo, dst_lo, keep = real(*a, **k)
        return n_new, w_new, src_lo + 1, dst_lo, keep - 1 + 1     # reads one column late
    monkeypatch.setattr(O, "realign_plan", off_by_one)
    with pytest.raises(AssertionError):
        for st in _simulate(3):
            _rebuild(st)


def test_planted_residual_sign_error_is_caught(monkeypatch):
    real = np.maximum

    class NP:
        def __getattr__(self, k):
            return getattr(np, k)

        @staticmethod
        def maximum(x, y):
            return real(x, -y)                                  # max(0, q - p) instead
    monkeypatch.setattr(O, "np", NP())
    rng = np.random.default_rng(6)
    V, n = 8, 30000
    p0, p1, q0 = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    a, y, draft, first = _sample_trials([p0, p1], [q0], n, 0.7, 7)
    assert stats.chisquare(np.bincount(first, minlength=V), p0 * n).pvalue < 1e-3


def test_planted_all_matches_count_is_caught(monkeypatch):
    def count_all(logits, draft):
        L = np.asarray(logits, dtype=np.float64)
        ch = L.argmax(-1)
        a = (ch[:, :-1] == np.asarray(draft)).sum(1).astype(np.int32)
        return a, ch[np.arange(len(a)), a].astype(np.int32)
    monkeypatch.setattr(O, "verify_greedy", count_all)
    with pytest.raises(AssertionError):
        test_cycle_counts(golden("cycle_counts.json")["cases"][2])


# ------------------------------------------------------------------------------------ grouping

def _check_grouping(lengths, bs):
    perm, off, uni, nu = O.group_by_length(lengths, bs)
    N = len(lengths)
    assert sorted(perm.tolist()) == list(range(N))
    assert off[0] == 0 and off[-1] == N and len(uni) == len(off) - 1
    assert list(uni[:nu]) == [1] * nu and list(uni[nu:]) == [0] * (len(uni) - nu)
    lens = np.asarray(lengths)
    left = []
    for k in range(len(uni)):
        rows = perm[off[k]:off[k + 1]]
        if uni[k]:
            assert len(rows) == bs and len(set(lens[rows])) == 1
            assert list(rows) == sorted(rows)
        else:
            left.extend(rows.tolist())
            assert 1 <= len(rows) <= bs
            if k < len(uni) - 1:
                assert len(rows) == bs
    assert left == sorted(left, key=lambda i: (lens[i], i))          # (length, index) order
    for v in set(lens.tolist()):
        c = int((lens == v).sum())
        assert sum(1 for i in left if lens[i] == v) == c % bs
        # the uniform rows of a length are its lowest indices
        all_v = sorted(np.nonzero(lens == v)[0].tolist())
        uni_v = [i for k in range(nu) for i in perm[off[k]:off[k + 1]] if lens[i] == v]
        assert sorted(uni_v) == all_v[:len(uni_v)]
    lens_u = [lens[perm[off[k]]] for k in range(nu)]
    assert lens_u == sorted(lens_u)


@pytest.mark.parametrize("seed", range(20))
def test_group_by_length_properties(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(0, 40))
    bs = int(rng.integers(1, 6))
    lengths = rng.integers(1, 5, size=N)
    _check_grouping(lengths, bs)


def test_group_by_length_tiny_exact():
    perm, off, uni, nu = O.group_by_length([3, 1, 3, 3, 1], 2)
    # length 1: rows 1, 4 -> one uniform batch; length 3: rows 0, 2 uniform, 3 left over
    assert perm.tolist() == [1, 4, 0, 2, 3]
    assert off.tolist() == [0, 2, 4, 5] and uni.tolist() == [1, 1, 0] and nu == 2


# ------------------------------------------------------------------------------------ pool

def test_pool_gather_append_rebuild():
    """Mixed rows gathered from unpadded slots, verified and appended back equal a from-scratch
    rebuild of each sequence."""
    gen = synth.make_gen(13)
    L, H, hd, D, V = 2, 2, 4, 3, 30
    S = 5
    cap = 40
    n = np.array([3, 5, 2, 5, 4])
    slot_cols = np.arange(S) * cap
    arena = torch.zeros(L, 2, 1, H, S * cap, hd)
    toks = [list(torch.randint(0, V, (int(n[s]),), generator=gen).numpy()) for s in range(S)]
    for s in range(S):
        synth.write_tagged_columns(arena, 0, int(slot_cols[s]), s, list(range(n[s] - 1)),
                                   toks[s][:-1])
    arena = arena[:, :, 0].numpy()
    pool_ids = np.zeros((S, cap), np.int32)
    for s in range(S):
        pool_ids[s, :n[s]] = toks[s]
    for _ in range(4):
        rows = [4, 0, 2]
        scratch = np.full((L, 2, 3, H, 12 + D, hd), 7.0)
        sc, W, ids, mask, pos = O.pool_gather(arena, slot_cols, n, rows, scratch, 0, pool_ids)
        assert O.check_invariants(mask, pos, n[rows], W) == []
        for i, s in enumerate(rows):
            assert list(ids[i, W - n[s]:W]) == toks[s]
        logits, draft = synth.greedy_round(gen, 3, D, V, 0.6, dtype=torch.float32)
        dr = draft.numpy()
        sct = torch.from_numpy(sc)
        for i, s in enumerate(rows):
            synth.write_tagged_columns(sct, i, W - 1, s, list(range(n[s] - 1, n[s] + D)),
                                       [toks[s][-1]] + list(dr[i]))
        a, y = O.verify_greedy(logits.double().numpy(), dr)
        arena, n, pool_ids = O.pool_append(arena, slot_cols, n, rows, sct.numpy(), W, a, y, dr,
                                           pool_ids)
        for i, s in enumerate(rows):
            toks[s] = toks[s] + list(dr[i, :a[i]]) + [int(y[i])]
        for s in range(S):
            ref = torch.zeros(L, 2, 1, H, n[s] - 1, hd)
            synth.write_tagged_columns(ref, 0, 0, s, list(range(n[s] - 1)), toks[s][:-1])
            c0 = int(slot_cols[s])
            np.testing.assert_array_equal(arena[:, :, :, c0:c0 + n[s] - 1], ref[:, :, 0].numpy())
            assert list(pool_ids[s, :n[s]]) == toks[s]
