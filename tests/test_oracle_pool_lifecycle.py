"""Pins of the oracle's SequencePool lifecycle ("Batch Speculative Decoding Done Right", section
2.3: a pool of active sequences, same-length ones grouped so that only mixed-length ones are
realigned).

The window grouping is pinned by brute force (the number of windowed batches is the largest number
of disjoint batch_size-row groups of span <= w), by the exact-length rule at window 0, and by
properties that follow from its definition; retirement and admission by hand examples; the first-fit
arena by a hand sequence; and the whole lifecycle by running every sequence alone: a pooled run must
commit, for every sequence, exactly the tokens it commits on its own.
"""
import itertools

import numpy as np
import pytest

import oracle.specdec_oracle as O
import specdec_testlib as testlib


# ------------------------------------------------------------------------- window grouping

def _brute_max_groups(lengths, bs, w):
    """Largest number of disjoint groups of bs rows, each of length span <= w (exhaustive)."""
    lengths = sorted(lengths)

    def best(rest):
        if len(rest) < bs:
            return 0
        x, others = rest[0], rest[1:]
        top = best(others)                       # the smallest row is in no group
        for comb in itertools.combinations(range(len(others)), bs - 1):
            if all(others[j] - x <= w for j in comb):
                left = [others[j] for j in range(len(others)) if j not in comb]
                top = max(top, 1 + best(left))
        return top

    return best(lengths)


def _check_window(lengths, bs, w):
    perm, off, uni, nw = O.group_by_window(lengths, bs, w)
    N = len(lengths)
    assert sorted(perm.tolist()) == list(range(N))
    assert off[0] == 0 and off[-1] == N
    L = np.asarray(lengths)
    for k in range(len(off) - 1):
        rows = perm[off[k]:off[k + 1]]
        if k < nw:
            assert len(rows) == bs and L[rows].max() - L[rows].min() <= w
            assert uni[k] == (L[rows].max() == L[rows].min())
        else:
            assert 1 <= len(rows) <= bs and uni[k] == 0
            assert k == len(off) - 2 or len(rows) == bs
    mins = [L[perm[off[k]:off[k + 1]]].min() for k in range(nw)]
    assert mins == sorted(mins)                               # windowed batches: ascending length
    left = perm[off[nw]:].tolist()
    assert left == sorted(left, key=lambda i: (lengths[i], i))   # leftovers in (length, index)
    # maximal: no bs leftovers span <= w (the smallest of them would have started a batch)
    ll = sorted(L[left].tolist())
    assert all(ll[i + bs - 1] - ll[i] > w for i in range(len(ll) - bs + 1))
    return perm, off, uni, nw


def test_window_hand_example():
    # (length, index) order: (3,1) (3,5) (4,2) (4,4) (5,0) (9,3) (10,6); bs 2, window 1:
    # [3,3] uniform, [4,4] uniform, 5 -> leftover (9 - 5 > 1), [9,10] windowed, leftover [0].
    perm, off, uni, nw = O.group_by_window([5, 3, 4, 9, 4, 3, 10], 2, 1)
    assert perm.tolist() == [1, 5, 2, 4, 3, 6, 0]
    assert off.tolist() == [0, 2, 4, 6, 7]
    assert uni.tolist() == [1, 1, 0, 0] and nw == 3


@pytest.mark.parametrize("seed", range(40))
def test_window_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(0, 8))
    bs = int(rng.integers(1, 4))
    w = int(rng.integers(0, 4))
    lengths = rng.integers(1, 7, size=N).tolist()
    _, _, _, nw = _check_window(lengths, bs, w)
    assert nw == _brute_max_groups(lengths, bs, w)


@pytest.mark.parametrize("seed", range(10))
def test_window_zero_is_exact_length_rule(seed):
    rng = np.random.default_rng(100 + seed)
    N, bs = int(rng.integers(0, 300)), int(rng.integers(1, 10))
    lengths = rng.integers(1, 12, size=N).tolist()
    p0, o0, u0, n0 = O.group_by_length(lengths, bs)
    p1, o1, u1, n1 = _check_window(lengths, bs, 0)
    assert p0.tolist() == p1.tolist() and o0.tolist() == o1.tolist()
    assert u0.tolist() == u1.tolist() and n0 == n1


def test_window_wide_takes_sorted_runs():
    rng = np.random.default_rng(7)
    lengths = rng.integers(1, 500, size=37).tolist()
    perm, off, uni, nw = _check_window(lengths, 8, 10 ** 6)
    assert nw == 4 and off.tolist() == [0, 8, 16, 24, 32, 37]
    assert perm.tolist() == sorted(range(37), key=lambda i: (lengths[i], i))


# ------------------------------------------------------------------------- schedule

def test_schedule_active_only_and_finished_reported_once():
    F, A, E, L = O.FREE, O.ACTIVE, O.FINISHED_EOS, O.FINISHED_LENGTH
    state = np.array([A, F, E, A, L, A, A], np.uint8)
    lens = np.array([4, 0, 9, 4, 3, 6, 4])
    r = O.pool_schedule(state, lens, 2, 0)
    assert r["perm"].tolist() == [0, 3, 6, 5]        # [4,4] uniform; leftovers 6 (len 4), 5 (6)
    assert r["offsets"].tolist() == [0, 2, 4] and r["uniform"].tolist() == [1, 0]
    assert r["num_windowed"] == 1 and r["num_active"] == 4
    assert r["finished"].tolist() == [2, 4] and r["reason"].tolist() == [E, L]
    assert r["state"].tolist() == [A, F, F, A, F, A, A]
    r2 = O.pool_schedule(r["state"], lens, 2, 0)
    assert r2["finished"].tolist() == []


def test_schedule_leftover_order():
    A = O.ACTIVE
    r = O.pool_schedule(np.array([A, A, A, A], np.uint8), np.array([7, 4, 4, 5]), 2, 0)
    # [4,4] (slots 1,2) uniform; leftovers by (length, slot): 5 (slot 3), 7 (slot 0)
    assert r["perm"].tolist() == [1, 2, 3, 0]


# ------------------------------------------------------------------------- retirement

def test_retire_cases():
    A, E, Lr = O.ACTIVE, O.FINISHED_EOS, O.FINISHED_LENGTH
    eos = 0
    ids = np.array([[5, 6, 7, 8, 3, 0, 9, 1, 1, 1, 1, 1],     # EOS at q=5 among the new tokens
                    [5, 6, 7, 8, 9, 9, 9, 9, 9, 9, 9, 9],     # limit 6 reached at q=5
                    [5, 6, 7, 0, 4, 0, 9, 9, 9, 9, 9, 9],     # EOS in the prompt does not count
                    [5, 6, 7, 8, 9, 0, 9, 9, 9, 9, 9, 9],     # EOS at the limit position
                    [5, 6, 7, 8, 9, 9, 9, 9, 9, 9, 9, 9]])    # still active
    before = np.array([4, 4, 4, 4, 4])
    after = np.array([7, 7, 7, 7, 7])
    limit = np.array([12, 6, 12, 6, 12])
    ln, st = O.retire(before, after, ids, range(5), limit, eos, np.full(5, A, np.uint8))
    assert ln.tolist() == [6, 6, 6, 6, 7]
    assert st.tolist() == [E, Lr, E, E, A]


# ------------------------------------------------------------------------- admission

def _empty_pool(S, ids_cap):
    z = np.zeros(S, np.int32)
    return (np.zeros(S, np.uint8), z.copy(), z.copy(), z.copy(), z.copy(),
            np.zeros((S, ids_cap), np.int32))


def test_admit_writes_and_errors():
    D = 3
    pool = _empty_pool(4, 20)
    st, col, cap, ln, lim, ids = O.pool_admit(*pool, [2, 0], [10, 0], [12, 8], [10, 6],
                                              [[4, 5, 6], [7]], D, 40)
    assert st.tolist() == [1, 0, 1, 0] and col.tolist() == [0, 0, 10, 0]
    assert cap.tolist() == [8, 0, 12, 0] and ln.tolist() == [1, 0, 3, 0]
    assert lim.tolist() == [6, 0, 10, 0]
    assert ids[2, :3].tolist() == [4, 5, 6] and ids[0, 0] == 7
    new = (st, col, cap, ln, lim, ids)
    bad = [
        (([2], [20], [12], [10], [[1]]), "range"),          # slot 2 is not free
        (([1, 1], [20, 30], [5, 5], [3, 3], [[1], [1]]), "range"),   # slot named twice
        (([1], [20], [5], [3], [[]]), "range"),             # empty prompt
        (([1], [20], [5], [3], [[1, 2, 3]]), "range"),      # prompt not shorter than the limit
        (([1], [38], [5], [3], [[1]]), "range"),            # range past the arena
        (([4], [20], [5], [3], [[1]]), "range"),            # slot out of range
        (([1], [20], [5], [4], [[1]]), "capacity"),         # limit + D - 1 = 6 > cap 5
        (([1], [5], [30], [18], [[1]]), "capacity"),        # limit + D = 21 > ids_cap 20
    ]
    for args, kind in bad:
        with pytest.raises(O.OracleError, match=kind):
            O.pool_admit(*new, *args[:4], args[4], D, 40)


# ------------------------------------------------------------------------- first-fit arena

def test_first_fit_sequence():
    a = O.FirstFitArena(10)
    assert [a.alloc(3), a.alloc(4), a.alloc(2)] == [0, 3, 7]
    a.free(3)
    assert a.free_cols() == 5 and a.largest_free() == 4
    with pytest.raises(O.OracleError):
        a.alloc(5)
    assert a.alloc(2) == 3 and a.alloc(1) == 5 and a.alloc(1) == 6 and a.alloc(1) == 9
    for c in (0, 3, 5, 6, 7, 9):
        a.free(c)
    assert a.alloc(10) == 0
    with pytest.raises(O.OracleError):
        a.free(4)


# ------------------------------------------------------------------------- whole lifecycle

D, V, EOS = testlib.D, testlib.V, testlib.EOS
_alone = testlib.alone


def _pooled(requests, S, bs, window, arena_cols):
    """Run the requests through a pool of S slots, admitting in arrival order into the lowest
    free slots; K/V columns carry the token id they belong to."""
    ids_cap = max(lim for _, lim in requests) + D + 1
    state, col, cap, ln, lim, ids = _empty_pool(S, ids_cap)
    arena = np.full((1, 2, 1, arena_cols, 1), -1.0)          # [L, 2, H, C, hd]
    alloc = O.FirstFitArena(arena_cols)
    seq_of, rnd = [-1] * S, [0] * S
    waiting = list(range(len(requests)))
    results = {}
    for _ in range(500):
        sch = O.pool_schedule(state, ln, bs, window)
        for s, why in zip(sch["finished"].tolist(), sch["reason"].tolist()):
            n = int(ln[s])
            kv = arena[0, 0, 0, col[s]:col[s] + n - 1, 0]
            assert kv.tolist() == ids[s, :n - 1].tolist()    # K/V of all but the pending token
            results[seq_of[s]] = (ids[s, :n].tolist(), why)
            alloc.free(int(col[s]))
        state = sch["state"]
        adm = []
        for s in range(S):
            if state[s] == O.FREE and waiting and s not in [x[0] for x in adm]:
                q = waiting[0]
                need = requests[q][1] + D - 1
                try:
                    c = alloc.alloc(need)
                except O.OracleError:
                    break
                adm.append((s, c, need, q))
                waiting.pop(0)
        if adm:
            state, col, cap, ln, lim, ids = O.pool_admit(
                state, col, cap, ln, lim, ids, [x[0] for x in adm], [x[1] for x in adm],
                [x[2] for x in adm], [requests[x[3]][1] for x in adm],
                [requests[x[3]][0] for x in adm], D, arena_cols)
            for s, c, _, q in adm:
                seq_of[s], rnd[s] = q, 0
                p = requests[q][0]
                arena[0, :, 0, c:c + len(p) - 1, 0] = p[:-1]       # prefill K/V
        if not waiting and not (state == O.ACTIVE).any():
            break
        if adm:
            continue                                           # newly admitted: schedule again
        perm, off = sch["perm"], sch["offsets"]
        before = ln.copy()
        for k in range(len(off) - 1):
            rows = perm[off[k]:off[k + 1]].tolist()
            logits = np.stack([testlib.round_scores(seq_of[s], rnd[s])[0] for s in rows])
            draft = np.stack([testlib.round_scores(seq_of[s], rnd[s])[1] for s in rows])
            a, y = O.verify_greedy(logits, draft)
            if sch["uniform"][k]:
                for i, s in enumerate(rows):               # verified in place in the slot
                    n = int(ln[s])
                    arena[0, :, 0, col[s] + n - 1:col[s] + n + a[i], 0] = (
                        [ids[s, n - 1]] + draft[i, :a[i]].tolist())
                    ids[s, n:n + a[i]] = draft[i, :a[i]]
                    ids[s, n + a[i]] = y[i]
                    ln[s] = n + a[i] + 1
            else:
                scratch = np.full((1, 2, len(rows), 1, int(ln.max()) + 2 * D + 2, 1), -2.0)
                sc, W, _, _, _ = O.pool_gather(arena, col, ln, rows, scratch, 0, ids)
                for i, s in enumerate(rows):               # the verification pass writes K/V
                    sc[0, :, i, 0, W - 1:W + D, 0] = [ids[s, int(ln[s]) - 1]] + draft[i].tolist()
                arena, ln, ids = O.pool_append(arena, col, ln, rows, sc, W, a, y, draft, ids)
        act = perm.tolist()
        ln, state = O.retire(before, ln, ids, act, lim, EOS, state)
        for s in act:
            rnd[s] += 1
    return results


@pytest.mark.parametrize("S,bs,window,seed", [(4, 2, 0, 1), (6, 3, 2, 2), (5, 2, 100, 3),
                                              (3, 1, 0, 4)])
def test_pooled_equals_alone(S, bs, window, seed):
    rng = np.random.default_rng(seed)
    requests = []
    for _ in range(12):
        n = int(rng.integers(2, 9))
        requests.append((rng.integers(1, V, size=n).tolist(), n + int(rng.integers(2, 16))))
    results = _pooled(requests, S, bs, window, arena_cols=60)
    assert sorted(results) == list(range(len(requests)))
    for q, (prompt, limit) in enumerate(requests):
        assert results[q] == _alone(prompt, limit, q)
