"""SequencePool lifecycle on the GPU against the CPU oracle: the device schedule (window grouping of
the active slots, finished slots reported once and freed), admission, retirement inside the append,
and a whole pool run in which every sequence must commit exactly the tokens it commits alone."""
import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
import specdec_testlib as testlib
from speculative_decoding_specdec_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENT = -7


def _i32(x):
    return torch.as_tensor(np.asarray(x), dtype=torch.int32, device=DEV)


def _u8(x):
    return torch.as_tensor(np.asarray(x), dtype=torch.uint8, device=DEV)


def gpu_schedule(state, lens, bs, window):
    import speculative_decoding_specdec_gb300.specdec as sd
    S = len(state)
    st = _u8(state)
    ln = _i32(lens)
    out = dict(perm=torch.full((max(S, 1),), SENT, dtype=torch.int32, device=DEV),
               offsets=torch.full((S + 1,), SENT, dtype=torch.int32, device=DEV),
               uniform=torch.full((max(S, 1),), 77, dtype=torch.uint8, device=DEV),
               finished=torch.full((max(S, 1),), SENT, dtype=torch.int32, device=DEV),
               reason=torch.full((max(S, 1),), 77, dtype=torch.uint8, device=DEV),
               counts=torch.full((4,), SENT, dtype=torch.int32, device=DEV))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd.pool_schedule(st, ln, bs, window, out["perm"], out["offsets"], out["uniform"],
                     out["finished"], out["reason"], out["counts"], status)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["state"] = st.cpu().numpy()
    res["status"] = int(status.item())
    return res


def check_schedule(state, lens, bs, window):
    g = gpu_schedule(state, lens, bs, window)
    e = O.pool_schedule(state, lens, bs, window)
    assert g["status"] == 0
    nb = len(e["offsets"]) - 1
    na, nf = e["num_active"], len(e["finished"])
    assert g["counts"].tolist() == [nb, e["num_windowed"], na, nf]
    np.testing.assert_array_equal(g["perm"][:na], e["perm"])
    np.testing.assert_array_equal(g["offsets"][:nb + 1], e["offsets"])
    np.testing.assert_array_equal(g["uniform"][:nb], e["uniform"])
    np.testing.assert_array_equal(g["finished"][:nf], e["finished"])
    np.testing.assert_array_equal(g["reason"][:nf], e["reason"])
    np.testing.assert_array_equal(g["state"], e["state"])
    # nothing past the counts is written
    assert (g["perm"][na:] == SENT).all() and (g["offsets"][nb + 1:] == SENT).all()
    assert (g["uniform"][nb:] == 77).all() and (g["finished"][nf:] == SENT).all()
    return e


@pytest.mark.parametrize("S,bs,window,seed,hi", [
    (0, 8, 0, 1, 10),            # empty pool
    (1, 1, 0, 2, 10),
    (7, 3, 1, 3, 6),
    (256, 8, 0, 4, 2048),        # the pool workload's shape, exact lengths
    (256, 8, 0, 5, 8),           # many equal lengths: mostly uniform batches
    (256, 8, 64, 6, 2048),       # windowed
    (1000, 16, 3, 7, 40),
    (4096, 8, 0, 8, 50),         # largest pool
    (4096, 64, 100, 9, 1 << 20), # lengths up to the limit
    (4096, 4096, 10 ** 6, 10, 9),
    (300, 1, 0, 11, 30),         # batch size 1: every row its own uniform batch
    (33, 40, 0, 12, 5),          # batch larger than the pool: all leftovers
])
def test_schedule_matches_oracle(S, bs, window, seed, hi):
    rng = np.random.default_rng(seed)
    state = rng.choice(np.array([0, 1, 1, 1, 1, 2, 3], np.uint8), size=S)
    lens = rng.integers(1, hi, size=S).astype(np.int32)
    lens[state == O.FREE] = rng.integers(0, 3, size=int((state == O.FREE).sum()))  # any value
    check_schedule(state, lens, bs, window)


def test_schedule_all_active_discrete_lengths():
    """The pool workload's length mix: 256 sequences over 8 discrete lengths."""
    gen = synth.make_gen(3)
    lens = synth.lengths_discrete(gen, 256, [256, 468, 680, 892, 1104, 1316, 1528, 2048]).numpy()
    state = np.ones(256, np.uint8)
    for w in (0, 1, 300, 10 ** 6):
        e = check_schedule(state, lens.astype(np.int32), 8, w)
        assert e["num_active"] == 256


def test_schedule_errors_write_nothing():
    state = np.array([1, 1, 4, 1], np.uint8)               # state 4 is not a state
    g = gpu_schedule(state, np.array([3, 3, 3, 3], np.int32), 2, 0)
    assert g["status"] == 5 and (g["counts"] == SENT).all() and (g["perm"] == SENT).all()
    assert g["state"].tolist() == state.tolist()
    for bad_len in (0, 1 << 20):
        state = np.array([1, 2, 1], np.uint8)
        g = gpu_schedule(state, np.array([3, 3, bad_len], np.int32), 2, 0)
        assert g["status"] == 5 and (g["counts"] == SENT).all()
        assert g["state"].tolist() == [1, 2, 1]          # the finished slot is not freed


# --------------------------------------------------------------------------------- admission

def _pool_arrays(S, ids_cap, rng):
    state = rng.choice(np.array([0, 0, 1, 2], np.uint8), size=S)
    col = rng.integers(0, 50, size=S).astype(np.int32)
    cap = rng.integers(1, 50, size=S).astype(np.int32)
    ln = rng.integers(0, 20, size=S).astype(np.int32)
    lim = rng.integers(0, 30, size=S).astype(np.int32)
    ids = rng.integers(0, 100, size=(S, ids_cap)).astype(np.int32)
    return [state, col, cap, ln, lim, ids]


def gpu_admit(pool, slots, cols, caps, limits, prompts, D, arena_cols, status0=0):
    import speculative_decoding_specdec_gb300.specdec as sd
    t = [_u8(pool[0])] + [_i32(x) for x in pool[1:]]
    off = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int32)
    flat = np.array([v for p in prompts for v in p] or [0], np.int32)
    status = torch.full((1,), status0, dtype=torch.int32, device=DEV)
    sd.pool_admit(_i32(slots), _i32(cols), _i32(caps), _i32(limits), _i32(flat), _i32(off), D,
                  arena_cols, *t, status)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in t], int(status.item())


def test_admit_matches_oracle():
    rng = np.random.default_rng(4)
    D, S, ids_cap, arena_cols = 4, 300, 64, 100000
    pool = _pool_arrays(S, ids_cap, rng)
    free = np.nonzero(pool[0] == O.FREE)[0]
    slots = rng.permutation(free)[:120].tolist()
    n = len(slots)
    lens = rng.integers(1, 40, size=n)
    limits = (lens + rng.integers(1, 20, size=n)).clip(max=ids_cap - D)
    caps = limits + D - 1 + rng.integers(0, 5, size=n)
    cols = np.cumsum(np.concatenate([[0], caps[:-1]]))
    prompts = [rng.integers(0, 1000, size=int(k)).tolist() for k in lens]
    got, st = gpu_admit(pool, slots, cols, caps, limits, prompts, D, arena_cols)
    assert st == 0
    want = O.pool_admit(*pool, slots, cols, caps, limits, prompts, D, arena_cols)
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)


def test_admit_errors_write_nothing():
    rng = np.random.default_rng(5)
    D, S, ids_cap, arena_cols = 3, 8, 20, 40
    pool = _pool_arrays(S, ids_cap, rng)
    pool[0][:] = [0, 0, 1, 0, 2, 0, 0, 0]
    ok = ([1], [0], [8], [6], [[5, 6]])
    got, st = gpu_admit(pool, *ok, D, arena_cols)
    assert st == 0 and got[0][1] == O.ACTIVE
    bad = [
        (([2], [0], [12], [10], [[1]]), 5),                 # slot 2 is active
        (([4], [0], [12], [10], [[1]]), 5),                 # slot 4 is finished, not yet freed
        (([1, 1], [0, 10], [5, 5], [3, 3], [[1], [1]]), 5), # slot named twice
        (([1, 3], [0, 10], [5, 5], [3, 3], [[1], []]), 5),  # empty prompt
        (([1], [0], [5], [3], [[1, 2, 3]]), 5),             # prompt not shorter than its limit
        (([1], [38], [5], [3], [[1]]), 5),                  # range past the arena
        (([8], [0], [5], [3], [[1]]), 5),                   # slot out of range
        (([-1], [0], [5], [3], [[1]]), 5),
        (([1], [0], [5], [4], [[1]]), 4),                   # limit + D - 1 > cap
        (([1], [5], [30], [18], [[1]]), 4),                 # limit + D > ids_cap
    ]
    for args, code in bad:
        got, st = gpu_admit(pool, *args, D, arena_cols)
        assert st == code, args
        for g, w in zip(got, pool):
            np.testing.assert_array_equal(g, w)
    got, st = gpu_admit(pool, *ok, D, arena_cols, status0=6)  # an earlier error: no writes
    assert st == 6
    for g, w in zip(got, pool):
        np.testing.assert_array_equal(g, w)


# --------------------------------------------------------------------------------- retirement

@pytest.mark.parametrize("in_place,eos", [(False, 3), (True, 3), (False, -1)])
def test_append_retires_like_oracle(in_place, eos):
    import speculative_decoding_specdec_gb300.specdec as sd
    rng = np.random.default_rng(6)
    S, D, L, H, hd, cap, V = 10, 4, 2, 2, 64, 40, 8           # small V: EOS shows up often
    arena = torch.zeros((L, 2, 1, H, S * cap, hd), device=DEV)
    scratch = torch.zeros((L, 2, S, H, cap, hd), device=DEV)
    n = rng.integers(2, 12, size=S).astype(np.int32)
    if in_place:
        n[:] = 7
    limit = (n + rng.integers(1, 7, size=S)).astype(np.int32)
    ids = rng.integers(0, V, size=(S, cap)).astype(np.int32)
    state = np.ones(S, np.uint8)
    state[8] = O.FINISHED_EOS                                 # slot 8 not active: reported
    rows = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8], np.int32)
    t = dict(slot_col=_i32(np.arange(S) * cap), slot_cap=_i32([cap] * S), slot_len=_i32(n),
             pool_ids=_i32(ids), state=_u8(state), limit=_i32(limit))
    blen = torch.zeros(len(rows), dtype=torch.int32, device=DEV)
    width = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sids = torch.zeros((S, cap), dtype=torch.int32, device=DEV)
    smask = torch.zeros((S, cap), dtype=torch.uint8, device=DEV)
    spos = torch.zeros((S, cap), dtype=torch.int32, device=DEV)
    sd.pool_gather(arena, scratch, _i32(rows), D, t["slot_col"], t["slot_cap"], t["slot_len"],
                   t["pool_ids"], blen, width, st, sids, smask, spos, in_place=in_place)
    a = rng.integers(0, D + 1, size=len(rows)).astype(np.int32)
    y = rng.integers(0, V, size=len(rows)).astype(np.int32)
    draft = rng.integers(0, V, size=(len(rows), D)).astype(np.int32)
    sd.pool_append(arena, scratch, _i32(rows), D, t["slot_col"], t["slot_cap"], t["slot_len"],
                   t["pool_ids"], blen, width, _i32(a), _i32(y), _i32(draft), st,
                   in_place=in_place, slot_state=t["state"], slot_limit=t["limit"], eos_id=eos)
    torch.cuda.synchronize()
    assert int(st.item()) == 5                                 # the row of slot 8
    act = rows[:8]
    _, len_app, ids_app = O.pool_append(np.zeros((L, 2, H, S * cap, hd)), np.arange(S) * cap, n,
                                        act.tolist(), np.zeros((L, 2, S, H, cap, hd)),
                                        int(width.item()), a[:8], y[:8], draft[:8], ids)
    want_len, want_state = O.retire(n, len_app, ids_app, act.tolist(), limit, eos, state)
    np.testing.assert_array_equal(t["slot_len"].cpu().numpy(), want_len)
    np.testing.assert_array_equal(t["state"].cpu().numpy(), want_state)
    np.testing.assert_array_equal(t["pool_ids"].cpu().numpy(), ids_app)
    assert want_len[8] == n[8] and want_state[8] == O.FINISHED_EOS
    if eos >= 0:
        assert (want_state == O.FINISHED_EOS).sum() >= 2
    assert (want_state[:8] == O.FINISHED_LENGTH).any()


# --------------------------------------------------------------------------------- whole pool

@pytest.mark.parametrize("S,bs,window,seed", [(4, 2, 0, 1), (6, 3, 2, 2), (5, 2, 100, 3),
                                              (3, 1, 0, 4)])
def test_sequence_pool_commits_what_each_sequence_commits_alone(S, bs, window, seed):
    from speculative_decoding_specdec_gb300.engine import SequencePool
    D, V, EOS = testlib.D, testlib.V, testlib.EOS
    L, H, hd = 2, 2, 64
    rng = np.random.default_rng(seed)
    requests = []
    for _ in range(12):
        n = int(rng.integers(2, 9))
        requests.append((rng.integers(1, V, size=n).tolist(), n + int(rng.integers(2, 16))))
    max_len = max(lim for _, lim in requests)
    pool = SequencePool(L, H, hd, torch.float32, S, 60, D, max_len, batch_size=bs, window=window,
                        eos_id=EOS, device=DEV)
    seq_of, rnd = [-1] * S, [0] * S
    waiting = list(range(len(requests)))
    results = {}
    for _ in range(500):
        batches, fin = pool.schedule()
        for s, why in fin:
            toks = pool.tokens(s)
            n = len(toks)
            exp = torch.zeros((L, 2, 1, H, n - 1, hd), device=DEV)
            synth.write_tagged_columns(exp, 0, 0, seq_of[s], list(range(n - 1)), toks[:-1])
            c = int(pool.slot_col[s].item())
            assert torch.equal(pool.arena[:, :, :, :, c:c + n - 1], exp)   # committed K/V
            results[seq_of[s]] = (toks, why)
        slots = pool.admit([requests[q][0] for q in waiting], [requests[q][1] for q in waiting])
        for s in slots:
            q = waiting.pop(0)
            seq_of[s], rnd[s] = q, 0
            p = requests[q][0]
            c = int(pool.slot_col[s].item())
            synth.write_tagged_columns(pool.arena, 0, c, q, list(range(len(p) - 1)), p[:-1])
        if not waiting and not batches and not slots:
            break
        if slots:
            continue                                           # newly admitted: schedule again
        logits = torch.zeros((S, D + 1, V))
        draft = torch.zeros((S, D), dtype=torch.int32)
        for s in range(S):
            if pool.taken[s]:
                logits[s], draft[s] = testlib.round_scores(seq_of[s], rnd[s])
        dl, dd = logits.to(DEV), draft.to(DEV)
        pool.verify_greedy(dl, dd)
        lens = pool.slot_len.cpu().tolist()
        ids = pool.pool_ids.cpu()
        perm = pool.perm.cpu().tolist()
        for off, k, uni in batches:
            pool.gather(off, k, uni)
            W = int(pool.width.item())
            for i, s in enumerate(perm[off:off + k]):      # the verification pass writes K/V
                n = lens[s]
                toks = [int(ids[s, n - 1])] + draft[s].tolist()
                if uni:
                    synth.write_tagged_columns(pool.arena, 0, int(pool.slot_col[s].item()) + n - 1,
                                               seq_of[s], list(range(n - 1, n + D)), toks)
                else:
                    synth.write_tagged_columns(pool.scratch, i, W - 1, seq_of[s],
                                               list(range(n - 1, n + D)), toks)
            pool.append(off, k, uni, dd)
        for off, k, _ in batches:
            for s in perm[off:off + k]:
                rnd[s] += 1
        torch.cuda.synchronize()
        assert int(pool.status.item()) == 0
    assert sorted(results) == list(range(len(requests)))
    for q, (prompt, limit) in enumerate(requests):
        assert results[q] == testlib.alone(prompt, limit, q)
