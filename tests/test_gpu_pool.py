"""Pool gather / append (EXSPEC mixed leftovers) on the GPU against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth

pytestmark = pytest.mark.gpu


def _pool(S, cap, L, H, hd, V, gen, lo, hi):
    dev = "cuda"
    arena = torch.full((L, 2, 1, H, S * cap, hd), -9.0, device=dev)
    n = synth.lengths_uniform(gen, S, lo, hi)
    toks = [torch.randint(0, V, (int(n[s]),), generator=gen).tolist() for s in range(S)]
    for s in range(S):
        synth.write_tagged_columns(arena, 0, s * cap, s, list(range(len(toks[s]) - 1)),
                                   toks[s][:-1])
    pool_ids = torch.zeros(S, cap, dtype=torch.int32)
    for s in range(S):
        pool_ids[s, :len(toks[s])] = torch.tensor(toks[s], dtype=torch.int32)
    i32 = lambda x: torch.as_tensor(x, dtype=torch.int32, device=dev)  # noqa: E731
    return dict(arena=arena, slot_col=i32(np.arange(S) * cap), slot_cap=i32([cap] * S),
                slot_len=i32(n.numpy()), pool_ids=pool_ids.to(dev), toks=toks)


@pytest.mark.parametrize("scheduled", [False, True])
def test_gather_append_rounds_match_oracle(scheduled):
    """Gather / append against the oracle, with fixed CTA shares or with work items taken from
    a pair of scheduling words (back at zero after every call)."""
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(21)
    S, cap, L, H, hd, D, V, R = 12, 80, 2, 3, 64, 4, 50, 5
    P = _pool(S, cap, L, H, hd, V, gen, 2, 40)
    dev = "cuda"
    Sc = 40 + 8 * (D + 1) + D + 1
    scratch = torch.full((L, 2, R, H, Sc, hd), 5.0, device=dev)
    s_ids = torch.zeros(R, Sc, dtype=torch.int32, device=dev)
    s_mask = torch.zeros(R, Sc, dtype=torch.uint8, device=dev)
    s_pos = torch.zeros(R, Sc, dtype=torch.int32, device=dev)
    blen = torch.zeros(R, dtype=torch.int32, device=dev)
    width = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sched = torch.zeros(2, dtype=torch.int32, device=dev) if scheduled else None
    rng = np.random.default_rng(2)
    for _ in range(6):
        k = int(rng.integers(1, R + 1))
        rows_np = rng.choice(S, size=k, replace=False).astype(np.int32)
        rows = torch.as_tensor(rows_np, device=dev)
        ar0 = P["arena"][:, :, 0].cpu().numpy()
        n_np = P["slot_len"].cpu().numpy()
        ids_np = P["pool_ids"].cpu().numpy()
        sc0 = scratch.cpu().numpy()
        sd.pool_gather(P["arena"], scratch, rows, D, P["slot_col"], P["slot_cap"], P["slot_len"],
                       P["pool_ids"], blen, width, st, s_ids, s_mask, s_pos, schedule=sched)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert sched is None or sched.tolist() == [0, 0]
        exp_sc, W, eids, emask, epos = O.pool_gather(ar0, np.arange(S) * cap, n_np, rows_np.tolist(),
                                                   sc0, 0, ids_np)
        assert int(width.item()) == W
        np.testing.assert_array_equal(blen.cpu().numpy()[:k], n_np[rows_np])
        np.testing.assert_array_equal(scratch.cpu().numpy(), exp_sc)
        np.testing.assert_array_equal(s_ids.cpu().numpy()[:k], eids)
        np.testing.assert_array_equal(s_mask.cpu().numpy()[:k], emask)
        np.testing.assert_array_equal(s_pos.cpu().numpy()[:k], epos)
        # synthetic verification pass on the padded batch, then greedy verification
        logits, draft = synth.greedy_round(gen, k, D, V, 0.6, dtype=torch.float32)
        for i, s in enumerate(rows_np):
            t = P["toks"][s]
            synth.write_tagged_columns(scratch, i, W - 1, int(s), list(range(len(t) - 1, len(t) + D)),
                                       [t[-1]] + draft[i].tolist())
        a, y = O.verify_greedy(logits.double().numpy(), draft.numpy())
        ar1 = P["arena"][:, :, 0].cpu().numpy()
        sc1 = scratch.cpu().numpy()
        ga = torch.as_tensor(a, device=dev)
        gy = torch.as_tensor(y, device=dev)
        sd.pool_append(P["arena"], scratch, rows, D, P["slot_col"], P["slot_cap"], P["slot_len"],
                       P["pool_ids"], blen, width, ga, gy, draft.to(dev), st, schedule=sched)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert sched is None or sched.tolist() == [0, 0]
        exp_ar, exp_len, exp_ids = O.pool_append(ar1, np.arange(S) * cap, n_np, rows_np.tolist(),
                                                 sc1, W, a, y, draft.numpy(), ids_np)
        np.testing.assert_array_equal(P["arena"][:, :, 0].cpu().numpy(), exp_ar)
        np.testing.assert_array_equal(P["slot_len"].cpu().numpy(), exp_len)
        np.testing.assert_array_equal(P["pool_ids"].cpu().numpy(), exp_ids)
        for i, s in enumerate(rows_np):
            P["toks"][s] = P["toks"][s] + draft[i, :a[i]].tolist() + [int(y[i])]
    # every slot equals a from-scratch rebuild of its sequence
    got = P["arena"][:, :, 0].cpu().numpy()
    for s in range(S):
        t = P["toks"][s]
        ref = torch.zeros(L, 2, 1, H, len(t) - 1, hd)
        synth.write_tagged_columns(ref, 0, 0, s, list(range(len(t) - 1)), t[:-1])
        np.testing.assert_array_equal(got[:, :, :, s * cap:s * cap + len(t) - 1], ref[:, :, 0].numpy())


def test_in_place_uniform_batch():
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(22)
    S, cap, L, H, hd, D, V = 6, 60, 1, 2, 32, 3, 40
    P = _pool(S, cap, L, H, hd, V, gen, 9, 9)          # all length 9
    dev = "cuda"
    scratch = torch.zeros(L, 2, 4, H, 16, hd, device=dev)
    blen = torch.zeros(4, dtype=torch.int32, device=dev)
    width = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    rows_np = np.array([4, 1, 2, 5], dtype=np.int32)
    rows = torch.as_tensor(rows_np, device=dev)
    sd.pool_gather(P["arena"], scratch, rows, D, P["slot_col"], P["slot_cap"], P["slot_len"],
                   P["pool_ids"], blen, width, st, in_place=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(width.item()) == 9 and (blen == 9).all()
    assert (scratch == 0).all()                         # nothing was gathered
    logits, draft = synth.greedy_round(gen, 4, D, V, 0.6, dtype=torch.float32)
    for i, s in enumerate(rows_np):                     # the pass writes into the slots
        t = P["toks"][s]
        synth.write_tagged_columns(P["arena"], 0, int(s) * cap + 8, int(s), list(range(8, 9 + D)),
                                   [t[-1]] + draft[i].tolist())
    a, y = O.verify_greedy(logits.double().numpy(), draft.numpy())
    ar1 = P["arena"][:, :, 0].cpu().numpy()
    n_np = P["slot_len"].cpu().numpy()
    ids_np = P["pool_ids"].cpu().numpy()
    sd.pool_append(P["arena"], scratch, rows, D, P["slot_col"], P["slot_cap"], P["slot_len"],
                   P["pool_ids"], blen, width, torch.as_tensor(a, device=dev),
                   torch.as_tensor(y, device=dev), draft.to(dev), st, in_place=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # expected: the slot columns stay where the pass wrote them; lengths and ids advance
    fake = np.zeros((L, 2, 4, H, 9 + D, hd), np.float32)
    for i, s in enumerate(rows_np):
        fake[:, :, i, :, 8:9 + D] = ar1[:, :, :, s * cap + 8:s * cap + 9 + D]
    exp_ar, exp_len, exp_ids = O.pool_append(ar1, np.arange(S) * cap, n_np, rows_np.tolist(), fake,
                                             9, a, y, draft.numpy(), ids_np)
    np.testing.assert_array_equal(P["arena"][:, :, 0].cpu().numpy(), exp_ar)
    np.testing.assert_array_equal(P["slot_len"].cpu().numpy(), exp_len)
    np.testing.assert_array_equal(P["pool_ids"].cpu().numpy(), exp_ids)


def test_capacity_and_range_errors():
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(23)
    P = _pool(3, 20, 1, 1, 16, 30, gen, 15, 18)
    dev = "cuda"
    scratch = torch.zeros(1, 2, 3, 1, 12, 16, device=dev)    # too narrow for W + D
    s_ids = torch.zeros(3, 12, dtype=torch.int32, device=dev)
    s_mask = torch.zeros(3, 12, dtype=torch.uint8, device=dev)
    s_pos = torch.zeros(3, 12, dtype=torch.int32, device=dev)
    blen = torch.zeros(3, dtype=torch.int32, device=dev)
    width = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    rows = torch.tensor([0, 1, 2], dtype=torch.int32, device=dev)
    sd.pool_gather(P["arena"], scratch, rows, 2, P["slot_col"], P["slot_cap"], P["slot_len"],
                   P["pool_ids"], blen, width, st, s_ids, s_mask, s_pos)
    torch.cuda.synchronize()
    assert int(st.item()) == 4 and (scratch == 0).all() and int(width.item()) == 0
    st.zero_()
    blen.fill_(5)
    width.fill_(6)
    bad = torch.tensor([0, 3, 1], dtype=torch.int32, device=dev)   # 3 > D = 2
    before = P["slot_len"].clone()
    sd.pool_append(P["arena"], scratch, rows, 2, P["slot_col"], P["slot_cap"], P["slot_len"],
                   P["pool_ids"], blen, width, bad, bad, torch.zeros(3, 2, dtype=torch.int32, device=dev),
                   st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5 and torch.equal(before, P["slot_len"])


def test_pool_engine_rounds_match_oracle():
    """ExspecPool rounds (grouping, one verification over the pool, per-batch gather/append with
    pool-wide accept lengths) against the oracle, with a synthetic verification pass writing the
    new K/V columns in between; every slot equals its from-scratch rebuild after every round."""
    from speculative_decoding_specdec_gb300.engine import ExspecPool
    gen = synth.make_gen(24)
    L, H, hd, D, V, S, bs, rounds = 1, 2, 16, 3, 40, 22, 4, 4
    n0 = synth.lengths_discrete(gen, S, [4, 6, 9]).tolist()
    toks = [torch.randint(0, V, (n,), generator=gen).tolist() for n in n0]
    pool = ExspecPool(L, H, hd, torch.float32, toks, D, rounds, batch_size=bs)
    pool.arena.fill_(-9.0)
    cols = pool.slot_col.cpu().numpy()
    for s in range(S):
        synth.write_tagged_columns(pool.arena, 0, int(cols[s]), s, list(range(n0[s] - 1)),
                                   toks[s][:-1])
    n = np.array(n0)
    saw_uniform = saw_mixed = False
    for _ in range(rounds):
        batches = pool.schedule()
        ep, eo, eu, enu = O.group_by_length(n, bs)
        assert [(int(eo[k]), int(eo[k + 1] - eo[k]), bool(eu[k])) for k in range(len(eu))] == batches
        np.testing.assert_array_equal(pool.perm.cpu().numpy(), ep)
        logits, draft = synth.greedy_round(gen, S, D, V, 0.6, dtype=torch.float32)
        dd = draft.cuda()
        pool.verify_greedy(logits.cuda(), dd)
        a, y = O.verify_greedy(logits.double().numpy(), draft.numpy())
        for off, k, uniform in batches:
            rows = ep[off:off + k].tolist()
            pool.gather(off, k, uniform)
            torch.cuda.synchronize()
            W = int(pool.width.item())
            assert W == max(n[s] for s in rows)
            for i, s in enumerate(rows):       # the verification pass writes [pending, d_1..d_D]
                pos = list(range(n[s] - 1, n[s] + D))
                tk = [toks[s][-1]] + draft[s].tolist()
                if uniform:
                    synth.write_tagged_columns(pool.arena, 0, int(cols[s]) + n[s] - 1, s, pos, tk)
                else:
                    synth.write_tagged_columns(pool.scratch, i, W - 1, s, pos, tk)
            pool.append(off, k, uniform, dd)
            torch.cuda.synchronize()
            assert int(pool.status.item()) == 0
            for s in rows:
                toks[s] = toks[s] + draft[s, :a[s]].tolist() + [int(y[s])]
                n[s] += a[s] + 1
            saw_uniform |= uniform
            saw_mixed |= not uniform
        np.testing.assert_array_equal(pool.slot_len.cpu().numpy(), n)
        np.testing.assert_array_equal(pool.accept_len.cpu().numpy(), a)
        arena = pool.arena[:, :, 0].cpu().numpy()
        ids = pool.pool_ids.cpu().numpy()
        for s in range(S):
            ref = torch.zeros(L, 2, 1, H, n[s] - 1, hd)
            synth.write_tagged_columns(ref, 0, 0, s, list(range(n[s] - 1)), toks[s][:-1])
            c0 = int(cols[s])
            np.testing.assert_array_equal(arena[:, :, :, c0:c0 + n[s] - 1], ref[:, :, 0].numpy())
            assert list(ids[s, :n[s]]) == toks[s]
    assert saw_uniform and saw_mixed
