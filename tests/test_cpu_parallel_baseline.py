"""The row-parallel CPU baseline (oracle/specdec_cpu_parallel.cpp) against the oracle.

bench.py reports it as a multi-core CPU baseline next to the single-threaded oracle; before its
times mean anything it must compute what the oracle computes: bit-exact accept lengths, tokens,
moved K/V bytes, ids, mask, position IDs, lengths and width, and the same errors.
"""
import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
from oracle import _build_cpu


@pytest.fixture(scope="module")
def lib():
    return _build_cpu.load()


def _p(a):
    return a.ctypes.data


def _verify(lib, logits, draft, threads):
    B, Dp1, V = logits.shape
    if logits.dtype == torch.bfloat16:
        raw, dt = np.ascontiguousarray(logits.view(torch.int16).numpy()), 1
    else:
        raw, dt = np.ascontiguousarray(logits.numpy().astype(np.float32)), 0
    d = np.ascontiguousarray(draft.numpy().astype(np.int32))
    a = np.zeros(B, np.int32)
    y = np.zeros(B, np.int32)
    rc = lib.cpu_verify_greedy(_p(raw), dt, B, Dp1 - 1, V, _p(d), _p(a), _p(y), threads)
    return rc, a, y


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_greedy_matches_oracle(lib, dtype, threads):
    g = torch.Generator().manual_seed(5)
    B, D, V = 11, 5, 300
    # few distinct values: many ties, so the lowest-index rule is exercised
    logits = torch.randint(-4, 4, (B, D + 1, V), generator=g).to(dtype)
    draft = torch.randint(0, V, (B, D), generator=g, dtype=torch.int32)
    # plant the target's choices as drafts in some rows so that acceptance runs long
    choice = np.array([[O.greedy_choice(logits[b, j].double().numpy()) for j in range(D)]
                       for b in range(B)])
    for b in range(0, B, 2):
        k = b % (D + 1)
        draft[b, :k] = torch.as_tensor(choice[b, :k], dtype=torch.int32)
    exp_a, exp_y = O.verify_greedy(logits.double().numpy(), draft.numpy())
    rc, a, y = _verify(lib, logits, draft, threads)
    assert rc == 0
    np.testing.assert_array_equal(a, exp_a)
    np.testing.assert_array_equal(y, exp_y)
    assert exp_a.max() >= 2


def test_greedy_errors_like_oracle(lib):
    g = torch.Generator().manual_seed(6)
    logits = torch.randn(3, 4, 50, generator=g)
    draft = torch.randint(0, 50, (3, 3), generator=g, dtype=torch.int32)
    nan = logits.clone()
    nan[1, 2, 7] = float("nan")
    with pytest.raises(O.OracleError):
        O.verify_greedy(nan.double().numpy(), draft.numpy())
    assert _verify(lib, nan, draft, 4)[0] == 1
    bad = draft.clone()
    bad[2, 2] = 50
    with pytest.raises(O.OracleError):
        O.verify_greedy(logits.double().numpy(), bad.numpy())
    assert _verify(lib, logits, bad, 4)[0] == 1


def _realign(lib, src, dst, n, W, a, y, draft, ids_src, threads, pad_id=0):
    L, _, B, H, S_src, hd = src.shape
    S_dst = dst.shape[4]
    col_bytes = hd * src.itemsize
    out = np.array(dst, copy=True)
    ids = np.zeros((B, S_dst), np.int32)
    mask = np.zeros((B, S_dst), np.uint8)
    pos = np.zeros((B, S_dst), np.int32)
    n_out = np.zeros(B, np.int32)
    w_out = np.zeros(1, np.int32)
    args = [np.ascontiguousarray(x, dtype=np.int32) for x in (n, a, y, draft, ids_src)]
    rc = lib.cpu_realign(_p(src), _p(out), L, B, H, S_src, S_dst, col_bytes, draft.shape[1],
                         _p(args[0]), int(W), _p(args[1]), _p(args[2]), _p(args[3]), _p(args[4]),
                         _p(ids), _p(mask), _p(pos), _p(n_out), _p(w_out), pad_id, threads)
    return rc, out, ids, mask, pos, n_out, int(w_out[0])


@pytest.mark.parametrize("threads", [1, 2, 7])
def test_realign_matches_oracle(lib, threads):
    rng = np.random.default_rng(3)
    L, B, H, hd, D = 2, 6, 3, 8, 4
    for _ in range(4):
        n = rng.integers(1, 30, size=B)
        W = int(n.max()) + int(rng.integers(0, 3))
        S_src, S_dst = W + D + 2, W + 2 * D + 3
        src = rng.integers(-30000, 30000, size=(L, 2, B, H, S_src, hd), dtype=np.int16)
        dst = rng.integers(-30000, 30000, size=(L, 2, B, H, S_dst, hd), dtype=np.int16)
        a = rng.integers(0, D + 1, size=B)
        y = rng.integers(0, 1000, size=B)
        draft = rng.integers(0, 1000, size=(B, D))
        ids_src = rng.integers(0, 1000, size=(B, S_src)).astype(np.int32)
        exp = O.realign(src, dst, n, W, a, y, draft, ids_src, 7)
        rc, out, ids, mask, pos, n_out, w_out = _realign(lib, src, dst, n, W, a, y, draft,
                                                         ids_src, threads, pad_id=7)
        assert rc == 0
        np.testing.assert_array_equal(out, exp[0])
        np.testing.assert_array_equal(ids, exp[1])
        np.testing.assert_array_equal(mask, exp[2])
        np.testing.assert_array_equal(pos, exp[3])
        np.testing.assert_array_equal(n_out, exp[4])
        assert w_out == exp[5]


def test_realign_errors_like_oracle(lib):
    rng = np.random.default_rng(4)
    L, B, H, hd, D = 1, 3, 2, 8, 3
    n = np.array([5, 9, 2])
    W = 9
    src = rng.integers(-100, 100, size=(L, 2, B, H, W + D, hd), dtype=np.int16)
    ids_src = np.zeros((B, W + D), np.int32)
    draft = np.zeros((B, D), np.int32)
    y = np.zeros(B, np.int32)
    small = np.zeros((L, 2, B, H, W + D, hd), np.int16)    # W' = 13 > W + D - D
    a = np.array([3, 3, 0])
    with pytest.raises(O.OracleError):
        O.realign(src, small, n, W, a, y, draft, ids_src)
    before = small.copy()
    rc, out, *_ = _realign(lib, src, small, n, W, a, y, draft, ids_src, 2)
    assert rc == 2 and np.array_equal(out, before)
    big = np.zeros((L, 2, B, H, W + 2 * D + 2, hd), np.int16)
    for bad_a, bad_n in ((np.array([4, 0, 0]), n), (a, np.array([0, 9, 2])),
                         (a, np.array([5, 10, 2]))):
        with pytest.raises(O.OracleError):
            O.realign(src, big, bad_n, W, bad_a, y, draft, ids_src)
        assert _realign(lib, src, big, bad_n, W, bad_a, y, draft, ids_src, 2)[0] == 1


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sampled_matches_oracle(lib, dtype):
    from speculative_decoding_specdec_gb300 import synth
    gen = synth.make_gen(12)
    B, D, V, T = 9, 4, 257, 0.7
    lg, dl, d, u = synth.sampled_round(gen, B, D, V, T, dtype=dtype)
    a_exp, y_exp, _, _ = O.verify_sample(lg.double().numpy(), dl.double().numpy(), d.numpy(),
                                        u.double().numpy(), T)
    dt = 1 if dtype == torch.bfloat16 else 0
    conv = (lambda t: np.ascontiguousarray(t.view(torch.int16).numpy())) if dt else \
        (lambda t: np.ascontiguousarray(t.numpy()))
    tl, dr = conv(lg), conv(dl)
    dd = np.ascontiguousarray(d.numpy().astype(np.int32))
    uu = np.ascontiguousarray(u.numpy().astype(np.float32))
    a = np.zeros(B, np.int32)
    y = np.zeros(B, np.int32)
    assert lib.cpu_verify_sample(_p(tl), _p(dr), dt, B, D, V, _p(dd), _p(uu), T, _p(a), _p(y),
                                 3) == 0
    np.testing.assert_array_equal(a, a_exp)
    np.testing.assert_array_equal(y, y_exp)
    assert 0 < a_exp.sum() < B * D      # both rejections and acceptances occur
    bad = dd.copy()
    bad[0, 0] = V
    assert lib.cpu_verify_sample(_p(tl), _p(dr), dt, B, D, V, _p(bad), _p(uu), T, _p(a), _p(y),
                                 3) == 1
