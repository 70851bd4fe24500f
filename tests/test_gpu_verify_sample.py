"""Sampled verification on the GPU against the CPU oracle.

Tolerance (decisions are taken in fp32/fp64 on the GPU and in fp64 in the oracle):
* accept decisions must match except where |u - p(d)/q(d)| < 1e-6 (p/q as the oracle computes it);
* with equal accept lengths, the drawn token must match except where u[b][D] * R lies within
  1e-5 * R of a boundary of the oracle's running sum (a boundary-straddling draw may pick the
  neighbouring token);
* residual probabilities within 1e-5 absolute.
Shapes: the GLM-4-9B-shaped full size (B=32, D=6, V=151552, T=0.7) and smaller, ragged,
unaligned, D=1 / D=31, q == p; plus a chi-square check that the GPU's emitted token follows p.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_ACCEPT = 1e-6
TOL_DRAW = 1e-5
TOL_RESID = 1e-5


def gpu_sample(tl, dl, draft, u, T, row_stride=None, residual=True, top_k=0, top_p=1.0,
               bounds_out=None):
    import speculative_decoding_specdec_gb300.specdec as sd
    B, Dp1, V = tl.shape

    def place(x):
        if row_stride is None:
            return x.to(DEV)
        R = x.shape[1]
        buf = torch.zeros(B * R * row_stride + 8, dtype=x.dtype, device=DEV)
        y = buf[:B * R * row_stride].view(B, R, row_stride)[:, :, :V]
        y.copy_(x.to(DEV))
        return y
    a = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    y = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = torch.full((B, V), -1.0, device=DEV) if residual else None
    tl_d, dl_d = place(tl), place(dl)
    bounds = None
    if top_k or top_p < 1.0:
        bounds = torch.zeros((B, 2 * Dp1 - 1, 2), dtype=torch.int32, device=DEV)
        sd.sampling_filter(tl_d, dl_d, T, top_k, top_p, bounds, st)
        if bounds_out is not None:
            bounds_out.append(bounds)
    sd.verify_sample(tl_d, dl_d, draft.to(DEV), u.to(DEV), T, a, y, st, res, keep_bounds=bounds)
    torch.cuda.synchronize()
    return (a.cpu().numpy(), y.cpu().numpy(), None if res is None else res.cpu().numpy(),
            int(st.item()))


def compare(tl, dl, draft, u, T, row_stride=None, max_excused=0.02):
    a, y, res, st = gpu_sample(tl, dl, draft, u, T, row_stride)
    assert st == 0
    ea, ey, eres, tr = O.verify_sample(tl.double().numpy(), dl.double().numpy(), draft.numpy(),
                                       u.double().numpy(), T)
    uu = u.double().numpy()
    excused = 0
    for b in range(len(a)):
        if a[b] != ea[b]:
            j = min(a[b], ea[b])            # first decision that differs
            assert abs(uu[b, j] - tr["ratio"][b, j]) < TOL_ACCEPT, (b, j, uu[b, j], tr["ratio"][b, j])
            excused += 1
            continue
        if y[b] != ey[b]:
            R = tr["R"][b]
            near = min(abs(tr["t"][b] - tr["cdf_lo"][b]), abs(tr["t"][b] - tr["cdf_hi"][b]))
            assert near < TOL_DRAW * R, (b, y[b], ey[b], near / R)
            excused += 1
            continue
        np.testing.assert_allclose(res[b], eres[b], rtol=0, atol=TOL_RESID)
    assert excused <= max(1, max_excused * len(a))
    return a, y


@pytest.mark.parametrize("B,D,V,T,dtype", [
    (32, 6, 151552, 0.7, torch.bfloat16),     # GLM-4-9B-shaped, full size
    (8, 5, 32000, 0.7, torch.bfloat16),
    (4, 4, 1000, 1.0, torch.float32),
    (5, 3, 1003, 0.5, torch.bfloat16),        # ragged V
    (3, 1, 40000, 1.3, torch.bfloat16),       # D = 1
    (2, 31, 600, 0.9, torch.float32),         # D = 31
    (1, 2, 9, 0.7, torch.float32),            # tiny V
    (64, 2, 4096, 0.7, torch.bfloat16),       # many rows
    (16, 4, 151936, 0.7, torch.bfloat16),     # Qwen3-8B-shaped: two CTAs per SM, clusters of 13
])
def test_sample_matches_oracle(B, D, V, T, dtype):
    gen = synth.make_gen(2000 + B + D)
    tl, dl, draft, u = synth.sampled_round(gen, B, D, V, T, dtype=dtype)
    compare(tl, dl, draft, u, T)


@pytest.mark.parametrize("extra", [8, 3])
def test_padded_and_unaligned_rows(extra):
    gen = synth.make_gen(31)
    for dtype in (torch.bfloat16, torch.float32):
        tl, dl, draft, u = synth.sampled_round(gen, 6, 3, 5000, 0.7, dtype=dtype)
        compare(tl, dl, draft, u, 0.7, row_stride=5000 + extra)


def test_q_equal_p_accepts_all():
    gen = synth.make_gen(32)
    tl, _, draft, u = synth.sampled_round(gen, 16, 4, 20000, 0.7)
    a, y, res, st = gpu_sample(tl, tl[:, :4].contiguous(), draft, u, 0.7)
    assert st == 0 and (a == 4).all()


def test_low_acceptance_sharp_temperature():
    gen = synth.make_gen(33)
    tl, dl, draft, u = synth.sampled_round(gen, 24, 5, 30000, 0.25, sigma=1.5)
    compare(tl, dl, draft, u, 0.25)


@pytest.mark.parametrize("T,scale,dtype", [
    (0.05, 1.0, torch.bfloat16),    # nearly greedy: most exponents underflow
    (4.0, 1.0, torch.bfloat16),     # nearly flat
    (1.0, 12.0, torch.bfloat16),    # scores spread like a real model's (tens of units)
    (0.05, 1.0, torch.float32),
    (1.0, 30.0, torch.float32),
])
def test_sample_extreme_temperature_and_scale(T, scale, dtype):
    """Sharp and flat temperatures and widely spread scores, under the same tolerances."""
    gen = synth.make_gen(50 + int(T * 100) + int(scale))
    tl, dl, draft, u = synth.sampled_round(gen, 8, 4, 32000, T, dtype=dtype)
    tl = (tl.float() * scale).to(dtype)
    dl = (dl.float() * scale).to(dtype)
    compare(tl, dl, draft, u, T)


def test_emitted_token_follows_p_chi_square():
    """Distribution preservation on the GPU: with drafts drawn from q, the first emitted token of
    many independent rows is distributed as p."""
    rng = np.random.default_rng(34)
    V, n, T = 8, 200000, 0.7
    p0, p1, q0 = (rng.dirichlet(np.ones(V)) for _ in range(3))
    tl = torch.tensor(np.stack([T * np.log(p0), T * np.log(p1)]), dtype=torch.float32)
    dl = torch.tensor((T * np.log(q0))[None], dtype=torch.float32)
    tl = tl[None].expand(n, 2, V).contiguous()
    dl = dl[None].expand(n, 1, V).contiguous()
    draft = torch.tensor(rng.choice(V, size=(n, 1), p=q0), dtype=torch.int32)
    u = torch.tensor(rng.random((n, 2)), dtype=torch.float32)
    a, y, _, st = gpu_sample(tl, dl, draft, u, T, residual=False)
    assert st == 0
    first = np.where(a >= 1, draft[:, 0].numpy(), y)
    assert stats.chisquare(np.bincount(first, minlength=V), p0 * n).pvalue > 1e-3
    bonus = y[a == 1]
    assert stats.chisquare(np.bincount(bonus, minlength=V), p1 * len(bonus)).pvalue > 1e-3
    pacc = np.minimum(p0, q0).sum()
    assert abs((a == 1).mean() - pacc) < 4 * np.sqrt(pacc * (1 - pacc) / n)


def test_bad_inputs_set_status():
    gen = synth.make_gen(35)
    tl, dl, draft, u = synth.sampled_round(gen, 3, 2, 500, 0.7, dtype=torch.float32)
    u[1, 0] = 1.0                                  # uniform outside [0, 1)
    assert gpu_sample(tl, dl, draft, u, 0.7)[3] == 5
    tl2, dl2, draft2, u2 = synth.sampled_round(gen, 3, 2, 500, 0.7, dtype=torch.float32)
    draft2[2, 1] = 500                             # token outside [0, V)
    assert gpu_sample(tl2, dl2, draft2, u2, 0.7)[3] == 5
    tl2[0, 1, 3] = float("nan")                    # NaN score
    draft2[2, 1] = 1
    assert gpu_sample(tl2, dl2, draft2, u2, 0.7)[3] == 5


def test_host_errors():
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(36)
    tl, dl, draft, u = synth.sampled_round(gen, 2, 2, 100, 0.7, dtype=torch.float32)
    with pytest.raises(sd.SpecdecError):
        gpu_sample(tl, dl, draft, u, 0.0)
    with pytest.raises(sd.SpecdecError):
        gpu_sample(tl, dl, draft, u, float("inf"))


def test_repeated_calls_deterministic():
    gen = synth.make_gen(38)
    tl, dl, draft, u = synth.sampled_round(gen, 32, 6, 151552, 0.7)
    r1 = gpu_sample(tl, dl, draft, u, 0.7, residual=False)
    r2 = gpu_sample(tl, dl, draft, u, 0.7, residual=False)
    assert (r1[0] == r2[0]).all() and (r1[1] == r2[1]).all()


# ------------------------------------------------------------------ top-k / top-p

def kept_from_bounds(scores, bound):
    """Host decoding of one specdec_keep_bound: the order-preserving key of the float score
    (-0 as +0; sign bit set for x >= 0, all bits inverted for x < 0) against (key, index)."""
    x = np.asarray(scores, dtype=np.float32).copy()
    x[x == 0] = 0.0
    u = x.view(np.uint32)
    key = np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)
    bkey, bidx = np.uint32(bound[0] & 0xffffffff), int(bound[1])
    return (key > bkey) | ((key == bkey) & (np.arange(len(x)) <= bidx))


def rows_of(tl, dl):
    """The 2D+1 score rows of every batch row, in the bounds' order (target rows, then draft)."""
    return np.concatenate([tl, dl], axis=1)


@pytest.mark.parametrize("B,D,V,dtype,top_k,top_p", [
    (4, 3, 1000, torch.float32, 10, 1.0),
    (4, 3, 1000, torch.float32, 0, 0.9),
    (5, 3, 1003, torch.bfloat16, 37, 0.8),
    (8, 5, 32000, torch.bfloat16, 50, 1.0),
    (8, 5, 32000, torch.bfloat16, 0, 0.95),
    (32, 6, 151552, torch.bfloat16, 0, 0.9),        # GLM-4-9B-shaped, top-p only
    (32, 6, 151552, torch.bfloat16, 100, 0.95),     # top-k then top-p
])
def test_keep_bounds_match_the_oracle(B, D, V, dtype, top_k, top_p):
    """Every row's kept set from the GPU bounds equals the oracle's (top-k exactly; top-p except
    where top_p lies within 2e-6 of a cumulative mass, which fixed-point sums may cut either way)."""
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(3000 + B + D + top_k)
    tl, dl, draft, u = synth.sampled_round(gen, B, D, V, 0.7, dtype=dtype)
    bounds = torch.zeros((B, 2 * D + 1, 2), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd.sampling_filter(tl.to(DEV), dl.to(DEV), 0.7, top_k, top_p, bounds, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bnd = bounds.cpu().numpy().astype(np.int64)
    rows = rows_of(tl.float().numpy(), dl.float().numpy())
    excused = 0
    for b in range(B):
        for q in range(2 * D + 1):
            got = kept_from_bounds(rows[b, q], bnd[b, q])
            exp = O.sampling_keep(rows[b, q].astype(np.float64), 0.7, top_k, top_p)
            if not np.array_equal(got, exp):
                assert O.top_p_margin(rows[b, q].astype(np.float64), 0.7, top_k, top_p) < 2e-6, (b, q)
                excused += 1
    assert excused <= max(1, 0.02 * B * (2 * D + 1))


@pytest.mark.parametrize("T,scale,top_k,top_p", [
    (0.05, 1.0, 0, 0.9),       # nearly all mass on the highest score or two
    (4.0, 12.0, 0, 0.9),       # widely spread scores at a flat temperature
    (0.05, 12.0, 40, 0.95),
    (4.0, 1.0, 100, 0.5),
])
def test_keep_bounds_extreme_temperature_and_scale(T, scale, top_k, top_p):
    """Keep bounds at sharp and flat temperatures and on widely spread bf16 scores."""
    import speculative_decoding_specdec_gb300.specdec as sd
    B, D, V = 4, 3, 32000
    gen = synth.make_gen(60 + top_k + int(scale))
    tl, dl, _, _ = synth.sampled_round(gen, B, D, V, T, dtype=torch.bfloat16)
    tl = (tl.float() * scale).to(torch.bfloat16)
    dl = (dl.float() * scale).to(torch.bfloat16)
    bounds = torch.zeros((B, 2 * D + 1, 2), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd.sampling_filter(tl.to(DEV), dl.to(DEV), T, top_k, top_p, bounds, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bnd = bounds.cpu().numpy().astype(np.int64)
    rows = rows_of(tl.float().numpy(), dl.float().numpy())
    for b in range(B):
        for q in range(2 * D + 1):
            got = kept_from_bounds(rows[b, q], bnd[b, q])
            exp = O.sampling_keep(rows[b, q].astype(np.float64), T, top_k, top_p)
            if not np.array_equal(got, exp):
                assert O.top_p_margin(rows[b, q].astype(np.float64), T, top_k, top_p) < 2e-6, (b, q)


def filtered_drafts(dl, T, top_k, top_p, seed):
    """Drafts drawn from the oracle's filtered draft distribution q' of every draft row (so that
    q'(d) > 0, as a draft model using the same sampling settings would propose)."""
    rng = np.random.default_rng(seed)
    w = dl.double().numpy()
    B, D, V = w.shape
    out = np.zeros((B, D), dtype=np.int32)
    for b in range(B):
        for j in range(D):
            out[b, j] = rng.choice(V, p=O.filtered_softmax(w[b, j], T, top_k, top_p))
    return torch.tensor(out)


def compare_filtered(tl, dl, draft, u, T, top_k, top_p, max_excused=0.05, row_stride=None):
    a, y, res, st = gpu_sample(tl, dl, draft, u, T, row_stride=row_stride, top_k=top_k,
                               top_p=top_p)
    assert st == 0
    tl64, dl64 = tl.double().numpy(), dl.double().numpy()
    ea, ey, eres, tr = O.verify_sample(tl64, dl64, draft.numpy(), u.double().numpy(), T,
                                       top_k=top_k, top_p=top_p)
    rows = rows_of(tl64, dl64)
    uu = u.double().numpy()
    excused = 0
    for b in range(len(a)):
        close_cut = min(O.top_p_margin(r, T, top_k, top_p) for r in rows[b]) < 2e-6
        if a[b] != ea[b]:
            j = min(a[b], ea[b])
            assert close_cut or abs(uu[b, j] - tr["ratio"][b, j]) < TOL_ACCEPT, (b, j)
            excused += 1
            continue
        if y[b] != ey[b]:
            near = min(abs(tr["t"][b] - tr["cdf_lo"][b]), abs(tr["t"][b] - tr["cdf_hi"][b]))
            assert close_cut or near < TOL_DRAW * tr["R"][b], b
            excused += 1
            continue
        if not close_cut:
            np.testing.assert_allclose(res[b], eres[b], rtol=0, atol=TOL_RESID)
    assert excused <= max(1, max_excused * len(a))
    return a, y


@pytest.mark.parametrize("B,D,V,T,dtype,top_k,top_p", [
    (4, 4, 1000, 1.0, torch.float32, 20, 1.0),
    (5, 3, 1003, 0.5, torch.bfloat16, 0, 0.9),      # ragged V: the cluster kernel's tail path
    (8, 5, 32000, 0.7, torch.bfloat16, 64, 0.95),
    (32, 6, 151552, 0.7, torch.bfloat16, 0, 0.9),   # GLM-4-9B-shaped
    (16, 4, 151936, 0.7, torch.bfloat16, 200, 1.0), # Qwen3-8B-shaped: two CTAs per SM
])
def test_filtered_sample_matches_oracle(B, D, V, T, dtype, top_k, top_p):
    gen = synth.make_gen(4000 + B + D)
    tl, dl, _, u = synth.sampled_round(gen, B, D, V, T, dtype=dtype)
    draft = filtered_drafts(dl, T, top_k, top_p, seed=B + D)
    compare_filtered(tl, dl, draft, u, T, top_k, top_p)


@pytest.mark.parametrize("extra", [3, 8])
def test_filtered_padded_rows(extra):
    """Sampling settings on rows inside wider buffers: 3 extra elements (rows not 16-byte
    aligned: plain loads) and 8 (aligned, strided: per-row slices), bf16 and fp32, element by
    element against the oracle under the same tolerances as every other sampled test."""
    gen = synth.make_gen(41 + extra)
    for dtype in (torch.bfloat16, torch.float32):
        tl, dl, _, u = synth.sampled_round(gen, 6, 3, 5000, 0.7, dtype=dtype)
        for top_k, top_p in ((30, 1.0), (0, 0.9), (50, 0.8)):
            draft = filtered_drafts(dl, 0.7, top_k, top_p, seed=6 + top_k)
            compare_filtered(tl, dl, draft, u, 0.7, top_k, top_p, row_stride=5000 + extra)


@pytest.mark.parametrize("top_k", [0, 5])
def test_drafts_outside_the_kept_sets(top_k):
    """Drafts the target cannot emit: outside both rows' kept sets (p(d) = q(d) = 0) and with a
    -inf score in both rows are rejected; outside the draft row's kept set only (q(d) = 0 < p(d))
    accepted -- as the oracle decides, element by element."""
    gen = synth.make_gen(45 + top_k)
    B, D, V, T = 18, 3, 1000, 0.7
    tl, dl, draft, u = synth.sampled_round(gen, B, D, V, T, dtype=torch.float32)
    tl64, dl64 = tl.double().numpy(), dl.double().numpy()
    rng = np.random.default_rng(top_k)
    for b in range(B):
        for j in range(D):
            case = (b + j) % 3
            if case == 2 or top_k == 0:      # -inf in both rows: 0/0
                d = int(rng.integers(0, V))
                tl[b, j, d] = float("-inf")
                dl[b, j, d] = float("-inf")
            else:
                kp = O.sampling_keep(tl64[b, j], T, top_k)
                kq = O.sampling_keep(dl64[b, j], T, top_k)
                pick = np.nonzero(~kp & ~kq)[0] if case == 0 else np.nonzero(kp & ~kq)[0]
                if len(pick) == 0:
                    pick = np.nonzero(~kp & ~kq)[0]
                d = int(pick[rng.integers(0, len(pick))])
            draft[b, j] = d
    a, y = compare_filtered(tl, dl, draft, u, T, top_k, 1.0, max_excused=0.0)
    ea = O.verify_sample(tl.double().numpy(), dl.double().numpy(), draft.numpy(),
                         u.double().numpy(), T, top_k=top_k)[0]
    np.testing.assert_array_equal(a, ea)
    assert (a < D).any()


def test_top_k_one_is_greedy_on_the_gpu():
    """top_k = 1 with drafts equal to the draft rows' argmax gives the greedy verifier's result."""
    gen = synth.make_gen(42)
    B, D, V = 16, 5, 32000
    tl, dl, _, u = synth.sampled_round(gen, B, D, V, 0.7, dtype=torch.bfloat16)
    draft = dl.float().argmax(-1).to(torch.int32)
    a, y, _, st = gpu_sample(tl, dl, draft, u, 0.7, residual=False, top_k=1)
    ga, gy = O.verify_greedy(tl.double().numpy(), draft.numpy())
    assert st == 0
    np.testing.assert_array_equal(a, ga)
    np.testing.assert_array_equal(y, gy)


def test_filtered_emitted_token_follows_filtered_p():
    rng = np.random.default_rng(43)
    V, n, T = 8, 200000, 0.7
    for k, tp in ((5, 1.0), (0, 0.8)):
        zp0, zp1, zq = (rng.normal(size=V) for _ in range(3))
        p0 = O.filtered_softmax(zp0, T, k, tp)
        p1 = O.filtered_softmax(zp1, T, k, tp)
        q0 = O.filtered_softmax(zq, T, k, tp)
        tl = torch.tensor(np.stack([zp0, zp1]), dtype=torch.float32)[None].expand(n, 2, V).contiguous()
        dl = torch.tensor(zq[None], dtype=torch.float32)[None].expand(n, 1, V).contiguous()
        draft = torch.tensor(rng.choice(V, size=(n, 1), p=q0), dtype=torch.int32)
        u = torch.tensor(rng.random((n, 2)), dtype=torch.float32)
        a, y, _, st = gpu_sample(tl, dl, draft, u, T, residual=False, top_k=k, top_p=tp)
        assert st == 0
        first = np.where(a >= 1, draft[:, 0].numpy(), y)
        m0, m1 = p0 > 0, p1 > 0
        assert (np.bincount(first, minlength=V)[~m0] == 0).all()
        assert stats.chisquare(np.bincount(first, minlength=V)[m0], p0[m0] * n).pvalue > 1e-3
        bonus = y[a == 1]
        assert stats.chisquare(np.bincount(bonus, minlength=V)[m1], p1[m1] * len(bonus)).pvalue > 1e-3


def test_filter_host_errors():
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(44)
    tl, dl, draft, u = synth.sampled_round(gen, 2, 2, 100, 0.7, dtype=torch.float32)
    bounds = torch.zeros((2, 5, 2), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for k, p in ((0, 0.0), (0, 1.5), (-1, 1.0)):
        with pytest.raises(sd.SpecdecError):
            sd.sampling_filter(tl.to(DEV), dl.to(DEV), 0.7, k, p, bounds, st)


@pytest.mark.parametrize("ties,top_k,top_p", [
    (65535, 1000, 1.0),      # a counter filled exactly: the histogram path, cut inside the ties
    (65535, 0, 0.9),
    (65536, 1000, 1.0),      # one more: the counter overflows, the row takes the radix path
    (70000, 0, 0.9),
    (70000, 100, 0.95),
])
def test_keep_bounds_many_equal_scores(ties, top_k, top_p):
    """bf16 rows (V = 151552) whose highest score is shared by `ties` tokens at spread-out
    indices: the value histogram holds up to 65535 equal scores; more send the row to the radix
    selection.  Either way the kept set equals the oracle's."""
    import speculative_decoding_specdec_gb300.specdec as sd
    B, D, V = 1, 1, 151552
    gen = synth.make_gen(77 + ties + top_k)
    tl, dl, _, _ = synth.sampled_round(gen, B, D, V, 0.7, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(ties)
    for row in (tl[0, 0], tl[0, 1], dl[0, 0]):
        idx = torch.randperm(V, generator=g)[:ties]
        row[idx] = 8.0                                  # above every N(0,1) score
    bounds = torch.zeros((B, 2 * D + 1, 2), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd.sampling_filter(tl.to(DEV), dl.to(DEV), 0.7, top_k, top_p, bounds, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bnd = bounds.cpu().numpy().astype(np.int64)
    rows = rows_of(tl.float().numpy(), dl.float().numpy())
    for q in range(2 * D + 1):
        got = kept_from_bounds(rows[0, q], bnd[0, q])
        exp = O.sampling_keep(rows[0, q].astype(np.float64), 0.7, top_k, top_p)
        if not np.array_equal(got, exp):   # top_p on a cumulative mass: either cut is exact
            assert O.top_p_margin(rows[0, q].astype(np.float64), 0.7, top_k, top_p) < 2e-6, q
            assert abs(int(got.sum()) - int(exp.sum())) == 1
        assert 0 < got.sum() < ties


@pytest.mark.parametrize("V,top_k,top_p,plant", [
    (20480, 128, 1.0, None),
    (20483, 7, 1.0, None),                 # ragged rows: aligned and unaligned rows in one CTA
    (32000, 100, 1.0, ((300, 8.0),)),      # the cut inside 300 equal top scores
    (32000, 100, 1.0, ((700, 8.0),)),
    (32000, 100, 1.0, ((5000, 8.0),)),
    (32000, 100, 1.0, ((60, 9.0), (200, 8.0))),   # the cut inside the second score value
    (32000, 10, 1.0, "constant"),          # every score equal
    (32000, 120, 0.5, ((300, 8.0),)),      # top-k then top-p, the cut inside equal scores
    (151552, 128, 0.9, None),              # top-p inside the top 128
    (151552, 1, 1.0, None),
])
def test_keep_bounds_ties_at_the_cut(V, top_k, top_p, plant):
    """Top-k (and top-k then top-p) cuts that fall inside a run of equal scores, so the bound's
    index comes from the tie search: kept sets equal the oracle's, with exactly k tokens kept,
    also on ragged rows and on a row of equal scores."""
    import speculative_decoding_specdec_gb300.specdec as sd
    B, D = 3, 2
    gen = synth.make_gen(900 + V + top_k)
    tl, dl, _, _ = synth.sampled_round(gen, B, D, V, 0.7, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(V + top_k)
    for rows3 in (tl, dl):
        for b in range(B):
            for j in range(rows3.shape[1]):
                if plant == "constant":
                    rows3[b, j] = 0.25
                elif plant:
                    idx = torch.randperm(V, generator=g)
                    at = 0
                    for n, val in plant:
                        rows3[b, j, idx[at:at + n]] = val
                        at += n
    bounds = torch.zeros((B, 2 * D + 1, 2), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd.sampling_filter(tl.to(DEV), dl.to(DEV), 0.7, top_k, top_p, bounds, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bnd = bounds.cpu().numpy().astype(np.int64)
    rows = rows_of(tl.float().numpy(), dl.float().numpy())
    for b in range(B):
        for q in range(2 * D + 1):
            got = kept_from_bounds(rows[b, q], bnd[b, q])
            exp = O.sampling_keep(rows[b, q].astype(np.float64), 0.7, top_k, top_p)
            if not np.array_equal(got, exp):
                assert top_p < 1.0, (b, q)
                assert O.top_p_margin(rows[b, q].astype(np.float64), 0.7, top_k, top_p) < 2e-6
            if top_p == 1.0:
                assert got.sum() == top_k


@pytest.mark.parametrize("seed,offset,B,D", [
    (0, 0, 3, 4),
    (2024, 7, 64, 6),
    (2 ** 64 - 1, 2 ** 40 + 3, 33, 31),        # every bit of seed and offset in use
    (5, 2 ** 32 - 1, 1, 1),
])
def test_philox_uniforms_match_the_oracle(seed, offset, B, D):
    """The uniforms the fused round draws in-kernel (Philox4x32-10) equal the oracle's, bit for
    bit (24-bit values are exact in fp32)."""
    import speculative_decoding_specdec_gb300.specdec as sd
    out = torch.full((B, D + 1), -1.0, device=DEV)
    sd.philox_uniforms(seed, offset, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64),
                                  O.philox_uniforms(seed, offset, B, D))


@pytest.mark.parametrize("B,D,V,dtype,top_k", [
    (32, 6, 151552, torch.bfloat16, 0),        # GLM-4-9B-shaped
    (8, 5, 32000, torch.bfloat16, 50),         # with top-k bounds
    (4, 31, 1000, torch.float32, 0),
])
def test_sample_with_in_kernel_uniforms(B, D, V, dtype, top_k):
    """Uniforms drawn in-kernel give exactly the result of passing the same uniforms explicitly,
    which matches the oracle."""
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(5000 + B + D)
    tl, dl, draft, _ = synth.sampled_round(gen, B, D, V, 0.7, dtype=dtype, draft_candidates=top_k)
    seed, offset = 99, 3
    u = torch.empty((B, D + 1), device=DEV)
    sd.philox_uniforms(seed, offset, u)
    torch.cuda.synchronize()
    if top_k:
        a1, y1, r1, st1 = gpu_sample(tl, dl, draft, u.cpu(), 0.7, top_k=top_k)
    else:
        a1, y1 = compare(tl, dl, draft, u.cpu(), 0.7)
        _, _, r1, st1 = gpu_sample(tl, dl, draft, u.cpu(), 0.7)
    assert st1 == 0
    tl_d, dl_d = tl.to(DEV), dl.to(DEV)
    bounds = None
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if top_k:
        bounds = torch.zeros((B, 2 * D + 1, 2), dtype=torch.int32, device=DEV)
        sd.sampling_filter(tl_d, dl_d, 0.7, top_k, 1.0, bounds, st)
    a = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    y = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    res = torch.full((B, V), -1.0, device=DEV)
    sd.verify_sample_philox(tl_d, dl_d, draft.to(DEV), seed, offset, 0.7, a, y, st, res,
                            keep_bounds=bounds)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(a.cpu().numpy(), a1)
    np.testing.assert_array_equal(y.cpu().numpy(), y1)
    np.testing.assert_array_equal(res.cpu().numpy(), r1)
