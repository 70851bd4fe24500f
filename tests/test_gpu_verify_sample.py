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


def gpu_sample(tl, dl, draft, u, T, row_stride=None, residual=True):
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
    sd.verify_sample(place(tl), place(dl), draft.to(DEV), u.to(DEV), T, a, y, st, res)
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
