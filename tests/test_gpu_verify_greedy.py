"""Greedy verification on the GPU against the CPU oracle: bit-exact accept lengths and tokens.

Shapes: the tiny fp32 case, the Vicuna-7B-shaped (B=8, V=32000), Qwen3-8B-shaped (B=16,
V=151936) and pool-shaped (B=256, V=32000) full sizes, ragged vocabularies, padded and unaligned
row strides, ties, -inf/NaN rows, D from 1 to 31, and out-of-range drafts.
"""
import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_greedy(logits, draft, row_stride=None, ws=None):
    import speculative_decoding_specdec_gb300.specdec as sd
    B, Dp1, V = logits.shape
    if row_stride is None:
        x = logits.to(DEV)
    else:
        buf = torch.zeros(B * Dp1 * row_stride + 8, dtype=logits.dtype, device=DEV)
        x = buf[:B * Dp1 * row_stride].view(B, Dp1, row_stride)[:, :, :V]
        x.copy_(logits.to(DEV))
    a = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    y = torch.full((B,), -5, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if ws is None:
        ws = torch.zeros(sd.greedy_workspace_bytes(B, Dp1 - 1), dtype=torch.uint8,
                         device=DEV)
    sd.verify_greedy(x, draft.to(DEV), a, y, st, ws)
    torch.cuda.synchronize()
    return a.cpu().numpy(), y.cpu().numpy(), int(st.item())


def oracle_greedy(logits, draft):
    L = logits.double().numpy().copy()
    L[np.isnan(L)] = -np.inf        # NaN is never chosen (a NaN-only row is flagged separately)
    return O.verify_greedy(L, draft.numpy())


def check(logits, draft, row_stride=None):
    a, y, st = gpu_greedy(logits, draft, row_stride)
    ea, ey = oracle_greedy(logits, draft)
    assert st == 0
    np.testing.assert_array_equal(a, ea)
    np.testing.assert_array_equal(y, ey)
    return a


@pytest.mark.parametrize("B,D,V,dtype,alpha", [
    (2, 4, 1000, torch.float32, 0.7),          # tiny
    (8, 5, 32000, torch.bfloat16, 0.7),        # Vicuna-7B-shaped, full size
    (16, 4, 151936, torch.bfloat16, 0.6),      # Qwen3-8B-shaped, full size
    (256, 5, 32000, torch.bfloat16, 0.7),      # pool verification shape, full size
    (3, 3, 1003, torch.bfloat16, 0.5),         # ragged V (not a multiple of 8)
    (5, 2, 7, torch.bfloat16, 0.5),            # V smaller than one vector per slice
    (4, 1, 1, torch.float32, 0.5),             # V == 1
    (1, 31, 4099, torch.float32, 0.9),         # D = 31
    (1, 1, 50000, torch.bfloat16, 0.5),        # B = 1, D = 1
    (33, 6, 151552, torch.bfloat16, 0.7),      # GLM-4-shaped vocabulary
    (300, 3, 100, torch.bfloat16, 0.6),        # many batch rows per CTA share
    (97, 2, 1003, torch.float32, 0.6),         # shares cross rows and batch rows, ragged V
])
def test_greedy_matches_oracle(B, D, V, dtype, alpha):
    gen = synth.make_gen(1000 + B * 7 + D)
    logits, draft = synth.greedy_round(gen, B, D, V, alpha, dtype=dtype)
    check(logits, draft)


@pytest.mark.parametrize("alpha,expect", [(1.0, "all"), (0.0, "none")])
def test_all_and_none_accepted(alpha, expect):
    gen = synth.make_gen(11)
    logits, draft = synth.greedy_round(gen, 16, 5, 32000, alpha, dtype=torch.bfloat16)
    a = check(logits, draft)
    if expect == "all":
        assert (a == 5).all()
    else:
        assert (a == 0).mean() > 0.99


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ties_lowest_index(dtype):
    g = torch.Generator().manual_seed(3)
    B, D, V = 12, 4, 20000
    logits = torch.randint(0, 4, (B, D + 1, V), generator=g).to(dtype)   # many exact ties
    draft = torch.randint(0, 3, (B, D), generator=g, dtype=torch.int32)
    check(logits, draft)


@pytest.mark.parametrize("extra", [24, 3, 1])
def test_padded_row_stride(extra):
    """Rows padded to V + extra elements: 16-byte aligned rows (24) and the unaligned path."""
    gen = synth.make_gen(4)
    for dtype in (torch.bfloat16, torch.float32):
        logits, draft = synth.greedy_round(gen, 6, 3, 9000, 0.6, dtype=dtype)
        check(logits, draft, row_stride=9000 + extra)


def test_inf_and_nan_rows():
    gen = synth.make_gen(5)
    B, D, V = 6, 3, 4000
    logits, draft = synth.greedy_round(gen, B, D, V, 0.5, dtype=torch.float32)
    logits[0, 0, :] = -float("inf")             # all -inf: the lowest index wins
    logits[1, 1, ::3] = float("nan")            # NaN never chosen
    logits[2, 0, 17] = float("nan")
    logits[3, 2, 5] = float("inf")
    logits[3, 2, 900] = float("inf")            # tie of +inf: index 5
    draft[0, 0] = 0
    check(logits, draft)


def test_nan_only_row_sets_status():
    gen = synth.make_gen(6)
    logits, draft = synth.greedy_round(gen, 2, 2, 3000, 0.5, dtype=torch.float32)
    logits[1, 0, :] = float("nan")
    _, _, st = gpu_greedy(logits, draft)
    assert st == 5


def test_out_of_range_draft_sets_status_and_mismatches():
    gen = synth.make_gen(7)
    logits, draft = synth.greedy_round(gen, 4, 4, 3000, 1.0, dtype=torch.bfloat16)
    draft[2, 1] = 3000
    draft[3, 0] = -1
    a, y, st = gpu_greedy(logits, draft)
    assert st == 5
    assert a[0] == 4 and a[1] == 4 and a[2] == 1 and a[3] == 0
    L = logits.double().numpy()
    assert y[2] == int(np.argmax(L[2, 1])) and y[3] == int(np.argmax(L[3, 0]))


def test_empty_batch_and_host_errors():
    import speculative_decoding_specdec_gb300.specdec as sd
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    x = torch.zeros(0, 5, 100, dtype=torch.bfloat16, device=DEV)
    d = torch.zeros(0, 4, dtype=torch.int32, device=DEV)
    z = torch.zeros(0, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd.verify_greedy(x, d, z, z, st, ws)
    x = torch.zeros(1, 33, 100, dtype=torch.bfloat16, device=DEV)
    d = torch.zeros(1, 32, dtype=torch.int32, device=DEV)
    o = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(sd.SpecdecError) as e:
        sd.verify_greedy(x, d, o, o, st, ws)
    assert e.value.code == sd.ERR_UNSUPPORTED
    x = torch.zeros(8, 6, 32000, dtype=torch.bfloat16, device=DEV)   # workspace too small
    d = torch.zeros(8, 5, dtype=torch.int32, device=DEV)
    o = torch.zeros(8, dtype=torch.int32, device=DEV)
    rc = sd.lib.specdec_verify_greedy(x.data_ptr(), sd.BF16, 8, 5, 32000, 32000, d.data_ptr(),
                                      o.data_ptr(), o.data_ptr(), ws.data_ptr(), 64, st.data_ptr(),
                                      None)
    assert rc == sd.ERR_INVALID_ARG
    rc = sd.lib.specdec_verify_greedy(x.data_ptr(), sd.BF16, 8, 5, 32000, 32000, d.data_ptr(),
                                      o.data_ptr(), o.data_ptr(), ws.data_ptr() + 128, 1 << 19,
                                      st.data_ptr(), None)
    assert rc == sd.ERR_INVALID_ARG                                   # workspace not 256-aligned


def test_workspace_reused_across_calls():
    """One workspace, zero-filled once, serves consecutive calls of several shapes: every call
    (including one that reports an out-of-range draft) leaves it all zero again."""
    import speculative_decoding_specdec_gb300.specdec as sd
    gen = synth.make_gen(9)
    shapes = [(16, 4, 151936), (8, 5, 32000), (256, 5, 32000), (3, 3, 1003), (97, 2, 1003)]
    need = max(sd.greedy_workspace_bytes(B, D) for B, D, V in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for _ in range(2):
        for B, D, V in shapes:
            logits, draft = synth.greedy_round(gen, B, D, V, 0.6, dtype=torch.bfloat16)
            a, y, st = gpu_greedy(logits, draft, ws=ws)
            ea, ey = oracle_greedy(logits, draft)
            assert st == 0
            np.testing.assert_array_equal(a, ea)
            np.testing.assert_array_equal(y, ey)
            assert int(ws.count_nonzero()) == 0
    logits, draft = synth.greedy_round(gen, 4, 4, 3000, 1.0, dtype=torch.bfloat16)
    draft[1, 2] = 3000
    _, _, st = gpu_greedy(logits, draft, ws=ws)
    assert st == 5 and int(ws.count_nonzero()) == 0


def test_repeated_calls_deterministic():
    gen = synth.make_gen(8)
    logits, draft = synth.greedy_round(gen, 16, 4, 151936, 0.6, dtype=torch.bfloat16)
    r1 = gpu_greedy(logits, draft)
    r2 = gpu_greedy(logits, draft)
    assert (r1[0] == r2[0]).all() and (r1[1] == r2[1]).all()
