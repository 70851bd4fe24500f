"""EQSPEC realignment on the GPU against the CPU oracle.

Small and mid-size batches compare everything bit-exactly after every round (both copy engines).
The full-size Vicuna-7B-, Qwen3-8B- and GLM-4-9B-shaped caches run in the benchmark's launch
configuration and are checked through the oracle's column plan: every content column of every
row equals its source column (compared on the device), the metadata equals the oracle's, and a
sample of whole (layer, k/v) planes is realigned by the oracle itself and compared.
"""
import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth
from specdec_testlib import eqspec_rounds

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("copy_engine", [0, 1])
def test_tiny_fp32(copy_engine):
    eqspec_rounds(1, 2, 64, torch.float32, B=2, D=4, V=1000, rounds=3, prompt_lo=5, prompt_hi=20,
                  seed=0, copy_engine=copy_engine, alpha=0.7)


@pytest.mark.parametrize("copy_engine", [0, 1])
def test_multi_tile_ragged_bf16(copy_engine):
    # runs of up to ~730 columns x 256 B span several tiles (64 KB bulk, 32 KB vector) with a
    # ragged last tile
    eqspec_rounds(2, 4, 128, torch.bfloat16, B=8, D=5, V=500, rounds=4, prompt_lo=20,
                  prompt_hi=700, seed=1, copy_engine=copy_engine, alpha=0.7)


@pytest.mark.parametrize("B,D,lo,hi,hd,dtype", [
    (1, 4, 1, 40, 128, torch.bfloat16),       # one row
    (64, 3, 1, 12, 64, torch.bfloat16),       # many short rows (zero-shift and one-column runs)
    (5, 1, 3, 200, 32, torch.float32),        # D = 1
    (3, 31, 2, 100, 8, torch.bfloat16),       # D = 31, 16-byte columns
    (300, 2, 1, 6, 64, torch.float32),        # more rows than one CTA's threads
])
def test_shapes(B, D, lo, hi, hd, dtype):
    eqspec_rounds(2, 2, hd, dtype, B=B, D=D, V=300, rounds=3, prompt_lo=lo, prompt_hi=hi,
                  seed=B + D, alpha=0.6)


@pytest.mark.parametrize("B,D,lo,hi,hd,dtype,L,H", [
    (2, 4, 5, 20, 64, torch.float32, 1, 2),      # tiny
    (8, 5, 20, 300, 128, torch.bfloat16, 2, 4),  # multi-tile runs, ragged last tiles
    (4, 5, 300, 1300, 128, torch.bfloat16, 1, 2),  # runs of 2-6 tiles of 64 KB
    (64, 3, 1, 12, 64, torch.bfloat16, 2, 2),    # many short rows: zero-shift and one-column runs
    (3, 31, 2, 100, 8, torch.bfloat16, 2, 2),    # D = 31, 16-byte columns
    (300, 2, 1, 6, 64, torch.float32, 2, 2),     # more rows than one CTA's threads
])
def test_in_place(B, D, lo, hi, hd, dtype, L, H):
    """The whole buffer after an in-place realignment equals the oracle's realignment into a
    copy of the source: surviving columns moved, every other column untouched."""
    eqspec_rounds(L, H, hd, dtype, B=B, D=D, V=300, rounds=4, prompt_lo=lo, prompt_hi=hi,
                  seed=50 + B + D, alpha=0.6, in_place=True)


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("B,lo,hi,L,H", [
    (8, 20, 700, 2, 4),      # multi-tile runs with ragged last tiles
    (300, 1, 6, 2, 2),       # many one-tile runs, zero-shift rows
    (4, 300, 1300, 1, 2),    # runs of 2-6 tiles of 64 KB
])
def test_fixed_shares(in_place, B, lo, hi, L, H):
    """Without scheduling words every CTA moves one fixed share of the tiles: same results."""
    eqspec_rounds(L, H, 128, torch.bfloat16, B=B, D=5, V=300, rounds=3, prompt_lo=lo,
                  prompt_hi=hi, seed=90 + B, alpha=0.7, in_place=in_place, scheduled=False)


@pytest.mark.parametrize("copy_engine", [0, 1])
def test_in_place_long_shifts(copy_engine):
    # prompts of very different lengths: runs of up to ~730 columns shifting both ways
    eqspec_rounds(2, 2, 128, torch.bfloat16, B=6, D=6, V=200, rounds=5, prompt_lo=1,
                  prompt_hi=700, seed=77, alpha=0.9, in_place=True, copy_engine=copy_engine)


def test_in_place_rejects_a_different_destination():
    import speculative_decoding_specdec_gb300.specdec as sd
    buf = _one_round_buffers()
    a = sd.RealignArgs()
    a.src = sd.kv_view(buf["kv"][0])
    a.dst = sd.kv_view(buf["kv"][1])
    a.B, a.D = 4, 3
    for name, key in (("n_committed", "n"), ("width", "w"), ("accept_len", "a"), ("out_token", "y"),
                      ("draft", "d"), ("ids_src", None), ("ids_dst", None), ("pos_dst", "pos"),
                      ("n_committed_dst", "n2"), ("width_dst", "w2"), ("dev_status", "st")):
        t = buf["ids"][0] if name == "ids_src" else buf["ids"][1] if name == "ids_dst" else buf[key]
        setattr(a, name, t.data_ptr())
    a.mask_dst = buf["mask"].data_ptr()
    assert sd.lib.specdec_realign_inplace(sd.ctypes.byref(a), None) == sd.ERR_INVALID_ARG
    a.dst = sd.kv_view(buf["kv"][0])
    assert sd.lib.specdec_realign(sd.ctypes.byref(a), None) == sd.ERR_INVALID_ARG  # overlap


def test_all_rows_accept_everything():
    eqspec_rounds(1, 3, 64, torch.bfloat16, B=6, D=4, V=200, rounds=3, prompt_lo=10,
                  prompt_hi=90, seed=7, alpha=1.0)


def _one_round_buffers(B=4, D=3, L=2, H=2, hd=64, cap=40):
    dev = "cuda"
    kv = [torch.randn(L, 2, B, H, cap, hd, device=dev).to(torch.bfloat16) for _ in range(2)]
    ids = [torch.zeros(B, cap, dtype=torch.int32, device=dev) for _ in range(2)]
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32, device=dev)  # noqa: E731
    return dict(kv=kv, ids=ids, mask=torch.zeros(B, cap, dtype=torch.uint8, device=dev),
                pos=i32(B, cap), n=i32(B), n2=i32(B), w=i32(1), w2=i32(1), a=i32(B), y=i32(B),
                d=i32(B, D), st=i32(1))


def _call(buf, **over):
    import speculative_decoding_specdec_gb300.specdec as sd
    b = dict(buf, **over)
    sd.realign(b["kv"][0], b["kv"][1], b["n"], b["w"], b["a"], b["y"], b["d"], b["ids"][0],
               b["ids"][1], b["mask"], b["pos"], b["n2"], b["w2"], b["st"])
    torch.cuda.synchronize()
    return int(b["st"].item())


def test_capacity_error_writes_nothing():
    buf = _one_round_buffers(cap=40)
    buf["n"].copy_(torch.tensor([30, 10, 5, 36], dtype=torch.int32))
    buf["w"].fill_(36)
    buf["a"].fill_(3)                         # W' = 40 -> W' + D = 43 > 40
    before = buf["kv"][1].clone()
    assert _call(buf) == 4
    assert torch.equal(before, buf["kv"][1])
    assert int(buf["w2"].item()) == 0 and (buf["n2"] == 0).all()


@pytest.mark.parametrize("bad", ["accept", "length", "width"])
def test_range_errors_write_nothing(bad):
    buf = _one_round_buffers(cap=40)
    buf["n"].copy_(torch.tensor([3, 10, 5, 6], dtype=torch.int32))
    buf["w"].fill_(10)
    buf["a"].fill_(1)
    if bad == "accept":
        buf["a"][2] = 4                       # > D
    elif bad == "length":
        buf["n"][1] = 11                      # > W
    else:
        buf["w"].fill_(38)                    # W + D > source capacity
        buf["n"].fill_(3)
    before = buf["kv"][1].clone()
    assert _call(buf) == 5
    assert torch.equal(before, buf["kv"][1]) and (buf["n2"] == 0).all()


def test_host_errors():
    import speculative_decoding_specdec_gb300.specdec as sd
    buf = _one_round_buffers()
    kv0 = buf["kv"][0]
    n, hd = kv0.numel(), kv0.shape[-1]
    big = torch.zeros(n + hd, dtype=kv0.dtype, device=kv0.device)
    with pytest.raises(sd.SpecdecError):                    # overlapping, not the same view
        _call(buf, kv=[big[:n].view(kv0.shape), big[hd:].view(kv0.shape)])
    with pytest.raises(sd.SpecdecError):                    # lengths aliasing
        _call(buf, n2=buf["n"])
    odd = torch.zeros(1, 2, 4, 2, 40, 4, dtype=torch.bfloat16, device="cuda")   # 8-byte columns
    with pytest.raises(sd.SpecdecError) as e:
        _call(buf, kv=[odd, odd.clone()])
    assert e.value.code == sd.ERR_UNSUPPORTED


# ---------------------------------------------------------------------------------- full size

FULL = {
    "vicuna7b": dict(L=32, H=32, B=8, D=5, V=32000, lo=128, hi=1024, alpha=0.7, rounds=64),
    "qwen3_8b": dict(L=36, H=8, B=16, D=4, V=151936, lo=None, hi=None, alpha=0.6, rounds=64),
    "glm4_9b": dict(L=40, H=2, B=32, D=6, V=151552, lo=1024, hi=8192, alpha=0.7, rounds=32),
}


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("name", list(FULL))
def test_full_size_rounds(name, in_place):
    """Three rounds at the full cache size (capacity for the workload's full round count), with
    two cache buffers or one realigned in place."""
    from speculative_decoding_specdec_gb300.engine import EqspecBatch
    c = FULL[name]
    w = synth.WORKLOADS[name]
    gen = synth.make_gen(50 + w.seed)
    n0 = w.prompt_lengths(gen)
    cap = w.capacity(int(n0.max()))
    eng = EqspecBatch(c["L"], c["H"], 128, torch.bfloat16, c["B"], c["D"], cap, 3,
                      in_place=in_place)
    prompts = [torch.randint(0, c["V"], (int(n),), generator=gen).tolist() for n in n0]
    W = eng.start(prompts)
    g = torch.Generator(device="cuda").manual_seed(1)
    for k in eng.kv:                       # distinct random bits in every column
        k.view(torch.int16).random_(-32768, 32767, generator=g)
    n = n0.numpy().astype(np.int64)
    ids = eng.ids[0].cpu().numpy()
    rng = np.random.default_rng(0)
    for _ in range(3):
        logits, draft = synth.greedy_round(gen, c["B"], c["D"], c["V"], c["alpha"],
                                           dtype=torch.bfloat16)
        src = eng.cache.clone() if in_place else eng.cache   # the in-place move overwrites it
        dd = draft.cuda()
        eng.verify_greedy(logits.cuda(), dd)
        planes = [(int(rng.integers(c["L"])), int(rng.integers(2))) for _ in range(2)]
        src_planes = [src[l, kv].view(torch.int16).cpu().numpy() for l, kv in planes]
        dst_planes = [(src if in_place else eng.kv[1 - eng.cur])[l, kv].view(torch.int16)
                      .cpu().numpy() for l, kv in planes]
        eng.realign(dd)
        torch.cuda.synchronize()
        assert int(eng.status.item()) == 0
        a, y = O.verify_greedy(logits.double().numpy(), draft.numpy())
        np.testing.assert_array_equal(eng.accept_len.cpu().numpy(), a)
        n_new, W_new, src_lo, dst_lo, keep = O.realign_plan(n, W, a, c["D"])
        assert int(eng.width.item()) == W_new
        np.testing.assert_array_equal(eng.n_committed.cpu().numpy(), n_new)
        dst = eng.cache
        for b in range(c["B"]):            # every content column of every (layer, kv, head)
            s0, d0, k = int(src_lo[b]), int(dst_lo[b]), int(keep[b])
            assert torch.equal(dst[:, :, b, :, d0:d0 + k].view(torch.int16),
                               src[:, :, b, :, s0:s0 + k].view(torch.int16)), b
        for (l, kv), sp, dp in zip(planes, src_planes, dst_planes):
            exp = O.realign(sp[None, None], dp[None, None], n, W,
                            a, y, draft.numpy(), ids, 0)
            got = dst[l, kv].view(torch.int16).cpu().numpy()
            np.testing.assert_array_equal(got, exp[0][0, 0])
        _, ids, mask, pos, n, W = O.realign(np.zeros((1, 2, c["B"], 1, src.shape[4], 1), np.int8),
                                           np.zeros((1, 2, c["B"], 1, cap, 1), np.int8), n, W,
                                           a, y, draft.numpy(), ids, 0)
        np.testing.assert_array_equal(eng.ids[eng.cur].cpu().numpy(), ids)
        np.testing.assert_array_equal(eng.mask[eng.cur].cpu().numpy(), mask)
        np.testing.assert_array_equal(eng.pos[eng.cur].cpu().numpy(), pos)
        n = n.astype(np.int64)


@pytest.mark.parametrize("in_place", [False, True])
def test_rounds_with_programmatic_dependent_launch(in_place):
    """Realignment launched as a programmatic dependent of the verification (SPECDEC_REALIGN_PDL)
    gives the oracle's result in every round."""
    eqspec_rounds(2, 4, 128, torch.bfloat16, B=8, D=5, V=500, rounds=5, prompt_lo=20,
                  prompt_hi=300, seed=11, alpha=0.7, in_place=in_place, pdl=True)


@pytest.mark.parametrize("in_place", [False, True])
def test_graph_replay_rounds(in_place):
    """Rounds captured once into a CUDA graph (verification, then realignment as its programmatic
    dependent, taking work items from the batch's scheduling words) and replayed: every round's
    results, and both caches and the metadata after the last round, equal the oracle's.  The
    words are back at zero after every launch, or a later round would skip its items."""
    from speculative_decoding_specdec_gb300.engine import EqspecBatch
    from specdec_testlib import host_bits
    L, H, hd, B, D, V, R = 2, 4, 128, 8, 5, 500, 5
    gen = synth.make_gen(21)
    n0 = synth.lengths_uniform(gen, B, 20, 300)
    prompts = [torch.randint(0, V, (int(n),), generator=gen).tolist() for n in n0]
    cap = int(n0.max()) + R * (D + 1) + D + 1
    eng = EqspecBatch(L, H, hd, torch.bfloat16, B, D, cap, R, in_place=in_place, pdl=True)
    W = eng.start(prompts)
    g = torch.Generator(device="cuda").manual_seed(3)
    for k in eng.kv:
        k.view(torch.int16).random_(-32768, 32767, generator=g)
    rounds = [synth.greedy_round(gen, B, D, V, 0.7, dtype=torch.bfloat16) for _ in range(R)]
    dev_rounds = [(lg.cuda(), d.cuda()) for lg, d in rounds]
    eng.workspaces.greedy(dev_rounds[0][0], dev_rounds[0][1])      # allocated before capture
    bufs = [host_bits(k) for k in eng.kv]
    ids = eng.ids[0].cpu().numpy()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for lg, d in dev_rounds:
            eng.verify_greedy(lg, d)
            eng.realign(d)
    graph.replay()
    torch.cuda.synchronize()
    assert int(eng.status.item()) == 0
    assert eng.sched_words.tolist() == [0, 0]
    n = n0.numpy().astype(np.int64)
    hist = eng.hist.cpu().numpy()
    for r, (lg, d) in enumerate(rounds):
        a, y = O.verify_greedy(lg.double().numpy(), d.numpy())
        s_, d_ = (0, 0) if in_place else (r % 2, 1 - r % 2)
        src = bufs[s_]
        dst_before = src.copy() if in_place else bufs[d_]
        kv, ids, mask, pos, n, W = O.realign(src, dst_before, n, W, a, y, d.numpy(), ids, 0)
        bufs[d_] = kv
        np.testing.assert_array_equal(hist[r, B + 1:2 * B + 1], a)
        np.testing.assert_array_equal(hist[r, 2 * B + 1:], y)
        np.testing.assert_array_equal(hist[r + 1, :B], n)
        assert int(hist[r + 1, B]) == W
    for k, exp in zip(eng.kv, bufs):
        np.testing.assert_array_equal(host_bits(k), exp)
    np.testing.assert_array_equal(eng.ids[eng.cur].cpu().numpy(), ids)
    np.testing.assert_array_equal(eng.mask[eng.cur].cpu().numpy(), mask)
    np.testing.assert_array_equal(eng.pos[eng.cur].cpu().numpy(), pos)
