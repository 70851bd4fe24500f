"""Rounds fed from pinned host memory (engine.HostRounds): the copy stream's overlap must not
change what a round computes.  Each round's accept lengths, tokens, lengths and width come back to
the host and are compared with the oracle run on the same inputs, and the cache's content columns
with the oracle's realigned cache, for greedy and sampled rounds."""
import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth
from specdec_testlib import host_bits

pytestmark = pytest.mark.gpu


def _batch(B, D, V, rounds, seed, in_place, L=2, H=2, hd=64):
    from speculative_decoding_specdec_gb300.engine import EqspecBatch
    gen = synth.make_gen(seed)
    n0 = synth.lengths_uniform(gen, B, 3, 30)
    prompts = [torch.randint(0, V, (int(n),), generator=gen).tolist() for n in n0]
    cap = int(n0.max()) + rounds * (D + 1) + D + 1
    eng = EqspecBatch(L, H, hd, torch.float32, B, D, cap, rounds, in_place=in_place, pdl=True)
    W = eng.start(prompts)
    eng.cache.normal_(generator=torch.Generator(device="cuda").manual_seed(seed))
    return gen, eng, prompts, W


@pytest.mark.parametrize("in_place,depth", [(True, 2), (False, 2), (True, 1), (True, 4),
                                            (False, 8)])
@pytest.mark.parametrize("B,D,V", [(3, 4, 1000), (8, 5, 4099)])
def test_greedy_host_rounds_match_oracle(B, D, V, in_place, depth):
    """Staging depths 1 (no overlap), 2, 4 and 8 (more sets than rounds) commit the same."""
    from speculative_decoding_specdec_gb300.engine import HostRounds
    rounds = 6
    gen, eng, prompts, W = _batch(B, D, V, rounds, 11 + B, in_place)
    host = []
    for _ in range(rounds):
        lg, d = synth.greedy_round(gen, B, D, V, 0.7, dtype=torch.float32)
        host.append({"logits": lg.pin_memory(), "draft": d.pin_memory()})
    feed = HostRounds(eng, host[0], depth=depth)
    assert feed.h2d_bytes == B * (D + 1) * V * 4 + B * D * 4
    out = torch.zeros((rounds, 3 * B + 1), dtype=torch.int32).pin_memory()
    src0 = host_bits(eng.cache)
    dst0 = src0.copy() if in_place else host_bits(eng.kv[1])
    ids = eng.ids[0].cpu().numpy()
    feed.run(host, lambda d: eng.verify_greedy(d["logits"], d["draft"]), out)
    torch.cuda.synchronize()
    assert int(eng.status.item()) == 0
    n = np.array([len(p) for p in prompts])
    kv, other = src0, dst0
    for r in range(rounds):
        d = host[r]["draft"].numpy()
        a, y = O.verify_greedy(host[r]["logits"].double().numpy(), d)
        kv_new, ids, _, _, n, W = O.realign(kv, kv.copy() if in_place else other, n, W, a, y, d,
                                            ids, 0)
        kv, other = kv_new, kv
        got = out[r].numpy()
        np.testing.assert_array_equal(got[:B], a)
        np.testing.assert_array_equal(got[B:2 * B], y)
        np.testing.assert_array_equal(got[2 * B:3 * B], n)
        assert got[3 * B] == W
    got_kv = host_bits(eng.cache)
    for b in range(B):   # content columns [W - n_b, W - 1)
        np.testing.assert_array_equal(got_kv[:, :, b, :, W - n[b]:W - 1],
                                      kv[:, :, b, :, W - n[b]:W - 1])


def test_sampled_host_rounds_match_device_rounds():
    """Sampled rounds with uniforms as host inputs: the host-fed run commits exactly what the same
    rounds commit from device-resident inputs (the sampled parity itself is tested elsewhere)."""
    from speculative_decoding_specdec_gb300.engine import HostRounds
    B, D, V, T, rounds = 4, 3, 2000, 0.7, 5
    gen, eng, prompts, W = _batch(B, D, V, rounds, 5, True)
    host = []
    for _ in range(rounds):
        tl, dl, d, u = synth.sampled_round(gen, B, D, V, T, dtype=torch.float32)
        host.append({"logits": tl.pin_memory(), "draft_logits": dl.pin_memory(),
                     "draft": d.pin_memory(), "uniforms": u.pin_memory()})
    want = []
    for h in host:
        dv = {k: v.cuda() for k, v in h.items()}
        eng.verify_sample(dv["logits"], dv["draft_logits"], dv["draft"], dv["uniforms"], T)
        eng.realign(dv["draft"])
        want.append(torch.cat([eng.accept_len, eng.out_token, eng.n_committed,
                               eng.width]).cpu())
    for depth in (2, 3):
        eng.start(prompts)
        feed = HostRounds(eng, host[0], depth=depth)
        out = torch.zeros((rounds, 3 * B + 1), dtype=torch.int32).pin_memory()
        feed.run(host, lambda d: eng.verify_sample(d["logits"], d["draft_logits"], d["draft"],
                                                   d["uniforms"], T), out)
        torch.cuda.synchronize()
        assert int(eng.status.item()) == 0
        for r in range(rounds):
            assert out[r].tolist() == want[r].tolist()


def test_host_rounds_rejects_unpinned_output():
    from speculative_decoding_specdec_gb300.engine import HostRounds
    gen, eng, _, _ = _batch(2, 2, 100, 1, 1, True)
    lg, d = synth.greedy_round(gen, 2, 2, 100, 0.5, dtype=torch.float32)
    feed = HostRounds(eng, {"logits": lg, "draft": d})
    with pytest.raises(ValueError):
        feed.run([{"logits": lg, "draft": d}], lambda x: None, torch.zeros((1, 7), dtype=torch.int32))
