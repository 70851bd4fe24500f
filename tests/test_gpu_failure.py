"""Device-side failure reporting on the GPU, without a fault: the bounded wait every streaming
kernel uses runs out on a barrier that nothing completes (no copy is in flight), the kernel
records SPECDEC_ERR_TIMEOUT in the caller's status word and exits, and the context stays usable
(a greedy verification right after it matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("polls,sleep_ns", [(1, 0), (64, 1000), (2000, 5000)])
def test_bounded_wait_runs_out_and_reports_timeout(polls, sleep_ns):
    import speculative_decoding_specdec_gb300.specdec as sd
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sd.wait_selftest(polls, sleep_ns, st)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(st.item()) == sd.ERR_TIMEOUT
    assert elapsed < 2.0
    # the first code written stays
    st2 = torch.full((1,), sd.ERR_CAPACITY, dtype=torch.int32, device=DEV)
    sd.wait_selftest(polls, sleep_ns, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == sd.ERR_CAPACITY


def test_context_usable_after_a_timeout():
    import speculative_decoding_specdec_gb300.specdec as sd
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sd.wait_selftest(100, 1000, st)
    gen = synth.make_gen(61)
    B, D, V = 8, 5, 32000
    logits, draft = synth.greedy_round(gen, B, D, V, 0.7)
    a = torch.empty(B, dtype=torch.int32, device=DEV)
    y = torch.empty(B, dtype=torch.int32, device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.zeros(sd.greedy_workspace_bytes(B, D), dtype=torch.uint8, device=DEV)
    sd.verify_greedy(logits.to(DEV), draft.to(DEV), a, y, st2, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == sd.ERR_TIMEOUT and int(st2.item()) == 0
    ea, ey = O.verify_greedy(logits.double().numpy(), draft.numpy())
    np.testing.assert_array_equal(a.cpu().numpy(), ea)
    np.testing.assert_array_equal(y.cpu().numpy(), ey)


def test_selftest_host_checks():
    import speculative_decoding_specdec_gb300.specdec as sd
    L = sd.lib
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert L.specdec_wait_selftest(0, 0, st.data_ptr(), None) == sd.ERR_INVALID_ARG
    assert L.specdec_wait_selftest((1 << 20) + 1, 0, st.data_ptr(), None) == sd.ERR_INVALID_ARG
    assert L.specdec_wait_selftest(1, 1000001, st.data_ptr(), None) == sd.ERR_INVALID_ARG
    assert L.specdec_wait_selftest(1, 0, None, None) == sd.ERR_INVALID_ARG
