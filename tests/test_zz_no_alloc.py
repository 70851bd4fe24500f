"""The workspace-free greedy entry point against the workspace one, through the C ABI.

specdec_verify_greedy_noalloc runs the greedy kernel on a static per-device scratch array; two
calls in a row (different shapes, so the second reuses what the first left behind) must give
exactly the accept lengths and tokens of specdec_verify_greedy with a fresh workspace, and both
those of the CPU oracle.  The file is named to be collected last, so it also runs after every
other test in one process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O
from speculative_decoding_specdec_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outputs(B):
    a = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    y = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    return a, y, st


def test_noalloc_matches_workspace_entry_point_two_calls():
    import speculative_decoding_specdec_gb300.specdec as sd
    L = sd.lib
    gen = synth.make_gen(21, DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for B, D, V in ((16, 4, 151936), (8, 5, 32000)):
        logits, draft = synth.greedy_round(gen, B, D, V, 0.6, dtype=torch.bfloat16, device=DEV)
        a0, y0, s0 = _outputs(B)
        ws = torch.zeros(L.specdec_verify_greedy_workspace(B, D), dtype=torch.uint8, device=DEV)
        assert L.specdec_verify_greedy(logits.data_ptr(), sd.BF16, B, D, V, V, draft.data_ptr(),
                                       a0.data_ptr(), y0.data_ptr(), ws.data_ptr(), ws.numel(),
                                       s0.data_ptr(), stream) == sd.OK
        a1, y1, s1 = _outputs(B)
        assert L.specdec_verify_greedy_noalloc(logits.data_ptr(), sd.BF16, B, D, V, V,
                                               draft.data_ptr(), a1.data_ptr(), y1.data_ptr(),
                                               s1.data_ptr(), stream) == sd.OK
        torch.cuda.synchronize()
        assert int(s0.item()) == 0 and int(s1.item()) == 0
        np.testing.assert_array_equal(a1.cpu().numpy(), a0.cpu().numpy())
        np.testing.assert_array_equal(y1.cpu().numpy(), y0.cpu().numpy())
        ea, ey = O.verify_greedy(logits.cpu().double().numpy(), draft.cpu().numpy())
        np.testing.assert_array_equal(a1.cpu().numpy(), ea)
        np.testing.assert_array_equal(y1.cpu().numpy(), ey)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import speculative_decoding_specdec_gb300.specdec as sd
    B, D, V = 4096, 5, 8          # 4096 * 6 keys of 8 bytes: more than the static scratch
    assert sd.lib.specdec_verify_greedy_workspace(B, D) > sd.GREEDY_SCRATCH_BYTES
    logits = torch.zeros(B, D + 1, V, dtype=torch.bfloat16, device=DEV)
    draft = torch.zeros(B, D, dtype=torch.int32, device=DEV)
    a, y, st = _outputs(B)
    with pytest.raises(sd.SpecdecError) as e:
        sd.verify_greedy_noalloc(logits, draft, a, y, st)
    assert e.value.code == sd.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and (a.cpu().numpy() == -7).all()
