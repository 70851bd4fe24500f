"""Host-side argument checks of the engine's caller-side state (no GPU needed)."""
import types

import pytest
import torch

from speculative_decoding_specdec_gb300.engine import HostRounds


@pytest.mark.parametrize("depth", [0, -1])
def test_host_rounds_rejects_depth_below_one(depth):
    batch = types.SimpleNamespace(status=torch.zeros(1, dtype=torch.int32), B=2)
    with pytest.raises(ValueError):
        HostRounds(batch, {}, depth=depth)
