"""EXSPEC length grouping on the GPU against the CPU oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle.specdec_oracle as O

pytestmark = pytest.mark.gpu


def gpu_group(lengths, bs, max_len):
    import speculative_decoding_specdec_gb300.specdec as sd
    N = len(lengths)
    dev = "cuda"
    L = torch.as_tensor(np.asarray(lengths, dtype=np.int32), device=dev)
    perm = torch.full((max(N, 1),), -1, dtype=torch.int32, device=dev)
    off = torch.full((N + 1,), -1, dtype=torch.int32, device=dev)
    uni = torch.full((max(N, 1),), 9, dtype=torch.uint8, device=dev)
    nb = torch.full((1,), -1, dtype=torch.int32, device=dev)
    nu = torch.full((1,), -1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    sd.group_by_length(L, bs, max_len, perm, off, uni, nb, nu, st)
    torch.cuda.synchronize()
    k = int(nb.item())
    return (perm.cpu().numpy()[:N], off.cpu().numpy()[:k + 1], uni.cpu().numpy()[:k],
            int(nu.item()), int(st.item()), k)


def check(lengths, bs, max_len):
    perm, off, uni, nu, st, k = gpu_group(lengths, bs, max_len)
    assert st == 0
    ep, eo, eu, enu = O.group_by_length(lengths, bs)
    assert k == len(eu) and nu == enu
    np.testing.assert_array_equal(perm, ep)
    np.testing.assert_array_equal(off, eo)
    np.testing.assert_array_equal(uni, eu)


@pytest.mark.parametrize("seed", range(12))
def test_random_pools(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 600))
    bs = int(rng.integers(1, 12))
    distinct = int(rng.integers(1, 20))
    values = rng.choice(3000, size=distinct, replace=False)
    check(rng.choice(values, size=N), bs, 3000)


def test_pool_shape():
    """256 rows, batch size 8, lengths from {256, 512, ..., 2048} (and after some growth)."""
    rng = np.random.default_rng(4)
    lens = rng.choice(np.arange(256, 2049, 256), size=256)
    check(lens, 8, 2048 + 128 * 6 + 6)
    check(lens + rng.integers(1, 7, size=256), 8, 4096)


@pytest.mark.parametrize("lengths,bs,max_len", [
    ([], 8, 10), ([5], 8, 10), ([3] * 16, 8, 10), ([3] * 17, 8, 10), ([0, 16383, 0], 2, 16383),
    (list(range(40)), 1, 100), ([7, 7, 7], 4, 7), (list(np.arange(4096) % 5), 8, 4),
])
def test_edges(lengths, bs, max_len):
    check(lengths, bs, max_len)


def test_out_of_range_length_sets_status():
    perm, off, uni, nu, st, k = gpu_group([3, 11, 2], 2, 10)
    assert st == 5 and k == -1
