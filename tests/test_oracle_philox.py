"""Pins of the oracle's counter-based generator (Philox, "Parallel Random Numbers: As Easy as 1,
2, 3", SC11), used for the uniforms a fused round draws in-kernel.

The 32-bit-word instance the uniforms use is checked against the published Philox4x32-10
known-answer vectors of the Random123 library (tests/golden/philox4x32_10_kat.json): a wrong digit
in either multiplier or Weyl increment, or a wrong round or key schedule, changes every output
word.  The 64-bit-word instance is checked against numpy's Philox4x64-10 bit generator (a library
routine).  Properties pin the rest."""
import json
import os

import numpy as np
import pytest

import oracle.specdec_oracle as O


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def _kat():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _kat()["cases"])
def test_philox4x32_10_known_answers(case):
    """The published Random123 known-answer vectors: zero counter and key, all ones, and the
    counter and key taken from the hexadecimal digits of pi."""
    h = lambda words: [int(w, 16) for w in words]  # noqa: E731
    assert O.philox(h(case["ctr"]), h(case["key"]), bits=32, rounds=_kat()["rounds"]) == h(case["out"])


@pytest.mark.parametrize("which", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_philox4x32_known_answers_catch_a_changed_constant(monkeypatch, which):
    """Planted mistakes: one multiplier or Weyl increment with its lowest digit changed no
    longer reproduces any of the known answers."""
    M, W = O.PHILOX_CONSTANTS[32]
    consts = [list(M), list(W)]
    consts[which[0]][which[1]] ^= 0x2
    monkeypatch.setitem(O.PHILOX_CONSTANTS, 32, (tuple(consts[0]), tuple(consts[1])))
    h = lambda words: [int(w, 16) for w in words]  # noqa: E731
    for case in _kat()["cases"]:
        assert O.philox(h(case["ctr"]), h(case["key"]), bits=32) != h(case["out"])


@pytest.mark.parametrize("ctr,key", [
    ((0, 0, 0, 0), (0, 0)),
    ((5, 7, 11, 13), (123456789, 987654321)),
    ((2 ** 64 - 2, 3, 0, 9), (2 ** 63 + 5, 77)),        # the counter's low word carries
    ((2 ** 64 - 1, 2 ** 64 - 1, 2 ** 64 - 1, 2 ** 64 - 7), (2 ** 64 - 1, 2 ** 64 - 1)),
])
def test_philox4x64_matches_numpy(ctr, key):
    bg = np.random.Philox(counter=np.array(ctr, dtype=np.uint64),
                          key=np.array(key, dtype=np.uint64))
    raw = [int(x) for x in bg.random_raw(8)]
    c = list(ctr)
    for blk in range(2):                 # numpy advances the counter before each block
        c[0] = (c[0] + 1) % 2 ** 64
        k = 1
        while c[k - 1] == 0 and k < 4:
            c[k] = (c[k] + 1) % 2 ** 64
            if c[k]:
                break
            k += 1
        assert raw[4 * blk:4 * blk + 4] == O.philox(c, key, bits=64)


def test_weyl_constants_of_the_two_widths_agree():
    """The 32-bit key increments are the top halves of the 64-bit ones (both the golden ratio
    and sqrt(3) - 1 in fixed point): checked through the key schedule itself."""
    one32 = O.philox((0, 0, 0, 0), (0, 0), bits=32, rounds=1)
    two32 = O.philox((0, 0, 0, 0), (0, 0), bits=32, rounds=2)
    assert one32 == [0, 0, 0, 0]          # M * 0 = 0 and key 0: the first round maps 0 to 0
    # second round: key = (W0, W1), counter 0 -> (W0, 0, W1, 0)
    assert two32 == [0x9E3779B9, 0, 0xBB67AE85, 0]
    two64 = O.philox((0, 0, 0, 0), (0, 0), bits=64, rounds=2)
    assert two64[0] >> 32 == two32[0] and two64[2] >> 32 == two32[2]
    assert abs(two64[0] / 2 ** 64 - (np.sqrt(5) - 1) / 2) < 1e-15
    assert abs(two64[2] / 2 ** 64 - (np.sqrt(3) - 1)) < 1e-15


def test_uniforms_range_layout_and_distribution():
    u = O.philox_uniforms(seed=2024, offset=7, B=64, D=6)
    assert u.shape == (64, 7) and (u >= 0).all() and (u < 1).all()
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))          # 24-bit values
    # the same (seed, offset) gives the same uniforms; another offset or seed others
    assert np.array_equal(u, O.philox_uniforms(2024, 7, 64, 6))
    assert not np.array_equal(u, O.philox_uniforms(2024, 8, 64, 6))
    assert not np.array_equal(u, O.philox_uniforms(2025, 7, 64, 6))
    # u[b][j] for j < 4 and 4 <= j < 8 come from consecutive counters of row b
    x = O.philox((1, 5, 7, 0), (2024, 0))
    assert [int(v * 2 ** 24) for v in u[5, 4:7]] == [w >> 8 for w in x[:3]]
    # uniformity: chi-square over 64 bins of 20000 draws
    v = O.philox_uniforms(seed=1, offset=0, B=2500, D=7).ravel()
    h = np.bincount((v * 64).astype(int), minlength=64)
    e = len(v) / 64
    chi2 = float(((h - e) ** 2 / e).sum())
    assert chi2 < 120                      # 63 degrees of freedom: p ~ 1e-5 at 120
