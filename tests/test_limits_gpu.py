"""GPU parity at the limits the library accepts: the largest outlier pool
whose flush staging fits one CTA's shared memory, a batch with more
(sequence, kv head) units than the decode grid has warps, one or two units
long enough that every decode warp holds a piece of them, and a ragged batch
of the maximum 256 sequences. Same bar as the other parity tests: state
bit-exact against the CPU oracle, outputs within max |d| <= 2e-3 and mean
|d| <= 2e-4 of its double result.
"""
import numpy as np
import pytest

from tests.test_parity_gpu import _run_small
from tests.test_ragged_gpu import _run as _run_ragged

pytestmark = pytest.mark.gpu


def _largest_pool(ott, d, G):
    """The largest P that ott_create accepts for (d, G), found by asking it."""
    P = 1024
    while P > 0:
        try:
            with ott.OTTCache(1, 1, 1, d, G, 4, P, max_tokens=64):
                return P
        except ott.OTTError as e:
            assert e.code == ott.OTT_ERR_INVALID
            P -= 2
    raise AssertionError("no pool size accepted")


def test_largest_pool_accepted(oracle_mod, ott):
    """d=128, G=128: the pool at its largest; 9 flushes fill it and keep evicting."""
    P = _largest_pool(ott, 128, 128)
    assert 200 <= P <= 320, P
    with pytest.raises(ott.OTTError):
        ott.OTTCache(1, 1, 1, 128, 128, 4, P + 2, max_tokens=64)
    _run_small(oracle_mod, ott, 1, 2, 1, 128, 128, 32, P, 1100, 30, seed=P, check_every_step=False)


def test_more_units_than_decode_warps(oracle_mod, ott):
    """64 sequences x 32 kv heads = 2048 units (the grid has 16 warps per SM)."""
    _run_small(oracle_mod, ott, 64, 32, 32, 128, 16, 4, 5, 90, 6, seed=64, check_every_step=False)


def test_ragged_at_the_sequence_limit(oracle_mod, ott):
    rng = np.random.default_rng(256)
    lens = [int(x) for x in rng.integers(1, 70, size=256)]
    _run_ragged(oracle_mod, ott, 256, 2, 1, 64, 16, 2, 3, lens, 20, seed=256, every=10)


@pytest.mark.parametrize("B,Hq,Hkv,G,R,P,L", [
    (1, 2, 1, 4, 1, 2, 10000),     # one unit of 2,500 blocks: every decode warp holds a piece of it
    (1, 8, 2, 8, 2, 5, 12000),     # two GQA units of 1,500 blocks
])
def test_one_long_unit(oracle_mod, ott, B, Hq, Hkv, G, R, P, L):
    """Thousands of blocks in one or two units: every decode warp holds a
    piece of a unit, and the combine merges thousands of partials per head."""
    _run_small(oracle_mod, ott, B, Hq, Hkv, 128, G, R, P, L, 3, seed=L + G, check_every_step=False)
