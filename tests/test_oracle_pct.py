"""Pins for the oracle's channel-conditioned outlier criterion
(zijie-tian.site sec. 3.1: a candidate is an outlier when it lies in an
outlier channel and its magnitude is among the globally smallest p%; sec.
3.2: the pool of capacity P keeps the outliers). The reading (oracle R14):
per flush, the n_oc channels with the largest max |k| over the candidates
are the outlier channels, the score is the squared norm over them, the
smallest ceil(p * candidates) scores are outliers, and the pool keeps the
min(P, that) most outlying; the rest are written back.

Nothing here touches the CUDA path. Pins:
- p = 100% over all d channels is the norm criterion itself, bit for bit;
- p = 0 keeps nothing: the norm criterion with P = 0;
- membership and pool scores against ``bruteforce.state_pct`` after every
  append, with forced ties;
- the pool sizes follow min(P, ceil(p (previous + G))) in every unit;
- a case worked by hand (``golden/pct_tiny.json``).
"""
import json
import os

import numpy as np
import pytest

from tests import bruteforce as bf

HERE = os.path.dirname(os.path.abspath(__file__))


def _keys(seed, B, Hkv, T, d, ties=True):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((B, Hkv, T, d))
    ch = rng.choice(d, size=4, replace=False)
    K[..., ch] *= 15
    K[rng.random((B, Hkv, T)) < 0.08] *= 0.03
    V = rng.standard_normal((B, Hkv, T, d))
    K, V = K.astype(np.float16), V.astype(np.float16)
    if ties and T > 12:
        K[:, :, 9::11] = K[:, :, 4:5]
    return K, V


def _coarse_keys(seed, T, d):
    """Small integers: max |k| ties across channels at almost every flush,
    so the channel tie rule decides the scores."""
    rng = np.random.default_rng(seed)
    K = rng.integers(-3, 4, size=(1, 1, T, d)).astype(np.float16)
    K[..., : d // 2] *= rng.integers(0, 2, size=(1, 1, T, d // 2)).astype(np.float16)
    return K


def _state_equal(a, b, units):
    for u in range(units):
        ea, eb = a.export_unit(u), b.export_unit(u)
        for k in ("bcount", "bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "tk", "tv", "pidx", "pnorm", "pk", "pv"):
            assert np.array_equal(ea[k], eb[k]), (u, k)


@pytest.mark.parametrize("B,Hkv,d,G,R,P,T", [(2, 2, 32, 8, 3, 5, 90), (1, 3, 64, 16, 0, 20, 150)])
def test_full_percent_over_all_channels_is_the_norm_criterion(oracle_mod, B, Hkv, d, G, R, P, T):
    K, V = _keys(1, B, Hkv, T, d)
    a = oracle_mod.OracleCache(B, Hkv, Hkv, d, G, R, P, pct=(10000, d))
    b = oracle_mod.OracleCache(B, Hkv, Hkv, d, G, R, P)
    a.prefill(K, V)
    b.prefill(K, V)
    _state_equal(a, b, B * Hkv)
    q = np.random.default_rng(2).standard_normal((B, Hkv, d)).astype(np.float16)
    assert np.array_equal(a.decode(q), b.decode(q))


def test_zero_percent_keeps_nothing(oracle_mod):
    B, Hkv, d, G, R, P, T = 1, 2, 32, 8, 2, 6, 70
    K, V = _keys(3, B, Hkv, T, d)
    a = oracle_mod.OracleCache(B, Hkv, Hkv, d, G, R, P, pct=(0, 4))
    b = oracle_mod.OracleCache(B, Hkv, Hkv, d, G, R, 0)
    a.prefill(K, V)
    b.prefill(K, V)
    for u in range(B * Hkv):
        ea, eb = a.export_unit(u), b.export_unit(u)
        assert ea["npool"] == 0
        for k in ("bcount", "bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "tk", "tv"):
            assert np.array_equal(ea[k], eb[k]), (u, k)


@pytest.mark.parametrize("d,G,R,P,pct,n_oc,T", [
    (32, 4, 1, 3, 3000, 2, 60),
    (32, 8, 0, 2, 2500, 4, 70),
    (64, 8, 3, 10, 5000, 6, 90),
    (32, 4, 2, 50, 10000, 3, 50),   # P larger than any candidate set
    (64, 16, 4, 4, 100, 8, 120),    # 1%: at most one outlier per flush
])
def test_membership_against_brute_force(oracle_mod, d, G, R, P, pct, n_oc, T):
    K, _ = _keys(d + G + pct, 1, 1, T, d)
    V = np.zeros_like(K)
    orc = oracle_mod.OracleCache(1, 1, 1, d, G, R, P, pct=(pct, n_oc))
    for t in range(T):
        orc.append(K[:, :, t], V[:, :, t])
        blocks, pool, tail, scores = bf.state_pct(K[0, 0, : t + 1], G, R, P, pct, n_oc)
        e = orc.export_unit(0)
        assert e["nf"] == len(blocks) and e["tail"] == len(tail)
        for j, blk in enumerate(blocks):
            assert e["bcount"][j] == len(blk)
            assert e["bidx"][j][: len(blk)].tolist() == blk, (t, j)
        got_pool = sorted(int(x) for x in e["pidx"][: e["npool"]])
        assert got_pool == pool, t
        for i in range(e["npool"]):
            want = np.float32(scores[int(e["pidx"][i])]).view(np.uint32)
            assert e["pnorm"][i] == want, (t, i)
        # every token once
        seen = [x for blk in blocks for x in blk] + pool + tail
        assert sorted(seen) == list(range(t + 1))


@pytest.mark.parametrize("n_oc", [1, 3, 7])
def test_channel_ties_against_brute_force(oracle_mod, n_oc):
    d, G, R, P, pct, T = 32, 8, 1, 6, 4000, 80
    K = _coarse_keys(n_oc, T, d)
    orc = oracle_mod.OracleCache(1, 1, 1, d, G, R, P, pct=(pct, n_oc))
    orc.prefill(K, np.zeros_like(K))
    blocks, pool, tail, scores = bf.state_pct(K[0, 0], G, R, P, pct, n_oc)
    e = orc.export_unit(0)
    assert [e["bidx"][j][: e["bcount"][j]].tolist() for j in range(e["nf"])] == blocks
    assert sorted(e["pidx"][: e["npool"]].tolist()) == pool


@pytest.mark.parametrize("P,pct,G", [(32, 100, 128), (32, 2000, 128), (5, 5000, 8), (64, 10000, 16), (3, 1, 7)])
def test_pool_sizes_follow_the_recurrence(oracle_mod, P, pct, G):
    d, R, T = 32, 2, 8 * G + 5
    K, V = _keys(P + pct, 2, 2, T, d, ties=False)
    orc = oracle_mod.OracleCache(2, 2, 2, d, G, R, P, pct=(pct, 5))
    orc.prefill(K, V)
    nf = bf.flush_count(T, G, R)
    want = bf.pct_pool_sizes(nf, G, P, pct)
    for u in range(4):
        e = orc.export_unit(u)
        assert e["npool"] == want[-1]
        prev = 0
        for j in range(nf):
            assert e["bcount"][j] == prev + G - want[j]
            prev = want[j]


def test_worked_by_hand(oracle_mod):
    g = json.load(open(os.path.join(HERE, "golden", "pct_tiny.json")))
    d, G, R, P = g["d"], g["G"], g["R"], g["P"]
    K = np.zeros((1, 1, len(g["keys_ch012"]), d), np.float16)
    K[0, 0, :, :3] = np.array(g["keys_ch012"], np.float16)
    V = np.zeros_like(K)
    orc = oracle_mod.OracleCache(1, 1, 1, d, G, R, P, pct=(g["pct"], g["n_oc"]))
    orc.prefill(K, V)
    e = orc.export_unit(0)
    assert [e["bidx"][j][: e["bcount"][j]].tolist() for j in range(e["nf"])] == g["blocks"]
    assert e["pidx"][: e["npool"]].tolist() == g["pool"]
    assert e["pnorm"][: e["npool"]].view(np.float32).tolist() == g["pool_scores"]
