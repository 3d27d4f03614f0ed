"""Pins for the oracle's cold-pool policy (zijie-tian.site sec. 3.2: a token
displaced from the outlier pool may go to a small "cold" pool instead of
being written back; the pages give it 32 slots). The reading: displaced
tokens enter an fp16 first-in-first-out pool of capacity C in ascending token
order, the earliest leave (discarded) when it overflows, the new block is the
group's tokens that did not enter the pool, and decode attends the cold pool
like the outlier pool.

Nothing here touches the CUDA path. The pins are independent of the oracle's
flush-by-flush merge:
- membership against ``bruteforce.state_cold``, which states it globally
  from the P smallest of every flushed prefix;
- decode on two-level inputs, where 2-bit quantization is exact, against
  float64 softmax attention over exactly the tokens that were not discarded;
- with no eviction possible (P >= T) the policy changes nothing.
"""
import numpy as np
import pytest
import torch

from tests import bruteforce as bf


def _falling_keys(seed, T, d):
    """fp16 keys whose norms tend to fall with the token index, so that new
    groups keep displacing pool tokens; a few exact duplicates force ties."""
    rng = np.random.default_rng(seed)
    base = rng.standard_normal((T, d)) * np.linspace(3.0, 0.3, T)[:, None]
    base[rng.random(T) < 0.1] *= 0.05
    K = base.astype(np.float16)
    if T > 8:
        K[5::7] = K[3]
    return K


def _two_level(seed, T, d, falling=True):
    """Keys and values that 2-bit quantization represents exactly: every
    channel of a key takes one of two values lo_c, lo_c + 3*2^-4, and every
    32-channel group of a value one of two values lo, lo + 3*2^-3. Later keys
    pick the high level less often, so their norms tend to fall."""
    rng = np.random.default_rng(seed)
    lo_k = rng.integers(-8, 9, size=d) * 2.0 ** -4
    p_hi = np.linspace(0.9, 0.1, T) if falling else np.full(T, 0.5)
    hi = rng.random((T, d)) < p_hi[:, None]
    K = (lo_k[None, :] + hi * 3 * 2.0 ** -4).astype(np.float16)
    ng = d // 32
    lo_v = rng.integers(-16, 17, size=(T, ng)) * 2.0 ** -3
    hv = rng.random((T, d)) < 0.5
    V = (np.repeat(lo_v, 32, axis=1) + hv * 3 * 2.0 ** -3).astype(np.float16)
    return K, V


def _attend(q16, K16, V16, toks):
    q = q16.astype(np.float64)
    k = K16[toks].astype(np.float64)
    v = V16[toks].astype(np.float64)
    s = (k @ q) / np.sqrt(len(q))
    w = np.exp(s - s.max())
    return (w[:, None] * v).sum(0) / w.sum()


@pytest.mark.parametrize("d,G,R,P,C,T", [
    (32, 8, 2, 3, 2, 90),      # the cold pool overflows often
    (32, 8, 0, 4, 0, 70),      # C = 0: every displaced token is discarded
    (64, 16, 4, 5, 32, 640),   # the pages' C = 32
    (32, 4, 1, 9, 3, 60),      # P > G: several flushes before the pool is full
    (32, 8, 3, 0, 4, 50),      # P = 0: nothing is pooled, nothing displaced
])
def test_cold_membership_matches_bruteforce_every_append(oracle_mod, d, G, R, P, C, T):
    K = _falling_keys(d + G + P + C, T, d)
    V = np.random.default_rng(1).standard_normal((T, d)).astype(np.float16)
    orc = oracle_mod.OracleCache(1, 1, 1, d, G, R, P, cold=C)
    evictions = 0
    for t in range(T):
        orc.append(K[t][None, None], V[t][None, None])
        blocks, pool, tail, cold, dropped = bf.state_cold(K[: t + 1], G, R, P, C)
        e = orc.export_unit(0)
        assert e["nf"] == len(blocks) and e["tail"] == len(tail) and e["npool"] == len(pool)
        for j, blk in enumerate(blocks):
            assert e["bcount"][j] == len(blk)
            assert e["bidx"][j][: len(blk)].tolist() == blk
            assert np.all(e["bidx"][j][len(blk):] == -1)
        assert sorted(x for x in e["pidx"].tolist() if x >= 0) == pool
        assert e["ncold"] == len(cold)
        assert e["cidx"][: len(cold)].tolist() == cold
        # the cold rows hold the tokens' own fp16 values
        for i, tok in enumerate(cold):
            assert np.array_equal(e["ck"][i], K[tok].view(np.uint16))
            assert np.array_equal(e["cv"][i], V[tok].view(np.uint16))
        # every token seen sits in exactly one place
        placed = sum((list(b) for b in blocks), []) + pool + tail + cold + dropped
        assert sorted(placed) == list(range(t + 1))
        evictions = len(cold) + len(dropped)
    if P > 0:
        assert evictions > C, "the inputs must overflow the cold pool"


@pytest.mark.parametrize("C", [0, 3, 32, 10_000])
def test_cold_decode_is_exact_attention_over_the_kept_tokens(oracle_mod, C):
    d, G, R, P, T = 64, 16, 4, 6, 260
    K, V = _two_level(11 + C, T, d)
    orc = oracle_mod.OracleCache(1, 2, 1, d, G, R, P, cold=C)
    orc.prefill(K[None, None], V[None, None])
    _, _, _, cold, dropped = bf.state_cold(K, G, R, P, C)
    if C == 10_000:
        assert not dropped
    else:
        assert dropped
    kept = sorted(set(range(T)) - set(dropped))
    q = np.random.default_rng(3).standard_normal((1, 2, d)).astype(np.float16)
    out = orc.decode(q)
    for h in range(2):
        ref = _attend(q[0, h], K, V, kept)
        assert np.allclose(out[0, h], ref, rtol=1e-12, atol=1e-13), h


def test_cold_changes_nothing_without_evictions(oracle_mod):
    """P >= T: no token is ever displaced, so the two policies agree bit for bit."""
    d, G, R, P, T = 64, 8, 2, 64, 60
    K = _falling_keys(4, T, d)
    V = np.random.default_rng(2).standard_normal((T, d)).astype(np.float16)
    a = oracle_mod.OracleCache(1, 1, 1, d, G, R, P)
    b = oracle_mod.OracleCache(1, 1, 1, d, G, R, P, cold=32)
    a.prefill(K[None, None], V[None, None])
    b.prefill(K[None, None], V[None, None])
    ea, eb = a.export_unit(0), b.export_unit(0)
    for k in ("bcount", "bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "pidx", "pk", "pv"):
        assert np.array_equal(ea[k], eb[k]), k
    assert eb["ncold"] == 0
    q = torch.randn(1, 1, d, generator=torch.Generator().manual_seed(0)).half()
    assert np.array_equal(a.decode(q), b.decode(q))


def test_cold_golden_hand_worked(oracle_mod):
    """tests/golden/cold_pool_tiny.json: membership worked out by hand."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "cold_pool_tiny.json")))
    sh = g["shape"]
    d = sh["d"]
    K = np.stack([np.full(d, a, np.float16) for a in g["inputs"]["key_level"]])
    V = np.zeros_like(K)
    orc = oracle_mod.OracleCache(1, 1, 1, d, sh["G"], sh["R"], sh["P"], cold=sh["C"])
    for t in range(len(K)):
        orc.append(K[t][None, None], V[t][None, None])
    e = orc.export_unit(0)
    ex = g["expect"]
    blocks = [e["bidx"][j][: e["bcount"][j]].tolist() for j in range(e["nf"])]
    assert blocks == ex["blocks"]
    assert [x for x in e["pidx"].tolist() if x >= 0] == ex["pool"]
    assert e["cidx"][: e["ncold"]].tolist() == ex["cold"]
    assert e["tail"] == len(ex["tail"])
