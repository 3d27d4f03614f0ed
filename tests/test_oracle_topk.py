"""Pins for the oracle's Top-K sparse decode (zijie-tian.site sec. 6:
combining OTT with sparse access to the quantized KV). The reading: a decode
call attends only the K non-empty quantized blocks of each (sequence, kv
head) with the largest score bound (ties to the lower block index), plus
every residual and pool token. The bound of block j for query head h is the
largest q.k that a key dequantized from the block's per-channel scale s and
zero z can reach, sum_c max(q_c z_c, q_c (z_c + 3 s_c)), in fp32; the
block's bound is the largest over the query heads of the kv head.

Nothing here touches the CUDA path. Pins, independent of the oracle's code:
- the bound is an upper bound of every dequantized key's score (float64 from
  the canonical export), and it is reached when the block holds the key at
  the box corner that q points to;
- the selection equals a brute-force sort of the bounds;
- the decode equals float64 softmax attention over exactly the selected
  blocks' dequantized tokens plus the residual and pool tokens;
- K >= the block count gives the full decode; K = 0 (where residual or pool
  tokens exist) gives attention over them alone.
"""
import numpy as np
import pytest
import torch

from tests import bruteforce as bf


def _gen(seed, B, Hkv, T, d):
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    ch = torch.randint(0, d, (4,), generator=g)
    K[..., ch] *= 15
    low = torch.rand(B, Hkv, T, generator=g) < 0.05
    K[low] *= 0.03
    V = torch.randn(B, Hkv, T, d, generator=g)
    return K.half(), V.half()


def _dequant_blocks(e, d):
    """Dequantized keys and values of every block of one unit's export, float64."""
    nf, G = e["bidx"].shape
    kc = bf.unpack_rows(e["kcode"].reshape(nf * G, d // 4), d).reshape(nf, G, d).astype(np.float64)
    vc = bf.unpack_rows(e["vcode"].reshape(nf * G, d // 4), d).reshape(nf, G, d).astype(np.float64)
    ks = e["ks"].view(np.float16).astype(np.float64)
    kz = e["kz"].view(np.float16).astype(np.float64)
    vs = np.repeat(e["vs"].view(np.float16).astype(np.float64), 32, axis=2)
    vz = np.repeat(e["vz"].view(np.float16).astype(np.float64), 32, axis=2)
    return kc * ks[:, None, :] + kz[:, None, :], vc * vs + vz


def _attend(q, keys, vals):
    s = keys @ q / np.sqrt(len(q))
    w = np.exp(s - s.max())
    return (w[:, None] * vals).sum(0) / w.sum()


SHAPES = [  # B, Hq, Hkv, d, G, R, P, T
    (2, 2, 2, 64, 16, 4, 5, 300),
    (1, 8, 2, 128, 32, 8, 40, 700),     # GQA 4, P > G (empty first blocks)
    (2, 3, 1, 64, 20, 0, 0, 260),       # GQA 3, R = 0, P = 0
]


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,T", SHAPES)
def test_bound_is_an_upper_bound(oracle_mod, B, Hq, Hkv, d, G, R, P, T):
    K, V = _gen(T + G, B, Hkv, T, d)
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill(K, V)
    q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(3)).half()
    _, bounds = orc.topk_select(q, 1)
    g = Hq // Hkv
    for u in range(B * Hkv):
        b, hk = divmod(u, Hkv)
        e = orc.export_unit(u)
        kh, _ = _dequant_blocks(e, d)
        for j in range(e["nf"]):
            c = int(e["bcount"][j])
            if c == 0:
                assert bounds[u, j] == -np.inf
                continue
            ks = e["ks"][j].view(np.float16).astype(np.float64)
            kz = e["kz"][j].view(np.float16).astype(np.float64)
            best = -np.inf
            for x in range(g):
                qv = q[b, hk * g + x].double().numpy()
                top = float((kh[j, :c] @ qv).max())
                slack = 1e-5 * float(np.abs(qv) @ np.maximum(np.abs(kz), np.abs(kz + 3 * ks))) + 1e-6
                corner = float(np.maximum(qv * kz, qv * (kz + 3 * ks)).sum())
                assert top <= corner + slack, (u, j, x)
                best = max(best, corner)
            assert abs(float(bounds[u, j]) - best) <= 1e-5 * abs(best) + 1e-3


def test_bound_is_reached_by_the_corner_key(oracle_mod):
    """Two-level keys (every channel takes lo_c or hi_c, both in every block)
    and, in every group, the key at the corner the query points to: the
    bound equals that key's score."""
    d, G, R, P, T = 64, 16, 4, 0, 20 * 16 + 4
    rng = np.random.default_rng(8)
    lo = rng.integers(-8, 9, size=d) * 2.0 ** -3
    hi = lo + 3 * 2.0 ** -3
    pick = rng.random((T, d)) < 0.5
    q = rng.standard_normal(d).astype(np.float16)
    corner = np.where(q.astype(np.float64) > 0, hi, lo)
    Kx = np.where(pick, hi, lo)
    Kx[5::G] = corner
    Kx[0::G] = lo       # both levels appear in every block
    Kx[1::G] = hi
    Kh = Kx.astype(np.float16)
    V = rng.standard_normal((T, d)).astype(np.float16)
    orc = oracle_mod.OracleCache(1, 1, 1, d, G, R, P)
    orc.prefill(Kh[None, None], V[None, None])
    _, bounds = orc.topk_select(q[None, None], 1)
    want = float(q.astype(np.float64) @ corner)
    assert np.allclose(bounds[0], want, rtol=1e-6, atol=1e-4), (bounds[0][:4], want)


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,T", SHAPES)
@pytest.mark.parametrize("Kb", [1, 3, 7])
def test_selection_and_sparse_decode(oracle_mod, B, Hq, Hkv, d, G, R, P, T, Kb):
    K, V = _gen(T + Kb, B, Hkv, T, d)
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill(K, V)
    q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(Kb)).half()
    sel, bounds = orc.topk_select(q, Kb)
    out = orc.decode_topk(q, Kb)
    g = Hq // Hkv
    for u in range(B * Hkv):
        b, hk = divmod(u, Hkv)
        e = orc.export_unit(u)
        # brute force: sort the non-empty blocks by (bound desc, index)
        cand = [j for j in range(e["nf"]) if e["bcount"][j] > 0]
        want = sorted(sorted(cand, key=lambda j: (-float(bounds[u, j]), j))[:Kb])
        got = [int(x) for x in sel[u] if x >= 0]
        assert got == want, (u, got, want)
        # attention over exactly those blocks + residual + pool, from the export
        kh, vh = _dequant_blocks(e, d)
        keys = [kh[j, : e["bcount"][j]] for j in want]
        vals = [vh[j, : e["bcount"][j]] for j in want]
        keys.append(e["tk"].view(np.float16).astype(np.float64))
        vals.append(e["tv"].view(np.float16).astype(np.float64))
        npool = e["npool"]
        keys.append(e["pk"][:npool].view(np.float16).astype(np.float64))
        vals.append(e["pv"][:npool].view(np.float16).astype(np.float64))
        keys, vals = np.concatenate(keys), np.concatenate(vals)
        for x in range(g):
            hq = hk * g + x
            ref = _attend(q[b, hq].double().numpy(), keys, vals)
            assert np.allclose(out[b, hq], ref, rtol=1e-10, atol=1e-12), (u, x)


def test_all_blocks_is_the_full_decode(oracle_mod):
    B, Hq, Hkv, d, G, R, P, T = 2, 4, 2, 64, 16, 4, 5, 300
    K, V = _gen(1, B, Hkv, T, d)
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill(K, V)
    q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(2)).half()
    nf = orc.counts()[1]
    assert np.array_equal(orc.decode_topk(q, nf), orc.decode(q))
    assert np.array_equal(orc.decode_topk(q, nf + 10), orc.decode(q))


def test_topk_with_the_cold_pool(oracle_mod):
    """Under the cold-pool policy the cold tokens are always attended."""
    B, Hq, Hkv, d, G, R, P, T = 1, 2, 1, 64, 16, 4, 6, 400
    g = torch.Generator().manual_seed(4)
    K = (torch.randn(B, Hkv, T, d, generator=g) * torch.linspace(3, 0.3, T)[None, None, :, None]).half()
    V = torch.randn(B, Hkv, T, d, generator=g).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P, cold=5)
    orc.prefill(K, V)
    q = torch.randn(B, Hq, d, generator=g).half()
    e = orc.export_unit(0)
    assert e["ncold"] > 0
    out = orc.decode_topk(q, 0)
    keys = np.concatenate([e["tk"], e["pk"][: e["npool"]], e["ck"][: e["ncold"]]]).view(np.float16).astype(np.float64)
    vals = np.concatenate([e["tv"], e["pv"][: e["npool"]], e["cv"][: e["ncold"]]]).view(np.float16).astype(np.float64)
    for h in range(Hq):
        assert np.allclose(out[0, h], _attend(q[0, h].double().numpy(), keys, vals), rtol=1e-10, atol=1e-12)


def test_topk_golden_hand_worked(oracle_mod):
    """tests/golden/topk_tiny.json: bounds and selections worked out by hand."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "topk_tiny.json")))
    sh = g["shape"]
    d = sh["d"]
    rows = []
    for lo, hi in g["inputs"]["block_levels"]:
        rows += [np.full(d, lo, np.float16), np.full(d, hi, np.float16)]
    K = np.stack(rows)
    V = np.zeros_like(K)
    orc = oracle_mod.OracleCache(1, 1, 1, d, sh["G"], sh["R"], sh["P"])
    for t in range(len(K)):
        orc.append(K[t][None, None], V[t][None, None])
    for name, sign in (("q_plus", 1.0), ("q_minus", -1.0)):
        q = np.full((1, 1, d), sign, np.float16)
        ex = g["expect"][name]
        sel, bounds = orc.topk_select(q, 2)
        assert bounds[0].tolist() == ex["bounds"], name
        assert sel[0].tolist() == ex["top2"], name
        if "top3" in ex:
            sel3, _ = orc.topk_select(q, 3)
            assert sel3[0].tolist() == ex["top3"], name
