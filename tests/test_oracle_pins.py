"""Pins for the CPU oracle: closed forms, hand-derived goldens, invariants,
library routines and brute force. No GPU; nothing here touches the CUDA path.

Sources: "Accurate KV Cache Quantization with Outlier Tokens Tracing"
(zijie-tian.site sec. 3.1-3.3 and the flowchart; sciencestack.ai TL;DR,
Abstract, Fig. 1(c), Fig. 2).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from tests import bruteforce as bf

hyp = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _h(x):
    return int(x, 16) if isinstance(x, str) else int(x)


# ----------------------------------------------------------------- fp16 I/O

def test_h2f_exhaustive_matches_numpy(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.h2f(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f32_sample():
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x0fff, 0x1000, 0x1001, 0x1fff, 0x2000, 0x2001,
                     0x2fff, 0x3000, 0x3001, 0x4000, 0x7fff, 0x8000, 0x8001, 0xefff,
                     0xf000, 0xffff], np.uint32)
    rng = np.random.default_rng(5)
    rand = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([(hi[:, None] | lows[None, :]).ravel(), rand]).view(np.float32)


def test_f2h_round_to_nearest_even_matches_libraries(oracle_mod):
    """Every fp32 exponent, the tie and near-tie fraction patterns, and 1M random
    patterns: bit-identical to numpy's and torch's fp32->fp16 conversion."""
    x = _f32_sample()
    got = oracle_mod.f2h(x)
    ref_np = x.astype(np.float16).view(np.uint16)
    ref_t = torch.from_numpy(x.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.all((got[nan] & 0x7c00) == 0x7c00) and np.all((got[nan] & 0x3ff) != 0)
    assert np.array_equal(got[~nan], ref_np[~nan])
    assert np.array_equal(got[~nan], ref_t[~nan])


# ----------------------------------------------------------------- norm

def test_norm_integer_closed_form(oracle_mod):
    rng = np.random.default_rng(1)
    for d in (32, 64, 128):
        k = rng.integers(-40, 41, size=d)
        got = oracle_mod.norm(k.astype(np.float16))
        assert got == float(np.sum(k.astype(np.int64) ** 2))


def test_norm_is_sequential_fp32(oracle_mod):
    """Bit-equal to numpy's strictly sequential fp32 accumulate; the sample is
    chosen so that pairwise summation gives different bits for some keys."""
    rng = np.random.default_rng(2)
    differs = 0
    for _ in range(400):
        k = (rng.standard_normal(128) * np.exp(rng.uniform(-6, 6, 128))).astype(np.float16)
        got = np.float32(oracle_mod.norm(k))
        seq = bf.norms_fp32(k[None])[0]
        assert got.view(np.uint32) == seq.view(np.uint32)
        pair = np.sum(k.astype(np.float32) ** 2, dtype=np.float32)
        differs += int(pair.view(np.uint32) != seq.view(np.uint32))
    assert differs > 0


# ----------------------------------------------------------------- quantization

def test_quant_golden_cases(oracle_mod):
    cases = json.load(open(os.path.join(GOLD, "quant_cases.json")))["cases"]
    for c in cases:
        if "x_bits" in c:
            x = np.array([_h(b) for b in c["x_bits"]], np.uint16).view(np.float16)
        else:
            x = np.array(c["x"], np.float16)
        s, z, codes = oracle_mod.quant_group(x)
        assert s == _h(c["s_bits"]), c["name"]
        assert z == _h(c["z_bits"]), c["name"]
        assert codes.tolist() == c["codes"], c["name"]


@settings(max_examples=300, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(st.integers(1, 64), st.floats(-8, 8), st.floats(-12, 4), st.integers(0, 2**31 - 1))
def test_quant_invariants(oracle_mod, n, center_log, spread_log, seed):
    rng = np.random.default_rng(seed)
    x = (np.sign(center_log) * 2.0 ** abs(center_log) +
         rng.standard_normal(n) * 2.0 ** spread_log).astype(np.float16)
    x = x[np.isfinite(x)]
    if x.size == 0:
        return
    s16, z16, codes = oracle_mod.quant_group(x)
    s = float(np.uint16(s16).view(np.float16))
    z = float(np.uint16(z16).view(np.float16))
    xf = x.astype(np.float64)
    assert codes.max() <= 3
    assert z == xf.min()
    if s == 0:
        assert np.all(codes == 0) and xf.max() - xf.min() < 2.0 ** -24 * 1.5
        return
    assert codes[np.argmin(xf)] == 0
    assert codes[np.argmax(xf)] == 3
    err = np.abs(xf - (codes * s + z))
    if (xf.max() - xf.min()) / 3 >= 2.0 ** -14:  # s is a normal fp16 number
        assert np.all(err <= s / 2 * (1 + 2.0 ** -9) + np.abs(xf) * 2.0 ** -22)


# ----------------------------------------------------------------- golden cache

def test_flush_tiny_golden(oracle_mod):
    gd = json.load(open(os.path.join(GOLD, "flush_tiny.json")))
    sh, ex = gd["shape"], gd["expect"]
    d = sh["d"]
    a = gd["inputs"]["a"]
    keys = np.array([[v] * d for v in a], np.float16)
    vals = np.array([[t + 0.5 * (c % 4) for c in range(d)] for t in range(len(a))], np.float16)
    o = oracle_mod.OracleCache(sh["B"], sh["Hq"], sh["Hkv"], d, sh["G"], sh["R"], sh["P"])
    for t in range(len(a)):
        o.append(keys[t].reshape(1, 1, d), vals[t].reshape(1, 1, d))
    e = o.export_unit(0)
    assert (e["T"], e["nf"], e["tail"], e["npool"]) == (ex["T"], ex["nf"], ex["tail"], ex["npool"])
    assert e["bcount"].tolist() == ex["bcount"]
    assert e["bidx"].tolist() == ex["bidx"]
    assert [set(r.tolist()) for r in e["kcode"][0]] == [{_h(x)} for x in ex["kcode_rows"]]
    assert [set(r.tolist()) for r in e["vcode"][0]] == [{_h(x)} for x in ex["vcode_rows"]]
    assert set(e["ks"][0].tolist()) == {_h(ex["ks"])} and set(e["kz"][0].tolist()) == {_h(ex["kz"])}
    assert e["vs"][0, :, 0].tolist() == [_h(x) for x in ex["vs"]]
    assert e["vz"][0, :, 0].tolist() == [_h(x) for x in ex["vz"]]
    assert e["pidx"].tolist() == ex["pidx"] and e["pnorm"][0] == _h(ex["pnorm"])
    assert e["tidx"].tolist() == ex["tidx"]
    # decode closed form: out[c] = sum_t softmax(sqrt(2)*khat)_t * t + 0.5*(c%4)
    q = np.full((1, 1, d), 0.25, np.float16)
    out = o.decode(q)[0, 0]
    kh = ex["decode_khat"]
    base = ex["decode_base"]
    w = {t: math.exp(math.sqrt(2.0) * kh[t]) for t in kh}
    mean = sum(w[t] * base[t] for t in w) / sum(w.values())
    ref = np.array([mean + 0.5 * (c % 4) for c in range(d)])
    assert np.max(np.abs(out - ref)) < 1e-12


# ----------------------------------------------------------------- brute force

def _inputs(rng, B, Hkv, T, d, dup=False):
    K = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
    K[..., rng.integers(0, d)] *= 15
    low = rng.random((B, Hkv, T)) < 0.1
    K[low] *= 0.03
    if dup and T > 3:  # forced norm ties: repeated key vectors
        K[:, :, 1::3] = K[:, :, 0:1]
    V = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
    return K.astype(np.float16), V.astype(np.float16)


def check_unit_against_bruteforce(e, K16, V16, G, R, P):
    """Compare one unit's canonical export with the brute-force statement."""
    T = len(K16)
    d = K16.shape[1]
    blocks, pool, tail, norms = bf.state(K16, G, R, P)
    assert e["T"] == T and e["nf"] == len(blocks)
    assert e["tail"] == len(tail) and e["npool"] == len(pool)
    # accounting: every token exactly once across blocks, tail and pool
    seen = [t for b in blocks for t in b] + tail + pool
    assert sorted(seen) == list(range(T))
    assert sum(e["bcount"].tolist()) + e["tail"] + e["npool"] == T
    for j, blk in enumerate(blocks):
        c = len(blk)
        assert e["bcount"][j] == c
        assert e["bidx"][j, :c].tolist() == blk and np.all(e["bidx"][j, c:] == -1)
        if c == 0:
            continue
        kb = K16[blk].astype(np.float32)
        vb = V16[blk].astype(np.float32)
        s, z, code = bf.np_quant(kb, axis=0)                          # keys per channel
        assert np.array_equal(e["ks"][j], s[0].view(np.uint16))
        assert np.array_equal(e["kz"][j].view(np.float16).astype(np.float32), z[0])
        assert np.array_equal(bf.unpack_rows(e["kcode"][j, :c], d), code)
        vs, vz, vcode = bf.np_quant(vb.reshape(c, d // 32, 32), axis=2)  # values per token/32
        assert np.array_equal(e["vs"][j, :c], vs[..., 0].view(np.uint16))
        assert np.array_equal(e["vz"][j, :c].view(np.float16).astype(np.float32), vz[..., 0])
        assert np.array_equal(bf.unpack_rows(e["vcode"][j, :c], d), vcode.reshape(c, d))
        assert np.all(e["kcode"][j, c:] == 0) and np.all(e["vs"][j, c:] == 0)
    assert e["tidx"].tolist() == tail
    assert np.array_equal(e["tk"], K16[tail].view(np.uint16))
    assert np.array_equal(e["tv"], V16[tail].view(np.uint16))
    npool = len(pool)
    assert e["pidx"][:npool].tolist() == pool and np.all(e["pidx"][npool:] == -1)
    assert np.array_equal(e["pnorm"][:npool], norms[pool].view(np.uint32))
    assert np.array_equal(e["pk"][:npool], K16[pool].view(np.uint16))
    assert np.array_equal(e["pv"][:npool], V16[pool].view(np.uint16))


@settings(max_examples=60, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(d=st.sampled_from([32, 64]), G=st.sampled_from([4, 8]), R=st.sampled_from([0, 1, 3]),
       P=st.sampled_from([0, 1, 2, 5]), T=st.integers(1, 64), dup=st.booleans(),
       seed=st.integers(0, 2**31 - 1))
def test_state_matches_bruteforce_every_append(oracle_mod, d, G, R, P, T, dup, seed):
    rng = np.random.default_rng(seed)
    K, V = _inputs(rng, 1, 2, T, d, dup)
    o = oracle_mod.OracleCache(1, 2, 2, d, G, R, P)
    for t in range(T):
        o.append(K[:, :, t], V[:, :, t])
        for u in range(2):
            check_unit_against_bruteforce(o.export_unit(u), K[0, u, : t + 1], V[0, u, : t + 1], G, R, P)


def test_prefill_equals_appends(oracle_mod):
    rng = np.random.default_rng(9)
    B, H, T, d, G, R, P = 2, 2, 300, 64, 16, 5, 7
    K, V = _inputs(rng, B, H, T, d, dup=True)
    a = oracle_mod.OracleCache(B, H, H, d, G, R, P)
    b = oracle_mod.OracleCache(B, H, H, d, G, R, P)
    a.prefill(K, V)
    for t in range(T):
        b.append(K[:, :, t], V[:, :, t])
    for u in range(B * H):
        ea, eb = a.export_unit(u), b.export_unit(u)
        for k in ea:
            assert np.array_equal(np.asarray(ea[k]), np.asarray(eb[k])), k
        check_unit_against_bruteforce(ea, K[u // H, u % H], V[u // H, u % H], G, R, P)


# ----------------------------------------------------------------- decode

def _torch_attention(q16, K16, V16, Hq, Hkv):
    """float64 softmax attention with the library routine; GQA by repeat."""
    q = torch.from_numpy(q16.astype(np.float64))              # [Hq][d]
    K = torch.from_numpy(K16.astype(np.float64))              # [Hkv][n][d]
    V = torch.from_numpy(V16.astype(np.float64))
    g = Hq // Hkv
    K = K.repeat_interleave(g, 0)
    V = V.repeat_interleave(g, 0)
    s = torch.einsum("hd,hnd->hn", q, K) / math.sqrt(q.shape[-1])
    return torch.einsum("hn,hnd->hd", torch.softmax(s, -1), V).numpy()


@pytest.mark.parametrize("T,G,R,P", [(40, 64, 8, 4), (40, 8, 4, 64), (100, 16, 4, 200)])
def test_decode_exact_attention_when_nothing_is_quantized(oracle_mod, T, G, R, P):
    """P >= T or G+R > T: no token is quantized, so the result is plain softmax
    attention over the fp16 keys and values."""
    rng = np.random.default_rng(T + G)
    B, Hq, Hkv, d = 2, 4, 2, 64
    K, V = _inputs(rng, B, Hkv, T, d)
    q = rng.standard_normal((B, Hq, d)).astype(np.float16)
    o = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    o.prefill(K, V)
    for u in range(B * Hkv):
        assert sum(o.export_unit(u)["bcount"].tolist()) == 0
    out = o.decode(q)
    for b in range(B):
        ref = _torch_attention(q[b], K[b], V[b], Hq, Hkv)
        assert np.max(np.abs(out[b] - ref)) < 1e-12


def dequantized_tokens(e, d):
    """All tokens of one unit from its export, dequantized, in any order."""
    ks, vs = [], []
    for j in range(e["nf"]):
        c = int(e["bcount"][j])
        if c == 0:
            continue
        code_k = bf.unpack_rows(e["kcode"][j, :c], d).astype(np.float64)
        s = e["ks"][j].view(np.float16).astype(np.float64)
        z = e["kz"][j].view(np.float16).astype(np.float64)
        ks.append(code_k * s + z)
        code_v = bf.unpack_rows(e["vcode"][j, :c], d).astype(np.float64).reshape(c, d // 32, 32)
        sv = e["vs"][j, :c].view(np.float16).astype(np.float64)[..., None]
        zv = e["vz"][j, :c].view(np.float16).astype(np.float64)[..., None]
        vs.append((code_v * sv + zv).reshape(c, d))
    n = e["npool"]
    ks += [e["tk"].view(np.float16).astype(np.float64), e["pk"][:n].view(np.float16).astype(np.float64)]
    vs += [e["tv"].view(np.float16).astype(np.float64), e["pv"][:n].view(np.float16).astype(np.float64)]
    return np.concatenate(ks), np.concatenate(vs)


@settings(max_examples=40, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(d=st.sampled_from([32, 64]), G=st.sampled_from([4, 8, 16]), R=st.sampled_from([0, 1, 3]),
       P=st.sampled_from([0, 1, 5]), T=st.integers(1, 90), gq=st.sampled_from([(1, 1), (4, 2), (4, 1)]),
       seed=st.integers(0, 2**31 - 1))
def test_decode_is_softmax_attention_over_three_stores(oracle_mod, d, G, R, P, T, gq, seed):
    """The three-segment decode equals one softmax over the concatenation of
    dequantized-block, residual and pool tokens (sciencestack.ai Fig. 2), with
    query head h reading kv head h // (Hq/Hkv)."""
    Hq, Hkv = gq
    rng = np.random.default_rng(seed)
    K, V = _inputs(rng, 1, Hkv, T, d)
    q = rng.standard_normal((1, Hq, d)).astype(np.float16)
    o = oracle_mod.OracleCache(1, Hq, Hkv, d, G, R, P)
    o.prefill(K, V)
    out = o.decode(q)[0]
    g = Hq // Hkv
    for h in range(Hq):
        kh, vh = dequantized_tokens(o.export_unit(h // g), d)
        ref = _torch_attention(q[0, h:h + 1], kh[None], vh[None], 1, 1)[0]
        assert np.max(np.abs(out[h] - ref)) < 1e-11


def test_ragged_batch_is_independent_sequences(oracle_mod):
    """Reading R10: a ragged batch (per-sequence prefill lengths, then appends
    to every sequence) is each sequence's cache side by side. Sequence b's
    state and decode output equal a one-sequence oracle fed only its own
    lens[b] tokens and then the same appends -- through flushes that happen
    at different steps for different sequences."""
    B, Hq, Hkv, d, G, R, P = 4, 4, 2, 32, 8, 3, 5
    lens = [1, 9, 23, 40]       # before the first flush, around it, several flushes
    Lmax = max(lens)
    rng = np.random.default_rng(11)
    K = rng.standard_normal((B, Hkv, Lmax, d)).astype(np.float16)
    V = rng.standard_normal((B, Hkv, Lmax, d)).astype(np.float16)
    rag = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    rag.prefill_lens(K, V, lens)
    solo = []
    for b in range(B):
        o = oracle_mod.OracleCache(1, Hq, Hkv, d, G, R, P)
        o.prefill(np.ascontiguousarray(K[b:b + 1, :, :lens[b]]), np.ascontiguousarray(V[b:b + 1, :, :lens[b]]))
        solo.append(o)
    for step in range(25):
        k = rng.standard_normal((B, Hkv, d)).astype(np.float16)
        v = rng.standard_normal((B, Hkv, d)).astype(np.float16)
        q = rng.standard_normal((B, Hq, d)).astype(np.float16)
        rag.append(k, v)
        out = rag.decode(q)
        for b in range(B):
            solo[b].append(np.ascontiguousarray(k[b:b + 1]), np.ascontiguousarray(v[b:b + 1]))
            np.testing.assert_array_equal(out[b], solo[b].decode(np.ascontiguousarray(q[b:b + 1]))[0])
            for h in range(Hkv):
                assert rag.counts(b * Hkv + h) == solo[b].counts(h)
                e_r, e_s = rag.export_unit(b * Hkv + h), solo[b].export_unit(h)
                for key in e_s:
                    np.testing.assert_array_equal(e_r[key], e_s[key], err_msg=f"step {step} seq {b} {key}")
    with pytest.raises(RuntimeError):
        rag.prefill_lens(K, V, lens)                       # only on an empty cache
    bad = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    with pytest.raises(RuntimeError):
        bad.prefill_lens(K, V, [1, 2, 3, Lmax + 1])       # a length beyond the staged tokens


def test_released_and_refilled_sequence_is_a_fresh_one(oracle_mod):
    """A released sequence refilled with a new prompt equals a one-sequence
    cache that only ever saw that prompt (state bit for bit, outputs exactly),
    and the other sequences are untouched by the release."""
    B, Hq, Hkv, d, G, R, P = 3, 4, 2, 64, 8, 2, 3
    g = torch.Generator().manual_seed(9)
    K = torch.randn(B, Hkv, 90, d, generator=g).half()
    V = torch.randn(B, Hkv, 90, d, generator=g).half()
    K2 = torch.randn(Hkv, 37, d, generator=g).half()
    V2 = torch.randn(Hkv, 37, d, generator=g).half()
    steps = [(torch.randn(B, Hkv, d, generator=g).half(), torch.randn(B, Hkv, d, generator=g).half())
             for _ in range(20)]
    lens = [90, 60, 75]
    big = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    big.prefill_lens(K, V, lens)
    for k, v in steps[:5]:
        big.append(k, v)
    before = [big.export_unit(u) for u in range(B * Hkv)]
    big.release_seq(1)
    with pytest.raises(RuntimeError):
        big.append(*steps[5])                  # an empty sequence blocks appends
    big.prefill_seq(1, K2, V2)
    fresh = oracle_mod.OracleCache(1, Hq, Hkv, d, G, R, P)
    fresh.prefill(K2[None], V2[None])
    for u in (0, 1, 4, 5):                     # sequences 0 and 2 untouched
        e = big.export_unit(u)
        for key in ("bidx", "kcode", "ks", "vcode", "tidx", "tk", "pidx", "pk"):
            assert np.array_equal(e[key], before[u][key]), (u, key)
    for k, v in steps[5:]:
        big.append(k, v)
        fresh.append(k[1:2], v[1:2])
    for x in range(Hkv):
        a, f = big.export_unit(1 * Hkv + x), fresh.export_unit(x)
        assert (a["T"], a["nf"], a["tail"], a["npool"]) == (f["T"], f["nf"], f["tail"], f["npool"]) == (52, 6, 4, 3)
        for key in ("bcount", "bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "tidx", "tk", "tv", "pidx", "pnorm",
                    "pk", "pv"):
            assert np.array_equal(a[key], f[key]), (x, key)
    q = torch.randn(B, Hq, d, generator=g).half()
    assert np.array_equal(big.decode(q)[1], fresh.decode(q[1:2])[0])
