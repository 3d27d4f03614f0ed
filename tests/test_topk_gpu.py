"""GPU parity for Top-K sparse decode (ott_decode_attn_topk; zijie-tian.site
sec. 6, OTT combined with sparse access to the quantized KV): every
(sequence, kv head) attends its K non-empty blocks with the largest fp32
score bound plus all fp16 tokens. The CUDA path through the C ABI against the
CPU oracle on the same seeded inputs: the selected blocks bit-exact (the
bound is an fp32 computation both sides take in the same order), outputs
within max |d| <= 2e-3 and mean |d| <= 2e-4 of the oracle's double result.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from bit_kv_cache_ott_gb300 import synth
from tests.parity_util import compare_out

pytestmark = pytest.mark.gpu


def _gen(seed, B, Hkv, T, d, falling=False):
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    ch = torch.randint(0, d, (4,), generator=g)
    K[..., ch] *= 15
    if falling:
        K *= torch.linspace(3.0, 0.3, T)[None, None, :, None]
    low = torch.rand(B, Hkv, T, generator=g) < 0.05
    K[low] *= 0.03
    V = torch.randn(B, Hkv, T, d, generator=g)
    return K.half(), V.half()


def _check(c, orc, q, Kb, where):
    dev = torch.device("cuda")
    nf = max(c.seq_counts(b)[1] for b in range(c.B)) if c.ragged else c.counts()[1]
    kc = min(Kb, nf)
    sel = torch.full((c.B * c.Hkv, kc), -7, dtype=torch.int32, device=dev)
    out = c.decode_attn_topk(q.to(dev), Kb, sel=sel if kc > 0 else None)
    want, _ = orc.topk_select(q, Kb)
    if kc > 0:
        got = sel.cpu().numpy()
        if not np.array_equal(got, want[:, :kc]):
            bad = np.argwhere(got != want[:, :kc])
            raise AssertionError(f"{where}: selection differs at {bad[:3].tolist()}")
    compare_out(out, orc.decode_topk(q, Kb), where)


def _run(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, L, steps, Ks, seed, cold=None, every=1):
    K, V = _gen(seed, B, Hkv, L + steps, d, falling=cold is not None)
    q_all = torch.randn(steps + 1, B, Hq, d, generator=torch.Generator().manual_seed(seed + 1)).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P, cold=cold)
    orc.prefill(K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L + steps + 1, cold=cold) as c:
        c.prefill(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev))
        for s in range(steps + 1):
            if s % every == 0 or s == steps:
                for Kb in Ks:
                    _check(c, orc, q_all[s], Kb, f"step {s} K={Kb}")
            if s < steps:
                k, v = K[:, :, L + s].contiguous(), V[:, :, L + s].contiguous()
                c.append(k.to(dev), v.to(dev))
                orc.append(k, v)
        c.check_device()


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,L,steps,Ks", [
    (2, 2, 2, 128, 16, 4, 5, 300, 30, (1, 4, 100)),     # K above the block count: every block
    (1, 8, 2, 128, 32, 8, 40, 700, 40, (1, 3, 7)),      # GQA 4, P > G (empty first blocks)
    (2, 4, 2, 64, 16, 0, 7, 260, 30, (2, 5)),           # GQA 2, d = 64, R = 0
    (3, 3, 3, 128, 20, 5, 0, 200, 25, (1, 6)),          # G not a multiple of 16, P = 0
    (1, 1, 1, 128, 8, 2, 3, 40, 30, (1, 2)),            # the first flushes happen during the steps
    (1, 16, 2, 128, 32, 8, 40, 700, 40, (1, 3, 7)),     # GQA 8: bounds over both slices' heads
    (2, 6, 2, 64, 16, 0, 7, 260, 30, (2, 5)),           # GQA 3 (a padded slice), d = 64
])
def test_topk_every_step(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, L, steps, Ks):
    _run(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, L, steps, Ks, seed=L + G)


def test_topk_with_cold_pool(oracle_mod, ott):
    _run(oracle_mod, ott, 2, 4, 2, 128, 16, 4, 6, 400, 30, (1, 5), seed=9, cold=4)


def test_topk_pages_shape(oracle_mod, ott):
    """G=128, R=32, P=32 over ~2K tokens: 16 blocks, K = 4."""
    _run(oracle_mod, ott, 2, 8, 2, 128, 128, 32, 32, 2100, 140, (4,), seed=3, every=20)


def test_topk_all_blocks_matches_full_decode(ott):
    B, Hq, Hkv, d, G, R, P = 2, 4, 2, 128, 16, 3, 5
    K, V = _gen(4, B, Hkv, 300, d)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=400) as c:
        c.prefill(K.contiguous().to(dev), V.contiguous().to(dev))
        q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(1)).half().to(dev)
        full = c.decode_attn(q)
        for Kb in (c.counts()[1], 10_000):
            assert float((c.decode_attn_topk(q, Kb).float() - full.float()).abs().max()) <= 1e-3


def test_topk_argument_errors(ott):
    L = ott.load()
    dev = torch.device("cuda")
    K = torch.zeros(2, 1, 40, 128, device=dev, dtype=torch.float16)
    q = torch.zeros(2, 1, 128, device=dev, dtype=torch.float16)
    out = torch.empty_like(q)
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    with ott.OTTCache(2, 1, 1, 128, 16, 2, 4, max_tokens=64) as c:
        assert L.ott_decode_attn_topk(C.c_void_p(c.handle), C.c_void_p(q.data_ptr()), C.c_void_p(out.data_ptr()),
                                      1, None, st) == ott.OTT_ERR_STATE     # empty cache
        c.prefill(K, K.clone())
        for Kb in (0, -3):
            assert L.ott_decode_attn_topk(C.c_void_p(c.handle), C.c_void_p(q.data_ptr()),
                                          C.c_void_p(out.data_ptr()), Kb, None, st) == ott.OTT_ERR_INVALID
    with ott.OTTCache(2, 1, 1, 128, 16, 2, 4, max_tokens=64, ragged=True) as r:
        r.prefill_lens(K, K.clone(), [20, 40])
        r.release_seq(0)
        with pytest.raises(ott.OTTError) as ei:
            r.decode_attn_topk(q, 2)              # a released sequence must be refilled first
        assert ei.value.code == ott.OTT_ERR_STATE


@pytest.mark.parametrize("name,Kb", [("mistral_gqa_g128", 32), ("llama31_8b_131k", 64)])
def test_topk_fullsize(oracle_mod, ott, name, Kb):
    """Full-size long-context layers: the selection of every unit bit-exact and
    every output within tolerance at a few steps, one of them after a flush."""
    w = synth.WORKLOADS[name]
    steps = 40
    K, V = synth.prefill_kv(w)
    orc = oracle_mod.OracleCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P)
    orc.prefill(K, V)
    with ott.OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + steps) as c:
        c.prefill(K.cuda(), V.cuda())
        del K, V
        for s in range(steps):
            k, v, q = synth.step_kvq(w, s)
            c.append(k.cuda(), v.cuda())
            orc.append(k, v)
            if s in (0, 33, 39):
                _check(c, orc, q, Kb, f"{name} step {s}")
        c.check_device()


@pytest.mark.parametrize("paged", [False, True])
def test_topk_ragged_and_paged(oracle_mod, ott, paged):
    """Sequences of different lengths (and, paged, blocks from one pool):
    each unit selects among its own blocks; selection bit-exact, outputs
    within tolerance, through flushes, a release and a refill."""
    from tests.test_ragged_gpu import _gen as _rgen
    B, Hq, Hkv, d, G, R, P = 4, 8, 2, 128, 16, 3, 5
    lens, steps, Kb = [300, 40, 170, 95], 30, 4
    Lmax = max(lens)
    K, V = _rgen(31, B, Hkv, Lmax + steps, d)
    kk, vv = _rgen(32, 1, Hkv, 120, d)
    q_all = torch.randn(steps, B, Hq, d, generator=torch.Generator().manual_seed(33)).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill_lens(K[:, :, :Lmax].contiguous(), V[:, :, :Lmax].contiguous(), lens)
    dev = torch.device("cuda")
    kw = dict(pool_blocks=2 * (Lmax + steps) // G * B * Hkv) if paged else dict(ragged=True)
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=Lmax + steps + 1, **kw) as c:
        c.prefill_lens(K[:, :, :Lmax].contiguous().to(dev), V[:, :, :Lmax].contiguous().to(dev), lens)
        for s in range(steps):
            if s == 12:
                c.release_seq(1)
                orc.release_seq(1)
                c.prefill_seq(1, kk[0].contiguous().to(dev), vv[0].contiguous().to(dev))
                orc.prefill_seq(1, kk[0].contiguous(), vv[0].contiguous())
            _check(c, orc, q_all[s], Kb, f"step {s}")
            k, v = K[:, :, Lmax + s].contiguous(), V[:, :, Lmax + s].contiguous()
            c.append(k.to(dev), v.to(dev))
            orc.append(k, v)
        c.check_device()
