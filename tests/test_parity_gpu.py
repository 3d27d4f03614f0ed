"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. State bit-exact after every flush checked; outputs within
max |d| <= 2e-3, mean |d| <= 2e-4 of the oracle's double result.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_ott_gb300 import synth
from tests.parity_util import compare_out, compare_state

pytestmark = pytest.mark.gpu


def _gen(seed, B, Hkv, T, d, dup=False, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    ch = torch.randint(0, d, (4,), generator=g)
    K[..., ch] *= 15
    low = torch.rand(B, Hkv, T, generator=g) < 0.05
    K[low] *= 0.03
    if dup and T > 3:
        K[:, :, 1::3] = K[:, :, 0:1]
    V = torch.randn(B, Hkv, T, d, generator=g)
    return (K * scale).half(), V.half()


def _run_small(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, L, steps, seed, dup=False, scale=1.0,
               check_every_step=True):
    K, V = _gen(seed, B, Hkv, L + steps, d, dup, scale)
    q_all = (torch.randn(steps + 1, B, Hq, d, generator=torch.Generator().manual_seed(seed + 1)) * scale).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L + steps + 1) as c:
        Kd, Vd = K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev)
        c.prefill(Kd, Vd)
        orc.prefill(K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
        nf_seen = -1
        for s in range(steps + 1):
            T, nf, _, _ = c.counts()
            if T > 0 and (check_every_step or nf != nf_seen or s == steps):
                compare_state(c.export_state(), orc)
                nf_seen = nf
                out = c.decode_attn(q_all[s].to(dev))
                compare_out(out, orc.decode(q_all[s]), f"step {s} T={T}")
            if s < steps:
                k = K[:, :, L + s].contiguous()
                v = V[:, :, L + s].contiguous()
                c.append(k.to(dev), v.to(dev))
                orc.append(k, v)
        c.check_device()


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,L,steps", [
    (1, 1, 1, 128, 128, 32, 32, 300, 40),     # default shape, flushes during the steps
    (2, 4, 2, 128, 16, 3, 5, 100, 40),        # GQA 2, small groups
    (2, 8, 2, 64, 32, 0, 7, 150, 70),         # GQA 4, d=64, R=0
    (3, 3, 3, 64, 20, 5, 0, 90, 30),          # G not a multiple of 16, P=0
    (1, 4, 1, 128, 48, 4, 60, 200, 30),       # P > G (empty first blocks), GQA 4
    (2, 2, 2, 128, 4, 1, 2, 60, 20),          # tiny G
    (2, 6, 2, 128, 16, 3, 5, 100, 30),        # GQA 3: one slice of four, padded
    (1, 16, 2, 64, 32, 0, 7, 150, 40),        # GQA 8: two slices, d=64, R=0
    (2, 5, 1, 128, 20, 5, 40, 120, 30),       # GQA 5: slices of 4 and 1, P > G
    (1, 32, 1, 128, 16, 4, 8, 90, 20),        # multi-query (GQA 32): eight slices
])
def test_small_shapes_every_step(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, L, steps):
    _run_small(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, L, steps, seed=L * 7 + G)


def test_norm_ties_pick_lower_index(oracle_mod, ott):
    _run_small(oracle_mod, ott, 2, 2, 2, 128, 16, 2, 6, 120, 20, seed=5, dup=True)


@pytest.mark.parametrize("L", [1, 10, 159, 160, 161])
def test_around_first_flush(oracle_mod, ott, L):
    """T below, at and above G+R, including a single token."""
    _run_small(oracle_mod, ott, 1, 2, 1, 128, 128, 32, 32, L, 3, seed=L)


def test_pool_holds_everything(oracle_mod, ott):
    """P >= T: nothing is quantized; decode is plain attention."""
    _run_small(oracle_mod, ott, 2, 2, 2, 128, 16, 4, 300, 200, 10, seed=3)


def test_pool_too_large_for_flush_staging_is_rejected(ott):
    """(P + G) candidate rows must fit one CTA's shared memory; beyond that
    ott_create refuses the shape instead of failing later."""
    with pytest.raises(ott.OTTError) as ei:
        ott.OTTCache(1, 1, 1, 128, 16, 4, 500, max_tokens=100)
    assert ei.value.code == ott.OTT_ERR_INVALID


def test_large_magnitudes(oracle_mod, ott):
    """Keys and queries scaled by 50: q*s overflows fp16 unless the per-block
    exponent rescales the score operand."""
    _run_small(oracle_mod, ott, 1, 4, 2, 128, 32, 8, 8, 100, 10, seed=11, scale=50.0,
               check_every_step=False)


def test_tiny_workload_every_step(oracle_mod, ott):
    """The tiny single-head workload, all 64 decode steps, state at every step."""
    w = synth.WORKLOADS["tiny"]
    K, V = synth.prefill_kv(w)
    orc = oracle_mod.OracleCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P)
    orc.prefill(K, V)
    with ott.OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + w.steps) as c:
        c.prefill(K.cuda(), V.cuda())
        for s in range(w.steps):
            k, v, q = synth.step_kvq(w, s)
            c.append(k.cuda(), v.cuda())
            orc.append(k, v)
            compare_state(c.export_state(), orc)
            compare_out(c.decode_attn(q.cuda()), orc.decode(q), f"tiny step {s}")
        c.check_device()
