"""GPU parity for ragged batches: every sequence has its own length, flushes
on its own schedule and is attended over its own tokens. The CUDA path
(ott_create_ragged / ott_prefill_lens / ott_append / ott_decode_attn through
the C ABI) against the CPU oracle's ragged batch on the same seeded inputs:
state bit-exact per sequence, outputs within max |d| <= 2e-3 and mean
|d| <= 2e-4 of the oracle's double result, at every step.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from tests.parity_util import STATE_KEYS, compare_out

pytestmark = pytest.mark.gpu


def _gen(seed, B, Hkv, T, d):
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    ch = torch.randint(0, d, (4,), generator=g)
    K[..., ch] *= 15
    low = torch.rand(B, Hkv, T, generator=g) < 0.05
    K[low] *= 0.03
    V = torch.randn(B, Hkv, T, d, generator=g)
    return K.half(), V.half()


def _compare_seq(c, orc, b, Hkv):
    """Bit-exact state of sequence b's units against the oracle."""
    gpu = c.export_state(b * Hkv, Hkv)
    for h in range(Hkv):
        e = orc.export_unit(b * Hkv + h)
        assert (gpu["T"], gpu["nf"], gpu["tail"], gpu["npool"]) == (e["T"], e["nf"], e["tail"], e["npool"]), (b, h)
        assert np.array_equal(gpu["bcount"], e["bcount"]), (b, h)
        for k in STATE_KEYS:
            if not np.array_equal(gpu[k][h], e[k]):
                bad = np.argwhere(gpu[k][h] != e[k])
                raise AssertionError(f"seq {b} head {h} field {k}: {len(bad)} mismatches, first {bad[:3].tolist()}")


def _run(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, lens, steps, seed, every=1):
    Lmax = max(lens)
    K, V = _gen(seed, B, Hkv, Lmax + steps, d)
    q_all = torch.randn(steps + 1, B, Hq, d, generator=torch.Generator().manual_seed(seed + 1)).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill_lens(K[:, :, :Lmax].contiguous(), V[:, :, :Lmax].contiguous(), lens)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=Lmax + steps + 1, ragged=True) as c:
        c.prefill_lens(K[:, :, :Lmax].contiguous().to(dev), V[:, :, :Lmax].contiguous().to(dev), lens)
        T = list(lens)
        for s in range(steps + 1):
            if s % every == 0 or s == steps:
                for b in range(B):
                    assert c.seq_counts(b)[0] == T[b]
                    _compare_seq(c, orc, b, Hkv)
            out = c.decode_attn(q_all[s].to(dev))
            compare_out(out, orc.decode(q_all[s]), f"step {s} lens {T}")
            if s < steps:
                # token Lmax + s of the staged stream goes to every sequence
                k = K[:, :, Lmax + s].contiguous()
                v = V[:, :, Lmax + s].contiguous()
                c.append(k.to(dev), v.to(dev))
                orc.append(k, v)
                T = [t + 1 for t in T]
        c.check_device()


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,lens,steps", [
    (4, 4, 4, 128, 16, 3, 5, [1, 18, 40, 97], 40),        # before, at and past the first flush; staggered flushes
    (3, 8, 2, 64, 32, 0, 7, [150, 5, 66], 50),            # GQA 4, d=64, R=0
    (5, 2, 1, 128, 20, 4, 0, [19, 20, 23, 24, 60], 30),   # G not a multiple of 16, P=0, lengths around G+R
    (2, 4, 1, 128, 48, 4, 60, [200, 7], 30),              # P > G (empty first blocks), GQA 4
    (6, 6, 6, 128, 128, 32, 32, [300, 161, 160, 159, 33, 1], 40),   # the pages' G, R, P
    (3, 15, 3, 128, 32, 0, 7, [150, 5, 66], 50),          # GQA 5: slices of 4 and 1 per kv head
])
def test_ragged_every_step(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, lens, steps):
    _run(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, lens, steps, seed=sum(lens) + G)


def test_ragged_many_sequences(oracle_mod, ott):
    """Enough short sequences that a decode warp's range crosses several of
    them, with lengths spread over a few groups."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 90, size=40)]
    _run(oracle_mod, ott, 40, 2, 2, 64, 16, 4, 6, lens, 24, seed=77, every=8)


def test_ragged_cache_with_equal_lengths_and_uniform_prefill(oracle_mod, ott):
    """A ragged-capable cache prefilled with ott_prefill behaves as the plain
    one; with ott_prefill_lens and equal lengths it matches the oracle too."""
    B, Hq, Hkv, d, G, R, P, L = 3, 6, 3, 128, 16, 2, 4, 70
    K, V = _gen(3, B, Hkv, L + 8, d)
    dev = torch.device("cuda")
    for mode in ("uniform", "lens"):
        orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
        with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L + 8, ragged=True) as c:
            if mode == "uniform":
                c.prefill(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev))
                orc.prefill(K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
            else:
                c.prefill_lens(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev), [L] * B)
                orc.prefill_lens(K[:, :, :L].contiguous(), V[:, :, :L].contiguous(), [L] * B)
            for s in range(8):
                q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(s)).half()
                compare_out(c.decode_attn(q.to(dev)), orc.decode(q), f"{mode} step {s}")
                k, v = K[:, :, L + s].contiguous(), V[:, :, L + s].contiguous()
                c.append(k.to(dev), v.to(dev))
                orc.append(k, v)
            for b in range(B):
                _compare_seq(c, orc, b, Hkv)


def test_ragged_static_decode_matches(oracle_mod, ott):
    """The allocation-free entry point on a ragged batch gives the same output."""
    B, Hq, Hkv, d, G, R, P = 4, 4, 2, 128, 16, 3, 5
    lens = [3, 40, 17, 61]
    K, V = _gen(9, B, Hkv, max(lens), d)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=100, ragged=True) as c:
        c.prefill_lens(K.contiguous().to(dev), V.contiguous().to(dev), lens)
        q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(1)).half().to(dev)
        ref = c.decode_attn(q)
        out = torch.full_like(ref, float("nan"))
        rc = ott.load().ott_decode_attn_static(C.c_void_p(c.handle), C.c_void_p(q.data_ptr()),
                                               C.c_void_p(out.data_ptr()),
                                               C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == ott.OTT_OK
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the same bits
        assert torch.equal(out, ref)


def test_ragged_argument_errors(ott):
    dev = torch.device("cuda")
    K = torch.zeros(2, 1, 8, 64, device=dev, dtype=torch.float16)
    with ott.OTTCache(2, 1, 1, 64, 4, 1, 1, max_tokens=16) as plain:
        with pytest.raises(ott.OTTError) as ei:
            plain.prefill_lens(K, K.clone(), [3, 8])         # not created ragged
        assert ei.value.code == ott.OTT_ERR_STATE
    with ott.OTTCache(2, 1, 1, 64, 4, 1, 1, max_tokens=16, ragged=True) as c:
        for bad in ([0, 8], [3, 9]):                          # lengths must lie in [1, Lmax]
            with pytest.raises(ott.OTTError) as ei:
                c.prefill_lens(K, K.clone(), bad)
            assert ei.value.code == ott.OTT_ERR_INVALID
        c.prefill_lens(K, K.clone(), [3, 8])
        with pytest.raises(ott.OTTError) as ei:
            c.prefill_lens(K, K.clone(), [3, 8])             # only on an empty cache
        assert ei.value.code == ott.OTT_ERR_STATE
        with pytest.raises(ott.OTTError) as ei:
            c.export_state(0, 2)                              # units of two sequences at once
        assert ei.value.code == ott.OTT_ERR_INVALID
    out = C.c_void_p(123)
    assert ott.load().ott_create_ragged(300, 1, 1, 64, 4, 1, 1, 16, C.byref(out)) == ott.OTT_ERR_INVALID
    assert out.value is None
