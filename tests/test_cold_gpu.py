"""GPU parity for the cold-pool eviction policy (ott_create_cold): pool
tokens displaced at a flush enter a first-in-first-out fp16 cold pool of C
slots instead of the new block (zijie-tian.site sec. 3.2, the alternative to
writing them back). The CUDA path through the C ABI against the CPU oracle's
same policy on the same seeded inputs: per-unit block sizes, block indices,
codes, scales, residual, pool and cold pool (indices, keys, values, order)
bit-exact; outputs within max |d| <= 2e-3 and mean |d| <= 2e-4 of the
oracle's double result.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from tests.parity_util import compare_out

pytestmark = pytest.mark.gpu

KEYS = ("bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "tk", "tv", "pidx", "pnorm", "pk", "pv")


def _gen(seed, B, Hkv, T, d):
    """Keys whose norms tend to fall with the token index (new groups keep
    displacing pool tokens), the usual outlier channels and low-norm tokens,
    and some exact duplicates for ties."""
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    ch = torch.randint(0, d, (4,), generator=g)
    K[..., ch] *= 15
    K *= torch.linspace(3.0, 0.3, T)[None, None, :, None]
    low = torch.rand(B, Hkv, T, generator=g) < 0.05
    K[low] *= 0.03
    if T > 12:
        K[:, :, 9::11] = K[:, :, 4:5]
    V = torch.randn(B, Hkv, T, d, generator=g)
    return K.half(), V.half()


def _compare(c, orc, where):
    gpu = c.export_state()
    for u in range(c.B * c.Hkv):
        e = orc.export_unit(u)
        assert (gpu["T"], gpu["nf"], gpu["tail"], gpu["npool"]) == (e["T"], e["nf"], e["tail"], e["npool"]), where
        assert np.array_equal(gpu["bcount"][u], e["bcount"]), (where, u, gpu["bcount"][u], e["bcount"])
        assert gpu["ncold"][u] == e["ncold"], (where, u)
        for k in KEYS + ("cidx", "ck", "cv"):
            if not np.array_equal(gpu[k][u], e[k]):
                bad = np.argwhere(gpu[k][u] != e[k])
                raise AssertionError(f"{where} unit {u} field {k}: {len(bad)} mismatches, first {bad[:3].tolist()}")


def _run(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, Cc, L, steps, seed, every=1):
    K, V = _gen(seed, B, Hkv, L + steps, d)
    q_all = torch.randn(steps + 1, B, Hq, d, generator=torch.Generator().manual_seed(seed + 1)).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P, cold=Cc)
    orc.prefill(K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L + steps + 1, cold=Cc) as c:
        c.prefill(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev))
        for s in range(steps + 1):
            if s % every == 0 or s == steps:
                _compare(c, orc, f"step {s}")
            out = c.decode_attn(q_all[s].to(dev))
            compare_out(out, orc.decode(q_all[s]), f"step {s}")
            if s < steps:
                k, v = K[:, :, L + s].contiguous(), V[:, :, L + s].contiguous()
                c.append(k.to(dev), v.to(dev))
                orc.append(k, v)
        c.check_device()
    # once the pool is full, a block short of G tokens means that group tokens
    # entered the pool and displaced as many pool tokens
    jfull = -(-P // G)
    return sum(int(G - n) for u in range(B * Hkv) for n in orc.export_unit(u)["bcount"][jfull:])


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,Cc,L,steps", [
    (1, 1, 1, 128, 16, 4, 5, 3, 300, 40),        # the cold ring wraps many times
    (2, 4, 2, 128, 32, 8, 6, 32, 500, 70),       # GQA 2, the pages' C = 32
    (2, 8, 2, 64, 16, 0, 7, 5, 260, 40),         # GQA 4, d = 64, R = 0
    (3, 3, 3, 128, 20, 5, 9, 0, 200, 30),        # C = 0: displaced tokens are discarded
    (2, 2, 2, 128, 16, 3, 0, 4, 120, 30),        # P = 0: nothing is ever displaced
    (1, 4, 1, 128, 8, 2, 20, 6, 180, 30),        # P > G: several flushes before the pool is full
    (2, 12, 2, 128, 16, 4, 6, 5, 260, 40),       # GQA 6: slices of 4 and 2 (padded)
])
def test_cold_every_step(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, Cc, L, steps):
    ev = _run(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, Cc, L, steps, seed=L + G + Cc)
    if P > 0:
        assert ev > 0, "the inputs must displace pool tokens"


def test_cold_pages_shape(oracle_mod, ott):
    """G=128, R=32, P=32, C=32 over a few thousand tokens, checked at every 16th step."""
    _run(oracle_mod, ott, 2, 4, 4, 128, 128, 32, 32, 32, 2100, 140, seed=5, every=16)


def test_cold_static_decode_matches(ott):
    B, Hq, Hkv, d, G, R, P, Cc = 2, 4, 2, 128, 16, 3, 5, 4
    K, V = _gen(2, B, Hkv, 300, d)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=400, cold=Cc) as c:
        c.prefill(K.contiguous().to(dev), V.contiguous().to(dev))
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


def test_cold_argument_errors(ott):
    L = ott.load()
    h = C.c_void_p(123)
    assert L.ott_create_cold(1, 1, 1, 128, 16, 2, 4, -1, 64, C.byref(h)) == ott.OTT_ERR_INVALID
    assert h.value is None
    assert L.ott_create_cold(1, 1, 1, 128, 16, 2, 4, 4097, 64, C.byref(h)) == ott.OTT_ERR_INVALID
    with ott.OTTCache(1, 1, 1, 128, 16, 2, 4, max_tokens=64) as plain:
        n = np.zeros(1, np.int32)
        assert L.ott_export_cold(C.c_void_p(plain.handle), 0, 1, None, n.ctypes.data, None, None, None) \
            == ott.OTT_ERR_STATE
    K = torch.zeros(1, 1, 40, 128, device="cuda", dtype=torch.float16)
    with ott.OTTCache(1, 1, 1, 128, 16, 2, 4, max_tokens=64, cold=4) as c:
        c.prefill(K, K.clone())
        with pytest.raises(ott.OTTError) as ei:
            c.block_count(0)                      # sizes differ per unit under this policy
        assert ei.value.code == ott.OTT_ERR_STATE
        with pytest.raises(ott.OTTError) as ei:
            c.prefill(K, K.clone())               # only on an empty cache
        assert ei.value.code == ott.OTT_ERR_STATE
