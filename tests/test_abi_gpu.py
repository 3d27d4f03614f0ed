"""C ABI contract on a GPU: argument/state checks leave the cache unchanged,
capacity is enforced, a failed allocation is reported (host-side fault
injection through OTT_FAULT=alloc), and the status word stays clear after
normal work.
"""
import ctypes as C
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_state_errors_leave_the_cache_unchanged(ott):
    dev = torch.device("cuda")
    with ott.OTTCache(2, 4, 2, 128, 16, 4, 8, max_tokens=64) as c:
        q = torch.randn(2, 4, 128, device=dev).half()
        with pytest.raises(ott.OTTError) as ei:
            c.decode_attn(q)                              # empty cache
        assert ei.value.code == ott.OTT_ERR_STATE
        K = torch.randn(2, 2, 40, 128, device=dev).half()
        c.prefill(K, K.clone())
        before = c.export_state()
        with pytest.raises(ott.OTTError) as ei:
            c.prefill(K, K)                                # not empty any more
        assert ei.value.code == ott.OTT_ERR_STATE
        L = ott.load()
        k = torch.randn(2, 2, 128, device=dev).half()
        # misaligned pointer (2 bytes past a 16-byte boundary)
        rc = L.ott_append(c.handle, C.c_void_p(k.data_ptr() + 2), C.c_void_p(k.data_ptr()),
                          C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == ott.OTT_ERR_INVALID
        rc = L.ott_decode_attn(c.handle, C.c_void_p(q.data_ptr()), C.c_void_p(q.data_ptr()), None)
        assert rc == ott.OTT_ERR_INVALID                   # out aliases q
        rc = L.ott_export_state(c.handle, 3, 2, None)
        assert rc == ott.OTT_ERR_INVALID
        after = c.export_state()
        for key in before:
            assert np.array_equal(np.asarray(before[key]), np.asarray(after[key])), key
        c.check_device()


def test_capacity_is_enforced(ott):
    dev = torch.device("cuda")
    with ott.OTTCache(1, 1, 1, 64, 16, 2, 4, max_tokens=20) as c:
        K = torch.randn(1, 1, 19, 64, device=dev).half()
        with pytest.raises(ott.OTTError) as ei:
            c.prefill(torch.randn(1, 1, 21, 64, device=dev).half(), torch.randn(1, 1, 21, 64, device=dev).half())
        assert ei.value.code == ott.OTT_ERR_CAPACITY
        c.prefill(K, K.clone())
        k = torch.randn(1, 1, 64, device=dev).half()
        c.append(k, k.clone())                             # T = 20
        with pytest.raises(ott.OTTError) as ei:
            c.append(k, k.clone())
        assert ei.value.code == ott.OTT_ERR_CAPACITY
        assert c.counts()[0] == 20


def test_allocation_failure_is_reported(ott):
    os.environ["OTT_FAULT"] = "alloc"
    try:
        with pytest.raises(ott.OTTError) as ei:
            ott.OTTCache(1, 1, 1, 128, 128, 32, 32, max_tokens=1000)
        assert ei.value.code == ott.OTT_ERR_OOM
    finally:
        del os.environ["OTT_FAULT"]
    with ott.OTTCache(1, 1, 1, 128, 128, 32, 32, max_tokens=1000) as c:
        assert c.device_bytes() > 0


def test_handles_are_independent_and_streams_are_honoured(ott, oracle_mod):
    """Two caches of different shapes on two streams; results match the oracle."""
    dev = torch.device("cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.Generator().manual_seed(3)
    shapes = [(2, 2, 2, 128, 32, 4, 5, 120), (1, 4, 1, 64, 16, 8, 3, 90)]
    outs = []
    for (B, Hq, Hkv, d, G, R, P, L), s in zip(shapes, (s1, s2)):
        K = torch.randn(B, Hkv, L, d, generator=g).half()
        V = torch.randn(B, Hkv, L, d, generator=g).half()
        q = torch.randn(B, Hq, d, generator=g).half()
        orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
        orc.prefill(K, V)
        c = ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L)
        with torch.cuda.stream(s):
            Kd, Vd, qd = K.to(dev, non_blocking=False), V.to(dev), q.to(dev)
            c.prefill(Kd, Vd, stream=s)
            out = c.decode_attn(qd, stream=s)
        outs.append((c, out, orc.decode(q), s))
    for c, out, ref, s in outs:
        s.synchronize()
        assert float(np.abs(out.float().cpu().numpy() - ref).max()) <= 2e-3
        c.check_device()
        c.close()
