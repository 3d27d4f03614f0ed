"""ott_step_host: one step (append + decode) fed from and answered into
pinned host memory by the kernels themselves. Against the same cache driven
through device buffers (copies, ott_append, ott_decode_attn): every step's
output equal (torch.equal) and the final state equal, across flushes, for a
uniform batch (MHA and GQA) and a ragged one; plus the argument checks.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from tests.parity_util import STATE_KEYS

pytestmark = pytest.mark.gpu


def _gen(seed, B, Hkv, Hq, T, d):
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    K[..., 3] *= 15
    V = torch.randn(B, Hkv, T, d, generator=g)
    Q = torch.randn(T, B, Hq, d, generator=g)
    return K.half(), V.half(), Q.half()


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,L,steps,ragged", [
    (2, 2, 2, 128, 16, 4, 5, 100, 40, False),     # MHA, two flushes during the steps
    (2, 8, 2, 128, 16, 4, 8, 130, 40, False),     # GQA 4
    (1, 4, 2, 64, 32, 8, 6, 60, 50, False),       # d = 64, GQA 2, the first flush during the steps
    (3, 4, 4, 128, 16, 4, 5, 90, 30, True),       # ragged batch
    (2, 12, 2, 128, 16, 4, 8, 130, 40, False),    # GQA 6: slices of 4 and 2
])
def test_step_host_equals_device_path(ott, B, Hq, Hkv, d, G, R, P, L, steps, ragged):
    K, V, Q = _gen(B + G, B, Hkv, Hq, L + steps, d)
    dev = torch.device("cuda")
    kw = dict(max_tokens=L + steps + 1, ragged=ragged)
    lens = [L - 7 * b for b in range(B)]
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as a, ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as b:
        for c in (a, b):
            if ragged:
                c.prefill_lens(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev), lens)
            else:
                c.prefill(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev))
        kh = [K[:, :, L + s].contiguous().pin_memory() for s in range(steps)]
        vh = [V[:, :, L + s].contiguous().pin_memory() for s in range(steps)]
        qh = [Q[L + s].contiguous().pin_memory() for s in range(steps)]
        outs = [torch.empty(B, Hq, d, dtype=torch.float16).pin_memory() for _ in range(steps)]
        stream = torch.cuda.current_stream()
        for s in range(steps):
            a.step_host(kh[s], vh[s], qh[s], outs[s], stream=stream)
            b.append(kh[s].to(dev), vh[s].to(dev))
            ref = b.decode_attn(qh[s].to(dev))
            torch.cuda.synchronize()
            assert torch.equal(outs[s], ref.cpu()), s
        if not ragged:
            ea, eb = a.export_state(), b.export_state()
            assert (ea["T"], ea["nf"], ea["npool"]) == (eb["T"], eb["nf"], eb["npool"])
            for key in STATE_KEYS:
                assert np.array_equal(ea[key], eb[key]), key
        a.check_device()
        b.check_device()


def test_step_host_argument_checks(ott):
    B, Hq, Hkv, d = 1, 2, 1, 128
    with ott.OTTCache(B, Hq, Hkv, d, 16, 4, 4, max_tokens=64) as c:
        k = torch.zeros(B, Hkv, d, dtype=torch.float16).pin_memory()
        q = torch.zeros(B, Hq, d, dtype=torch.float16).pin_memory()
        out = torch.zeros(B, Hq, d, dtype=torch.float16).pin_memory()
        with pytest.raises(TypeError):
            c.step_host(k, k.clone(), q, torch.zeros(B, Hq, d, dtype=torch.float16))   # not pinned
        with pytest.raises(TypeError):
            c.step_host(k.cuda(), k, q, out)                                           # on the device
        L = ott.load()
        sp = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = L.ott_step_host(c.handle, k.data_ptr(), k.data_ptr(), q.data_ptr(), q.data_ptr(), 0, sp)
        assert rc == ott.OTT_ERR_INVALID                      # out aliases q
        rc = L.ott_step_host(c.handle, k.data_ptr() + 2, k.data_ptr(), q.data_ptr(), out.data_ptr(), 0, sp)
        assert rc == ott.OTT_ERR_INVALID                      # k not 16-byte aligned
        rc = L.ott_step_host(c.handle, None, k.data_ptr(), q.data_ptr(), out.data_ptr(), 0, sp)
        assert rc == ott.OTT_ERR_INVALID                      # no k
        assert c.counts()[0] == 0                             # nothing queued
        c.step_host(k, k.clone().pin_memory(), q, out)
        torch.cuda.synchronize()
        assert c.counts()[0] == 1 and torch.isfinite(out.float()).all()
        c.check_device()


@pytest.mark.parametrize("ragged", [False, True])
def test_step_host_topk_equals_device_path(ott, ragged):
    """Top-K steps from host memory against ott_append + ott_decode_attn_topk
    on device buffers: every output equal, across a flush."""
    B, Hq, Hkv, d, G, R, P, L, steps, Kb = 2, 8, 2, 128, 16, 4, 6, 300, 30, 3
    K, V, Q = _gen(7, B, Hkv, Hq, L + steps, d)
    dev = torch.device("cuda")
    kw = dict(max_tokens=L + steps + 1, ragged=ragged)
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as a, ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as b:
        for c in (a, b):
            if ragged:
                c.prefill_lens(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev), [L, L - 40])
            else:
                c.prefill(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev))
        out = torch.empty(B, Hq, d, dtype=torch.float16).pin_memory()
        for s in range(steps):
            kh, vh, qh = (K[:, :, L + s].contiguous().pin_memory(), V[:, :, L + s].contiguous().pin_memory(),
                          Q[L + s].contiguous().pin_memory())
            a.step_host(kh, vh, qh, out, topk=Kb)
            b.append(kh.to(dev), vh.to(dev))
            ref = b.decode_attn_topk(qh.to(dev), Kb)
            torch.cuda.synchronize()
            assert torch.equal(out, ref.cpu()), s
        a.check_device()
        b.check_device()


@pytest.mark.parametrize("kind", ["paged", "pct", "cold"])
def test_step_host_on_other_caches(ott, kind):
    """The host-buffer step on a paged, a channel-criterion and a cold-pool
    cache, against the device path on the same kind of cache; then the
    allocation-free decode agrees with the last step."""
    B, Hq, Hkv, d, G, R, P, L, steps = 2, 4, 2, 128, 16, 4, 6, 120, 30
    K, V, Q = _gen(11, B, Hkv, Hq, L + steps, d)
    dev = torch.device("cuda")
    kw = dict(max_tokens=L + steps + 1)
    if kind == "paged":
        kw["pool_blocks"] = B * Hkv * 16
    elif kind == "pct":
        kw["pct"] = (2500, 4)
    else:
        kw["cold"] = 3
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as a, ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as b:
        for c in (a, b):
            c.prefill(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev))
        out = torch.empty(B, Hq, d, dtype=torch.float16).pin_memory()
        for s in range(steps):
            kh, vh, qh = (K[:, :, L + s].contiguous().pin_memory(), V[:, :, L + s].contiguous().pin_memory(),
                          Q[L + s].contiguous().pin_memory())
            a.step_host(kh, vh, qh, out)
            b.append(kh.to(dev), vh.to(dev))
            ref = b.decode_attn(qh.to(dev))
            torch.cuda.synchronize()
            assert torch.equal(out, ref.cpu()), (kind, s)
        st = torch.empty(B, Hq, d, dtype=torch.float16, device=dev)
        qd = qh.to(dev)
        L_ = ott.load()
        assert L_.ott_decode_attn_static(a.handle, qd.data_ptr(), st.data_ptr(),
                                         C.c_void_p(torch.cuda.current_stream().cuda_stream)) == ott.OTT_OK
        torch.cuda.synchronize()
        assert torch.equal(st.cpu(), out)
        a.check_device()
        b.check_device()
