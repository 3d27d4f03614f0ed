"""ott_decode_attn_static: the allocation-free decode entry point.

Callers on a decode path where no device memory may be allocated (an engine
that gave all free memory to its own pool, a latency-critical loop) use this
variant; its split-K partials live in a fixed device array inside libott.
Here it is called through the C ABI and checked against ott_decode_attn on
two calls in a row (with an append between them): both run the same kernels
on the same inputs, so the outputs must agree bit for bit; one case is also
checked against the CPU oracle within the parity tests' output tolerance.
The file runs last so that, if it fails, a stop-at-first-failure run has
already run everything else; it must also pass alone in a fresh process,
where its first call sets up the array's address.
"""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu



def _static_decode(ott, cache, q, out):
    rc = ott.load().ott_decode_attn_static(C.c_void_p(cache.handle), C.c_void_p(q.data_ptr()),
                                          C.c_void_p(out.data_ptr()),
                                          C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,L", [
    (4, 8, 8, 128, 128, 32, 32, 700),     # MHA, several flushes
    (2, 8, 2, 128, 32, 4, 6, 300),        # GQA 4
    (3, 2, 1, 64, 16, 3, 5, 120),         # d = 64, GQA 2
    (2, 16, 2, 128, 32, 4, 6, 300),       # GQA 8: two slices
    (3, 3, 1, 64, 16, 3, 5, 120),         # GQA 3: a padded slice
])
def test_static_decode_matches_decode_twice(ott, B, Hq, Hkv, d, G, R, P, L):
    g = torch.Generator().manual_seed(L + G)
    dev = torch.device("cuda")
    K = torch.randn(B, Hkv, L + 1, d, generator=g).half().to(dev)
    V = torch.randn(B, Hkv, L + 1, d, generator=g).half().to(dev)
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L + 1) as c:
        c.prefill(K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
        for call in range(2):
            q = torch.randn(B, Hq, d, generator=g).half().to(dev)
            ref = c.decode_attn(q)
            out = torch.full_like(ref, float("nan"))
            assert _static_decode(ott, c, q, out) == ott.OTT_OK
            torch.cuda.synchronize()
            assert torch.isfinite(out.float()).all()
            assert torch.equal(out, ref), f"call {call}: max |d| {float((out.float() - ref.float()).abs().max())}"
            if call == 0:   # change the cache between the two calls
                c.append(K[:, :, L].contiguous(), V[:, :, L].contiguous())
        c.check_device()


def test_static_decode_matches_the_oracle(oracle_mod, ott):
    """The allocation-free decode against the CPU oracle (GQA 2, several flushes)."""
    from tests.parity_util import compare_out
    B, Hq, Hkv, d, G, R, P, L = 2, 4, 2, 128, 32, 8, 12, 250
    g = torch.Generator().manual_seed(3)
    K = torch.randn(B, Hkv, L, d, generator=g).half()
    V = torch.randn(B, Hkv, L, d, generator=g).half()
    q = torch.randn(B, Hq, d, generator=g).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill(K, V)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L) as c:
        c.prefill(K.to(dev), V.to(dev))
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.float16, device=dev)
        assert _static_decode(ott, c, q.to(dev), out) == ott.OTT_OK
        torch.cuda.synchronize()
        compare_out(out, orc.decode(q), "static decode")
        c.check_device()


def test_static_decode_rejects_a_shape_beyond_its_array(ott):
    """Enough (sequence, kv head) units that the partials outgrow the fixed
    array: the call says so instead of writing past it."""
    dev = torch.device("cuda")
    B, Hq, Hkv, d = 160, 128, 32, 128          # 5120 units, 4 query heads each
    with ott.OTTCache(B, Hq, Hkv, d, 16, 4, 4, max_tokens=24) as c:
        K = torch.zeros(B, Hkv, 24, d, device=dev, dtype=torch.float16)
        c.prefill(K, K.clone())
        q = torch.zeros(B, Hq, d, device=dev, dtype=torch.float16)
        out = torch.empty_like(q)
        assert _static_decode(ott, c, q, out) == ott.OTT_ERR_CAPACITY
        c.decode_attn(q, out)                   # the regular entry point still works
        torch.cuda.synchronize()
        c.check_device()


def test_static_decode_argument_errors(ott):
    dev = torch.device("cuda")
    with ott.OTTCache(1, 1, 1, 128, 16, 2, 2, max_tokens=8) as c:
        q = torch.zeros(1, 1, 128, device=dev, dtype=torch.float16)
        out = torch.empty_like(q)
        assert _static_decode(ott, c, q, out) == ott.OTT_ERR_STATE     # empty cache
        L = ott.load()
        assert L.ott_decode_attn_static(None, None, None, None) == ott.OTT_ERR_INVALID
