"""The parallel prefill (every flush of a prompt in one pass: group norms and
smallest keys, a per-unit merge into the pool history, then all blocks at
once) against the same tokens appended one by one (each flush in order, from
the residual ring): the device state bit for bit and the decode outputs equal
(torch.equal), for the uniform, ragged and one-sequence prefill entry points,
with P below, equal to and above G, P = 0, d = 64 and GQA; plus the oracle
on the largest case.
"""
import numpy as np
import pytest
import torch

from tests.parity_util import STATE_KEYS, compare_out, compare_state

pytestmark = pytest.mark.gpu


def _gen(seed, B, Hkv, T, d):
    g = torch.Generator().manual_seed(seed)
    K = torch.randn(B, Hkv, T, d, generator=g)
    ch = torch.randint(0, d, (4,), generator=g)
    K[..., ch] *= 15
    low = torch.rand(B, Hkv, T, generator=g) < 0.05
    K[low] *= 0.03
    if T > 12:
        K[:, :, 9::11] = K[:, :, 4:5]       # ties in the norm
    V = torch.randn(B, Hkv, T, d, generator=g)
    return K.half().cuda(), V.half().cuda()


def _appended(ott, K, V, args, kw, L):
    c = ott.OTTCache(*args, **kw)
    for t in range(L):
        c.append(K[:, :, t].contiguous(), V[:, :, t].contiguous())
    return c


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,L", [
    (2, 2, 2, 128, 16, 4, 5, 300),       # P < G
    (1, 4, 2, 128, 16, 0, 16, 200),      # P = G, R = 0
    (2, 8, 2, 128, 16, 3, 40, 330),      # P > G: the first blocks are empty or short
    (2, 4, 1, 64, 32, 8, 7, 400),        # d = 64, GQA 4
    (3, 3, 3, 128, 20, 5, 0, 210),       # P = 0, G not a multiple of 16
    (1, 1, 1, 128, 128, 32, 32, 1200),   # the pages' G, R, P
    # enough groups on few units that the pool scan is cut into chunks with
    # a carry pass (3, 9 and 6 chunks per unit)
    (1, 4, 2, 128, 16, 4, 40, 1400),     # P > G
    (2, 2, 2, 64, 8, 2, 5, 2100),        # d = 64, P < G
    (1, 8, 1, 128, 16, 0, 64, 3000),     # P = 4 G, R = 0, GQA 8
])
def test_prefill_equals_appends(ott, B, Hq, Hkv, d, G, R, P, L):
    K, V = _gen(B + G + P, B, Hkv, L, d)
    args, kw = (B, Hq, Hkv, d, G, R, P), dict(max_tokens=L + 8)
    with ott.OTTCache(*args, **kw) as a, _appended(ott, K, V, args, kw, L) as b:
        a.prefill(K, V)
        ea, eb = a.export_state(), b.export_state()
        assert (ea["T"], ea["nf"], ea["tail"], ea["npool"]) == (eb["T"], eb["nf"], eb["tail"], eb["npool"])
        for k in STATE_KEYS + ("bcount",):
            assert np.array_equal(ea[k], eb[k]), k
        q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(3)).half().cuda()
        assert torch.equal(a.decode_attn(q), b.decode_attn(q))
        for t in range(3):   # decode continues identically from either state
            k_, v_ = K[:, :, t].contiguous(), V[:, :, t].contiguous()
            a.append(k_, v_)
            b.append(k_, v_)
            assert torch.equal(a.decode_attn(q), b.decode_attn(q))
        a.check_device()
        b.check_device()


@pytest.mark.parametrize("paged", [False, True])
def test_prefill_lens_and_seq_equal_appends(ott, paged):
    """Ragged prefill (each sequence its own parallel pass, sequences with
    fewer than two groups flushed group by group) and the one-sequence
    prefill of a serving slot, against token-by-token appends of each
    sequence on its own cache."""
    B, Hq, Hkv, d, G, R, P = 4, 4, 2, 128, 16, 4, 6
    lens = [170, 19, 35, 260]      # 10, 0, 1 and 16 flushes
    Lmax = max(lens)
    K, V = _gen(21, B, Hkv, Lmax, d)
    kw = dict(max_tokens=Lmax + 8, ragged=not paged, pool_blocks=(B * Hkv * 20) if paged else None)
    q = torch.randn(1, Hq, d, generator=torch.Generator().manual_seed(4)).half().cuda()
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as a, ott.OTTCache(B, Hq, Hkv, d, G, R, P, **kw) as s:
        a.prefill_lens(K, V, lens)
        for b in range(B):
            s.prefill_seq(b, K[b, :, : lens[b]].contiguous(), V[b, :, : lens[b]].contiguous())
        qa = q.expand(B, Hq, d).contiguous()
        oa, os_ = a.decode_attn(qa), s.decode_attn(qa)
        assert torch.equal(oa, os_)
        for b in range(B):
            L = lens[b]
            one = _appended(ott, K[b:b + 1, :, :L].contiguous(), V[b:b + 1, :, :L].contiguous(),
                            (1, Hq, Hkv, d, G, R, P), dict(max_tokens=Lmax + 8), L)
            with one:
                eo = one.export_state()
                for src in (a, s):
                    es = src.export_state(b * Hkv, Hkv)
                    assert (es["T"], es["nf"], es["npool"]) == (eo["T"], eo["nf"], eo["npool"]), b
                    for k in STATE_KEYS:
                        assert np.array_equal(es[k], eo[k]), (b, k)
                # another batch splits the work differently: equal up to the merge order
                d_ = (one.decode_attn(q).float() - oa[b:b + 1].float()).abs().max().item()
                assert d_ <= 2e-3, (b, d_)
        a.check_device()
        s.check_device()


def test_prefill_many_groups_against_oracle(oracle_mod, ott):
    """A long prompt in one parallel pass (2000 groups, a pool history two
    thousand merges deep): state bit-exact against the oracle, output within
    the bar."""
    B, Hq, Hkv, d, G, R, P, L = 1, 2, 2, 64, 16, 4, 24, 32004
    K, V = _gen(33, B, Hkv, L, d)
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill(K.cpu(), V.cpu())
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L) as c:
        c.prefill(K, V)
        compare_state(c.export_state(), orc)
        q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(5)).half()
        compare_out(c.decode_attn(q.cuda()), orc.decode(q), "long prefill")
        c.check_device()


@pytest.mark.parametrize("d", [64, 128])
def test_signed_zeros_and_repeated_values(oracle_mod, ott, d):
    """Blocks whose channels and value groups hold +0 and -0 together, runs
    of equal values, channels that are constant, and values exactly on the
    code boundaries: the scales, zeros (their sign included) and codes
    bit-exact against the oracle, through the parallel prefill and through
    the flushes of appends."""
    B, Hq, Hkv, G, R, P, L, steps = 2, 2, 2, 16, 4, 5, 200, 40
    g = torch.Generator().manual_seed(d)
    K = torch.randint(-2, 3, (B, Hkv, L + steps, d), generator=g).float() * 0.5
    V = torch.randint(-3, 4, (B, Hkv, L + steps, d), generator=g).float() * 0.25
    sign = torch.rand(B, Hkv, L + steps, d, generator=g) < 0.5
    K[(K == 0) & sign] = -0.0
    V[(V == 0) & sign] = -0.0
    K[:, :, :, 3] = 0.75                          # a constant channel: scale 0
    V[:, :, ::7, :32] = -0.0                      # a whole value group of -0
    K, V = K.half(), V.half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill(K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L + steps) as c:
        c.prefill(K[:, :, :L].contiguous().cuda(), V[:, :, :L].contiguous().cuda())
        compare_state(c.export_state(), orc)
        for s in range(steps):
            k, v = K[:, :, L + s].contiguous(), V[:, :, L + s].contiguous()
            c.append(k.cuda(), v.cuda())
            orc.append(k, v)
        compare_state(c.export_state(), orc)
        c.check_device()
