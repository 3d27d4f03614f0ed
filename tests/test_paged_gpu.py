"""GPU parity for the paged block pool and for serving a batch whose
sequences finish and are replaced (ott_create_paged, ott_release_seq,
ott_prefill_seq). The blocks of all units come from one pool through a block
table; the state read back through the table must equal the CPU oracle's bit
for bit, per sequence, and the outputs must be within max |d| <= 2e-3 and
mean |d| <= 2e-4 of its double result. A released and refilled sequence is a
fresh sequence of its own (the oracle pins that).
"""
import ctypes as C

import numpy as np
import pytest
import torch

from tests.parity_util import compare_out
from tests.test_ragged_gpu import _compare_seq, _gen

pytestmark = pytest.mark.gpu


def _blocks(lens, G, R, Hkv):
    return sum(((t - R) // G if t >= G + R else 0) for t in lens) * Hkv


def _serve(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, lens, steps, events, seed, pool=None, paged=True):
    """Prefill, then `steps` appends and decodes; events[s] = [(b, new prompt
    length), ...] releases sequence b before step s and refills it."""
    Lmax = max(lens) + 64
    K, V = _gen(seed, B, Hkv, Lmax + steps, d)
    g = torch.Generator().manual_seed(seed + 7)
    q_all = torch.randn(steps + 1, B, Hq, d, generator=g).half()
    prompts = {}
    for s, evs in events.items():
        for b, L in evs:
            kk, vv = _gen(seed + 100 * s + b, 1, Hkv, L, d)
            prompts[(s, b)] = (kk[0].contiguous(), vv[0].contiguous())
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill_lens(K[:, :, :Lmax].contiguous(), V[:, :, :Lmax].contiguous(), lens)
    dev = torch.device("cuda")
    kw = dict(pool_blocks=pool) if paged else dict(ragged=True)
    longest = max([Lmax] + [L for evs in events.values() for _, L in evs])
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=longest + steps + 1, **kw) as c:
        c.prefill_lens(K[:, :, :Lmax].contiguous().to(dev), V[:, :, :Lmax].contiguous().to(dev), lens)
        T = list(lens)
        for s in range(steps + 1):
            for b, L in events.get(s, []):
                free0 = c.free_blocks()
                c.release_seq(b)
                orc.release_seq(b)
                if paged:
                    assert c.free_blocks() == free0 + _blocks([T[b]], G, R, Hkv)
                kk, vv = prompts[(s, b)]
                c.prefill_seq(b, kk.to(dev), vv.to(dev))
                orc.prefill_seq(b, kk, vv)
                T[b] = L
            if paged:
                assert c.free_blocks() == pool - _blocks(T, G, R, Hkv)
            for b in range(B):
                assert c.seq_counts(b)[0] == T[b]
                if s % 5 == 0 or s == steps:
                    _compare_seq(c, orc, b, Hkv)
            out = c.decode_attn(q_all[s].to(dev))
            compare_out(out, orc.decode(q_all[s]), f"step {s} lens {T}")
            if s < steps:
                k = K[:, :, Lmax + s].contiguous()
                v = V[:, :, Lmax + s].contiguous()
                c.append(k.to(dev), v.to(dev))
                orc.append(k, v)
                T = [t + 1 for t in T]
        c.check_device()


@pytest.mark.parametrize("B,Hq,Hkv,d,G,R,P,lens,steps,events", [
    (4, 4, 2, 128, 16, 3, 5, [40, 97, 18, 130], 30, {6: [(1, 50)], 17: [(0, 3), (3, 77)]}),
    (3, 8, 2, 64, 32, 0, 7, [150, 5, 66], 40, {10: [(0, 200)], 25: [(2, 1)]}),     # GQA 4, d=64, R=0
    (6, 6, 6, 128, 128, 32, 32, [300, 161, 160, 159, 33, 1], 30, {12: [(4, 400)]}),   # the pages' G, R, P
    (3, 16, 2, 64, 32, 0, 7, [150, 5, 66], 40, {10: [(0, 200)], 25: [(2, 1)]}),   # GQA 8: two slices
])
def test_paged_serving(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, lens, steps, events):
    # a pool just large enough for the run
    need = 0
    T = list(lens)
    for s in range(steps + 1):
        for b, L in events.get(s, []):
            T[b] = L
        need = max(need, _blocks(T, G, R, Hkv))
        T = [t + 1 for t in T]
    _serve(oracle_mod, ott, B, Hq, Hkv, d, G, R, P, lens, steps, events, seed=sum(lens) + G, pool=need + 1)


def test_release_and_refill_without_a_pool(oracle_mod, ott):
    """The same serving calls on a ragged cache with its own blocks per unit."""
    _serve(oracle_mod, ott, 4, 4, 2, 128, 16, 3, 5, [40, 97, 18, 130], 30, {6: [(1, 50)], 17: [(3, 77)]},
           seed=11, paged=False)


def test_pool_exhaustion_is_refused_and_recovers(ott):
    """A flush that needs more free blocks than the pool has is refused before
    anything is queued; releasing a sequence makes room."""
    B, Hq, Hkv, d, G, R, P = 2, 2, 1, 128, 16, 2, 3
    dev = torch.device("cuda")
    K, V = _gen(3, B, Hkv, 200, d)
    lens = [17, 33]                       # 0 and 1 flushes (a flush is due when 18 tokens wait)
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=256, pool_blocks=3) as c:
        c.prefill_lens(K[:, :, :40].contiguous().to(dev), V[:, :, :40].contiguous().to(dev), lens)
        assert c.free_blocks() == 2
        k, v = K[:, :, 40].contiguous().to(dev), V[:, :, 40].contiguous().to(dev)
        c.append(k, v)                     # T = 18, 34: both flush, taking the last two blocks
        assert c.free_blocks() == 0
        for _ in range(15):                # up to T = 33, 49: both flush at the next append
            c.append(k, v)
        t_before = [c.seq_counts(b)[0] for b in range(B)]
        with pytest.raises(ott.OTTError) as ei:
            c.append(k, v)
        assert ei.value.code == ott.OTT_ERR_CAPACITY
        assert [c.seq_counts(b)[0] for b in range(B)] == t_before     # nothing happened
        c.release_seq(1)
        with pytest.raises(ott.OTTError) as ei:
            c.append(k, v)                 # an empty sequence blocks appends
        assert ei.value.code == ott.OTT_ERR_STATE
        c.prefill_seq(1, K[1, :, :10].contiguous().to(dev), V[1, :, :10].contiguous().to(dev))
        assert c.free_blocks() == 2        # sequence 1 gave back its two blocks
        c.append(k, v)                     # sequence 0 flushes into a returned block
        assert c.seq_counts(0)[1] == 2 and c.free_blocks() == 1
        c.decode_attn(torch.zeros(B, Hq, d, dtype=torch.float16, device=dev))
        c.check_device()


def test_paged_argument_errors(ott):
    L = ott.load()
    h = C.c_void_p(123)
    assert L.ott_create_paged(2, 1, 1, 128, 16, 2, 4, 64, 0, C.byref(h)) == ott.OTT_ERR_INVALID
    assert h.value is None
    assert L.ott_create_paged(300, 1, 1, 128, 16, 2, 4, 64, 10, C.byref(h)) == ott.OTT_ERR_INVALID
    dev = torch.device("cuda")
    K = torch.zeros(2, 1, 40, 128, device=dev, dtype=torch.float16)
    with ott.OTTCache(2, 1, 1, 128, 16, 2, 4, max_tokens=64, pool_blocks=10) as c:
        with pytest.raises(ott.OTTError) as ei:
            c.release_seq(0)               # nothing to release yet
        assert ei.value.code == ott.OTT_ERR_STATE
        c.prefill_lens(K, K.clone(), [20, 40])
        with pytest.raises(ott.OTTError) as ei:
            c.prefill_seq(0, K[0].contiguous(), K[0].contiguous())   # sequence 0 is not empty
        assert ei.value.code == ott.OTT_ERR_STATE
    with ott.OTTCache(2, 1, 1, 128, 16, 2, 4, max_tokens=64) as plain:
        plain.prefill(K, K.clone())
        with pytest.raises(ott.OTTError) as ei:
            plain.release_seq(0)           # not created for per-sequence lengths
        assert ei.value.code == ott.OTT_ERR_STATE
        assert plain.free_blocks() == -1


@pytest.mark.parametrize("paged", [True, False])
def test_release_after_a_uniform_prefill(oracle_mod, ott, paged):
    """A cache filled by ott_prefill (one length for all) switches to
    per-sequence counts at its first release; it then serves like the others."""
    B, Hq, Hkv, d, G, R, P, L, steps = 3, 6, 3, 128, 16, 2, 4, 70, 24
    K, V = _gen(21, B, Hkv, L + steps, d)
    kk, vv = _gen(22, 1, Hkv, 45, d)
    q_all = torch.randn(steps, B, Hq, d, generator=torch.Generator().manual_seed(23)).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    orc.prefill(K[:, :, :L].contiguous(), V[:, :, :L].contiguous())
    dev = torch.device("cuda")
    kw = dict(pool_blocks=_blocks([L + steps] * B, G, R, Hkv) + 1) if paged else dict(ragged=True)
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=L + steps + 1, **kw) as c:
        c.prefill(K[:, :, :L].contiguous().to(dev), V[:, :, :L].contiguous().to(dev))
        for s in range(steps):
            if s == 9:
                c.release_seq(2)
                orc.release_seq(2)
                c.prefill_seq(2, kk[0].contiguous().to(dev), vv[0].contiguous().to(dev))
                orc.prefill_seq(2, kk[0].contiguous(), vv[0].contiguous())
            compare_out(c.decode_attn(q_all[s].to(dev)), orc.decode(q_all[s]), f"step {s}")
            k, v = K[:, :, L + s].contiguous(), V[:, :, L + s].contiguous()
            c.append(k.to(dev), v.to(dev))
            orc.append(k, v)
        for b in range(B):
            _compare_seq(c, orc, b, Hkv)
        c.check_device()


def test_paged_cache_filled_by_appends(oracle_mod, ott):
    """No prefill: every token arrives through ott_append, from an empty cache."""
    B, Hq, Hkv, d, G, R, P, T = 2, 4, 2, 128, 16, 3, 5, 90
    K, V = _gen(41, B, Hkv, T, d)
    q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(42)).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=T + 1, pool_blocks=_blocks([T] * B, G, R, Hkv)) as c:
        for t in range(T):
            k, v = K[:, :, t].contiguous(), V[:, :, t].contiguous()
            c.append(k.to(dev), v.to(dev))
            orc.append(k, v)
            if t % 23 == 0 or t == T - 1:
                compare_out(c.decode_attn(q.to(dev)), orc.decode(q), f"T={t + 1}")
        assert c.free_blocks() == 0
        for b in range(B):
            _compare_seq(c, orc, b, Hkv)
        c.check_device()


def test_paged_static_decode_matches(ott):
    """The allocation-free entry point reads the pool through the table too."""
    B, Hq, Hkv, d, G, R, P = 3, 4, 2, 128, 16, 3, 5
    lens = [40, 97, 18]
    K, V = _gen(51, B, Hkv, max(lens), d)
    dev = torch.device("cuda")
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=128, pool_blocks=_blocks(lens, G, R, Hkv) + 2) as c:
        c.prefill_lens(K.contiguous().to(dev), V.contiguous().to(dev), lens)
        q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(5)).half().to(dev)
        ref = c.decode_attn(q)
        out = torch.full_like(ref, float("nan"))
        rc = ott.load().ott_decode_attn_static(C.c_void_p(c.handle), C.c_void_p(q.data_ptr()),
                                               C.c_void_p(out.data_ptr()),
                                               C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == ott.OTT_OK
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the same bits
        assert torch.equal(out, ref)


@pytest.mark.parametrize("paged", [True, False])
def test_rotation_beyond_max_tokens(oracle_mod, ott, paged):
    """A serving loop that keeps releasing and refilling sequences runs for
    more appends than max_tokens: the capacity is per sequence, so no call is
    refused while every sequence stays below it."""
    B, Hq, Hkv, d, G, R, P, M = 3, 3, 3, 64, 8, 2, 3, 40
    steps = 3 * M
    K, V = _gen(61, B, Hkv, steps + M, d)
    q_all = torch.randn(steps, B, Hq, d, generator=torch.Generator().manual_seed(62)).half()
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    dev = torch.device("cuda")
    # a pool for every sequence at its longest
    kw = dict(pool_blocks=_blocks([M] * B, G, R, Hkv) + 1) if paged else dict(ragged=True)
    lens = [5, 12, 20]
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=M, **kw) as c:
        c.prefill_lens(K[:, :, :20].contiguous().to(dev), V[:, :, :20].contiguous().to(dev), lens)
        orc.prefill_lens(K[:, :, :20].contiguous(), V[:, :, :20].contiguous(), lens)
        T = list(lens)
        refills = 0
        for s in range(steps):
            for b in range(B):
                if T[b] + 1 > M:                # about to outgrow max_tokens: replace it
                    c.release_seq(b)
                    orc.release_seq(b)
                    L = 1 + (s + 3 * b) % 7
                    kk, vv = _gen(1000 + s * B + b, 1, Hkv, L, d)
                    c.prefill_seq(b, kk[0].contiguous().to(dev), vv[0].contiguous().to(dev))
                    orc.prefill_seq(b, kk[0].contiguous(), vv[0].contiguous())
                    T[b] = L
                    refills += 1
            k, v = K[:, :, M + s].contiguous(), V[:, :, M + s].contiguous()
            c.append(k.to(dev), v.to(dev))
            orc.append(k, v)
            T = [t + 1 for t in T]
            if s % 11 == 0 or s == steps - 1:
                compare_out(c.decode_attn(q_all[s].to(dev)), orc.decode(q_all[s]), f"step {s} lens {T}")
        assert refills >= 6 and steps > M
        for b in range(B):
            _compare_seq(c, orc, b, Hkv)
        c.check_device()


@pytest.mark.parametrize("paged", [True, False])
def test_empty_cache_filled_one_sequence_at_a_time(oracle_mod, ott, paged):
    """An empty serving cache takes its prompts through ott_prefill_seq, one
    sequence at a time; appends wait until every sequence holds a token."""
    B, Hq, Hkv, d, G, R, P = 3, 6, 3, 128, 16, 2, 4
    lens, steps = [37, 5, 60], 12
    dev = torch.device("cuda")
    orc = oracle_mod.OracleCache(B, Hq, Hkv, d, G, R, P)
    kw = dict(pool_blocks=_blocks([L + steps for L in lens], G, R, Hkv)) if paged else dict(ragged=True)
    K, V = _gen(71, B, Hkv, steps, d)
    q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(72)).half()
    with ott.OTTCache(B, Hq, Hkv, d, G, R, P, max_tokens=max(lens) + steps, **kw) as c:
        for b, L in enumerate(lens):
            kk, vv = _gen(80 + b, 1, Hkv, L, d)
            c.prefill_seq(b, kk[0].contiguous().to(dev), vv[0].contiguous().to(dev))
            orc.prefill_seq(b, kk[0].contiguous(), vv[0].contiguous())
            if b < B - 1:
                with pytest.raises(ott.OTTError) as ei:   # sequence b+1 is still empty
                    c.append(K[:, :, 0].contiguous().to(dev), V[:, :, 0].contiguous().to(dev))
                assert ei.value.code == ott.OTT_ERR_STATE
        for s in range(steps):
            k, v = K[:, :, s].contiguous(), V[:, :, s].contiguous()
            c.append(k.to(dev), v.to(dev))
            orc.append(k, v)
        compare_out(c.decode_attn(q.to(dev)), orc.decode(q), "after the appends")
        for b in range(B):
            assert c.seq_counts(b)[0] == lens[b] + steps
            _compare_seq(c, orc, b, Hkv)
        c.check_device()
