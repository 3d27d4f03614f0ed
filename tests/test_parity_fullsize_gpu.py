"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: the whole quantized state bit-exact against the oracle at
every flush boundary the run crosses, and at the chosen decode steps the
attention output of every (sequence, query head) against the oracle (max and
mean |d| over the whole output).

The Llama-3.1-8B-shaped workload has 32 layers with identical shapes; each
layer's cache is independent, so one layer is checked here.
"""
import numpy as np
import pytest

from bit_kv_cache_ott_gb300 import synth
from tests.parity_util import compare_out, compare_state, oracle_decode_all

pytestmark = pytest.mark.gpu


def _units_to_check(w, limit):
    U = w.B * w.Hkv
    if U <= limit:
        return range(U)
    rng = np.random.default_rng(7)
    return sorted({0, U - 1, *rng.choice(U, limit - 2, replace=False).tolist()})


def run_fullsize(oracle_mod, ott, name, steps, decode_steps, unit_limit=64):
    w = synth.WORKLOADS[name]
    K, V = synth.prefill_kv(w)
    orc = oracle_mod.OracleCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P)
    orc.prefill(K, V)
    with ott.OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + steps) as c:
        c.prefill(K.cuda(), V.cuda())
        del K, V
        nf_prev = c.counts()[1]
        units = _units_to_check(w, unit_limit)
        compare_state(c.export_state(), orc)   # every unit after the prefill
        for s in range(steps):
            k, v, q = synth.step_kvq(w, s)
            c.append(k.cuda(), v.cuda())
            orc.append(k, v)
            nf = c.counts()[1]
            if nf != nf_prev:
                compare_state(c.export_state(), orc, units)
                nf_prev = nf
            if s in decode_steps:
                compare_out(c.decode_attn(q.cuda()), oracle_decode_all(orc, q), f"{name} step {s}")
        c.check_device()


def test_llama2_7b_layer(oracle_mod, ott):
    run_fullsize(oracle_mod, ott, "llama2_7b_layer", 256, {0, 31, 32, 100, 255})


def test_batch_b32_headline(oracle_mod, ott):
    run_fullsize(oracle_mod, ott, "batch_b32", 300, {0, 31, 32, 160, 299}, unit_limit=48)


@pytest.mark.parametrize("name", ["batch_b1", "batch_b8", "batch_b16"])
def test_batch_sweep(oracle_mod, ott, name):
    """The rest of the batch sweep (B = 1, 8, 16; B = 32 is the headline
    test): 140 steps across the flush after step 31, state at every flush,
    every output before and after it."""
    run_fullsize(oracle_mod, ott, name, 140, {0, 31, 32, 139}, unit_limit=40)


@pytest.mark.parametrize("name", ["mistral_gqa_g128", "mistral_gqa_g256"])
def test_mistral_gqa(oracle_mod, ott, name):
    run_fullsize(oracle_mod, ott, name, 256, {0, 63, 64, 200, 255})


def test_llama31_8b_131k_one_layer(oracle_mod, ott):
    run_fullsize(oracle_mod, ott, "llama31_8b_131k", 128, {0, 31, 32, 127})


def _compare_seq_state(c, orc, b, Hkv, STATE_KEYS):
    gpu = c.export_state(b * Hkv, Hkv)
    for h in range(Hkv):
        e = orc.export_unit(b * Hkv + h)
        assert (gpu["T"], gpu["nf"], gpu["tail"], gpu["npool"]) == (e["T"], e["nf"], e["tail"], e["npool"]), (b, h)
        assert np.array_equal(gpu["bcount"], e["bcount"]), (b, h)
        for k in STATE_KEYS:
            assert np.array_equal(gpu[k][h], e[k]), f"seq {b} head {h} field {k}"


def test_batch_b32_ragged(oracle_mod, ott):
    """The ragged serving batch (32 sequences of 1K..7K tokens): the state of
    every sequence that flushes is checked at the step it flushes, every
    output at chosen steps."""
    from tests.parity_util import STATE_KEYS
    w = synth.WORKLOADS["batch_b32_ragged"]
    lens = synth.seq_lens(w)
    steps, decode_steps = 200, {0, 37, 38, 120, 199}
    K, V = synth.prefill_kv(w)
    orc = oracle_mod.OracleCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P)
    orc.prefill_lens(K, V, lens)
    with ott.OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + steps, ragged=True) as c:
        c.prefill_lens(K.cuda(), V.cuda(), lens)
        del K, V
        for b in (0, 7, 19, w.B - 1):
            _compare_seq_state(c, orc, b, w.Hkv, STATE_KEYS)
        nf_prev = [c.seq_counts(b)[1] for b in range(w.B)]
        flushed = 0
        for s in range(steps):
            k, v, q = synth.step_kvq(w, s)
            c.append(k.cuda(), v.cuda())
            orc.append(k, v)
            for b in range(w.B):
                nf = c.seq_counts(b)[1]
                if nf != nf_prev[b]:
                    _compare_seq_state(c, orc, b, w.Hkv, STATE_KEYS)
                    nf_prev[b] = nf
                    flushed += 1
            if s in decode_steps:
                compare_out(c.decode_attn(q.cuda()), oracle_decode_all(orc, q), f"ragged step {s}")
        assert flushed > w.B // 2        # the sequences flushed at different steps
        c.check_device()


def test_batch_b32_cold(oracle_mod, ott):
    """The headline batch under the cold-pool policy (32 slots): per-unit
    block sizes, blocks, pool and cold pool bit-exact on sampled units after
    the prefill and at every flush; every output at chosen steps."""
    from tests.parity_util import STATE_KEYS
    w = synth.WORKLOADS["batch_b32_cold"]
    steps, decode_steps = 300, {0, 31, 32, 160, 299}
    K, V = synth.prefill_kv(w)
    orc = oracle_mod.OracleCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, cold=w.cold)
    orc.prefill(K, V)
    units = _units_to_check(w, 48)

    def check():
        gpu = c.export_state()
        for u in units:
            e = orc.export_unit(u)
            assert (gpu["T"], gpu["nf"], gpu["npool"]) == (e["T"], e["nf"], e["npool"])
            assert np.array_equal(gpu["bcount"][u], e["bcount"]), u
            assert gpu["ncold"][u] == e["ncold"], u
            for k in STATE_KEYS + ("cidx", "ck", "cv"):
                assert np.array_equal(gpu[k][u], e[k]), f"unit {u} field {k}"

    with ott.OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + steps, cold=w.cold) as c:
        c.prefill(K.cuda(), V.cuda())
        del K, V
        check()
        bc, nc = c.cold_sizes()
        assert nc.min() > 0 and (bc[:, 1:] < w.G).any()   # pool tokens were displaced
        nf_prev = c.counts()[1]
        for s in range(steps):
            k, v, q = synth.step_kvq(w, s)
            c.append(k.cuda(), v.cuda())
            orc.append(k, v)
            nf = c.counts()[1]
            if nf != nf_prev:
                check()
                nf_prev = nf
            if s in decode_steps:
                compare_out(c.decode_attn(q.cuda()), oracle_decode_all(orc, q), f"cold step {s}")
        c.check_device()
