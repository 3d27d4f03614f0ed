"""Shared helpers for the GPU-vs-oracle parity tests.

Acceptance (the stated bar): the quantized state is bit-exact (codes,
scales/zeros, block token indices and counts, residual tokens, pool
membership, pool norms); the attention output, fp16 on the device, is
within max |d| <= 2e-3 and mean |d| <= 2e-4 of the oracle's double result.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

MAX_ABS = 2e-3
MEAN_ABS = 2e-4
STATE_KEYS = ("bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "tk", "tv", "pidx", "pnorm", "pk", "pv")


def compare_state(gpu: dict, orc_cache, units=None):
    """Bit-exact comparison of the device export with the oracle, unit by unit."""
    U = gpu["bidx"].shape[0]
    units = range(U) if units is None else units
    for u in units:
        e = orc_cache.export_unit(u)
        assert (gpu["T"], gpu["nf"], gpu["tail"], gpu["npool"]) == (e["T"], e["nf"], e["tail"], e["npool"]), u
        assert np.array_equal(gpu["bcount"], e["bcount"]), u
        for k in STATE_KEYS:
            g = gpu[k][u]
            o = e[k]
            if not np.array_equal(g, o):
                bad = np.argwhere(g != o)
                raise AssertionError(f"unit {u} field {k}: {len(bad)} mismatches, first at {bad[:3].tolist()}: "
                                     f"gpu {g[tuple(bad[0])]} oracle {o[tuple(bad[0])]}")


def compare_out(out_gpu: torch.Tensor, ref: np.ndarray, where: str = ""):
    g = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    d = np.abs(g - ref)
    assert np.all(np.isfinite(g)), f"non-finite output {where}"
    mx, mean = float(d.max()), float(d.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{where}: max|d|={mx:.3e} mean|d|={mean:.3e}"
    return mx, mean


def oracle_decode_all(orc, q, threads: int | None = None) -> np.ndarray:
    """The oracle's decode of every (sequence, query head), [B][Hq][d] float64,
    one head per call spread over host threads (the oracle's C call releases
    the interpreter lock and only reads the cache)."""
    B, Hq = q.shape[0], q.shape[1]
    out = np.zeros((B, Hq, q.shape[2]), np.float64)
    pairs = [(b, h) for b in range(B) for h in range(Hq)]

    def one(bh):
        b, h = bh
        out[b, h] = orc.decode_head(b, h, q[b, h])

    n = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(n) as ex:
        list(ex.map(one, pairs))
    return out
