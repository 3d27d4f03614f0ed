"""Time ott_decode_attn on one layer of a workload.

    python -m bit_kv_cache_ott_gb300.decode_loop WORKLOAD [CALLS] [--appends N]

Builds one layer's cache from the workload's seeded prefill (on the device),
optionally appends N tokens to every sequence (N >= G crosses a flush), makes
5 warm-up calls and CALLS timed calls on the current stream, and prints the
mean time per call (decode + combine, CUDA events) with the algorithmic bytes
and GB/s. Meant for profiling a single layer of large workloads whose full
bench runs many layers, and (with --appends) the flush of one group.
"""
from __future__ import annotations

import sys

import torch

from . import OTTCache, metrics, synth


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    if not argv or argv[0] not in synth.WORKLOADS:
        print(__doc__)
        print("workloads:", ", ".join(sorted(synth.WORKLOADS)))
        return 2
    w = synth.WORKLOADS[argv[0]]
    appends = 0
    if "--appends" in argv:
        k = argv.index("--appends")
        appends = int(argv[k + 1])
        argv = argv[:k] + argv[k + 2:]
    calls = int(argv[1]) if len(argv) > 1 else 20
    lens = synth.seq_lens(w)
    K, V = synth.prefill_kv(w, 0, w.L, "cuda")
    c = OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + appends + 1, ragged=w.ragged)
    if w.ragged:
        c.prefill_lens(K, V, lens)
    else:
        c.prefill(K, V)
    del K, V
    for s in range(appends):
        k_, v_, _ = synth.step_kvq(w, s)
        c.append(k_.cuda(), v_.cuda())
    lens = [t + appends for t in lens]
    q = torch.randn(w.B, w.Hq, w.d, device="cuda").half()
    out = torch.empty_like(q)
    for _ in range(5):
        c.decode_attn(q, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls):
        c.decode_attn(q, out)
    e1.record()
    torch.cuda.synchronize()
    c.check_device()
    us = e0.elapsed_time(e1) * 1e3 / calls
    byts = sum(metrics.decode_bytes(t, 1, w.Hq, w.Hkv, w.d, w.G, w.R, w.P) for t in lens)
    print(f"{w.name}: decode+combine {us:.1f} us/call, {byts / 1e6:.1f} MB, {byts / us / 1e3:.0f} GB/s")
    c.close()
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
