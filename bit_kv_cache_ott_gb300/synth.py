"""Seeded synthetic inputs and the named workloads.

This module holds no part of the method's arithmetic: it only draws the keys,
values and queries that both the CUDA library and the CPU oracle consume.

The key distribution stands in for the activations the OTT pages describe
("Accurate KV Cache Quantization with Outlier Tokens Tracing", sciencestack.ai
Fig. 1(a),(d),(e), Fig. 4, Fig. 5; zijie-tian.site sec. 2.1): keys carry a few
outlier channels of large magnitude, and inside them a few tokens whose keys
are small. Values show no structure. Recipe, per (layer, kv head):

* K ~ N(0, 1) per element; 4 channels, drawn without replacement, are scaled
  by 15 (the outlier channels, shared by every sequence of the batch).
* Each token independently (probability ``outlier_rate``) has its whole key
  vector scaled by 0.03: the low-norm outlier tokens.
* V ~ N(0, 1), q ~ N(0, 1).
* Everything is drawn in fp32 with a CPU ``torch.Generator`` and rounded to
  fp16; the same host tensors feed the oracle and the device.

Decode step ``s`` draws its k, v, q from its own generator, so any step can be
produced without replaying the earlier ones.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

OUTLIER_CHANNELS = 4
OUTLIER_CHANNEL_SCALE = 15.0
LOW_NORM_SCALE = 0.03


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    L: int            # prefill length
    steps: int        # decode steps
    G: int
    R: int
    P: int
    outlier_rate: float = 0.005
    layers: int = 1   # independent caches (one per layer)
    seed: int = 1000
    len_lo: int = 0   # > 0: sequence b's prefill length is drawn uniformly from [len_lo, L]
    cold: int = -1    # >= 0: the cold-pool eviction policy with this capacity
    topk: int = 0     # > 0: decode with ott_decode_attn_topk, this many blocks per (sequence, kv head)
    paged: bool = False   # ragged workloads: the blocks come from one pool (ott_create_paged)

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def ragged(self) -> bool:
        return self.len_lo > 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The pages' shapes (defaults G=128, R=32, P=32 from zijie-tian.site sec. 4 and
# sec. 6; model shapes of Llama-2-7B, Mistral-7B and Llama-3.1-8B layers).
WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hq=1, Hkv=1, d=128, L=512, steps=64,
                     G=128, R=32, P=32, seed=1000),
    "llama2_7b_layer": Workload("llama2_7b_layer", B=1, Hq=32, Hkv=32, d=128, L=4096,
                                steps=256, G=128, R=32, P=32, seed=1001),
    "batch_b1": Workload("batch_b1", B=1, Hq=32, Hkv=32, d=128, L=4096, steps=512,
                         G=128, R=32, P=32, seed=1002),
    "batch_b8": Workload("batch_b8", B=8, Hq=32, Hkv=32, d=128, L=4096, steps=512,
                         G=128, R=32, P=32, seed=1002),
    "batch_b16": Workload("batch_b16", B=16, Hq=32, Hkv=32, d=128, L=4096, steps=512,
                          G=128, R=32, P=32, seed=1002),
    "batch_b32": Workload("batch_b32", B=32, Hq=32, Hkv=32, d=128, L=4096, steps=512,
                          G=128, R=32, P=32, seed=1002),
    "mistral_gqa_g128": Workload("mistral_gqa_g128", B=4, Hq=32, Hkv=8, d=128, L=32768,
                                 steps=256, G=128, R=32, P=32, seed=1003),
    "mistral_gqa_g256": Workload("mistral_gqa_g256", B=4, Hq=32, Hkv=8, d=128, L=32768,
                                 steps=256, G=256, R=64, P=32, seed=1003),
    "llama31_8b_131k": Workload("llama31_8b_131k", B=1, Hq=32, Hkv=8, d=128, L=131072,
                                steps=128, G=128, R=32, P=64, outlier_rate=0.002,
                                layers=32, seed=1004),
    # a serving batch whose sequences differ in length (mean ~4096 tokens)
    "batch_b32_ragged": Workload("batch_b32_ragged", B=32, Hq=32, Hkv=32, d=128, L=7168, steps=512,
                                 G=128, R=32, P=32, seed=1005, len_lo=1024),
    # the ragged serving batch with its blocks drawn from one pool through a block table
    "batch_b32_paged": Workload("batch_b32_paged", B=32, Hq=32, Hkv=32, d=128, L=7168, steps=512,
                                G=128, R=32, P=32, seed=1005, len_lo=1024, paged=True),
    # the headline batch under the cold-pool policy with the pages' 32 slots
    # long contexts decoded with Top-K sparse access (1/8 and 1/16 of the blocks)
    "mistral_gqa_g128_topk32": Workload("mistral_gqa_g128_topk32", B=4, Hq=32, Hkv=8, d=128, L=32768,
                                        steps=256, G=128, R=32, P=32, seed=1003, topk=32),
    "llama31_8b_131k_topk64": Workload("llama31_8b_131k_topk64", B=1, Hq=32, Hkv=8, d=128, L=131072,
                                       steps=128, G=128, R=32, P=64, outlier_rate=0.002,
                                       layers=32, seed=1004, topk=64),
    "batch_b32_cold": Workload("batch_b32_cold", B=32, Hq=32, Hkv=32, d=128, L=4096, steps=512,
                               G=128, R=32, P=32, seed=1002, cold=32),
}

HEADLINE = "batch_b32"


def seq_lens(w: Workload) -> list[int]:
    """Prefill length of every sequence: w.L for all, or (ragged workloads)
    drawn uniformly from [w.len_lo, w.L] by the workload's seed."""
    if not w.ragged:
        return [w.L] * w.B
    g = _gen(w.seed * 104729 + 11)
    return [int(x) for x in torch.randint(w.len_lo, w.L + 1, (w.B,), generator=g)]


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def outlier_channels(w: Workload, layer: int = 0) -> torch.Tensor:
    """[Hkv][4] channel indices scaled by 15 in layer ``layer``'s keys."""
    g = _gen(w.seed * 7919 + 17 * layer + 3)
    rows = [torch.randperm(w.d, generator=g)[:OUTLIER_CHANNELS] for _ in range(w.Hkv)]
    return torch.stack(rows)


def _channel_scale(w: Workload, layer: int) -> torch.Tensor:
    """[Hkv][d] fp32 multiplier: 15 on the outlier channels, 1 elsewhere."""
    sc = torch.ones(w.Hkv, w.d)
    ch = outlier_channels(w, layer)
    sc.scatter_(1, ch, OUTLIER_CHANNEL_SCALE)
    return sc


def _keys(w: Workload, g: torch.Generator, shape_tokens: tuple, layer: int) -> torch.Tensor:
    """fp32 keys of shape [B][Hkv][*tokens][d] with outlier channels and tokens."""
    dev = g.device
    k = torch.randn(w.B, w.Hkv, *shape_tokens, w.d, generator=g, device=dev)
    sc = _channel_scale(w, layer).to(dev).view(1, w.Hkv, *([1] * len(shape_tokens)), w.d)
    k.mul_(sc)
    low = torch.rand(w.B, w.Hkv, *shape_tokens, generator=g, device=dev) < w.outlier_rate
    k[low] *= LOW_NORM_SCALE
    return k


def prefill_kv(w: Workload, layer: int = 0, L: int | None = None, device: str = "cpu"):
    """(K, V) fp16 tensors [B][Hkv][L][d] for the prefill of layer ``layer``.

    ``device="cpu"`` is the reference draw that tests share with the oracle.
    Drawing on a CUDA device follows the same recipe with the device's own
    generator (different numbers, same distribution): the benchmark uses it
    to build large caches quickly.
    """
    L = w.L if L is None else L
    g = _gen(w.seed * 1_000_003 + 101 * layer, device)
    K = _keys(w, g, (L,), layer).half()
    V = torch.randn(w.B, w.Hkv, L, w.d, generator=g, device=g.device).half()
    return K, V


def step_kvq(w: Workload, step: int, layer: int = 0):
    """(k, v, q) for decode step ``step``: [B][Hkv][d], [B][Hkv][d], [B][Hq][d] fp16."""
    g = _gen(w.seed * 1_000_003 + 101 * layer + 7_777_777 + 13 * step)
    k = _keys(w, g, (), layer)
    v = torch.randn(w.B, w.Hkv, w.d, generator=g)
    q = torch.randn(w.B, w.Hq, w.d, generator=g)
    return k.half(), v.half(), q.half()


def query(w: Workload, step: int, layer: int = 0) -> torch.Tensor:
    """Only the query of decode step ``step`` (same draw as ``step_kvq``)."""
    return step_kvq(w, step, layer)[2]
