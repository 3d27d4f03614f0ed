"""Independent brute-force statement of the OTT cache state, for tiny inputs.

Where the oracle merges the pool flush by flush, this module states the result
globally: after flush j the pool is the P smallest (norm, index) pairs among
ALL tokens flushed so far, and block j is (pool_{j-1} + group_j) - pool_j.
(Keeping the P smallest of a union is associative, so the two statements must
agree; a mistake in either one shows up as a mismatch.)

Sources: "Accurate KV Cache Quantization with Outlier Tokens Tracing"
(zijie-tian.site sec. 3.1, 3.2; sciencestack.ai TL;DR, Fig. 1(c)).
Norms use numpy's strictly sequential ``np.add.accumulate`` in fp32.
"""
from __future__ import annotations

import numpy as np


def norms_fp32(keys16: np.ndarray) -> np.ndarray:
    """[n][d] fp16 -> [n] fp32 squared norms, accumulated in channel order."""
    sq = keys16.astype(np.float32) ** 2          # exact: fp16 squares fit fp32
    return np.add.accumulate(sq, axis=1, dtype=np.float32)[:, -1]


def flush_count(T: int, G: int, R: int) -> int:
    return (T - R) // G if T >= G + R else 0


def state(keys16: np.ndarray, G: int, R: int, P: int):
    """Membership of one (sequence, kv head) after T = len(keys16) appends.

    Returns (blocks, pool, tail): blocks is a list of ascending token lists,
    pool the pool's tokens ascending, tail the residual tokens ascending.
    """
    T = len(keys16)
    nf = flush_count(T, G, R)
    n = norms_fp32(keys16[: nf * G]) if nf else np.zeros(0, np.float32)
    order_key = lambda t: (float(n[t]), t)
    prev: set[int] = set()
    blocks = []
    for j in range(nf):
        flushed = range((j + 1) * G)
        pool_j = set(sorted(flushed, key=order_key)[:P])
        group = set(range(j * G, (j + 1) * G))
        blocks.append(sorted((prev | group) - pool_j))
        prev = pool_j
    return blocks, sorted(prev), list(range(nf * G, T)), n


def state_cold(keys16: np.ndarray, G: int, R: int, P: int, C: int):
    """Membership under the cold-pool policy (capacity C) after T appends.

    Stated globally from the same pool sets: pool_j is the P smallest pairs
    among all tokens flushed by flush j; the tokens evicted at flush j are
    pool_{j-1} - pool_j, ranked by (j, index); the cold pool holds the last C
    of that ranking, oldest first; block j is group_j - pool_j.
    Returns (blocks, pool, tail, cold, dropped).
    """
    T = len(keys16)
    nf = flush_count(T, G, R)
    n = norms_fp32(keys16[: nf * G]) if nf else np.zeros(0, np.float32)
    order_key = lambda t: (float(n[t]), t)
    prev: set[int] = set()
    blocks, evicted = [], []
    for j in range(nf):
        pool_j = set(sorted(range((j + 1) * G), key=order_key)[:P])
        group = set(range(j * G, (j + 1) * G))
        blocks.append(sorted(group - pool_j))
        evicted += sorted(prev - pool_j)
        prev = pool_j
    cold = evicted[max(0, len(evicted) - C):] if C > 0 else []
    dropped = sorted(set(evicted) - set(cold))
    return blocks, sorted(prev), list(range(nf * G, T)), cold, dropped


def np_quant(x32: np.ndarray, axis: int):
    """Vectorized restatement of the 2-bit rule along ``axis`` (cross-check only)."""
    mn = x32.min(axis=axis, keepdims=True)
    mx = x32.max(axis=axis, keepdims=True)
    s16 = ((mx - mn) / np.float32(3.0)).astype(np.float16)
    s = s16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.rint((x32 - mn) / np.where(s == 0, np.float32(1), s))
    code = np.where(s == 0, 0, np.clip(y, 0, 3)).astype(np.uint8)
    return s16, mn, code


def unpack_rows(packed: np.ndarray, d: int) -> np.ndarray:
    """[..., d/4] canonical bytes -> [..., d] codes (channel c at bits 2(c%4))."""
    sh = np.array([0, 2, 4, 6], np.uint8)
    codes = (packed[..., :, None] >> sh) & 3
    return codes.reshape(*packed.shape[:-1], d)


def state_pct(keys16: np.ndarray, G: int, R: int, P: int, pct: int, n_oc: int):
    """Membership under the channel-conditioned criterion after T appends,
    restated with numpy (blocks, pool, tail, pool scores).

    At each flush the candidates are the pool and the group; the outlier
    channels are the n_oc channels with the largest max |k| over them (ties
    to the lower channel); a candidate's score is its fp32 squared norm over
    those channels in ascending channel order; the pool keeps the
    min(P, ceil(pct * n / 10000)) smallest (score, index) pairs; every other
    candidate joins the block, in token order."""
    T = len(keys16)
    nf = flush_count(T, G, R)
    pool: list[int] = []
    blocks = []
    scores = {}
    for j in range(nf):
        cand = pool + list(range(j * G, (j + 1) * G))
        a = np.abs(keys16[cand].astype(np.float32)).max(axis=0)
        order = np.lexsort((np.arange(a.size), -a))          # largest first, lower channel on ties
        oc = np.sort(order[:n_oc])
        sq = keys16[cand][:, oc].astype(np.float32) ** 2
        sc = np.add.accumulate(sq, axis=1, dtype=np.float32)[:, -1]
        ranked = sorted(range(len(cand)), key=lambda x: (float(sc[x]), cand[x]))
        m = -(-pct * len(cand) // 10000)
        keep = min(P, m)
        pool = [cand[x] for x in ranked[:keep]]
        scores = {cand[x]: sc[x] for x in ranked[:keep]}
        blocks.append(sorted(cand[x] for x in ranked[keep:]))
    return blocks, sorted(pool), list(range(nf * G, T)), scores


def pct_pool_sizes(nf: int, G: int, P: int, pct: int) -> list[int]:
    """Pool size after each flush: min(P, ceil(pct * (previous + G) / 10000))."""
    out, prev = [], 0
    for _ in range(nf):
        prev = min(P, -(-pct * (prev + G) // 10000))
        out.append(prev)
    return out
