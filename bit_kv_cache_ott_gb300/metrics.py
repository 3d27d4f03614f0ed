"""Counting rules for the measurements (no timing here).

Algorithmic bytes of one decode-attention call, per (sequence, kv head),
counting only what the method must read or write once:

    K codes   n_q * d/4          V codes   n_q * d/4
    K scale/zero  (non-empty blocks) * d * 4
    V scale/zero  n_q * (d/32) * 4
    fp16 residual + pool tokens   (tail + n_pool) * d * 4   (K and V)
    queries in and outputs out    g * d * 4

with n_q = nf*G - n_pool quantized tokens. Padding slots, split-K partials,
token indices, norms and block counts are not credited. At d = 128 this is
84 bytes per quantized token and 512 bytes per fp16 token.
"""
from __future__ import annotations


def flush_count(T: int, G: int, R: int) -> int:
    return (T - R) // G if T >= G + R else 0


def pool_size(T: int, G: int, R: int, P: int) -> int:
    return min(P, flush_count(T, G, R) * G)


def block_count(j: int, G: int, P: int) -> int:
    return min(P, j * G) + G - min(P, (j + 1) * G)


def decode_bytes_per_unit(T: int, d: int, g: int, G: int, R: int, P: int) -> int:
    nf = flush_count(T, G, R)
    npool = pool_size(T, G, R, P)
    nq = nf * G - npool
    tail = T - nf * G
    # block j is empty exactly when the pool absorbs its whole group: (j+1)G <= P
    nonempty = nf - min(nf, P // G)
    return (2 * nq * d // 4 + nonempty * d * 4 + nq * (d // 32) * 4
            + (tail + npool) * d * 4 + g * d * 4)


def decode_bytes(T: int, B: int, Hq: int, Hkv: int, d: int, G: int, R: int, P: int) -> int:
    return B * Hkv * decode_bytes_per_unit(T, d, Hq // Hkv, G, R, P)


def hot_bytes(T: int, B: int, Hq: int, Hkv: int, d: int, G: int, R: int, P: int) -> int:
    """Bytes of one decode call outside the quantized blocks and the cold
    pool: residual and pool tokens (fp16 K and V), the query and the output."""
    nf = flush_count(T, G, R)
    npool = pool_size(T, G, R, P)
    return B * Hkv * ((T - nf * G + npool) * d * 4 + (Hq // Hkv) * d * 4)


def cold_unit_bytes(bcount, ncold: int, d: int) -> int:
    """Cold-pool policy: bytes of one unit's quantized blocks (sizes bcount,
    read from the device) and of its ncold fp16 cold-pool tokens."""
    nq = int(sum(int(n) for n in bcount))
    nonempty = sum(1 for n in bcount if n > 0)
    return 2 * nq * d // 4 + nonempty * d * 4 + nq * (d // 32) * 4 + int(ncold) * d * 4


def topk_bytes_per_unit(T: int, d: int, g: int, G: int, R: int, P: int, K: int) -> int:
    """Top-K sparse decode of one unit: the bound pass reads every non-empty
    block's K scale/zero header and the queries; the decode reads the K
    selected blocks, the residual and pool tokens, the queries, and writes the
    output. Which blocks are selected depends on the data; they are counted
    as the K smallest non-empty blocks, so this is a lower bound."""
    nf = flush_count(T, G, R)
    npool = pool_size(T, G, R, P)
    sizes = sorted(n for n in (block_count(j, G, P) for j in range(nf)) if n > 0)
    kc = min(K, len(sizes))
    nq = sum(sizes[:kc])
    bound_pass = len(sizes) * d * 4 + g * d * 2
    return (bound_pass + 2 * nq * d // 4 + kc * d * 4 + nq * (d // 32) * 4
            + (T - nf * G + npool) * d * 4 + g * d * 4)


def topk_bytes(T: int, B: int, Hq: int, Hkv: int, d: int, G: int, R: int, P: int, K: int) -> int:
    return B * Hkv * topk_bytes_per_unit(T, d, Hq // Hkv, G, R, P, K)


def fp16_cache_bytes(T: int, B: int, Hkv: int, d: int) -> int:
    """The same cache held entirely in fp16 (K and V)."""
    return B * Hkv * T * d * 4


def block_bytes(d: int, G: int) -> int:
    """One packed block as stored: K scale/zero per channel (4d), then per 16
    token slots the K and V codes and the V scale/zero (10d)."""
    return 4 * d + -(-G // 16) * 10 * d


def flush_bytes_per_unit(j: int, d: int, G: int, P: int) -> int:
    """Algorithmic bytes of flush j of one (sequence, kv head) unit: read the
    group's G fp16 tokens and the pool's tokens (K and V, 4d each) with the
    pool's norms and indices (8 each); write the packed block, its G token
    indices, and the new pool (tokens, norms, indices)."""
    np0, np1 = min(P, j * G), min(P, (j + 1) * G)
    return G * 4 * d + np0 * (4 * d + 8) + block_bytes(d, G) + 4 * G + np1 * (4 * d + 8)


def prefill_bytes_per_unit(L: int, d: int, G: int, R: int, P: int) -> int:
    """Algorithmic bytes of a prefill of L tokens into one empty unit: read
    every token once (K and V); write the nf packed blocks with their token
    indices, the final pool (tokens, norms, indices) and the fp16 residual."""
    nf = flush_count(L, G, R)
    return (L * 4 * d + nf * (block_bytes(d, G) + 4 * G) + pool_size(L, G, R, P) * (4 * d + 8)
            + (L - nf * G) * 4 * d)
