"""Python handle on the plain-C OTT oracle (``ott_oracle.c``).

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
leg of the benchmark import this module. It never touches the CUDA library.

The C file follows "Accurate KV Cache Quantization with Outlier Tokens
Tracing" (zijie-tian.site, sec. 3.1-3.3 and the flowchart; sciencestack.ai,
TL;DR, Abstract, Fig. 1(c), Fig. 2). Its header lists the readings taken
where those pages are silent.

Arrays cross the boundary as numpy arrays: fp16 values travel as their raw
``uint16`` bit patterns so that nothing rounds on the way.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ott_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
# No contraction of a*b+c into fused multiply-adds and no fast-math: the
# fp32 decisions (norms, scales, codes) must be the plain IEEE operations.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            i32, i64, u16 = C.c_int, C.c_longlong, C.c_uint16
            L.orc_create.restype = P
            L.orc_create.argtypes = [i32] * 7
            L.orc_create_policy.restype = P
            L.orc_create_policy.argtypes = [i32] * 8
            L.orc_create_pct.restype = P
            L.orc_create_pct.argtypes = [i32] * 9
            L.orc_export_cold.argtypes = [P, i32, P, P, P]
            L.orc_topk_select.argtypes = [P, i32, i32, P, i32, P, P]
            L.orc_release_seq.argtypes = [P, i32]
            L.orc_prefill_seq.argtypes = [P, i32, P, P, i32]
            L.orc_decode_topk.argtypes = [P, P, i32, P]
            L.orc_destroy.argtypes = [P]
            L.orc_append.argtypes = [P, P, P]
            L.orc_prefill.argtypes = [P, P, P, i32]
            L.orc_prefill_lens.argtypes = [P, P, P, P, i32]
            L.orc_decode.argtypes = [P, P, P]
            L.orc_decode_head.argtypes = [P, i32, i32, P, P]
            L.orc_counts.argtypes = [P, i32, P, P, P, P]
            L.orc_block_count.argtypes = [P, i32, i32]
            L.orc_export_unit.argtypes = [P, i32] + [P] * 15
            L.orc_h2f.restype = C.c_float
            L.orc_h2f.argtypes = [u16]
            L.orc_f2h.restype = u16
            L.orc_f2h.argtypes = [C.c_float]
            L.orc_f2h_array.argtypes = [P, P, i64]
            L.orc_h2f_array.argtypes = [P, P, i64]
            L.orc_norm.restype = C.c_float
            L.orc_norm.argtypes = [P, i32]
            L.orc_quant_group.argtypes = [P, i32, i32, P, P, P, i32]
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _bits(a) -> np.ndarray:
    """fp16 data (numpy float16/uint16 or a CPU torch tensor) -> contiguous uint16 bits."""
    if hasattr(a, "numpy"):  # torch tensor
        a = a.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected fp16 data, got {a.dtype}")
    return a


# ---------------------------------------------------------------- primitives

def f2h(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 bits, round to nearest even (the oracle's own routine)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f2h_array(_ptr(x), _ptr(out), x.size)
    return out


def h2f(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_h2f_array(_ptr(h), _ptr(out), h.size)
    return out


def norm(k) -> float:
    """Squared L2 norm of one fp16 key, fp32, summed in channel order."""
    kb = _bits(k)
    return float(lib().orc_norm(_ptr(kb), kb.size))


def quant_group(x) -> tuple[int, int, np.ndarray]:
    """2-bit asymmetric quantization of one group: (scale bits, zero bits, codes)."""
    xb = _bits(x).ravel()
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(max(xb.size, 1), np.uint8)
    lib().orc_quant_group(_ptr(xb), xb.size, 1, _ptr(s), _ptr(z), _ptr(codes), 1)
    return int(s[0]), int(z[0]), codes[: xb.size]


# ---------------------------------------------------------------- the cache

class OracleCache:
    """The oracle's OTT cache: same create/prefill/append/decode calls as the library.

    ``cold=None`` writes displaced pool tokens back into the new block;
    ``cold=C`` (an int >= 0) is the cold-pool policy with capacity C.
    ``pct=(p, n_oc)`` selects the channel-conditioned outlier criterion: p in
    units of 1/10000, n_oc outlier channels per flush (written back)."""

    def __init__(self, B, Hq, Hkv, d, G, R, P, cold=None, pct=None):
        self.B, self.Hq, self.Hkv, self.d, self.G, self.R, self.P = B, Hq, Hkv, d, G, R, P
        self.cold = cold
        self.pct = pct
        if pct is not None:
            if cold is not None:
                raise ValueError("the criterion and the cold-pool policy do not combine")
            self._h = lib().orc_create_pct(B, Hq, Hkv, d, G, R, P, int(pct[0]), int(pct[1]))
        else:
            self._h = lib().orc_create_policy(B, Hq, Hkv, d, G, R, P, -1 if cold is None else int(cold))
        if not self._h:
            raise ValueError("invalid OTT shape")

    def close(self):
        if self._h:
            lib().orc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, K, V):
        """K, V: fp16 [B][Hkv][L][d]."""
        Kb, Vb = _bits(K), _bits(V)
        L = Kb.shape[2]
        rc = lib().orc_prefill(self._h, _ptr(Kb), _ptr(Vb), L)
        if rc:
            raise RuntimeError("prefill on a non-empty oracle cache")

    def prefill_lens(self, K, V, lens):
        """Ragged prefill: K, V fp16 [B][Hkv][Lmax][d]; sequence b takes its
        first lens[b] tokens."""
        Kb, Vb = _bits(K), _bits(V)
        Lmax = Kb.shape[2]
        ln = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
        if ln.shape != (self.B,):
            raise ValueError("lens must hold one length per sequence")
        rc = lib().orc_prefill_lens(self._h, _ptr(Kb), _ptr(Vb), _ptr(ln), Lmax)
        if rc:
            raise RuntimeError("ragged prefill rejected (non-empty cache or bad lengths)")

    def append(self, k, v):
        """k, v: fp16 [B][Hkv][d]."""
        kb, vb = _bits(k), _bits(v)
        if lib().orc_append(self._h, _ptr(kb), _ptr(vb)):
            raise RuntimeError("append while a sequence is empty")

    def release_seq(self, b: int):
        """Sequence b drops every token; it must be refilled before the next append or decode."""
        if lib().orc_release_seq(self._h, int(b)):
            raise ValueError("bad sequence index")

    def prefill_seq(self, b: int, K, V):
        """Fill the empty sequence b: K, V fp16 [Hkv][L][d]."""
        Kb, Vb = _bits(K), _bits(V)
        rc = lib().orc_prefill_seq(self._h, int(b), _ptr(Kb), _ptr(Vb), Kb.shape[1])
        if rc:
            raise RuntimeError("prefill_seq rejected (sequence not empty or bad length)")

    def decode(self, q) -> np.ndarray:
        """q: fp16 [B][Hq][d] -> float64 [B][Hq][d]."""
        qb = _bits(q)
        out = np.zeros(qb.shape, np.float64)
        if lib().orc_decode(self._h, _ptr(qb), _ptr(out)):
            raise RuntimeError("decode on an empty oracle cache")
        return out

    def decode_topk(self, q, K: int) -> np.ndarray:
        """Top-K sparse decode: q fp16 [B][Hq][d] -> float64 [B][Hq][d]; each
        (sequence, kv head) attends its K best-bounded quantized blocks."""
        qb = _bits(q)
        out = np.zeros(qb.shape, np.float64)
        if lib().orc_decode_topk(self._h, _ptr(qb), int(K), _ptr(out)):
            raise RuntimeError("decode on an empty oracle cache")
        return out

    def topk_select(self, q, K: int):
        """The blocks a top-K decode attends: (sel int32 [B*Hkv][K] ascending,
        -1 padded; bounds float32 [B*Hkv][nf], -inf for empty blocks)."""
        qb = _bits(q)
        U = self.B * self.Hkv
        nf = max(self.counts(u)[1] for u in range(U))   # units may differ (ragged batches)
        sel = np.full((U, max(K, 1)), -1, np.int32)
        bounds = np.full((U, max(nf, 1)), -np.inf, np.float32)
        for u in range(U):
            b, hk = divmod(u, self.Hkv)
            row = np.zeros(max(nf, 1), np.int32)
            qrow = np.ascontiguousarray(qb[b])
            brow = np.full(max(nf, 1), -np.inf, np.float32)
            m = lib().orc_topk_select(self._h, b, hk, _ptr(qrow), int(K), _ptr(row), _ptr(brow))
            sel[u, :m] = row[:m]
            bounds[u] = brow
        return sel[:, :K], bounds[:, :nf]

    def decode_head(self, b, hq, qv) -> np.ndarray:
        """One query head: qv fp16 [d] -> float64 [d]."""
        qb = _bits(qv)
        out = np.zeros(self.d, np.float64)
        if lib().orc_decode_head(self._h, b, hq, _ptr(qb), _ptr(out)):
            raise RuntimeError("bad decode_head arguments")
        return out

    def counts(self, u: int = 0):
        T, nf, tail, npool = (C.c_longlong(), C.c_int(), C.c_int(), C.c_int())
        lib().orc_counts(self._h, u, C.byref(T), C.byref(nf), C.byref(tail), C.byref(npool))
        return T.value, nf.value, tail.value, npool.value

    def export_unit(self, u: int) -> dict:
        """Canonical state of unit u = b*Hkv + hkv (see ``orc_export_unit``)."""
        T, nf, nt, npool = self.counts(u)
        G, P, d = self.G, self.P, self.d
        e = dict(
            bcount=np.zeros(nf, np.int32),
            bidx=np.zeros((nf, G), np.int32),
            kcode=np.zeros((nf, G, d // 4), np.uint8),
            ks=np.zeros((nf, d), np.uint16),
            kz=np.zeros((nf, d), np.uint16),
            vcode=np.zeros((nf, G, d // 4), np.uint8),
            vs=np.zeros((nf, G, d // 32), np.uint16),
            vz=np.zeros((nf, G, d // 32), np.uint16),
            tidx=np.zeros(nt, np.int32),
            tk=np.zeros((nt, d), np.uint16),
            tv=np.zeros((nt, d), np.uint16),
            pidx=np.zeros(P, np.int32),
            pnorm=np.zeros(P, np.uint32),
            pk=np.zeros((P, d), np.uint16),
            pv=np.zeros((P, d), np.uint16),
        )
        order = ["bcount", "bidx", "kcode", "ks", "kz", "vcode", "vs", "vz",
                 "tidx", "tk", "tv", "pidx", "pnorm", "pk", "pv"]
        # zero-size arrays still need a valid pointer
        ptrs = [_ptr(e[k]) if e[k].size else None for k in order]
        lib().orc_export_unit(self._h, u, *ptrs)
        e.update(T=T, nf=nf, tail=nt, npool=npool)
        if self.cold is not None:
            Cc = int(self.cold)
            cidx = np.zeros(max(Cc, 1), np.int32)
            ck = np.zeros((max(Cc, 1), d), np.uint16)
            cv = np.zeros((max(Cc, 1), d), np.uint16)
            n = lib().orc_export_cold(self._h, u, _ptr(cidx), _ptr(ck), _ptr(cv))
            e.update(ncold=n, cidx=cidx[:Cc], ck=ck[:Cc], cv=cv[:Cc])
        return e
