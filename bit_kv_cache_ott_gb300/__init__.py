"""bit_kv_cache_ott_gb300 -- Outlier Tokens Tracing (OTT) KV-cache quantization
on one GB300 GPU.

A thin ctypes binding over ``libott.so`` (C ABI in ``include/ott.h``): it only
marshals torch tensors into device pointers and streams. Every step of the
path (append, flush, prefill, decode attention) runs in the library's CUDA
kernels. There is no CPU fallback: if the library is missing or cannot load,
``load()`` raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import synth  # noqa: F401  (seeded workloads)

__all__ = ["OTTCache", "OTTError", "load", "status_str", "lib_path", "hbm_copy"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libott.so")
_lib = None

OTT_OK, OTT_ERR_INVALID, OTT_ERR_STATE, OTT_ERR_CAPACITY = 0, -1, -2, -3
OTT_ERR_OOM, OTT_ERR_CUDA, OTT_ERR_DEVICE = -4, -5, -6


class OTTError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_str(code)} ({code})")
        self.code = code


class StateExport(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("bidx", "kcode", "ks", "kz", "vcode", "vs", "vz", "tk", "tv", "pidx", "pnorm", "pk", "pv")]


SYMBOLS = ("ott_create", "ott_create_ragged", "ott_create_paged", "ott_release_seq", "ott_prefill_seq",
           "ott_free_blocks", "ott_create_cold", "ott_create_pct", "ott_export_cold", "ott_destroy", "ott_prefill", "ott_prefill_lens", "ott_append", "ott_step_host",
           "ott_decode_attn", "ott_decode_attn_static", "ott_decode_attn_topk", "ott_get_counts", "ott_get_seq_counts", "ott_block_count",
           "ott_export_state", "ott_check_device", "ott_device_bytes", "ott_status_str", "ott_hbm_copy", "ott_ex2_probe")


def lib_path() -> str:
    return _LIB_PATH


def load(build_if_missing: bool = False):
    """Load libott.so (raises if it is absent or broken)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        if not build_if_missing:
            raise RuntimeError(f"libott.so not built ({_LIB_PATH}); run __graft_entry__.build()")
        from .build import build
        build()
    L = C.CDLL(_LIB_PATH)
    P, i32, i64 = C.c_void_p, C.c_int, C.c_longlong
    L.ott_create.argtypes = [i32] * 8 + [C.POINTER(P)]
    L.ott_create_ragged.argtypes = [i32] * 8 + [C.POINTER(P)]
    L.ott_create_cold.argtypes = [i32] * 9 + [C.POINTER(P)]
    L.ott_create_pct.argtypes = [i32] * 10 + [C.POINTER(P)]
    L.ott_create_paged.argtypes = [i32] * 8 + [i64, C.POINTER(P)]
    L.ott_release_seq.argtypes = [P, i32, P]
    L.ott_prefill_seq.argtypes = [P, i32, P, P, i32, P]
    L.ott_free_blocks.argtypes = [P]
    L.ott_free_blocks.restype = i64
    L.ott_export_cold.argtypes = [P, i32, i32, P, P, P, P, P]
    L.ott_destroy.argtypes = [P]
    L.ott_prefill.argtypes = [P, P, P, i32, P]
    L.ott_prefill_lens.argtypes = [P, P, P, C.POINTER(i32), i32, P]
    L.ott_append.argtypes = [P, P, P, P]
    L.ott_step_host.argtypes = [P, P, P, P, P, i32, P]
    L.ott_decode_attn.argtypes = [P, P, P, P]
    L.ott_decode_attn_static.argtypes = [P, P, P, P]
    L.ott_decode_attn_topk.argtypes = [P, P, P, i32, P, P]
    L.ott_get_counts.argtypes = [P, C.POINTER(i64), C.POINTER(i32), C.POINTER(i32), C.POINTER(i32)]
    L.ott_get_seq_counts.argtypes = [P, i32, C.POINTER(i64), C.POINTER(i32), C.POINTER(i32), C.POINTER(i32)]
    L.ott_block_count.argtypes = [P, i32]
    L.ott_export_state.argtypes = [P, i32, i32, C.POINTER(StateExport)]
    L.ott_check_device.argtypes = [P]
    L.ott_device_bytes.argtypes = [P]
    L.ott_device_bytes.restype = i64
    L.ott_status_str.argtypes = [i32]
    L.ott_status_str.restype = C.c_char_p
    L.ott_hbm_copy.argtypes = [P, P, i64, P]
    L.ott_ex2_probe.argtypes = [P, P, i32, P]
    _lib = L
    return L


def status_str(code: int) -> str:
    return load().ott_status_str(code).decode()


def hbm_copy(dst: torch.Tensor, src: torch.Tensor, stream=None):
    """Copy src into dst (same byte size, CUDA tensors) with the library's
    streaming copy kernel: the bandwidth probe that times HBM in the same run
    as the decode."""
    if not (dst.is_cuda and src.is_cuda and dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("hbm_copy: contiguous CUDA tensors")
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("hbm_copy: sizes differ")
    _check(load().ott_hbm_copy(dst.data_ptr(), src.data_ptr(), n, _stream(stream)), "ott_hbm_copy")


def _check(rc: int, what: str):
    if rc != OTT_OK:
        raise OTTError(rc, what)


def _dev_ptr(t: torch.Tensor, shape, name) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float16:
        raise TypeError(f"{name}: expected a CUDA float16 tensor")
    if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class OTTCache:
    """One OTT cache (one attention layer): ``create/prefill/append/decode_attn/destroy``.
    ``ragged=True`` creates it with ``ott_create_ragged`` so that ``prefill_lens``
    can give every sequence its own length. ``cold=C`` creates it with
    ``ott_create_cold``: displaced pool tokens go to a first-in-first-out
    fp16 cold pool of C slots instead of the new block. ``pct=(p, n_oc)``
    creates it with ``ott_create_pct``: the channel-conditioned outlier
    criterion, p in units of 1/10000 over n_oc outlier channels."""

    def __init__(self, B, Hq, Hkv, d, G=128, R=32, P=32, max_tokens=8192, ragged=False, cold=None,
                 pool_blocks=None, pct=None):
        L = load()
        self.B, self.Hq, self.Hkv, self.d, self.G, self.R, self.P = B, Hq, Hkv, d, G, R, P
        self.max_tokens = max_tokens
        self.ragged = ragged
        self.cold = cold
        h = C.c_void_p()
        if pool_blocks is not None:
            self.ragged = True
            _check(L.ott_create_paged(B, Hq, Hkv, d, G, R, P, max_tokens, int(pool_blocks), C.byref(h)),
                   "ott_create_paged")
        elif pct is not None:
            if ragged or cold is not None:
                raise ValueError("the channel criterion takes sequences of one length and writes tokens back")
            _check(L.ott_create_pct(B, Hq, Hkv, d, G, R, P, int(pct[0]), int(pct[1]), max_tokens, C.byref(h)),
                   "ott_create_pct")
        elif cold is not None:
            if ragged:
                raise ValueError("the cold-pool policy takes sequences of one length")
            _check(L.ott_create_cold(B, Hq, Hkv, d, G, R, P, int(cold), max_tokens, C.byref(h)), "ott_create_cold")
        else:
            create = L.ott_create_ragged if ragged else L.ott_create
            _check(create(B, Hq, Hkv, d, G, R, P, max_tokens, C.byref(h)),
                   "ott_create_ragged" if ragged else "ott_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            load().ott_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def handle(self) -> int:
        return self._h.value

    def prefill(self, K: torch.Tensor, V: torch.Tensor, stream=None):
        Lq = K.shape[2] if K.dim() == 4 else -1
        shp = (self.B, self.Hkv, Lq, self.d)
        _check(load().ott_prefill(self._h, _dev_ptr(K, shp, "K"), _dev_ptr(V, shp, "V"), Lq,
                                  _stream(stream)), "ott_prefill")

    def prefill_lens(self, K: torch.Tensor, V: torch.Tensor, lens, stream=None):
        """Ragged prefill: K, V [B][Hkv][Lmax][d]; sequence b takes its first lens[b] tokens."""
        Lmax = K.shape[2] if K.dim() == 4 else -1
        shp = (self.B, self.Hkv, Lmax, self.d)
        ln = (C.c_int * self.B)(*[int(x) for x in lens])
        if len(lens) != self.B:
            raise ValueError("lens must hold one length per sequence")
        _check(load().ott_prefill_lens(self._h, _dev_ptr(K, shp, "K"), _dev_ptr(V, shp, "V"), ln, Lmax,
                                       _stream(stream)), "ott_prefill_lens")

    def append(self, k: torch.Tensor, v: torch.Tensor, stream=None):
        shp = (self.B, self.Hkv, self.d)
        _check(load().ott_append(self._h, _dev_ptr(k, shp, "k"), _dev_ptr(v, shp, "v"),
                                 _stream(stream)), "ott_append")

    def step_host(self, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, out: torch.Tensor, topk: int = 0,
                  stream=None):
        """One step from pinned host memory: append k, v (fp16 [B][Hkv][d]) and
        decode q (fp16 [B][Hq][d]) into out (fp16 [B][Hq][d]), all pinned CPU
        tensors; the kernels read and write them in place (ott_step_host).
        topk >= 1 decodes with Top-K sparse access over that many blocks.
        out is complete when the stream has passed the step."""
        for name, t, shp in (("k", k, (self.B, self.Hkv, self.d)), ("v", v, (self.B, self.Hkv, self.d)),
                             ("q", q, (self.B, self.Hq, self.d)), ("out", out, (self.B, self.Hq, self.d))):
            if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.float16 or not t.is_pinned():
                raise TypeError(f"{name}: expected a pinned CPU float16 tensor")
            if tuple(t.shape) != shp or not t.is_contiguous():
                raise ValueError(f"{name}: expected contiguous shape {shp}, got {tuple(t.shape)}")
        _check(load().ott_step_host(self._h, k.data_ptr(), v.data_ptr(), q.data_ptr(), out.data_ptr(), int(topk),
                                    _stream(stream)), "ott_step_host")

    def decode_attn(self, q: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        shp = (self.B, self.Hq, self.d)
        if out is None:
            out = torch.empty(shp, dtype=torch.float16, device=q.device)
        _check(load().ott_decode_attn(self._h, _dev_ptr(q, shp, "q"), _dev_ptr(out, shp, "out"),
                                      _stream(stream)), "ott_decode_attn")
        return out

    def decode_attn_topk(self, q: torch.Tensor, K: int, out: torch.Tensor | None = None,
                         sel: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Top-K sparse decode: each (sequence, kv head) attends its K blocks
        with the largest score bound plus all fp16 tokens. ``sel``, if given,
        is a CUDA int32 tensor [B*Hkv][min(K, nf)] that receives the blocks
        (nf: the largest block count of any sequence)."""
        shp = (self.B, self.Hq, self.d)
        if out is None:
            out = torch.empty(shp, dtype=torch.float16, device=q.device)
        sp = None
        if sel is not None:
            nf = max(self.seq_counts(b)[1] for b in range(self.B)) if self.ragged else self.counts()[1]
            kc = min(int(K), nf)
            if (not sel.is_cuda or sel.dtype != torch.int32 or not sel.is_contiguous()
                    or tuple(sel.shape) != (self.B * self.Hkv, kc)):
                raise ValueError(f"sel: expected a contiguous CUDA int32 tensor {(self.B * self.Hkv, kc)}")
            sp = sel.data_ptr()
        _check(load().ott_decode_attn_topk(self._h, _dev_ptr(q, shp, "q"), _dev_ptr(out, shp, "out"), int(K), sp,
                                           _stream(stream)), "ott_decode_attn_topk")
        return out

    def counts(self):
        T, nf, tail, npool = C.c_longlong(), C.c_int(), C.c_int(), C.c_int()
        _check(load().ott_get_counts(self._h, C.byref(T), C.byref(nf), C.byref(tail), C.byref(npool)),
               "ott_get_counts")
        return T.value, nf.value, tail.value, npool.value

    def seq_counts(self, b: int):
        T, nf, tail, npool = C.c_longlong(), C.c_int(), C.c_int(), C.c_int()
        _check(load().ott_get_seq_counts(self._h, b, C.byref(T), C.byref(nf), C.byref(tail), C.byref(npool)),
               "ott_get_seq_counts")
        return T.value, nf.value, tail.value, npool.value

    def release_seq(self, b: int, stream=None):
        """Sequence b finishes: it drops its tokens (and its pool blocks)."""
        _check(load().ott_release_seq(self._h, int(b), _stream(stream)), "ott_release_seq")

    def prefill_seq(self, b: int, K: torch.Tensor, V: torch.Tensor, stream=None):
        """Fill the empty sequence b with a prompt: K, V fp16 [Hkv][L][d] on the device."""
        L = K.shape[1] if K.dim() == 3 else -1
        shp = (self.Hkv, L, self.d)
        _check(load().ott_prefill_seq(self._h, int(b), _dev_ptr(K, shp, "K"), _dev_ptr(V, shp, "V"), L,
                                      _stream(stream)), "ott_prefill_seq")

    def free_blocks(self) -> int:
        """Free blocks of the paged pool (-1 without one)."""
        return int(load().ott_free_blocks(self._h))

    def cold_sizes(self):
        """Cold-pool policy: (block sizes [U][nf], cold-pool sizes [U]) from the device."""
        import numpy as np
        U, nf = self.B * self.Hkv, self.counts()[1]
        bc = np.zeros((U, max(nf, 1)), np.int32)
        nc = np.zeros(U, np.int32)
        _check(load().ott_export_cold(self._h, 0, U, bc.ctypes.data, nc.ctypes.data, None, None, None),
               "ott_export_cold")
        return bc[:, :nf], nc

    def block_count(self, j: int) -> int:
        rc = load().ott_block_count(self._h, j)
        if rc < 0:
            raise OTTError(rc, "ott_block_count")
        return rc

    def device_bytes(self) -> int:
        return int(load().ott_device_bytes(self._h))

    def check_device(self):
        _check(load().ott_check_device(self._h), "ott_check_device")

    def export_state(self, u0: int = 0, nu: int | None = None) -> dict:
        """Canonical host arrays of units [u0, u0+nu) (numpy). In a ragged
        batch the units must belong to one sequence."""
        import numpy as np
        nu = self.B * self.Hkv - u0 if nu is None else nu
        T, nf, nt, npool = self.seq_counts(u0 // self.Hkv)
        G, P, d = self.G, self.P, self.d
        e = dict(
            bidx=np.zeros((nu, nf, G), np.int32),
            kcode=np.zeros((nu, nf, G, d // 4), np.uint8),
            ks=np.zeros((nu, nf, d), np.uint16), kz=np.zeros((nu, nf, d), np.uint16),
            vcode=np.zeros((nu, nf, G, d // 4), np.uint8),
            vs=np.zeros((nu, nf, G, d // 32), np.uint16), vz=np.zeros((nu, nf, G, d // 32), np.uint16),
            tk=np.zeros((nu, nt, d), np.uint16), tv=np.zeros((nu, nt, d), np.uint16),
            pidx=np.zeros((nu, P), np.int32), pnorm=np.zeros((nu, P), np.uint32),
            pk=np.zeros((nu, P, d), np.uint16), pv=np.zeros((nu, P, d), np.uint16),
        )
        st = StateExport(**{k: (v.ctypes.data if v.size else None) for k, v in e.items()})
        _check(load().ott_export_state(self._h, u0, nu, C.byref(st)), "ott_export_state")
        if self.cold is None:
            e["bcount"] = np.array([self.block_count(j) for j in range(nf)], np.int32)
        else:
            Cc = int(self.cold)
            bc = np.zeros((nu, max(nf, 1)), np.int32)
            nc = np.zeros(nu, np.int32)
            ci = np.zeros((nu, max(Cc, 1)), np.int32)
            ck = np.zeros((nu, max(Cc, 1), d), np.uint16)
            cv = np.zeros((nu, max(Cc, 1), d), np.uint16)
            _check(load().ott_export_cold(self._h, u0, nu, bc.ctypes.data, nc.ctypes.data, ci.ctypes.data,
                                          ck.ctypes.data, cv.ctypes.data), "ott_export_cold")
            e.update(bcount=bc[:, :nf], ncold=nc, cidx=ci[:, :Cc], ck=ck[:, :Cc], cv=cv[:, :Cc])
        e.update(T=T, nf=nf, tail=nt, npool=npool)
        return e
