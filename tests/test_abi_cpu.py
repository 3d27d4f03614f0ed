"""The C ABI library loads without a GPU and exports every symbol that
include/ott.h declares; host-only paths (status strings, NULL handles) work.
No compute call is made here.
"""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ott.h")


@pytest.fixture(scope="module")
def libott():
    from bit_kv_cache_ott_gb300 import build
    path = build.build()
    return C.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ott_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("ott_create", "ott_prefill", "ott_append", "ott_decode_attn", "ott_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(libott):
    missing = [n for n in declared_functions() if not hasattr(libott, n)]
    assert not missing, missing


def test_binding_lists_every_symbol():
    import bit_kv_cache_ott_gb300 as pkg
    assert set(declared_functions()) <= set(pkg.SYMBOLS)


def test_status_strings_and_null_handles(libott):
    libott.ott_status_str.restype = C.c_char_p
    assert libott.ott_status_str(0) == b"ok"
    assert b"capacity" in libott.ott_status_str(-3)
    assert libott.ott_status_str(12345) == b"unknown status"
    assert libott.ott_destroy(None) == 0
    assert libott.ott_prefill(None, None, None, 0, None) == -1
    assert libott.ott_append(None, None, None, None) == -1
    assert libott.ott_decode_attn(None, None, None, None) == -1
    assert libott.ott_get_counts(None, None, None, None, None) == -1
    assert libott.ott_export_state(None, 0, 0, None) == -1
    assert libott.ott_check_device(None) == -1
    out = C.c_void_p(123)
    assert libott.ott_create(1, 1, 1, 128, 128, 32, 32, 100, None) == -1
    # unsupported shapes are rejected before any device call
    assert libott.ott_create(1, 3, 2, 128, 128, 32, 32, 100, C.byref(out)) == -1   # Hq % Hkv != 0
    assert out.value is None
    assert libott.ott_create(1, 1, 1, 96, 128, 32, 32, 100, C.byref(out)) == -1    # d = 96
    assert libott.ott_create(1, 2, 4, 128, 128, 32, 32, 100, C.byref(out)) == -1   # Hq < Hkv
    assert libott.ott_create(1, 1, 1, 128, 0, 32, 32, 100, C.byref(out)) == -1     # G = 0


def test_decode_bytes_formula():
    """The closed-form byte count against a direct per-block sum, and the
    hand-computed figure per unit at T = 4096, G = 128, R = 32, P = 32, d = 128:
    3936 quantized tokens x 80 B (codes and value scale/zero) + 31 blocks x
    512 B (key scale/zero) + 160 fp16 tokens x 512 B + 512 B (query, output)
    = 413,184 B."""
    from bit_kv_cache_ott_gb300 import metrics
    assert metrics.decode_bytes_per_unit(4096, 128, 1, 128, 32, 32) == 413184
    for T, G, R, P in [(300, 16, 4, 40), (1000, 32, 0, 200), (77, 8, 3, 0), (5000, 128, 32, 64)]:
        nf = metrics.flush_count(T, G, R)
        npool = metrics.pool_size(T, G, R, P)
        nq = nf * G - npool
        nonempty = sum(1 for j in range(nf) if metrics.block_count(j, G, P) > 0)
        direct = (nq * 128 // 4) * 2 + nonempty * 128 * 4 + nq * 4 * 4 + (T - nf * G + npool) * 128 * 4 + 128 * 4
        assert metrics.decode_bytes_per_unit(T, 128, 1, G, R, P) == direct
