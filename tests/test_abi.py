"""CPU-side checks of the C ABI: the library builds, loads, exports every
declared symbol, and rejects bad arguments on the host before launching.

No call here reaches a kernel: each one either fails validation or has an
empty problem (m == 0 or n == 0), which the ABI defines as a no-op.
"""

import ctypes
import glob
import os
import re

import pytest

from int8_hadamard_rotated_convrot_gb300 import build as cbuild
from int8_hadamard_rotated_convrot_gb300 import convrot as cr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced on these paths


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cr.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(convrot_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(cr.EXPORTED) <= set(names) | {"convrot_status_string"}
    for name in names:
        assert hasattr(lib, name), name
    # and the binding knows about all of them
    assert set(names) <= set(cr.EXPORTED) | set(getattr(cr, "EXPORTED_EXTRA", []))


def test_ldq(lib):
    assert lib.convrot_ldq(1) == 128
    assert lib.convrot_ldq(128) == 128
    assert lib.convrot_ldq(129) == 256
    assert lib.convrot_ldq(3072) == 3072
    assert lib.convrot_ldq(0) == 0


def test_status_strings(lib):
    for s in range(8):
        assert len(cr.status_string(s)) > 0
    assert cr.status_string(999) == "unknown status"


def packed(q=FAKE, scale=FAKE, ldq=128, codes=cr.CODES_I8, rows=0, k=0, G=0):
    return cr._Packed(q, scale, rows, k, ldq, G, codes)


def pack(lib, X=FAKE, m=4, k=256, ldx=256, G=256, out=None):
    out = out or packed(ldq=cr.convrot_ldq(k) if k > 0 else 128)
    return lib.convrot_pack_activations(X, m, k, ldx, G, ctypes.byref(out), None, None)


@pytest.mark.parametrize("G", [1, 2, 8, 32, 128, 0, -4, 16384])
def test_pack_rejects_bad_group(lib, G):
    assert pack(lib, G=G) == cr.ERR_GROUP_SIZE


def test_group_size_limits(lib):
    """4^8 = 65536 is the largest power of four dividing a k within the range; 4^9 is rejected."""
    assert pack(lib, k=131072, ldx=131072, G=65536, out=packed(ldq=131072)) != cr.ERR_GROUP_SIZE
    assert pack(lib, k=131072, ldx=131072, G=16384, out=packed(ldq=131072)) != cr.ERR_GROUP_SIZE
    assert pack(lib, k=131072, ldx=131072, G=262144, out=packed(ldq=131072)) == cr.ERR_GROUP_SIZE


def test_pack_rejects_group_not_dividing_k(lib):
    assert pack(lib, k=96, ldx=96, G=64) == cr.ERR_GROUP_SIZE


@pytest.mark.parametrize("k", [0, -1, 133148])
def test_pack_rejects_k_range(lib, k):
    assert pack(lib, k=k, ldx=max(k, 4), G=4) == cr.ERR_K_RANGE


def test_pack_rejects_bad_pointers_and_lds(lib):
    assert pack(lib, X=None) == cr.ERR_INVALID_ARG
    assert pack(lib, X=FAKE + 4) == cr.ERR_ALIGNMENT
    assert pack(lib, ldx=255) == cr.ERR_INVALID_ARG
    assert pack(lib, k=256, ldx=258) == cr.ERR_ALIGNMENT
    assert pack(lib, m=-1) == cr.ERR_INVALID_ARG
    assert lib.convrot_pack_activations(FAKE, 4, 256, 256, 256, None, None, None) == cr.ERR_INVALID_ARG
    assert pack(lib, out=packed(q=None)) == cr.ERR_INVALID_ARG
    assert pack(lib, out=packed(scale=None)) == cr.ERR_INVALID_ARG
    assert pack(lib, out=packed(q=FAKE + 8, ldq=256)) == cr.ERR_ALIGNMENT
    assert pack(lib, out=packed(ldq=128)) == cr.ERR_INVALID_ARG  # ldq < convrot_ldq(256)
    assert pack(lib, out=packed(ldq=264)) == cr.ERR_ALIGNMENT
    assert pack(lib, out=packed(codes=2, ldq=256)) == cr.ERR_INVALID_ARG


def test_pack_empty_is_noop_and_fills_shape(lib):
    out = packed(q=None, scale=None, ldq=256)
    assert lib.convrot_pack_activations(None, 0, 256, 256, 64, ctypes.byref(out), None, None) == cr.OK
    assert (out.rows, out.k, out.group_size) == (0, 256, 64)
    out = packed(q=None, scale=None, ldq=256)
    assert lib.convrot_quantize_weights(None, 0, 192, 192, 64, ctypes.byref(out), None, None) == cr.OK


def pair(mx=4, nw=4, k=256, G=256, codes=cr.CODES_I8):
    ld = cr.convrot_ldq(k)
    return (packed(rows=mx, k=k, G=G, ldq=ld, codes=codes), packed(rows=nw, k=k, G=G, ldq=ld, codes=codes))


def linear(lib, x, w, Y=FAKE, ldy=64, bias=None, status=None):
    return lib.convrot_linear(ctypes.byref(x), ctypes.byref(w), bias, Y, ldy, status, None)


def test_linear_rejects_mismatches(lib):
    x, w = pair()
    w.k = 512
    assert linear(lib, x, w) == cr.ERR_INVALID_ARG
    x, w = pair()
    w.group_size = 64
    assert linear(lib, x, w) == cr.ERR_GROUP_SIZE
    x, w = pair()
    w.codes = cr.CODES_BF16
    assert linear(lib, x, w) == cr.ERR_INVALID_ARG
    x, w = pair(G=8)
    assert linear(lib, x, w) == cr.ERR_GROUP_SIZE
    x, w = pair()
    assert linear(lib, x, w, ldy=2) == cr.ERR_INVALID_ARG
    assert linear(lib, x, w, Y=None) == cr.ERR_INVALID_ARG
    assert linear(lib, x, w, Y=FAKE + 4) == cr.ERR_ALIGNMENT
    assert linear(lib, x, w, ldy=6) == cr.ERR_ALIGNMENT
    assert linear(lib, x, w, bias=FAKE + 2) == cr.ERR_ALIGNMENT
    x.q = None
    assert linear(lib, x, w) == cr.ERR_INVALID_ARG
    assert lib.convrot_linear(None, ctypes.byref(w), None, FAKE, 64, None, None) == cr.ERR_INVALID_ARG


def test_linear_empty_is_noop(lib):
    x, w = pair(mx=0)
    assert linear(lib, x, w, Y=None) == cr.OK
    x, w = pair(nw=0)
    assert linear(lib, x, w, Y=None) == cr.OK


def test_gemm_i32_validation(lib):
    x, w = pair()
    assert lib.convrot_gemm_i32(ctypes.byref(x), ctypes.byref(w), None, 4, None, None) == cr.ERR_INVALID_ARG
    assert lib.convrot_gemm_i32(ctypes.byref(x), ctypes.byref(w), FAKE, 3, None, None) == cr.ERR_INVALID_ARG
    x, w = pair(mx=0)
    assert lib.convrot_gemm_i32(ctypes.byref(x), ctypes.byref(w), None, 4, None, None) == cr.OK


def test_linear_act_rejects_unknown_activation(lib):
    x, w = pair()
    for act in (-1, 3, 99):
        assert lib.convrot_linear_act(ctypes.byref(x), ctypes.byref(w), None, act, FAKE, 64, None, None) == \
            cr.ERR_INVALID_ARG
    x, w = pair(mx=0)
    assert lib.convrot_linear_act(ctypes.byref(x), ctypes.byref(w), None, cr.ACT_GELU_ERF, None, 64, None, None) == cr.OK


def test_lora_cols(lib):
    assert lib.convrot_lora_cols(16) == 64
    assert lib.convrot_lora_cols(64) == 192
    assert lib.convrot_lora_cols(48) == 192
    assert lib.convrot_lora_cols(256) == 768
    for r in (0, 8, 24, 272, -16):
        assert lib.convrot_lora_cols(r) == 0


def test_lora_entry_points_validate(lib):
    assert lib.convrot_lora_prepare(FAKE, 4, 24, 24, 1.0, FAKE, 128, None) == cr.ERR_INVALID_ARG  # r % 16
    assert lib.convrot_lora_prepare(FAKE, 4, 16, 8, 1.0, FAKE, 64, None) == cr.ERR_INVALID_ARG   # ldb < r
    assert lib.convrot_lora_prepare(FAKE, 4, 16, 16, 1.0, FAKE, 32, None) == cr.ERR_INVALID_ARG  # lde < cols
    assert lib.convrot_lora_prepare(FAKE, 4, 16, 16, 1.0, FAKE + 8, 64, None) == cr.ERR_ALIGNMENT
    assert lib.convrot_lora_prepare(None, 0, 16, 16, 1.0, None, 64, None) == cr.OK
    assert lib.convrot_lora_down(FAKE, 4, 0, 256, FAKE, 16, 256, FAKE, 64, None, None) == cr.ERR_K_RANGE
    assert lib.convrot_lora_down(FAKE, 4, 256, 250, FAKE, 16, 256, FAKE, 64, None, None) == cr.ERR_INVALID_ARG
    assert lib.convrot_lora_down(FAKE + 4, 4, 256, 256, FAKE, 16, 256, FAKE, 64, None, None) == cr.ERR_ALIGNMENT
    assert lib.convrot_lora_down(FAKE, 4, 256, 256, FAKE, 16, 256, FAKE, 60, None, None) == cr.ERR_INVALID_ARG
    assert lib.convrot_lora_down(None, 0, 256, 256, None, 16, 256, None, 64, None, None) == cr.OK
    assert lib.convrot_lora_prepare_down(FAKE, 16, 0, 256, FAKE, 256, None) == cr.ERR_K_RANGE
    assert lib.convrot_lora_prepare_down(FAKE, 16, 256, 256, FAKE + 4, 256, None) == cr.ERR_ALIGNMENT
    assert lib.convrot_lora_prepare_down(FAKE, 12, 256, 256, FAKE, 256, None) == cr.ERR_INVALID_ARG


def test_linear_lora_validates(lib):
    x, w = pair(codes=cr.CODES_BF16)
    call = lambda x, w, r=16, t=FAKE, ldt=64, b=FAKE, ldb=64: lib.convrot_linear_lora(
        ctypes.byref(x), ctypes.byref(w), None, 0, t, ldt, b, ldb, r, FAKE, 64, None, None)
    assert call(x, w, r=0) == cr.ERR_INVALID_ARG
    assert call(x, w, r=20) == cr.ERR_INVALID_ARG
    assert call(x, w, ldt=32) == cr.ERR_INVALID_ARG
    assert call(x, w, t=FAKE + 8) == cr.ERR_ALIGNMENT
    assert call(x, w, t=None) == cr.ERR_INVALID_ARG
    xi, wi = pair(codes=cr.CODES_I8)
    assert call(xi, wi) == cr.ERR_UNSUPPORTED


def test_wait_check_validates_before_launching(lib):
    assert lib.convrot_wait_check(None, 1000, 0, None) == cr.ERR_INVALID_ARG
    assert lib.convrot_wait_check(FAKE, 0, 0, None) == cr.ERR_INVALID_ARG
    assert lib.convrot_wait_check(FAKE, cr.WAIT_LIMIT_NS + 1, 0, None) == cr.ERR_INVALID_ARG
    assert "bounded wait" in cr.status_string(cr.ERR_TIMEOUT)
