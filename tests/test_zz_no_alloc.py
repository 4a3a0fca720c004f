"""convrot_linear_lora_noalloc: the LoRA linear in one call that allocates no
device memory. It is for callers that must not call cudaMalloc: a plug-in
whose host application owns all device memory through its own pool, a
latency-bound loop that cannot pay for an allocation (or the synchronization
a free brings), or code held to a device-memory budget fixed at load time.
T_ext then lives in a 32 MiB array that the library declares at file scope
on each device.

Two calls in a row, with different shapes and ranks so that the second
overwrites what the first left in the shared array, must equal the existing
two-call path (convrot_lora_down into a caller-allocated T_ext, then
convrot_linear_lora) bit for bit: the same kernels run on the same inputs.
Requests larger than the array are refused before any launch. This file is
named to be collected last."""

import ctypes

import numpy as np
import pytest
import torch

from int8_hadamard_rotated_convrot_gb300 import build as cbuild
from int8_hadamard_rotated_convrot_gb300 import convrot as cr

FAKE = 0x10000


def test_noalloc_rejects_requests_beyond_the_scratch():
    cbuild.build()
    lib = cr.load()
    r = 64
    cols = lib.convrot_lora_cols(r)
    rows = cr.NOALLOC_SCRATCH_BYTES // (cols * 2) + 1
    ld = cr.convrot_ldq(256)
    x = cr._Packed(FAKE, FAKE, rows, 256, ld, 256, cr.CODES_BF16)
    w = cr._Packed(FAKE, FAKE, 8, 256, ld, 256, cr.CODES_BF16)
    st = lib.convrot_linear_lora_noalloc(ctypes.byref(x), ctypes.byref(w), None, 0, FAKE, 256, FAKE, 256, FAKE, cols,
                                         r, FAKE, 8, None, None)
    assert st == cr.ERR_SCRATCH
    assert "static scratch" in cr.status_string(cr.ERR_SCRATCH)
    assert lib.convrot_linear_lora_noalloc(ctypes.byref(x), ctypes.byref(w), None, 0, FAKE, 256, FAKE, 256, FAKE,
                                           cols, 20, FAKE, 8, None, None) == cr.ERR_INVALID_ARG


def test_noalloc_checks_the_linear_before_any_device_work():
    """The linear's own argument errors come back before the scratch lookup and
    before the down kernel would run (here, without a GPU, any device call would
    answer CONVROT_ERR_CUDA instead)."""
    cbuild.build()
    lib = cr.load()
    r = 64
    cols = lib.convrot_lora_cols(r)
    ld = cr.convrot_ldq(256)
    args = lambda x, w, ldy, Y: (ctypes.byref(x), ctypes.byref(w), None, 0, FAKE, 256, FAKE, 256, FAKE, cols, r,
                                 Y, ldy, None, None)
    x = cr._Packed(FAKE, FAKE, 8, 256, ld, 256, cr.CODES_I8)
    w = cr._Packed(FAKE, FAKE, 8, 256, ld, 256, cr.CODES_I8)
    assert lib.convrot_linear_lora_noalloc(*args(x, w, 8, FAKE)) == cr.ERR_UNSUPPORTED  # I8 codes: no LoRA chunk
    x = cr._Packed(FAKE, FAKE, 8, 256, ld, 256, cr.CODES_BF16)
    w = cr._Packed(FAKE, FAKE, 8, 256, ld, 256, cr.CODES_BF16)
    assert lib.convrot_linear_lora_noalloc(*args(x, w, 8, FAKE + 4)) == cr.ERR_ALIGNMENT  # Y not 16-byte aligned
    assert lib.convrot_linear_lora_noalloc(*args(x, w, 7, FAKE)) == cr.ERR_INVALID_ARG  # ldy < n
    assert lib.convrot_linear_lora_noalloc(*args(x, w, 8, None)) == cr.ERR_INVALID_ARG  # no Y
    w_other_g = cr._Packed(FAKE, FAKE, 8, 256, ld, 64, cr.CODES_BF16)
    assert lib.convrot_linear_lora_noalloc(*args(x, w_other_g, 8, FAKE)) == cr.ERR_GROUP_SIZE


def test_noalloc_wrapper_rejects_tensors_the_c_side_cannot_check():
    """The C entry point takes X's and A_ext's sizes from x and r, so the binding
    checks the tensors before the call: wrong dtype, layout, shape or device
    raise here, on the host, and nothing reaches the library."""
    cbuild.build()
    cr.load()
    m, k, n, r = 8, 256, 16, 64
    cols = cr.lora_cols(r)
    x = cr.Packed(torch.zeros((m, cr.convrot_ldq(k)), dtype=torch.bfloat16), torch.zeros(m), m, k, 256,
                  cr.CODES_BF16)
    w = cr.Packed(torch.zeros((n, cr.convrot_ldq(k)), dtype=torch.bfloat16), torch.zeros(n), n, k, 256,
                  cr.CODES_BF16)
    X = torch.zeros((m, k))
    A_ext = torch.zeros((2 * r, k))
    B_ext = torch.zeros((n, cols), dtype=torch.bfloat16)
    call = lambda X=X, A=A_ext, B=B_ext: cr.convrot_linear_lora_noalloc(x, w, None, 0, X, A, B, r,
                                                                         out=torch.zeros((m, n)))
    with pytest.raises(TypeError):
        call(X=X.double())                        # not fp32
    with pytest.raises(TypeError):
        call(X=torch.zeros((k, m)).t())           # not row-major
    with pytest.raises(ValueError):
        call(X=X[: m - 1])                        # fewer rows than x was packed from
    with pytest.raises(ValueError):
        call(X=torch.zeros((m, k - 4)))           # fewer columns than x.k
    with pytest.raises(ValueError):
        call(A=torch.zeros((2 * 32, k)))          # prepared for another rank
    with pytest.raises(ValueError):
        call(A=torch.zeros((2 * r, k - 4)))       # narrower than x.k
    with pytest.raises(TypeError):
        call(B=B_ext.float())                     # B_ext is bf16
    with pytest.raises(ValueError):
        call(B=B_ext[:, : cols - 8])              # fewer columns than lora_cols(r)
    with pytest.raises(TypeError, match="CUDA"):
        call()                                    # right shapes, but host tensors


def _case(rng, m, n, k, r):
    X = rng.standard_normal((m, k)).astype(np.float32)
    W = (0.02 * rng.standard_normal((n, k))).astype(np.float32)
    b = rng.standard_normal(n).astype(np.float32)
    A = (0.05 * rng.standard_normal((r, k))).astype(np.float32)
    B = (0.05 * rng.standard_normal((n, r))).astype(np.float32)
    dev = lambda a: torch.from_numpy(a).cuda()
    Xd = dev(X)
    px = cr.convrot_pack_activations(Xd, 64, cr.CODES_BF16)
    pw = cr.convrot_quantize_weights(dev(W), 64, cr.CODES_BF16)
    A_ext = cr.convrot_lora_prepare_down(dev(A))
    B_ext = cr.convrot_lora_prepare(dev(B), 2.0)
    return Xd, px, pw, dev(b), A_ext, B_ext


@pytest.mark.gpu
def test_noalloc_lora_linear_twice_equals_two_call_path():
    cbuild.build()
    rng = np.random.default_rng(2024)
    cases = [(_case(rng, 300, 512, 1024, 64), 64, cr.ACT_NONE), (_case(rng, 129, 256, 512, 32), 32, cr.ACT_GELU_ERF)]
    outs = []
    for (Xd, px, pw, b, A_ext, B_ext), r, act in cases:  # two calls in a row
        outs.append(cr.convrot_linear_lora_noalloc(px, pw, b, act, Xd, A_ext, B_ext, r))
    for ((Xd, px, pw, b, A_ext, B_ext), r, act), y in zip(cases, outs):
        T_ext = cr.convrot_lora_down(Xd, A_ext)
        y_ref = cr.convrot_linear_lora(px, pw, b, act, T_ext, B_ext, r)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        assert torch.isfinite(y).all() and y.abs().max() > 0


@pytest.mark.gpu
def test_noalloc_at_the_largest_accepted_request():
    """r = 256 at the most rows the array holds (21845 x 768 bf16 fills all but 512
    bytes of it): the last rows of T_ext sit at the array's end, and the result still
    equals the two-call path; one more row is refused."""
    cbuild.build()
    r = 256
    m = cr.NOALLOC_SCRATCH_BYTES // (cr.lora_cols(r) * 2)
    assert m == 21845
    rng = np.random.default_rng(77)
    Xd, px, pw, b, A_ext, B_ext = _case(rng, m, 256, 256, r)
    y = cr.convrot_linear_lora_noalloc(px, pw, b, cr.ACT_NONE, Xd, A_ext, B_ext, r)
    y_ref = cr.convrot_linear_lora(px, pw, b, cr.ACT_NONE, cr.convrot_lora_down(Xd, A_ext), B_ext, r)
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)
    Xd1, px1, pw1, b1, A1, B1 = _case(rng, m + 1, 256, 256, r)
    with pytest.raises(cr.ConvrotError):
        cr.convrot_linear_lora_noalloc(px1, pw1, b1, cr.ACT_NONE, Xd1, A1, B1, r)
