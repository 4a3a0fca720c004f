"""Python binding of libconvrot's C ABI (ctypes; argument marshalling only).

The names mirror ``include/convrot.h``. Every step of the layer runs in the
library's CUDA kernels; this module only turns torch CUDA tensors into device
pointers and the current torch stream into a ``cudaStream_t``. There is no
fallback: if the library is missing, calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from . import build as _build

OK, ERR_INVALID_ARG, ERR_GROUP_SIZE, ERR_ALIGNMENT, ERR_K_RANGE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED, ERR_SCRATCH = range(9)
NOALLOC_SCRATCH_BYTES = 32 << 20
WAIT_LIMIT_NS = 4_000_000_000
CODES_I8, CODES_BF16 = 0, 1
MAX_K = 133144
MAX_GROUP = 65536

EXPORTED = [
    "convrot_ldq",
    "convrot_quantize_weights",
    "convrot_pack_activations",
    "convrot_linear",
    "convrot_linear_act",
    "convrot_linear_pack_work_bytes",
    "convrot_linear_act_pack",
    "convrot_lora_cols",
    "convrot_lora_prepare",
    "convrot_lora_prepare_down",
    "convrot_lora_down",
    "convrot_linear_lora",
    "convrot_linear_lora_noalloc",
    "convrot_gemm_i32",
    "convrot_wait_check",
    "convrot_status_string",
]


class ConvrotError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class _Packed(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("k", ctypes.c_int64),
        ("ldq", ctypes.c_int64),
        ("group_size", ctypes.c_int32),
        ("codes", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Loads libconvrot.so (built in-tree by ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libconvrot.so is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        P = ctypes.POINTER(_Packed)
        lib.convrot_ldq.argtypes = [i64]
        lib.convrot_ldq.restype = i64
        lib.convrot_quantize_weights.argtypes = [vp, i64, i64, i64, i32, P, vp, vp]
        lib.convrot_quantize_weights.restype = ctypes.c_int
        lib.convrot_pack_activations.argtypes = [vp, i64, i64, i64, i32, P, vp, vp]
        lib.convrot_pack_activations.restype = ctypes.c_int
        lib.convrot_linear.argtypes = [P, P, vp, vp, i64, vp, vp]
        lib.convrot_linear.restype = ctypes.c_int
        lib.convrot_linear_act.argtypes = [P, P, vp, i32, vp, i64, vp, vp]
        lib.convrot_linear_act.restype = ctypes.c_int
        lib.convrot_linear_pack_work_bytes.argtypes = [i64, i64]
        lib.convrot_linear_pack_work_bytes.restype = i64
        lib.convrot_linear_act_pack.argtypes = [P, P, vp, i32, i32, vp, i64, P, vp, vp]
        lib.convrot_linear_act_pack.restype = ctypes.c_int
        lib.convrot_lora_cols.argtypes = [i32]
        lib.convrot_lora_cols.restype = i64
        lib.convrot_lora_prepare.argtypes = [vp, i64, i32, i64, ctypes.c_float, vp, i64, vp]
        lib.convrot_lora_prepare.restype = ctypes.c_int
        lib.convrot_lora_prepare_down.argtypes = [vp, i32, i64, i64, vp, i64, vp]
        lib.convrot_lora_prepare_down.restype = ctypes.c_int
        lib.convrot_lora_down.argtypes = [vp, i64, i64, i64, vp, i32, i64, vp, i64, vp, vp]
        lib.convrot_lora_down.restype = ctypes.c_int
        lib.convrot_linear_lora.argtypes = [P, P, vp, i32, vp, i64, vp, i64, i32, vp, i64, vp, vp]
        lib.convrot_linear_lora.restype = ctypes.c_int
        lib.convrot_linear_lora_noalloc.argtypes = [P, P, vp, i32, vp, i64, vp, i64, vp, i64, i32, vp, i64, vp, vp]
        lib.convrot_linear_lora_noalloc.restype = ctypes.c_int
        lib.convrot_gemm_i32.argtypes = [P, P, vp, i64, vp, vp]
        lib.convrot_gemm_i32.restype = ctypes.c_int
        lib.convrot_wait_check.argtypes = [vp, ctypes.c_uint64, i32, vp]
        lib.convrot_wait_check.restype = ctypes.c_int
        lib.convrot_status_string.argtypes = [ctypes.c_int]
        lib.convrot_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().convrot_status_string(int(status)).decode()


convrot_status_string = status_string


def convrot_ldq(k: int) -> int:
    return int(load().convrot_ldq(int(k)))


@dataclass
class Packed:
    """Owner of a packed block: codes q [rows, ldq] and fp32 scale [rows] (torch CUDA tensors)."""

    q: torch.Tensor
    scale: torch.Tensor
    rows: int
    k: int
    group_size: int
    codes: int

    @property
    def ldq(self) -> int:
        return self.q.stride(0)

    def struct(self) -> _Packed:
        return _Packed(self.q.data_ptr() if self.q.numel() else None,
                       self.scale.data_ptr() if self.scale.numel() else None,
                       self.rows, self.k, self.ldq, self.group_size, self.codes)

    def codes_as_int8(self) -> torch.Tensor:
        """[rows, k] int8 view of the codes (a copy for bf16 codes)."""
        q = self.q[:, : self.k]
        return q if self.codes == CODES_I8 else q.to(torch.int8)


def empty_packed(rows: int, k: int, codes: int = CODES_I8, device=None) -> Packed:
    """Allocates (with torch) the buffers a pack call fills."""
    ldq = convrot_ldq(k)
    dtype = torch.int8 if codes == CODES_I8 else torch.bfloat16
    device = device or torch.device("cuda", torch.cuda.current_device())
    q = torch.empty((rows, ldq), dtype=dtype, device=device)
    s = torch.empty((rows,), dtype=torch.float32, device=device)
    return Packed(q, s, rows, k, 0, codes)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status: int, what: str):
    if status != OK:
        raise ConvrotError(status, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None or t.numel() == 0 else t.data_ptr()


def _padded_out(m: int, n: int, dtype, device) -> torch.Tensor:
    """[m, n] output whose row pitch is a multiple of 4 elements (16-byte rows), as the ABI asks."""
    ld = (n + 3) // 4 * 4
    return torch.empty((m, ld), dtype=dtype, device=device)[:, :n]


def _pack(fn, X: torch.Tensor, G: int, codes: int, out: Packed | None, dev_status, stream,
          what: str) -> Packed:
    if X.dtype != torch.float32 or not X.is_cuda or X.dim() != 2 or X.stride(1) != 1:
        raise TypeError("X must be a 2-D row-major float32 CUDA tensor")
    rows, k = X.shape
    out = out or empty_packed(rows, k, codes, X.device)
    st = out.struct()
    _check(fn(_ptr(X), rows, k, X.stride(0), int(G), ctypes.byref(st), _ptr(dev_status), _stream(stream)),
           what)
    out.rows, out.k, out.group_size = int(st.rows), int(st.k), int(st.group_size)
    return out


def convrot_quantize_weights(W: torch.Tensor, G: int, codes: int = CODES_I8, out: Packed | None = None,
                             dev_status: torch.Tensor | None = None, stream=None) -> Packed:
    """Offline: Q_w, s_w of W [n, k] fp32 (page section "Weight quantization")."""
    return _pack(load().convrot_quantize_weights, W, G, codes, out, dev_status, stream,
                 "convrot_quantize_weights")


def convrot_pack_activations(X: torch.Tensor, G: int, codes: int = CODES_I8, out: Packed | None = None,
                             dev_status: torch.Tensor | None = None, stream=None) -> Packed:
    """Runtime: Q_x, s_x of X [m, k] fp32 (page section "Runtime activation quantization")."""
    return _pack(load().convrot_pack_activations, X, G, codes, out, dev_status, stream,
                 "convrot_pack_activations")


def convrot_linear(x: Packed, w: Packed, bias: torch.Tensor | None = None, out: torch.Tensor | None = None,
                   dev_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y [m, n] fp32 = (Q_x Q_w^T) * s_x s_w + b."""
    if out is None:
        out = _padded_out(x.rows, w.rows, torch.float32, x.q.device)
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda):
        raise TypeError("bias must be a float32 CUDA tensor")
    xs, ws = x.struct(), w.struct()
    _check(load().convrot_linear(ctypes.byref(xs), ctypes.byref(ws), _ptr(bias), _ptr(out),
                                 out.stride(0) if out.dim() == 2 else 0, _ptr(dev_status),
                                 _stream(stream)), "convrot_linear")
    return out


ACT_NONE, ACT_GELU_ERF, ACT_GELU_TANH = 0, 1, 2


def convrot_linear_act(x: Packed, w: Packed, bias: torch.Tensor | None, act: int,
                       out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Y [m, n] fp32 = act((Q_x Q_w^T) * s_x s_w + b), act one of ACT_*."""
    if out is None:
        out = _padded_out(x.rows, w.rows, torch.float32, x.q.device)
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda):
        raise TypeError("bias must be a float32 CUDA tensor")
    xs, ws = x.struct(), w.struct()
    _check(load().convrot_linear_act(ctypes.byref(xs), ctypes.byref(ws), _ptr(bias), int(act), _ptr(out),
                                     out.stride(0) if out.dim() == 2 else 0, _ptr(dev_status),
                                     _stream(stream)), "convrot_linear_act")
    return out


def linear_pack_work_bytes(m: int, n: int) -> int:
    """Bytes of the workspace convrot_linear_act_pack needs for an [m, n] output."""
    return int(load().convrot_linear_pack_work_bytes(int(m), int(n)))


def convrot_linear_act_pack(x: Packed, w: Packed, bias: torch.Tensor | None, act: int, G: int,
                            codes: int = CODES_BF16, out: Packed | None = None, work: torch.Tensor | None = None,
                            dev_status: torch.Tensor | None = None, stream=None) -> Packed:
    """The linear with an activation, then the pack of its output H = act(...) for the next
    linear with group size G: the same codes and scales as convrot_linear_act followed by
    convrot_pack_activations, with the rotation and row absmax in the GEMM's epilogue.
    ``work`` (uint8 CUDA tensor of linear_pack_work_bytes(m, n) bytes) is allocated here
    when not given."""
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda):
        raise TypeError("bias must be a float32 CUDA tensor")
    m, n = x.rows, w.rows
    need = linear_pack_work_bytes(m, n)
    if work is None:
        work = torch.empty((max(need, 1),), dtype=torch.uint8, device=x.q.device)
    elif work.dtype != torch.uint8 or not work.is_cuda or work.dim() != 1 or work.numel() < need:
        raise ValueError(f"work must be a 1-D uint8 CUDA tensor of at least {need} bytes")
    out = out or empty_packed(m, n, codes, x.q.device)
    xs, ws, os_ = x.struct(), w.struct(), out.struct()
    _check(load().convrot_linear_act_pack(ctypes.byref(xs), ctypes.byref(ws), _ptr(bias), int(act), int(G),
                                          _ptr(work), int(work.numel()), ctypes.byref(os_), _ptr(dev_status),
                                          _stream(stream)), "convrot_linear_act_pack")
    out.rows, out.k, out.group_size = int(os_.rows), int(os_.k), int(os_.group_size)
    return out


def lora_cols(r: int) -> int:
    """K extent of the LoRA operands: 3 r rounded up to 64 (0 if r is not accepted)."""
    return int(load().convrot_lora_cols(int(r)))


def _lora_out(rows: int, r: int, device) -> torch.Tensor:
    cols = lora_cols(r)
    if cols == 0:
        raise ConvrotError(ERR_INVALID_ARG, "lora rank")
    return torch.empty((rows, cols), dtype=torch.bfloat16, device=device)


def convrot_lora_prepare(B: torch.Tensor, scale: float, out: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Offline: B [n, r] fp32 (the adapter's up matrix) -> B_ext [n, lora_cols(r)] bf16 with
    the scale folded in."""
    if B.dtype != torch.float32 or not B.is_cuda or B.dim() != 2 or B.stride(1) != 1:
        raise TypeError("B must be a 2-D row-major float32 CUDA tensor")
    n, r = B.shape
    if out is None:
        out = _lora_out(n, r, B.device)
    _check(load().convrot_lora_prepare(_ptr(B), n, r, B.stride(0), float(scale), _ptr(out), out.stride(0),
                                       _stream(stream)), "convrot_lora_prepare")
    return out


def convrot_lora_prepare_down(A: torch.Tensor, stream=None) -> torch.Tensor:
    """Offline: the adapter's down matrix A [r, k] fp32 -> A_ext [2r, k rounded up to 4] fp32
    = [hi(A); lo(A)] (hi exact in TF32)."""
    if A.dtype != torch.float32 or not A.is_cuda or A.dim() != 2 or A.stride(1) != 1:
        raise TypeError("A must be a 2-D row-major float32 CUDA tensor")
    r, k = A.shape
    out = torch.zeros((2 * r, (k + 3) // 4 * 4), dtype=torch.float32, device=A.device)
    _check(load().convrot_lora_prepare_down(_ptr(A), r, k, A.stride(0), _ptr(out), out.stride(0), _stream(stream)),
           "convrot_lora_prepare_down")
    return out


def convrot_lora_down(X: torch.Tensor, A_ext: torch.Tensor, out: torch.Tensor | None = None,
                      dev_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per call: T = X A^T from the unrotated X [m, k] and A_ext (convrot_lora_prepare_down),
    as T_ext [m, lora_cols(r)] bf16."""
    for t, name in ((X, "X"), (A_ext, "A_ext")):
        if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise TypeError(f"{name} must be a 2-D row-major float32 CUDA tensor")
    m, k = X.shape
    r = A_ext.shape[0] // 2
    if out is None:
        out = _lora_out(m, r, X.device)
    _check(load().convrot_lora_down(_ptr(X), m, k, X.stride(0), _ptr(A_ext), r, A_ext.stride(0), _ptr(out),
                                    out.stride(0), _ptr(dev_status), _stream(stream)), "convrot_lora_down")
    return out


def _check_matrix(t: torch.Tensor, name: str, dtype, rows: int, min_cols: int, exact_cols: bool = False):
    """t must be a 2-D row-major `dtype` tensor with `rows` rows and at least (or
    exactly) `min_cols` columns. The C side receives only a pointer and a leading
    dimension and cannot check any of this; a tensor that breaks it would make a kernel
    read outside the buffer. (That it lives on the GPU is checked by _check_cuda.)"""
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.dim() != 2 or t.stride(1) != 1:
        raise TypeError(f"{name} must be a 2-D row-major {str(dtype).replace('torch.', '')} tensor")
    if t.shape[0] != rows or (t.shape[1] != min_cols if exact_cols else t.shape[1] < min_cols):
        want = f"[{rows}, {min_cols}]" if exact_cols else f"[{rows}, >= {min_cols}]"
        raise ValueError(f"{name} has shape {list(t.shape)}; expected {want}")


def _check_cuda(**tensors):
    for name, t in tensors.items():
        if not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")


def _check_lora_up(w: Packed, b_ext: torch.Tensor, r: int):
    cols = lora_cols(r)
    if cols == 0:
        raise ConvrotError(ERR_INVALID_ARG, "lora rank")
    _check_matrix(b_ext, "B_ext", torch.bfloat16, w.rows, cols)


def convrot_linear_lora(x: Packed, w: Packed, bias: torch.Tensor | None, act: int, t_ext: torch.Tensor,
                        b_ext: torch.Tensor, r: int, out: torch.Tensor | None = None,
                        dev_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = act((Q_x Q_w^T) s_x s_w + b + T_ext B_ext^T): the linear with the LoRA correction."""
    _check_lora_up(w, b_ext, r)
    _check_matrix(t_ext, "T_ext", torch.bfloat16, x.rows, lora_cols(r))
    _check_cuda(T_ext=t_ext, B_ext=b_ext)
    if out is None:
        out = _padded_out(x.rows, w.rows, torch.float32, x.q.device)
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda):
        raise TypeError("bias must be a float32 CUDA tensor")
    xs, ws = x.struct(), w.struct()
    _check(load().convrot_linear_lora(ctypes.byref(xs), ctypes.byref(ws), _ptr(bias), int(act), _ptr(t_ext),
                                      t_ext.stride(0), _ptr(b_ext), b_ext.stride(0), int(r), _ptr(out),
                                      out.stride(0) if out.dim() == 2 else 0, _ptr(dev_status), _stream(stream)),
           "convrot_linear_lora")
    return out


def convrot_linear_lora_noalloc(x: Packed, w: Packed, bias: torch.Tensor | None, act: int, X: torch.Tensor,
                                A_ext: torch.Tensor, b_ext: torch.Tensor, r: int, out: torch.Tensor | None = None,
                                dev_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The LoRA linear in one call that allocates no device memory, for callers that must
    not call cudaMalloc (device memory owned by a host application's pool, no room for an
    allocation's cost in a latency-bound loop, a fixed memory budget). T_ext goes to the
    library's 32 MiB per-device static array; larger requests raise ERR_SCRATCH. The first
    call on a device looks up that array's address: make it before any stream capture.
    Every call shares the array, so calls that overlap on the GPU race on it. ``out`` is
    allocated here only when the caller passes none; the C entry point allocates nothing.

    X must be the activations x was packed from, [x.rows, x.k] fp32, and A_ext the
    convrot_lora_prepare_down output for this r ([2 r, >= x.k] fp32); B_ext is
    [w.rows, >= lora_cols(r)] bf16. These are checked here, before the call, because
    the C entry point takes their sizes from x, w and r and cannot verify them."""
    _check_matrix(X, "X", torch.float32, x.rows, x.k, exact_cols=True)
    _check_matrix(A_ext, "A_ext", torch.float32, 2 * int(r), x.k)
    _check_lora_up(w, b_ext, r)
    _check_cuda(X=X, A_ext=A_ext, B_ext=b_ext)
    if out is None:
        out = _padded_out(x.rows, w.rows, torch.float32, x.q.device)
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda):
        raise TypeError("bias must be a float32 CUDA tensor")
    xs, ws = x.struct(), w.struct()
    _check(load().convrot_linear_lora_noalloc(ctypes.byref(xs), ctypes.byref(ws), _ptr(bias), int(act), _ptr(X),
                                              X.stride(0), _ptr(A_ext), A_ext.stride(0), _ptr(b_ext),
                                              b_ext.stride(0), int(r), _ptr(out),
                                              out.stride(0) if out.dim() == 2 else 0, _ptr(dev_status),
                                              _stream(stream)), "convrot_linear_lora_noalloc")
    return out


def convrot_gemm_i32(x: Packed, w: Packed, out: torch.Tensor | None = None,
                     dev_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """A [m, n] int32 = Q_x Q_w^T."""
    if out is None:
        out = _padded_out(x.rows, w.rows, torch.int32, x.q.device)
    xs, ws = x.struct(), w.struct()
    _check(load().convrot_gemm_i32(ctypes.byref(xs), ctypes.byref(ws), _ptr(out),
                                   out.stride(0) if out.dim() == 2 else 0, _ptr(dev_status),
                                   _stream(stream)), "convrot_gemm_i32")
    return out


def convrot_wait_check(dev_status: torch.Tensor, limit_ns: int, arrive: bool, stream=None) -> None:
    """Launch the bounded-wait check: with arrive False the kernel's wait runs
    out after limit_ns and it writes ERR_TIMEOUT into dev_status (int32, one
    element); with arrive True dev_status is left as it is."""
    _check(load().convrot_wait_check(_ptr(dev_status), int(limit_ns), int(bool(arrive)), _stream(stream)),
           "convrot_wait_check")


def quantize_weights_grouped(Ws, G: int, codes: int = CODES_I8, stream=None) -> Packed:
    """Quantize several weights that will multiply the same packed input into one packed block.

    Row block i of the result holds W_i's codes and scales (each W_i quantized by
    the same kernel as convrot_quantize_weights, written in place). One
    convrot_linear against it computes every linear at once; its output
    [m, sum(n_i)] holds linear i in columns [off_i, off_i + n_i) -- the page's
    packed activation is reused by all of them ("Runtime activation quantization").
    """
    Ws = list(Ws)
    if not Ws:
        raise ValueError("no weights")
    k = Ws[0].shape[1]
    if any(W.shape[1] != k for W in Ws):
        raise ValueError("grouped weights need the same input features")
    rows = sum(W.shape[0] for W in Ws)
    out = empty_packed(rows, k, codes, Ws[0].device)
    r0 = 0
    for W in Ws:
        n = W.shape[0]
        part = Packed(out.q[r0:r0 + n], out.scale[r0:r0 + n], n, k, 0, codes)
        convrot_quantize_weights(W, G, codes, out=part, stream=stream)
        r0 += n
    out.group_size = int(G)
    return out


def split_columns(Y: torch.Tensor, sizes):
    """Views of the column blocks of a grouped linear's output."""
    views, c0 = [], 0
    for n in sizes:
        views.append(Y[:, c0:c0 + n])
        c0 += n
    return views


def packed_from_codes(q_int8: torch.Tensor, scale: torch.Tensor, group_size: int, codes: int = CODES_I8) -> Packed:
    """Wraps externally produced codes (e.g. a checkpoint's I8 weight and its scales) as a Packed.

    Copies into the padded layout the GEMM reads: [rows, convrot_ldq(k)], zero past k.
    """
    rows, k = q_int8.shape
    p = empty_packed(rows, k, codes, q_int8.device)
    p.q.zero_()
    p.q[:, :k].copy_(q_int8 if codes == CODES_I8 else q_int8.to(torch.bfloat16))
    p.scale.copy_(scale.reshape(-1).to(torch.float32))
    p.group_size = int(group_size)
    return p
