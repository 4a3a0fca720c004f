"""Oracle for the INT8 convrot linear layer: a plain fp64 CPU statement.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library and the CUDA library never calls it.

The arithmetic lives in ``convrot_oracle.c`` (plain C, fp64), written from the
page "INT8 Convrot Safetensors" (stable-diffusion.cpp docs): sections "How
INT8 convrot works", "Weight quantization" and "Runtime activation
quantization". This module only builds that file with gcc and marshals numpy
arrays through ctypes.

Every function here is pinned by ``tests/test_oracle.py`` to facts that do not
come from the oracle itself (the printed H4, a closed form of R_G, orthogonality,
the rotation identity, hand-worked rows, brute force and error bounds).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "convrot_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile convrot_oracle.c into _build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.oracle_log4.argtypes = [i64]
        lib.oracle_log4.restype = ctypes.c_int
        lib.oracle_h4.argtypes = [vp]
        lib.oracle_h4.restype = None
        lib.oracle_rotation_matrix.argtypes = [i64, vp]
        lib.oracle_rotation_matrix.restype = ctypes.c_int
        lib.oracle_rotate_dense.argtypes = [vp, i64, i64, i64, i64, vp, vp]
        lib.oracle_rotate_dense.restype = None
        lib.oracle_rotate_fast.argtypes = [vp, i64, i64, i64, i64, vp]
        lib.oracle_rotate_fast.restype = None
        lib.oracle_quantize_rows.argtypes = [vp, i64, i64, vp, vp, i64, vp]
        lib.oracle_quantize_rows.restype = None
        lib.oracle_gemm_i32.argtypes = [vp, i64, i64, vp, i64, i64, i64, vp, i64]
        lib.oracle_gemm_i32.restype = ctypes.c_int
        lib.oracle_reconstruct.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, i64, vp]
        lib.oracle_reconstruct.restype = None
        lib.oracle_pack_rows.argtypes = [vp, i64, i64, i64, i64, vp, vp, i64, vp]
        lib.oracle_pack_rows.restype = ctypes.c_int
        lib.oracle_lora_delta.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, ctypes.c_double, vp, vp]
        lib.oracle_lora_delta.restype = None
        lib.oracle_activation.argtypes = [vp, i64, ctypes.c_int]
        lib.oracle_activation.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _rows_f32(X: np.ndarray) -> np.ndarray:
    X = np.asarray(X)
    if X.dtype != np.float32:
        raise TypeError("X must be float32")
    if X.ndim != 2:
        raise ValueError("X must be 2-D")
    if X.strides[1] != 4:
        X = np.ascontiguousarray(X)
    return X


def num_threads() -> int:
    """Threads the oracle's row loops use (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def log4(G: int) -> int:
    """n if G == 4**n with n >= 1, else -1."""
    return int(_load().oracle_log4(int(G)))


def h4() -> np.ndarray:
    """The 4x4 matrix printed in "How INT8 convrot works", divided by 2."""
    out = np.empty((4, 4), np.float64)
    _load().oracle_h4(_ptr(out))
    return out


def rotation_matrix(G: int) -> np.ndarray:
    """Dense R_G: the normalized Kronecker power of H4 with G = 4**n."""
    R = np.empty((G, G), np.float64)
    if _load().oracle_rotation_matrix(int(G), _ptr(R)) != 0:
        raise ValueError(f"group size {G} is not a power of four >= 4")
    return R


def rotate_dense(X: np.ndarray, G: int) -> np.ndarray:
    """X_rot = X R by the definition (dense R_G per contiguous group), fp64."""
    X = _rows_f32(X)
    m, k = X.shape
    if k % G:
        raise ValueError("G must divide k")
    R = rotation_matrix(G)
    out = np.empty((m, k), np.float64)
    _load().oracle_rotate_dense(_ptr(X), m, k, X.strides[0] // 4, G, _ptr(R), _ptr(out))
    return out


def rotate_fast(X: np.ndarray, G: int) -> np.ndarray:
    """X_rot = X R by H4 along each base-4 digit (Kronecker mixed product), fp64."""
    X = _rows_f32(X)
    m, k = X.shape
    if log4(G) < 0 or k % G:
        raise ValueError("G must be a power of four >= 4 dividing k")
    out = np.empty((m, k), np.float64)
    _load().oracle_rotate_fast(_ptr(X), m, k, X.strides[0] // 4, G, _ptr(out))
    return out


def quantize_rows(rot: np.ndarray, ldq: int | None = None):
    """Row scales and int8 codes of fp64 rotated rows.

    Returns (Q int8 [m, ldq] zero past k, scale fp32 [m], pre_round fp64 [m, k]).
    """
    rot = np.ascontiguousarray(rot, dtype=np.float64)
    m, k = rot.shape
    ldq = k if ldq is None else int(ldq)
    Q = np.zeros((m, ldq), np.int8)
    s = np.empty((m,), np.float32)
    v = np.empty((m, k), np.float64)
    _load().oracle_quantize_rows(_ptr(rot), m, k, _ptr(s), _ptr(Q), ldq, _ptr(v))
    return Q, s, v


def pack_rows(X: np.ndarray, G: int, ldq: int | None = None, want_pre_round: bool = True):
    """Rotate then quantize each row: (Q int8 [m, ldq], scale fp32 [m], pre_round or None).

    The same routine serves activations (runtime) and weights (offline): the
    page defines both with the same formulas.
    """
    X = _rows_f32(X)
    m, k = X.shape
    ldq = k if ldq is None else int(ldq)
    Q = np.zeros((m, ldq), np.int8)
    s = np.empty((m,), np.float32)
    v = np.empty((m, k), np.float64) if want_pre_round else None
    rc = _load().oracle_pack_rows(_ptr(X), m, k, X.strides[0] // 4, int(G), _ptr(s), _ptr(Q),
                                  ldq, _ptr(v))
    if rc != 0:
        raise ValueError(f"bad group size {G} for k={k}")
    return Q, s, v


def gemm_i32(Qx: np.ndarray, Qw: np.ndarray, k: int) -> np.ndarray:
    """A = Q_x Q_w^T over the first k columns, int64 sums stored as int32."""
    Qx = np.ascontiguousarray(Qx, dtype=np.int8)
    Qw = np.ascontiguousarray(Qw, dtype=np.int8)
    m, n = Qx.shape[0], Qw.shape[0]
    A = np.empty((m, n), np.int32)
    rc = _load().oracle_gemm_i32(_ptr(Qx), m, Qx.shape[1], _ptr(Qw), n, Qw.shape[1], int(k),
                                 _ptr(A), n)
    if rc != 0:
        raise OverflowError("an accumulator left the signed 32-bit range")
    return A


def activation(v: np.ndarray, act: int) -> np.ndarray:
    """GELU (act 1: erf form, 2: tanh form) or identity (0) in fp64, elementwise."""
    out = np.ascontiguousarray(v, dtype=np.float64).copy()
    _load().oracle_activation(_ptr(out), out.size, int(act))
    return out


def lora_delta(X: np.ndarray, A: np.ndarray, B: np.ndarray, scale: float):
    """(T = X A^T, D = scale * T B^T), both fp64, from the unrotated X (r <= 256)."""
    X = _rows_f32(X)
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    m, k = X.shape
    r = A.shape[0]
    n = B.shape[0]
    if A.shape[1] != k or B.shape[1] != r or r > 256:
        raise ValueError("shapes: X [m, k], A [r, k], B [n, r], r <= 256")
    T = np.empty((m, r), np.float64)
    D = np.empty((m, n), np.float64)
    _load().oracle_lora_delta(_ptr(X), m, k, X.strides[0] // 4, _ptr(A), r, _ptr(B), n, float(scale), _ptr(T),
                              _ptr(D))
    return T, D


def reconstruct(A: np.ndarray, sx: np.ndarray, sw: np.ndarray, bias: np.ndarray | None, act: int = 0,
                add: np.ndarray | None = None):
    """Y = act(A * s_x[r] * s_w[o] + b[o] + add[r, o]) in fp64 (add: e.g. a LoRA
    correction, added before the activation); returns (Y fp32, Y fp64)."""
    A = np.ascontiguousarray(A, dtype=np.int32)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    m, n = A.shape
    Y = np.empty((m, n), np.float32)
    Y64 = np.empty((m, n), np.float64)
    _load().oracle_reconstruct(_ptr(A), n, m, n, _ptr(sx), _ptr(sw), _ptr(b), _ptr(Y), n,
                               _ptr(Y64))
    if add is not None:
        Y64 = Y64 + np.asarray(add, np.float64)
    if act:
        Y64 = activation(Y64, act)
    if add is not None or act:
        Y = Y64.astype(np.float32)
    return Y, Y64


def linear(X: np.ndarray, W: np.ndarray, bias: np.ndarray | None, G: int, act: int = 0):
    """End to end: pack X, quantize W, integer GEMM, reconstruct (then the activation).

    Returns a dict with Qx, sx, vx (pre-round), Qw, sw, A, Y (fp32), Y64.
    """
    X = _rows_f32(X)
    W = _rows_f32(W)
    k = X.shape[1]
    Qx, sx, vx = pack_rows(X, G)
    Qw, sw, _ = pack_rows(W, G, want_pre_round=False)
    A = gemm_i32(Qx, Qw, k)
    Y, Y64 = reconstruct(A, sx, sw, bias, act)
    return {"Qx": Qx, "sx": sx, "vx": vx, "Qw": Qw, "sw": sw, "A": A, "Y": Y, "Y64": Y64}
