"""Tolerance rules for comparing the CUDA path with the oracle.

The rules (stated for the INT8 convrot linear, page "INT8 Convrot
Safetensors", stable-diffusion.cpp docs):

  - row scales: |s - s_ref| <= 1e-6 * s_ref;
  - codes: at most ceil(1e-4 * count) entries differ from the oracle's, each
    by exactly 1, and only where the oracle's fp64 pre-round value lies within
    1e-4 of a .5 rounding boundary (the kernel rotates in fp32, the oracle in
    fp64, so values that close to a boundary may round either way);
  - given identical codes: the int32 accumulators are bit-exact, and
    |Y - Y_ref| <= 1e-6 * (|A s_x s_w| + |b|) elementwise (Y_ref in fp64);
  - end to end from X: |Y - Y_ref| <= 1e-3 * max |Y_ref|
    + 127 * s_x[r] s_w[o] * (flips_x[r] + flips_w[o]), where flips counts the
    codes of row r of X (row o of W) that the previous rule let differ: each
    such code moves the integer product by at most 127, times the scales.
"""

from __future__ import annotations

import math

import numpy as np

S_RTOL = 1e-6
CODE_FRAC = 1e-4
BOUNDARY = 1e-4
Y_RTOL_SAME_CODES = 1e-6
Y_END_TO_END = 1e-3


def check_scales(s_gpu: np.ndarray, s_ref: np.ndarray):
    s_gpu = np.asarray(s_gpu, np.float64)
    s_ref = np.asarray(s_ref, np.float64)
    err = np.abs(s_gpu - s_ref)
    bad = err > S_RTOL * np.abs(s_ref)
    assert not bad.any(), (f"{bad.sum()} scales off; worst rel "
                           f"{np.max(err / np.maximum(np.abs(s_ref), 1e-300)):.3e}")


def check_codes(q_gpu: np.ndarray, q_ref: np.ndarray, pre_round: np.ndarray):
    """q_gpu, q_ref: int [rows, k]; pre_round: the oracle's fp64 v = rot / s."""
    q_gpu = np.asarray(q_gpu, np.int32)
    q_ref = np.asarray(q_ref, np.int32)
    diff = q_gpu != q_ref
    n_diff = int(diff.sum())
    if n_diff == 0:
        return 0
    assert n_diff <= math.ceil(CODE_FRAC * q_ref.size), f"{n_diff} of {q_ref.size} codes differ"
    assert np.all(np.abs(q_gpu[diff] - q_ref[diff]) == 1), "a code differs by more than 1"
    v = pre_round[diff]
    dist = np.abs(np.abs(v - np.trunc(v)) - 0.5)
    assert np.all(dist <= BOUNDARY), f"a differing code is {dist.max():.3e} from a .5 boundary"
    return n_diff


def check_y_same_codes(y_gpu: np.ndarray, y64_ref: np.ndarray, A: np.ndarray, sx, sw, bias):
    base = np.abs(A.astype(np.float64) * np.asarray(sx, np.float64)[:, None]
                  * np.asarray(sw, np.float64)[None, :])
    if bias is not None:
        base = base + np.abs(np.asarray(bias, np.float64))[None, :]
    err = np.abs(np.asarray(y_gpu, np.float64) - y64_ref)
    bad = err > Y_RTOL_SAME_CODES * base + 1e-30
    assert not bad.any(), f"{bad.sum()} outputs off; worst {np.max(err / np.maximum(base, 1e-300)):.3e}"


def check_y_act_same_codes(y_gpu: np.ndarray, y64_ref: np.ndarray, A: np.ndarray, sx, sw, bias):
    """Y = act(A s_x s_w + b), given identical codes: the pre-activation rule
    (1e-6 of |A s_x s_w| + |b|) times GELU's largest slope (1.13), rounded up
    to 1.5e-6, plus 3e-7 |Y| for erff/tanhf and the fp32 products after them."""
    base = np.abs(A.astype(np.float64) * np.asarray(sx, np.float64)[:, None]
                  * np.asarray(sw, np.float64)[None, :])
    if bias is not None:
        base = base + np.abs(np.asarray(bias, np.float64))[None, :]
    err = np.abs(np.asarray(y_gpu, np.float64) - y64_ref)
    tol = 1.5e-6 * base + 3e-7 * np.abs(y64_ref) + 1e-30
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} outputs off; worst {np.max(err / tol):.3e} of the tolerance"


def check_y_end_to_end(y_gpu: np.ndarray, y_ref: np.ndarray, qx=None, qw=None, sx=None, sw=None):
    """qx = (gpu codes, oracle codes) of the rows of X behind y, qw likewise for W,
    sx, sw the GPU's scales; without them no code may have flipped."""
    err = np.abs(np.asarray(y_gpu, np.float64) - np.asarray(y_ref, np.float64))
    ref = np.max(np.abs(np.asarray(y_ref, np.float64)))
    tol = np.full(err.shape, Y_END_TO_END * ref)
    if qx is not None:
        fx = (np.asarray(qx[0], np.int32) != np.asarray(qx[1], np.int32)).sum(axis=1).astype(np.float64)
        fw = (np.asarray(qw[0], np.int32) != np.asarray(qw[1], np.int32)).sum(axis=1).astype(np.float64)
        tol = tol + 127.0 * (1 + 1e-6) * (np.asarray(sx, np.float64)[:, None] * np.asarray(sw, np.float64)[None, :]
                                          * (fx[:, None] + fw[None, :]))
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} outputs off end to end; worst |dY| = {err.max():.3e}, 1e-3 * max|Y| = {Y_END_TO_END * ref:.3e}"
