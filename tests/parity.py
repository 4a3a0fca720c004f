"""Tolerance rules for comparing the CUDA path with the oracle.

The rules (stated for the INT8 convrot linear, page "INT8 Convrot
Safetensors", stable-diffusion.cpp docs):

  - row scales: |s - s_ref| <= 1e-6 * s_ref;
  - codes: at most 1e-4 of the entries (floor(1e-4 * count)) differ from the oracle's, each
    by exactly 1, and only where the oracle's fp64 pre-round value lies within
    1e-4 of a .5 rounding boundary (the kernel rotates in fp32, the oracle in
    fp64, so values that close to a boundary may round either way);
  - given identical codes: the int32 accumulators are bit-exact, and
    |Y - Y_ref| <= 1e-6 * (|A s_x s_w| + |b|) elementwise (Y_ref in fp64);
  - end to end from X: |Y - Y_ref| <= 1e-3 * max |Y_ref|
    + 127 * s_x[r] s_w[o] * (flips_x[r] + flips_w[o]), where flips counts the
    codes of row r of X (row o of W) that the previous rule let differ: each
    such code moves the integer product by at most 127, times the scales.
    check_y_end_to_end returns how often that flip term was needed, and
    whether the plain bound |Y - Y_ref| <= 1e-3 * max |Y_ref| held on its own.

Tests may record those statistics with record(); when the environment names a
file in CONVROT_PARITY_RECORD, the session writes every record there as JSON.
"""

from __future__ import annotations

import math

import numpy as np

RECORDS: list = []


def record(case: str, **stats):
    """Keeps one line of parity statistics (written out at the end of the session)."""
    RECORDS.append({"case": case, **stats})

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
    assert n_diff <= math.floor(CODE_FRAC * q_ref.size), f"{n_diff} of {q_ref.size} codes differ"
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
    to 1.5e-6 (this also covers the erf approximation's 1.5e-7 |v| / 2), plus
    3e-7 |Y| for the fast exponential and division and the fp32 products."""
    base = np.abs(A.astype(np.float64) * np.asarray(sx, np.float64)[:, None]
                  * np.asarray(sw, np.float64)[None, :])
    if bias is not None:
        base = base + np.abs(np.asarray(bias, np.float64))[None, :]
    err = np.abs(np.asarray(y_gpu, np.float64) - y64_ref)
    tol = 1.5e-6 * base + 3e-7 * np.abs(y64_ref) + 1e-30
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} outputs off; worst {np.max(err / tol):.3e} of the tolerance"


def check_y_end_to_end(y_gpu: np.ndarray, y_ref: np.ndarray, qx=None, qw=None, sx=None, sw=None) -> dict:
    """qx = (gpu codes, oracle codes) of the rows of X behind y, qw likewise for W,
    sx, sw the GPU's scales; without them no code may have flipped.

    Returns: outputs compared; code flips in those rows of X and in W; how many
    outputs needed the flip term (their error is above the plain bound); whether
    the plain bound held everywhere; and the largest error over the plain bound."""
    err = np.abs(np.asarray(y_gpu, np.float64) - np.asarray(y_ref, np.float64))
    ref = np.max(np.abs(np.asarray(y_ref, np.float64)))
    plain = Y_END_TO_END * ref
    tol = np.full(err.shape, plain)
    flips_x = flips_w = 0
    if qx is not None:
        fx = (np.asarray(qx[0], np.int32) != np.asarray(qx[1], np.int32)).sum(axis=1).astype(np.float64)
        fw = (np.asarray(qw[0], np.int32) != np.asarray(qw[1], np.int32)).sum(axis=1).astype(np.float64)
        flips_x, flips_w = int(fx.sum()), int(fw.sum())
        tol = tol + 127.0 * (1 + 1e-6) * (np.asarray(sx, np.float64)[:, None] * np.asarray(sw, np.float64)[None, :]
                                          * (fx[:, None] + fw[None, :]))
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} outputs off end to end; worst |dY| = {err.max():.3e}, 1e-3 * max|Y| = {plain:.3e}"
    needed = int((err > plain).sum())
    return {"outputs": int(err.size), "flips_x": flips_x, "flips_w": flips_w, "needed_flip_term": needed,
            "plain_bound_held": needed == 0, "max_err_over_plain": float(err.max() / plain) if plain > 0 else 0.0}


def lora_t_tolerance(k: int) -> float:
    """Relative bound (to sum_i |X_i||A_i|) on T = X A^T from three-term TF32:
    every product is formed exactly from the split parts except the dropped
    lo*lo term and lo's own TF32 rounding (together < 2^-20), and the sum
    runs over 3k terms in fp32 with at most one ulp (2^-23) lost per add."""
    return 3 * k * 2.0 ** -23 + 2.0 ** -20


def lora_t_rms_tolerance(k: int) -> float:
    """Typical size of the same error: independent roundings over 3k adds grow
    like sqrt(3k) * 2^-24; four of those."""
    return 4 * math.sqrt(3 * k) * 2.0 ** -24


def check_lora_t(t_gpu, t_ref, l1, k):
    """T against the fp64 oracle; l1 = |X| |A|^T."""
    err = np.abs(np.asarray(t_gpu, np.float64) - t_ref)
    tol = lora_t_tolerance(k) * l1 + 2.0 ** -17 * np.abs(t_ref) + 1e-30  # + the bf16 hi/lo form of T
    assert not (err > tol).any(), f"{(err > tol).sum()} of T off; worst {np.max(err / tol):.3e} of the tolerance"
    rms = math.sqrt(float(np.mean(err ** 2)))
    rms_l1 = math.sqrt(float(np.mean(l1 ** 2)))
    assert rms <= lora_t_rms_tolerance(k) * rms_l1 + 2.0 ** -17 * math.sqrt(float(np.mean(t_ref ** 2))), \
        f"rms error {rms:.3e} vs {lora_t_rms_tolerance(k) * rms_l1:.3e}"


def check_y_lora_same_codes(y_gpu, y64_ref, A, sx, sw, bias, lora_l1, k, r, act):
    """Y = act(base + D): the base rule (1e-6 of |A s_x s_w| + |b|), plus for the
    correction D (magnitude lora_l1 = scale |X| |A|^T |B|^T) the T bound, the
    two-term bf16 split of T and of scale*B (2^-15) and the fp32 sum over
    3r terms (3r * 2^-23); times GELU's largest slope 1.13 when act, plus 3e-7 |Y|."""
    base = np.abs(A.astype(np.float64) * np.asarray(sx, np.float64)[:, None] * np.asarray(sw, np.float64)[None, :])
    if bias is not None:
        base = base + np.abs(np.asarray(bias, np.float64))[None, :]
    c = lora_t_tolerance(k) + 2.0 ** -15 + 3 * r * 2.0 ** -23
    tol = 1e-6 * base + c * lora_l1
    if act:
        tol = 1.13 * tol + 3e-7 * np.abs(y64_ref)
    tol = tol + 1e-30
    err = np.abs(np.asarray(y_gpu, np.float64) - y64_ref)
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} outputs off; worst {np.max(err / tol):.3e} of the tolerance"
    # typical size: a dropped hi/lo term (2^-9 relative) would stand far above this
    rms = lambda a: math.sqrt(float(np.mean(np.square(a))))
    typ = (lora_t_rms_tolerance(k) + 2.0 ** -15 + 4 * math.sqrt(3 * r) * 2.0 ** -24) * rms(lora_l1) + 1e-6 * rms(base)
    assert rms(err) <= (1.13 if act else 1.0) * typ + (3e-7 * rms(y64_ref) if act else 0.0), \
        f"rms error {rms(err):.3e} above the typical bound {typ:.3e}"
