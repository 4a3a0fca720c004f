"""Seeded synthetic inputs for the convrot linear, shared by tests and bench.

This module draws random numbers only. It holds none of the layer's
arithmetic (no rotation, no quantization, no GEMM), so the oracle side and the
CUDA side of every parity test can both start from it.

Shapes follow DiT denoisers of the kind the page "INT8 Convrot Safetensors"
(stable-diffusion.cpp docs) targets: M = image or video tokens, K = hidden or
MLP width. Activations are N(0, 1) with a few fixed outlier channels scaled up
(the case the rotation exists for, "How INT8 convrot works"); weights are
N(0, 0.02^2) and biases N(0, 0.01^2), fp32 (the bias stays fp32 as in sd.cpp).

Each tensor comes from its own numpy substream keyed by (seed, tag), so that a
weight can be drawn without drawing the activation first.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_TAG_COLS, _TAG_X, _TAG_W, _TAG_B = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    """One convrot linear problem: Y[M, N] = X[M, K] W[N, K]^T + b[N]."""

    name: str
    m: int
    k: int
    n: int
    G: int
    seed: tuple
    outlier_frac: float = 0.001
    outlier_scale: float = 50.0
    outlier_cols: tuple | None = None  # fixed columns; overrides outlier_frac
    gelu_input: bool = False  # X = GELU(N(0,1)) before the outlier scaling
    linears: int = 1  # linears sharing one packed X (q, k, v -> 3)
    act: int = 0      # activation after the (first) linear: 0 none, 1 GELU erf form, 2 GELU tanh form
    down_n: int = 0   # > 0: a DiT MLP pair; the activated output feeds a down projection to down_n features
    lora_r: int = 0   # > 0: a runtime LoRA of this rank on the (first) linear
    lora_scale: float = 2.0  # alpha / r
    notes: str = field(default="", compare=False)

    @property
    def int_ops(self) -> int:
        """2*M*N*K integer operations of one GEMM."""
        return 2 * self.m * self.n * self.k

    @property
    def step_ops(self) -> int:
        """2*M*N*K summed over every GEMM of one step (all linears, both MLP projections).
        A LoRA's own multiply-adds (2 M r (K + N)) are not counted: the metric is the
        convrot linear's."""
        return sum(2 * self.m * st.n * st.k for st in stage_shapes(self))

    @property
    def pack_bytes(self) -> int:
        """Algorithmic bytes of one pack: 4 B read + 1 B code written per element, 4 B scale per row."""
        return self.m * (5 * self.k + 4)


def _rng(seed: tuple, tag: int) -> np.random.Generator:
    return np.random.default_rng(list(seed) + [tag])


def outlier_columns(wl: Workload) -> np.ndarray:
    if wl.outlier_cols is not None:
        return np.asarray(wl.outlier_cols, dtype=np.int64)
    count = int(round(wl.outlier_frac * wl.k))
    cols = _rng(wl.seed, _TAG_COLS).choice(wl.k, size=count, replace=False)
    return np.sort(cols).astype(np.int64)


def _gelu_exact(x: np.ndarray) -> np.ndarray:
    from scipy.special import erf

    return (0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))).astype(np.float32)


def activations(wl: Workload, rows: slice | None = None) -> np.ndarray:
    """X fp32 [M, K] (or the given row slice of it: the full draw, then sliced)."""
    X = _rng(wl.seed, _TAG_X).standard_normal((wl.m, wl.k), dtype=np.float32)
    if wl.gelu_input:
        X = _gelu_exact(X)
    cols = outlier_columns(wl)
    if cols.size:
        X[:, cols] *= np.float32(wl.outlier_scale)
    return X if rows is None else np.ascontiguousarray(X[rows])


def weights(wl: Workload, index: int = 0) -> np.ndarray:
    """W fp32 [N, K] ~ N(0, 0.02^2); `index` picks one of the linears sharing the input."""
    rng = _rng(wl.seed, _TAG_W) if index == 0 else np.random.default_rng(list(wl.seed) + [_TAG_W, index])
    return rng.standard_normal((wl.n, wl.k), dtype=np.float32) * np.float32(0.02)


def bias(wl: Workload, index: int = 0) -> np.ndarray:
    """b fp32 [N] ~ N(0, 0.01^2)."""
    rng = _rng(wl.seed, _TAG_B) if index == 0 else np.random.default_rng(list(wl.seed) + [_TAG_B, index])
    return rng.standard_normal((wl.n,), dtype=np.float32) * np.float32(0.01)


@dataclass(frozen=True)
class StageShape:
    k: int   # input features
    n: int   # output features (all linears of the stage)
    act: int


def stage_shapes(wl: Workload):
    """The pack + linear stages of one step: one for a single (or grouped) linear,
    two for an MLP pair (the second packs the first's activated output)."""
    if wl.down_n:
        return [StageShape(wl.k, wl.n, wl.act), StageShape(wl.n, wl.down_n, 0)]
    return [StageShape(wl.k, wl.n * wl.linears, wl.act)]


_DOWN = 10  # substream index of the down projection's weights and bias


def stage_weights(wl: Workload, s: int):
    """(list of W_i fp32 [n_i, k], concatenated bias fp32 [n]) of stage s."""
    if s == 1:
        W = np.random.default_rng(list(wl.seed) + [_TAG_W, _DOWN]).standard_normal(
            (wl.down_n, wl.n), dtype=np.float32) * np.float32(0.02)
        b = np.random.default_rng(list(wl.seed) + [_TAG_B, _DOWN]).standard_normal(
            (wl.down_n,), dtype=np.float32) * np.float32(0.01)
        return [W], b
    count = 1 if wl.down_n else wl.linears
    return [weights(wl, i) for i in range(count)], np.concatenate([bias(wl, i) for i in range(count)])


_LORA_A, _LORA_B = 20, 21  # substream indices of the adapter's matrices


def lora_weights(wl: Workload):
    """(A [r, k], B [n, r]) fp32 of the workload's adapter, both ~ N(0, 0.02^2)."""
    r, n = wl.lora_r, wl.n * wl.linears
    A = np.random.default_rng(list(wl.seed) + [_TAG_W, _LORA_A]).standard_normal((r, wl.k), dtype=np.float32)
    B = np.random.default_rng(list(wl.seed) + [_TAG_W, _LORA_B]).standard_normal((n, r), dtype=np.float32)
    return A * np.float32(0.02), B * np.float32(0.02)


def _sweep(G: int) -> Workload:
    return Workload(f"sweep_G{G}", 4096, 3072, 3072, G, (3, G))


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 64, 256, 256, 256, (0,), outlier_cols=(7, 200)),
        Workload("attn_qkv", 4096, 3072, 3072, 256, (1,), linears=3),
        Workload("mlp_up", 4096, 3072, 12288, 256, (2, 0)),
        Workload("mlp_down", 4096, 12288, 3072, 256, (2, 1), gelu_input=True),
        Workload("mlp_up_lora", 4096, 3072, 12288, 256, (2, 0), lora_r=64, lora_scale=2.0,
                 notes="MLP up with a rank-64 runtime LoRA, scale 128/64 (the rank and lora_alpha of the "
                       "few-step LoRA in the stable-diffusion-cpp article, section \"A LoRA that loaded "
                       "320 of its 448 tensors\")"),
        Workload("mlp_pair", 4096, 3072, 12288, 256, (2, 2), act=1, down_n=3072,
                 notes="up projection with GELU fused in its epilogue, then pack + down projection"),
        *[_sweep(G) for G in (4, 16, 64, 256, 1024)],
        Workload("video_n5120", 32760, 5120, 5120, 256, (4,), outlier_frac=0.0005,
                 outlier_scale=100.0),
        Workload("video_n13824", 32760, 5120, 13824, 256, (4,), outlier_frac=0.0005,
                 outlier_scale=100.0),
    ]
}

HEADLINE = "mlp_up"
