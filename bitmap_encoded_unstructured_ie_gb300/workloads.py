"""Seeded synthetic inputs for the bitmap SpMM / spMspV workloads.

The only module that both the CUDA path's callers (tests, benchmark) and the CPU
oracle's tests take inputs from.  It draws matrices and activations and quantises
them to int4 codes; it holds none of the format's or the product's arithmetic
(no bitmap, no offsets, no multiply).

Stand-ins: the pages evaluate on pruned LLaMA / OPT / Qwen projection weights and
on real activations.  None of those is available, so each workload takes only
their shapes and sparsity statistics:

* weights ~ N(0, 0.02), activations ~ N(0, 1), drawn with numpy's PCG64;
  W uses ``seed``, X uses ``seed + 1``, activation thresholds ``seed + 2``;
* "uniform" sparsity keeps each position independently with probability
  ``1 - s``; "magnitude" sparsity keeps, per row, the ``round(keep * K)``
  largest |w| (ties to the lower column index), with ``keep`` fixed or drawn
  per row as ``0.3 + 0.4 * Beta(2, 2)``;
* int4 quantisation (W4A4): per row (weights) or per token (activations),
  ``s = fp16(max|v| / 7)`` and ``q = clip(rint(v / s), -8, 7)``; a kept weight
  that rounds to 0 is a zero of the quantised matrix;
* int2 quantisation (W2A4, the plain reading of a setting the pages only name):
  per row ``s = fp16(max|w| / 2)`` and ``q = clip(rint(w / s), -2, 1)``;
* spMspV activations: ``x ~ N(0, 1)`` with its ``round(p * K)`` smallest entries
  set to 0 (a ReLU-style threshold at the empirical p-quantile).
"""
from __future__ import annotations

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal(seed: int, shape, std: float) -> np.ndarray:
    return (rng(seed).standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def uniform_mask(seed: int, shape, keep: float) -> np.ndarray:
    """Each position kept independently with probability ``keep``."""
    return rng(seed).random(size=shape, dtype=np.float32) < np.float32(keep)


def magnitude_mask(W: np.ndarray, keep_per_row: np.ndarray) -> np.ndarray:
    """Per row, keep the round(keep*K) largest |w|; ties go to the lower column."""
    M, K = W.shape
    counts = np.rint(np.asarray(keep_per_row, dtype=np.float64) * K).astype(np.int64)
    counts = np.clip(counts, 0, K)
    order = np.argsort(-np.abs(W), axis=1, kind="stable")
    ranks = np.empty_like(order)
    np.put_along_axis(ranks, order, np.arange(K)[None, :].repeat(M, axis=0), axis=1)
    return ranks < counts[:, None]


def beta_row_keep(seed: int, M: int) -> np.ndarray:
    """Per-row keep rate 0.3 + 0.4 * Beta(2, 2): mean 0.5, range [0.3, 0.7]."""
    return 0.3 + 0.4 * rng(seed).beta(2.0, 2.0, size=M)


def quantize_int4_rows(V: np.ndarray):
    """Symmetric int4 per row: codes int8 in [-8, 7] and an fp16 scale per row."""
    V = np.asarray(V, dtype=np.float32)
    amax = np.abs(V).max(axis=1)
    s = (amax / np.float32(7.0)).astype(np.float16)
    s = np.where(s == 0, np.float16(1.0), s).astype(np.float16)
    q = np.clip(np.rint(V / s.astype(np.float32)[:, None]), -8, 7).astype(np.int8)
    return q, s


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Row-major int4 codes -> bytes, two per byte, element 2i in the low nibble."""
    flat = np.ascontiguousarray(codes, dtype=np.int8).reshape(-1)
    if flat.size % 2:
        flat = np.concatenate([flat, np.zeros(1, np.int8)])
    u = flat.view(np.uint8) & np.uint8(0x0F)
    return (u[0::2] | (u[1::2] << np.uint8(4))).astype(np.uint8)


# ---------------------------------------------------------------------------
def f16_weights(M: int, K: int, sparsity: float, seed: int, mode: str = "uniform") -> np.ndarray:
    """fp16 W (M x K) ~ N(0, 0.02) with unstructured sparsity."""
    W = _normal(seed, (M, K), 0.02)
    if mode == "uniform":
        mask = uniform_mask(seed + 1000003, (M, K), 1.0 - sparsity)
    else:
        mask = magnitude_mask(W, np.full(M, 1.0 - sparsity))
    return np.where(mask, W, np.float32(0)).astype(np.float16)


def clustered_importance(seed: int, M: int, K: int, group: int = 4, sigma: float = 3.0) -> np.ndarray:
    """Per-row column scales shared by groups of `group` consecutive rows:
    exp(sigma * N(0, 1)) per (group, column).  A magnitude mask taken on
    W * scales keeps mostly the same positions within a group: rows that share
    sparsity patterns, the structure the bitmap-aware row reordering of
    UnionSparse (section V-B) groups into one union mask."""
    rng = np.random.default_rng(seed)
    g = np.exp(rng.standard_normal(((M + group - 1) // group, K)) * sigma).astype(np.float32)
    return np.repeat(g, group, axis=0)[:M]


def scatter_within_tiles(seed: int, M: int, TM: int) -> np.ndarray:
    """A row order that shuffles the rows inside every TM-row block (seeded),
    so that only a reordering finds the groups again."""
    rng = np.random.default_rng(seed)
    order = np.arange(M)
    for b in range(0, M - M % TM, TM):
        order[b:b + TM] = b + rng.permutation(TM)
    return order


def w4a4(M: int, K: int, N: int, sparsity: float, seed: int, rows: str = "fixed"):
    """W4A4 workload: magnitude-pruned, per-row int4 W; per-token int4 X.
    rows: "fixed" (every row keeps 1 - sparsity), "beta" (per-row keep rates
    from Beta(2, 2)), "clustered" (groups of four rows share column scales
    before pruning, then the rows are shuffled within each 16-row block).

    Returns dict with Wq (int8 M x K), s_w (fp16 M), Xq (int8 N x K),
    Xq_packed (uint8 N*K/2), s_x (fp16 N).
    """
    W = _normal(seed, (M, K), 0.02)
    keep = beta_row_keep(seed + 2, M) if rows == "beta" else np.full(M, 1.0 - sparsity)
    # clustered: the mask comes from the magnitudes under the shared column
    # scales; the kept values stay N(0, 0.02)
    score = W * clustered_importance(seed + 3, M, K) if rows == "clustered" else W
    W = np.where(magnitude_mask(score, keep), W, np.float32(0))
    if rows == "clustered":
        W = W[scatter_within_tiles(seed + 4, M, 16)]
    Wq, s_w = quantize_int4_rows(W)
    X = _normal(seed + 1, (N, K), 1.0)
    Xq, s_x = quantize_int4_rows(X)
    return {"Wq": Wq, "s_w": s_w, "Xq": Xq, "Xq_packed": pack_int4(Xq), "s_x": s_x}


def quantize_int2_rows(V: np.ndarray):
    """Per-row int2 codes in [-2, 1] with an fp16 scale amax / 2 per row (the
    positive end saturates at +1; zeros of V stay zero)."""
    V = np.asarray(V, dtype=np.float32)
    amax = np.abs(V).max(axis=1)
    s = (amax / np.float32(2.0)).astype(np.float16)
    s = np.where(s == 0, np.float16(1.0), s).astype(np.float16)
    q = np.clip(np.rint(V / s.astype(np.float32)[:, None]), -2, 1).astype(np.int8)
    return q, s


def w2a4(M: int, K: int, N: int, sparsity: float, seed: int):
    """W2A4 workload (UnionSparse Fig. 11 names the setting): the W4A4 recipe
    with magnitude-pruned weights quantised per row to int2 codes in [-2, 1];
    activations per-token int4.  Same keys as ``w4a4``."""
    W = _normal(seed, (M, K), 0.02)
    W = np.where(magnitude_mask(W, np.full(M, 1.0 - sparsity)), W, np.float32(0))
    Wq, s_w = quantize_int2_rows(W)
    X = _normal(seed + 1, (N, K), 1.0)
    Xq, s_x = quantize_int4_rows(X)
    return {"Wq": Wq, "s_w": s_w, "Xq": Xq, "Xq_packed": pack_int4(Xq), "s_x": s_x}


def f16_spmm(M: int, K: int, N: int, sparsity: float, seed: int):
    """fp16 SpMM workload: uniform-random sparse W and dense X (N x K)."""
    W = f16_weights(M, K, sparsity, seed, "uniform")
    X = _normal(seed + 1, (N, K), 1.0).astype(np.float16)
    return {"W": W, "X": X}


def relu_threshold(x: np.ndarray, zero_frac: float) -> np.ndarray:
    """Zero the round(zero_frac * K) smallest entries (ties to the lower index)."""
    K = x.size
    n0 = int(round(zero_frac * K))
    order = np.argsort(x, kind="stable")
    out = x.copy()
    out[order[:n0]] = 0
    return out


def spmspv(M: int, K: int, sparsity: float, act_zero_frac: float, seed: int):
    """fp16 spMspV workload: uniform-random sparse W and a thresholded x."""
    W = f16_weights(M, K, sparsity, seed, "uniform")
    x = relu_threshold(_normal(seed + 2, (K,), 1.0), act_zero_frac).astype(np.float16)
    return {"W": W, "x": x}


# Named configurations (shapes and statistics of the evaluated workloads).
CONFIGS = {
    "f16_256x512_n1": dict(kind="f16", M=256, K=512, N=1, sparsity=0.5, TM=64, TK=64),
    "w4a4_4096_s30": dict(kind="w4a4", M=4096, K=4096, sparsity=0.3, rows="fixed"),
    "w4a4_4096_s50": dict(kind="w4a4", M=4096, K=4096, sparsity=0.5, rows="fixed"),
    "w4a4_4096_s70": dict(kind="w4a4", M=4096, K=4096, sparsity=0.7, rows="fixed"),
    "w4a4_11008x4096_beta": dict(kind="w4a4", M=11008, K=4096, sparsity=0.5, rows="beta"),
    "w4a4_4096x11008_beta": dict(kind="w4a4", M=4096, K=11008, sparsity=0.5, rows="beta"),
    "f16_prefill_4096_s60": dict(kind="f16", M=4096, K=4096, sparsity=0.6),
    "spmspv_14336x4096": dict(kind="spmspv", M=14336, K=4096, sparsity=0.5),
}
