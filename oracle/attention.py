"""CPU oracle for attention forward: O = softmax(scale * Q K^T [+ causal mask]) V, fp64.

TEST INFRASTRUCTURE ONLY (same rules as the GEMM oracle in this package: only the tests,
the smoke check and the benchmark's CPU-baseline leg may use it; the GPU library never
does).

Sources (page title and section):
  * the aikraft.ru TileLang tutorial survey ("TileLang: создание высокопроизводительных
    GPU-ядер"), section 6 ("FlashAttention: Слияние внимания"): attention computed without
    materialising the full score matrix, with online softmax updates (running maxima,
    normalisation sums, rescaling factors) and causal masks.  The oracle computes the same
    function the plain way: the whole score matrix, one softmax per row;
  * "TileLang异步协作终极指南：如何实现2倍性能提升的GPU并行计算": the multi-head attention
    whose K/V loads, QK^T and softmax/output steps the page assigns to separate roles.

Readings where the pages are silent:
  * layout (batch, heads, seq, head_dim), row-major, fp16 in and out, fp64 here;
  * the default scale is 1/sqrt(head_dim);
  * causal masking keeps key j for query i when j <= i + (seq_kv - seq_q) (the mask aligned
    to the bottom-right corner, which is the usual lower triangle when seq_q == seq_kv);
  * a query row whose keys are all masked has no softmax: its output is 0 and its
    log-sum-exp is -inf;
  * the output is rounded once to fp16 (nearest, ties to even); lse is returned in fp64.
"""
from __future__ import annotations

import numpy as np


def attention(Q, K, V, scale: float | None = None, causal: bool = False, return_lse=False):
    """Q (B,H,Sq,D), K and V (B,H,Skv,D) fp16 (numpy or CPU torch).  Returns O as float16
    (B,H,Sq,D) and, with ``return_lse``, the fp64 log-sum-exp of the scaled scores (B,H,Sq)
    and the fp64 output before rounding."""
    q = _f64(Q)
    k = _f64(K)
    v = _f64(V)
    if q.ndim != 4 or k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("shapes: Q %s K %s V %s" % (q.shape, k.shape, v.shape))
    D = q.shape[3]
    sq, skv = q.shape[2], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    s = np.einsum("bhqd,bhkd->bhqk", q, k) * float(np.float32(scale))
    if causal:
        qi = np.arange(sq)[:, None]
        kj = np.arange(skv)[None, :]
        s = np.where(kj <= qi + (skv - sq), s, -np.inf)
    m = s.max(axis=-1, keepdims=True) if skv else np.full(s.shape[:-1] + (1,), -np.inf)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - safe_m)                       # masked entries give exp(-inf) = 0
    l = p.sum(axis=-1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l > 0, np.einsum("bhqk,bhkd->bhqd", p, v) / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[..., 0] > 0, safe_m[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)),
                       -np.inf)
    o16 = o.astype(np.float16)
    return (o16, lse, o) if return_lse else o16


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("attention oracle inputs must be float16, got %s" % x.dtype)
    return x.astype(np.float64)
