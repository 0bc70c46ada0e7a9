"""Exact attention written out in float64 (test infrastructure only).

Every array argument is converted to float64 first; batch/head axes in front
of the last two are carried along by numpy broadcasting. Nothing here is
blocked, fused or reordered: the score matrix is materialised in full.

Sources (page title, then section):
  * "Flash attention, f32" (Phobos examples) -- opening statement
    O = softmax(Q K^T * scale) V.
  * "Flash Attention" (notes) -- Definition 1 (softmax) and Proposition 1
    (safe softmax, subtract the row maximum); "IO complexity" for the backward
    identity D_i = rowsum(dO o O), dS = P o (dP - D).
  * "06: Fused attention" (Phobos tutorial) -- the causal rule (key j is kept
    for query i iff j <= i), the stored row statistic L = m + log(l), and the
    gradient kernels' outputs dQ, dK, dV with the factor ``scale``.
  * "Flash decoding" (linear algebra for programmers, part 4) -- "Overview of
    the algorithm": the per-split (m, l, O) equations and the combine.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _t(x: np.ndarray) -> np.ndarray:
    return np.swapaxes(x, -1, -2)


def scores(Q, K, scale: float, causal: bool = False) -> np.ndarray:
    """S = scale * Q K^T, with S[i, j] = -inf where a causal mask hides key j.

    Causal masking follows the fused-attention tutorial's forward kernel, which
    keeps key j for query i only when j <= i; for M != N this is read as
    top-left alignment (the same rule on absolute indices).
    """
    Q, K = _f64(Q), _f64(K)
    S = float(scale) * np.matmul(Q, _t(K))
    if causal:
        M, N = S.shape[-2], S.shape[-1]
        keep = np.arange(N)[None, :] <= np.arange(M)[:, None]
        S = np.where(keep, S, -np.inf)
    return S


def _safe_softmax(S: np.ndarray):
    """Row softmax with the row maximum subtracted (notes, Proposition 1).

    Returns P, the row maxima m and the row sums l of exp(S - m).
    """
    m = np.max(S, axis=-1, keepdims=True)
    E = np.exp(S - m)
    l = np.sum(E, axis=-1, keepdims=True)
    return E / l, m, l


def forward(Q, K, V, scale: float, causal: bool = False):
    """O = softmax(scale * Q K^T) V and LSE = m + ln(l) per query row.

    Q [..., M, D], K and V [..., N, D]. LSE is in natural-log units of the
    scaled scores, the statistic the tutorial's forward kernel stores.
    """
    S = scores(Q, K, scale, causal)
    P, m, l = _safe_softmax(S)
    O = np.matmul(P, _f64(V))
    lse = (m + np.log(l))[..., 0]
    return O, lse


def probabilities(Q, K, scale: float, causal: bool = False) -> np.ndarray:
    """The full matrix P = softmax(scale * Q K^T)."""
    return _safe_softmax(scores(Q, K, scale, causal))[0]


def backward(Q, K, V, dO, scale: float, causal: bool = False):
    """Gradients of sum(dO o O) with respect to Q, K, V by the chain rule.

    dV = P^T dO; dP = dO V^T; through the softmax Jacobian
    dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik); through S = scale Q K^T,
    dQ = scale dS K and dK = scale dS^T Q. The row term sum_k P_ik dP_ik is
    taken in this form, not as rowsum(dO o O), so that the identity between the
    two (notes, "IO complexity") is something the tests check rather than assume.
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    P = probabilities(Q, K, scale, causal)
    dV = np.matmul(_t(P), dO)
    dP = np.matmul(dO, _t(V))
    row = np.sum(P * dP, axis=-1, keepdims=True)
    dS = P * (dP - row)
    dQ = float(scale) * np.matmul(dS, K)
    dK = float(scale) * np.matmul(_t(dS), Q)
    return dQ, dK, dV


def delta(O, dO) -> np.ndarray:
    """D_i = rowsum(dO o O) (notes, "IO complexity"; tutorial's delta kernel)."""
    return np.sum(_f64(O) * _f64(dO), axis=-1)


def decode(q, K, V, scale: float):
    """Decode attention: the forward with a single query row.

    q [..., 1, D] (or [..., D]), K and V [..., N, D]; returns O [..., 1, D].
    """
    q, K = _f64(q), _f64(K)
    if q.ndim == K.ndim - 1:
        q = q[..., None, :]
    return forward(q, K, V, scale, causal=False)[0]


def split_bounds(N: int, n_splits: int):
    """Key ranges [n_s, n_{s+1}) of the splits: chunks of ceil(N / n_splits) keys.

    The flash-decoding page's split kernel starts split s at s*S and ends it at
    min(s*S + S, N) for a split size S; S = ceil(N / n_splits) is the reading
    taken here, so trailing splits can be empty when n_splits does not divide N.
    """
    size = -(-N // n_splits)
    return [(min(s * size, N), min(s * size + size, N)) for s in range(n_splits)]


def decode_partials(q, K, V, scale: float, n_splits: int):
    """Per-split unnormalised partials for one query row (flash decoding).

    q [D], K and V [N, D]. For split s over keys [n_s, n_{s+1}):
      m_s = max_j x_j,  l_s = sum_j e^{x_j - m_s},  O_s = sum_j e^{x_j - m_s} V_j
    with x_j = scale * q . K_j. An empty split is the identity of the merge:
    m_s = -inf, l_s = 0, O_s = 0. Returns O_s [n_splits, D], m_s, l_s [n_splits].
    """
    q, K, V = _f64(q).reshape(-1), _f64(K), _f64(V)
    D = q.shape[0]
    Os = np.zeros((n_splits, D))
    ms = np.full(n_splits, -np.inf)
    ls = np.zeros(n_splits)
    for s, (lo, hi) in enumerate(split_bounds(K.shape[0], n_splits)):
        if lo >= hi:
            continue
        x = float(scale) * (K[lo:hi] @ q)
        ms[s] = np.max(x)
        e = np.exp(x - ms[s])
        ls[s] = np.sum(e)
        Os[s] = e @ V[lo:hi]
    return Os, ms, ls


def decode_combine(Os, ms, ls) -> np.ndarray:
    """Merge per-split partials (flash decoding, "combine"):

      m_g = max_s m_s,  l_g = sum_s e^{m_s - m_g} l_s,
      O = (1 / l_g) sum_s e^{m_s - m_g} O_s.
    """
    Os, ms, ls = _f64(Os), _f64(ms), _f64(ls)
    m_g = np.max(ms)
    w = np.where(np.isneginf(ms), 0.0, np.exp(ms - m_g))
    l_g = np.sum(w * ls)
    return (w @ Os) / l_g
