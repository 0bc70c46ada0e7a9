"""The FP8 forward's steps written out in float64 (test infrastructure only).

"Flash Attention" (notes), section "FlashAttention 3", the FP8 bullets: Q and K are
multiplied on the right by a random orthogonal M = diag(signs) H / sqrt(d) (H the
Hadamard matrix; Q M (K M)^T = Q K^T exactly, while outliers spread over all d
columns), then quantised to FP8 with one scale per block of rows (a B_r x d tile).
FP8 here is E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, largest
finite value 448), rounded to nearest with ties to even and saturated to +-448.

Readings where the page is silent (also listed with the design notes): a block is
128 rows of Q or 128 keys of K; V is quantised with one scale per (batch, head),
because the key blocks of P V are summed into one accumulator; the weights P are
quantised without a scale (they lie in [0, 1] here, in [0, 2^8] in the kernel,
inside E4M3's range); O is divided by the sum of the quantised weights (so a
dominant key's rounding cancels), LSE uses the exact sum.

Nothing is blocked or reordered beyond the block scales the method defines: the score
matrix is formed in full from the dequantised operands.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e4m3_positive_values() -> np.ndarray:
    """Every finite non-negative E4M3 value, in code order 0x00 .. 0x7E (0x7F is NaN)."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


_E4M3 = _e4m3_positive_values()


def e4m3_round(x) -> np.ndarray:
    """x rounded to the nearest E4M3 value (ties to the even code), saturated to +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    i = np.clip(np.searchsorted(_E4M3, a), 1, len(_E4M3) - 1)
    lo, hi = _E4M3[i - 1], _E4M3[i]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & (i % 2 == 0))  # code i even
    r = np.where(pick_hi, hi, lo)
    return np.copysign(r, x)


def hadamard(d: int) -> np.ndarray:
    """The d x d Sylvester Hadamard matrix (entries +-1, H H^T = d I); d a power of two."""
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    assert H.shape[0] == d, "d must be a power of two"
    return H


def incoherent(X, signs) -> np.ndarray:
    """X M with M = diag(signs) H / sqrt(d), on the last axis (the head dimension)."""
    X = np.asarray(X, dtype=np.float64)
    s = np.asarray(signs, dtype=np.float64)
    d = X.shape[-1]
    return (X * s) @ hadamard(d) / np.sqrt(d)


def quantize_blocks(X, rows: int):
    """Blocks of `rows` rows along axis -2 quantised to E4M3 with one scale each,
    scale = amax(block) / 448 (1 for an all-zero block). Returns (E4M3 values, scales
    [..., blocks])."""
    X = np.asarray(X, dtype=np.float64)
    n = X.shape[-2]
    nb = (n + rows - 1) // rows
    pad = nb * rows - n
    Xp = np.concatenate([X, np.zeros(X.shape[:-2] + (pad, X.shape[-1]))], axis=-2) if pad else X
    Xb = Xp.reshape(X.shape[:-2] + (nb, rows, X.shape[-1]))
    amax = np.max(np.abs(Xb), axis=(-2, -1))
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    q = e4m3_round(Xb / scale[..., None, None])
    return q.reshape(Xp.shape)[..., :n, :], scale


def forward_fp8(Q, K, V, scale: float, causal: bool, signs, block: int = 128):
    """The FP8 forward on one or more heads: returns (O, LSE) as float64.

    Q [..., M, d], K and V [..., N, d]; signs [d] of +-1 (drawn by the caller)."""
    Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    M, N = Q.shape[-2], K.shape[-2]
    q8, sq = quantize_blocks(incoherent(Q, signs), block)
    k8, sk = quantize_blocks(incoherent(K, signs), block)
    v8, sv = quantize_blocks(V, N)
    row_scale = np.repeat(sq, block, axis=-1)[..., :M]
    col_scale = np.repeat(sk, block, axis=-1)[..., :N]
    S = float(scale) * (q8 @ np.swapaxes(k8, -1, -2)) * row_scale[..., :, None] * col_scale[..., None, :]
    if causal:
        S = np.where(np.arange(N)[None, :] <= np.arange(M)[:, None], S, -np.inf)
    m = np.max(S, axis=-1, keepdims=True)
    E = np.exp(S - m)
    P8 = e4m3_round(E)
    O = (P8 @ v8) * sv[..., 0][..., None, None] / np.sum(P8, axis=-1, keepdims=True)
    L = m[..., 0] + np.log(np.sum(E, axis=-1))
    return O, L
