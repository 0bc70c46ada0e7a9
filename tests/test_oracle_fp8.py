"""Pins for the FP8 steps of the oracle (oracle/fp8.py), against things other than themselves.

* E4M3 rounding: a brute-force nearest-value search over every finite E4M3 value (ties to the
  even code), and PyTorch's float8_e4m3fn conversion (a library routine) inside the finite range;
  fixed points, saturation and the relative error bound of a 3-bit mantissa.
* The Hadamard-times-sign transform: H H^T = d I, Q M (K M)^T = Q K^T in float64, norms kept, and
  a one-hot outlier spread evenly over all d columns (the closed form).
* Block quantisation: each block's largest magnitude lands on +-448, every element within half an
  E4M3 step of its value.
* The FP8 forward: closed forms (V = 1 gives O = 1; one key gives its quantised value), and its
  error against exact attention within the stated FP8 tolerance on the workload's inputs.
Planted mistakes in copies of the transform fail at least one pin.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from exact_attention_gb300 import synth
from oracle import fp8

from helpers import TOL_FP8, fp8_rmse


def _all_e4m3():
    v = fp8._e4m3_positive_values()
    codes = np.arange(len(v))
    return np.concatenate([-v[::-1], v[1:]]), np.concatenate([codes[::-1], codes[1:]])


def _brute_round(x):
    vals, codes = _all_e4m3()
    out = np.empty_like(x)
    for i, xi in enumerate(x):
        a = min(abs(xi), 448.0) * (1 if xi >= 0 else -1)
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:  # a tie: the even code
            best = [b for b in best if codes[b] % 2 == 0]
        out[i] = vals[best[0]]
    return out


def test_e4m3_round_matches_brute_force_nearest_even():
    rng = np.random.default_rng(0)
    vals, _ = _all_e4m3()
    mids = (vals[:-1] + vals[1:]) / 2  # exact ties
    x = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(500) * 0.01, mids,
                        mids * (1 + 1e-12), mids * (1 - 1e-12), [0.0, -0.0, 447.9, 448.0, 460.0, 1e6, -1e6]])
    assert np.array_equal(fp8.e4m3_round(x), _brute_round(x))


def test_e4m3_round_matches_torch_float8_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch has no float8_e4m3fn")
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 30, rng.standard_normal(2000) * 0.003]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_round(x.astype(np.float64)), ref)


def test_e4m3_properties():
    vals, _ = _all_e4m3()
    assert len(vals) == 253 and vals.max() == 448.0 and fp8._e4m3_positive_values()[1] == 2.0 ** -9
    assert np.array_equal(fp8.e4m3_round(vals), vals)  # representable values are fixed points
    assert fp8.e4m3_round(np.array([1e9, -1e9, 449.0])).tolist() == [448.0, -448.0, 448.0]
    x = np.random.default_rng(2).uniform(2.0 ** -6, 448, 20000)
    assert np.max(np.abs(fp8.e4m3_round(x) / x - 1)) <= 2.0 ** -4


def test_hadamard_transform_is_orthogonal_and_keeps_scores():
    for d in (2, 8, 64, 128):
        H = fp8.hadamard(d)
        assert np.array_equal(np.abs(H), np.ones((d, d))) and np.array_equal(H, H.T)
        assert np.array_equal(H @ H.T, d * np.eye(d))
    rng = np.random.default_rng(3)
    signs = np.where(rng.standard_normal(64) > 0, 1.0, -1.0)
    Q, K = rng.standard_normal((50, 64)), rng.standard_normal((70, 64))
    Qt, Kt = fp8.incoherent(Q, signs), fp8.incoherent(K, signs)
    assert np.max(np.abs(Qt @ Kt.T - Q @ K.T)) <= 1e-12
    assert np.allclose(np.linalg.norm(Qt, axis=1), np.linalg.norm(Q, axis=1), rtol=1e-14)
    # a one-hot outlier spreads evenly: every column gets |a| / sqrt(d)
    x = np.zeros((1, 64))
    x[0, 17] = 40.0
    assert np.allclose(np.abs(fp8.incoherent(x, signs)), 40.0 / 8.0, rtol=0, atol=1e-13)


def test_block_quantisation():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((2, 300, 64)) * np.array([1.0, 30.0])[:, None, None]
    X[0, 128:256] = 0.0  # an all-zero block
    q, s = fp8.quantize_blocks(X, 128)
    assert s.shape == (2, 3) and s[0, 1] == 1.0 and np.all(q[0, 128:256] == 0)
    for h in range(2):
        for b in range(3):
            blk = q[h, 128 * b:128 * (b + 1)]
            if s[h, b] != 1.0 or np.any(blk):
                assert np.max(np.abs(blk)) == 448.0
    deq = q * np.repeat(s, 128, axis=-1)[..., :300, None]
    step = np.maximum(np.abs(X) * 2.0 ** -4, np.repeat(s, 128, axis=-1)[..., :300, None] * 2.0 ** -10)
    assert np.all(np.abs(deq - X) <= step * (1 + 1e-12))


def test_forward_fp8_closed_forms():
    rng = np.random.default_rng(5)
    signs = np.where(rng.standard_normal(64) > 0, 1.0, -1.0)
    Q, K = rng.standard_normal((40, 64)), rng.standard_normal((300, 64))
    O, _ = fp8.forward_fp8(Q, K, np.ones((300, 64)), 0.125, False, signs)
    assert np.allclose(O, 1.0, rtol=0, atol=1e-14)
    V1 = rng.standard_normal((1, 64))
    O1, L1 = fp8.forward_fp8(Q, K[:1], V1, 0.125, False, signs)
    v8, sv = fp8.quantize_blocks(V1, 1)
    assert np.allclose(O1, v8 * sv[0], rtol=0, atol=1e-14)
    # causal row 0 sees key 0 only
    Oc, _ = fp8.forward_fp8(rng.standard_normal((300, 64)), K, K, 0.125, True, signs)
    k8, sk = fp8.quantize_blocks(K, 300)
    assert np.allclose(Oc[0], k8[0] * sk[0], rtol=0, atol=1e-14)


@pytest.mark.parametrize("N,causal", [(512, False), (512, True), (1024, False)])
def test_forward_fp8_error_within_tolerance(N, causal):
    """The FP8 method itself against exact attention on the workload's inputs (fp16 N(0,1),
    scale 1/8): RMSE (rows seeing 256 keys or more) within the pages' FP8 figure, max |error|
    within the fp16 bound times the E4M3/fp16 unit-roundoff ratio."""
    q, k, v = synth.attention_inputs(1, 2, N, N, 64, "f16", seed=N)
    q, k, v = (synth.to_f64(x, "f16") for x in (q, k, v))
    signs = np.where(np.random.default_rng(6).standard_normal(64) > 0, 1.0, -1.0)
    Oe, Le = oracle.forward(q, k, v, 0.125, causal)
    Of, Lf = fp8.forward_fp8(q, k, v, 0.125, causal, signs)
    for h in range(2):
        assert fp8_rmse(Of[0, h] - Oe[0, h], N, causal) <= TOL_FP8["rmse"]
    assert np.max(np.abs(Of - Oe)) <= TOL_FP8["max_abs"]
    assert np.max(np.abs(Lf - Le)) <= TOL_FP8["lse"]


def _no_normalisation(X, signs):
    X = np.asarray(X, dtype=np.float64)
    return (X * np.asarray(signs)) @ fp8.hadamard(X.shape[-1])


def _hadamard_without_sign_flip(d):
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, H]])  # the lower-right block should be -H
    return H


@pytest.mark.parametrize("name,mutant", [("incoherent", _no_normalisation), ("hadamard", _hadamard_without_sign_flip)])
def test_planted_transform_mistakes_fail_a_pin(monkeypatch, name, mutant):
    monkeypatch.setattr(fp8, name, mutant)
    with pytest.raises(AssertionError):
        test_hadamard_transform_is_orthogonal_and_keeps_scores()
