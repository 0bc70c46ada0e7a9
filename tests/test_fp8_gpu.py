"""FP8 forward on the GPU (fa_fwd_fp8, D = 64): against exact attention (the oracle's definition)
within the stated FP8 tolerance, against the oracle's FP8 steps, and its quantised operands (the
workspace) against the oracle's transform and block quantisation."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import exact_attention_gb300 as fa
from exact_attention_gb300 import synth
from oracle import fp8

from helpers import TOL_FP8, f64, fp8_rmse, to_device, to_f64

pytestmark = pytest.mark.gpu


def run_fp8(B, H, M, N, dtype, causal, scale, seed):
    import torch
    q, k, v = synth.attention_inputs(B, H, M, N, 64, dtype, seed=seed)
    signs = synth.hadamard_signs(64, seed)
    sd = torch.from_numpy(signs).cuda()
    out, lse, ws = fa.forward_fp8(to_device(q, dtype), to_device(k, dtype), to_device(v, dtype), scale, causal, sd)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    return (q, k, v), signs, to_f64(out), to_f64(lse), ws


def check_fp8(inputs, signs, out, lse, dtype, causal, scale):
    q, k, v = inputs
    B, H = q.shape[:2]
    worst = {}
    for b in range(B):
        for h in range(H):
            qh, kh, vh = f64(q[b, h], dtype), f64(k[b, h], dtype), f64(v[b, h], dtype)
            Oe, Le = oracle.forward(qh, kh, vh, scale, causal)
            Of, Lf = fp8.forward_fp8(qh, kh, vh, scale, causal, signs)
            o, l_ = out[b, h], lse[b, h]
            assert np.all(np.isfinite(o)) and np.all(np.isfinite(l_))
            for name, ref in (("exact", Oe), ("fp8 steps", Of)):
                mx = float(np.max(np.abs(o - ref)))
                assert mx <= TOL_FP8["max_abs"], f"O[{b},{h}] vs {name}: max {mx:.3e}"
                rmse = fp8_rmse(o - ref, kh.shape[0], causal)
                if rmse is not None:
                    assert rmse <= TOL_FP8["rmse"], f"O[{b},{h}] vs {name}: rmse {rmse:.3e}"
                    worst[name] = max(worst.get(name, 0.0), rmse)
            dl = float(np.max(np.abs(l_ - Le)))
            assert dl <= TOL_FP8["lse"], f"LSE[{b},{h}] vs exact: {dl:.3e}"
            dl = float(np.max(np.abs(l_ - Lf)))
            assert dl <= TOL_FP8["lse_steps"], f"LSE[{b},{h}] vs fp8 steps: {dl:.3e}"
    return worst


SHAPES = [
    (1, 2, 256, 256),
    (1, 2, 300, 200),    # ragged M and N (the transposed V padded to 16 keys)
    (2, 3, 1000, 900),
    (1, 1, 5, 700),
    (1, 2, 1024, 1024),
    (1, 1, 128, 33),     # N not a multiple of 16
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,M,N", SHAPES)
def test_fp8_forward_matches_oracle(dtype, causal, B, H, M, N):
    inputs, signs, out, lse, _ = run_fp8(B, H, M, N, dtype, causal, 0.125, seed=M + 3 * N)
    check_fp8(inputs, signs, out, lse, dtype, causal, 0.125)


def test_fp8_forward_negative_scale():
    inputs, signs, out, lse, _ = run_fp8(1, 2, 384, 300, "f16", False, -0.125, seed=4)
    check_fp8(inputs, signs, out, lse, "f16", False, -0.125)


def test_fp8_forward_workload_heads():
    """The fp16 workload's shape (B4 H12 M=N=2048), checked on sampled heads."""
    q, k, v = synth.attention_inputs(4, 12, 2048, 2048, 64, "f16", seed=0)
    signs = synth.hadamard_signs(64, 0)
    import torch
    out, lse, _ = fa.forward_fp8(to_device(q, "f16"), to_device(k, "f16"), to_device(v, "f16"), 0.125, False,
                                 torch.from_numpy(signs).cuda())
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    o, l_ = to_f64(out), to_f64(lse)
    sub = lambda a: a[[0, 3], :][:, [0, 11]]  # noqa: E731
    check_fp8((sub(q), sub(k), sub(v)), signs, sub(o), sub(l_), "f16", False, 0.125)


def _e4m3_decode(b: np.ndarray) -> np.ndarray:
    mag = fp8._e4m3_positive_values()[b & 0x7F]
    return np.where(b & 0x80, -mag, mag)


def test_fp8_quantised_operands_match_the_oracle():
    """The workspace's E4M3 copies of Q M, K M and V, and their scales, against the oracle's
    transform and block quantisation: the scales agree to f32 rounding, and every element is the
    oracle's E4M3 value or (where the f32 transform lands next to a rounding boundary) one
    E4M3 step from it."""
    B, H, M, N = 1, 2, 300, 200
    (q, k, v), signs, _, _, ws = run_fp8(B, H, M, N, "f16", False, 0.125, seed=5)
    w = ws.cpu().numpy()
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    BH, npad, nqb, nkb = B * H, (N + 15) // 16 * 16, (M + 127) // 128, (N + 127) // 128
    o_k8 = a256(BH * M * 64)
    o_vt = o_k8 + a256(BH * N * 64)
    o_sq = o_vt + a256(BH * 64 * npad)
    o_sk = o_sq + a256(BH * nqb * 4)
    o_sv = o_sk + a256(BH * nkb * 4) + a256(BH * nkb * 4)
    q8 = _e4m3_decode(w[:BH * M * 64].reshape(B, H, M, 64))
    k8 = _e4m3_decode(w[o_k8:o_k8 + BH * N * 64].reshape(B, H, N, 64))
    vt8 = _e4m3_decode(w[o_vt:o_vt + BH * 64 * npad].reshape(B, H, 64, npad))
    sq = w[o_sq:o_sq + BH * nqb * 4].view(np.float32).reshape(B, H, nqb)
    sk = w[o_sk:o_sk + BH * nkb * 4].view(np.float32).reshape(B, H, nkb)
    sv = w[o_sv:o_sv + BH * 4].view(np.float32).reshape(B, H)
    rq, rsq = fp8.quantize_blocks(fp8.incoherent(f64(q, "f16"), signs), 128)
    rk, rsk = fp8.quantize_blocks(fp8.incoherent(f64(k, "f16"), signs), 128)
    rv, rsv = fp8.quantize_blocks(f64(v, "f16"), N)
    for got, ref in ((sq, rsq), (sk, rsk), (sv, rsv[..., 0])):
        assert np.allclose(got, ref, rtol=1e-6, atol=0)
    for got, ref in ((q8, rq), (k8, rk), (np.swapaxes(vt8[..., :N], -1, -2), rv)):
        step = np.maximum(np.abs(ref) * 2.0 ** -3, 2.0 ** -9)
        assert np.all(np.abs(got - ref) <= step)
        assert np.mean(got == ref) >= 0.999
    assert np.all(vt8[..., N:] == 0)  # the padding keys are zero
