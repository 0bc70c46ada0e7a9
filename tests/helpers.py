"""Test helpers: moving synth arrays to the GPU and comparing results with the oracle."""
from __future__ import annotations

import numpy as np

from exact_attention_gb300 import synth

TORCH_DT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}

# Tolerances stated for this method: max |GPU - oracle| on O, on the gradients and on LSE.
# bf16 gradients have no stated bound: the fp16 one scaled by the ratio of the two types' unit
# roundoffs (2^-8 / 2^-11 = 8), since the same rounding steps (P and dS rounded once to the I/O
# type, outputs rounded once) dominate both.
TOL_O = {"f32": 1e-4, "f16": 2e-3, "bf16": 1e-2}
TOL_GRAD = {"f16": 1e-2, "bf16": 8e-2}
TOL_LSE = 1e-4
# The FP8 forward (E4M3 operands, fp16/bf16 I/O). Against exact attention: max |O error| within the
# fp16 bound times the E4M3/fp16 unit-roundoff ratio (2^-4 / 2^-11 = 128); RMSE of O within the FP8
# figure the "Flash Attention" notes print for FlashAttention-3's block quantisation with incoherent
# processing (9.1e-3), over the rows that see at least 256 keys (the figure is a long-sequence one:
# a row with a handful of keys does not average its weights' 2^-4 roundings); LSE within 0.2, four
# times the largest score error E4M3 operands give unit-variance rows of d = 64 at scale 1/8.
# Against the oracle's FP8 steps (same E4M3 operands): the same O bounds, and LSE within 1e-3 (f32
# against f64 scores of identical operands, plus the rare operand that lands on the other side of
# a rounding boundary in the f32 transform).
TOL_FP8 = {"rmse": 9.1e-3, "max_abs": 0.256, "lse": 0.2, "lse_steps": 1e-3, "rmse_min_keys": 256}


def fp8_rmse(err, n_keys: int, causal: bool):
    """RMSE of err [M, d] over the rows that see at least TOL_FP8["rmse_min_keys"] of the n_keys
    keys (row i sees i + 1 of them when causal), or None when no row does."""
    import numpy as np
    M = err.shape[-2]
    seen = np.minimum(np.arange(M) + 1, n_keys) if causal else np.full(M, n_keys)
    rows = seen >= TOL_FP8["rmse_min_keys"]
    if not np.any(rows):
        return None
    return float(np.sqrt(np.mean(err[rows] ** 2)))
REL_L2_F32 = 1e-5


def to_device(a: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda()


def to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def errs(got: np.ndarray, ref: np.ndarray):
    d = np.abs(got - ref)
    rel_l2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    return float(d.max()) if d.size else 0.0, rel_l2


def assert_close(got, ref, atol: float, what: str, rel_l2: float | None = None):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    mx, rl = errs(got, ref)
    assert mx <= atol, f"{what}: max abs err {mx:.3e} > {atol:.1e} (rel L2 {rl:.3e})"
    if rel_l2 is not None:
        assert rl <= rel_l2, f"{what}: rel L2 {rl:.3e} > {rel_l2:.1e} (max abs {mx:.3e})"
    return mx, rl


def f64(a, dtype):
    return synth.to_f64(a, dtype)
