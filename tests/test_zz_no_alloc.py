"""fa_decode_static: decode for callers that cannot allocate device memory.

Such callers (an allocator that must not grow, a runtime that owns every buffer,
a C caller without an allocator) get their split partials kept in the
library's own fixed scratch array instead of a workspace they pass in. This
file runs last so that a failure here leaves every other test already run; it
passes on its own in a fresh process too, since the first call on the device
does the one-time set-up.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import exact_attention_gb300 as fa
from exact_attention_gb300 import synth

from helpers import TOL_O, assert_close, to_device, to_f64

pytestmark = pytest.mark.gpu

DT = {"f32": fa.FA_F32, "f16": fa.FA_F16, "bf16": fa.FA_BF16}


def _decode_both(B, H, N, D, dtype, ns, seed):
    import torch
    q, k, v = synth.decode_inputs(B, H, N, D, dtype, seed)
    qd, kd, vd = to_device(q, dtype), to_device(k, dtype), to_device(v, dtype)
    scale = 1.0 / math.sqrt(D)
    ref = torch.empty_like(qd)
    ws = torch.empty(fa.fa_decode_workspace_bytes(B, H, D, ns) // 4, dtype=torch.float32, device="cuda")
    assert fa.fa_decode(qd, kd, vd, ref, ws, B, H, N, D, scale, ns, DT[dtype]) == fa.FA_OK
    out = torch.full_like(qd, float("nan"))
    s = fa.fa_decode_static(qd, kd, vd, out, B, H, N, D, scale, ns, DT[dtype])
    assert s == fa.FA_OK, fa.fa_last_error_message()
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    # the fp64 oracle on the same inputs, head by head
    want = np.stack([[oracle.decode(synth.to_f64(q[b, h], dtype), synth.to_f64(k[b, h], dtype),
                                    synth.to_f64(v[b, h], dtype), scale) for h in range(H)] for b in range(B)])
    return to_f64(out), to_f64(ref), want


def test_static_decode_matches_workspace_decode_twice_in_a_row():
    # two different problems back to back through the shared scratch
    got1, ref1, want1 = _decode_both(2, 4, 3000, 128, "bf16", 16, seed=11)
    got2, ref2, want2 = _decode_both(1, 3, 777, 64, "f16", 5, seed=12)
    assert_close(got1, want1.reshape(got1.shape), TOL_O["bf16"], "static decode vs oracle, first call")
    assert_close(got2, want2.reshape(got2.shape), TOL_O["f16"], "static decode vs oracle, second call")
    # the same kernels run on the same data: the results agree exactly
    assert np.array_equal(got1, ref1) and np.array_equal(got2, ref2)


def test_static_decode_rejects_requests_above_its_scratch():
    # B=8, H=32, D=128, 256 splits needs 8.5 M floats > 4 M: refused before any launch
    s = fa.fa_decode_static(1 << 20, 1 << 20, 1 << 20, 1 << 20, 8, 32, 32768, 128, 0.1, 256, fa.FA_BF16)
    assert s == fa.FA_ERR_INVALID
    assert "fixed scratch" in fa.fa_last_error_message()
