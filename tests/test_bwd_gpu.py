"""Backward pass on the GPU against the fp64 oracle: dQ, dK, dV and the delta workspace."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import exact_attention_gb300 as fa
from exact_attention_gb300 import synth

from helpers import TOL_GRAD, assert_close, f64, to_device, to_f64

pytestmark = pytest.mark.gpu


def run_bwd(B, H, M, N, D, dtype, causal, scale, seed=0, std=1.0, fused=False):
    q, k, v, do = synth.attention_inputs(B, H, M, N, D, dtype, seed=seed, std=std, with_dout=True)
    qd, kd, vd, dod = (to_device(x, dtype) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, scale, causal)
    if fused in (False, "pair"):  # fa_bwd, its D = 64 gradient kernels on single CTAs or on CTA pairs
        with fa.schedule(fa.FA_SCHED_BWD_PAIR, 1 if fused == "pair" else 0):
            dq, dk, dv, delta = fa.backward(qd, kd, vd, o, dod, lse, scale, causal)
    else:
        dq, dk, dv, delta = fa.backward(qd, kd, vd, o, dod, lse, scale, causal, fused=fused)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    return (q, k, v, do), to_f64(o), (to_f64(dq), to_f64(dk), to_f64(dv)), to_f64(delta)


def check(inputs, o_gpu, grads, delta, dtype, causal, scale, heads=None):
    q, k, v, do = inputs
    B, H = q.shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    worst = [0.0, 0.0, 0.0]
    for b, h in heads:
        ref = oracle.backward(f64(q[b, h], dtype), f64(k[b, h], dtype), f64(v[b, h], dtype), f64(do[b, h], dtype),
                              scale, causal)
        for n, (g, r) in enumerate(zip(grads, ref)):
            mx, _ = assert_close(g[b, h], r, TOL_GRAD[dtype], f"{'dQ dK dV'.split()[n]}[{b},{h}] {dtype} "
                                 f"causal={causal}")
            worst[n] = max(worst[n], mx)
        # delta is rowsum(dO o O) of the stored O (the tutorial's delta kernel)
        dref = oracle.delta(o_gpu[b, h], f64(do[b, h], dtype))
        assert_close(delta[b, h], dref, 1e-4 * max(1.0, float(np.max(np.abs(dref)))), f"delta[{b},{h}]")
    return worst


# fused: fa_bwd_ws (dQ formed in the dK/dV pass and accumulated in f32 for D = 64) instead of fa_bwd;
# "3kernels" / "pair": fa_bwd with its D = 64 dK/dV and dQ kernels on single CTAs / on CTA pairs
# (forced either way; the same kernels at D = 128)
FUSED = pytest.mark.parametrize("fused", [False, "pair", True], ids=["3kernels", "pair", "fused"])


@FUSED
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("std", [1.0, 0.5])
def test_backward_tutorial_shape(causal, std, fused):
    """Z=1, H=2, N_CTX=1024, D=64, sm_scale 0.5, fp16, N(0,1) and N(0, 0.5^2)."""
    inputs, o, grads, delta = run_bwd(1, 2, 1024, 1024, 64, "f16", causal, 0.5, seed=20, std=std, fused=fused)
    check(inputs, o, grads, delta, "f16", causal, 0.5)


@FUSED
@pytest.mark.parametrize("causal", [False, True])
def test_backward_tutorial_shape_bf16(causal, fused):
    """The tutorial's shape in bf16 with N(0,1) inputs and sm_scale 0.5, the most peaked case the
    workloads hold: |dQ|, |dK| reach about 14, where one bf16 output rounding alone is up to 2^-5."""
    inputs, o, grads, delta = run_bwd(1, 2, 1024, 1024, 64, "bf16", causal, 0.5, seed=20, fused=fused)
    check(inputs, o, grads, delta, "bf16", causal, 0.5)


SHAPES = [
    (1, 1, 128, 128),
    (1, 2, 256, 384),
    (2, 1, 300, 200),
    (1, 1, 129, 129),
    (1, 1, 1, 1),
    (1, 1, 77, 333),
    (1, 1, 333, 77),
]


@FUSED
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,M,N", SHAPES)
def test_backward_matches_oracle(dtype, D, causal, B, H, M, N, fused):
    scale = 1.0 / math.sqrt(D)
    inputs, o, grads, delta = run_bwd(B, H, M, N, D, dtype, causal, scale, seed=M * 7 + N, fused=fused)
    check(inputs, o, grads, delta, dtype, causal, scale)


@FUSED
@pytest.mark.parametrize("D", [64, 128])
def test_backward_causal_keys_past_every_query(D, fused):
    """Causal with N > M and more key tiles than SMs: a CTA takes a key tile that some query sees
    and then one past every query (no query block: zero gradients, no accumulators to hand
    over). The accumulators-final barrier must advance only for the first, or the compute warps'
    parity wait would see it two phases ahead; and every thread arriving on the barrier that frees
    K and V must first wait for them, or its arrivals for such tiles run ahead of the loads."""
    B, H, M, N = 4, 50, 128, 1024
    scale = 1.0 / math.sqrt(D)
    inputs, o, grads, delta = run_bwd(B, H, M, N, D, "f16", True, scale, seed=17, fused=fused)
    check(inputs, o, grads, delta, "f16", True, scale, heads=[(0, 0), (1, 31), (3, 49)])
    # keys past the last query get nothing
    assert np.all(grads[1][:, :, M:] == 0) and np.all(grads[2][:, :, M:] == 0)


def test_backward_gradient_identities():
    """sum_j dK_j = 0 (rows of dS sum to zero) and sum_j dV_j = sum_i dO_i."""
    inputs, o, (dq, dk, dv), _ = run_bwd(1, 2, 512, 512, 64, "f16", True, 0.125, seed=3)
    do = f64(inputs[3], "f16")
    assert np.max(np.abs(dk.sum(axis=2))) < 0.05
    assert np.max(np.abs(dv.sum(axis=2) - do.sum(axis=2))) < 0.05


@FUSED
@pytest.mark.parametrize("causal", [False, True])
def test_backward_full_workload_sampled_heads(causal, fused):
    """B4 H12 M=N=2048 D64 fp16 (the measured workload): every gradient entry of three heads
    spread over the batch against the oracle."""
    inputs, o, grads, delta = run_bwd(4, 12, 2048, 2048, 64, "f16", causal, 0.125, seed=5, fused=fused)
    check(inputs, o, grads, delta, "f16", causal, 0.125, heads=[(0, 0), (1, 7), (3, 11)])


def test_backward_fused_matches_three_kernels():
    """The fused pass gives dK and dV identical to the three kernels (same products, same order)
    and dQ equal up to the f32 summation order of its key blocks."""
    import torch
    for causal in (False, True):
        q, k, v, do = synth.attention_inputs(2, 3, 700, 900, 64, "f16", seed=11, with_dout=True)
        qd, kd, vd, dod = (to_device(x, "f16") for x in (q, k, v, do))
        o, lse = fa.forward(qd, kd, vd, 0.125, causal)
        a = fa.backward(qd, kd, vd, o, dod, lse, 0.125, causal)
        b = fa.backward(qd, kd, vd, o, dod, lse, 0.125, causal, fused=True)
        assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2]), causal
        assert torch.equal(a[3], b[3])  # delta
        assert float((a[0].float() - b[0].float()).abs().max()) <= 4e-3, causal


PAIR_SHAPES = [
    # B, H, M, N: one key tile per pair with an empty second half, ragged tails, more pair items
    # than pairs (the persistent loop), heads whose key range ends inside a pair
    (1, 1, 128, 128),
    (1, 1, 5, 700),
    (2, 3, 700, 900),
    (1, 2, 1024, 1024),
    (4, 12, 512, 512),
    (1, 3, 2048, 384),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,M,N", PAIR_SHAPES)
def test_backward_pair_matches_single_cta(dtype, causal, B, H, M, N):
    """fa_bwd's dK/dV and dQ kernels on CTA pairs against the single-CTA kernels on the same inputs
    (the same products, the same rounding points), then against the oracle."""
    import torch
    scale = 0.125
    q, k, v, do = synth.attention_inputs(B, H, M, N, 64, dtype, seed=M + 3 * N + H, with_dout=True)
    qd, kd, vd, dod = (to_device(x, dtype) for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, scale, causal)
    with fa.schedule(fa.FA_SCHED_BWD_PAIR, 0):
        a = fa.backward(qd, kd, vd, o, dod, lse, scale, causal)
    with fa.schedule(fa.FA_SCHED_BWD_PAIR, 1):
        b = fa.backward(qd, kd, vd, o, dod, lse, scale, causal)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    # dK and dV: the same products with the same rounding points, bit for bit; delta: the same
    # kernel; dQ: the same products, whose f32 sums can differ between runs in the last bit
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    assert float((a[0].float() - b[0].float()).abs().max()) <= 1e-3 * max(1.0, float(a[0].float().abs().max()))
    heads = [(0, 0), (B - 1, H - 1)]
    check((q, k, v, do), to_f64(o), (to_f64(b[0]), to_f64(b[1]), to_f64(b[2])), to_f64(b[3]), dtype, causal,
          scale, heads=heads)


SPLIT_SHAPES = [
    # B, H, M, N
    (1, 2, 1024, 1024),  # the tutorial's shape
    (2, 3, 384, 256),
    (1, 2, 300, 700),    # ragged M and N
    (1, 1, 8192, 256),   # 128 units for more CTAs: empty ranges, one key tile over many CTAs
    (3, 5, 640, 1000),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("B,H,M,N", SPLIT_SHAPES)
def test_backward_fused_split_schedule_matches_oracle(dtype, B, H, M, N):
    """The fused pass's split schedule forced on: every SM an equal share of the (key tile,
    query block) units; a key tile cut by a share boundary gets the partial dK/dV of the SMs
    holding its later query blocks added in by the SM holding its first ones."""
    with fa.schedule(fa.FA_SCHED_BWD_SPLIT, 1):
        inputs, o, grads, delta = run_bwd(B, H, M, N, 64, dtype, False, 0.125, seed=M + N, fused=True)
    check(inputs, o, grads, delta, dtype, False, 0.125)


def test_backward_fused_split_agrees_with_whole_tiles():
    """Split and whole key tiles run the same products; dK and dV differ only in the f32
    order in which a cut tile's two sums meet, dQ in the order of its reduce-adds."""
    import torch
    q, k, v, do = synth.attention_inputs(2, 3, 1000, 900, 64, "f16", seed=12, with_dout=True)
    qd, kd, vd, dod = (to_device(x, "f16") for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, 0.125, False)
    with fa.schedule(fa.FA_SCHED_BWD_SPLIT, 0):
        a = fa.backward(qd, kd, vd, o, dod, lse, 0.125, False)
    with fa.schedule(fa.FA_SCHED_BWD_SPLIT, 1):
        b = fa.backward(qd, kd, vd, o, dod, lse, 0.125, False)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    for n in range(3):
        assert float((a[n].float() - b[n].float()).abs().max()) <= 4e-3, n
    assert torch.equal(a[3], b[3])  # delta


def test_backward_fused_split_reused_workspace():
    """Three calls on one workspace: the ready flags the previous call left set are cleared by
    the next call's delta kernel before its fused pass reads them."""
    import torch
    B, H, M, N, D = 1, 3, 512, 640, 64
    nbytes = fa.fa_bwd_ws_workspace_bytes(B, H, M, D)
    ws = torch.empty((nbytes // 4,), dtype=torch.float32, device="cuda")
    for seed in (1, 2, 3):
        q, k, v, do = synth.attention_inputs(B, H, M, N, D, "f16", seed=seed, with_dout=True)
        qd, kd, vd, dod = (to_device(x, "f16") for x in (q, k, v, do))
        o, lse = fa.forward(qd, kd, vd, 0.125, False)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        with fa.schedule(fa.FA_SCHED_BWD_SPLIT, 1):
            st = fa.fa_bwd_ws(qd, kd, vd, o, dod, lse, dq, dk, dv, ws, nbytes, B, H, M, N, D, 0.125, False, fa.FA_F16)
        assert st == fa.FA_OK, fa.fa_last_error_message()
        torch.cuda.synchronize()
        check((q, k, v, do), to_f64(o), (to_f64(dq), to_f64(dk), to_f64(dv)), to_f64(ws[: B * H * M].view(B, H, M)),
              "f16", False, 0.125)


NEG_CASES = [
    # B, H, M, N, D, dtype, causal, scale
    (1, 2, 384, 300, 64, "f16", False, -0.5),
    (1, 2, 300, 384, 64, "f16", True, -0.125),
    (1, 2, 256, 256, 64, "bf16", False, -0.125),
    (1, 2, 300, 300, 128, "f16", True, -1 / math.sqrt(128)),
]


@FUSED
@pytest.mark.parametrize("B,H,M,N,D,dtype,causal,scale", NEG_CASES)
def test_backward_negative_scale(B, H, M, N, D, dtype, causal, scale, fused):
    """scale < 0: the score products are negated in the tensor core, the exponent uses |scale|
    and dK, dQ take the signed scale; compared with the oracle's chain rule at that scale."""
    inputs, o, grads, delta = run_bwd(B, H, M, N, D, dtype, causal, scale, seed=M + 2 * N, fused=fused)
    check(inputs, o, grads, delta, dtype, causal, scale)


def test_backward_negative_scale_split_forced():
    with fa.schedule(fa.FA_SCHED_BWD_SPLIT, 1):
        inputs, o, grads, delta = run_bwd(2, 3, 1000, 900, 64, "f16", False, -0.125, seed=9, fused=True)
    check(inputs, o, grads, delta, "f16", False, -0.125)


def test_backward_zero_scale():
    """scale = 0: every visible key gets the same weight; dK and dQ are exactly zero."""
    inputs, o, grads, delta = run_bwd(1, 2, 256, 300, 64, "f16", True, 0.0, seed=3, fused=True)
    check(inputs, o, grads, delta, "f16", True, 0.0)
    assert np.all(grads[0] == 0) and np.all(grads[1] == 0)
