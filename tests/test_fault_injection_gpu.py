"""Failure detection without a GPU fault: a bounded wait is made to run out on purpose.

The injection makes the first decode CTA skip loading its first stage of keys, so its compute
warps wait on a barrier that never completes. With a 20 ms wait budget the wait gives up, the CTA
drains and exits, and the host reads FA_ERR_TIMEOUT naming the kernel and the wait site. Nothing
traps or faults, and the following normal call must still match the oracle.
"""
from __future__ import annotations

import math

import pytest

import oracle
import exact_attention_gb300 as fa
from exact_attention_gb300 import synth

from helpers import TOL_GRAD, TOL_O, assert_close, f64, to_device, to_f64

pytestmark = pytest.mark.gpu

DEFAULT_BUDGET_NS = 2_000_000_000


def test_bounded_wait_reports_timeout_and_context_survives():
    B, H, N, D, ns = 1, 2, 4096, 128, 4
    q, k, v = synth.decode_inputs(B, H, N, D, "bf16", 7)
    qd, kd, vd = to_device(q, "bf16"), to_device(k, "bf16"), to_device(v, "bf16")
    scale = 1.0 / math.sqrt(D)
    assert fa.fa_set_wait_budget_ns(20_000_000) == fa.FA_OK
    try:
        assert fa.fa_debug_inject(1) == fa.FA_OK
        fa.decode(qd, kd, vd, scale, ns)
        status = fa.fa_last_status()
        msg = fa.fa_last_error_message()
        assert status == fa.FA_ERR_TIMEOUT, (status, msg)
        assert "decode_split" in msg and "block 0" in msg, msg
        # the status word was cleared by reading it
        assert fa.fa_last_status() == fa.FA_OK
    finally:
        fa.fa_debug_inject(0)
        fa.fa_set_wait_budget_ns(DEFAULT_BUDGET_NS)
    out, _ = fa.decode(qd, kd, vd, scale, ns)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    ref = oracle.decode(f64(q, "bf16"), f64(k, "bf16"), f64(v, "bf16"), scale)
    assert_close(to_f64(out), ref, TOL_O["bf16"], "decode after the injected timeout")


def _forward_after_timeout(B, H, M, N, kind, split):
    """Arms injection `kind`, runs one forward with a 20 ms wait budget, returns the status and its
    message; then runs the same forward normally and checks it against the oracle."""
    q, k, v = synth.attention_inputs(B, H, M, N, 64, "f16", seed=kind)
    qd, kd, vd = to_device(q, "f16"), to_device(k, "f16"), to_device(v, "f16")
    assert fa.fa_set_wait_budget_ns(20_000_000) == fa.FA_OK
    try:
        assert fa.fa_debug_inject(kind) == fa.FA_OK
        with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1 if split else 0):
            fa.forward(qd, kd, vd, 0.125, False)
        status = fa.fa_last_status()
        msg = fa.fa_last_error_message()
        assert fa.fa_last_status() == fa.FA_OK  # reading the status word cleared it
    finally:
        fa.fa_debug_inject(0)
        fa.fa_set_wait_budget_ns(DEFAULT_BUDGET_NS)
    with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1 if split else 0):
        out, lse = fa.forward(qd, kd, vd, 0.125, False)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    for b, h in ((0, 0), (B - 1, H - 1)):
        ro, _ = oracle.forward(f64(q[b, h], "f16"), f64(k[b, h], "f16"), f64(v[b, h], "f16"), 0.125, False)
        assert_close(to_f64(out)[b, h], ro, TOL_O["f16"], f"forward after the injected timeout [{b},{h}]")
    return status, msg


def test_forward_stage_wait_times_out_and_context_survives():
    """A wait inside one CTA: the first CTA's first K/V stage is never loaded, so the MMA issuers'
    and softmax warps' bounded waits on it run out."""
    status, msg = _forward_after_timeout(1, 2, 512, 512, 2, split=False)
    assert status == fa.FA_ERR_TIMEOUT, (status, msg)
    assert "kernel fwd " in msg and "block 0" in msg, msg


def test_forward_split_flag_wait_times_out_and_context_survives():
    """A wait between CTAs: on the split schedule CTA 1 never publishes the partial of its first
    piece (a later part of a pair CTA 0 finishes), so CTA 0's softmax warps wait on its flags (wait
    site 36) and CTA 0's epilogue warp waits on them (site 37); whichever budget runs out first is
    the one reported, in block 0."""
    status, msg = _forward_after_timeout(4, 12, 2048, 2048, 3, split=True)
    assert status == fa.FA_ERR_TIMEOUT, (status, msg)
    assert "kernel fwd " in msg and "block 0" in msg, msg
    assert "wait site 36 " in msg or "wait site 37 " in msg, msg


def test_backward_split_count_wait_times_out_and_context_survives():
    """A wait between CTAs in the fused backward: on its split schedule the lowest CTA whose share
    starts inside a key tile never counts its partial in, so the CTA holding that key tile's first
    query blocks gives up: its compute warps' wait for the count (wait site 39) or its drain warp's
    wait for the dV/dK tiles those warps never stage (site 38), which began earlier and so usually
    runs out first. The next call, whose delta kernel zeroes the counters again, must match the
    oracle."""
    import torch

    B, H, M, N = 2, 3, 1024, 1024
    q, k, v, do = synth.attention_inputs(B, H, M, N, 64, "f16", seed=39, with_dout=True)
    qd, kd, vd, dod = (to_device(x, "f16") for x in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, 0.125, False)
    # the CTA expected to report: the holder of the first blocks of the key tile that CTA c cuts
    G = torch.cuda.get_device_properties(0).multi_processor_count
    nqb = M // 128
    units = B * H * (N // 128) * nqb
    c = next(c for c in range(1, G) if (c * units // G) % nqb != 0)
    assert fa.fa_set_wait_budget_ns(20_000_000) == fa.FA_OK
    try:
        with fa.schedule(fa.FA_SCHED_BWD_SPLIT, 1):
            assert fa.fa_debug_inject(4) == fa.FA_OK
            fa.backward(qd, kd, vd, o, dod, lse, 0.125, False, fused=True)
            status = fa.fa_last_status()
            msg = fa.fa_last_error_message()
            assert fa.fa_last_status() == fa.FA_OK
            fa.fa_debug_inject(0)
            fa.fa_set_wait_budget_ns(DEFAULT_BUDGET_NS)
            dq, dk, dv, _ = fa.backward(qd, kd, vd, o, dod, lse, 0.125, False, fused=True)
            assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    finally:
        fa.fa_debug_inject(0)
        fa.fa_set_wait_budget_ns(DEFAULT_BUDGET_NS)
    assert status == fa.FA_ERR_TIMEOUT, (status, msg)
    assert "kernel bwd_dkdv " in msg and f"block {c - 1}" in msg, msg
    assert "wait site 39 " in msg or "wait site 38 " in msg, msg
    grads = (to_f64(dq), to_f64(dk), to_f64(dv))
    for b, h in ((0, 0), (B - 1, H - 1)):
        ref = oracle.backward(f64(q[b, h], "f16"), f64(k[b, h], "f16"), f64(v[b, h], "f16"), f64(do[b, h], "f16"),
                              0.125, False)
        for n, (g, r) in enumerate(zip(grads, ref)):
            assert_close(g[b, h], r, TOL_GRAD["f16"], f"{'dQ dK dV'.split()[n]}[{b},{h}] after the injected timeout")
