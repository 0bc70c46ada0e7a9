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

from helpers import TOL_O, assert_close, f64, to_device, to_f64

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
