"""Forward pass on the GPU against the fp64 oracle: O and LSE."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import exact_attention_gb300 as fa
from exact_attention_gb300 import synth

from helpers import TOL_LSE, TOL_O, REL_L2_F32, assert_close, errs, f64, to_device, to_f64

pytestmark = pytest.mark.gpu


def run_fwd(B, H, M, N, D, dtype, causal, scale, seed=0, std=1.0):
    q, k, v = synth.attention_inputs(B, H, M, N, D, dtype, seed=seed, std=std)
    out, lse = fa.forward(to_device(q, dtype), to_device(k, dtype), to_device(v, dtype), scale, causal)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    return (q, k, v), to_f64(out), to_f64(lse)


def check_heads(inputs, out, lse, dtype, causal, scale, heads=None, rel_l2=None):
    q, k, v = inputs
    B, H = q.shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    worst = (0.0, 0.0)
    for b, h in heads:
        ro, rl = oracle.forward(f64(q[b, h], dtype), f64(k[b, h], dtype), f64(v[b, h], dtype), scale, causal)
        mo, _ = assert_close(out[b, h], ro, TOL_O[dtype], f"O[{b},{h}] {dtype} causal={causal}", rel_l2)
        ml, _ = assert_close(lse[b, h], rl, TOL_LSE, f"LSE[{b},{h}]")
        worst = (max(worst[0], mo), max(worst[1], ml))
    return worst


SHAPES = [
    # B, H, M, N
    (1, 1, 128, 128),
    (1, 1, 256, 256),
    (2, 3, 384, 256),
    (1, 2, 300, 200),   # ragged M and N
    (1, 1, 1, 1),
    (1, 1, 5, 700),
    (1, 2, 1000, 1000),
    (1, 1, 200, 513),
    (1, 1, 777, 129),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,M,N", SHAPES)
def test_forward_matches_oracle(dtype, D, causal, B, H, M, N):
    scale = 1.0 / math.sqrt(D)
    inputs, out, lse = run_fwd(B, H, M, N, D, dtype, causal, scale, seed=B * 1000 + M + N)
    check_heads(inputs, out, lse, dtype, causal, scale)


@pytest.mark.parametrize("N", [512, 1024, 2048])
def test_forward_multihead_fp16_workload(N):
    """B=4, H=12, D=64, M=N, fp16, scale 0.125: sampled heads in full."""
    B, H, D = 4, 12, 64
    inputs, out, lse = run_fwd(B, H, N, N, D, "f16", False, 0.125, seed=0)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    check_heads(inputs, out, lse, "f16", False, 0.125, heads=[(0, 0), (1, 5), (2, 11), (3, 7)])


def test_forward_fp16_error_magnitude_matches_the_pages():
    """At B=4, H=12, M=N=2048, D=64 fp16 the flash-attention README's "Accuracy" table
    (tests/golden/fp16_forward_error_magnitudes.json) prints rel L2 2.819e-4 and max abs
    1.098e-4 for an fp16 kernel against an fp32 reference (output rounding dominates).
    Ours against the fp64 oracle must be of the same order."""
    import json
    import os
    pr = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fp16_forward_error_magnitudes.json")))
    pr = pr["printed"]
    inputs, out, lse = run_fwd(4, 12, 2048, 2048, 64, "f16", False, 0.125, seed=0)
    q, k, v = inputs
    num = den = 0.0
    mx = 0.0
    for b, h in [(0, 0), (3, 11)]:
        ro, _ = oracle.forward(f64(q[b, h], "f16"), f64(k[b, h], "f16"), f64(v[b, h], "f16"), 0.125, False)
        num += float(np.sum((out[b, h] - ro) ** 2))
        den += float(np.sum(ro ** 2))
        mx = max(mx, float(np.max(np.abs(out[b, h] - ro))))
    rel = math.sqrt(num / den)
    assert rel <= 2 * pr["rel_l2"] and mx <= 2 * pr["max_abs"], (rel, mx)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("std", [1.0, 0.5])
def test_forward_tutorial_shape(causal, std):
    """Z=1, H=2, N_CTX=1024, D=64, sm_scale 0.5, fp16, causal and not; inputs
    N(0,1) and the tutorial's own N(0, 0.5^2)."""
    inputs, out, lse = run_fwd(1, 2, 1024, 1024, 64, "f16", causal, 0.5, seed=20, std=std)
    check_heads(inputs, out, lse, "f16", causal, 0.5)


def test_forward_closed_forms():
    """Q = 0 gives the column mean of V; V = 1 gives 1; causal row 0 gives V[0]."""
    import torch
    B, H, M, N, D = 1, 2, 256, 384, 64
    _, k, v = synth.attention_inputs(B, H, M, N, D, "f16", seed=5)
    kd, vd = to_device(k, "f16"), to_device(v, "f16")
    q0 = torch.zeros((B, H, M, D), dtype=torch.float16, device="cuda")
    out, lse = fa.forward(q0, kd, vd, 0.125, False)
    mean = f64(v, "f16").mean(axis=2, keepdims=True)
    assert_close(to_f64(out), np.broadcast_to(mean, (B, H, M, D)), 2e-3, "Q=0")
    assert_close(to_f64(lse), np.full((B, H, M), math.log(N)), 1e-5, "LSE(Q=0)")
    ones = torch.ones((B, H, N, D), dtype=torch.float16, device="cuda")
    qd = to_device(synth.attention_inputs(B, H, M, N, D, "f16", seed=6)[0], "f16")
    out1, _ = fa.forward(qd, kd, ones, 0.125, True)
    assert_close(to_f64(out1), np.ones((B, H, M, D)), 1e-3, "V=1")
    outc, _ = fa.forward(qd, kd, vd, 0.125, True)
    assert_close(to_f64(outc)[:, :, 0], f64(v, "f16")[:, :, 0], 1e-3, "causal row 0")


F32_SHAPES = [
    # B, H, M, N
    (1, 1, 256, 256),    # single head, 256 x 256 (seed 0)
    (1, 1, 4096, 4096),  # single head, 4096 x 4096
    (2, 3, 300, 200),
    (1, 1, 1, 1),
    (1, 2, 129, 777),
    # few tiles, long key ranges: each tile's keys split over many CTAs (19, 12 and 30 parts),
    # merged by the part that counts in last
    (1, 1, 1000, 3000),
    (1, 2, 700, 2500),
    (1, 1, 640, 3900),
    # parts of a tile as one cluster, merged through shared memory: 2 parts (256^2 and 300 x 200
    # above), 4 (4096^2 above) and 8 here (19 tiles, the last ragged; causal: empty parts)
    (1, 1, 2400, 1000),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,M,N", F32_SHAPES)
def test_forward_f32_matches_oracle(causal, B, H, M, N):
    """f32 I/O (3xTF32 contraction): max abs <= 1e-4 and relative L2 <= 1e-5 against fp64."""
    scale = 0.125
    inputs, out, lse = run_fwd(B, H, M, N, 64, "f32", causal, scale, seed=0)
    heads = [(0, 0)] if B * H * M * N > 10**7 else None
    check_heads(inputs, out, lse, "f32", causal, scale, heads=heads, rel_l2=REL_L2_F32)


def test_forward_f32_head_dim_128_is_unsupported():
    import torch
    q = torch.zeros((1, 1, 8, 128), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(q, q, q, q, None, 1, 1, 8, 8, 128, 0.1, 0, fa.FA_F32) == fa.FA_ERR_UNSUPPORTED


SPLIT_SHAPES = [
    # B, H, M, N
    (1, 1, 256, 384),    # one pair cut into one-block pieces; most CTAs get no work
    (2, 3, 300, 200),    # ragged M and N
    (1, 2, 1024, 1024),  # 8 pairs x 8 key blocks spread over all SMs
    (3, 5, 700, 1500),   # pieces crossing pair boundaries, ragged tails
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("B,H,M,N", SPLIT_SHAPES)
def test_forward_split_schedule_matches_oracle(dtype, B, H, M, N, causal):
    """The split schedule (each SM an equal share of (query pair, key block) units, cut
    pairs merged with the online-softmax rescaling) forced on; causal pairs hold
    different numbers of units."""
    scale = 0.125
    with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1):
        inputs, out, lse = run_fwd(B, H, M, N, 64, dtype, causal, scale, seed=M + N)
    check_heads(inputs, out, lse, dtype, causal, scale)


@pytest.mark.parametrize("B,H,M,N,dtype,causal", [(1, 4, 2048, 2048, "bf16", False), (1, 2, 1024, 8192, "f16", False),
                                                    (1, 2, 4096, 4096, "f16", True)])
def test_forward_split_automatic_choice(B, H, M, N, dtype, causal):
    """Shapes whose pairs have many key blocks and fill few SMs take the split schedule without
    forcing: 32 pairs of 16 blocks; 8 pairs of 64 blocks, each cut into about 19 pieces, so the
    holder of a pair's first blocks merges about 18 partials; causal, 32 pairs of 1 to 31 blocks."""
    scale = 0.125
    inputs, out, lse = run_fwd(B, H, M, N, 64, dtype, causal, scale, seed=N + H)
    check_heads(inputs, out, lse, dtype, causal, scale)


def test_forward_split_schedule_repeated_calls():
    """Back-to-back calls reuse one workspace; each launch's flags carry a new epoch, and the
    merging CTAs put the flags they consumed back to zero."""
    import torch
    nbytes = fa.fa_fwd_workspace_bytes(1, 3, 512, 640, 64, 0, fa.FA_F16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    flags = ws[nbytes - sms * 8 * 4:]  # eight 32-bit flags per SM end the workspace
    for seed in (1, 2, 3):
        q, k, v = synth.attention_inputs(1, 3, 512, 640, 64, "f16", seed=seed)
        with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1):
            out, lse = fa.forward(to_device(q, "f16"), to_device(k, "f16"), to_device(v, "f16"), 0.125, False,
                                  workspace=ws)
        assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
        check_heads((q, k, v), to_f64(out), to_f64(lse), "f16", False, 0.125)
        assert int(torch.count_nonzero(flags)) == 0, "flags left set after the merge"



@pytest.mark.parametrize("causal", [False, True])
def test_forward_f32_without_workspace(causal):
    """The f32 path with one CTA per query tile (no key-range split): fa_fwd without a workspace."""
    import torch
    q, k, v = synth.attention_inputs(1, 2, 300, 700, 64, "f32", seed=4)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    fa.forward(to_device(q, "f32"), to_device(k, "f32"), to_device(v, "f32"), 0.125, causal, out=out, lse=lse,
               workspace=False)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    check_heads((q, k, v), to_f64(out), to_f64(lse), "f32", causal, 0.125, rel_l2=REL_L2_F32)


HOST_CASES = [
    # B, H, M, N, D, dtype, causal (default chunks: three, 4:2:1 from seven heads up)
    (1, 1, 256, 300, 64, "f16", False),    # one head: one chunk
    (2, 3, 300, 200, 64, "bf16", True),    # six heads: three equal chunks, ragged M and N
    (3, 5, 700, 1500, 64, "f16", False),   # 15 heads in chunks of 9, 4 and 2
    (2, 2, 512, 512, 128, "f16", True),    # D = 128
    (1, 3, 256, 384, 64, "f32", False),    # f32 (3xTF32 path)
    (1, 7, 256, 640, 64, "f32", False),    # f32, seven heads: 4, 2 and 1
]


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", HOST_CASES)
@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_buffers(B, H, M, N, D, dtype, causal, pinned):
    """fa_fwd_host: host inputs in, host O and LSE out, chunked over heads with the copies
    overlapped; same results as the device forward (checked against the oracle)."""
    import torch
    scale = 0.125
    q, k, v = synth.attention_inputs(B, H, M, N, D, dtype, seed=B * H + M)
    hq, hk, hv = (to_device(x, dtype).cpu() for x in (q, k, v))
    ho, hl = torch.empty_like(hq), torch.empty((B, H, M), dtype=torch.float32)
    if pinned:
        hq, hk, hv, ho, hl = (t.pin_memory() for t in (hq, hk, hv, ho, hl))
    dt = {"f32": fa.FA_F32, "f16": fa.FA_F16, "bf16": fa.FA_BF16}[dtype]
    nbytes = fa.fa_fwd_host_workspace_bytes(B, H, M, N, D, causal, dt)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the workspace
        s = fa.fa_fwd_host(hq, hk, hv, ho, hl, ws, nbytes, B, H, M, N, D, scale, causal, dt)
        assert s == fa.FA_OK, fa.fa_last_error_message()
        torch.cuda.synchronize()
        assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
        check_heads((q, k, v), to_f64(ho), to_f64(hl), dtype, causal, scale,
                    rel_l2=REL_L2_F32 if dtype == "f32" else None)


@pytest.mark.parametrize("chunks", [2, 5, 8])
def test_forward_host_buffers_forced_chunks(chunks):
    """fa_set_schedule(FA_SCHED_HOST_CHUNKS, n): n equal chunks (15 heads: two sizes each)."""
    import torch
    B, H, M, N, D = 3, 5, 384, 700, 64
    q, k, v = synth.attention_inputs(B, H, M, N, D, "bf16", seed=chunks)
    hq, hk, hv = (to_device(x, "bf16").cpu().pin_memory() for x in (q, k, v))
    ho, hl = torch.empty_like(hq).pin_memory(), torch.empty((B, H, M), dtype=torch.float32).pin_memory()
    with fa.schedule(fa.FA_SCHED_HOST_CHUNKS, chunks):
        nbytes = fa.fa_fwd_host_workspace_bytes(B, H, M, N, D, 0, fa.FA_BF16)
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        assert fa.fa_fwd_host(hq, hk, hv, ho, hl, ws, nbytes, B, H, M, N, D, 0.125, 0, fa.FA_BF16) == fa.FA_OK
        torch.cuda.synchronize()
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    check_heads((q, k, v), to_f64(ho), to_f64(hl), "bf16", False, 0.125)


def test_forward_host_buffers_without_lse_and_checks():
    import torch
    B, H, M, N, D = 2, 2, 256, 256, 64
    q, k, v = synth.attention_inputs(B, H, M, N, D, "f16", seed=4)
    hq, hk, hv = (to_device(x, "f16").cpu().pin_memory() for x in (q, k, v))
    ho = torch.empty_like(hq).pin_memory()
    nbytes = fa.fa_fwd_host_workspace_bytes(B, H, M, N, D, 0, fa.FA_F16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    assert fa.fa_fwd_host(hq, hk, hv, ho, None, ws, nbytes, B, H, M, N, D, 0.125, 0, fa.FA_F16) == fa.FA_OK
    torch.cuda.synchronize()
    ref = [oracle.forward(f64(q[b, h], "f16"), f64(k[b, h], "f16"), f64(v[b, h], "f16"), 0.125, False)[0]
           for b in range(B) for h in range(H)]
    assert_close(to_f64(ho).reshape(B * H, M, D), np.stack(ref), TOL_O["f16"], "host O without LSE")
    # a small workspace or a NULL host buffer is rejected before anything is queued
    assert fa.fa_fwd_host(hq, hk, hv, ho, None, ws, nbytes - 256, B, H, M, N, D, 0.125, 0, fa.FA_F16) == \
        fa.FA_ERR_INVALID
    assert fa.fa_fwd_host(hq, None, hv, ho, None, ws, nbytes, B, H, M, N, D, 0.125, 0, fa.FA_F16) == fa.FA_ERR_INVALID
    assert fa.fa_fwd_host(hq, hk, hv, ho, None, ws, nbytes, B, H, M, N, 96, 0.125, 0, fa.FA_F16) == \
        fa.FA_ERR_UNSUPPORTED


def test_forward_f32_and_half_splits_share_the_workspace():
    """The cached forward workspace serves, in turn, the f32 key-range split (partial slots and
    epoch-tagged counters, merged by the part that finishes last) and the half-precision split
    schedule (partials and epoch flags); neither is misled by what the other left there, and a
    repeated f32 call is not misled by its own earlier counts."""
    for seed in (1, 2):
        for dtype in ("f32", "f16", "f32"):
            with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1):
                inputs, out, lse = run_fwd(1, 2, 512, 768, 64, dtype, seed == 2, 0.125, seed=seed)
            check_heads(inputs, out, lse, dtype, seed == 2, 0.125, rel_l2=REL_L2_F32 if dtype == "f32" else None)


NEG_CASES = [
    # B, H, M, N, D, dtype, causal, scale
    (1, 2, 300, 200, 64, "f16", False, -0.125),
    (1, 2, 300, 700, 64, "bf16", True, -0.2),
    (1, 4, 2048, 2048, 64, "f16", False, -0.125),  # split schedule at automatic choice
    (1, 2, 384, 256, 128, "f16", True, -1 / math.sqrt(128)),
    (1, 1, 256, 300, 64, "f32", False, -0.125),
    (1, 1, 5, 700, 64, "f32", True, -0.3),
    (1, 2, 200, 200, 64, "f16", True, 0.0),        # scale 0: uniform weights over the visible keys
]


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal,scale", NEG_CASES)
def test_forward_negative_and_zero_scale(B, H, M, N, D, dtype, causal, scale):
    """Any finite scale: scale < 0 negates the score product in the tensor core (the row maximum
    is then taken over -q.k) and the exponent uses |scale|; the oracle applies scale as given."""
    inputs, out, lse = run_fwd(B, H, M, N, D, dtype, causal, scale, seed=7 * M + N)
    check_heads(inputs, out, lse, dtype, causal, scale, rel_l2=REL_L2_F32 if dtype == "f32" else None)


def test_forward_negative_scale_split_forced():
    with fa.schedule(fa.FA_SCHED_FWD_SPLIT, 1):
        inputs, out, lse = run_fwd(3, 5, 700, 1500, 64, "f16", False, -0.125, seed=3)
    check_heads(inputs, out, lse, "f16", False, -0.125)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_forward_rising_scores_rescale(dtype, causal, D):
    """Scores that rise along the keys: each key block's scores sit above the running maximum by
    far more than 2^8 in the exponent, and a block's second half above its first, so the halves
    formed against the running maximum overflow and are formed again after a rescale (both the
    first-half and the second-half paths), every block."""
    rng = np.random.default_rng(5)
    B, H, M, N = 1, 2, 512, 1024
    u = np.ones(D, dtype=np.float32) / np.sqrt(D)
    q = rng.standard_normal((B, H, M, D), dtype=np.float32) + 2.0 * u
    k = rng.standard_normal((B, H, N, D), dtype=np.float32) + (0.2 * np.arange(N, dtype=np.float32))[:, None] * u
    v = rng.standard_normal((B, H, N, D), dtype=np.float32)
    q, k, v = (synth.round_f32(x.astype(np.float32), dtype) for x in (q, k, v))
    scale = 1.0 / math.sqrt(D)
    out, lse = fa.forward(to_device(q, dtype), to_device(k, dtype), to_device(v, dtype), scale, causal)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    check_heads((q, k, v), to_f64(out), to_f64(lse), dtype, causal, scale)
