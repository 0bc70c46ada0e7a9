"""Flash decoding on the GPU against the fp64 oracle (split partials and combined output)."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import exact_attention_gb300 as fa
from exact_attention_gb300 import synth

from helpers import TOL_LSE, TOL_O, REL_L2_F32, assert_close, f64, to_device, to_f64

pytestmark = pytest.mark.gpu

# Elementwise bound for the rounded output: half an ulp of the storage type
# relative to |O| plus f32 accumulation slack.
REL_ROUND = {"f32": 2.0**-22, "f16": 2.0**-11, "bf16": 2.0**-8}


def run_decode(B, H, N, D, dtype, n_splits, seed=0):
    q, k, v = synth.decode_inputs(B, H, N, D, dtype, seed)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = to_device(q, dtype), to_device(k, dtype), to_device(v, dtype)
    out, ws = fa.decode(qd, kd, vd, scale, n_splits)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    return (q, k, v, scale), to_f64(out), ws


CASES = [
    # B, H, N, D, n_splits
    (1, 1, 1, 64, 1),
    (1, 2, 7, 64, 3),
    (2, 3, 1000, 128, 16),
    (1, 2, 4096, 128, 64),
    (2, 1, 333, 64, 333),
    (1, 1, 5000, 128, 7),
    (1, 1, 100, 128, 64),  # trailing empty splits: ceil(100/64) = 2 keys per split
]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("B,H,N,D,ns", CASES)
def test_decode_matches_oracle(dtype, B, H, N, D, ns):
    (q, k, v, scale), out, ws = run_decode(B, H, N, D, dtype, ns)
    q64, k64, v64 = f64(q, dtype), f64(k, dtype), f64(v, dtype)
    ref = oracle.decode(q64, k64, v64, scale)
    assert_close(out, ref, TOL_O[dtype], f"decode O {dtype}", REL_L2_F32 if dtype == "f32" else None)
    assert np.all(np.abs(out - ref) <= REL_ROUND[dtype] * np.abs(ref) + 2e-6)
    # the workspace holds the page's unnormalised partials
    Os, ms, ls = fa.split_workspace(ws, B, H, D, ns)
    Os, ms, ls = to_f64(Os), to_f64(ms), to_f64(ls)
    for b in range(B):
        for h in range(H):
            ro, rm, rl = oracle.decode_partials(q64[b, h, 0], k64[b, h], v64[b, h], scale, ns)
            bh = b * H + h
            empty = np.isneginf(rm)
            assert np.array_equal(np.isneginf(ms[bh]), empty)
            assert np.all(ls[bh][empty] == 0) and np.all(Os[bh][empty] == 0)
            assert np.max(np.abs(ms[bh][~empty] - rm[~empty])) <= 1e-5
            assert np.max(np.abs(ls[bh] - rl) / np.maximum(rl, 1e-30)) <= 1e-5
            assert np.max(np.abs(Os[bh] - ro)) <= 1e-5 * max(1.0, np.max(np.abs(ro)))


@pytest.mark.parametrize("ns", [1, 2, 5, 64])
def test_decode_split_count_invariance(ns):
    """Any number of splits gives the same O (the combine is exact)."""
    (q, k, v, scale), out, _ = run_decode(2, 2, 777, 128, "f32", ns, seed=3)
    ref = oracle.decode(f64(q, "f32"), f64(k, "f32"), f64(v, "f32"), scale)
    assert_close(out, ref, 1e-5, f"n_splits={ns}")


FULL = (8, 32, 32768, 128)  # B, H, N, D of the bf16 decode workload


@pytest.fixture(scope="module")
def full_cache():
    import torch
    B, H, N, D = FULL
    q = synth.decode_query(B, H, D, "bf16", 0)
    k = torch.empty((B, H, N, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    for b, h, kh, vh in synth.iter_decode_heads(B, H, N, D, "bf16", 0):
        k[b, h] = to_device(kh, "bf16")
        v[b, h] = to_device(vh, "bf16")
    yield q, k, v
    del k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("ns", [16, 64, 256])
def test_decode_full_size_sampled_heads(full_cache, ns):
    """B=8, H=32, N=32768, D=128 bf16 cache: outputs of sampled (b, h) checked against
    the oracle, which regenerates those heads on the host."""
    q, k, v = full_cache
    B, H, N, D = FULL
    scale = 1.0 / math.sqrt(D)
    out, _ = fa.decode(to_device(q, "bf16"), k, v, scale, ns)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    out = to_f64(out)
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(ns)
    for b, h in [(0, 0), (B - 1, H - 1)] + [tuple(x) for x in rng.integers(0, [B, H], size=(4, 2))]:
        kh, vh = synth.decode_head_kv(b, h, N, D, "bf16", 0)
        ref = oracle.decode(f64(q[b, h], "bf16"), f64(kh, "bf16"), f64(vh, "bf16"), scale)
        assert_close(out[b, h], ref, TOL_O["bf16"], f"decode head ({b},{h})")
        assert np.all(np.abs(out[b, h] - ref) <= REL_ROUND["bf16"] * np.abs(ref) + 2e-6)


ROW_CASES = [
    # B, H, R, N, D, n_splits
    (1, 1, 2, 1, 64, 1),
    (2, 3, 2, 1000, 128, 16),
    (1, 2, 3, 4096, 128, 64),   # three rows run the four-row kernel with a padding row
    (2, 1, 4, 333, 64, 333),
    (1, 1, 4, 5000, 128, 7),
    (1, 2, 4, 100, 128, 64),    # trailing empty splits
    (3, 2, 1, 777, 64, 5),      # one row with an LSE goes through fa_decode_ex too
]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("B,H,R,N,D,ns", ROW_CASES)
def test_decode_rows_match_oracle(dtype, B, H, R, N, D, ns):
    """R query rows per (batch, head) against the whole cache: O and LSE per row equal the
    oracle's forward over those R rows (no mask)."""
    q, k, v = synth.attention_inputs(B, H, R, N, D, dtype, seed=R * 100 + N)
    scale = 1.0 / math.sqrt(D)
    out, ws, lse = fa.decode(to_device(q, dtype), to_device(k, dtype), to_device(v, dtype), scale, ns, lse=True)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    out, lse = to_f64(out), to_f64(lse)
    q64, k64, v64 = f64(q, dtype), f64(k, dtype), f64(v, dtype)
    for b in range(B):
        for h in range(H):
            ro, rl = oracle.forward(q64[b, h], k64[b, h], v64[b, h], scale, False)
            assert_close(out[b, h], ro, TOL_O[dtype], f"decode rows O[{b},{h}] {dtype}",
                         REL_L2_F32 if dtype == "f32" else None)
            assert np.all(np.abs(out[b, h] - ro) <= REL_ROUND[dtype] * np.abs(ro) + 2e-6)
            assert_close(lse[b, h], rl, TOL_LSE, f"decode rows LSE[{b},{h}]")


def test_decode_rows_partials_are_the_pages():
    """Row r of head bh is partial row bh*R + r: each holds the page's unnormalised partials."""
    B, H, R, N, D, ns = 1, 2, 3, 1500, 64, 6
    q, k, v = synth.attention_inputs(B, H, R, N, D, "f32", seed=9)
    scale = 0.125
    _, ws = fa.decode(to_device(q, "f32"), to_device(k, "f32"), to_device(v, "f32"), scale, ns)
    Os, ms, ls = fa.split_workspace(ws, B, H * R, D, ns)
    Os, ms, ls = to_f64(Os), to_f64(ms), to_f64(ls)
    for h in range(H):
        for r in range(R):
            ro, rm, rl = oracle.decode_partials(f64(q, "f32")[0, h, r], f64(k, "f32")[0, h], f64(v, "f32")[0, h],
                                                scale, ns)
            row = h * R + r
            assert np.max(np.abs(ms[row] - rm)) <= 1e-5
            assert np.max(np.abs(ls[row] - rl) / np.maximum(rl, 1e-30)) <= 1e-5
            assert np.max(np.abs(Os[row] - ro)) <= 1e-5 * max(1.0, np.max(np.abs(ro)))


def test_decode_rows_limits():
    import torch
    q = torch.zeros((1, 1, 5, 64), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(4096, dtype=torch.float32, device="cuda")
    assert fa.fa_decode_ex(q, kv, kv, q, None, ws, 1, 1, 5, 8, 64, 0.1, 2, fa.FA_BF16) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_decode_ex(q, kv, kv, q, None, ws, 1, 1, 0, 8, 64, 0.1, 2, fa.FA_BF16) == fa.FA_ERR_INVALID
    assert fa.fa_decode_ex_workspace_bytes(2, 3, 4, 128, 16) == 2 * 3 * 4 * 16 * 130 * 4


def test_decode_rows_grouped_query_full_cache(full_cache):
    """Grouped-query decode on the B=8, H=32, N=32768, D=128 bf16 cache: four query rows per
    K/V head; sampled heads checked against the oracle."""
    import torch
    _, k, v = full_cache
    B, H, N, D = FULL
    R = 4
    rng = np.random.default_rng(5)
    q = synth.normal(rng, (B, H, R, D), "bf16")
    scale = 1.0 / math.sqrt(D)
    out, _, lse = fa.decode(to_device(q, "bf16"), k, v, scale, 64, lse=True)
    assert fa.fa_last_status() == fa.FA_OK, fa.fa_last_error_message()
    out, lse = to_f64(out), to_f64(lse)
    for b, h in [(0, 0), (B - 1, H - 1), (3, 17)]:
        kh, vh = synth.decode_head_kv(b, h, N, D, "bf16", 0)
        ro, rl = oracle.forward(f64(q[b, h], "bf16"), f64(kh, "bf16"), f64(vh, "bf16"), scale, False)
        assert_close(out[b, h], ro, TOL_O["bf16"], f"grouped decode head ({b},{h})")
        assert_close(lse[b, h], rl, TOL_LSE, f"grouped decode LSE ({b},{h})")
