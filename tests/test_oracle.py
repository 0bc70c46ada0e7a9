"""Pins for the fp64 oracle: it is checked against things other than itself.

* high-precision brute force (mpmath, 50 digits, pure-Python loops, no max
  subtraction) on tiny inputs, for the forward values, LSE, decode partials and,
  through mpmath's numerical differentiation, every gradient entry;
* closed forms: Q = 0 gives the column mean of V and LSE = ln(#keys); V = 1
  gives 1; a single key gives that key's value; causal row 0 gives V[0];
  a large scale turns the softmax into an argmax;
* invariants: split-and-combine equals the unsplit result for any number of
  splits, shifting K along a direction leaves O unchanged, permuting keys leaves
  O unchanged, sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, and
  rowsum(dO o O) = rowsum(P o dP);
* central finite differences of sum(dO o O) in float64.

The last test plants mistakes in copies of the oracle (dropped scale, wrong
mask direction, missing correction, transposed operand, ...) and checks that
each one fails at least one pin, so the pins have teeth.
"""
from __future__ import annotations

import types

import mpmath as mp
import numpy as np
import pytest

import oracle
from exact_attention_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

REAL = types.SimpleNamespace(
    forward=oracle.forward,
    backward=oracle.backward,
    delta=oracle.delta,
    probabilities=oracle.probabilities,
    decode_partials=oracle.decode_partials,
    decode_combine=oracle.decode_combine,
)


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


# ----------------------------------------------------------------- brute force
def mp_forward(Q, K, V, scale, causal):
    """Softmax attention at 50 digits, written from the definition (no max trick)."""
    with mp.workdps(50):
        M, D = Q.shape
        N = K.shape[0]
        O = np.empty((M, V.shape[1]), dtype=object)
        L = np.empty(M, dtype=object)
        sc = mp.mpf(float(scale))
        for i in range(M):
            keys = [j for j in range(N) if (not causal) or j <= i]
            s = {j: sc * mp.fsum(mp.mpf(float(Q[i, d])) * mp.mpf(float(K[j, d])) for d in range(D)) for j in keys}
            w = {j: mp.exp(s[j]) for j in keys}
            Z = mp.fsum(w.values())
            for d in range(V.shape[1]):
                O[i, d] = mp.fsum(w[j] * mp.mpf(float(V[j, d])) for j in keys) / Z
            L[i] = mp.log(Z)
        return O, L


def mp_grad(Q, K, V, dO, scale, causal, which, idx):
    """d/dx sum(dO o O) for one input entry, by mpmath's numerical differentiation."""
    def loss(t):
        arrs = {"q": Q.astype(object), "k": K.astype(object), "v": V.astype(object)}
        for a in arrs.values():
            for ix in np.ndindex(a.shape):
                a[ix] = mp.mpf(float(a[ix]))
        arrs[which][idx] = arrs[which][idx] + t
        q, k, v = arrs["q"], arrs["k"], arrs["v"]
        M, D = q.shape
        N = k.shape[0]
        total = mp.mpf(0)
        for i in range(M):
            keys = [j for j in range(N) if (not causal) or j <= i]
            s = {j: mp.mpf(float(scale)) * mp.fsum(q[i, d] * k[j, d] for d in range(D)) for j in keys}
            w = {j: mp.exp(s[j]) for j in keys}
            Z = mp.fsum(w.values())
            for d in range(v.shape[1]):
                total += mp.mpf(float(dO[i, d])) * mp.fsum(w[j] * v[j, d] for j in keys) / Z
        return total

    with mp.workdps(40):
        return mp.diff(loss, 0)


def pin_brute_forward(impl):
    rng = np.random.default_rng(1)
    # negative and zero scales too: the library takes any finite scale
    for (M, N, D, causal, scale) in [(3, 4, 2, False, 0.7), (4, 4, 3, True, 0.5), (2, 5, 4, False, 1.9),
                                     (5, 3, 2, True, 0.3), (3, 4, 3, False, -0.9), (4, 4, 2, True, -1.3),
                                     (2, 3, 2, False, 0.0)]:
        Q, K, V = _rand(rng, M, D), _rand(rng, N, D), _rand(rng, N, D)
        O, L = impl.forward(Q, K, V, scale, causal)
        Om, Lm = mp_forward(Q, K, V, scale, causal)
        Om = Om.astype(float)
        Lm = Lm.astype(float)
        assert np.all(np.isfinite(O)), "non-finite output"
        assert np.max(np.abs(O - Om)) <= 1e-13 * max(1.0, np.max(np.abs(Om))), (M, N, D, causal)
        assert np.max(np.abs(L - Lm)) <= 1e-13 * max(1.0, np.max(np.abs(Lm))), (M, N, D, causal)


def pin_brute_backward(impl):
    rng = np.random.default_rng(2)
    for (M, N, D, causal, scale) in [(3, 3, 2, False, 0.8), (3, 3, 2, True, 0.5), (2, 3, 2, False, 1.3),
                                     (3, 3, 2, False, -0.6), (3, 3, 2, True, -1.1)]:
        Q, K, V, dO = _rand(rng, M, D), _rand(rng, N, D), _rand(rng, N, D), _rand(rng, M, D)
        dQ, dK, dV = impl.backward(Q, K, V, dO, scale, causal)
        for which, g in (("q", dQ), ("k", dK), ("v", dV)):
            for idx in np.ndindex(g.shape):
                ref = float(mp_grad(Q, K, V, dO, scale, causal, which, idx))
                assert abs(g[idx] - ref) <= 1e-11 * max(1.0, abs(ref)), (which, idx, causal, g[idx], ref)


def pin_brute_decode(impl):
    rng = np.random.default_rng(3)
    N, D, scale = 11, 3, 0.6
    q, K, V = _rand(rng, D), _rand(rng, N, D), _rand(rng, N, D)
    Os, ms, ls = impl.decode_partials(q, K, V, scale, 4)  # splits of 3,3,3,2 keys
    size = 3
    with mp.workdps(50):
        for s in range(4):
            lo, hi = s * size, min(s * size + size, N)
            x = [mp.mpf(scale) * mp.fsum(mp.mpf(q[d]) * mp.mpf(K[j, d]) for d in range(D)) for j in range(lo, hi)]
            m = max(x)
            e = [mp.exp(xx - m) for xx in x]
            assert abs(ms[s] - float(m)) <= 1e-14 * max(1, abs(float(m)))
            assert abs(ls[s] - float(mp.fsum(e))) <= 1e-13 * float(mp.fsum(e))
            for d in range(D):
                ref = float(mp.fsum(e[t] * mp.mpf(V[lo + t, d]) for t in range(hi - lo)))
                assert abs(Os[s, d] - ref) <= 1e-13 * max(1.0, abs(ref))
    O = impl.decode_combine(Os, ms, ls)
    Om, _ = mp_forward(q[None, :], K, V, scale, False)
    assert np.max(np.abs(O - Om.astype(float)[0])) <= 1e-13


# ----------------------------------------------------------------- closed forms
def pin_closed_forms(impl):
    rng = np.random.default_rng(4)
    M, N, D = 9, 13, 5
    K, V = _rand(rng, N, D), _rand(rng, N, D)
    # Q = 0: uniform weights
    O, L = impl.forward(np.zeros((M, D)), K, V, 0.37, False)
    assert np.allclose(O, V.mean(0)[None, :].repeat(M, 0), rtol=0, atol=1e-14)
    assert np.allclose(L, np.log(N), rtol=0, atol=1e-14)
    Oc, Lc = impl.forward(np.zeros((N, D)), K, V, 0.37, True)
    for i in range(N):
        assert np.allclose(Oc[i], V[: i + 1].mean(0), rtol=0, atol=1e-14)
        assert abs(Lc[i] - np.log(i + 1)) <= 1e-14
    # V = 1: every output is 1
    Q = _rand(rng, M, D)
    O1, _ = impl.forward(Q, K, np.ones((N, D)), 0.9, False)
    assert np.allclose(O1, 1.0, rtol=0, atol=1e-14)
    O1c, _ = impl.forward(_rand(rng, N, D), K, np.ones((N, D)), 0.9, True)
    assert np.allclose(O1c, 1.0, rtol=0, atol=1e-14)
    # a single key: O = V[0], LSE = scale q.k0
    O2, L2 = impl.forward(Q, K[:1], V[:1], 0.45, False)
    assert np.allclose(O2, V[:1].repeat(M, 0), rtol=0, atol=1e-14)
    assert np.allclose(L2, 0.45 * Q @ K[0], rtol=0, atol=1e-13)
    # causal row 0 sees only key 0
    Q3 = _rand(rng, N, D)
    O3, L3 = impl.forward(Q3, K, V, 0.8, True)
    assert np.allclose(O3[0], V[0], rtol=0, atol=1e-14)
    assert abs(L3[0] - 0.8 * Q3[0] @ K[0]) <= 1e-13
    # huge scale: softmax becomes an argmax (needs the max subtraction to stay finite)
    Qh = _rand(rng, M, D)
    S = Qh @ K.T
    Oh, Lh = impl.forward(Qh, K, V, 1e4, False)
    assert np.all(np.isfinite(Oh)) and np.all(np.isfinite(Lh))
    srt = np.sort(S, axis=1)
    ok = (srt[:, -1] - srt[:, -2]) > 1e-2  # unique, well separated maxima only
    assert np.allclose(Oh[ok], V[np.argmax(S, axis=1)][ok], rtol=0, atol=1e-12)


def pin_invariants(impl):
    rng = np.random.default_rng(5)
    M, N, D, scale = 7, 300, 4, 0.4
    Q, K, V = _rand(rng, M, D), _rand(rng, N, D), _rand(rng, N, D)
    O, _ = impl.forward(Q, K, V, scale, False)
    # split-and-combine equals the unsplit result for any number of splits
    for ns in (1, 2, 3, 16, 64, 256, N):
        for i in range(M):
            Oi = impl.decode_combine(*impl.decode_partials(Q[i], K, V, scale, ns))
            assert np.max(np.abs(Oi - O[i])) <= 1e-13, (ns, i)
    # shift invariance: K -> K + 1 u^T adds q_i.u to row i of S
    u = _rand(rng, D)
    Os_, _ = impl.forward(Q, K + u[None, :], V, scale, False)
    assert np.max(np.abs(Os_ - O)) <= 1e-12
    # permuting the keys (with their values) leaves O unchanged
    perm = rng.permutation(N)
    Op, _ = impl.forward(Q, K[perm], V[perm], scale, False)
    assert np.max(np.abs(Op - O)) <= 1e-13
    # rows of P sum to one
    assert np.allclose(impl.probabilities(Q, K, scale, True if M <= N else False).sum(-1), 1.0, atol=1e-14)
    # backward invariants, causal and not
    for causal in (False, True):
        Qb, Kb, Vb, dO = _rand(rng, 12, D), _rand(rng, 12, D), _rand(rng, 12, D), _rand(rng, 12, D)
        dQ, dK, dV = impl.backward(Qb, Kb, Vb, dO, 0.6, causal)
        assert np.max(np.abs(dK.sum(0))) <= 1e-12
        assert np.max(np.abs(dV.sum(0) - dO.sum(0))) <= 1e-12
        Ob, _ = impl.forward(Qb, Kb, Vb, 0.6, causal)
        P = impl.probabilities(Qb, Kb, 0.6, causal)
        dP = dO @ Vb.T
        assert np.max(np.abs(impl.delta(Ob, dO) - (P * dP).sum(-1))) <= 1e-12


def pin_finite_differences(impl):
    rng = np.random.default_rng(6)
    M, N, D, scale, h = 5, 7, 3, 0.7, 1e-6
    for causal in (False, True):
        Mc = N if causal else M
        Q, K, V, dO = _rand(rng, Mc, D), _rand(rng, N, D), _rand(rng, N, D), _rand(rng, Mc, D)
        grads = impl.backward(Q, K, V, dO, scale, causal)

        def loss(q, k, v):
            return float(np.sum(dO * impl.forward(q, k, v, scale, causal)[0]))

        for t, (X, G) in enumerate(zip((Q, K, V), grads)):
            num = np.zeros_like(X)
            for ix in np.ndindex(X.shape):
                Xp, Xm = X.copy(), X.copy()
                Xp[ix] += h
                Xm[ix] -= h
                args_p = [Q, K, V]
                args_m = [Q, K, V]
                args_p[t], args_m[t] = Xp, Xm
                num[ix] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            rel = np.linalg.norm(num - G) / np.linalg.norm(num)
            assert rel <= 1e-6, (causal, t, rel)


PINS = [pin_brute_forward, pin_brute_backward, pin_brute_decode, pin_closed_forms, pin_invariants,
        pin_finite_differences]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pins(pin):
    pin(REAL)


# ------------------------------------------------------------- planted mistakes
def _mutant(**over):
    ns = types.SimpleNamespace(**vars(REAL))
    for k, v in over.items():
        setattr(ns, k, v)
    return ns


def _fwd_no_scale(Q, K, V, scale, causal=False):
    return oracle.forward(Q, K, V, 1.0, causal)


def _fwd_strict_mask(Q, K, V, scale, causal=False):
    if not causal:
        return oracle.forward(Q, K, V, scale, causal)
    S = oracle.scores(Q, K, scale, False)
    M, N = S.shape
    S = np.where(np.arange(N)[None, :] < np.arange(M)[:, None] + 0, S, -np.inf)
    S[0, 0] = oracle.scores(Q, K, scale, False)[0, 0]
    m = S.max(-1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(-1, keepdims=True)
    return (E / l) @ np.asarray(V, float), (m + np.log(l))[:, 0]


def _fwd_reversed_v(Q, K, V, scale, causal=False):
    return oracle.forward(Q, K, np.asarray(V)[::-1], scale, causal)


def _fwd_lse_no_max(Q, K, V, scale, causal=False):
    O, L = oracle.forward(Q, K, V, scale, causal)
    m = oracle.scores(Q, K, scale, causal).max(-1)
    return O, L - m


def _fwd_no_max_subtraction(Q, K, V, scale, causal=False):
    S = oracle.scores(Q, K, scale, causal)
    E = np.exp(S)
    l = E.sum(-1, keepdims=True)
    return (E / l) @ np.asarray(V, float), np.log(l)[..., 0]


def _bwd_no_row_term(Q, K, V, dO, scale, causal=False):
    P = oracle.probabilities(Q, K, scale, causal)
    dP = np.asarray(dO) @ np.asarray(V).T
    dS = P * dP
    return scale * dS @ K, scale * dS.T @ Q, P.T @ dO


def _bwd_dk_unscaled(Q, K, V, dO, scale, causal=False):
    dQ, dK, dV = oracle.backward(Q, K, V, dO, scale, causal)
    return dQ, dK / scale, dV


def _bwd_dv_untransposed(Q, K, V, dO, scale, causal=False):
    dQ, dK, dV = oracle.backward(Q, K, V, dO, scale, causal)
    P = oracle.probabilities(Q, K, scale, causal)
    if P.shape[0] == P.shape[1]:
        dV = P @ np.asarray(dO, float)
    return dQ, dK, dV


def _combine_unweighted(Os, ms, ls):
    return np.sum(Os, 0) / np.sum(ls)


def _partials_normalised(q, K, V, scale, n):
    Os, ms, ls = oracle.decode_partials(q, K, V, scale, n)
    return Os / np.where(ls > 0, ls, 1)[:, None], ms, ls


MUTANTS = {
    "forward without scale": _mutant(forward=_fwd_no_scale),
    "causal mask j < i": _mutant(forward=_fwd_strict_mask),
    "V rows reversed": _mutant(forward=_fwd_reversed_v),
    "LSE without the max": _mutant(forward=_fwd_lse_no_max),
    "softmax without max subtraction": _mutant(forward=_fwd_no_max_subtraction),
    "dS without the row term": _mutant(backward=_bwd_no_row_term),
    "dK without scale": _mutant(backward=_bwd_dk_unscaled),
    "dV = P dO": _mutant(backward=_bwd_dv_untransposed),
    "combine without split weights": _mutant(decode_combine=_combine_unweighted),
    "partials normalised per split": _mutant(decode_partials=_partials_normalised),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name):
    impl = MUTANTS[name]
    caught = []
    for pin in PINS:
        try:
            pin(impl)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake '{name}' passed every pin"


def test_synth_rounding_is_round_to_nearest_even():
    # bf16: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 and goes to the even one (1.0)
    x = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, -2.5, 3.140625], dtype=np.float32)
    got = synth.to_f64(synth.round_f32(x, "bf16"), "bf16")
    assert list(got) == [1.0, 1.0, 1 + 2**-6, -2.5, 3.140625]
    h = synth.to_f64(synth.round_f32(x, "f16"), "f16")
    assert h[1] == 1 + 2**-8  # exactly representable in fp16
    q, k, v = synth.attention_inputs(1, 2, 3, 4, 8, "bf16", seed=0)
    q2, _, _ = synth.attention_inputs(1, 2, 3, 4, 8, "bf16", seed=0)
    assert q.dtype == np.uint16 and np.array_equal(q, q2)


# ------------------------------------------------------------- page-printed error magnitudes
def test_fp16_error_magnitude_matches_the_printed_table():
    """The fp16 forward's error figures printed by the flash-attention README (section
    "Accuracy", tests/golden/fp16_forward_error_magnitudes.json) against the oracle: rounding the
    oracle's output to fp16 (the dominant error of any correct fp16 kernel at this shape) must give
    errors of the same order. A wrong normalisation or scale in the oracle moves |O|, and with it the
    max-abs figure, by orders of magnitude."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fp16_forward_error_magnitudes.json")))
    sh, pr = g["shape"], g["printed"]
    q, k, v = synth.attention_inputs(1, 2, sh["M"], sh["N"], sh["D"], "f16", seed=0)
    errs, refs = [], []
    for h in range(2):
        o, _ = oracle.forward(synth.to_f64(q[0, h], "f16"), synth.to_f64(k[0, h], "f16"),
                              synth.to_f64(v[0, h], "f16"), 0.125, False)
        errs.append(o.astype(np.float16).astype(np.float64) - o)
        refs.append(o)
    e, r = np.concatenate(errs), np.concatenate(refs)
    max_abs = float(np.max(np.abs(e)))
    rel_l2 = float(np.linalg.norm(e) / np.linalg.norm(r))
    assert pr["max_abs"] / 5 <= max_abs <= pr["max_abs"] * 5, max_abs
    assert pr["rel_l2"] / 3 <= rel_l2 <= pr["rel_l2"] * 3, rel_l2
