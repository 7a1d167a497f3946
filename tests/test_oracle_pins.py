"""Pins for the fp64 oracle, checked against things other than the oracle itself.

* the quadratic (semiseparable matrix) form y = (L o C B^T)(delta X) of page
  "长序列 Mamba 多卡训练算力和显存怎么同时省" §一, written out here by brute force;
* a closed form for constant delta with a single-token impulse in X;
* the printed worked value softplus(-4.6) ~ 0.01 (page "Mamba-2架构与LaCT并行计算
  技术解析" §1.1, fixture under tests/golden/);
* central finite differences of the oracle's forward for every gradient;
* invariants: linearity in X, head independence, packed sequences equal
  independent runs, the delta -> 0 and delta -> infinity limits, and splitting a
  sequence with the first part's final state carried over.
"""

import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(rng, bsz, L, H, P, N, G=1, raw_scale=0.5):
    x = rng.standard_normal((bsz, L, H, P))
    B = rng.standard_normal((bsz, L, G, N)) / np.sqrt(N)
    C = rng.standard_normal((bsz, L, G, N)) / np.sqrt(N)
    raw = rng.standard_normal((bsz, L, H)) * raw_scale
    return x, raw, B, C


def _quadratic_form(x, raw, B, C, delta_init):
    """y[t] = sum_{s<=t} exp(-sum_{k=s+1..t} delta_k) (C_t . B_s) delta_s x_s, per head,
    one sequence ([L, H, P] etc.), by explicit double loop over (t, s)."""
    L, H, P = x.shape
    G = B.shape[1]
    delta = np.logaddexp(0.0, raw + delta_init)  # softplus, independent of the oracle
    y = np.zeros_like(x)
    for h in range(H):
        g = h // (H // G)
        for t in range(L):
            for s in range(t + 1):
                decay = np.exp(-np.sum(delta[s + 1:t + 1, h]))
                y[t, h] += decay * np.dot(C[t, g], B[s, g]) * delta[s, h] * x[s, h]
    return y


@pytest.mark.parametrize("H,P,N,G", [(2, 3, 5, 1), (4, 2, 3, 2), (1, 4, 4, 1)])
def test_quadratic_form(oracle_mod, H, P, N, G):
    rng = np.random.default_rng(11)
    L = 37
    x, raw, B, C = _rand_problem(rng, 1, L, H, P, N, G, raw_scale=1.5)
    y, _ = oracle_mod.forward(x, raw, B, C, delta_init=-1.0)
    yq = _quadratic_form(x[0], raw[0], B[0], C[0], -1.0)
    np.testing.assert_allclose(y[0], yq, rtol=1e-11, atol=1e-13)


def test_final_state_is_sum_of_outer_products(oracle_mod):
    """final_state = sum_s exp(-sum_{k>s} delta_k) delta_s x_s B_s^T (P x N, not N x P)."""
    rng = np.random.default_rng(3)
    L, H, P, N = 23, 2, 3, 5
    x, raw, B, C = _rand_problem(rng, 1, L, H, P, N)
    _, hT = oracle_mod.forward(x, raw, B, C, delta_init=-2.0)
    delta = np.logaddexp(0.0, raw[0] - 2.0)
    for h in range(H):
        ref = np.zeros((P, N))
        for s in range(L):
            ref += np.exp(-delta[s + 1:, h].sum()) * delta[s, h] * np.outer(x[0, s, h], B[0, s, 0])
        np.testing.assert_allclose(hT[0, h], ref, rtol=1e-12, atol=1e-14)


def test_impulse_closed_form(oracle_mod):
    """Constant delta and x = e_p at t0 only: y_t = delta exp(-delta (t - t0)) (C_t . B_t0) e_p."""
    rng = np.random.default_rng(5)
    L, H, P, N = 50, 1, 4, 6
    t0, p = 17, 2
    raw_c, dinit = 0.3, -1.2
    x = np.zeros((1, L, H, P))
    x[0, t0, 0, p] = 1.0
    B = rng.standard_normal((1, L, 1, N))
    C = rng.standard_normal((1, L, 1, N))
    raw = np.full((1, L, H), raw_c)
    y, _ = oracle_mod.forward(x, raw, B, C, delta_init=dinit)
    delta = np.log1p(np.exp(raw_c + dinit))
    expect = np.zeros((L, P))
    for t in range(t0, L):
        expect[t, p] = delta * np.exp(-delta * (t - t0)) * np.dot(C[0, t, 0], B[0, t0, 0])
    np.testing.assert_allclose(y[0, :, 0, :], expect, rtol=1e-12, atol=1e-15)
    assert np.all(y[0, :t0] == 0.0)


def test_softplus_printed_value(oracle_mod):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "softplus_delta_init.txt"))
            if l.strip() and not l.startswith("#")]
    assert rows
    for dinit, printed, tol in rows:
        got = oracle_mod.softplus(float(dinit))
        assert abs(got - float(printed)) <= float(tol)
        # and the oracle's softplus is the exact log(1 + e^z) (checked at the same point
        # against the naive formula, which is accurate there)
        assert abs(got - np.log(1.0 + np.exp(float(dinit)))) < 1e-15


def test_softplus_extremes(oracle_mod):
    assert oracle_mod.softplus(-800.0) == 0.0
    assert oracle_mod.softplus(800.0) == 800.0
    assert abs(oracle_mod.softplus(0.0) - np.log(2.0)) < 1e-15


def _loss(oracle_mod, x, raw, B, C, dy, dinit, cu, h0, dhT):
    y, hT = oracle_mod.forward(x, raw, B, C, dinit, cu_seqlens=cu, initial_state=h0)
    return float(np.sum(y * dy) + np.sum(hT * dhT))


@pytest.mark.parametrize("varlen", [False, True])
def test_backward_finite_differences(oracle_mod, varlen):
    rng = np.random.default_rng(7 + varlen)
    L, H, P, N, G = 11, 2, 3, 4, 1
    x, raw, B, C = _rand_problem(rng, 1, L, H, P, N, G, raw_scale=1.0)
    cu = np.array([0, 4, 11], dtype=np.int32) if varlen else None
    nseq = 2 if varlen else 1
    dy = rng.standard_normal(x.shape)
    h0 = rng.standard_normal((nseq, H, P, N))
    dhT = rng.standard_normal((nseq, H, P, N))
    dinit = -0.7
    g = oracle_mod.backward(x, raw, B, C, dy, dinit, cu_seqlens=cu, initial_state=h0,
                            d_final_state=dhT)
    eps = 1e-6
    args = {"x": x, "raw": raw, "B": B, "C": C, "h0": h0}
    names = {"x": "dx", "raw": "d_raw_dt", "B": "dB", "C": "dC", "h0": "d_initial_state"}
    for key, arr in args.items():
        num = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp = _loss(oracle_mod, args["x"], args["raw"], args["B"], args["C"], dy, dinit, cu,
                       args["h0"], dhT)
            flat[i] = old - eps
            lm = _loss(oracle_mod, args["x"], args["raw"], args["B"], args["C"], dy, dinit, cu,
                       args["h0"], dhT)
            flat[i] = old
            num.reshape(-1)[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[names[key]], num, rtol=2e-6, atol=2e-8,
                                   err_msg="gradient of " + key)


def test_backward_long_sequence_crosses_checkpoints(oracle_mod):
    """Several checkpoint blocks: directional derivative against finite differences."""
    rng = np.random.default_rng(9)
    L, H, P, N = 700, 1, 2, 3
    x, raw, B, C = _rand_problem(rng, 1, L, H, P, N)
    dy = rng.standard_normal(x.shape)
    dinit = -3.0
    g = oracle_mod.backward(x, raw, B, C, dy, dinit)
    dirs = {k: rng.standard_normal(v.shape) for k, v in
            {"x": x, "raw": raw, "B": B, "C": C}.items()}
    eps = 1e-5

    def loss(s):
        y, _ = oracle_mod.forward(x + s * dirs["x"], raw + s * dirs["raw"], B + s * dirs["B"],
                                  C + s * dirs["C"], dinit)
        return float(np.sum(y * dy))

    num = (loss(eps) - loss(-eps)) / (2 * eps)
    ana = (np.sum(g["dx"] * dirs["x"]) + np.sum(g["d_raw_dt"] * dirs["raw"])
           + np.sum(g["dB"] * dirs["B"]) + np.sum(g["dC"] * dirs["C"]))
    assert abs(num - ana) <= 1e-6 * max(1.0, abs(ana))


def test_linear_in_x(oracle_mod):
    rng = np.random.default_rng(1)
    x1, raw, B, C = _rand_problem(rng, 2, 30, 3, 4, 5)
    x2 = rng.standard_normal(x1.shape)
    y1, s1 = oracle_mod.forward(x1, raw, B, C, -4.6)
    y2, s2 = oracle_mod.forward(x2, raw, B, C, -4.6)
    y3, s3 = oracle_mod.forward(2.5 * x1 - 0.75 * x2, raw, B, C, -4.6)
    np.testing.assert_allclose(y3, 2.5 * y1 - 0.75 * y2, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s3, 2.5 * s1 - 0.75 * s2, rtol=1e-11, atol=1e-13)


def test_heads_independent(oracle_mod):
    rng = np.random.default_rng(2)
    x, raw, B, C = _rand_problem(rng, 1, 40, 5, 3, 4)
    perm = np.array([3, 0, 4, 1, 2])
    y, s = oracle_mod.forward(x, raw, B, C, -2.0)
    yp, sp = oracle_mod.forward(x[:, :, perm], raw[:, :, perm], B, C, -2.0)
    np.testing.assert_array_equal(yp, y[:, :, perm])
    np.testing.assert_array_equal(sp, s[:, perm])


def test_packed_equals_independent_runs(oracle_mod):
    rng = np.random.default_rng(4)
    lens = [13, 1, 30, 7]
    T = sum(lens)
    x, raw, B, C = _rand_problem(rng, 1, T, 2, 3, 4)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    y, s = oracle_mod.forward(x, raw, B, C, -1.0, cu_seqlens=cu)
    for i, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        yi, si = oracle_mod.forward(x[:, a:b], raw[:, a:b], B[:, a:b], C[:, a:b], -1.0)
        np.testing.assert_array_equal(y[:, a:b], yi)
        np.testing.assert_array_equal(s[i], si[0])
    # and a dense batch is the packed run with equal lengths
    xb = x[:, :36].reshape(2, 18, 2, 3)
    yb, sb = oracle_mod.forward(xb, raw[:, :36].reshape(2, 18, 2), B[:, :36].reshape(2, 18, 1, 4),
                                C[:, :36].reshape(2, 18, 1, 4), -1.0)
    yc, sc = oracle_mod.forward(x[:, :36], raw[:, :36], B[:, :36], C[:, :36], -1.0,
                                cu_seqlens=np.array([0, 18, 36], dtype=np.int32))
    np.testing.assert_array_equal(yb.reshape(1, 36, 2, 3), yc)
    np.testing.assert_array_equal(sb, sc)


def test_small_delta_forgets_nothing_and_adds_nothing(oracle_mod):
    """raw -> -infinity: delta -> 0, so nothing enters the state and y -> 0."""
    rng = np.random.default_rng(6)
    x, raw, B, C = _rand_problem(rng, 1, 25, 2, 3, 4)
    y, s = oracle_mod.forward(x, np.full_like(raw, -60.0), B, C, -4.6)
    assert np.max(np.abs(y)) < 1e-25 and np.max(np.abs(s)) < 1e-25


def test_large_delta_is_memoryless(oracle_mod):
    """raw -> +infinity: exp(-delta) -> 0, so y_t = delta_t (C_t . B_t) x_t."""
    rng = np.random.default_rng(8)
    x, raw, B, C = _rand_problem(rng, 1, 25, 2, 3, 4)
    raw = 40.0 + rng.random(raw.shape)
    y, _ = oracle_mod.forward(x, raw, B, C, -1.0)
    delta = np.logaddexp(0.0, raw - 1.0)
    cb = np.sum(C[0, :, 0] * B[0, :, 0], axis=-1)
    expect = delta[0][:, :, None] * cb[:, None, None] * x[0]
    np.testing.assert_allclose(y[0], expect, rtol=1e-12, atol=1e-14)


def test_split_with_carried_state(oracle_mod):
    """Continuing from the first part's final state reproduces the whole run."""
    rng = np.random.default_rng(10)
    L, T1 = 60, 23
    x, raw, B, C = _rand_problem(rng, 1, L, 3, 2, 5)
    h0 = rng.standard_normal((1, 3, 2, 5))
    y, s = oracle_mod.forward(x, raw, B, C, -2.0, initial_state=h0)
    ya, sa = oracle_mod.forward(x[:, :T1], raw[:, :T1], B[:, :T1], C[:, :T1], -2.0,
                                initial_state=h0)
    yb, sb = oracle_mod.forward(x[:, T1:], raw[:, T1:], B[:, T1:], C[:, T1:], -2.0,
                                initial_state=sa)
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=1), y, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(sb, s, rtol=1e-13, atol=1e-15)


def test_rejects_bad_boundaries(oracle_mod):
    rng = np.random.default_rng(12)
    x, raw, B, C = _rand_problem(rng, 1, 10, 1, 2, 2)
    with pytest.raises(ValueError):
        oracle_mod.forward(x, raw, B, C, -1.0, cu_seqlens=np.array([0, 7, 5, 10]))
    with pytest.raises(ValueError):
        oracle_mod.forward(x, raw, B, C, -1.0, cu_seqlens=np.array([0, 4, 9]))


def _reverse_quadratic_form(x, raw, B, C, delta_init):
    """The right-to-left recurrence H_t = exp(-delta_t) H_{t+1} + delta_t x_t B_t^T,
    y_t = H_t C_t, written out as its upper-triangular quadratic form:
    y[t] = sum_{s>=t} exp(-sum_{k=t..s-1} delta_k) (C_t . B_s) delta_s x_s."""
    L, H, P = x.shape
    G = B.shape[1]
    delta = np.logaddexp(0.0, raw + delta_init)
    y = np.zeros_like(x)
    for h in range(H):
        g = h // (H // G)
        for t in range(L):
            for s in range(t, L):
                decay = np.exp(-np.sum(delta[t:s, h]))
                y[t, h] += decay * np.dot(C[t, g], B[s, g]) * delta[s, h] * x[s, h]
    return y


def test_bidirectional_halves(oracle_mod):
    """Bidirectional mode (page "Mamba-2架构与LaCT并行计算技术解析" §3.1): the first half
    of each output row is the causal quadratic form, the second the reverse one, per packed
    sequence."""
    rng = np.random.default_rng(17)
    H, P, N = 2, 3, 4
    cu = np.array([0, 9, 10, 25], dtype=np.int32)
    x, raw, B, C = _rand_problem(rng, 1, 25, H, P, N, raw_scale=1.0)
    y, ff, fr = oracle_mod.bidirectional_forward(x, raw, B, C, -1.0, cu_seqlens=cu)
    assert y.shape == (1, 25, H, 2 * P)
    for s in range(3):
        a, b = cu[s], cu[s + 1]
        np.testing.assert_allclose(y[0, a:b, :, :P], _quadratic_form(
            x[0, a:b], raw[0, a:b], B[0, a:b], C[0, a:b], -1.0), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(y[0, a:b, :, P:], _reverse_quadratic_form(
            x[0, a:b], raw[0, a:b], B[0, a:b], C[0, a:b], -1.0), rtol=1e-11, atol=1e-13)


def test_bidirectional_reversal_swaps_halves(oracle_mod):
    """Reversing every sequence swaps the two directions (and reverses the tokens)."""
    rng = np.random.default_rng(18)
    x, raw, B, C = _rand_problem(rng, 2, 14, 2, 3, 4)
    y, ff, fr = oracle_mod.bidirectional_forward(x, raw, B, C, -0.5)
    r = lambda a: np.ascontiguousarray(a[:, ::-1])  # noqa: E731
    y2, ff2, fr2 = oracle_mod.bidirectional_forward(r(x), r(raw), r(B), r(C), -0.5)
    np.testing.assert_allclose(y2[..., :3], r(y[..., 3:]), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y2[..., 3:], r(y[..., :3]), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ff2, fr, rtol=1e-12, atol=1e-14)


def test_bidirectional_backward_finite_differences(oracle_mod):
    rng = np.random.default_rng(19)
    cu = np.array([0, 5, 12], dtype=np.int32)
    x, raw, B, C = _rand_problem(rng, 1, 12, 2, 2, 3, raw_scale=1.0)
    dy = rng.standard_normal((1, 12, 2, 4))
    g = oracle_mod.bidirectional_backward(x, raw, B, C, dy, -1.0, cu_seqlens=cu)

    def loss(x_, raw_, B_, C_):
        y, _, _ = oracle_mod.bidirectional_forward(x_, raw_, B_, C_, -1.0, cu_seqlens=cu)
        return float(np.sum(y * dy))

    eps = 1e-6
    for name, arr, idx in (("dx", x, (0, 3, 1, 0)), ("dx", x, (0, 10, 0, 1)),
                           ("d_raw_dt", raw, (0, 2, 1)), ("d_raw_dt", raw, (0, 7, 0)),
                           ("dB", B, (0, 4, 0, 2)), ("dC", C, (0, 9, 0, 1))):
        hi, lo = arr.copy(), arr.copy()
        hi[idx] += eps
        lo[idx] -= eps
        args_hi = [hi if a is arr else a for a in (x, raw, B, C)]
        args_lo = [lo if a is arr else a for a in (x, raw, B, C)]
        fd = (loss(*args_hi) - loss(*args_lo)) / (2 * eps)
        assert abs(fd - g[name][idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[name][idx])
