"""Pins for the fp64 oracle: closed forms, a second library route, invariants, brute force.

None of these compare the oracle with a retyped copy of itself.  The Newton-Schulz
closed form follows from the iteration's algebra: for X = U diag(s) V^T with U, V
orthonormal columns, every iterate stays U diag(sigma) V^T with sigma <- p(sigma),
p(x) = a x + b x^3 + c x^5, starting from sigma = s/||s||_2; so the output is
U diag(p^k(s/||s||)) V^T.  p is evaluated here on scalars (exact rationals where the
singular values are rational), never through the oracle's matrix code.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import muon_ref as ref
from muon_optimizer_step_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))
A_EXACT = Fraction(34445, 10000)
B_EXACT = Fraction(-47750, 10000)
C_EXACT = Fraction(20315, 10000)


def p_exact(x: Fraction, k: int) -> Fraction:
    for _ in range(k):
        x = A_EXACT * x + B_EXACT * x ** 3 + C_EXACT * x ** 5
    return x


def p_float(x: float, k: int, coeffs=(3.4445, -4.7750, 2.0315)) -> float:
    a, b, c = coeffs
    for _ in range(k):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def rel(x, y):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    return float(np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300))


def random_orthonormal(rng, n, k):
    q, r = np.linalg.qr(rng.normal(size=(n, k)))
    return q * np.sign(np.diag(r))


# ------------------------------------------------------------------ hand-checkable values
def test_p_at_one_is_sum_of_coefficients():
    # p(1) = a + b + c = 3.4445 - 4.7750 + 2.0315 = 0.7010, by hand.
    assert p_exact(Fraction(1), 1) == Fraction(701, 1000)
    assert ref.NS_A + ref.NS_B + ref.NS_C == pytest.approx(0.701, abs=1e-15)


def test_coefficients_are_the_quintic_ones():
    assert (ref.NS_A, ref.NS_B, ref.NS_C) == (3.4445, -4.7750, 2.0315)


# ------------------------------------------------------------------ golden fixture
def _monomial_closed_form(X, k):
    """NS of a matrix with at most one nonzero per row and column, exactly.

    Such X is a scaled partial permutation: its singular values are |x_ij| and
    X X^T is diagonal, so each entry maps to sign(x) * p^k(|x| / ||X||_F).
    """
    X = [[Fraction(v).limit_denominator(10 ** 6) for v in row] for row in X]
    nu2 = sum(v * v for row in X for v in row)
    nu = Fraction(math.isqrt(nu2.numerator), math.isqrt(nu2.denominator))
    assert nu * nu == nu2, "fixture chosen with a rational norm"
    out = []
    for row in X:
        orow = []
        for v in row:
            if v == 0:
                orow.append(0.0)
            else:
                sgn = 1 if v > 0 else -1
                orow.append(float(sgn * p_exact(abs(v) / nu, k)))
        out.append(orow)
    return np.array(out)


def test_golden_fixture_matches_oracle_and_closed_form():
    with open(os.path.join(HERE, "golden", "ns_small_cases.json")) as f:
        gold = json.load(f)
    assert gold["coeffs"] == [3.4445, -4.775, 2.0315]
    for case in gold["cases"]:
        X = np.array(case["input"], dtype=np.float64)
        k = case["ns_steps"]
        O = ref.newton_schulz(X, k)
        np.testing.assert_allclose(O, np.array(case["output"]), rtol=1e-13, atol=1e-15,
                                   err_msg=case["name"])
        nz = (X != 0)
        if np.all(nz.sum(0) <= 1) and np.all(nz.sum(1) <= 1):
            np.testing.assert_allclose(O, _monomial_closed_form(case["input"], k), rtol=1e-13,
                                       atol=1e-15, err_msg=case["name"])
        else:  # rank-1 case: O = p^k(1) * X / ||X||
            np.testing.assert_allclose(O, p_float(1.0, k) * X / np.linalg.norm(X),
                                       rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ closed form, random U, V
@pytest.mark.parametrize("shape,k", [((6, 10), 6), ((12, 5), 5), ((8, 8), 8), ((7, 9), 3),
                                     ((256, 128), 128)])
def test_ns_closed_form_random_orthogonal(shape, k):
    rng = np.random.default_rng(hash(shape) % 2 ** 32)
    r, c = shape
    U = random_orthonormal(rng, r, k)
    V = random_orthonormal(rng, c, k)
    s = rng.uniform(0.05, 3.0, size=k)
    G = U @ np.diag(s) @ V.T
    want = U @ np.diag([p_float(x, 5) for x in s / np.linalg.norm(s)]) @ V.T
    got = ref.newton_schulz(G, 5)
    assert got.shape == G.shape
    assert rel(got, want) < 1e-12


def test_ns_closed_form_orthogonal_input_value():
    # A 128 x 128 orthogonal input has all s/||s|| = 1/sqrt(128).
    rng = np.random.default_rng(11)
    Q = random_orthonormal(rng, 128, 128)
    got = ref.newton_schulz(Q, 5)
    want = p_float(1 / math.sqrt(128), 5) * Q
    assert rel(got, want) < 1e-12


# ------------------------------------------------------------------ second route: SVD
@pytest.mark.parametrize("shape", [(5, 9), (9, 5), (7, 7), (1, 6), (6, 1), (33, 17)])
@pytest.mark.parametrize("steps", [0, 1, 5])
def test_ns_matches_svd_route(shape, steps):
    rng = np.random.default_rng(sum(shape) * 7 + steps)
    G = rng.normal(size=shape)
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    want = U @ np.diag([p_float(x, steps) for x in s / np.linalg.norm(s)]) @ Vt
    assert rel(ref.newton_schulz(G, steps), want) < 1e-12


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("shape", [(10, 16), (16, 10), (12, 12)])
def test_ns_invariants(shape):
    rng = np.random.default_rng(3)
    G = rng.normal(size=shape)
    O = ref.newton_schulz(G)
    for alpha in (1e-3, 7.5, 1e4):
        assert rel(ref.newton_schulz(alpha * G), O) < 1e-13       # scale invariance
    assert rel(ref.newton_schulz(-G), -O) < 1e-15                  # oddness
    assert rel(ref.newton_schulz(G.T), O.T) < 1e-13                # transpose symmetry
    Q = random_orthonormal(rng, shape[0], shape[0])
    R = random_orthonormal(rng, shape[1], shape[1])
    assert rel(ref.newton_schulz(Q @ G @ R), Q @ O @ R) < 1e-12    # orthogonal equivariance
    assert rel(ref.newton_schulz(G, 0), G / np.linalg.norm(G)) < 1e-15


def test_ns_rank_preserved_and_zero():
    rng = np.random.default_rng(5)
    G = rng.normal(size=(6, 2)) @ rng.normal(size=(2, 9))
    s = np.linalg.svd(ref.newton_schulz(G), compute_uv=False)
    assert np.all(s[2:] < 1e-12 * s[0])
    assert np.all(s[:2] > 0.4)
    Z = ref.newton_schulz(np.zeros((4, 7)))
    assert Z.shape == (4, 7) and not Z.any()


def test_ns_output_singular_values_in_known_band():
    # p^5 maps (0, 1] into roughly [0.47, 1.21] for inputs not too close to 0.
    rng = np.random.default_rng(8)
    G = rng.normal(size=(40, 64))
    s = np.linalg.svd(ref.newton_schulz(G), compute_uv=False)
    assert s.min() > 0.3 and s.max() < 1.25


# ------------------------------------------------------------------ planted mistakes
@pytest.mark.parametrize("coeffs", [(3.4445, 4.7750, 2.0315),    # sign of b
                                    (3.4445, -4.7750, 0.0),      # dropped c term
                                    (2.0315, -4.7750, 3.4445)])  # a and c swapped
def test_pins_catch_planted_coefficient_mistakes(coeffs):
    rng = np.random.default_rng(1)
    U = random_orthonormal(rng, 6, 4)
    V = random_orthonormal(rng, 10, 4)
    s = np.array([3.0, 1.0, 0.5, 0.1])
    G = U @ np.diag(s) @ V.T
    want = U @ np.diag([p_float(x, 5) for x in s / np.linalg.norm(s)]) @ V.T
    assert rel(ref.newton_schulz(G, 5, coeffs=coeffs), want) > 1e-3


def test_pins_catch_planted_operand_order_mistake(monkeypatch):
    # Plant "X <- a X + X B" (operands of the update swapped) into the oracle and check
    # that the SVD closed form catches it on a square input.
    def swapped(X, ns_steps=5, coeffs=(ref.NS_A, ref.NS_B, ref.NS_C)):
        a, b, c = coeffs
        X = np.asarray(X, dtype=np.float64)
        X = X / np.linalg.norm(X)
        for _ in range(ns_steps):
            A = X @ X.T
            X = a * X + X @ (b * A + c * A @ A)
        return X

    monkeypatch.setattr(ref, "newton_schulz", swapped)
    rng = np.random.default_rng(2)
    G = rng.normal(size=(9, 9))
    U, s, Vt = np.linalg.svd(G)
    want = U @ np.diag([p_float(x, 5) for x in s / np.linalg.norm(s)]) @ Vt
    assert rel(ref.newton_schulz(G, 5), want) > 1e-3


def test_pins_catch_planted_missing_transpose_back():
    # Forgetting to transpose a tall result back changes its shape.
    G = np.random.default_rng(3).normal(size=(12, 5))
    assert ref.newton_schulz(G).shape == (12, 5)
    assert ref.newton_schulz(G).T.shape != G.shape


def test_pins_catch_planted_nesterov_mistake():
    # Nesterov must use the momentum after the update; with M0 != 0 the two differ.
    rng = np.random.default_rng(4)
    G = rng.normal(size=16)
    M0 = rng.normal(size=16)
    mu = 0.9
    M1 = ref.momentum_update(M0, G, mu)
    np.testing.assert_allclose(ref.ns_input(G, M1, mu, True), G + mu * (mu * M0 + G),
                               rtol=1e-15)
    assert rel(ref.ns_input(G, M1, mu, True), G + mu * M0) > 1e-2


# ------------------------------------------------------------------ momentum / apply
def test_first_step_closed_form_single_256x128():
    wl = inputs.WORKLOADS["single_256x128"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    lay = ref.flat_layout(wl.shapes, 1, wl.is_matrix)
    W1, M1, upd = ref.muon_step(W0, Gs[0], M0, lay, wl.lr, wl.wd, wl.mu, True, 5)
    G1 = Gs[0].astype(np.float64)
    np.testing.assert_array_equal(M1, G1)                                  # M1 = G1
    O = ref.newton_schulz(G1.reshape(256, 128), 5)                         # NS(1.95 G) = NS(G)
    assert rel(upd[0], O) < 1e-13
    want = W0.astype(np.float64) * (1 - 0.02 * 0.01) - 0.02 * math.sqrt(2.0) * O.reshape(-1)
    assert rel(W1, want) < 1e-15
    # Second step by hand: M2 = mu G1 + G2, X2 = G2 + mu M2.
    W2, M2, upd2 = ref.muon_step(W1, Gs[1], M1, lay, wl.lr, wl.wd, wl.mu, True, 5)
    G2 = Gs[1].astype(np.float64)
    np.testing.assert_allclose(M2, 0.95 * G1 + G2, rtol=1e-15, atol=0)
    X2 = G2 + 0.95 * (0.95 * G1 + G2)
    assert rel(upd2[0], ref.newton_schulz(X2.reshape(256, 128))) < 1e-13


def test_plain_momentum_input_and_no_nesterov():
    G = np.arange(6.0)
    M = np.ones(6)
    M1 = ref.momentum_update(M, G, 0.5)
    np.testing.assert_array_equal(M1, 0.5 + G)
    np.testing.assert_array_equal(ref.ns_input(G, M1, 0.5, False), M1)


def test_update_scale_values():
    assert ref.update_scale(256, 128) == math.sqrt(2.0)
    assert ref.update_scale(128, 256) == 1.0
    assert ref.update_scale(14336, 4096) == math.sqrt(3.5)
    assert ref.update_scale(7, 7) == 1.0


# ------------------------------------------------------------------ layout / gather / scatter
def test_layout_shard_length_and_straddles():
    wl = inputs.WORKLOADS["llama3_8b_8shards"]
    lay = ref.flat_layout(wl.shapes, wl.n_shards, wl.is_matrix)
    assert lay["N"] == 6_979_325_952
    assert lay["L"] == 872_415_744 == -(-lay["N"] // 8)
    L = lay["L"]
    straddle = [i for i, (r, c) in enumerate(wl.shapes)
                if lay["offsets"][i] // L != (lay["offsets"][i] + r * c - 1) // L]
    # the down projection (index 6 in a layer) of layers 3, 7, ..., 27
    assert straddle == [1 + 7 * layer + 6 for layer in range(3, 28, 4)]
    plain = ref.flat_layout(inputs.WORKLOADS["llama3_8b_x32"].shapes, 8)
    Lp = plain["L"]
    assert not any(plain["offsets"][i] // Lp != (plain["offsets"][i] + r * c - 1) // Lp
                   for i, (r, c) in enumerate(plain["shapes"]))


@pytest.mark.parametrize("n_shards", [1, 2, 3, 7, 8])
def test_gather_scatter_brute_force(n_shards):
    shapes = [(3, 5), (4, 1), (2, 7), (1, 1), (6, 2)]
    is_matrix = [True, False, True, True, True]
    lay = ref.flat_layout(shapes, n_shards, is_matrix)
    N, L = lay["N"], lay["L"]
    # Label every flat position with its own index: the gather must hit each matrix
    # element exactly once, at the right row-major place.
    flat = np.arange(N, dtype=np.float64)
    shards = ref.shard_flat(flat, lay)
    assert all(len(s) == L for s in shards)
    full = ref.gather_full(shards, lay)
    seen = []
    for i, (r, c) in enumerate(shapes):
        if not is_matrix[i]:
            assert i not in full
            continue
        for rr in range(r):
            for cc in range(c):
                g = int(full[i][rr, cc])
                assert g == lay["offsets"][i] + rr * c + cc
                seen.append(g)
    assert len(seen) == len(set(seen))
    # scatter(gather(x)) = x everywhere; gather(scatter(y)) = y.
    back = ref.scatter_updates(full, lay, [np.full(L, -1.0) for _ in range(n_shards)])
    flat_back = np.concatenate(back)
    for i, (r, c) in enumerate(shapes):
        sl = slice(lay["offsets"][i], lay["offsets"][i] + r * c)
        if is_matrix[i]:
            np.testing.assert_array_equal(flat_back[sl], flat[sl])
        else:
            assert np.all(flat_back[sl] == -1.0)
    assert np.all(flat_back[N:] == -1.0)  # padding untouched
    rng = np.random.default_rng(n_shards)
    y = {i: rng.normal(size=s) for i, s in enumerate(shapes) if is_matrix[i]}
    y2 = ref.gather_full(ref.scatter_updates(y, lay, [np.zeros(L)] * n_shards), lay)
    for i in y:
        np.testing.assert_array_equal(y2[i], y[i])


@pytest.mark.parametrize("n_shards", [1, 3, 8])
def test_sharded_step_equals_unsharded_step(n_shards):
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    lay = ref.flat_layout(wl.shapes, n_shards, wl.is_matrix)
    W, M = W0.astype(np.float64), M0.astype(np.float64)
    Ws, Ms = ref.shard_flat(W, lay), ref.shard_flat(M, lay)
    for t in range(2):
        W, M, upd = ref.muon_step(W, Gs[t], M, lay, wl.lr, wl.wd, wl.mu, True, 5)
        Ws, Ms, upd_s = ref.muon_step_sharded(Ws, ref.shard_flat(Gs[t], lay), Ms, lay, wl.lr,
                                              wl.wd, wl.mu, True, 5)
        np.testing.assert_array_equal(ref.unshard_flat(Ws, lay), W)
        np.testing.assert_array_equal(ref.unshard_flat(Ms, lay), M)
        for i in upd:
            np.testing.assert_array_equal(upd_s[i], upd[i])


def test_non_matrix_parameters_untouched():
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    M0 = np.random.default_rng(0).normal(size=M0.size)
    lay = ref.flat_layout(wl.shapes, 1, wl.is_matrix)
    W1, M1, upd = ref.muon_step(W0, Gs[0], M0, lay, wl.lr, wl.wd, wl.mu, True, 5)
    off = lay["offsets"][1]
    n = lay["numels"][1]
    np.testing.assert_array_equal(W1[off:off + n], W0[off:off + n])
    np.testing.assert_array_equal(M1[off:off + n], M0[off:off + n])
    assert 1 not in upd


def test_input_generators_are_seeded_and_shaped():
    wl = inputs.WORKLOADS["single_256x128"]
    a = inputs.host_grads(wl, 0)
    b = inputs.host_grads(wl, 0)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, inputs.host_grads(wl, 1))
    G = a.reshape(256, 128).astype(np.float64)
    s = np.linalg.svd(G, compute_uv=False)
    # rank-4 part of norm 0.1 over N(0, 1e-3^2) noise (noise norm ~ 0.18)
    assert 0.15 < np.linalg.norm(G) < 0.25
    assert s[3] > 1.4 * s[4]
    assert inputs.WORKLOADS["llama3_8b_x32"].numel == 6_979_321_856
    assert inputs.WORKLOADS["gpt2_small_x12"].numel == 84_934_656
    assert inputs.WORKLOADS["moe_64e"].numel == 570_425_344
    assert inputs.WORKLOADS["moe_64e"].n_matrices == 196


def test_grouped_step_matches_per_group_steps_and_closed_form():
    wl = inputs.WORKLOADS["ragged_small"]
    W0, Gs, M0 = inputs.host_inputs(wl)
    M0 = np.random.default_rng(1).normal(0, 1e-3, M0.size)
    lay = ref.flat_layout(wl.shapes, 1, wl.is_matrix)
    group_of = [i % 3 for i in range(len(wl.shapes))]
    hp = [(0.02, 0.01, 0.95, True), (0.05, 0.0, 0.9, False), (0.001, 0.1, 0.5, True)]
    W, M, upd = ref.muon_step_grouped(W0, Gs[0], M0, lay, group_of, hp, 5)
    for g, (lr, wd, mu, nest) in enumerate(hp):
        Wg, Mg, ug = ref.muon_step(W0, Gs[0], M0, lay, lr, wd, mu, nest, 5)
        for i, (r, c) in enumerate(wl.shapes):
            if not wl.is_matrix[i] or group_of[i] != g:
                continue
            sl = slice(lay["offsets"][i], lay["offsets"][i] + r * c)
            np.testing.assert_array_equal(W[sl], Wg[sl])
            np.testing.assert_array_equal(M[sl], Mg[sl])
    # group 1 has no Nesterov: X = M1 = 0.9 M0 + G, W1 = W0 (1 - 0) - 0.05 s NS(X)
    i = 4  # (1, 50): group 1
    assert group_of[i] == 1
    r, c = wl.shapes[i]
    sl = slice(lay["offsets"][i], lay["offsets"][i] + r * c)
    X = (0.9 * M0[sl] + Gs[0][sl].astype(np.float64)).reshape(r, c)
    want = W0[sl].astype(np.float64) - 0.05 * 1.0 * ref.newton_schulz(X).reshape(-1)
    assert rel(W[sl], want) < 1e-15
