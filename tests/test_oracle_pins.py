"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each check below compares the oracle with an independent statement of the same
mathematics: the SVD closed form of a matrix polynomial iteration, scalar
recurrences on 1x1 / row / diagonal inputs, invariants of orthogonalisation,
the momentum recurrence's closed form, the IEEE definition of bf16 rounding
(checked against PyTorch's cast), and brute-force optima for the partition.
The mutation tests at the end plant plausible mistakes in copies of the oracle
and show that these pins reject them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import muon_oracle as mo

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _p(t, abc=oracle.NS_COEFFS):
    a, b, c = abc
    return a * t + b * t ** 3 + c * t ** 5


def _pk(t, k, abc=oracle.NS_COEFFS):
    for _ in range(k):
        t = _p(t, abc)
    return t


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def svd_closed_form(G, k, abc=oracle.NS_COEFFS, eps=oracle.NS_EPS):
    """U p^k(S) V^T of the normalised matrix, via numpy's SVD (no NS code)."""
    G = np.asarray(G, np.float64)
    X0 = G / (np.sqrt((G ** 2).sum()) + eps)
    U, S, Vt = np.linalg.svd(X0, full_matrices=False)
    return (U * _pk(S, k, abc)) @ Vt


# ---------------------------------------------------------------- constants
def test_constants_match_golden():
    g = json.load(open(os.path.join(GOLD, "muon_constants.json")))
    assert oracle.DEFAULT_LR == g["lr"]["value"]
    assert oracle.DEFAULT_NS_STEPS == g["ns_steps"]["value"]
    assert tuple(oracle.NS_COEFFS) == tuple(g["ns_coeffs"]["value"])
    assert oracle.NS_EPS == g["ns_eps"]["value"]
    assert oracle.DEFAULT_BETA == g["beta"]["value"]


# ------------------------------------------------------- NS: closed forms
@pytest.mark.parametrize("shape", [(256, 1024), (1024, 256), (64, 64), (2, 3), (3, 2),
                                   (37, 100), (100, 37), (1, 5), (5, 1)])
@pytest.mark.parametrize("k", [0, 1, 3, 5, 8])
def test_ns_matches_svd_closed_form(shape, k):
    G = np.random.default_rng(hash(shape) % 2 ** 31 + k).standard_normal(shape)
    O = oracle.newton_schulz(G, k)
    assert O.shape == G.shape
    assert _rel(O, svd_closed_form(G, k)) < 1e-12


@pytest.mark.parametrize("g", [3.0, -0.25, 1e-3, -7.5e4])
@pytest.mark.parametrize("k", [0, 1, 5])
def test_ns_scalar_brute_force(g, k):
    t = g / (abs(g) + 1e-7)
    exp = t
    for _ in range(k):
        exp = 3.4445 * exp - 4.7750 * exp ** 3 + 2.0315 * exp ** 5
    got = oracle.newton_schulz(np.array([[g]]), k)[0, 0]
    assert abs(got - exp) <= 1e-14 * max(1.0, abs(exp))


@pytest.mark.parametrize("n", [1, 4, 33])
def test_ns_row_and_column_vectors(n):
    u = np.random.default_rng(n).standard_normal(n)
    nu = math.sqrt(float(u @ u))
    exp = u * _pk(nu / (nu + 1e-7), 5) / nu
    row = oracle.newton_schulz(u[None, :], 5)
    col = oracle.newton_schulz(u[:, None], 5)
    assert np.allclose(row[0], exp, rtol=1e-13, atol=1e-15)
    assert np.allclose(col[:, 0], exp, rtol=1e-13, atol=1e-15)


def test_ns_diagonal_2x2_keeps_signs():
    D = np.diag([3.0, -4.0])
    fro = 5.0 + 1e-7
    O = oracle.newton_schulz(D, 5)
    assert abs(O[0, 1]) < 1e-15 and abs(O[1, 0]) < 1e-15
    assert abs(O[0, 0] - _pk(3.0 / fro, 5)) < 1e-14
    assert abs(O[1, 1] + _pk(4.0 / fro, 5)) < 1e-14


def test_ns_zero_matrix_is_zero():
    assert not np.any(oracle.newton_schulz(np.zeros((4, 9)), 5))
    assert not np.any(oracle.gram_newton_schulz(np.zeros((9, 4)), 5))


# ------------------------------------------------------------ invariants
def _band(k):
    t = np.linspace(0.0, 1.0, 200001)
    v = _pk(t, k)
    return float(v.min()), float(v.max())


@pytest.mark.parametrize("shape", [(256, 1024), (128, 128), (300, 40)])
def test_ns_singular_value_band(shape):
    lo, hi = _band(5)
    G = np.random.default_rng(7).standard_normal(shape)
    s = np.linalg.svd(oracle.newton_schulz(G, 5), compute_uv=False)
    assert s.max() <= hi + 1e-12 and s.min() >= lo - 1e-12
    # inputs well away from zero land in the narrow band of the quintic
    t = np.linspace(0.01, 1.0, 100001)
    v = _pk(t, 5)
    s0 = np.linalg.svd(G / (np.linalg.norm(G) + 1e-7), compute_uv=False)
    in_band = np.sum((s >= v.min() - 1e-12) & (s <= v.max() + 1e-12))
    assert in_band >= np.sum(s0 >= 0.01)


def _orth(n, seed):
    q, r = np.linalg.qr(np.random.default_rng(seed).standard_normal((n, n)))
    return q * np.sign(np.diag(r))


@pytest.mark.parametrize("shape", [(48, 80), (80, 48), (50, 50)])
def test_ns_rotation_invariance(shape):
    G = np.random.default_rng(11).standard_normal(shape)
    Q1, Q2 = _orth(shape[0], 1), _orth(shape[1], 2)
    lhs = oracle.newton_schulz(Q1 @ G @ Q2, 5)
    rhs = Q1 @ oracle.newton_schulz(G, 5) @ Q2
    assert _rel(lhs, rhs) < 1e-11


@pytest.mark.parametrize("shape", [(40, 90), (64, 64)])
def test_ns_transpose_symmetry(shape):
    G = np.random.default_rng(5).standard_normal(shape)
    assert _rel(oracle.newton_schulz(G.T, 5), oracle.newton_schulz(G, 5).T) < 1e-12


# ------------------------------------------------------------------ Gram
@pytest.mark.parametrize("shape", [(64, 256), (256, 64), (96, 96), (3, 7)])
@pytest.mark.parametrize("k", [0, 1, 3, 5, 8])
def test_gram_equals_svd_closed_form(shape, k):
    G = np.random.default_rng(k + 100).standard_normal(shape)
    assert _rel(oracle.gram_newton_schulz(G, k), svd_closed_form(G, k)) < 1e-6


# -------------------------------------------------------------- momentum
def test_momentum_constant_gradient_closed_form():
    beta = 0.95
    G = np.random.default_rng(3).standard_normal((5, 7))
    M = np.zeros_like(G)
    for t in range(1, 8):
        M, U = oracle.nesterov_momentum(G, M, beta)
        assert np.allclose(M, (1 - beta ** t) * G, rtol=1e-14, atol=0)
        assert np.allclose(U, (1 - beta) * G + beta * (1 - beta ** t) * G, rtol=1e-14, atol=0)


def test_momentum_hand_worked():
    # beta = 0.9; g1 = 1: M1 = 0.1, U1 = 0.1 + 0.9*0.1 = 0.19
    #             g2 = 2: M2 = 0.09 + 0.2 = 0.29, U2 = 0.2 + 0.9*0.29 = 0.461
    M1, U1 = oracle.nesterov_momentum(np.array([[1.0]]), np.zeros((1, 1)), 0.9)
    M2, U2 = oracle.nesterov_momentum(np.array([[2.0]]), M1, 0.9)
    assert abs(M1[0, 0] - 0.1) < 1e-15 and abs(U1[0, 0] - 0.19) < 1e-15
    assert abs(M2[0, 0] - 0.29) < 1e-15 and abs(U2[0, 0] - 0.461) < 1e-15


# ---------------------------------------------------------------- update
def test_update_scale_and_sign():
    assert oracle.update_scale(4, 1) == 2.0
    assert oracle.update_scale(1, 4) == 1.0 and oracle.update_scale(3, 3) == 1.0
    W = np.ones((4, 1))
    O = np.full((4, 1), 0.5)
    assert np.allclose(oracle.apply_update(W, O, 0.02), 1.0 - 0.02 * 2.0 * 0.5)


def test_muon_step_scalar_end_to_end():
    g, w = 2.0, 0.3
    M, O, Wn = oracle.muon_step(np.array([[g]]), np.zeros((1, 1)), np.array([[w]]),
                                lr=0.02, beta=0.95, ns_steps=5)
    u = 0.05 * g + 0.95 * 0.05 * g
    t = _pk(u / (abs(u) + 1e-7), 5)
    assert abs(M[0, 0] - 0.05 * g) < 1e-15
    assert abs(O[0, 0] - t) < 1e-14
    assert abs(Wn[0, 0] - (w - 0.02 * t)) < 1e-14


# --------------------------------------------------------- bf16 rounding
def test_round_bf16_hand_cases():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, 2.0 ** -133,
                  3 * 2.0 ** -134, 3.5e38, np.inf, -np.inf])
    exp = np.array([1.0, 1.0 + 2 ** -6, -1.0, 0.0, 2.0 ** -133, 2 * 2.0 ** -133, np.inf,
                    np.inf, -np.inf])
    assert np.array_equal(oracle.round_bf16(x), exp)
    assert np.isnan(oracle.round_bf16(np.array([np.nan]))[0])


def test_round_bf16_matches_torch_cast_on_fp32_values():
    rng = np.random.default_rng(0)
    parts = [rng.standard_normal(200000).astype(np.float32) * np.float32(s)
             for s in (1.0, 1e-3, 1e-38, 1e30)]
    # exact ties: bf16 value + half a bf16 spacing, representable in fp32
    base = rng.standard_normal(20000).astype(np.float32)
    bits = base.view(np.uint32) & np.uint32(0xFFFF0000)
    parts.append((bits | np.uint32(0x8000)).view(np.float32))
    x = np.concatenate(parts)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


# ------------------------------------------------------- partition / pack
def test_lpt_hand_worked_example():
    g = json.load(open(os.path.join(GOLD, "lpt_worked_example.json")))
    own = oracle.lpt_assign(g["sizes"], g["n_owners"])
    assert own == g["owner_of"]
    loads = [sum(s for s, o in zip(g["sizes"], own) if o == k) for k in range(g["n_owners"])]
    assert loads == g["loads"]


def test_lpt_within_graham_bound_of_brute_force_optimum():
    rng = np.random.default_rng(1)
    for _ in range(60):
        n, m = int(rng.integers(1, 8)), int(rng.integers(1, 4))
        sizes = [int(v) for v in rng.integers(1, 50, n)]
        own = oracle.lpt_assign(sizes, m)
        lpt_max = max(sum(s for s, o in zip(sizes, own) if o == k) for k in range(m))
        opt = min(max(sum(s for s, o in zip(sizes, a) if o == k) for k in range(m))
                  for a in itertools.product(range(m), repeat=n))
        assert lpt_max <= (4.0 / 3.0 - 1.0 / (3.0 * m)) * opt + 1e-9
        assert sorted(set(own)) <= list(range(m))


@pytest.mark.parametrize("n_owners", [1, 3, 8])
def test_pack_plan_layout(n_owners):
    shapes = [(7, 300), (256, 1536), (1, 1), (64, 64), (300, 7), (5, 129)] * 3
    own, off, oel = oracle.pack_plan(shapes, n_owners)
    A = oracle.PACK_ALIGN_ELEMS
    starts = np.cumsum([0] + oel[:-1])
    segs = []
    for i, (r, c) in enumerate(shapes):
        o = own[i]
        assert off[i] % A == 0
        assert starts[o] <= off[i] and off[i] + r * c <= starts[o] + oel[o]
        segs.append((off[i], off[i] + r * c))
    segs.sort()
    assert all(e0 <= s1 for (_, e0), (s1, _) in zip(segs, segs[1:]))
    for o in range(n_owners):   # parameter order inside one owner buffer
        mine = [off[i] for i in range(len(shapes)) if own[i] == o]
        assert mine == sorted(mine)


def test_flop_counts_hand_worked():
    # m = 2, n = 3: 3*m^2*n + m^3 = 36 + 8 = 44 per step
    assert oracle.ns_flops_algorithmic([(3, 2)], 1) == 44.0
    assert oracle.ns_flops_algorithmic([(2, 3)], 5) == 220.0
    # Gram, 1 step: 3 m^2 n + A^2 = 36 + 8
    assert oracle.gram_ns_flops_algorithmic([(2, 3)], 1) == 44.0
    # Gram, 2 steps: 36 + (8 + 16) + (8 + 8) = 76
    assert oracle.gram_ns_flops_algorithmic([(2, 3)], 2) == 76.0


# --------------------------------------------- planted mistakes are caught
def _ns_mutant(kind):
    def f(U, k=5, abc=oracle.NS_COEFFS, eps=oracle.NS_EPS):
        a, b, c = abc
        X, tr = mo.ns_working_matrix(U)
        X = X / (np.linalg.norm(X) + eps)
        for _ in range(k):
            A = X @ X.T
            if kind == "drop_c":
                B = b * A
            elif kind == "sign_b":
                B = -b * A + c * (A @ A)
            elif kind == "coeff":
                B = b * A + 2.0 * (A @ A)
            else:
                B = b * A + c * (A @ A)
            X = a * X + B @ X
        if kind == "no_untranspose":
            return X.copy()
        return X.T.copy() if tr else X
    return f


@pytest.mark.parametrize("kind", ["drop_c", "sign_b", "coeff", "no_untranspose"])
def test_planted_ns_mistakes_fail_the_pins(kind):
    G = np.random.default_rng(0).standard_normal((24, 40))
    Gt = G.T.copy()
    f = _ns_mutant(kind)
    bad = (_rel(f(G, 5), svd_closed_form(G, 5)) > 1e-6 or
           f(Gt, 5).shape != Gt.shape or _rel(f(Gt, 5), svd_closed_form(Gt, 5)) > 1e-6)
    assert bad, kind
    # the unmutated copy passes, so the check itself is not vacuous
    assert _rel(_ns_mutant("none")(G, 5), svd_closed_form(G, 5)) < 1e-12


# ------------------------------------------------------------------ AdamW
def test_adamw_matches_torch_optim_adamw():
    rng = np.random.default_rng(4)
    p0 = rng.standard_normal((7, 33))
    grads = [rng.standard_normal((7, 33)) for _ in range(4)]
    tp = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([tp], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    for t, g in enumerate(grads, start=1):
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = oracle.adamw_step(p, g, m, v, t)
        assert np.allclose(p, tp.detach().numpy(), rtol=1e-13, atol=1e-15)
        st = opt.state[tp]
        assert np.allclose(m, st["exp_avg"].numpy(), rtol=1e-13, atol=0)
        assert np.allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=0)


def test_adamw_constant_gradient_closed_form():
    # with a constant gradient the bias-corrected moments are exactly g and g^2,
    # so each step moves p by lr * g / (|g| + eps) after the decay
    g = np.array([[0.5, -2.0, 3e-3]])
    p = np.array([[1.0, 1.0, -1.0]])
    m = v = np.zeros_like(g)
    for t in range(1, 6):
        p_dec = p * (1 - 1e-3 * 0.01)
        p, m, v = oracle.adamw_step(p, g, m, v, t)
        assert np.allclose(p, p_dec - 1e-3 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=1e-15)


def test_adamw_defaults_golden():
    assert oracle.ADAMW_DEFAULT_LR == json.load(open(os.path.join(GOLD, "muon_constants.json")))[
        "adamw_lr"]["value"]
