"""Plain fp64 CPU oracle for the DMuon owner-side Muon step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``newton_schulz_owner_gb300``) and imports
nothing from it.

What it computes, and where that comes from
-------------------------------------------
DMuon home page ("DMuon", sections "What DMuon Can Do" / "LLM Pretraining"):
each 2-D projection parameter has one owner; the owner runs Muon for it --
momentum, one Newton-Schulz orthogonalisation, update -- once per step
(owner section: each matrix is orthogonalised once, by its owner), with a
learning rate of 0.02 and 5 Newton-Schulz steps in the usage example.  "Z2 vs Z3 Modes" ("The two packed-buffer lifecycles"): all
Muon-target matrices that share an owner sit in one contiguous buffer.

The pages name Muon and Newton-Schulz but never write the formulas.  The
readings used here are the standard Muon ones:

* Nesterov momentum  M <- beta*M + (1-beta)*G ;  U = (1-beta)*G + beta*M
* X = U^T if rows > cols else U ;  X0 = X / (||X||_F + eps), eps = 1e-7
* ns_steps times:  A = X X^T ;  B = b*A + c*A A ;  X = a*X + B X
  with (a, b, c) = (3.4445, -4.7750, 2.0315)
* O = X^T if transposed, else X
* W <- W - lr * sqrt(max(1, rows/cols)) * O

Gram Newton-Schulz (home page, "VLA and VLM" and the closing credits) is only
named on the pages.  Reading: iterate on the m x m Gram matrix A = X0 X0^T
with P_k = a I + b A_k + c A_k^2, Q <- P_k Q, A_{k+1} = A_k P_k^2, and finish
with O = Q X0.  In exact arithmetic this equals the standard iteration,
because every P_k is a polynomial in A_0.

Owner partition (home page, "MoE": "balanced partition ensures no single rank
becomes a straggler") has no stated algorithm.  Reading: greedy longest
processing time (LPT) by element count.

Pins (each checked by ``tests/test_oracle_*.py`` against something other than
this file): SVD closed form of the quintic, scalar brute force on 1x1 / 1xn /
diagonal cases, singular-value band, rotation invariance, transpose symmetry,
momentum closed form for a constant gradient, RNE bf16 rounding against the
IEEE definition, LPT hand-worked case plus the Graham bound against brute force
optimum, AdamW against torch.optim.AdamW (fp64) and its constant-gradient closed
form.  Every function below is pinned; none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

# Standard Muon quintic coefficients (a, b, c) and normalisation epsilon.
NS_COEFFS: Tuple[float, float, float] = (3.4445, -4.7750, 2.0315)
NS_EPS: float = 1e-7
# Home page, "LLM Pretraining" usage example: learning rate 0.02, 5 Newton-Schulz steps.
DEFAULT_LR: float = 0.02
DEFAULT_NS_STEPS: int = 5
DEFAULT_BETA: float = 0.95

# Packed-segment alignment: 256 bytes (= 128 bf16 elements).  "Z2 vs Z3 Modes",
# "The two packed-buffer lifecycles", only says that they share one contiguous buffer;
# the alignment is this library's reading so that every segment can be read
# with 16-byte vector loads and TMA.
PACK_ALIGN_BYTES: int = 256
PACK_ALIGN_ELEMS: int = PACK_ALIGN_BYTES // 2


# ---------------------------------------------------------------------------
# Momentum (reading: standard Muon Nesterov form)
# ---------------------------------------------------------------------------
def nesterov_momentum(G: np.ndarray, M: np.ndarray, beta: float) -> Tuple[np.ndarray, np.ndarray]:
    """Return (M_new, U): M_new = beta*M + (1-beta)*G, U = (1-beta)*G + beta*M_new.

    Home page "What DMuon Can Do": the owner runs the Muon update for its
    matrices.  The Nesterov form is the standard Muon one (pages silent).
    """
    G = np.asarray(G, dtype=np.float64)
    M = np.asarray(M, dtype=np.float64)
    M_new = beta * M + (1.0 - beta) * G
    U = (1.0 - beta) * G + beta * M_new
    return M_new, U


# ---------------------------------------------------------------------------
# Newton-Schulz
# ---------------------------------------------------------------------------
def ns_working_matrix(U: np.ndarray) -> Tuple[np.ndarray, bool]:
    """X = U^T when rows > cols (so that X is m x n with m <= n), else U."""
    U = np.asarray(U, dtype=np.float64)
    if U.shape[0] > U.shape[1]:
        return U.T, True
    return U, False


def ns_normalise(X: np.ndarray, eps: float = NS_EPS) -> np.ndarray:
    """X0 = X / (||X||_F + eps); eps is added to the norm, not under the root."""
    X = np.asarray(X, dtype=np.float64)
    return X / (math.sqrt(float(np.sum(X * X))) + eps)


def newton_schulz(U: np.ndarray, ns_steps: int = DEFAULT_NS_STEPS,
                  abc: Sequence[float] = NS_COEFFS, eps: float = NS_EPS) -> np.ndarray:
    """Standard quintic Newton-Schulz orthogonalisation of one matrix (fp64).

    Home page, owner section: each matrix is orthogonalised once per step, by
    its owner, with the number of steps as an optimizer argument.  Steps in the iteration's own order:
    transpose-if-tall, normalise, then ``ns_steps`` times A = X X^T,
    B = b A + c A A, X = a X + B X; undo the transpose.
    """
    a, b, c = (float(v) for v in abc)
    X, transposed = ns_working_matrix(U)
    X = ns_normalise(X, eps)
    for _ in range(int(ns_steps)):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T.copy() if transposed else X.copy()


def gram_newton_schulz(U: np.ndarray, ns_steps: int = DEFAULT_NS_STEPS,
                       abc: Sequence[float] = NS_COEFFS, eps: float = NS_EPS) -> np.ndarray:
    """Gram-matrix form of the same iteration (fp64).

    Home page, "VLA and VLM" (Gram Newton-Schulz named for tensor-parallel
    use) -- the pages give no algorithm.  Reading: with A_0 = X0 X0^T,
    P_k = a I + b A_k + c A_k^2, Q_k = P_k Q_{k-1} (Q_0 = P_0),
    A_{k+1} = A_k P_k^2, and the result O = Q_{last} X0.  ns_steps = 0 gives X0.
    """
    a, b, c = (float(v) for v in abc)
    X, transposed = ns_working_matrix(U)
    X0 = ns_normalise(X, eps)
    m = X0.shape[0]
    A = X0 @ X0.T
    Q: Optional[np.ndarray] = None
    eye = np.eye(m)
    for k in range(int(ns_steps)):
        P = a * eye + b * A + c * (A @ A)
        Q = P if Q is None else P @ Q
        if k + 1 < int(ns_steps):
            A = A @ (P @ P)
    O = X0.copy() if Q is None else Q @ X0
    return O.T.copy() if transposed else O


def update_scale(rows: int, cols: int) -> float:
    """sqrt(max(1, rows/cols)) with the parameter's own (rows, cols) = (out, in)."""
    return math.sqrt(max(1.0, rows / cols))


def apply_update(W: np.ndarray, O: np.ndarray, lr: float) -> np.ndarray:
    """W' = W - lr * sqrt(max(1, rows/cols)) * O, in fp64."""
    W = np.asarray(W, dtype=np.float64)
    r, c = W.shape
    return W - lr * update_scale(r, c) * np.asarray(O, dtype=np.float64)


def muon_step(G: np.ndarray, M: np.ndarray, W: np.ndarray, lr: float = DEFAULT_LR,
              beta: float = DEFAULT_BETA, ns_steps: int = DEFAULT_NS_STEPS,
              variant: str = "standard", abc: Sequence[float] = NS_COEFFS,
              eps: float = NS_EPS) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One owner-side Muon step for one matrix: returns (M_new, O, W_new), fp64."""
    M_new, U = nesterov_momentum(G, M, beta)
    if variant == "standard":
        O = newton_schulz(U, ns_steps, abc, eps)
    elif variant == "gram":
        O = gram_newton_schulz(U, ns_steps, abc, eps)
    else:
        raise ValueError(f"unknown Newton-Schulz variant {variant!r}")
    return M_new, O, apply_update(W, O, lr)


# ---------------------------------------------------------------------------
# AdamW for the parameters Muon does not own
# ---------------------------------------------------------------------------
ADAMW_DEFAULT_LR = 1e-3          # home page, "LLM Pretraining": AdamW learning rate in the usage example
ADAMW_DEFAULT_BETAS = (0.9, 0.999)
ADAMW_DEFAULT_EPS = 1e-8
ADAMW_DEFAULT_WD = 0.01


def adamw_step(p: np.ndarray, g: np.ndarray, m: np.ndarray, v: np.ndarray, step: int,
               lr: float = ADAMW_DEFAULT_LR, betas: Tuple[float, float] = ADAMW_DEFAULT_BETAS,
               eps: float = ADAMW_DEFAULT_EPS,
               weight_decay: float = ADAMW_DEFAULT_WD) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One AdamW step (decoupled weight decay), fp64.  Returns (p, m, v).

    Home page, "LLM Pretraining": parameters outside the Muon set (embeddings,
    norms, heads) use AdamW with its own learning rate.  The pages give no other
    hyper-parameter; the reading is the usual AdamW with decay applied to the
    parameter before the moment update:
      p <- p (1 - lr wd)
      m <- b1 m + (1 - b1) g;   v <- b2 v + (1 - b2) g^2
      p <- p - (lr / (1 - b1^t)) m / (sqrt(v) / sqrt(1 - b2^t) + eps)
    """
    if step < 1:
        raise ValueError("step counts from 1")
    b1, b2 = betas
    p = np.asarray(p, np.float64) * (1.0 - lr * weight_decay)
    g = np.asarray(g, np.float64)
    m = b1 * np.asarray(m, np.float64) + (1.0 - b1) * g
    v = b2 * np.asarray(v, np.float64) + (1.0 - b2) * g * g
    bc1 = 1.0 - b1 ** step
    bc2 = 1.0 - b2 ** step
    p = p - (lr / bc1) * m / (np.sqrt(v) / math.sqrt(bc2) + eps)
    return p, m, v


# ---------------------------------------------------------------------------
# bf16 round-to-nearest-even, from the IEEE definition
# ---------------------------------------------------------------------------
_BF16_MANT_BITS = 7          # explicit fraction bits
_BF16_EMIN = -126            # smallest normal exponent (same as fp32)
_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even; result in fp64.

    bf16 = 1 sign, 8 exponent, 7 fraction bits.  For |x| in [2^e, 2^(e+1)) the
    spacing is 2^(e-7); below 2^-126 the spacing is fixed at 2^-133
    (subnormals).  Values whose rounding exceeds the largest finite bf16 become
    +-inf.  NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    ax = np.abs(x[finite])
    e = np.floor(np.log2(ax))
    # log2 can be off by one ulp near powers of two: fix the exponent exactly.
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, _BF16_EMIN)
    spacing_exp = (e - _BF16_MANT_BITS).astype(np.int64)
    q = np.rint(np.ldexp(ax, -spacing_exp))      # exact scaling; rint = ties-to-even
    r = np.ldexp(q, spacing_exp)
    r = np.where(r > _BF16_MAX, np.inf, r)
    out[finite] = np.copysign(r, x[finite])
    return out


# ---------------------------------------------------------------------------
# Owner partition and packing (reading: greedy LPT, 256-byte aligned segments)
# ---------------------------------------------------------------------------
def lpt_assign(sizes: Sequence[int], n_owners: int) -> List[int]:
    """Greedy LPT: visit matrices by descending size (ties: lower index first),
    give each to the currently least-loaded owner (ties: lower owner index)."""
    if n_owners <= 0:
        raise ValueError("n_owners must be positive")
    order = sorted(range(len(sizes)), key=lambda i: (-int(sizes[i]), i))
    load = [0] * n_owners
    owner_of = [0] * len(sizes)
    for i in order:
        best = min(range(n_owners), key=lambda o: (load[o], o))
        owner_of[i] = best
        load[best] += int(sizes[i])
    return owner_of


def _round_up(v: int, a: int) -> int:
    return (v + a - 1) // a * a


def pack_plan(shapes: Sequence[Tuple[int, int]], n_owners: int = 1,
              align_elems: int = PACK_ALIGN_ELEMS) -> Tuple[List[int], List[int], List[int]]:
    """Owner map, element offsets and per-owner buffer sizes for one packed
    allocation holding every owner's buffer back to back.

    "Z2 vs Z3 Modes", "The two packed-buffer lifecycles": matrices that share
    an owner are packed into one contiguous buffer.  Within an owner buffer the
    segments follow parameter order; each segment and each owner buffer starts
    on an ``align_elems`` boundary.  Returns (owner_of, offset, owner_elems).
    """
    sizes = [int(r) * int(c) for r, c in shapes]
    owner_of = lpt_assign(sizes, n_owners) if n_owners > 1 else [0] * len(sizes)
    offset = [0] * len(sizes)
    owner_elems = [0] * n_owners
    base = 0
    for o in range(n_owners):
        cur = 0
        for i in range(len(sizes)):
            if owner_of[i] == o:
                offset[i] = base + cur
                cur = _round_up(cur + sizes[i], align_elems)
        owner_elems[o] = cur
        base += cur
    return owner_of, offset, owner_elems


# ---------------------------------------------------------------------------
# Whole-set helpers used by tests
# ---------------------------------------------------------------------------
def ns_flops_algorithmic(shapes: Iterable[Tuple[int, int]], ns_steps: int) -> float:
    """Algorithmic flops of standard NS: per step 3 m^2 n + m^3 (symmetric
    products X X^T and A A counted as half), m = min(r, c), n = max(r, c)."""
    tot = 0.0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        tot += (3.0 * m * m * n + float(m) ** 3) * ns_steps
    return tot


def gram_ns_flops_algorithmic(shapes: Iterable[Tuple[int, int]], ns_steps: int) -> float:
    """Algorithmic flops of Gram NS: m^2 n (A0, symmetric) + 2 m^2 n (Q X0)
    + per step A^2, P Q, P^2, A P^2 as symmetric m^3 products (4 m^3),
    minus the products the first/last steps skip."""
    tot = 0.0
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        if ns_steps == 0:
            continue
        per = 0.0
        for k in range(ns_steps):
            per += m ** 3                      # A^2
            if k > 0:
                per += m ** 3                  # P Q
            if k + 1 < ns_steps:
                per += 2.0 * m ** 3            # P^2, A P^2
        tot += 3.0 * m * m * n + per
    return tot
