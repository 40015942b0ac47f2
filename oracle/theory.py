"""Oracle of the selection theory: joint distributions over n positions.

TEST INFRASTRUCTURE ONLY (see package header).

Everything here follows section 5 of the zhongzhuzhou.org Fast-dLLM reading
notes ("what the theorem guarantees"):

* eq. 5: q = product of the marginals p_j of a joint p;
* eqs. 6-8 (Theorem 1): if every p_j(x_j*) > 1 - eps and (n+1) eps <= 1 then
  argmax p = argmax q = x*; the union bound p(x*) > 1 - n eps (eq. 6) and
  p(z) < eps for z != x* (eq. 7) are the two steps;
* the tightness family: mass 1/(n+1) - eta on the all-zero string and
  1/(n+1) + eta/n on each single-one string;
* eq. 9: sum_j eps_j + max_j eps_j < 1 is enough for argmax p = x*;
* eq. 10: TV(p, q) < (3n - 1)/2 * eps;
* eqs. 11-12: D_KL(p || q) equals the total correlation
  sum_j H(X_j) - H(X) = sum_{j>=2} I(X_j; X_1..X_{j-1}) and stays below
  (n - 1) [h_b(eps) + eps log(V - 1)] when every marginal is eps-concentrated;
* the two-position example of section 4 (eq. 4).

These are exact finite computations (brute force over all V^n strings).
Pins: tests/golden/worked_example.json (eq. 4 and its printed product and TV),
brute-force checks of the theorem and its tightness family, the chain-rule
identity of eq. 11 checked against an independent conditional-entropy sum.
"""
from __future__ import annotations

import itertools

import numpy as np


def marginals(p: np.ndarray) -> list[np.ndarray]:
    n = p.ndim
    return [p.sum(axis=tuple(a for a in range(n) if a != j)) for j in range(n)]


def product_of_marginals(p: np.ndarray) -> np.ndarray:
    ms = marginals(p)
    q = ms[0]
    for m in ms[1:]:
        q = np.multiply.outer(q, m)
    return q


def argmax_strings(p: np.ndarray, tol: float = 0.0) -> list[tuple]:
    """All strings whose probability is within ``tol`` of the maximum."""
    top = p.max()
    return [tuple(int(i) for i in ix) for ix in zip(*np.nonzero(p >= top - tol))]


def marginal_argmax(p: np.ndarray) -> tuple:
    return tuple(int(np.argmax(m)) for m in marginals(p))


def eps_per_position(p: np.ndarray) -> np.ndarray:
    """eps_j = 1 - max_x p_j(x): the non-top mass of each marginal."""
    return np.array([1.0 - m.max() for m in marginals(p)])


def theorem1_applies(p: np.ndarray) -> bool:
    """True if some eps with p_j(x_j*) > 1 - eps for all j has (n+1) eps <= 1,
    i.e. (n+1) * max_j eps_j < 1."""
    n = p.ndim
    return (n + 1) * eps_per_position(p).max() < 1.0


def eq9_holds(p: np.ndarray) -> bool:
    e = eps_per_position(p)
    return e.sum() + e.max() < 1.0


def tv(p: np.ndarray, q: np.ndarray) -> float:
    return 0.5 * float(np.abs(p - q).sum())


def entropy(p: np.ndarray) -> float:
    x = p[p > 0]
    return float(-(x * np.log(x)).sum())


def kl(p: np.ndarray, q: np.ndarray) -> float:
    """Forward KL D(p || q); infinite when p puts mass where q has none."""
    m = p > 0
    if np.any(q[m] <= 0):
        return float("inf")
    return float((p[m] * np.log(p[m] / q[m])).sum())


def total_correlation(p: np.ndarray) -> float:
    return sum(entropy(m) for m in marginals(p)) - entropy(p)


def chain_mutual_information(p: np.ndarray) -> float:
    """sum_{j>=2} I(X_j ; X_1..X_{j-1}), each term H(X_j) - H(X_j | X_<j)
    computed from conditional distributions string by string."""
    n = p.ndim
    total = 0.0
    for j in range(1, n):
        pj = p.sum(axis=tuple(range(j + 1, n)))          # joint of X_1..X_j
        prefix = pj.sum(axis=j)                           # joint of X_1..X_{j-1}
        h_cond = 0.0
        for ix in itertools.product(*[range(s) for s in prefix.shape]):
            w = prefix[ix]
            if w <= 0:
                continue
            cond = pj[ix] / w
            h_cond += w * entropy(cond)
        total += entropy(pj.sum(axis=tuple(range(j)))) - h_cond
    return total


def binary_entropy(e: float) -> float:
    if e <= 0.0 or e >= 1.0:
        return 0.0
    return float(-e * np.log(e) - (1 - e) * np.log(1 - e))


def tv_bound(n: int, eps: float) -> float:
    return (3 * n - 1) / 2.0 * eps


def kl_bound(n: int, eps: float, V: int) -> float:
    return (n - 1) * (binary_entropy(eps) + eps * np.log(V - 1))


def tightness_family(n: int, eta: float) -> np.ndarray:
    """Joint over {0,1}^n: 1/(n+1) - eta on 0..0, 1/(n+1) + eta/n on each e_j."""
    p = np.zeros((2,) * n)
    p[(0,) * n] = 1.0 / (n + 1) - eta
    for j in range(n):
        ix = [0] * n
        ix[j] = 1
        p[tuple(ix)] = 1.0 / (n + 1) + eta / n
    return p


def worked_example() -> np.ndarray:
    """Section 4, eq. 4: p(0,0)=0.32, p(0,1)=p(1,0)=0.34, p(1,1)=0."""
    return np.array([[0.32, 0.34], [0.34, 0.0]])
