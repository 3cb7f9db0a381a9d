"""CPU model of the elimination order the direct-solve kernels use.

Cyclic reduction on the block-Jacobi-scaled chain S_hat = I + Nhat (identity
diagonal blocks, coupling blocks Nhat_j at (j, j-1)): the first level
eliminates the odd knots (identity blocks, products only); at stride s >= 2
the odd multiples of s are factored and the even multiples updated; knot 0
is the last one left; back-substitution runs the levels in reverse.  This
model follows the same index sets and the same update formulas in fp64 and
is checked against a dense solve, for every horizon up to 40 and the powers
of two and their neighbours.  The chronological order (block Cholesky in
knot order) is modelled the same way.
"""
import numpy as np
import pytest


def odd_multiples(N, s):
    return (N - 1 - s) // (2 * s) + 1 if s < N else 0


def even_multiples(N, s):
    return (N - 1) // (2 * s) + 1


def chain(N, n, rng):
    Nh = [None] + [0.2 / np.sqrt(n) * rng.standard_normal((n, n)) for _ in range(N - 1)]
    S = np.eye(N * n)
    for j in range(1, N):
        S[j * n:(j + 1) * n, (j - 1) * n:j * n] = Nh[j]
        S[(j - 1) * n:j * n, j * n:(j + 1) * n] = Nh[j].T
    return Nh, S


def cyclic_reduction(Nh, g, N, n):
    D, E, Y = [None] * N, [None] * N, [None] * N
    seen = set()
    for k in range(even_multiples(N, 1)):
        i = 2 * k
        c = np.eye(n)
        if i >= 1:
            c -= Nh[i] @ Nh[i].T
        if i + 1 < N:
            c -= Nh[i + 1].T @ Nh[i + 1]
        D[i] = c
        if i >= 2:
            E[i] = -Nh[i] @ Nh[i - 1]
    s = 2
    while s < N:
        for k in range(odd_multiples(N, s)):
            j = (2 * k + 1) * s
            assert j < N and j not in seen
            seen.add(j)
            F = np.linalg.inv(np.linalg.cholesky(D[j]))
            D[j], E[j] = F, F @ E[j]
            if j + s < N:
                Y[j] = F @ E[j + s].T
        for k in range(even_multiples(N, s)):
            i = 2 * k * s
            assert i < N
            c = D[i].copy()
            if i >= s:
                c -= Y[i - s].T @ Y[i - s]
            if i + s < N:
                c -= E[i + s].T @ E[i + s]
            D[i] = c
            if i >= 2 * s:
                E[i] = -Y[i - s].T @ E[i - s]
        s *= 2
    D[0] = np.linalg.inv(np.linalg.cholesky(D[0]))
    # every knot but 0 is eliminated exactly once: the odd ones at the first
    # level, the rest at the level of their lowest set bit
    assert seen | set(range(1, N, 2)) | {0} == set(range(N))

    v, G = g.reshape(N, n).copy(), np.zeros((N, n))
    for k in range(even_multiples(N, 1)):
        i = 2 * k
        if i >= 1:
            v[i] -= Nh[i] @ v[i - 1]
        if i + 1 < N:
            v[i] -= Nh[i + 1].T @ v[i + 1]
    smax, s = 1, 2
    while s < N:
        smax = s
        for k in range(odd_multiples(N, s)):
            j = (2 * k + 1) * s
            G[j] = D[j] @ v[j]
        for k in range(even_multiples(N, s)):
            i = 2 * k * s
            if i >= s:
                v[i] -= Y[i - s].T @ G[i - s]
            if i + s < N:
                v[i] -= E[i + s].T @ G[i + s]
        s *= 2
    v[0] = D[0].T @ (D[0] @ v[0])
    s = smax
    while s >= 2:
        for k in range(odd_multiples(N, s)):
            j = (2 * k + 1) * s
            h = G[j] - E[j] @ v[j - s]
            if j + s < N:
                h -= Y[j] @ v[j + s]
            v[j] = D[j].T @ h
        s //= 2
    for k in range(odd_multiples(N, 1)):
        j = 2 * k + 1
        x = v[j] - Nh[j] @ v[j - 1]
        if j + 1 < N:
            x -= Nh[j + 1].T @ v[j + 1]
        v[j] = x
    return v.ravel()


def chronological(Nh, g, N, n):
    F, W = [np.eye(n)], [None]
    for j in range(1, N):
        W.append(Nh[j] @ F[j - 1].T)
        F.append(np.linalg.inv(np.linalg.cholesky(np.eye(n) - W[j] @ W[j].T)))
    gv, y, x = g.reshape(N, n), np.zeros((N, n)), np.zeros((N, n))
    for j in range(N):
        y[j] = F[j] @ (gv[j] - (W[j] @ y[j - 1] if j else 0))
    for j in range(N - 1, -1, -1):
        x[j] = F[j].T @ (y[j] - (W[j + 1].T @ x[j + 1] if j + 1 < N else 0))
    return x.ravel()


HORIZONS = list(range(1, 41)) + [63, 64, 65, 127, 128, 129, 255, 256, 257, 512]


@pytest.mark.parametrize("N", HORIZONS)
def test_elimination_orders_solve_the_chain(N):
    rng = np.random.default_rng(N)
    for n in (1, 3, 6):
        Nh, S = chain(N, n, rng)
        g = rng.standard_normal(N * n)
        ref = np.linalg.solve(S, g)
        for solver in (cyclic_reduction, chronological):
            x = solver(Nh, g, N, n)
            assert np.linalg.norm(x - ref) <= 1e-12 * np.linalg.norm(ref), (solver.__name__, n)


def test_level_counts():
    # ceil(log2 N) levels: the stride-1 level plus one per stride s = 2, 4, ... < N
    for N in range(1, 600):
        levels = 1 + sum(1 for s in (2 ** k for k in range(1, 12)) if s < N)
        assert levels == max(1, int(np.ceil(np.log2(N)))) or N == 1
        assert sum(odd_multiples(N, 2 ** k) for k in range(0, 12)) == N - 1
