"""Black-box measurement of the output law of a single-row verifier.

The verifier is treated as a function of its uniforms only: for every draft
sequence, the acceptance threshold of each position and the edges of the final
draw's token cells are located by bisection on the uniform that controls them.
The measure of each cell, times the draft probability, gives the exact law of
the emitted token tuple (to ~1e-14), without restating any formula of the method.
"""
from __future__ import annotations

import itertools

import numpy as np

ONE_BELOW = float(np.nextafter(1.0, 0.0))


def _sup_true(f, iters: int = 64) -> float:
    """sup{u in [0,1) : f(u)} for f true on [0, r] and false above; 0 if f(0) is false."""
    if not f(0.0):
        return 0.0
    if f(ONE_BELOW):
        return 1.0
    lo, hi = 0.0, ONE_BELOW
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if mid == lo or mid == hi:
            break
        if f(mid):
            lo = mid
        else:
            hi = mid
    return hi


def _token_cells(token_of) -> dict:
    """Measure of {u : token_of(u) = c} for a non-decreasing step function on [0, 1)."""
    cells: dict = {}
    start = 0.0
    while True:
        c = token_of(start)
        if token_of(ONE_BELOW) == c:
            end = 1.0
        else:
            lo, hi = start, ONE_BELOW  # token_of(lo) == c != token_of(hi)
            while True:
                mid = 0.5 * (lo + hi)
                if mid <= lo or mid >= hi:
                    break
                if token_of(mid) == c:
                    lo = mid
                else:
                    hi = mid
            end = hi
        cells[c] = cells.get(c, 0.0) + (end - start)
        if end >= 1.0:
            return cells
        start = end


def measure_law(run, p: np.ndarray, q: np.ndarray) -> dict:
    """Law of emitted tuples for `run(tl, dl, ids, u)` -> emitted list (or dict with 'emitted').

    p [gamma+1, V] and q [gamma, V] are probability rows; the verifier gets
    logits log p and log q (-inf where 0) and draft ids enumerated over V^gamma
    weighted by prod q_i(x_i).
    """
    gamma, V = q.shape[0], p.shape[1]
    with np.errstate(divide="ignore"):
        tl, dl = np.log(p), np.log(q)

    def call(ids, u):
        out = run(tl, dl, np.asarray(ids, dtype=np.int64), np.asarray(u, dtype=np.float64))
        if isinstance(out, dict):
            out = out["emitted"]
        return tuple(int(t) for t in out if t >= 0)

    law: dict = {}

    def add(key, m):
        if m > 0:
            law[key] = law.get(key, 0.0) + m

    def rec(i, prefix, mass):
        ids = list(prefix) + [0] * (gamma - len(prefix))
        if i == gamma:  # every guess accepted: bonus draw
            u = [0.0] * gamma + [0.0]

            def tok(uf):
                uu = list(u)
                uu[gamma] = uf
                return call(ids, uu)

            for c, m in _token_cells(tok).items():
                add(c, mass * m)
            return
        for x in range(V):
            wx = q[i][x]
            if wx <= 0:
                continue
            ids_x = list(prefix) + [x] + [0] * (gamma - i - 1)

            # accepted at i <=> more than i accepted guesses <=> emitted length > i + 1
            def acc(ui, ids_x=ids_x):
                u = [0.0] * i + [ui] + [0.0] * (gamma - i - 1) + [0.5]
                return len(call(ids_x, u)) >= i + 2

            r = _sup_true(acc)
            if r < 1.0:  # rejection at i, then the residual draw
                ur = 0.5 * (r + 1.0) if r < ONE_BELOW else ONE_BELOW

                def tok(uf, ids_x=ids_x, ur=ur):
                    u = [0.0] * i + [ur] + [0.0] * (gamma - i - 1) + [uf]
                    return call(ids_x, u)

                for c, m in _token_cells(tok).items():
                    add(c, mass * wx * (1.0 - r) * m)
            if r > 0.0:
                rec(i + 1, list(prefix) + [x], mass * wx * r)

    rec(0, [], 1.0)
    return law


def first_token_marginal(law: dict, V: int) -> np.ndarray:
    m = np.zeros(V)
    for k, v in law.items():
        m[k[0]] += v
    return m


def all_small_cases(seed: int = 7):
    """Random (p, q) for every V in 1..4 and gamma in 0..2, with zeros and ties mixed in."""
    rng = np.random.default_rng(seed)
    for V, gamma in itertools.product(range(1, 5), range(0, 3)):
        p = rng.dirichlet(np.ones(V), size=gamma + 1)
        q = rng.dirichlet(np.ones(V), size=max(gamma, 0)).reshape(gamma, V)
        if V >= 3 and gamma >= 1:
            p[0, 0] = 0.0
            p[0] /= p[0].sum()
            q[0, 1] = 0.0
            q[0] /= q[0].sum()
        yield V, gamma, p, q
