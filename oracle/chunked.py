"""Chunked (UT-transform) restatement of the KDA recurrence, numpy fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  This is an
independent second statement of the same map, used to pin the sequential
oracle: on tiny inputs the two must agree to rounding.  The pages state only
the token recurrence ("Colibri Kimi K3 Metal backend", architecture section);
the chunked form below is derived from it by unrolling the recurrence inside
a chunk of C tokens (b_r = sum_{t<=r} g_t, cumulative log-decay per channel):

  S_r = Diag(e^{b_r}) S_0 + sum_{s<=r} Diag(e^{b_r - b_s}) k_s u_s^T
  u_r = beta_r (v_r - (Diag(e^{g_r}) S_{r-1})^T k_r)

which, with G^kk_rs = sum_c k_rc k_sc e^{b_rc - b_sc} (s < r) and
G^qk_rs = sum_c q_rc k_sc e^{b_rc - b_sc} (s <= r), gives

  (I + Diag(beta) G^kk) U = Diag(beta) (V - K0 S_0),   K0_r = e^{b_r} * k_r
  U  = T Diag(beta) V - T Diag(beta) K0 S_0,           T = (I + Diag(beta) G^kk)^-1
  O  = Q0 S_0 + G^qk U,                                Q0_r = e^{b_r} * q_r
  S_C = Diag(e^{b_C}) S_0 + Kbar^T U,                  Kbar_s = e^{b_C - b_s} * k_s

The pairwise factor e^{b_r - b_s} (s <= r) is at most 1.  The ``subblock``
folding splits it as e^{b_r - rho_p} * e^{rho_p - b_s}, with rho_p the
cumulative decay just before the 16-row sub-block p that holds row r; each
factor then stays within [e^-80, e^80] on the diagonal block when g >= -5
(the model's gate lower bound, "Kimi K3 -> TPU v7x feasibility", section 2),
which is the folding a fixed-width float kernel needs.  ``direct`` evaluates
e^{b_r - b_s} elementwise.  Both are checked against the sequential oracle.
"""
from __future__ import annotations

import numpy as np

SUB = 16


def gated_gram(x: np.ndarray, k: np.ndarray, b: np.ndarray, inclusive: bool,
               fold: str = "subblock") -> np.ndarray:
    """G_rs = sum_c x_rc k_sc exp(b_rc - b_sc) for s < r (or s <= r), else 0."""
    L = x.shape[0]
    G = np.zeros((L, L), dtype=np.float64)
    if fold == "direct":
        for r in range(L):
            for s in range(r + 1 if inclusive else r):
                G[r, s] = np.sum(x[r] * k[s] * np.exp(b[r] - b[s]))
    else:
        for p0 in range(0, L, SUB):
            p1 = min(L, p0 + SUB)
            rho = b[p0 - 1] if p0 > 0 else np.zeros_like(b[0])
            xr = x[p0:p1] * np.exp(b[p0:p1] - rho)          # rows of sub-block p
            ks = k[:p1] * np.exp(rho - b[:p1])               # keys up to the sub-block end
            blk = xr @ ks.T                                   # [p1-p0, p1]
            for r in range(p0, p1):
                lim = r + 1 if inclusive else r
                G[r, :lim] = blk[r - p0, :lim]
    return G


def chunk_step(S0, q, k, v, g, beta, fold: str = "subblock"):
    """One chunk of L <= C tokens from state S0 [dk, dv]: returns (O [L, dv], S_C)."""
    L = q.shape[0]
    b = np.cumsum(g, axis=0)                                  # b_r, r = 1..L
    Gkk = gated_gram(k, k, b, inclusive=False, fold=fold)
    Gqk = gated_gram(q, k, b, inclusive=True, fold=fold)
    M = beta[:, None] * Gkk
    T = np.linalg.inv(np.eye(L) + M)                          # unit lower triangular
    K0 = np.exp(b) * k
    Q0 = np.exp(b) * q
    W = T @ (beta[:, None] * K0)
    Ut = T @ (beta[:, None] * v)
    U = Ut - W @ S0
    O = Q0 @ S0 + Gqk @ U
    bC = b[L - 1]
    Kbar = np.exp(bC[None, :] - b) * k
    S = np.exp(bC)[:, None] * S0 + Kbar.T @ U
    return O, S


def run_unit(q, k, v, g, beta, S0, chunk: int, fold: str = "subblock"):
    """Chunked recurrence of one (sequence, head) unit, fp64 arrays:
    q, k, g [L, dk]; v [L, dv]; beta [L]; S0 [dk, dv] or None."""
    L, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    O = np.zeros((L, dv))
    for c0 in range(0, L, chunk):
        c1 = min(L, c0 + chunk)
        O[c0:c1], S = chunk_step(S, q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1],
                                 fold=fold)
    return O, S
