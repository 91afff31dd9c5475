"""The KDA layer's prologue and epilogue around the recurrence, numpy fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it.  It shares
no code with the CUDA path.

What the pages fix ("Colibri Kimi K3 Metal backend"):
  - Per KDA layer: q/k/v projections, a depthwise conv1d of width K = 4 on
    each of them ("conv_q / conv_k / conv_v" taps), per-head L2 normalisation,
    the state recurrence, then per-head RMSNorm with a sigmoid full-rank gate
    (section 8 introduction: the order of the per-token loop is conv1d + SiLU,
    per-head L2 norm, per-head state scan, per-head RMSNorm + sigmoid gate).
  - Section 8.3, the conv: every channel keeps a window of its last K raw
    inputs; a token shifts the window left by one, puts the new input in the
    last slot (K - 1), takes the dot product with the channel's K taps and
    applies SiLU(x) = x / (1 + exp(-x)).  Done for q, k and v alike.
  - Section 8.3, the L2 norm: per head, n = 1 / sqrt(sum x^2 + eps) over the
    head's channels with eps = 1e-6; q is multiplied by n * qscale (qscale =
    1 / sqrt(head width)) and k by n.  v is not normalised.
  - Section 8.4: after the token step, per-head RMSNorm of o and a sigmoid of
    the full-rank gate projection give the layer's output.

Readings where the pages leave a step open (the same readings the kernels
take):
  - The window before a sequence's first token holds the previous segment's
    last K - 1 raw inputs (a carried conv state), or zeros.
  - Tap m (0-based) multiplies window slot m, slot K - 1 being the newest
    input: y_t = sum_m w_m x_{t - (K - 1) + m}.
  - RMSNorm: o_j / sqrt(mean_j o_j^2 + eps) * w_j over the head's dv channels,
    with one weight vector of length dv shared by all heads and eps an
    argument (the pages give none; 1e-6 by default, the L2 norm's eps); the
    gate multiplies by sigmoid(gate_j) per channel.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

L2_EPS = 1e-6
NORM_EPS = 1e-6


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x / (1 + exp(-x)) (section 8.3), fp64."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def sigmoid(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def conv_window(x: np.ndarray, w: np.ndarray, win0: Optional[np.ndarray]
                ) -> Tuple[np.ndarray, np.ndarray]:
    """Depthwise causal conv of one sequence, token by token, by the window
    rule of section 8.3 (before the SiLU).

    x    [L, C] fp64: raw inputs of the sequence (C channels)
    w    [C, K] fp64: taps; tap K-1 multiplies the newest input
    win0 [K-1, C]: the K-1 inputs before the sequence, oldest first, or None
    Returns (y [L, C] fp64, window after the last token [K-1, C] fp64).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    L, Cn = x.shape
    K = w.shape[1]
    win = np.zeros((K, Cn), dtype=np.float64)
    if win0 is not None:
        win[1:] = np.asarray(win0, dtype=np.float64)   # slot 0 is shifted out first
    y = np.empty((L, Cn), dtype=np.float64)
    for t in range(L):
        win[:-1] = win[1:].copy()          # shift left by one
        win[K - 1] = x[t]                  # the new input in the last slot
        acc = np.zeros(Cn, dtype=np.float64)
        for m in range(K):
            acc += w[:, m] * win[m]
        y[t] = acc
    return y, win[1:].copy()


def l2_normalise(z: np.ndarray, scale: float = 1.0, eps: float = L2_EPS) -> np.ndarray:
    """z * scale / sqrt(sum z^2 + eps) over the last axis (a head's channels)."""
    z = np.asarray(z, dtype=np.float64)
    n = 1.0 / np.sqrt(np.sum(z * z, axis=-1, keepdims=True) + eps)
    return z * (n * scale)


def prologue(xq, xk, xv, conv_w, conv0, cu_seqlens, q_scale: float,
             eps: float = L2_EPS):
    """conv1d + SiLU on q, k, v, then the per-head L2 norm of q (times
    q_scale) and k, for a packed varlen batch.

    xq, xk, xv [T, H, d]: raw projections (fp32/fp64 values; bf16 bit
               patterns must be converted by the caller)
    conv_w     [3, H, d, K] taps of the q, k, v convs
    conv0      [N, 3, K-1, H, d] windows before each sequence, or None
    Returns (q, k, v [T, H, d] fp64, conv_out [N, 3, K-1, H, d] fp64): the
    windows after each sequence's last token (conv0 itself, or zeros, for an
    empty sequence).
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = cu.size - 1
    T, H, d = np.shape(xq)
    K = conv_w.shape[-1]
    outs = [np.empty((T, H, d), dtype=np.float64) for _ in range(3)]
    conv_out = np.zeros((N, 3, K - 1, H, d), dtype=np.float64)
    for p, x in enumerate((xq, xk, xv)):
        x = np.asarray(x, dtype=np.float64)
        wp = np.asarray(conv_w[p], dtype=np.float64).reshape(H * d, K)
        for n in range(N):
            a, b = int(cu[n]), int(cu[n + 1])
            w0 = None if conv0 is None else np.asarray(conv0[n, p], dtype=np.float64).reshape(K - 1, H * d)
            y, win = conv_window(x[a:b].reshape(b - a, H * d), wp, w0)
            outs[p][a:b] = silu(y).reshape(b - a, H, d)
            conv_out[n, p] = win.reshape(K - 1, H, d)
    q = l2_normalise(outs[0], q_scale, eps)
    k = l2_normalise(outs[1], 1.0, eps)
    return q, k, outs[2], conv_out


def gated_rmsnorm(o, gate, norm_w, eps: float = NORM_EPS) -> np.ndarray:
    """Per-head RMSNorm of o with weight norm_w, times sigmoid(gate)
    (section 8.4).  o, gate [..., dv]; norm_w [dv]."""
    o = np.asarray(o, dtype=np.float64)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return o / np.sqrt(ms + eps) * np.asarray(norm_w, dtype=np.float64) * sigmoid(gate)


# ----------------------------------------------------------- the whole layer
def _f64(a):
    """bf16 bit patterns (uint16) -> exact fp64; float arrays -> fp64."""
    from . import bf16_bits_to_f64
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def prefill_layer(inp, q_scale: float, round_qkv_bf16: bool = True, eps: float = NORM_EPS,
                  l2_eps: float = L2_EPS, threads: Optional[int] = None):
    """Prologue, recurrence and gated-norm epilogue over a packed varlen batch
    (``kda_inputs.LayerInputs``), in the section 8 order.

    With ``round_qkv_bf16`` the prologue's q, k, v are rounded to bf16 before
    the recurrence (``round_bf16``): the form a prefill that stores them in
    bf16 between the two stages computes.  Returns (out [T, H, dv], o
    [T, H, dv], S_out [N, H, dk, dv], conv_out [N, 3, K-1, H, d]), all fp64.
    """
    from . import prefill as rec_prefill, round_bf16
    import kda_inputs as ki
    conv0 = None if inp.conv0 is None else _f64(inp.conv0)
    q, k, v, conv_out = prologue(_f64(inp.xq), _f64(inp.xk), _f64(inp.xv), inp.conv_w, conv0,
                                 inp.cu_seqlens, q_scale, l2_eps)
    if round_qkv_bf16:
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    rec = ki.PrefillInputs(np.ascontiguousarray(q), np.ascontiguousarray(k), np.ascontiguousarray(v),
                           inp.g, inp.beta, inp.S0, inp.cu_seqlens, "f64", 64)
    o, S = rec_prefill(rec, threads=threads)
    out = gated_rmsnorm(o, _f64(inp.gate), inp.norm_w, eps)
    return out, o, S, conv_out


def decode_layer(S_pool, conv_pool, step, conv_w, norm_w, q_scale: float,
                 state_indices=None, state_bf16: bool = False, eps: float = NORM_EPS,
                 l2_eps: float = L2_EPS):
    """One token of the whole layer per sequence on slot-indexed pools.

    S_pool    [P, H, dk, dv] fp32 (or bf16 bits if state_bf16)
    conv_pool [P, 3, K-1, H, d] bf16 bits: each row's window (oldest first)
    step      ``kda_inputs.LayerDecodeStep`` ([B, H, ...])
    Sequence b uses pool row state_indices[b] (identity when None; a
    negative row is padding: out = 0 and no pool row changes).  The
    prologue's q, k, v enter the recurrence unrounded (fp64).  The stored
    state is rounded to bf16 when state_bf16; the new window holds raw bf16
    inputs, so it is exact.
    Returns (out [B, H, dv], S_pool after, conv_pool after), fp64.
    """
    from . import run_unit, round_bf16
    B, H, d = np.shape(step.xq)
    pool = _f64(S_pool)
    conv = _f64(conv_pool)
    P = pool.shape[0]
    K = conv_w.shape[-1]
    idx = np.arange(B) if state_indices is None else np.asarray(state_indices, dtype=np.int64)
    pool_out = pool.copy()
    conv_out = conv.copy()
    out = np.zeros((B, H, d), dtype=np.float64)
    x = [_f64(step.xq), _f64(step.xk), _f64(step.xv)]
    gate = _f64(step.gate)
    for b in range(B):
        r = int(idx[b])
        if not 0 <= r < P:
            continue
        ys = []
        for p in range(3):
            y, win = conv_window(x[p][b].reshape(1, H * d), np.asarray(conv_w[p]).reshape(H * d, K),
                                 conv[r, p].reshape(K - 1, H * d))
            ys.append(silu(y).reshape(1, H, d))
            conv_out[r, p] = win.reshape(K - 1, H, d)
        q = np.ascontiguousarray(l2_normalise(ys[0], q_scale, l2_eps))
        k = np.ascontiguousarray(l2_normalise(ys[1], 1.0, l2_eps))
        v = np.ascontiguousarray(ys[2])
        g = np.ascontiguousarray(step.g[b:b + 1])
        beta = np.ascontiguousarray(step.beta[b:b + 1])
        for h in range(H):
            o, S = run_unit(q, k, v, g, beta, pool[r, h], 0, 1, h)
            pool_out[r, h] = round_bf16(S) if state_bf16 else S
            out[b, h] = gated_rmsnorm(o[0], gate[b, h], norm_w, eps)
    return out, pool_out, conv_out
