"""Seeded synthetic inputs for the KDA recurrence.

This module is the one thing the CPU oracle and the CUDA path share: it draws
the random tensors, and holds none of the recurrence's arithmetic.  The value
distributions follow the model the pages describe (96 heads of width 128,
"Kimi K3 -> TPU v7x feasibility", section 2 model table; per-head L2
normalisation of q and k with eps 1e-6, "Colibri Kimi K3 Metal backend",
section 8.3; the decay gate bounded below by -5, the same model table) and the
five workloads of the benchmark:

  q, k  ~ N(0, 1), then x / sqrt(sum x^2 + 1e-6) per token-head (fp32), then
          rounded to bf16 (round to nearest even) unless the workload is fp32
  v     ~ N(0, 1), rounded to bf16 likewise
  g     = -5 * sigmoid(N(0, 1)) per channel, fp32 (log-decay, in (-5, 0))
  beta  = sigmoid(N(0, 1)) per token-head, fp32
  S0    = 0, or N(0, 0.02^2) fp32 per (sequence, head) state

Draw order from one numpy PCG64 generator: q, k, v, g_raw, beta_raw, S0; for
a decode run the state first, then q, k, v, g_raw, beta_raw per step.

bf16 tensors are carried as uint16 bit patterns; ``f32(name)`` gives their
exact values as fp32.  Nothing here needs a GPU.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

DK = 128
DV = 128
L2_EPS = 1e-6
G_LOWER = -5.0


# --------------------------------------------------------------------------
# bf16 <-> fp32 bit conversions (round to nearest even; inputs are finite)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_u.size, step):
        blk = flat_u[s:s + step]
        lsb = (blk >> np.uint32(16)) & np.uint32(1)
        flat_o[s:s + step] = ((blk + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    """x / sqrt(sum(x^2) + eps) over the last axis, in fp32."""
    n = np.sqrt(np.einsum("...d,...d->...", x, x, dtype=np.float32) + np.float32(L2_EPS))
    return (x / n[..., None]).astype(np.float32)


def _normal(rng: np.random.Generator, shape, slab_rows: int = 4096) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    rows = shape[0]
    for s in range(0, rows, slab_rows):
        e = min(rows, s + slab_rows)
        out[s:e] = rng.standard_normal((e - s,) + tuple(shape[1:]), dtype=np.float32)
    return out


def _qk(rng, shape, bf16: bool, slab_rows: int = 2048):
    """Gaussian, L2-normalised per token-head, optionally rounded to bf16."""
    rows = shape[0]
    out = np.empty(shape, dtype=np.uint16 if bf16 else np.float32)
    for s in range(0, rows, slab_rows):
        e = min(rows, s + slab_rows)
        x = _l2_normalise(rng.standard_normal((e - s,) + tuple(shape[1:]), dtype=np.float32))
        out[s:e] = f32_to_bf16_bits(x) if bf16 else x
    return out


def _v(rng, shape, bf16: bool, slab_rows: int = 2048):
    rows = shape[0]
    out = np.empty(shape, dtype=np.uint16 if bf16 else np.float32)
    for s in range(0, rows, slab_rows):
        e = min(rows, s + slab_rows)
        x = rng.standard_normal((e - s,) + tuple(shape[1:]), dtype=np.float32)
        out[s:e] = f32_to_bf16_bits(x) if bf16 else x
    return out


def _g(rng, shape, slab_rows: int = 2048):
    rows = shape[0]
    out = np.empty(shape, dtype=np.float32)
    for s in range(0, rows, slab_rows):
        e = min(rows, s + slab_rows)
        x = rng.standard_normal((e - s,) + tuple(shape[1:]), dtype=np.float32)
        out[s:e] = np.float32(G_LOWER) * _sigmoid(x)
    return out


# --------------------------------------------------------------------------
# containers
# --------------------------------------------------------------------------
@dataclasses.dataclass
class PrefillInputs:
    """Packed varlen prefill inputs, token-major layout [T, H, d]."""
    q: np.ndarray            # [T,H,dk] uint16 (bf16 bits) or float32
    k: np.ndarray            # [T,H,dk]
    v: np.ndarray            # [T,H,dv]
    g: np.ndarray            # [T,H,dk] float32, log-decay
    beta: np.ndarray         # [T,H] float32
    S0: Optional[np.ndarray]  # [N,H,dk,dv] float32 or None (zeros)
    cu_seqlens: np.ndarray   # [N+1] int32
    dtype: str               # "bf16" | "f32"
    chunk: int

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.size - 1)

    @property
    def H(self) -> int:
        return int(self.g.shape[1])

    def f32(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a


@dataclasses.dataclass
class DecodeStep:
    q: np.ndarray     # [B,H,dk]
    k: np.ndarray     # [B,H,dk]
    v: np.ndarray     # [B,H,dv]
    g: np.ndarray     # [B,H,dk] float32
    beta: np.ndarray  # [B,H] float32
    dtype: str

    def f32(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------
def gen_prefill(seed: int, lens: Sequence[int], H: int, dtype: str = "bf16",
                chunk: int = 64, with_s0: bool = False, s0_std: float = 0.02,
                dk: int = DK, dv: int = DV,
                rng: Optional[np.random.Generator] = None) -> PrefillInputs:
    bf16 = dtype == "bf16"
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    lens = [int(x) for x in lens]
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    q = _qk(rng, (T, H, dk), bf16)
    k = _qk(rng, (T, H, dk), bf16)
    v = _v(rng, (T, H, dv), bf16)
    g = _g(rng, (T, H, dk))
    beta = _sigmoid(rng.standard_normal((T, H), dtype=np.float32))
    S0 = None
    if with_s0:
        S0 = (np.float32(s0_std) * _normal(rng, (len(lens), H, dk, dv), slab_rows=1))
    return PrefillInputs(q, k, v, g, beta, S0, cu, dtype, chunk)


def gen_decode_state(rng: np.random.Generator, B: int, H: int, s0_std: float = 0.02,
                     dk: int = DK, dv: int = DV) -> np.ndarray:
    return np.float32(s0_std) * _normal(rng, (B, H, dk, dv), slab_rows=1)


def gen_decode_step(rng: np.random.Generator, B: int, H: int, dtype: str = "bf16",
                    dk: int = DK, dv: int = DV) -> DecodeStep:
    bf16 = dtype == "bf16"
    q = _qk(rng, (B, H, dk), bf16)
    k = _qk(rng, (B, H, dk), bf16)
    v = _v(rng, (B, H, dv), bf16)
    g = _g(rng, (B, H, dk))
    beta = _sigmoid(rng.standard_normal((B, H), dtype=np.float32))
    return DecodeStep(q, k, v, g, beta, dtype)


# --------------------------------------------------------------------------
# the five benchmark workloads (names describe what they are)
# --------------------------------------------------------------------------
VARLEN_64K_LENS = [512, 1024, 2048, 4096, 8192, 16384, 16384, 17408]

WORKLOADS: Dict[str, dict] = {
    # all-fp32 prefill, B=1, H=2, T=64, chunk 16, S0 = 0, seed 0
    "tiny_fp32": dict(kind="prefill", seed=0, lens=[64], H=2, dtype="f32", chunk=16,
                      with_s0=False, tol=1e-5),
    # bf16 prefill, B=1, H=96, T=4096, chunk 64, S0 = 0
    "prefill_4k": dict(kind="prefill", seed=2, lens=[4096], H=96, dtype="bf16", chunk=64,
                       with_s0=False, tol=2e-3),
    # batched decode, B=64, H=96, state ~N(0,0.02^2), 100 consecutive steps
    "decode_b64": dict(kind="decode", seed=3, B=64, H=96, dtype="bf16", steps=100,
                       tol=2e-3),
    # long bf16 prefill with carry-in state, T=32768, H=96, chunk 64
    "prefill_32k_carry": dict(kind="prefill", seed=4, lens=[32768], H=96, dtype="bf16",
                              chunk=64, with_s0=True, tol=2e-3),
    # varlen packed prefill of 8 sequences (65536 tokens) + one decode step for all 8
    "varlen_64k": dict(kind="varlen+decode", seed=5, lens=VARLEN_64K_LENS, H=96,
                       dtype="bf16", chunk=64, with_s0=True, tol=2e-3),
}


def workload_prefill(name: str) -> PrefillInputs:
    w = WORKLOADS[name]
    assert w["kind"] in ("prefill", "varlen+decode")
    return gen_prefill(w["seed"], w["lens"], w["H"], w["dtype"], w["chunk"], w["with_s0"])


def workload_varlen_with_decode(name: str = "varlen_64k"):
    """Prefill inputs, then one decode step for every sequence, same stream."""
    w = WORKLOADS[name]
    rng = np.random.Generator(np.random.PCG64(w["seed"]))
    pre = gen_prefill(w["seed"], w["lens"], w["H"], w["dtype"], w["chunk"], w["with_s0"],
                      rng=rng)
    step = gen_decode_step(rng, len(w["lens"]), w["H"], w["dtype"])
    return pre, step


def workload_decode(name: str = "decode_b64", steps: Optional[int] = None):
    """(state [B,H,dk,dv] fp32, generator of DecodeStep) for a decode run."""
    w = WORKLOADS[name]
    rng = np.random.Generator(np.random.PCG64(w["seed"]))
    S = gen_decode_state(rng, w["B"], w["H"])
    n = w["steps"] if steps is None else steps

    def _steps():
        for _ in range(n):
            yield gen_decode_step(rng, w["B"], w["H"], w["dtype"])

    return S, _steps()


def ragged_lens(seed: int, n: int, lo: int, hi: int) -> List[int]:
    """Sequence lengths for ragged parity cases (uniform in [lo, hi])."""
    r = np.random.Generator(np.random.PCG64(seed + 7919))
    return [int(x) for x in r.integers(lo, hi + 1, size=n)]


# --------------------------------------------------------------------------
# the layer around the recurrence: raw projections, conv taps and windows,
# output gate and norm weight
# --------------------------------------------------------------------------
CONV_K = 4          # depthwise causal conv width of the model's KDA layer


@dataclasses.dataclass
class LayerInputs:
    """Inputs of the KDA layer's prologue and epilogue around the recurrence.

    xq, xk, xv  [T, H, d] bf16 bits: the q/k/v projections before the conv
    conv_w      [3, H, d, K] float32: depthwise taps of the q, k, v convs;
                tap m multiplies the input m positions before the newest
                one counted from the oldest (tap K-1 = the newest input)
    conv0       [N, 3, K-1, H, d] bf16 bits (oldest first) or None (zeros):
                the last K-1 raw inputs before each sequence
    gate        [T, H, dv] bf16 bits: the output gate's projection (before
                its sigmoid)
    norm_w      [dv] float32: the output RMSNorm weight
    g, beta     as for the recurrence
    """
    xq: np.ndarray
    xk: np.ndarray
    xv: np.ndarray
    conv_w: np.ndarray
    conv0: Optional[np.ndarray]
    gate: np.ndarray
    norm_w: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    cu_seqlens: np.ndarray
    S0: Optional[np.ndarray]

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.size - 1)

    @property
    def H(self) -> int:
        return int(self.g.shape[1])


def gen_layer(seed: int, lens: Sequence[int], H: int, with_conv0: bool = True,
              with_s0: bool = False, s0_std: float = 0.02, conv_std: float = 0.5,
              dk: int = DK, dv: int = DV,
              rng: Optional[np.random.Generator] = None) -> LayerInputs:
    """Draw order: xq, xk, xv ~ N(0,1) bf16; conv taps ~ N(0, conv_std^2)
    fp32; conv windows ~ N(0,1) bf16; gate ~ N(0,1) bf16; norm weight
    1 + 0.1 N(0,1) fp32; g, beta as for the recurrence; S0."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    lens = [int(x) for x in lens]
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T, N = int(cu[-1]), len(lens)
    xq = _v(rng, (T, H, dk), True)
    xk = _v(rng, (T, H, dk), True)
    xv = _v(rng, (T, H, dv), True)
    conv_w = (np.float32(conv_std) * _normal(rng, (3, H, dk, CONV_K), slab_rows=1)).astype(np.float32)
    conv0 = _v(rng, (N, 3, CONV_K - 1, H, dk), True) if with_conv0 else None
    gate = _v(rng, (T, H, dv), True)
    norm_w = (np.float32(1.0) + np.float32(0.1) * rng.standard_normal(dv, dtype=np.float32)).astype(np.float32)
    g = _g(rng, (T, H, dk))
    beta = _sigmoid(rng.standard_normal((T, H), dtype=np.float32))
    S0 = None
    if with_s0:
        S0 = np.float32(s0_std) * _normal(rng, (N, H, dk, dv), slab_rows=1)
    return LayerInputs(xq, xk, xv, conv_w, conv0, gate, norm_w, g, beta, cu, S0)


@dataclasses.dataclass
class LayerDecodeStep:
    """One token per sequence of the whole layer step: raw projections
    [B, H, d] bf16, gate [B, H, dv] bf16, g [B, H, dk] fp32, beta [B, H]."""
    xq: np.ndarray
    xk: np.ndarray
    xv: np.ndarray
    gate: np.ndarray
    g: np.ndarray
    beta: np.ndarray


def gen_layer_decode_step(rng: np.random.Generator, B: int, H: int,
                          dk: int = DK, dv: int = DV) -> LayerDecodeStep:
    xq = _v(rng, (B, H, dk), True)
    xk = _v(rng, (B, H, dk), True)
    xv = _v(rng, (B, H, dv), True)
    gate = _v(rng, (B, H, dv), True)
    g = _g(rng, (B, H, dk))
    beta = _sigmoid(rng.standard_normal((B, H), dtype=np.float32))
    return LayerDecodeStep(xq, xk, xv, gate, g, beta)
