"""CPU oracle for the KDA recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``kda_linear_attention_gb300``) never imports, links or runs
it, and the two share no code: the oracle is a plain fp64 statement of the
method that the CUDA kernels are checked against.

Contents
  kda_oracle.c  sequential token-by-token fp64 recurrence, one (sequence, head)
                unit per call ("Colibri Kimi K3 Metal backend", architecture
                section and section 8.2).  Compiled with gcc into
                ``oracle/_build/libkda_oracle.so`` on first use (or by
                ``__graft_entry__.build()``).
  chunked.py    an independent fp64 restatement in chunked (UT-transform)
                form, used to pin the sequential oracle (they must agree to
                rounding on tiny inputs).
  decode_pool   the decode step on a state pool addressed by slot indices,
                with an fp32 or a bf16-stored state (this file).
  layer.py      the layer around the recurrence: conv1d + SiLU + per-head L2
                norm before it, per-head RMSNorm + sigmoid gate after it
                ("Colibri Kimi K3 Metal backend", sections 8.3 and 8.4), and
                the whole-layer prefill and decode compositions.

Parity pins: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` and ``tests/test_oracle_layer_pins.py``
(closed forms, exact retrieval, brute force, hand-worked examples, numpy's
convolution, the chunked restatement, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Iterable, List, Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, i32, i64, dp, fp = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_void_p)
            lib.oracle_kda_unit.argtypes = [vp, vp, vp, i32, fp, fp, fp, i64, i64, i32, i32,
                                            i32, i32, dp, dp]
            lib.oracle_kda_unit.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def run_unit(q, k, v, g, beta, S0_unit, t0: int, t1: int, h: int,
             out_o: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Sequential recurrence for head ``h`` over tokens [t0, t1).

    q, k, v: [T, H, d] arrays, uint16 (bf16 bits), float32 or float64, C-contiguous.
    g: [T, H, dk] float32; beta: [T, H] float32; S0_unit: [dk, dv] float32 or
    float64 (upcast exactly), or None.  Returns (o [t1-t0, dv] float64, S_final [dk, dv] float64).
    """
    lib = _load()
    kind = {np.dtype(np.float32): 0, np.dtype(np.uint16): 1, np.dtype(np.float64): 2}[q.dtype]
    assert k.dtype == q.dtype and v.dtype == q.dtype
    for a in (q, k, v, g, beta):
        assert a.flags["C_CONTIGUOUS"]
    H, dk = q.shape[1], q.shape[2]
    dv = v.shape[2]
    L = t1 - t0
    o = out_o if out_o is not None else np.empty((L, dv), dtype=np.float64)
    S = np.empty((dk, dv), dtype=np.float64)
    if S0_unit is not None:
        S0_unit = np.ascontiguousarray(S0_unit, dtype=np.float64)   # exact upcast
    rc = lib.oracle_kda_unit(_ptr(q), _ptr(k), _ptr(v), kind, _ptr(g), _ptr(beta),
                             _ptr(S0_unit), int(t0), int(t1), int(H), int(h), int(dk), int(dv),
                             _ptr(o), _ptr(S))
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return o, S


def prefill(inp, units: Optional[Iterable[Tuple[int, int]]] = None,
            threads: Optional[int] = None):
    """Oracle for a packed varlen prefill (``kda_inputs.PrefillInputs``).

    With ``units=None`` every (sequence, head) pair is computed and the result
    is (o [T,H,dv] float64, S_out [N,H,dk,dv] float64).  With a list of
    (n, h) pairs only those are computed and the result is a dict
    {(n, h): (o [len_n, dv], S [dk, dv])}.
    """
    cu = inp.cu_seqlens
    H = inp.H
    threads = threads or default_threads()
    full = units is None
    todo: List[Tuple[int, int]] = ([(n, h) for n in range(inp.N) for h in range(H)]
                                   if full else [tuple(u) for u in units])
    # biggest first so the pool ends together
    todo.sort(key=lambda nh: -(int(cu[nh[0] + 1]) - int(cu[nh[0]])))

    def one(nh):
        n, h = nh
        s0 = None if inp.S0 is None else inp.S0[n, h]
        return nh, run_unit(inp.q, inp.k, inp.v, inp.g, inp.beta, s0,
                            int(cu[n]), int(cu[n + 1]), h)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = dict(ex.map(one, todo))
    if not full:
        return res
    dk, dv = inp.q.shape[2], inp.v.shape[2]
    o = np.zeros((inp.T, H, dv), dtype=np.float64)
    S = np.zeros((inp.N, H, dk, dv), dtype=np.float64)
    for (n, h), (on, Sn) in res.items():
        o[int(cu[n]):int(cu[n + 1]), h, :] = on
        S[n, h] = Sn
    return o, S


def decode(S_in: np.ndarray, step, units: Optional[Iterable[Tuple[int, int]]] = None,
           threads: Optional[int] = None):
    """Oracle for one decode token per sequence.

    S_in: [B,H,dk,dv] float32; step: ``kda_inputs.DecodeStep``.  Returns
    (o [B,H,dv] float64, S_out [B,H,dk,dv] float64), or a dict over the given
    (b, h) units.
    """
    B, H = step.q.shape[0], step.q.shape[1]
    threads = threads or default_threads()
    full = units is None
    todo = [(b, h) for b in range(B) for h in range(H)] if full else [tuple(u) for u in units]

    def one(bh):
        b, h = bh
        return bh, run_unit(step.q, step.k, step.v, step.g, step.beta, S_in[b, h], b, b + 1, h)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = dict(ex.map(one, todo))
    if not full:
        return {bh: (o[0], S) for bh, (o, S) in res.items()}
    dk, dv = step.q.shape[2], step.v.shape[2]
    o = np.zeros((B, H, dv), dtype=np.float64)
    S = np.zeros((B, H, dk, dv), dtype=np.float64)
    for (b, h), (ob, Sb) in res.items():
        o[b, h] = ob[0]
        S[b, h] = Sb
    return o, S


# ---------------------------------------------------------------- state pools
def round_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 value (8 significant bits, ties to even) of each fp64
    element, returned as fp64.  Written from the format's definition: with
    x = m * 2^e, 0.5 <= |m| < 1, the bf16 value is rint(m * 2^8) * 2^(e-8),
    rint rounding half to even.  Normal range only (|x| >= 2^-126), which
    covers every state this package stores."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact fp64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def decode_pool(S_pool: np.ndarray, step, state_indices: Optional[np.ndarray] = None,
                state_bf16: bool = False, threads: Optional[int] = None):
    """One decode token per sequence on a state pool.

    Sequence b updates pool row ``state_indices[b]`` (the identity when None;
    a negative entry is a padding row: o = 0 and no state changes), as the TPU
    KDA decode kernel indexes its states ("Kimi K3 -> TPU v7x feasibility",
    section 4.2).  ``S_pool`` is [P, H, dk, dv] float32, or uint16 bf16 bit
    patterns when ``state_bf16`` (the bf16-stored state of the same review,
    section 6): the state is read exactly, the token step runs in fp64 (the
    sequential oracle), o comes from the updated fp64 state, and the stored
    state is that state rounded to bf16 (``round_bf16``).

    Returns (o [B, H, dv] fp64, pool after the step [P, H, dk, dv] fp64).
    """
    B, H = step.q.shape[0], step.q.shape[1]
    dv = step.v.shape[2]
    pool = bf16_bits_to_f64(S_pool) if state_bf16 else np.asarray(S_pool, dtype=np.float64)
    P = pool.shape[0]
    idx = np.arange(B) if state_indices is None else np.asarray(state_indices, dtype=np.int64)
    out = pool.copy()
    o = np.zeros((B, H, dv), dtype=np.float64)
    todo = [(b, h) for b in range(B) for h in range(H) if 0 <= idx[b] < P]

    def one(bh):
        b, h = bh
        return bh, run_unit(step.q, step.k, step.v, step.g, step.beta, pool[idx[b], h], b, b + 1, h)

    with ThreadPoolExecutor(max_workers=threads or default_threads()) as ex:
        for (b, h), (ob, Sb) in ex.map(one, todo):
            o[b, h] = ob[0]
            out[idx[b], h] = round_bf16(Sb) if state_bf16 else Sb
    return o, out
