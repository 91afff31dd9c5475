"""Shared helpers of the GPU tests: move seeded inputs to the device, call
the library, and measure the parity error the way the acceptance bar states
it: max |x - x_ref| / max |x_ref| over a tensor."""
from __future__ import annotations

import numpy as np

import kda_inputs as ki

TOL_BF16 = 2e-3      # bf16 q/k/v with fp32 state (stated bar)
TOL_F32 = 1e-5       # all-fp32 inputs (stated bar)


def rel_err(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(x).max())
    return float(np.abs(x - ref).max() / den)


def assert_close(x, ref, tol, what):
    e = rel_err(x, ref)
    assert np.isfinite(np.asarray(x, dtype=np.float64)).all(), "%s: non-finite output" % what
    assert e <= tol, "%s: max rel err %.3e > %.1e" % (what, e, tol)
    return e


def dev_tensor(a: np.ndarray, device="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def prefill_on_gpu(inp: ki.PrefillInputs, chunk=None, S0=None, device="cuda"):
    """Run kda_prefill_chunked on the inputs; returns (o, S_out) as numpy."""
    import torch
    import kda_linear_attention_gb300 as kda
    d = {n: dev_tensor(getattr(inp, n), device) for n in ("q", "k", "v", "g", "beta")}
    cu = dev_tensor(inp.cu_seqlens, device)
    s0 = S0 if S0 is not None else (None if inp.S0 is None else dev_tensor(inp.S0, device))
    o, S = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S0=s0,
                               chunk=chunk or inp.chunk)
    torch.cuda.synchronize()
    assert kda.device_error() == 0, "a bounded wait inside the prefill kernel gave up"
    return o.cpu().numpy(), S.cpu().numpy()


def decode_on_gpu(S_dev, step: ki.DecodeStep, device="cuda"):
    import torch
    import kda_linear_attention_gb300 as kda
    d = {n: dev_tensor(getattr(step, n), device) for n in ("q", "k", "v", "g", "beta")}
    o = kda.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], S_dev)
    torch.cuda.synchronize()
    return o.cpu().numpy()
