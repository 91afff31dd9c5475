"""kda_prefill_chunked_noalloc: the prefill with its workspace in the
library's fixed device array.  Two calls in a row must match the pool-backed
entry point and, on their own, the fp64 oracle within the bf16 bar; inputs
that need more scratch than the array holds are rejected before any launch.
(This file is collected last on purpose: it must pass both alone and after
every other test.)"""
import ctypes

import numpy as np
import pytest

import kda_inputs as ki
import oracle

from kda_testlib import TOL_BF16, assert_close, dev_tensor, rel_err

KDA_ERR_WORKSPACE = 6
SCRATCH = 64 << 20
REC = 60416


def _needed(N, T, H):
    chunks = (T + 63) // 64 + N
    return ((4 * (N + 2) + 1023) // 1024) * 1024 + ((8 * chunks + 1023) // 1024) * 1024 + chunks * H * REC


def test_noalloc_rejects_oversize_before_launch():
    """Host-side: an input whose workspace exceeds the array is refused with
    KDA_ERR_WORKSPACE (fake pointers: nothing may be dereferenced)."""
    from kda_linear_attention_gb300 import build
    build.build()
    import kda_linear_attention_gb300 as kda
    L = kda.lib()
    fake = ctypes.c_void_p(1 << 20)
    N, H = 1, 96
    T = 704                                   # (11 + 1) * 96 records > 64 MiB
    assert _needed(N, T, H) > SCRATCH and _needed(N, 640, H) <= SCRATCH
    rc = L.kda_prefill_chunked_noalloc(fake, fake, fake, fake, fake, None, fake, fake, fake,
                                      N, T, H, 128, 128, 64, 0, None)
    assert rc == KDA_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("lens,H,with_s0", [([640], 96, False), ([70, 33, 129, 0, 64], 8, True)])
def test_noalloc_matches_pool_entry_point_twice(lens, H, with_s0):
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(11, lens, H=H, dtype="bf16", chunk=64, with_s0=with_s0)
    assert _needed(len(lens), sum(lens), H) <= SCRATCH
    d = {n: dev_tensor(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta")}
    cu = dev_tensor(inp.cu_seqlens)
    s0 = None if inp.S0 is None else dev_tensor(inp.S0)
    o_ref, S_ref = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S0=s0)
    o_ref, S_ref = o_ref.cpu().numpy(), S_ref.cpu().numpy()
    o_or, S_or = oracle.prefill(inp)
    T, N = sum(lens), len(lens)
    o = torch.empty((T, H, 128), dtype=torch.float32, device="cuda")
    S = torch.empty((N, H, 128, 128), dtype=torch.float32, device="cuda")
    for call in range(2):
        o.fill_(float("nan"))
        S.fill_(float("nan"))
        kda.prefill_chunked_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S0=s0,
                                    o=o, S_out=S)
        torch.cuda.synchronize()
        assert kda.device_error() == 0
        on, Sn = o.cpu().numpy(), S.cpu().numpy()
        assert np.isfinite(on).all() and np.isfinite(Sn).all(), "call %d left outputs unwritten" % call
        # same kernels and inputs; only the order of a shared-memory sum may differ
        assert rel_err(on, o_ref) <= 1e-5, "call %d: o differs from kda_prefill_chunked" % call
        assert rel_err(Sn, S_ref) <= 1e-5, "call %d: S differs from kda_prefill_chunked" % call
        assert_close(on, o_or, TOL_BF16, "call %d: o against the oracle" % call)
        assert_close(Sn, S_or, TOL_BF16, "call %d: S against the oracle" % call)
