"""kda_prefill_chunked_ws: the prefill in a workspace the caller owns (a
torch tensor here).  It must match the pool-backed entry point on the same
inputs, need no clearing between calls (the buffer starts as 0xFF bytes and
is reused), and work for the CUDA-core configurations that need no
workspace at all; the oracle ties the results to the method."""
import pytest

import kda_inputs as ki
import oracle
from kda_testlib import TOL_BF16, TOL_F32, assert_close, dev_tensor, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_linear_attention_gb300 import build
    build.build()
    yield


def _dev(inp):
    d = {n: dev_tensor(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta")}
    return d, dev_tensor(inp.cu_seqlens), (None if inp.S0 is None else dev_tensor(inp.S0))


@pytest.mark.parametrize("lens,H,with_s0", [([4096], 8, False), ([70, 0, 129, 64, 300], 6, True)])
def test_workspace_entry_matches_pool_and_oracle(lens, H, with_s0):
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(61, lens, H=H, dtype="bf16", chunk=64, with_s0=with_s0)
    d, cu, s0 = _dev(inp)
    o_ref, S_ref = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S0=s0)
    o_ref, S_ref = o_ref.cpu().numpy(), S_ref.cpu().numpy()
    N, T = len(lens), sum(lens)
    nbytes = kda.prefill_workspace_bytes(N, T, H)
    assert nbytes > 0
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    for call in range(2):
        o, S = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S0=s0,
                                   workspace=ws)
        torch.cuda.synchronize()
        assert kda.device_error() == 0
        # the same kernels on the same inputs; only a shared-memory sum's order may differ
        assert rel_err(o.cpu().numpy(), o_ref) <= 1e-5, "call %d: o differs" % call
        assert rel_err(S.cpu().numpy(), S_ref) <= 1e-5, "call %d: S differs" % call
    o_or, S_or = oracle.prefill(inp)
    assert_close(o.cpu().numpy(), o_or, TOL_BF16, "o against the oracle")
    assert_close(S.cpu().numpy(), S_or, TOL_BF16, "S_out against the oracle")


def test_workspace_entry_without_a_workspace_on_the_cuda_core_path():
    """fp32 inputs run the CUDA-core kernel, which needs no workspace: the
    size query gives 0 and an empty buffer is accepted."""
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(62, [40, 17], H=3, dtype="f32", chunk=16, with_s0=True)
    d, cu, s0 = _dev(inp)
    assert kda.prefill_workspace_bytes(2, 57, 3, chunk=16, dtype=kda.KDA_F32) == 0
    ws = torch.empty((0,), dtype=torch.uint8, device="cuda")
    o, S = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S0=s0, chunk=16,
                               workspace=ws)
    torch.cuda.synchronize()
    o_or, S_or = oracle.prefill(inp)
    assert_close(o.cpu().numpy(), o_or, TOL_F32, "o against the oracle")
    assert_close(S.cpu().numpy(), S_or, TOL_F32, "S_out against the oracle")


def test_workspace_too_small_is_refused_before_launch():
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(63, [130], H=2, dtype="bf16", chunk=64, with_s0=False)
    d, cu, s0 = _dev(inp)
    nbytes = kda.prefill_workspace_bytes(1, 130, 2)
    ws = torch.zeros((nbytes - 1024,), dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KDAError) as e:
        kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, workspace=ws)
    assert e.value.status == 6


def test_workspace_release_returns_the_pool_memory():
    """kda_workspace_release gives the pool's records back to the driver (the
    device's free memory grows by at least the 4K prefill's workspace), and
    the next prefill grows the pool again and gives the same bits."""
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.workload_prefill("prefill_4k")
    d = {n: dev_tensor(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta")}
    cu = dev_tensor(inp.cu_seqlens)
    o1, S1 = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu)
    torch.cuda.synchronize()
    need = kda.prefill_workspace_bytes(inp.N, inp.T, inp.H)
    free0 = torch.cuda.mem_get_info()[0]
    kda.workspace_release()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 - free0 >= need - (64 << 20), (free0, free1, need)
    o2, S2 = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu)
    torch.cuda.synchronize()
    assert kda.device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
