"""GPU edge cases of the recurrence through the C ABI: batches of more than
1024 sequences (the chunk plan's multi-pass scan, the state pass's identity
order past its longest-first limit), the extreme gates g = -5 everywhere
(largest decay-folding factors) and g = 0, and the method's degenerate
cases: beta = 0 with g = 0 leaves the state unchanged bit for bit, and with
beta = 1 and exactly unit-norm keys the delta rule retrieves v exactly
(o_t = v_t when q = k), a property that needs no oracle."""
import numpy as np
import pytest

import kda_inputs as ki
import oracle
from kda_testlib import TOL_BF16, TOL_F32, assert_close, dev_tensor, prefill_on_gpu

pytestmark = pytest.mark.gpu

PATHS = [("bf16", 64), ("bf16", 32), ("f32", 16)]   # tensor-core path, CUDA-core paths


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_linear_attention_gb300 import build
    build.build()
    yield


def _tol(dtype):
    return TOL_F32 if dtype == "f32" else TOL_BF16


def _compare(inp, o, S, tol, what):
    """Per sequence: o and S_out each within tol of the oracle."""
    o_ref, S_ref = oracle.prefill(inp)
    cu = inp.cu_seqlens
    for n in range(inp.N):
        a, b = int(cu[n]), int(cu[n + 1])
        if b > a:
            assert_close(o[a:b], o_ref[a:b], tol, "%s: o of sequence %d" % (what, n))
        assert_close(S[n], S_ref[n], tol, "%s: S_out of sequence %d" % (what, n))


@pytest.mark.parametrize("dtype,chunk", [("bf16", 64), ("f32", 16)])
def test_prefill_more_than_1024_sequences(dtype, chunk):
    """The scheduling machinery past its limits: the chunk plan's scan in
    several 1024-sequence passes, the state pass's identity order beyond 256
    sequences, empty sequences among them, each sequence 0 to 40 tokens with
    a carried state.  o and the final state are held to the bar per
    sequence."""
    lens = ki.ragged_lens(400 + chunk, 1300, 0, 40)
    assert 0 in lens and len(lens) > 1024
    inp = ki.gen_prefill(401, lens, H=2, dtype=dtype, chunk=chunk, with_s0=True)
    o, S = prefill_on_gpu(inp)
    o_ref, S_ref = oracle.prefill(inp)
    tol = _tol(dtype)
    cu = inp.cu_seqlens
    worst = 0.0
    for n in range(inp.N):
        a, b = int(cu[n]), int(cu[n + 1])
        if b > a:
            worst = max(worst, assert_close(o[a:b], o_ref[a:b], tol, "1300 sequences: o of sequence %d" % n))
        assert_close(S[n], S_ref[n], tol, "1300 sequences: S_out of sequence %d" % n)
    print("worst per-sequence o error over 1300 sequences: %.2e" % worst)


@pytest.mark.parametrize("dtype,chunk", PATHS)
@pytest.mark.parametrize("gate", [-5.0, 0.0])
def test_prefill_constant_gate_extremes(dtype, chunk, gate):
    inp = ki.gen_prefill(410, [64, 130, 17, 1], H=3, dtype=dtype, chunk=chunk, with_s0=True)
    inp.g[...] = np.float32(gate)
    o, S = prefill_on_gpu(inp)
    _compare(inp, o, S, _tol(dtype), "g = %g" % gate)


@pytest.mark.parametrize("dtype,chunk", PATHS)
def test_prefill_beta_zero_decays_only(dtype, chunk):
    """beta = 0: S_T = Diag(exp(sum g)) S0.  The sequences are short enough
    that exp(sum g) stays in fp32's normal range (sum g >= -5 T)."""
    inp = ki.gen_prefill(420, [9, 17, 1], H=2, dtype=dtype, chunk=chunk, with_s0=True)
    inp.beta[...] = np.float32(0.0)
    o, S = prefill_on_gpu(inp)
    _compare(inp, o, S, _tol(dtype), "beta = 0")


@pytest.mark.parametrize("dtype,chunk", PATHS)
def test_prefill_no_decay_no_update_keeps_state_exactly(dtype, chunk):
    """g = 0, beta = 0: every update is zero and every decay factor is 1, so
    S_out equals S0 bit for bit on every path."""
    inp = ki.gen_prefill(430, [150, 3, 64], H=2, dtype=dtype, chunk=chunk, with_s0=True)
    inp.g[...] = np.float32(0.0)
    inp.beta[...] = np.float32(0.0)
    o, S = prefill_on_gpu(inp)
    np.testing.assert_array_equal(S, inp.S0)
    _compare(inp, o, S, _tol(dtype), "g = 0, beta = 0")


def _unit_keys(rng, T, H, dk):
    """Keys with four entries of +-0.5 at distinct random channels: exactly
    unit norm in bf16 and fp32."""
    k = np.zeros((T, H, dk), dtype=np.float32)
    for t in range(T):
        for h in range(H):
            idx = rng.choice(dk, 4, replace=False)
            k[t, h, idx] = rng.choice([-0.5, 0.5], 4)
    return k


@pytest.mark.parametrize("dtype,chunk", PATHS)
def test_prefill_exact_retrieval_with_unit_keys(dtype, chunk):
    """beta = 1 and ||k_t|| = 1: S_t^T k_t = v_t after every token, so with
    q = k the output is o_t = v_t (no oracle involved)."""
    rng = np.random.Generator(np.random.PCG64(440))
    lens = [130, 64, 9]
    inp = ki.gen_prefill(441, lens, H=2, dtype=dtype, chunk=chunk, with_s0=True)
    k = _unit_keys(rng, inp.T, inp.H, 128)
    kk = ki.f32_to_bf16_bits(k) if dtype == "bf16" else k
    inp.k[...] = kk
    inp.q[...] = kk
    inp.beta[...] = np.float32(1.0)
    o, S = prefill_on_gpu(inp)
    v = inp.f32("v")
    assert_close(o, v, _tol(dtype), "o = v")
    # and the final states retrieve the last token's v
    cu = inp.cu_seqlens
    for n in range(inp.N):
        last = int(cu[n + 1]) - 1
        got = np.einsum("hij,hi->hj", S[n].astype(np.float64), k[last].astype(np.float64))
        assert_close(got, v[last], _tol(dtype), "S^T k = v, sequence %d" % n)


def test_decode_no_decay_no_update_keeps_state_exactly():
    import torch
    import kda_linear_attention_gb300 as kda
    rng = np.random.Generator(np.random.PCG64(450))
    B, H = 5, 4
    S0 = ki.gen_decode_state(rng, B, H)
    step = ki.gen_decode_step(rng, B, H, "bf16")
    step.g[...] = np.float32(0.0)
    step.beta[...] = np.float32(0.0)
    S = dev_tensor(S0)
    d = {n: dev_tensor(getattr(step, n)) for n in ("q", "k", "v", "g", "beta")}
    o = kda.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], S)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(S.cpu().numpy(), S0)
    o_ref, _ = oracle.decode(S0, step)
    assert_close(o.cpu().numpy(), o_ref, TOL_BF16, "o = S^T q")


def test_decode_exact_retrieval_with_unit_keys():
    import torch
    import kda_linear_attention_gb300 as kda
    rng = np.random.Generator(np.random.PCG64(460))
    B, H = 6, 3
    S0 = ki.gen_decode_state(rng, B, H)
    step = ki.gen_decode_step(rng, B, H, "bf16")
    k = _unit_keys(rng, B, H, 128)
    step.k[...] = ki.f32_to_bf16_bits(k)
    step.q[...] = step.k
    step.beta[...] = np.float32(1.0)
    S = dev_tensor(S0)
    d = {n: dev_tensor(getattr(step, n)) for n in ("q", "k", "v", "g", "beta")}
    o = kda.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], S)
    torch.cuda.synchronize()
    # fp32 arithmetic throughout: o = v to fp32 rounding
    assert_close(o.cpu().numpy(), step.f32("v"), 1e-5, "o = v")


@pytest.mark.parametrize("dtype,chunk", [("bf16", 64), ("f32", 16)])
def test_cu_seqlens_past_T_is_contained(dtype, chunk):
    """cu_seqlens ending past T breaks the call's precondition (the host
    cannot read the device array to check it).  The tensor-core path empties
    its chunk plan and raises the device error flag; the CUDA-core path
    clamps the tokens to [0, T) and raises the same flag.  Neither reads or
    writes past the buffers, and the next valid call is unaffected."""
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(470, [60, 40], H=2, dtype=dtype, chunk=chunk, with_s0=True)   # T = 100
    d = {n: dev_tensor(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta")}
    s0 = dev_tensor(inp.S0)
    bad_cu = dev_tensor(np.array([0, 60, 130], dtype=np.int32))
    kda.device_error(reset=True)
    kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], bad_cu, S0=s0, chunk=chunk)
    torch.cuda.synchronize()
    err = kda.device_error(reset=True)
    assert err & 1, "the inconsistent cu_seqlens was not flagged"
    o, S = prefill_on_gpu(inp)                  # a valid call afterwards
    o_ref, S_ref = oracle.prefill(inp)
    assert_close(o, o_ref, _tol(dtype), "o after the flagged call")
    assert_close(S, S_ref, _tol(dtype), "S_out after the flagged call")


@pytest.mark.parametrize("g_bad", [-8.0, 0.5, float("nan")])
def test_prefill_gate_outside_bound_is_flagged(g_bad):
    """The tensor-core prefill folds the decay into per-row and per-column
    factors sized for gates in [-5, 0] (the model's gate lower bound); one
    gate outside that range (or NaN) raises bit 2 of the device error word,
    and a valid call afterwards leaves the word clear."""
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(480, [100, 70], H=3, dtype="bf16", chunk=64, with_s0=True)
    bad = ki.PrefillInputs(inp.q, inp.k, inp.v, inp.g.copy(), inp.beta, inp.S0, inp.cu_seqlens,
                           "bf16", 64)
    bad.g[120, 1, 77] = np.float32(g_bad)
    d = {n: dev_tensor(getattr(bad, n)) for n in ("q", "k", "v", "g", "beta")}
    kda.device_error(reset=True)
    kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], dev_tensor(bad.cu_seqlens),
                        S0=dev_tensor(bad.S0), chunk=64)
    torch.cuda.synchronize()
    assert kda.device_error(reset=True) & 4, "gate %r was not flagged" % g_bad
    o, S = prefill_on_gpu(inp)               # asserts a clear error word
    _compare(inp, o, S, TOL_BF16, "valid call after a flagged gate")


@pytest.mark.parametrize("dtype,chunk", PATHS)
def test_prefill_is_deterministic(dtype, chunk):
    """Every reduction in the prefill kernels runs in a fixed order (no
    atomics), so the same call on the same inputs gives the same bits: three
    calls on a ragged batch with a carried state, o and S_out compared bit
    for bit."""
    inp = ki.gen_prefill(77, [0, 1, 17, 64, 65, 130, 300], H=3, dtype=dtype, chunk=chunk,
                         with_s0=True)
    runs = [prefill_on_gpu(inp, chunk=chunk) for _ in range(3)]
    for o, S in runs[1:]:
        assert np.array_equal(o, runs[0][0]) and np.array_equal(S, runs[0][1])


def test_prefill_mixed_lengths_many_sequences():
    """48 sequences of random lengths from 0 to 2,500 tokens (about 60 K
    tokens, 8 heads, carried states): many more jobs than the intra-chunk
    kernel's persistent grid holds, of every tail length, so that jobs are
    handed out from its counter across sequence boundaries.  o and the final
    state per sequence within the bar."""
    rng = np.random.Generator(np.random.PCG64(91))
    lens = [int(x) for x in rng.integers(0, 2500, size=48)]
    inp = ki.gen_prefill(92, lens, H=8, dtype="bf16", chunk=64, with_s0=True)
    o, S = prefill_on_gpu(inp)
    _compare(inp, o, S, TOL_BF16, "48 mixed-length sequences")
