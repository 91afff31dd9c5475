"""GPU parity of the layer around the recurrence, through the C ABI:
the conv1d + SiLU + L2-norm prologue (``kda_conv_prologue``), the prefill
with its gated RMSNorm epilogue (``kda_prefill_chunked_gated``), the two
composed, and the fused whole-layer decode step (``kda_decode_layer_step``),
each against the fp64 layer oracle on the same seeded inputs."""
import numpy as np
import pytest

import kda_inputs as ki
import oracle
from oracle import layer as olayer

from kda_testlib import TOL_BF16, TOL_F32, assert_close, dev_tensor

pytestmark = pytest.mark.gpu

QS = 128 ** -0.5
RAGGED = [0, 1, 2, 3, 5, 64, 65, 130, 200, 0]


def _kda():
    import kda_linear_attention_gb300 as kda
    return kda


def _bf16_np(t):
    """bf16 device tensor -> exact fp64 numpy."""
    import torch
    return t.float().cpu().numpy().astype(np.float64)


def _check_no_device_error():
    assert _kda().device_error() == 0


def _prologue_gpu(L, with_conv0=True):
    import torch
    kda = _kda()
    d = lambda a: dev_tensor(a)
    cin = d(L.conv0).view(torch.bfloat16) if (with_conv0 and L.conv0 is not None) else None
    q, k, v, co = kda.conv_prologue(d(L.xq), d(L.xk), d(L.xv), d(L.conv_w), d(L.cu_seqlens),
                                    conv_in=cin, q_scale=QS)
    torch.cuda.synchronize()
    return q, k, v, co


def _assert_bf16_rounding_of(x_gpu, ref, what):
    """x_gpu is ref computed in fp32 and rounded to bf16: within half a bf16
    ulp of ref plus the fp32 arithmetic's error."""
    err = np.abs(x_gpu - ref)
    # |ref| = m 2^e with 0.5 <= m < 1: bf16 values there are 2^(e-8) apart
    half_ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 9)
    bound = half_ulp + 2e-5 * np.abs(ref).max()
    bad = err > bound
    assert not bad.any(), "%s: %d elements off by more than half a bf16 ulp (worst %.3e)" % (
        what, int(bad.sum()), float((err - bound).max()))


def assert_gated_close(out, out_ref, o_ref, gate, norm_w, tol_o, what, eps=1e-6):
    """The gated output inherits o's error through the row normalisation.
    With o within tol_o * max|o_ref| (the bar on o), x -> x / rms(x) turns an
    error d in row r into at most (1 + max|x_r| / rms_r) d / rms_r (first
    order), times |norm_w sigmoid(gate)|; rows whose o is small next to the
    tensor's largest values are amplified the most.  Checked row by row."""
    o_ref = np.asarray(o_ref, dtype=np.float64)
    rms = np.sqrt(np.mean(o_ref ** 2, axis=-1) + eps)
    mx_row = np.abs(o_ref).max(axis=-1)
    ws = np.abs(norm_w * olayer.sigmoid(gate)).max(axis=-1)
    d = tol_o * np.abs(o_ref).max()
    bound = (1.0 + mx_row / rms) * d / rms * ws + 1e-6
    err = np.abs(np.asarray(out, dtype=np.float64) - out_ref).max(axis=-1)
    bad = err > bound
    assert np.isfinite(out).all(), "%s: non-finite output" % what
    assert not bad.any(), "%s: %d rows beyond the bound inherited from o (worst ratio %.2f)" % (
        what, int(bad.sum()), float((err / bound).max()))
    return float((err / bound).max())


@pytest.mark.parametrize("with_conv0", [True, False])
@pytest.mark.parametrize("H", [1, 3])
def test_conv_prologue_ragged(with_conv0, H):
    L = ki.gen_layer(101 + H, RAGGED, H=H, with_conv0=with_conv0)
    q, k, v, co = _prologue_gpu(L, with_conv0)
    f = olayer._f64
    rq, rk, rv, rco = olayer.prologue(f(L.xq), f(L.xk), f(L.xv), L.conv_w,
                                      None if L.conv0 is None else f(L.conv0), L.cu_seqlens, QS)
    for name, x, r in (("q", q, rq), ("k", k, rk), ("v", v, rv)):
        _assert_bf16_rounding_of(_bf16_np(x), r, "prologue " + name)
    # the windows hold raw inputs: exact
    assert np.array_equal(_bf16_np(co), rco)


def test_conv_prologue_split_calls_carry_the_window():
    """Prologue over [0, T1) then [T1, T) with the window carried = one call."""
    import torch
    kda = _kda()
    T, T1, H = 150, 67, 2
    L = ki.gen_layer(105, [T], H=H)
    d = dev_tensor
    xs = [d(a) for a in (L.xq, L.xk, L.xv)]
    w = d(L.conv_w)
    cin = d(L.conv0).view(torch.bfloat16)
    q, k, v, co = kda.conv_prologue(*xs, w, d(np.array([0, T], np.int32)), conv_in=cin, q_scale=QS)
    a = [x[:T1].contiguous() for x in xs]
    b = [x[T1:].contiguous() for x in xs]
    q1, k1, v1, c1 = kda.conv_prologue(*a, w, d(np.array([0, T1], np.int32)), conv_in=cin, q_scale=QS)
    q2, k2, v2, c2 = kda.conv_prologue(*b, w, d(np.array([0, T - T1], np.int32)), conv_in=c1,
                                       q_scale=QS)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([q1, q2]), q) and torch.equal(torch.cat([v1, v2]), v)
    assert torch.equal(torch.cat([k1, k2]), k) and torch.equal(c2, co)


def _gated_gpu(inp, gate, norm_w, chunk, eps=1e-6):
    import torch
    kda = _kda()
    d = {n: dev_tensor(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta")}
    s0 = None if inp.S0 is None else dev_tensor(inp.S0)
    out, S = kda.prefill_chunked_gated(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                       dev_tensor(inp.cu_seqlens), dev_tensor(gate),
                                       dev_tensor(norm_w), S0=s0, chunk=chunk, eps=eps)
    torch.cuda.synchronize()
    _check_no_device_error()
    return out.cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("dtype,chunk", [("bf16", 64), ("bf16", 32), ("f32", 16)])
@pytest.mark.parametrize("with_s0", [False, True])
def test_gated_prefill_ragged(dtype, chunk, with_s0):
    lens = [0, 1, 17, 63, 64, 65, 130, 200]
    inp = ki.gen_prefill(110 + chunk, lens, H=3, dtype=dtype, chunk=chunk, with_s0=with_s0)
    rng = np.random.Generator(np.random.PCG64(111))
    gate = ki.f32_to_bf16_bits(rng.standard_normal((inp.T, 3, 128)).astype(np.float32))
    norm_w = (1.0 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    out, S = _gated_gpu(inp, gate, norm_w, chunk)
    o_ref, S_ref = oracle.prefill(inp)
    gf = olayer._f64(gate)
    out_ref = olayer.gated_rmsnorm(o_ref, gf, norm_w)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    cu = inp.cu_seqlens
    for n in range(inp.N):
        a, b = int(cu[n]), int(cu[n + 1])
        if b > a:
            assert_gated_close(out[a:b], out_ref[a:b], o_ref[a:b], gf[a:b], norm_w, tol,
                               "gated out, sequence %d" % n)
        assert_close(S[n], S_ref[n], tol, "S_out, sequence %d" % n)


@pytest.mark.parametrize("dtype,chunk", [("bf16", 64), ("f32", 16)])
def test_gated_prefill_saturated_gates(dtype, chunk):
    """Gates far in both tails: sigmoid saturates to 1 or underflows to 0
    (e^{-x} overflows), and a zero weight silences its channel."""
    lens = [70, 64, 5]
    inp = ki.gen_prefill(120 + chunk, lens, H=2, dtype=dtype, chunk=chunk, with_s0=True)
    rng = np.random.Generator(np.random.PCG64(121))
    vals = np.array([-200.0, -90.0, -20.0, -1.0, 0.0, 1.0, 20.0, 90.0, 200.0], np.float32)
    gate = ki.f32_to_bf16_bits(rng.choice(vals, size=(inp.T, 2, 128)).astype(np.float32))
    norm_w = (1.0 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    norm_w[::7] = 0.0
    out, S = _gated_gpu(inp, gate, norm_w, chunk)
    assert np.isfinite(out).all()
    assert (out[:, :, ::7] == 0).all()
    o_ref, S_ref = oracle.prefill(inp)
    gf = olayer._f64(gate)
    out_ref = olayer.gated_rmsnorm(o_ref, gf, norm_w)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    cu = inp.cu_seqlens
    for n in range(inp.N):
        a, b = int(cu[n]), int(cu[n + 1])
        assert_gated_close(out[a:b], out_ref[a:b], o_ref[a:b], gf[a:b], norm_w, tol,
                           "gated out, sequence %d" % n)
        assert_close(S[n], S_ref[n], tol, "S_out, sequence %d" % n)


def test_gated_prefill_4k_full():
    """The full 4K bf16 prefill (H = 96, chunk 64), every output."""
    inp = ki.workload_prefill("prefill_4k")
    rng = np.random.Generator(np.random.PCG64(112))
    gate = ki.f32_to_bf16_bits(rng.standard_normal((inp.T, inp.H, 128)).astype(np.float32))
    norm_w = (1.0 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    out, S = _gated_gpu(inp, gate, norm_w, 64)
    o_ref, S_ref = oracle.prefill(inp)
    gf = olayer._f64(gate)
    assert_gated_close(out, olayer.gated_rmsnorm(o_ref, gf, norm_w), o_ref, gf, norm_w, TOL_BF16,
                       "gated out")
    assert_close(S, S_ref, TOL_BF16, "S_out")


LAYER_CASES = [([0, 1, 70, 3, 129], 3, True, True),
               (RAGGED, 2, True, False),
               ([2, 1, 66, 0, 3, 190], 3, False, True),
               ([4096], 96, False, True)]


@pytest.mark.parametrize("one_call", [True, False], ids=["one_call", "two_calls"])
@pytest.mark.parametrize("lens,H,with_s0,with_conv0", LAYER_CASES)
def test_prefill_layer_against_the_layer_oracle(lens, H, with_s0, with_conv0, one_call):
    """The layer prefill from raw projections, in one call
    (``kda_layer_prefill``) and as two calls (prologue, then the gated
    tensor-core prefill), against the oracle's layer prefill with q, k, v
    rounded to bf16.  Sequences of 1 and 2 tokens carry part of the window
    before them into the window after them."""
    import torch
    kda = _kda()
    L = ki.gen_layer(120 + H, lens, H=H, with_s0=with_s0, with_conv0=with_conv0)
    d = dev_tensor
    s0 = None if L.S0 is None else d(L.S0)
    cin = d(L.conv0).view(torch.bfloat16) if with_conv0 else None
    out, S, co = kda.prefill_layer(d(L.xq), d(L.xk), d(L.xv), d(L.conv_w), d(L.g), d(L.beta),
                                   d(L.gate), d(L.norm_w), d(L.cu_seqlens),
                                   conv_in=cin, S0=s0, one_call=one_call)
    torch.cuda.synchronize()
    _check_no_device_error()
    out_ref, o_ref, S_ref, co_ref = olayer.prefill_layer(L, QS, round_qkv_bf16=True)
    cu = L.cu_seqlens
    out, S = out.cpu().numpy(), S.cpu().numpy()
    gf = olayer._f64(L.gate)
    for n in range(L.N):
        a, b = int(cu[n]), int(cu[n + 1])
        if b > a:
            assert_gated_close(out[a:b], out_ref[a:b], o_ref[a:b], gf[a:b], L.norm_w, TOL_BF16,
                               "layer out, sequence %d" % n)
        assert_close(S[n], S_ref[n], TOL_BF16, "layer S_out, sequence %d" % n)
    assert np.array_equal(_bf16_np(co), co_ref)


@pytest.mark.parametrize("lens,H", [(RAGGED, 2), ([4096], 96)])
def test_layer_prefill_equals_the_two_calls(lens, H):
    """kda_layer_prefill runs the prologue and the gated prefill on the same
    bf16 q, k, v as the two public calls, and every prefill kernel sums in a
    fixed order, so its outputs, final states and windows are the two-call
    path's bit for bit."""
    import torch
    kda = _kda()
    L = ki.gen_layer(150 + H, lens, H=H, with_s0=True)
    d = dev_tensor
    args = (d(L.xq), d(L.xk), d(L.xv), d(L.conv_w), d(L.g), d(L.beta), d(L.gate), d(L.norm_w),
            d(L.cu_seqlens))
    cin = d(L.conv0).view(torch.bfloat16)
    a = kda.prefill_layer(*args, conv_in=cin, S0=d(L.S0), one_call=True)
    b = kda.prefill_layer(*args, conv_in=cin, S0=d(L.S0), one_call=False)
    torch.cuda.synchronize()
    _check_no_device_error()
    for x, y, what in zip(a, b, ("out", "S_out", "conv_out")):
        assert torch.equal(x, y), what


def _pools(rng, P, H, state_bf16):
    S = (0.02 * rng.standard_normal((P, H, 128, 128))).astype(np.float32)
    if state_bf16:
        S = ki.f32_to_bf16_bits(S)
    conv = ki.f32_to_bf16_bits(rng.standard_normal((P, 3, 3, H, 128)).astype(np.float32))
    return S, conv


def _layer_step_gpu(step, conv_w, norm_w, S_dev, conv_dev, slots=None):
    import torch
    kda = _kda()
    d = dev_tensor
    out = kda.decode_layer_step(d(step.xq), d(step.xk), d(step.xv), conv_w, conv_dev, d(step.g),
                                d(step.beta), d(step.gate), norm_w, S_dev,
                                state_indices=None if slots is None else d(slots), q_scale=QS)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("state_bf16", [False, True])
def test_decode_layer_slots_padding_and_pools(state_bf16):
    import torch
    B, H, P = 5, 3, 8
    rng = np.random.Generator(np.random.PCG64(130 + state_bf16))
    L = ki.gen_layer(131, [1], H=H)
    step = ki.gen_layer_decode_step(rng, B, H)
    S, conv = _pools(rng, P, H, state_bf16)
    slots = np.array([6, -1, 0, 3, 7], dtype=np.int32)
    S_dev = dev_tensor(S)
    if state_bf16:
        S_dev = S_dev.view(torch.bfloat16)
    conv_dev = dev_tensor(conv).view(torch.bfloat16)
    out = _layer_step_gpu(step, dev_tensor(L.conv_w), dev_tensor(L.norm_w), S_dev, conv_dev, slots)
    _check_no_device_error()
    out_ref, S_ref, conv_ref = olayer.decode_layer(S, conv, step, L.conv_w, L.norm_w, QS,
                                                   state_indices=slots, state_bf16=state_bf16)
    assert np.all(out[1] == 0.0)
    assert_close(out, out_ref, TOL_BF16 if state_bf16 else 1e-4, "layer step out")
    S_after = _bf16_np(S_dev) if state_bf16 else S_dev.cpu().numpy()
    # rows 1, 2, 4, 5 are untouched (bit for bit)
    for r in (1, 2, 4, 5):
        assert np.array_equal(S_after[r], S_ref[r])
    used = [6, 0, 3, 7]
    if not state_bf16:
        for r in used:
            assert_close(S_after[r], S_ref[r], 1e-5, "pool row %d" % r)
    else:
        # each stored value is a bf16 neighbour of the exact (unrounded) update
        start = oracle.bf16_bits_to_f64(S).astype(np.float32)
        _, S_exact, _ = olayer.decode_layer(start, conv, step, L.conv_w, L.norm_w, QS,
                                            state_indices=slots)
        ex = S_exact[used]
        ulp = np.ldexp(1.0, np.frexp(np.abs(ex))[1] - 8)
        assert np.all(np.abs(S_after[used] - ex) <= ulp + 1e-6 * np.abs(ex).max())
        assert np.mean(S_after[used] == S_ref[used]) > 0.99
    assert np.array_equal(_bf16_np(conv_dev), conv_ref)


def test_decode_layer_invalid_slot_is_flagged():
    import torch
    kda = _kda()
    kda.device_error(reset=True)
    B, H, P = 2, 2, 3
    rng = np.random.Generator(np.random.PCG64(132))
    L = ki.gen_layer(133, [1], H=H)
    step = ki.gen_layer_decode_step(rng, B, H)
    S, conv = _pools(rng, P, H, False)
    S_dev, conv_dev = dev_tensor(S), dev_tensor(conv).view(torch.bfloat16)
    slots = np.array([5, 1], dtype=np.int32)
    out = _layer_step_gpu(step, dev_tensor(L.conv_w), dev_tensor(L.norm_w), S_dev, conv_dev, slots)
    assert kda.device_error(reset=True) & 2
    assert np.all(out[0] == 0.0)
    S_after = S_dev.cpu().numpy()
    assert np.array_equal(S_after[0], S[0]) and np.array_equal(S_after[2], S[2])


def test_prefill_layer_then_20_decode_layer_steps():
    """The GPU layer prefill over 97 tokens, then 20 fused layer steps on the
    carried windows and states, against the oracle doing the same."""
    import torch
    kda = _kda()
    H, T, steps = 4, 97, 20
    L = ki.gen_layer(140, [T, 33], H=H, with_s0=True)
    d = dev_tensor
    out, S, co = kda.prefill_layer(d(L.xq), d(L.xk), d(L.xv), d(L.conv_w), d(L.g), d(L.beta),
                                   d(L.gate), d(L.norm_w), d(L.cu_seqlens),
                                   conv_in=d(L.conv0).view(torch.bfloat16), S0=d(L.S0))
    _, _, S_ref, co_ref = olayer.prefill_layer(L, QS, round_qkv_bf16=True)
    conv_np = ki.f32_to_bf16_bits(co_ref.astype(np.float32))
    S_np = S_ref.astype(np.float32)
    rng = np.random.Generator(np.random.PCG64(141))
    for i in range(steps):
        step = ki.gen_layer_decode_step(rng, 2, H)
        o_gpu = _layer_step_gpu(step, d(L.conv_w), d(L.norm_w), S, co)
        o_ref, S_new, conv_new = olayer.decode_layer(S_np, conv_np, step, L.conv_w, L.norm_w, QS)
        assert_close(o_gpu, o_ref, TOL_BF16, "layer step %d out" % i)
        S_np = S_new.astype(np.float32)
        conv_np = ki.f32_to_bf16_bits(conv_new.astype(np.float32))
    _check_no_device_error()
    assert_close(S.cpu().numpy(), S_np, TOL_BF16, "state after 20 layer steps")
    assert np.array_equal(_bf16_np(co), olayer._f64(conv_np))


def test_decode_layer_b64_full():
    """The batched layer step at the decode workload's size (B = 64, H = 96),
    every output, fp32 pool with a permuted slot table."""
    import torch
    B, H = 64, 96
    rng = np.random.Generator(np.random.PCG64(150))
    L = ki.gen_layer(151, [1], H=H)
    step = ki.gen_layer_decode_step(rng, B, H)
    S, conv = _pools(rng, B, H, False)
    slots = rng.permutation(B).astype(np.int32)
    S_dev, conv_dev = dev_tensor(S), dev_tensor(conv).view(torch.bfloat16)
    out = _layer_step_gpu(step, dev_tensor(L.conv_w), dev_tensor(L.norm_w), S_dev, conv_dev, slots)
    _check_no_device_error()
    out_ref, S_ref, conv_ref = olayer.decode_layer(S, conv, step, L.conv_w, L.norm_w, QS,
                                                   state_indices=slots)
    assert_close(out, out_ref, 1e-4, "layer step out")
    assert_close(S_dev.cpu().numpy(), S_ref, 1e-5, "pool")
    assert np.array_equal(_bf16_np(conv_dev), conv_ref)


def test_conv_prologue_negative_cu_start_is_contained():
    """cu_seqlens starting below 0 breaks the call's precondition (the host
    cannot read the device array).  The prologue takes zeros for the window
    slots before token 0 instead of reading before the input buffer, raises
    bit 0 of the device error word, and a valid call afterwards is clean and
    matches the oracle."""
    import torch
    kda = _kda()
    L = ki.gen_layer(490, [50, 50], H=2, with_conv0=True)
    d = dev_tensor
    cin = d(L.conv0).view(torch.bfloat16)
    kda.device_error(reset=True)
    kda.conv_prologue(d(L.xq), d(L.xk), d(L.xv), d(L.conv_w), d(np.array([-3, 50, 100], np.int32)),
                      conv_in=cin, q_scale=QS)
    torch.cuda.synchronize()
    assert kda.device_error(reset=True) & 1, "the negative sequence start was not flagged"
    q, k, v, co = _prologue_gpu(L)
    _check_no_device_error()
    f = olayer._f64
    rq, rk, rv, rco = olayer.prologue(f(L.xq), f(L.xk), f(L.xv), L.conv_w, f(L.conv0),
                                      L.cu_seqlens, QS)
    for name, x, r in (("q", q, rq), ("k", k, rk), ("v", v, rv)):
        _assert_bf16_rounding_of(_bf16_np(x), r, "prologue " + name)
    assert np.array_equal(_bf16_np(co), rco)


def test_layer_prefill_without_tokens_passes_windows_and_states_through():
    """kda_layer_prefill on sequences that are all empty: every window and
    every state comes out as it went in (zeros where none came in)."""
    import torch
    kda = _kda()
    H = 2
    L = ki.gen_layer(160, [0, 0, 0], H=H, with_s0=True)
    d = dev_tensor
    cin = d(L.conv0).view(torch.bfloat16)
    out, S, co = kda.prefill_layer(d(L.xq), d(L.xk), d(L.xv), d(L.conv_w), d(L.g), d(L.beta),
                                   d(L.gate), d(L.norm_w), d(L.cu_seqlens), conv_in=cin, S0=d(L.S0))
    torch.cuda.synchronize()
    _check_no_device_error()
    assert out.shape[0] == 0
    assert torch.equal(co, cin)
    assert np.array_equal(S.cpu().numpy(), L.S0)
    _, S2, co2 = kda.prefill_layer(d(L.xq), d(L.xk), d(L.xv), d(L.conv_w), d(L.g), d(L.beta),
                                   d(L.gate), d(L.norm_w), d(L.cu_seqlens))
    torch.cuda.synchronize()
    _check_no_device_error()
    assert not co2.float().abs().max().item() and not S2.abs().max().item()
