"""CPU pins of the layer oracle (``oracle/layer.py``): the conv1d + SiLU +
L2-norm prologue and the RMSNorm + sigmoid-gate epilogue of the KDA layer
("Colibri Kimi K3 Metal backend", sections 8.3 and 8.4), and the whole-layer
compositions.  Each check compares the oracle with something other than
itself: closed forms, numpy's own convolution, a hand-worked impulse
response, invariants, and the continuity of a prefill followed by a decode
step."""
import numpy as np
import pytest

import kda_inputs as ki
import oracle
from oracle import layer


def test_silu_closed_forms():
    x = np.linspace(-30.0, 30.0, 601)
    s = layer.silu(x)
    # x sigma(x) - (-x) sigma(-x) = x (sigma(x) + sigma(-x)) = x
    assert np.allclose(s - layer.silu(-x), x, rtol=0, atol=1e-13)
    assert layer.silu(np.array([0.0]))[0] == 0.0
    # sigma(2) = 1 / (1 + e^-2)
    assert abs(layer.silu(np.array([2.0]))[0] - 2.0 / (1.0 + np.exp(-2.0))) < 1e-15
    assert abs(layer.silu(np.array([50.0]))[0] - 50.0) < 1e-12
    assert abs(layer.silu(np.array([-50.0]))[0]) < 1e-18


def test_conv_impulse_response_by_hand():
    # taps (w0, w1, w2, w3) = (1, 2, 3, 4), w3 on the newest input; a unit
    # impulse at t = 0 with an empty window gives y_t = w_{3-t}: 4, 3, 2, 1, 0
    w = np.array([[1.0, 2.0, 3.0, 4.0]])
    x = np.array([[1.0], [0.0], [0.0], [0.0], [0.0]])
    y, win = layer.conv_window(x, w, None)
    assert y[:, 0].tolist() == [4.0, 3.0, 2.0, 1.0, 0.0]
    assert win[:, 0].tolist() == [0.0, 0.0, 0.0]
    # a window (oldest first) of (5, 6, 7) and x_0 = 1: y_0 = 1*5 + 2*6 + 3*7 + 4*1
    y, win = layer.conv_window(np.array([[1.0]]), w, np.array([[5.0], [6.0], [7.0]]))
    assert y[0, 0] == 5 + 12 + 21 + 4
    assert win[:, 0].tolist() == [6.0, 7.0, 1.0]


def test_conv_matches_numpy_convolve():
    rng = np.random.default_rng(1)
    L, Cn, K = 37, 5, 4
    x = rng.standard_normal((L, Cn))
    w = rng.standard_normal((Cn, K))
    y, _ = layer.conv_window(x, w, None)
    for c in range(Cn):
        # y_t = sum_j h_j x_{t-j} with h_j = w_{K-1-j}: numpy's full convolution
        ref = np.convolve(x[:, c], w[c, ::-1])[:L]
        assert np.allclose(y[:, c], ref, rtol=0, atol=1e-13)


def test_conv_window_carry_equals_one_pass():
    rng = np.random.default_rng(2)
    L, Cn, K = 20, 3, 4
    x = rng.standard_normal((L, Cn))
    w = rng.standard_normal((Cn, K))
    y_all, win_all = layer.conv_window(x, w, None)
    for cut in (0, 1, 2, 3, 9, 20):
        y1, win1 = layer.conv_window(x[:cut], w, None)
        y2, win2 = layer.conv_window(x[cut:], w, win1)
        assert np.allclose(np.concatenate([y1, y2]), y_all, rtol=0, atol=1e-13)
        assert np.allclose(win2, win_all, rtol=0, atol=0)
    # a carried window = the same inputs placed before the sequence
    pre = rng.standard_normal((K - 1, Cn))
    y_c, _ = layer.conv_window(x, w, pre)
    y_p, _ = layer.conv_window(np.concatenate([pre, x]), w, None)
    assert np.allclose(y_c, y_p[K - 1:], rtol=0, atol=1e-13)


def test_l2_normalise_closed_form():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((7, 128))
    scale = 128 ** -0.5
    out = layer.l2_normalise(z, scale, 1e-6)
    nz = np.linalg.norm(z, axis=-1)
    assert np.allclose(np.linalg.norm(out, axis=-1), scale * nz / np.sqrt(nz ** 2 + 1e-6), rtol=1e-14)
    # same direction
    cos = np.sum(out * z, axis=-1) / (np.linalg.norm(out, axis=-1) * nz)
    assert np.allclose(cos, 1.0, rtol=0, atol=1e-14)
    assert np.all(layer.l2_normalise(np.zeros((2, 128))) == 0.0)


def test_gated_rmsnorm_closed_forms():
    rng = np.random.default_rng(4)
    o = rng.standard_normal((6, 3, 128))
    one = np.ones(128)
    big = np.full_like(o, 60.0)              # sigmoid(60) = 1 to double precision
    out = layer.gated_rmsnorm(o, big, one, eps=0.0)
    # with eps = 0 the result is o * sqrt(d) / ||o||: unit RMS per head
    assert np.allclose(out, o * np.sqrt(128) / np.linalg.norm(o, axis=-1, keepdims=True), rtol=1e-13)
    assert np.allclose(np.sqrt(np.mean(out ** 2, axis=-1)), 1.0, rtol=1e-13)
    # invariant to the scale of o (eps = 0), linear in the weight
    assert np.allclose(layer.gated_rmsnorm(3.7 * o, big, one, 0.0), out, rtol=1e-13)
    w = rng.standard_normal(128)
    assert np.allclose(layer.gated_rmsnorm(o, big, w, 0.0), out * w, rtol=1e-13)
    # a zero gate halves the output; sigmoid(x) + sigmoid(-x) = 1
    gz = layer.gated_rmsnorm(o, np.zeros_like(o), one, 0.0)
    assert np.allclose(gz, 0.5 * out, rtol=1e-13)
    gg = rng.standard_normal(o.shape)
    s = layer.gated_rmsnorm(o, gg, one, 0.0) + layer.gated_rmsnorm(o, -gg, one, 0.0)
    assert np.allclose(s, out, rtol=1e-12)
    # eps keeps a zero row at zero
    assert np.all(layer.gated_rmsnorm(np.zeros((1, 128)), np.zeros((1, 128)), one, 1e-6) == 0.0)


def test_prologue_varlen_independent_and_windows():
    L = ki.gen_layer(11, [5, 0, 1, 9], H=2)
    f = layer._f64
    s = 128 ** -0.5
    q, k, v, co = layer.prologue(f(L.xq), f(L.xk), f(L.xv), L.conv_w, f(L.conv0), L.cu_seqlens, s)
    cu = L.cu_seqlens
    for n in range(L.N):
        a, b = int(cu[n]), int(cu[n + 1])
        qn, kn, vn, con = layer.prologue(f(L.xq)[a:b], f(L.xk)[a:b], f(L.xv)[a:b], L.conv_w,
                                         f(L.conv0)[n:n + 1], np.array([0, b - a]), s)
        assert np.array_equal(qn, q[a:b]) and np.array_equal(kn, k[a:b]) and np.array_equal(vn, v[a:b])
        assert np.array_equal(con[0], co[n])
    # the empty sequence keeps its window; a one-token sequence shifts it by one
    assert np.array_equal(co[1], f(L.conv0)[1])
    n, t = 2, int(cu[2])
    assert np.array_equal(co[n, :, :2], f(L.conv0)[n, :, 1:])
    assert np.array_equal(co[n, 0, 2], f(L.xq)[t]) and np.array_equal(co[n, 2, 2], f(L.xv)[t])
    # q and k come out with norms s and 1 (up to eps), v is the plain SiLU
    nz = np.linalg.norm(q, axis=-1)
    assert np.all(nz <= s * (1 + 1e-12)) and np.all(nz > 0.9 * s)
    assert np.all(np.linalg.norm(k, axis=-1) <= 1 + 1e-12)


def test_prologue_zero_window_is_zero_padding():
    L = ki.gen_layer(12, [6], H=1, with_conv0=False)
    f = layer._f64
    q0, k0, v0, _ = layer.prologue(f(L.xq), f(L.xk), f(L.xv), L.conv_w, None, L.cu_seqlens, 1.0)
    zeros = np.zeros((1, 3, 3, 1, 128))
    q1, k1, v1, _ = layer.prologue(f(L.xq), f(L.xk), f(L.xv), L.conv_w, zeros, L.cu_seqlens, 1.0)
    assert np.array_equal(q0, q1) and np.array_equal(v0, v1)
    # v = SiLU(conv), brute force per channel with numpy's convolution
    x = f(L.xv)[:, 0, :]
    w = L.conv_w[2, 0].astype(np.float64)
    for c in (0, 17, 127):
        ref = layer.silu(np.convolve(x[:, c], w[c, ::-1])[:6])
        assert np.allclose(v0[:, 0, c], ref, rtol=0, atol=1e-13)


def test_oracle_takes_fp64_inputs_exactly():
    inp = ki.gen_prefill(13, [9], H=2, dtype="f32", with_s0=True)
    o32, S32 = oracle.prefill(inp)
    inp64 = ki.PrefillInputs(inp.q.astype(np.float64), inp.k.astype(np.float64),
                             inp.v.astype(np.float64), inp.g, inp.beta, inp.S0, inp.cu_seqlens,
                             "f64", 64)
    o64, S64 = oracle.prefill(inp64)
    assert np.array_equal(o32, o64) and np.array_equal(S32, S64)


@pytest.mark.parametrize("state_bf16", [False, True])
def test_prefill_layer_then_decode_layer_continues(state_bf16):
    """Prefill over T tokens, then one decode-layer step for token T, equals
    the prefill layer over T + 1 tokens at its last token (fp64 q/k/v on both
    sides)."""
    T, H = 7, 2
    L = ki.gen_layer(14, [T + 1], H=H, with_s0=True)
    s = 128 ** -0.5
    out_full, _, S_full, co_full = layer.prefill_layer(L, s, round_qkv_bf16=False)

    def cut(a, b):
        return a[:b]
    head = ki.LayerInputs(cut(L.xq, T), cut(L.xk, T), cut(L.xv, T), L.conv_w, L.conv0,
                          cut(L.gate, T), L.norm_w, cut(L.g, T), cut(L.beta, T),
                          np.array([0, T], dtype=np.int32), L.S0)
    out_h, _, S_h, co_h = layer.prefill_layer(head, s, round_qkv_bf16=False)
    assert np.allclose(out_h, out_full[:T], rtol=0, atol=1e-12)
    step = ki.LayerDecodeStep(L.xq[T:], L.xk[T:], L.xv[T:], L.gate[T:], L.g[T:], L.beta[T:])
    conv_pool = ki.f32_to_bf16_bits(co_h.astype(np.float32))   # raw bf16 inputs: exact
    pool = S_h.astype(np.float32)
    if state_bf16:
        pool = ki.f32_to_bf16_bits(pool)
    out_d, pool_d, conv_d = layer.decode_layer(pool, conv_pool, step, L.conv_w, L.norm_w, s,
                                               state_bf16=state_bf16)
    assert np.array_equal(conv_d, co_full)
    if state_bf16:
        # the stored state was rounded once before the step and once after it
        assert np.allclose(out_d[0], out_full[T], rtol=0, atol=2e-2)
        assert np.array_equal(pool_d[0], oracle.round_bf16(pool_d[0]))
    else:
        # the pool was stored as fp32: agreement to fp32 rounding of S
        assert np.allclose(out_d[0], out_full[T], rtol=0, atol=1e-5)
        assert np.allclose(pool_d[0], S_full[0], rtol=0, atol=1e-7)


def test_decode_layer_slots_and_padding():
    B, H, P = 3, 2, 5
    rng = np.random.Generator(np.random.PCG64(15))
    L = ki.gen_layer(15, [1], H=H)
    step = ki.gen_layer_decode_step(rng, B, H)
    pool = (0.02 * rng.standard_normal((P, H, 128, 128))).astype(np.float32)
    conv = ki.f32_to_bf16_bits(rng.standard_normal((P, 3, 3, H, 128)).astype(np.float32))
    slots = np.array([4, -1, 1], dtype=np.int32)
    out, pool2, conv2 = layer.decode_layer(pool, conv, step, L.conv_w, L.norm_w, 0.1,
                                           state_indices=slots)
    assert np.all(out[1] == 0.0)
    untouched = [0, 2, 3]
    assert np.array_equal(pool2[untouched], pool[untouched].astype(np.float64))
    assert np.array_equal(conv2[untouched], layer._f64(conv)[untouched])
    # the slot-4 row equals the identity-slot step of sequence 0 alone
    one = ki.LayerDecodeStep(step.xq[:1], step.xk[:1], step.xv[:1], step.gate[:1], step.g[:1],
                             step.beta[:1])
    o1, p1, c1 = layer.decode_layer(pool[4:5], conv[4:5], one, L.conv_w, L.norm_w, 0.1)
    assert np.array_equal(out[0], o1[0]) and np.array_equal(pool2[4], p1[0])
    assert np.array_equal(conv2[4], c1[0])
