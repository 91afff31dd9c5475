"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle on
the same seeded inputs, element by element over every output: the small
ragged cases and all five full-size workloads (the all-fp32 prefill, the
4K prefill, the 100-step batched decode, the 32K prefill with carried
state, and the 65,536-token varlen batch with its decode step), plus
properties that hold at any size."""
import numpy as np
import pytest

import kda_inputs as ki
import oracle
from kda_testlib import (TOL_BF16, TOL_F32, assert_close, decode_on_gpu, dev_tensor,
                         prefill_on_gpu, rel_err)

pytestmark = pytest.mark.gpu


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


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,H", [(1, 1), (3, 5), (7, 96)])
def test_decode_small(dtype, B, H):
    rng = np.random.Generator(np.random.PCG64(1000 + B * H))
    S = ki.gen_decode_state(rng, B, H)
    step = ki.gen_decode_step(rng, B, H, dtype)
    o_ref, S_ref = oracle.decode(S, step)
    Sd = dev_tensor(S)
    o = decode_on_gpu(Sd, step)
    assert_close(o, o_ref, _tol(dtype), "decode o")
    assert_close(Sd.cpu().numpy(), S_ref, _tol(dtype), "decode S")


def test_decode_b64_100_steps_full():
    """Batched decode, B=64, H=96, 100 consecutive in-place steps: every
    state is followed by the oracle in fp64 along the whole run; o of every
    step and every final state against it."""
    S, steps = ki.workload_decode("decode_b64")
    S_ref = S.astype(np.float64)
    Sd = dev_tensor(S)
    worst = 0.0
    for it, step in enumerate(steps):
        o = decode_on_gpu(Sd, step)
        o_ref, S_ref = oracle.decode(S_ref, step)
        worst = max(worst, assert_close(o, o_ref, TOL_BF16, "decode o at step %d" % it))
    S_fin = Sd.cpu().numpy()
    e = assert_close(S_fin, S_ref, TOL_BF16, "decode S after 100 steps")
    print("decode B=64 x 100 steps: worst o %.2e, final S %.2e" % (worst, e))


# ---------------------------------------------------------------- prefill, small
def test_prefill_tiny_fp32_full():
    """All-fp32 prefill: B=1, H=2, T=64, chunk 16 (element by element, 1e-5)."""
    inp = ki.workload_prefill("tiny_fp32")
    o_ref, S_ref = oracle.prefill(inp)
    o, S = prefill_on_gpu(inp)
    assert_close(o, o_ref, TOL_F32, "o")
    assert_close(S, S_ref, TOL_F32, "S_out")


RAGGED = [1, 63, 64, 65, 130, 0, 200, 17, 16, 33]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("with_s0", [False, True])
def test_prefill_ragged_varlen(dtype, chunk, with_s0):
    inp = ki.gen_prefill(300 + chunk, RAGGED, H=3, dtype=dtype, chunk=chunk, with_s0=with_s0)
    o_ref, S_ref = oracle.prefill(inp)
    o, S = prefill_on_gpu(inp)
    cu = inp.cu_seqlens
    tol = _tol(dtype)
    for n in range(inp.N):
        if cu[n + 1] > cu[n]:
            assert_close(o[cu[n]:cu[n + 1]], o_ref[cu[n]:cu[n + 1]], tol, "o seq %d" % n)
        if with_s0 or cu[n + 1] > cu[n]:
            assert_close(S[n], S_ref[n], tol, "S_out seq %d" % n)
        else:
            assert np.all(S[n] == 0)


def test_prefill_empty_batch_copies_state():
    inp = ki.gen_prefill(5, [0, 0], H=2, dtype="bf16", chunk=64, with_s0=True)
    o, S = prefill_on_gpu(inp)
    assert o.shape == (0, 2, 128)
    np.testing.assert_array_equal(S, inp.S0)


def test_prefill_in_place_state():
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(6, [70, 5], H=4, dtype="bf16", chunk=64, with_s0=True)
    o_ref, S_ref = oracle.prefill(inp)
    d = {n: dev_tensor(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta")}
    S = dev_tensor(inp.S0)
    o, S2 = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                dev_tensor(inp.cu_seqlens), S0=S, S_out=S, chunk=64)
    torch.cuda.synchronize()
    assert S2.data_ptr() == S.data_ptr()
    assert_close(o.cpu().numpy(), o_ref, TOL_BF16, "o")
    assert_close(S.cpu().numpy(), S_ref, TOL_BF16, "S in place")


def test_prefill_events_variant_matches_and_times_each_kernel():
    """kda_prefill_chunked_events computes the same prefill and brackets the
    chunk plan, intra-chunk kernel and state pass with the caller's events."""
    import torch
    import kda_linear_attention_gb300 as kda
    inp = ki.gen_prefill(12, [300, 64, 1], H=6, dtype="bf16", chunk=64, with_s0=True)
    d = {n: dev_tensor(getattr(inp, n)) for n in ("q", "k", "v", "g", "beta")}
    cu, s0 = dev_tensor(inp.cu_seqlens), dev_tensor(inp.S0)
    o1, S1 = kda.prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, S0=s0)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    o2, S2 = kda.prefill_chunked_events(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, evs, S0=s0)
    torch.cuda.synchronize()
    assert kda.device_error() == 0
    assert rel_err(o2.cpu().numpy(), o1.cpu().numpy()) <= 1e-5
    assert rel_err(S2.cpu().numpy(), S1.cpu().numpy()) <= 1e-5
    ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(3)]
    assert all(m >= 0 for m in ms) and ms[1] > 0 and ms[2] > 0
    o_ref, S_ref = oracle.prefill(inp)
    assert_close(o2.cpu().numpy(), o_ref, TOL_BF16, "o")
    assert_close(S2.cpu().numpy(), S_ref, TOL_BF16, "S")


def test_prefill_split_calls_and_decode_continuation():
    """prefill(T1) then prefill(T2, S0=S_out) and prefill(T-1) then one decode
    step reproduce the single call prefill(T1+T2): each piece is checked
    against the oracle of the whole sequence (the pieces chunk the tokens
    differently, so GPU-vs-GPU agreement is only at rounding level)."""
    T1, T2, H = 100, 77, 4
    full = ki.gen_prefill(8, [T1 + T2], H=H, dtype="bf16", chunk=64, with_s0=True)
    o_ref, S_ref = oracle.prefill(full)
    o_all, S_all = prefill_on_gpu(full)
    assert_close(o_all, o_ref, TOL_BF16, "whole o")

    def part(a, b):
        return ki.PrefillInputs(*(np.ascontiguousarray(x[a:b]) for x in
                                  (full.q, full.k, full.v, full.g, full.beta)),
                                None, np.array([0, b - a], dtype=np.int32), "bf16", 64)

    p1, p2 = part(0, T1), part(T1, T1 + T2)
    p1.S0 = full.S0
    o1, S1 = prefill_on_gpu(p1)
    o2, S2 = prefill_on_gpu(p2, S0=dev_tensor(S1))
    assert_close(np.concatenate([o1, o2]), o_ref, TOL_BF16, "split o")
    assert_close(S2, S_ref, TOL_BF16, "split S")
    assert rel_err(S2, S_all) < 2 * TOL_BF16
    # prefill(T-1) + decode of the last token
    pa = part(0, T1 + T2 - 1)
    pa.S0 = full.S0
    _, Sa = prefill_on_gpu(pa)
    Sd = dev_tensor(Sa)
    step = ki.DecodeStep(*(np.ascontiguousarray(x[-1:]) for x in
                           (full.q, full.k, full.v, full.g, full.beta)), "bf16")
    od = decode_on_gpu(Sd, step)
    assert_close(od[0], o_ref[-1], TOL_BF16, "decode after prefill o")
    assert_close(Sd.cpu().numpy(), S_ref, TOL_BF16, "decode after prefill S")


def test_prefill_split_calls_fp32_path():
    """The same split property on the fp32 CUDA-core path (chunk 32), where
    GPU-vs-GPU agreement is close to fp32 rounding."""
    T1, T2, H = 70, 45, 2
    full = ki.gen_prefill(18, [T1 + T2], H=H, dtype="f32", chunk=32, with_s0=True)
    o_all, S_all = prefill_on_gpu(full)

    def part(a, b):
        return ki.PrefillInputs(*(np.ascontiguousarray(x[a:b]) for x in
                                  (full.q, full.k, full.v, full.g, full.beta)),
                                None, np.array([0, b - a], dtype=np.int32), "f32", 32)

    p1, p2 = part(0, T1), part(T1, T1 + T2)
    p1.S0 = full.S0
    o1, S1 = prefill_on_gpu(p1)
    o2, S2 = prefill_on_gpu(p2, S0=dev_tensor(S1))
    assert rel_err(np.concatenate([o1, o2]), o_all) < 1e-5
    assert rel_err(S2, S_all) < 1e-5


# ---------------------------------------------------------------- full-size workloads
def test_prefill_4k_full():
    """bf16 prefill, H=96, T=4096, chunk 64, S0 = 0: every output against the oracle."""
    inp = ki.workload_prefill("prefill_4k")
    o, S = prefill_on_gpu(inp)
    o_ref, S_ref = oracle.prefill(inp)
    assert_close(o, o_ref, TOL_BF16, "o")
    assert_close(S, S_ref, TOL_BF16, "S_out")


def _oracle_heads(inp, n, heads):
    """The oracle's o [len_n, len(heads), dv] and S [len(heads), dk, dv] of
    sequence n on the given heads."""
    ref = oracle.prefill(inp, units=[(n, h) for h in heads])
    o = np.stack([ref[(n, h)][0] for h in heads], axis=1)
    S = np.stack([ref[(n, h)][1] for h in heads])
    return o, S


def test_prefill_32k_carry_full():
    """bf16 prefill, H=96, T=32768, S0 ~ N(0, 0.02^2): every head, every
    element of o and of the final state against the oracle (the long chain
    of carried fp32 state is where accumulated error would show).  The
    oracle runs 16 heads at a time to bound host memory; the bar applies to
    the whole tensor."""
    inp = ki.workload_prefill("prefill_32k_carry")
    o, S = prefill_on_gpu(inp)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    o_ref_max = S_ref_max = 0.0
    o_err = S_err = 0.0
    for h0 in range(0, inp.H, 16):
        heads = list(range(h0, min(inp.H, h0 + 16)))
        o_r, S_r = _oracle_heads(inp, 0, heads)
        o_err = max(o_err, float(np.abs(o[:, heads].astype(np.float64) - o_r).max()))
        S_err = max(S_err, float(np.abs(S[0, heads].astype(np.float64) - S_r).max()))
        o_ref_max = max(o_ref_max, float(np.abs(o_r).max()))
        S_ref_max = max(S_ref_max, float(np.abs(S_r).max()))
    print("32K carry: o %.2e, S %.2e" % (o_err / o_ref_max, S_err / S_ref_max))
    assert o_err <= TOL_BF16 * o_ref_max, "o: max rel err %.3e" % (o_err / o_ref_max)
    assert S_err <= TOL_BF16 * S_ref_max, "S_out: max rel err %.3e" % (S_err / S_ref_max)


def test_varlen_64k_then_decode_full():
    """Varlen packed prefill (8 sequences, 65536 tokens) with per-sequence
    S0, then one decode step for all 8 from the final states: every
    (sequence, head) unit against the oracle, the bar applied per sequence
    (o and S_out of each sequence over all its heads), and the decode step's
    o and states against the oracle's decode from the oracle's own final
    states."""
    pre, step = ki.workload_varlen_with_decode("varlen_64k")
    o, S = prefill_on_gpu(pre)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    Sd = dev_tensor(S)
    od = decode_on_gpu(Sd, step)
    Sd_np = Sd.cpu().numpy()
    cu = pre.cu_seqlens
    heads = list(range(pre.H))
    S_ref = np.empty((pre.N, pre.H, 128, 128), dtype=np.float64)
    worst = 0.0
    for n in range(pre.N):
        o_r, S_ref[n] = _oracle_heads(pre, n, heads)
        worst = max(worst, assert_close(o[cu[n]:cu[n + 1]], o_r, TOL_BF16, "o of sequence %d" % n))
        assert_close(S[n], S_ref[n], TOL_BF16, "S_out of sequence %d" % n)
        del o_r
    od_ref, Sd_ref = oracle.decode(S_ref, step)
    for n in range(pre.N):
        assert_close(od[n], od_ref[n], TOL_BF16, "decode o of sequence %d" % n)
        assert_close(Sd_np[n], Sd_ref[n], TOL_BF16, "decode S of sequence %d" % n)
    print("varlen 64K: worst per-sequence o error %.2e" % worst)


# ---------------------------------------------------------------- state pools
def _pool_gpu(pool_in, state_bf16):
    return dev_tensor(pool_in)     # uint16 bit patterns become a bf16 tensor


def _pool_host(t, state_bf16):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_decode_pool_slots_padding_and_storage(state_dtype):
    """Pool decode through kda_decode_step_pool against the oracle: permuted
    slots, padding rows (o = 0, state untouched), rows nobody names untouched;
    a bf16 pool stores a correct bf16 rounding of the updated state."""
    import torch
    import kda_linear_attention_gb300 as kda
    bf = state_dtype == "bf16"
    r = np.random.Generator(np.random.PCG64(46))
    P, B, H = 9, 6, 8
    pool32 = ki.gen_decode_state(r, P, H)
    step = ki.gen_decode_step(r, B, H, "bf16")
    idx = np.array([4, -1, 0, 8, 2, -1], dtype=np.int32)
    pool_in = ki.f32_to_bf16_bits(pool32) if bf else pool32
    o_ref, pool_ref = oracle.decode_pool(pool_in, step, idx, state_bf16=bf)
    S = _pool_gpu(pool_in, bf)
    d = {n: dev_tensor(getattr(step, n)) for n in ("q", "k", "v", "g", "beta")}
    o = kda.decode_step_pool(d["q"], d["k"], d["v"], d["g"], d["beta"], S,
                             state_indices=dev_tensor(idx))
    torch.cuda.synchronize()
    assert kda.device_error() == 0
    o = o.cpu().numpy()
    assert_close(o, o_ref, TOL_BF16, "o")
    for b in np.nonzero(idx < 0)[0]:
        np.testing.assert_array_equal(o[b], 0.0)
    got = _pool_host(S, bf)
    start = oracle.bf16_bits_to_f64(pool_in) if bf else pool32.astype(np.float64)
    used = {int(i) for i in idx if i >= 0}
    for row in set(range(P)) - used:
        np.testing.assert_array_equal(got[row], start[row])
    rows = sorted(used)
    if not bf:
        assert_close(got[rows], pool_ref[rows], TOL_BF16, "S")
        return
    # the exact (unrounded) update, and the bf16 spacing at each value
    gathered = np.stack([start[max(i, 0)] for i in idx]).astype(np.float32)
    _, S_exact = oracle.decode(gathered, step)
    exact = np.stack([S_exact[list(idx).index(i)] for i in rows])
    # a bf16 neighbour of the exact value, up to the kernel's fp32 arithmetic
    # (which matters only where cancellation leaves a value near zero)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    slack = 1e-6 * np.abs(exact).max()
    assert np.all(np.abs(got[rows] - exact) <= ulp + slack), "a stored value is not a neighbour"
    same = np.mean(got[rows] == pool_ref[rows])
    assert same > 0.99, "rounding decisions differ from the oracle's on %.2f%%" % (100 * (1 - same))


def test_decode_pool_invalid_slot_is_flagged_and_skipped():
    import torch
    import kda_linear_attention_gb300 as kda
    r = np.random.Generator(np.random.PCG64(47))
    P, B, H = 3, 2, 4
    pool = ki.gen_decode_state(r, P, H)
    step = ki.gen_decode_step(r, B, H, "bf16")
    S = dev_tensor(pool)
    d = {n: dev_tensor(getattr(step, n)) for n in ("q", "k", "v", "g", "beta")}
    kda.device_error(reset=True)
    o = kda.decode_step_pool(d["q"], d["k"], d["v"], d["g"], d["beta"], S,
                             state_indices=dev_tensor(np.array([1, 3], dtype=np.int32)))
    torch.cuda.synchronize()
    assert kda.device_error(reset=True) & 2
    np.testing.assert_array_equal(o.cpu().numpy()[1], 0.0)
    o_ref, pool_ref = oracle.decode_pool(pool, step, np.array([1, -1], dtype=np.int32))
    assert_close(o.cpu().numpy()[0], o_ref[0], TOL_BF16, "o")
    assert_close(S.cpu().numpy(), pool_ref, TOL_BF16, "pool")


def test_decode_bf16_state_trajectory_against_both_oracles():
    """50 in-place steps on a bf16 pool: against the bf16-storing oracle
    (same rounding points) within the bf16 bar, and against the fp32/fp64
    oracle (the drift a bf16 state costs), which must stay bounded."""
    import torch
    import kda_linear_attention_gb300 as kda
    r = np.random.Generator(np.random.PCG64(48))
    B, H, steps = 4, 16, 50
    S32 = ki.gen_decode_state(r, B, H)
    bits = ki.f32_to_bf16_bits(S32)
    S = dev_tensor(bits)
    ref_bf = bits
    ref_f = oracle.bf16_bits_to_f64(bits).astype(np.float32)
    worst_bf = worst_f = 0.0
    for _ in range(steps):
        step = ki.gen_decode_step(r, B, H, "bf16")
        d = {n: dev_tensor(getattr(step, n)) for n in ("q", "k", "v", "g", "beta")}
        o = kda.decode_step_pool(d["q"], d["k"], d["v"], d["g"], d["beta"], S).cpu().numpy()
        o_bf, pool_bf = oracle.decode_pool(ref_bf, step, state_bf16=True)
        ref_bf = ki.f32_to_bf16_bits(pool_bf.astype(np.float32))   # exact: values are bf16
        o_f, S_f = oracle.decode(ref_f, step)
        ref_f = S_f.astype(np.float32)
        worst_bf = max(worst_bf, rel_err(o, o_bf))
        worst_f = max(worst_f, rel_err(o, o_f))
    torch.cuda.synchronize()
    assert worst_bf <= TOL_BF16, worst_bf
    assert worst_f <= 1e-2, worst_f
    S_end = S.float().cpu().numpy()
    assert rel_err(S_end, oracle.bf16_bits_to_f64(ref_bf)) <= TOL_BF16
    print("bf16 state, %d steps: o vs bf16 oracle %.2e, vs fp32 state %.2e, S vs fp32 %.2e"
          % (steps, worst_bf, worst_f, rel_err(S_end, ref_f)))
