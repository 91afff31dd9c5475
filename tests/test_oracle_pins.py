"""Pins for the CPU oracle (no GPU).

The oracle is checked against what the pages and the mathematics fix, never
against a retyping of itself:
  * a hand-worked two-token example in exact fractions (tests/golden)
  * exact retrieval: beta = 1 and |k| = 1 give k_t^T S_t = v_t^T
  * beta = 0: the state only decays, channel by channel (closed form)
  * g = 0, beta = 0: the state is unchanged and o_t = S0^T q_t
  * the chunked (UT-transform) restatement agrees with the sequential form
  * brute force with explicit dense (I - beta k k^T) Diag(e^g) matrices
  * g = 0, beta = 1, orthonormal keys: every stored pair is retrieved exactly
  * linearity in (S0, V); split calls; varlen independence; head permutation
  * the Frobenius contraction bound for |k| = 1, beta in [0,1], g <= 0
A plausible slip in the oracle (decay after the update, readout from the old
state, S k instead of S^T k, per-column decay, a dropped beta, exp(-g), a
wrong token or head offset) fails at least one of these.
"""
import json
import os

import numpy as np
import pytest

import kda_inputs as ki
import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit_inputs(seed, L, dk, dv, H=1):
    r = np.random.Generator(np.random.PCG64(seed))
    q = r.standard_normal((L, H, dk)).astype(np.float32)
    k = r.standard_normal((L, H, dk)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = r.standard_normal((L, H, dv)).astype(np.float32)
    g = (-5.0 / (1.0 + np.exp(-r.standard_normal((L, H, dk))))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-r.standard_normal((L, H))))).astype(np.float32)
    S0 = r.standard_normal((H, dk, dv)).astype(np.float32) * np.float32(0.5)
    return q, k, v, g, beta, S0


def _c(a):
    return np.ascontiguousarray(a)


def test_hand_example_exact():
    with open(os.path.join(GOLDEN, "hand_2x2.json")) as f:
        gold = json.load(f)
    toks = gold["tokens"]
    L = len(toks)

    def lg(s):
        return {"0": 0.0, "ln(1/2)": np.log(0.5), "ln(1/4)": np.log(0.25)}[s]

    q = np.array([[t["q"]] for t in toks], dtype=np.float32)
    k = np.array([[t["k"]] for t in toks], dtype=np.float32)
    v = np.array([[t["v"]] for t in toks], dtype=np.float32)
    g = np.array([[[lg(x) for x in t["g"]]] for t in toks], dtype=np.float32)
    beta = np.array([[t["beta"]] for t in toks], dtype=np.float32)
    # 0.6 / 0.8 are not exact in binary; compare at the fp32 rounding of the inputs
    o, S = oracle.run_unit(q, k, v, g, beta, np.array(gold["S0"], dtype=np.float64), 0, L, 0)
    np.testing.assert_allclose(o, np.array(gold["o"]), rtol=0, atol=2e-6)
    np.testing.assert_allclose(S, np.array(gold["S_final"]), rtol=0, atol=2e-6)


@pytest.mark.parametrize("dk,dv", [(4, 4), (8, 6), (128, 128)])
def test_exact_retrieval_beta1_unit_k(dk, dv):
    r = np.random.Generator(np.random.PCG64(11))
    L = 9
    q, _, v, g, beta, S0 = _unit_inputs(1, L, dk, dv)
    # keys with four entries of +-1/2: exactly unit norm in fp32 and fp64
    k = np.zeros((L, 1, dk), dtype=np.float32)
    for t in range(L):
        idx = r.choice(dk, size=4, replace=False)
        k[t, 0, idx] = r.choice([-0.5, 0.5], size=4)
    beta[:] = 1.0
    # o_t = S_t^T k_t must equal v_t when q = k
    o, S = oracle.run_unit(_c(k), _c(k), v, g, beta, S0[0], 0, L, 0)
    np.testing.assert_allclose(o, v[:, 0, :].astype(np.float64), rtol=0, atol=1e-13)
    np.testing.assert_allclose(k[-1, 0].astype(np.float64) @ S, v[-1, 0], rtol=0, atol=1e-13)
    if dk == dv:  # a non-symmetric S0, so a transposed product (S k) would be caught
        assert np.abs(S0[0] - S0[0].T).max() > 0.1


def test_beta0_decay_only_closed_form():
    L, dk, dv = 7, 6, 5
    q, k, v, g, beta, S0 = _unit_inputs(2, L, dk, dv)
    beta[:] = 0.0
    o, S = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L, 0)
    b = np.cumsum(g[:, 0, :].astype(np.float64), axis=0)
    for t in range(L):
        St = np.exp(b[t])[:, None] * S0[0].astype(np.float64)
        np.testing.assert_allclose(o[t], St.T @ q[t, 0].astype(np.float64), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S, np.exp(b[-1])[:, None] * S0[0], rtol=1e-13, atol=1e-15)


def test_g0_beta0_identity():
    L, dk, dv = 5, 8, 3
    q, k, v, g, beta, S0 = _unit_inputs(3, L, dk, dv)
    g[:] = 0.0
    beta[:] = 0.0
    o, S = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L, 0)
    np.testing.assert_array_equal(S, S0[0].astype(np.float64))
    for t in range(L):
        np.testing.assert_allclose(o[t], S0[0].astype(np.float64).T @ q[t, 0], rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("L", [1, 15, 16, 17, 63, 64, 65, 130])
@pytest.mark.parametrize("fold", ["subblock", "direct"])
def test_chunked_matches_sequential(chunk, L, fold):
    if fold == "direct" and L > 65:
        pytest.skip("direct fold is O(L^2 dk) python loops")
    dk, dv = 32, 16
    q, k, v, g, beta, S0 = _unit_inputs(100 + L, L, dk, dv)
    o_seq, S_seq = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L, 0)
    f = lambda a: a[:, 0].astype(np.float64)
    o_ch, S_ch = chunked.run_unit(f(q), f(k), f(v), f(g), beta[:, 0].astype(np.float64),
                                  S0[0].astype(np.float64), chunk, fold=fold)
    scale_o = max(1.0, np.abs(o_seq).max())
    scale_S = max(1.0, np.abs(S_seq).max())
    assert np.abs(o_ch - o_seq).max() / scale_o < 1e-12
    assert np.abs(S_ch - S_seq).max() / scale_S < 1e-12


def test_chunked_matches_sequential_full_width_bf16_inputs():
    """dk = dv = 128 with bf16-rounded q, k, v drawn by the input recipe."""
    inp = ki.gen_prefill(7, [150], H=2, dtype="bf16", chunk=64, with_s0=True)
    o_seq, S_seq = oracle.prefill(inp)
    for h in range(2):
        f = lambda name: inp.f32(name)[:, h].astype(np.float64)
        o_ch, S_ch = chunked.run_unit(f("q"), f("k"), f("v"), f("g"),
                                      inp.beta[:, h].astype(np.float64),
                                      inp.S0[0, h].astype(np.float64), 64)
        assert np.abs(o_ch - o_seq[:, h]).max() / np.abs(o_seq[:, h]).max() < 1e-12
        assert np.abs(S_ch - S_seq[0, h]).max() / np.abs(S_seq[0, h]).max() < 1e-12


def test_brute_force_dense_matrices():
    L, dk, dv = 6, 5, 4
    q, k, v, g, beta, S0 = _unit_inputs(4, L, dk, dv)
    o, S = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L, 0)
    Sb = S0[0].astype(np.float64)
    for t in range(L):
        kt = k[t, 0].astype(np.float64)[:, None]
        vt = v[t, 0].astype(np.float64)[:, None]
        A = (np.eye(dk) - beta[t, 0] * (kt @ kt.T)) @ np.diag(np.exp(g[t, 0].astype(np.float64)))
        Sb = A @ Sb + beta[t, 0] * (kt @ vt.T)
        np.testing.assert_allclose(o[t], Sb.T @ q[t, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, Sb, rtol=1e-12, atol=1e-14)


def _hadamard(n):
    Hm = np.array([[1.0]])
    while Hm.shape[0] < n:
        Hm = np.block([[Hm, Hm], [Hm, -Hm]])
    return Hm


def test_orthonormal_keys_exact_retrieval():
    dk, dv = 16, 8
    Hm = _hadamard(dk) / 4.0          # entries +-1/4: exactly orthonormal rows
    L = dk
    q, _, v, g, beta, _ = _unit_inputs(5, L, dk, dv)
    k = Hm[:, None, :].astype(np.float32)
    g[:] = 0.0
    beta[:] = 1.0
    o, S = oracle.run_unit(q, _c(k), v, g, beta, None, 0, L, 0)
    for s in range(L):
        np.testing.assert_allclose(k[s, 0].astype(np.float64) @ S, v[s, 0], rtol=0, atol=1e-13)


def test_linearity_in_state_and_values():
    L, dk, dv = 9, 8, 6
    q, k, v, g, beta, S0 = _unit_inputs(6, L, dk, dv)
    _, _, v2, _, _, S02 = _unit_inputs(7, L, dk, dv)
    a, c = 0.75, -1.25
    o1, S1 = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L, 0)
    o2, S2 = oracle.run_unit(q, k, v2, g, beta, S02[0], 0, L, 0)
    v3 = (a * v.astype(np.float64) + c * v2).astype(np.float32)   # exact in fp32 here? no: compare loosely
    S03 = a * S0[0].astype(np.float64) + c * S02[0].astype(np.float64)
    o3, S3 = oracle.run_unit(q, k, v3, g, beta, S03, 0, L, 0)
    # v3 carries one fp32 rounding; the map itself is linear to fp64 rounding
    tol = 4e-7 * (np.abs(o1).max() + np.abs(o2).max())
    assert np.abs(o3 - (a * o1 + c * o2)).max() < tol
    assert np.abs(S3 - (a * S1 + c * S2)).max() < 4e-7 * (np.abs(S1).max() + np.abs(S2).max())


def test_split_calls_equal_one_call_and_decode_continues_prefill():
    L1, L2, dk, dv = 11, 7, 8, 8
    q, k, v, g, beta, S0 = _unit_inputs(8, L1 + L2, dk, dv)
    o, S = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L1 + L2, 0)
    oa, Sa = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L1, 0)
    ob, Sb = oracle.run_unit(q, k, v, g, beta, Sa, L1, L1 + L2, 0)
    np.testing.assert_array_equal(np.concatenate([oa, ob]), o)
    np.testing.assert_array_equal(Sb, S)
    # a decode step is one more token of the same recurrence
    step = ki.DecodeStep(_c(q[-1:]), _c(k[-1:]), _c(v[-1:]), _c(g[-1:]), _c(beta[-1:]), "f32")
    oc, Sc = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L1 + L2 - 1, 0)
    od, Sd = oracle.decode(Sc[None, None], step)
    np.testing.assert_array_equal(od[0, 0], o[-1])
    np.testing.assert_array_equal(Sd[0, 0], S)


def test_varlen_packed_equals_separate_and_head_permutation():
    lens = [5, 0, 17, 3]
    inp = ki.gen_prefill(9, lens, H=3, dtype="bf16", chunk=16, with_s0=True, dk=8, dv=4)
    o, S = oracle.prefill(inp)
    cu = inp.cu_seqlens
    for n, ln in enumerate(lens):
        sep = ki.PrefillInputs(*(np.ascontiguousarray(a[cu[n]:cu[n + 1]])
                                 for a in (inp.q, inp.k, inp.v, inp.g, inp.beta)),
                               inp.S0[n:n + 1].copy(), np.array([0, ln], dtype=np.int32),
                               inp.dtype, inp.chunk)
        on, Sn = oracle.prefill(sep)
        np.testing.assert_array_equal(on, o[cu[n]:cu[n + 1]])
        np.testing.assert_array_equal(Sn[0], S[n])
    # empty sequence: state passes through
    np.testing.assert_array_equal(S[1], inp.S0[1].astype(np.float64))
    perm = [2, 0, 1]
    pin = ki.PrefillInputs(*(np.ascontiguousarray(a[:, perm]) for a in
                             (inp.q, inp.k, inp.v, inp.g, inp.beta)),
                           np.ascontiguousarray(inp.S0[:, perm]), cu, inp.dtype, inp.chunk)
    op, Sp = oracle.prefill(pin)
    np.testing.assert_array_equal(op, o[:, perm])
    np.testing.assert_array_equal(Sp, S[:, perm])


def test_frobenius_contraction_bound():
    L, dk, dv = 40, 16, 16
    q, k, v, g, beta, S0 = _unit_inputs(10, L, dk, dv)
    S = S0[0].astype(np.float64)
    for t in range(L):
        Sn = oracle.run_unit(q, k, v, g, beta, S, t, t + 1, 0)[1]
        kn = np.linalg.norm(k[t, 0].astype(np.float64))
        # |k| is 1 up to fp32 rounding of the normalised key
        assert abs(kn - 1) < 1e-6
        bound = np.linalg.norm(S) + beta[t, 0] * np.linalg.norm(v[t, 0].astype(np.float64))
        assert np.linalg.norm(Sn) <= bound * (1 + 1e-6)
        S = Sn


def test_bf16_bits_upcast_exact():
    inp = ki.gen_prefill(12, [20], H=2, dtype="bf16", chunk=16, with_s0=True, dk=16, dv=8)
    o1, S1 = oracle.prefill(inp)
    f32 = ki.PrefillInputs(inp.f32("q"), inp.f32("k"), inp.f32("v"), inp.g, inp.beta,
                           inp.S0, inp.cu_seqlens, "f32", inp.chunk)
    o2, S2 = oracle.prefill(f32)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)


def test_input_recipe_ranges():
    inp = ki.gen_prefill(0, [64], H=2, dtype="f32", chunk=16)
    assert (inp.g < 0).all() and (inp.g > -5).all()
    assert (inp.beta > 0).all() and (inp.beta < 1).all()
    nq = np.linalg.norm(inp.q.astype(np.float64), axis=-1)
    assert np.abs(nq - 1).max() < 1e-5
    b = ki.gen_prefill(0, [64], H=2, dtype="bf16", chunk=16)
    x = b.f32("q")
    # the bf16 values are the fp32 ones rounded to nearest even
    np.testing.assert_array_equal(ki.f32_to_bf16_bits(x), b.q)


# ---------------------------------------------------------------- state pools
def test_round_bf16_matches_the_format():
    """round_bf16 against torch's bfloat16 conversion (round to nearest even)
    on fp32-representable values, including exact ties and both signs."""
    torch = pytest.importorskip("torch")
    r = np.random.Generator(np.random.PCG64(41))
    x = (r.standard_normal(200000) * np.exp(r.uniform(-20, 20, 200000))).astype(np.float32)
    # exact ties: 8 significant bits plus a half unit in the last place
    base = r.integers(128, 256, 2000).astype(np.float64)
    ties = np.ldexp(base + 0.5, r.integers(-30, 10, 2000) - 8).astype(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, 1.0, -1.0, 3.0e38])])
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_pool_identity_is_the_plain_decode():
    r = np.random.Generator(np.random.PCG64(42))
    S = ki.gen_decode_state(r, 3, 2)
    step = ki.gen_decode_step(r, 3, 2, "bf16")
    o1, S1 = oracle.decode(S, step)
    o2, S2 = oracle.decode_pool(S, step)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)


def test_pool_slots_gather_update_scatter_and_padding():
    """Sequence b updates row idx[b]; rows no sequence names are untouched;
    a negative slot gives o = 0 and touches nothing."""
    r = np.random.Generator(np.random.PCG64(43))
    P, B, H = 7, 4, 2
    pool = ki.gen_decode_state(r, P, H)
    step = ki.gen_decode_step(r, B, H, "bf16")
    idx = np.array([5, -1, 0, 3], dtype=np.int32)
    o, out = oracle.decode_pool(pool, step, idx)
    gathered = np.stack([pool[max(i, 0)] for i in idx])
    o_ref, S_ref = oracle.decode(gathered, step)
    for b, i in enumerate(idx):
        if i < 0:
            np.testing.assert_array_equal(o[b], 0.0)
        else:
            np.testing.assert_array_equal(o[b], o_ref[b])
            np.testing.assert_array_equal(out[i], S_ref[b])
    for row in set(range(P)) - {int(i) for i in idx if i >= 0}:
        np.testing.assert_array_equal(out[row], pool[row].astype(np.float64))


def test_bf16_pool_stores_the_rounded_updated_state():
    """A bf16 pool: the state is read exactly, updated in fp64, o is read out
    from the unrounded update, and the stored state is its bf16 rounding."""
    r = np.random.Generator(np.random.PCG64(44))
    B, H = 3, 2
    pool32 = ki.gen_decode_state(r, B, H)
    bits = ki.f32_to_bf16_bits(pool32)
    exact = oracle.bf16_bits_to_f64(bits)
    step = ki.gen_decode_step(r, B, H, "bf16")
    o, out = oracle.decode_pool(bits, step, state_bf16=True)
    o_ref, S_ref = oracle.decode(exact.astype(np.float32), step)   # bf16 values are exact in fp32
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(out, oracle.round_bf16(S_ref))
    # every stored value is a bf16 value
    np.testing.assert_array_equal(oracle.round_bf16(out), out)


def test_bf16_pool_identity_step_is_exact():
    """g = 0, beta = 0: a bf16 state comes back bit for bit."""
    r = np.random.Generator(np.random.PCG64(45))
    B, H = 2, 3
    bits = ki.f32_to_bf16_bits(ki.gen_decode_state(r, B, H))
    step = ki.gen_decode_step(r, B, H, "bf16")
    step.g[...] = 0.0
    step.beta[...] = 0.0
    o, out = oracle.decode_pool(bits, step, state_bf16=True)
    np.testing.assert_array_equal(out, oracle.bf16_bits_to_f64(bits))
    q = oracle.bf16_bits_to_f64(step.q)
    want = np.einsum("bhi,bhij->bhj", q, oracle.bf16_bits_to_f64(bits))
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-14)
