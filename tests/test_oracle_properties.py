"""Randomised properties of the oracle (CPU, hypothesis): over arbitrary
lengths, widths, chunk sizes, gate ranges (down to the -5 bound, and all-zero
gates) and beta in [0, 1], the chunked restatement with the 16-row
sub-block folding must agree with the sequential recurrence to fp64
rounding, and a prefill split anywhere must equal one call."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import chunked  # noqa: E402


def _draw(seed, L, dk, dv, gmin, beta_hi):
    r = np.random.Generator(np.random.PCG64(seed))
    q = r.standard_normal((L, 1, dk)).astype(np.float32)
    k = r.standard_normal((L, 1, dk)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((L, 1, dv)).astype(np.float32)
    g = (gmin * r.random((L, 1, dk))).astype(np.float32)          # in [gmin, 0]
    beta = (beta_hi * r.random((L, 1))).astype(np.float32)
    S0 = (0.5 * r.standard_normal((1, dk, dv))).astype(np.float32)
    return q, k, v, g, beta, S0


@settings(max_examples=25, deadline=None)
@given(seed=st.integers(0, 2 ** 31 - 1), L=st.integers(1, 140),
       dk=st.sampled_from([16, 32]), dv=st.sampled_from([8, 16]),
       chunk=st.sampled_from([16, 32, 64]), gmin=st.sampled_from([0.0, -0.5, -5.0]),
       beta_hi=st.sampled_from([0.0, 1.0]))
def test_chunked_restatement_matches_sequential(seed, L, dk, dv, chunk, gmin, beta_hi):
    q, k, v, g, beta, S0 = _draw(seed, L, dk, dv, gmin, beta_hi)
    o_seq, S_seq = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L, 0)
    f = lambda a: a[:, 0].astype(np.float64)
    o_ch, S_ch = chunked.run_unit(f(q), f(k), f(v), f(g), beta[:, 0].astype(np.float64),
                                  S0[0].astype(np.float64), chunk)
    assert np.abs(o_ch - o_seq).max() <= 1e-12 * max(1.0, np.abs(o_seq).max())
    assert np.abs(S_ch - S_seq).max() <= 1e-12 * max(1.0, np.abs(S_seq).max())


@settings(max_examples=25, deadline=None)
@given(seed=st.integers(0, 2 ** 31 - 1), L=st.integers(2, 120), data=st.data())
def test_split_prefill_equals_one_call(seed, L, data):
    cut = data.draw(st.integers(1, L - 1))
    q, k, v, g, beta, S0 = _draw(seed, L, 16, 8, -5.0, 1.0)
    o_all, S_all = oracle.run_unit(q, k, v, g, beta, S0[0], 0, L, 0)
    o_a, S_a = oracle.run_unit(q, k, v, g, beta, S0[0], 0, cut, 0)
    o_b, S_b = oracle.run_unit(q, k, v, g, beta, S_a.astype(np.float32), cut, L, 0)
    # the carried state passes through fp32 between the calls, as a caller's S_out does
    tol = 1e-6 * max(1.0, np.abs(S_all).max())
    assert np.abs(np.concatenate([o_a, o_b]) - o_all).max() <= 1e-5 * max(1.0, np.abs(o_all).max())
    assert np.abs(S_b - S_all).max() <= tol
