"""The float64 chunked (WY) restatement against the float64 token recurrence, by brute
force on small inputs, and the algebraic properties of its intermediates."""
import math

import numpy as np
import pytest

import oracle
from oracle import chunked
from oracle_pins import _random_case


@pytest.mark.parametrize("C", [1, 16, 32, 64])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 31, 33, 63, 64, 65, 130])
def test_chunked_equals_recurrence(C, T):
    c = _random_case(100 + T, T=T, H=2, K=8, V=6)
    o_ref, s_ref = oracle.forward(**c)
    o, s = chunked.forward(**c, chunk_size=C)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-11)
    assert np.allclose(s, s_ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("gscale", [1.0, 40.0])
def test_chunked_equals_recurrence_nonsafe(gscale):
    """The non-safe gate -exp(A_log) softplus(g + dt_bias) is unbounded below; with raw g up to
    about +-120 single tokens decay by e^-1000 and more, and the chunked form (decay ratios
    2^(G_i - G_j), j <= i) still equals the token recurrence."""
    c = _random_case(55, T=130, H=2, K=8, V=6)
    c["g"] = c["g"] * gscale
    c["mode"] = oracle.GATE_NONSAFE
    o_ref, s_ref = oracle.forward(**c)
    assert np.isfinite(o_ref).all()
    for C in (16, 64):
        o, s = chunked.forward(**c, chunk_size=C)
        assert np.allclose(o, o_ref, rtol=0, atol=1e-11)
        assert np.allclose(s, s_ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("mode", [oracle.GATE_PRE, oracle.GATE_SAFE, oracle.GATE_NONSAFE])
def test_chunked_equals_recurrence_varlen(mode):
    c = _random_case(7, T=200, H=2, K=8, V=8, mode=mode)
    lens = [0, 70, 1, 0, 64, 33, 0]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    c["initial_state"] = np.random.default_rng(1).normal(size=(len(lens), 2, 8, 8))
    o_ref, s_ref = oracle.forward(**c, cu_seqlens=cu)
    for C in (32, 64):
        o, s = chunked.forward(**c, cu_seqlens=cu, chunk_size=C)
        valid = slice(0, int(cu[-1]))
        assert np.allclose(o[:, valid], o_ref[:, valid], atol=1e-11)
        assert np.allclose(s, s_ref, atol=1e-11)


def test_intermediates_properties():
    c = _random_case(11, T=64, H=1, K=16, V=8)
    a = chunked.gate_act(c["g"][0, :, 0], c["A_log"][0], c["dt_bias"][0], c["mode"], -5.0)
    rec = chunked.chunk_unit(c["q"][0, :, 0], c["k"][0, :, 0], c["v"][0, :, 0], a,
                             c["beta"][0, :, 0], c["initial_state"][0, 0], 32)
    for Akk, Aqk, T, G in zip(rec["Akk"], rec["Aqk"], rec["T"], rec["G"]):
        n = Akk.shape[0]
        assert np.allclose(np.triu(Akk), 0)  # strictly lower
        assert np.allclose(np.triu(Aqk, 1), 0)  # lower, diagonal included
        assert np.allclose((np.eye(n) + Akk) @ T, np.eye(n), atol=1e-12)
        assert np.allclose(np.triu(T, 1), 0) and np.allclose(np.diag(T), 1)  # unit lower
        assert (np.diff(G, axis=0) <= 0).all()  # monotone non-increasing cumulative decay
    # diagonal of Aqk is s * q_i . k_i (the decay factor is 2^0 there)
    q, k = c["q"][0, :32, 0], c["k"][0, :32, 0]
    assert np.allclose(np.diag(rec["Aqk"][0]), (q * k).sum(-1) / math.sqrt(16))
