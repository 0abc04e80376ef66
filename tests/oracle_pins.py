"""Checks that pin the float64 oracle to facts it does not itself compute.

Each ``pin_*`` function takes an oracle library handle (``lib=None`` is the
built oracle) and raises AssertionError when the oracle disagrees with:
hand-worked values (tests/golden/), closed forms the KDA recurrence reduces to
in special cases, or exact invariants of the recurrence.  The same functions
run against deliberately broken builds of the oracle source
(tests/test_oracle_mutants.py) to show that they catch plausible mistakes.

The recurrence (per head, state S in R^{K x V}, rows = key channels):
  S = Diag(exp a_t) S;  S += beta_t k_t (v_t - S^T k_t)^T;  o_t = S^T q_t / sqrt(K).
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = np.array([float(x) for x in rest.split()])
    return vals


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def pin_gate_points(lib=None):
    """Hand-derived activation values (FLA skill "fla-kda", "Gate modes")."""
    with open(os.path.join(GOLDEN, "gate_points.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            mode, g, al, db, lb, exp_, tol = line.split()
            got = oracle.gate_act(float(g), float(al), float(db), int(mode), float(lb), lib=lib)
            assert abs(got - float(exp_)) <= float(tol), (line, got)


def pin_gate_cumsum_closed_form(lib=None):
    """Pre-gated constant decay -c*ln2 per token: G_i (log2 units) = -c * (i - chunk_start + 1)
    with resets at every chunk start and every sequence start (varlen)."""
    c = 0.75
    T, H, K, C = 50, 2, 3, 16
    cu = np.array([0, 7, 7, 40], dtype=np.int32)  # an empty slot in the middle, tail 40..49
    g = np.full((1, T, H, K), -c * math.log(2.0))
    out = oracle.gate(g, mode=oracle.GATE_PRE, cu_seqlens=cu, chunk_size=C, lib=lib)
    for n in range(3):
        for t in range(cu[n], cu[n + 1]):
            want = -c * ((t - cu[n]) % C + 1)
            assert np.allclose(out[0, t], want, rtol=0, atol=1e-12), (t, out[0, t], want)
    assert np.isnan(out[0, 40:]).all()  # capacity tail is not written


def pin_gate_chunk1_is_per_token(lib=None):
    """chunk_size=1 gives the per-token log2 decay, and the chunked cumulative gate is its
    running sum inside each chunk (attention-gym PR #317 Test Plan: chunk_size 1 vs 64)."""
    r = _rng(1)
    T, H, K = 70, 2, 4
    g = r.normal(size=(1, T, H, K))
    al = r.uniform(0, math.log(16), size=(H, K))
    db = r.normal(0, 0.5, size=(H, K))
    one = oracle.gate(g, al, db, oracle.GATE_SAFE, -5.0, chunk_size=1, lib=lib)
    big = oracle.gate(g, al, db, oracle.GATE_SAFE, -5.0, chunk_size=32, lib=lib)
    for t in range(T):
        start = (t // 32) * 32
        assert np.allclose(big[0, t], one[0, start:t + 1].sum(axis=0), atol=1e-12)
    # safe gate in natural-log units lies in [lb, 0]
    nat = one * math.log(2.0)
    assert (nat <= 0).all() and (nat >= -5.0).all()


def pin_hand_worked(lib=None):
    """Two tokens, K=V=2, worked by hand (tests/golden/hand_worked_k2_v2.txt)."""
    gv = _read_golden("hand_worked_k2_v2.txt")
    q = gv["q"].reshape(1, 2, 1, 2)
    k = gv["k"].reshape(1, 2, 1, 2)
    v = gv["v"].reshape(1, 2, 1, 2)
    g = gv["g"].reshape(1, 2, 1, 2)
    beta = gv["beta"].reshape(1, 2, 1)
    S0 = gv["S0"].reshape(1, 1, 2, 2)
    o, ST = oracle.forward(q, k, v, g, beta, mode=oracle.GATE_PRE, initial_state=S0, lib=lib)
    assert np.allclose(o.reshape(-1) * math.sqrt(2.0), gv["o_times_sqrtK"], atol=1e-14), o
    assert np.allclose(ST.reshape(-1), gv["ST"], atol=1e-14), ST


def pin_beta_zero(lib=None):
    """beta = 0: the state is only decayed, o_t = (Diag(exp(sum_{u<=t} a_u)) S0)^T q_t / sqrt(K)."""
    r = _rng(2)
    T, H, K, V = 9, 2, 4, 3
    q = r.normal(size=(1, T, H, K))
    k = r.normal(size=(1, T, H, K))
    v = r.normal(size=(1, T, H, V))
    g = -r.uniform(0.01, 2.0, size=(1, T, H, K))
    S0 = r.normal(size=(1, H, K, V))
    o, ST = oracle.forward(q, k, v, g, np.zeros((1, T, H)), mode=oracle.GATE_PRE,
                           initial_state=S0, lib=lib)
    for h in range(H):
        for t in range(T):
            dec = np.exp(g[0, :t + 1, h].sum(axis=0))
            want = (dec[:, None] * S0[0, h]).T @ q[0, t, h] / math.sqrt(K)
            assert np.allclose(o[0, t, h], want, atol=1e-12)
        assert np.allclose(ST[0, h], np.exp(g[0, :, h].sum(axis=0))[:, None] * S0[0, h],
                           atol=1e-12)


def pin_linear_attention(lib=None):
    """g = 0, beta = 1, orthonormal keys, S0 = 0: causal linear attention
    o_t = sum_{s<=t} (q_t . k_s) v_s / sqrt(K)."""
    r = _rng(3)
    T, K, V = 6, 8, 5
    Qm, _ = np.linalg.qr(r.normal(size=(K, K)))
    k = Qm[:T].reshape(1, T, 1, K)  # orthonormal rows
    q = r.normal(size=(1, T, 1, K))
    v = r.normal(size=(1, T, 1, V))
    o, _ = oracle.forward(q, k, v, np.zeros((1, T, 1, K)), np.ones((1, T, 1)),
                          mode=oracle.GATE_PRE, lib=lib)
    for t in range(T):
        want = sum((q[0, t, 0] @ k[0, s, 0]) * v[0, s, 0] for s in range(t + 1)) / math.sqrt(K)
        assert np.allclose(o[0, t, 0], want, atol=1e-12)


def pin_one_hot_gated(lib=None):
    """One-hot keys on distinct channels pi_s, S0 = 0: per-channel gated linear attention
    o_t = sum_{s<=t} beta_s q_t[pi_s] exp(sum_{s<u<=t} a_u[pi_s]) v_s / sqrt(K)."""
    r = _rng(4)
    T, K, V = 7, 8, 3
    perm = r.permutation(K)[:T]
    k = np.zeros((1, T, 1, K))
    for s in range(T):
        k[0, s, 0, perm[s]] = 1.0
    q = r.normal(size=(1, T, 1, K))
    v = r.normal(size=(1, T, 1, V))
    g = -r.uniform(0.01, 1.5, size=(1, T, 1, K))
    beta = r.uniform(0.1, 1.0, size=(1, T, 1))
    o, _ = oracle.forward(q, k, v, g, beta, mode=oracle.GATE_PRE, lib=lib)
    for t in range(T):
        want = np.zeros(V)
        for s in range(t + 1):
            c = perm[s]
            want += beta[0, s, 0] * q[0, t, 0, c] * math.exp(g[0, s + 1:t + 1, 0, c].sum()) * v[0, s, 0]
        assert np.allclose(o[0, t, 0], want / math.sqrt(K), atol=1e-12)


def pin_repeated_key_ema(lib=None):
    """The same one-hot key every token: row c of S follows
    x_t = (1 - beta_t) e^{a_t} x_{t-1} + beta_t v_t, i.e. in closed form
    x_t = prod_{u<=t}(1-beta_u)e^{a_u} x_0 + sum_{s<=t} beta_s e^{a_{s+1..t}} prod_{s<u<=t}(1-beta_u) v_s."""
    r = _rng(5)
    T, K, V, c = 8, 4, 3, 2
    k = np.zeros((1, T, 1, K))
    k[0, :, 0, c] = 1.0
    q = np.zeros((1, T, 1, K))
    q[0, :, 0, c] = 1.0
    v = r.normal(size=(1, T, 1, V))
    g = -r.uniform(0.01, 1.0, size=(1, T, 1, K))
    beta = r.uniform(0.05, 0.95, size=(1, T, 1))
    S0 = r.normal(size=(1, 1, K, V))
    o, ST = oracle.forward(q, k, v, g, beta, mode=oracle.GATE_PRE, initial_state=S0, lib=lib)
    a = g[0, :, 0, c]
    b = beta[0, :, 0]
    for t in range(T):
        lead = np.prod([(1 - b[u]) * math.exp(a[u]) for u in range(t + 1)])
        want = lead * S0[0, 0, c]
        for s in range(t + 1):
            f = b[s] * np.prod([(1 - b[u]) * math.exp(a[u]) for u in range(s + 1, t + 1)])
            want = want + f * v[0, s, 0]
        assert np.allclose(o[0, t, 0] * math.sqrt(K), want, atol=1e-12)
        if t == T - 1:
            assert np.allclose(ST[0, 0, c], want, atol=1e-12)
    # other rows only decay
    for d in range(K):
        if d != c:
            assert np.allclose(ST[0, 0, d], math.exp(g[0, :, 0, d].sum()) * S0[0, 0, d], atol=1e-12)


def pin_single_token_delta(lib=None):
    """One token with ||k|| = 1: S_1^T k = (1 - beta) S'^T k + beta v, S' = Diag(e^a) S0,
    and the read-out o = S_1^T q / sqrt(K) of the updated state."""
    r = _rng(6)
    K, V = 5, 4
    k = _unit(r.normal(size=(1, 1, 1, K)))
    q = r.normal(size=(1, 1, 1, K))
    v = r.normal(size=(1, 1, 1, V))
    g = -r.uniform(0.01, 2.0, size=(1, 1, 1, K))
    beta = np.array([[[0.3]]])
    S0 = r.normal(size=(1, 1, K, V))
    o, ST = oracle.forward(q, k, v, g, beta, mode=oracle.GATE_PRE, initial_state=S0, lib=lib)
    Sd = np.exp(g[0, 0, 0])[:, None] * S0[0, 0]
    kk = k[0, 0, 0]
    assert np.allclose(ST[0, 0].T @ kk, 0.7 * (Sd.T @ kk) + 0.3 * v[0, 0, 0], atol=1e-12)
    assert np.allclose(o[0, 0, 0], ST[0, 0].T @ q[0, 0, 0] / math.sqrt(K), atol=1e-12)
    # the update is rank one along k: S_1 - S' is parallel to k in the key dimension
    D = ST[0, 0] - Sd
    assert np.allclose(D - np.outer(kk, kk @ D), 0, atol=1e-12)


def _random_case(seed, B=1, T=20, H=2, K=6, V=5, mode=oracle.GATE_SAFE):
    r = _rng(seed)
    q = _unit(r.normal(size=(B, T, H, K)))
    k = _unit(r.normal(size=(B, T, H, K)))
    v = r.normal(size=(B, T, H, V))
    g = r.normal(size=(B, T, H, K)) if mode == oracle.GATE_SAFE else -r.uniform(
        0.01, 5, size=(B, T, H, K))
    beta = 1 / (1 + np.exp(-r.normal(size=(B, T, H))))
    al = r.uniform(0, math.log(16), size=(H, K))
    db = r.normal(0, 0.5, size=(H, K))
    S0 = r.normal(0, 0.05, size=(B, H, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=al, dt_bias=db, mode=mode,
                lower_bound=-5.0, initial_state=S0)


def pin_scale_exact(lib=None):
    """The map (v, S0) -> (o, S_T) is linear: doubling v and S0 doubles o and S_T exactly."""
    c = _random_case(7)
    o1, s1 = oracle.forward(**c, lib=lib)
    c2 = dict(c, v=2 * c["v"], initial_state=2 * c["initial_state"])
    o2, s2 = oracle.forward(**c2, lib=lib)
    assert np.array_equal(o2, 2 * o1) and np.array_equal(s2, 2 * s1)


def pin_state_carry(lib=None):
    """Splitting a sequence at t1 and feeding the first part's final state as the second
    part's initial state reproduces one call (attention-gym PR #317: initial_state /
    output_final_state)."""
    c = _random_case(8, T=23)
    o, ST = oracle.forward(**c, lib=lib)
    t1 = 9
    first = {n: (x[:, :t1] if n in ("q", "k", "v", "g", "beta") else x) for n, x in c.items()}
    second = {n: (x[:, t1:] if n in ("q", "k", "v", "g", "beta") else x) for n, x in c.items()}
    oa, Sa = oracle.forward(**first, lib=lib)
    second["initial_state"] = Sa
    ob, Sb = oracle.forward(**second, lib=lib)
    assert np.allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-12)
    assert np.allclose(Sb, ST, atol=1e-12)


def pin_varlen_contract(lib=None):
    """Packed sequences equal the same sequences run alone; a repeated offset (empty slot)
    passes its state through; the capacity tail is not written (attention-gym PR #317,
    Agent note)."""
    r = _rng(9)
    lens = [5, 0, 11, 1, 0, 7]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cap = int(cu[-1]) + 4
    H, K, V = 2, 4, 3
    q = _unit(r.normal(size=(1, cap, H, K)))
    k = _unit(r.normal(size=(1, cap, H, K)))
    v = r.normal(size=(1, cap, H, V))
    g = r.normal(size=(1, cap, H, K))
    beta = r.uniform(size=(1, cap, H))
    al = r.uniform(0, 2, size=(H, K))
    S0 = r.normal(size=(len(lens), H, K, V))
    o, ST = oracle.forward(q, k, v, g, beta, al, None, oracle.GATE_SAFE, -3.0, S0, cu, lib=lib)
    assert np.isnan(o[0, cu[-1]:]).all()
    for n, L in enumerate(lens):
        if L == 0:
            assert np.array_equal(ST[n], S0[n])
            continue
        sl = slice(cu[n], cu[n + 1])
        on, Sn = oracle.forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], al, None,
                                oracle.GATE_SAFE, -3.0, S0[n:n + 1], lib=lib)
        assert np.array_equal(on[0], o[0, sl]) and np.array_equal(Sn[0], ST[n])


def pin_q_l2norm_single_token(lib=None):
    """Query l2 normalisation (attention-gym PR #345, eps floor of the callers' l2norm): one
    token, S_1 = S' + beta k (v - S'^T k)^T with S' = Diag(e^a) S0, o = S_1^T q^ / sqrt(K),
    q^ = q / sqrt(|q|^2 + eps); the state does not see q."""
    r = _rng(10)
    K, V = 5, 4
    k = _unit(r.normal(size=(1, 1, 1, K)))
    q = 3.7 * r.normal(size=(1, 1, 1, K))
    v = r.normal(size=(1, 1, 1, V))
    g = -r.uniform(0.01, 2.0, size=(1, 1, 1, K))
    beta = np.array([[[0.6]]])
    S0 = r.normal(size=(1, 1, K, V))
    o, ST = oracle.forward(q, k, v, g, beta, mode=oracle.GATE_PRE, initial_state=S0, lib=lib,
                           q_l2norm=True)
    Sd = np.exp(g[0, 0, 0])[:, None] * S0[0, 0]
    kk, qq = k[0, 0, 0], q[0, 0, 0]
    S1 = Sd + 0.6 * np.outer(kk, v[0, 0, 0] - Sd.T @ kk)
    qh = qq / math.sqrt(qq @ qq + oracle.Q_L2NORM_EPS)
    assert np.allclose(ST[0, 0], S1, atol=1e-12)
    assert np.allclose(o[0, 0, 0], S1.T @ qh / math.sqrt(K), atol=1e-12)


def pin_q_l2norm_rows(lib=None):
    """The read-out is linear in the query row, so normalising row t scales o_t by
    1 / sqrt(|q_t|^2 + eps): rows scaled by 1e-3 .. 1e3 and all-zero rows; the final
    state is the same bit for bit."""
    c = _random_case(11, T=24)
    r = _rng(12)
    scales = 10.0 ** r.uniform(-3, 3, size=(1, 24, 2, 1))
    scales[0, 5] = 0.0  # zero query rows (both heads)
    scales[0, 17, 1] = 0.0
    c["q"] = c["q"] * scales
    o1, s1 = oracle.forward(**c, lib=lib)
    o2, s2 = oracle.forward(**c, lib=lib, q_l2norm=True)
    assert np.array_equal(s1, s2)
    ss = (c["q"] ** 2).sum(-1, keepdims=True)
    assert np.allclose(o2, o1 / np.sqrt(ss + oracle.Q_L2NORM_EPS), rtol=1e-12, atol=1e-14)
    assert (o2[0, 5] == 0).all() and (o2[0, 17, 1] == 0).all()


def pin_decode_preprocessing_single_token(lib=None):
    """Decode-side preprocessing (attention-gym PR #317; FLA skill "fla-kda", "Correctness
    checklist": raw beta logits, qk l2norm in kernel): one token with k^ = k / sqrt(|k|^2 + eps),
    q^ likewise and beta = sigmoid(x): S_1 = S' + beta k^ (v - S'^T k^)^T, o = S_1^T q^ / sqrt(K)."""
    r = _rng(13)
    K, V = 6, 3
    k = 5.0 * r.normal(size=(1, 1, 1, K))
    q = 0.2 * r.normal(size=(1, 1, 1, K))
    v = r.normal(size=(1, 1, 1, V))
    g = -r.uniform(0.01, 2.0, size=(1, 1, 1, K))
    x = np.array([[[-0.4]]])
    S0 = r.normal(size=(1, 1, K, V))
    o, ST = oracle.forward(q, k, v, g, x, mode=oracle.GATE_PRE, initial_state=S0, lib=lib,
                           q_l2norm=True, k_l2norm=True, beta_logits=True)
    eps = oracle.Q_L2NORM_EPS
    kk, qq = k[0, 0, 0], q[0, 0, 0]
    kh, qh = kk / math.sqrt(kk @ kk + eps), qq / math.sqrt(qq @ qq + eps)
    b = 1.0 / (1.0 + math.exp(0.4))
    Sd = np.exp(g[0, 0, 0])[:, None] * S0[0, 0]
    S1 = Sd + b * np.outer(kh, v[0, 0, 0] - Sd.T @ kh)
    assert np.allclose(ST[0, 0], S1, atol=1e-12)
    assert np.allclose(o[0, 0, 0], S1.T @ qh / math.sqrt(K), atol=1e-12)


def pin_k_l2norm_scale_free(lib=None):
    """With the key rows normalised, scaling every key row by any c > 0 leaves the result
    unchanged up to the eps floor: keys of norm 1e3 (eps negligible) give the same o and S_T
    as keys of norm 1e3 scaled again by 7."""
    c = _random_case(14, T=21)
    c["k"] = c["k"] * 1e3
    o1, s1 = oracle.forward(**c, lib=lib, k_l2norm=True)
    o2, s2 = oracle.forward(**dict(c, k=7.0 * c["k"]), lib=lib, k_l2norm=True)
    assert np.allclose(o1, o2, rtol=1e-9, atol=1e-12) and np.allclose(s1, s2, rtol=1e-9, atol=1e-12)
    o3, _ = oracle.forward(**c, lib=lib)  # without the option the keys of norm 1e3 blow up
    assert not np.allclose(o3, o1, atol=1e-3)


def pin_gva_is_repeated_heads(lib=None):
    """Grouped value heads (HV > H, FLA skill "fla-kda", "Correctness checklist"): with Hk
    query / key heads shared by H = 3 Hk value heads, value head h reads head h / 3, which is
    the multi-head forward on q and k with every head repeated 3 times in a row."""
    r = _rng(15)
    B, T, Hk, H, K, V = 2, 19, 2, 6, 5, 4
    q = _unit(r.normal(size=(B, T, Hk, K)))
    k = _unit(r.normal(size=(B, T, Hk, K)))
    v = r.normal(size=(B, T, H, V))
    g = r.normal(size=(B, T, H, K))
    beta = r.uniform(size=(B, T, H))
    al = r.uniform(0, 2, size=(H, K))
    S0 = r.normal(size=(B, H, K, V))
    o1, s1 = oracle.forward(q, k, v, g, beta, al, None, oracle.GATE_SAFE, -4.0, S0, lib=lib)
    q3, k3 = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    o2, s2 = oracle.forward(q3, k3, v, g, beta, al, None, oracle.GATE_SAFE, -4.0, S0, lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


ALL_PINS = [pin_gate_points, pin_gate_cumsum_closed_form, pin_gate_chunk1_is_per_token,
            pin_hand_worked, pin_beta_zero, pin_linear_attention, pin_one_hot_gated,
            pin_repeated_key_ema, pin_single_token_delta, pin_scale_exact, pin_state_carry,
            pin_varlen_contract, pin_q_l2norm_single_token, pin_q_l2norm_rows,
            pin_decode_preprocessing_single_token, pin_k_l2norm_scale_free, pin_gva_is_repeated_heads]
