"""Float64 numpy restatement of the chunked (WY / UT-transform) KDA forward.

TEST INFRASTRUCTURE ONLY (see the package docstring).  It writes out, chunk by
chunk and with no blocking or fusion, the steps the pages name, and returns
every intermediate so that a kernel can be checked stage by stage.

Steps, per (sequence, head), chunk of C tokens i, j in [0, C), G in log2 units:

  a1  G_i   = sum_{j<=i} a_j / ln 2                 chunk-local cumulative gate
      (FLA skill "fla-kda", "Safe gate numerical note": RCP_LN2 conversion
       before exp2; resets at each chunk start)
  a2  Akk[i,j] = beta_i sum_d k_i[d] k_j[d] 2^(G_i[d]-G_j[d])      j <  i
      Aqk[i,j] = s      sum_d q_i[d] k_j[d] 2^(G_i[d]-G_j[d])      j <= i
      (Helion PR #3290 "Read only the causal columns in
       chunk_fwd_A_diag_anchored": the intra-chunk score matrix is causal)
  a3  T = (I + Akk)^-1                    (FLA skill "fla-kda", "Safe gate
       numerical note": triangular solve on masked lower-triangular blocks)
  a4  w = T (beta * k * 2^G),  u = T (beta * v)
       (FLA skill "fla-kda", "Public code map": recompute_w_u_fwd)
  a5  v_new = u - w h;   h <- Diag(2^G_last) h + (k * 2^(G_last - G))^T v_new
  a6  o = s (q * 2^G) h + Aqk v_new
      (attention-gym PR #345: the output kernel's k-tile loop over q . h)

with s = 1/sqrt(K) and h the K x V state at the chunk start.  In exact
arithmetic this equals the token recurrence of ``kda_oracle.c`` for every C;
the tests check that by brute force.  float64 has the range to evaluate
2^(G_i - G_j) directly (|G| <= 64 * 5 / ln 2 < 1023 for |a| <= 5), so no
anchor offsets are needed here; the masked entries are never exponentiated.
"""
from __future__ import annotations

import math

import numpy as np

LN2 = math.log(2.0)


def gate_act(g, A_log=None, dt_bias=None, mode=1, lower_bound=-5.0):
    """Natural-log per-token decay a (FLA skill "fla-kda", "Gate modes"): 0 pre-gated,
    1 safe lb * sigmoid(exp(A_log) (g + dt_bias)), 2 non-safe -exp(A_log) softplus(g + dt_bias),
    3 a per-token log2 decay."""
    g = np.asarray(g, dtype=np.float64)
    if mode == 0:
        return g.copy()
    if mode == 3:
        return g * LN2
    x = g + (0.0 if dt_bias is None else np.asarray(dt_bias, dtype=np.float64))
    expA = np.exp(np.asarray(A_log, dtype=np.float64))
    if mode == 2:
        return -expA * np.logaddexp(0.0, x)  # softplus(x) = ln(1 + e^x)
    return lower_bound / (1.0 + np.exp(-expA * x))


def chunk_unit(q, k, v, a, beta, h0, C):
    """One (sequence, head) unit.

    q, k: [L, K]; v: [L, V]; a: [L, K] natural-log decay; beta: [L]; h0: [K, V].
    Returns dict with o [L, V], final [K, V] and per-chunk lists.
    """
    L, K = k.shape
    V = v.shape[1]
    s = 1.0 / math.sqrt(K)
    h = np.array(h0, dtype=np.float64, copy=True)
    o = np.zeros((L, V))
    rec = {k_: [] for k_ in ("G", "Akk", "Aqk", "T", "w", "u", "v_new", "h")}
    for c0 in range(0, L, C):
        c1 = min(c0 + C, L)
        n = c1 - c0
        qc, kc, vc, bc = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1]
        G = np.cumsum(a[c0:c1], axis=0) / LN2  # a1
        Akk = np.zeros((n, n))
        Aqk = np.zeros((n, n))
        for i in range(n):  # a2, causal entries only
            for j in range(i + 1):
                dec = np.exp2(G[i] - G[j])
                if j < i:
                    Akk[i, j] = bc[i] * np.sum(kc[i] * kc[j] * dec)
                Aqk[i, j] = s * np.sum(qc[i] * kc[j] * dec)
        Tm = np.linalg.inv(np.eye(n) + Akk)  # a3
        w = Tm @ (bc[:, None] * kc * np.exp2(G))  # a4
        u = Tm @ (bc[:, None] * vc)
        rec["h"].append(h.copy())
        v_new = u - w @ h  # a5
        o[c0:c1] = s * (qc * np.exp2(G)) @ h + Aqk @ v_new  # a6
        Gl = G[-1]
        h = np.exp2(Gl)[:, None] * h + (kc * np.exp2(Gl[None, :] - G)).T @ v_new
        for name, val in (("G", G), ("Akk", Akk), ("Aqk", Aqk), ("T", Tm), ("w", w), ("u", u),
                          ("v_new", v_new)):
            rec[name].append(val)
    rec["o"] = o
    rec["final"] = h
    return rec


def forward(q, k, v, g, beta, A_log=None, dt_bias=None, mode=1, lower_bound=-5.0,
            initial_state=None, cu_seqlens=None, chunk_size=64):
    """Chunked float64 forward over all units; same contract as ``oracle.forward``."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None:
        bounds = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        bounds = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    N = len(bounds)
    o = np.full((B, T, H, V), np.nan)
    ST = np.zeros((N, H, K, V))
    for n, (b, bos, eos) in enumerate(bounds):
        for hh in range(H):
            h0 = np.zeros((K, V)) if initial_state is None else np.asarray(
                initial_state[n, hh], dtype=np.float64)
            if eos == bos:
                ST[n, hh] = h0
                continue
            al = None if A_log is None else np.asarray(A_log, dtype=np.float64)[hh]
            db = None if dt_bias is None else np.asarray(dt_bias, dtype=np.float64)[hh]
            a = gate_act(g[b, bos:eos, hh], al, db, mode, lower_bound)
            rec = chunk_unit(q[b, bos:eos, hh], k[b, bos:eos, hh], v[b, bos:eos, hh], a,
                             beta[b, bos:eos, hh], h0, chunk_size)
            o[b, bos:eos, hh] = rec["o"]
            ST[n, hh] = rec["final"]
    return o, ST
