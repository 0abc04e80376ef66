"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (always against the float64 oracle on the exact quantised inputs):
  float32 inputs: rel-L2 <= 1e-4 on o and on the final state;
  bf16 inputs:    rel-L2 <= 2e-2 on o and on the final state, and
                  max |o - o_ref| <= 5e-2 * RMS(o_ref) for the forward's value.
When o is stored in bf16, the storage rounding adds up to half a bf16 ulp,
2^-8 |o|, to each element on top of the forward's own error (it is at most
2^-8 max|o|, which alone exceeds 5e-2 RMS wherever max|o| > 12.8 RMS), so a
bf16 o is held to |o - o_ref| <= 5e-2 RMS (1 + 2^-8) + 2^-8 |o_ref| element by
element; a float32 o from bf16 inputs is held to the plain bound.
"""
from __future__ import annotations

import numpy as np
import torch

F32_REL = 1e-4
BF16_REL = 2e-2
BF16_MAXABS_RMS = 5e-2


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_o(o_gpu, o_ref, dtype, mask=None, what="o", out_bf16=None):
    """Compare an output tensor (valid rows only when ``mask`` is given).

    ``dtype`` is the input dtype; ``out_bf16`` says whether o was stored in bf16
    (taken from o_gpu's dtype when o_gpu is a tensor)."""
    if out_bf16 is None:
        out_bf16 = isinstance(o_gpu, torch.Tensor) and o_gpu.dtype == torch.bfloat16
    a = to_np(o_gpu) if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu)
    b = np.asarray(o_ref)
    if mask is not None:
        a, b = a[mask], b[mask]
    assert np.isfinite(a).all(), f"{what}: non-finite values"
    e = rel_l2(a, b)
    if dtype == torch.float32:
        assert e <= F32_REL, f"{what}: rel-L2 {e:.3e} > {F32_REL}"
    else:
        assert e <= BF16_REL, f"{what}: rel-L2 {e:.3e} > {BF16_REL}"
        if what.startswith("o") and b.size:
            rms = float(np.sqrt(np.mean(b * b)))
            d = np.abs(a - b)
            if out_bf16:
                excess = float((d - 2.0 ** -8 * np.abs(b)).max())
                bound = BF16_MAXABS_RMS * rms * (1 + 2.0 ** -8)
                assert excess <= bound, (f"{what}: max(|o-o_ref| - 2^-8|o_ref|) {excess:.3e} > "
                                         f"5e-2*RMS {rms:.3e}")
            else:
                mx = float(d.max())
                assert mx <= BF16_MAXABS_RMS * rms, f"{what}: max-abs {mx:.3e} > 5e-2*RMS {rms:.3e}"
    return e


def check_state(s_gpu, s_ref, dtype, what="final_state"):
    a = to_np(s_gpu)
    assert np.isfinite(a).all(), f"{what}: non-finite values"
    e = rel_l2(a, s_ref)
    tol = F32_REL if dtype == torch.float32 else BF16_REL
    assert e <= tol, f"{what}: rel-L2 {e:.3e} > {tol}"
    return e


def to_device(w, dev="cuda"):
    return {n: (None if x is None else x.to(dev)) for n, x in w.tensors().items()}


def valid_mask(w):
    """Boolean [B, T] of rows inside some sequence."""
    m = np.zeros((w.B, w.T), dtype=bool)
    if w.cu_seqlens is None:
        m[:] = True
    else:
        m[0, :int(w.cu_seqlens[-1])] = True
    return m


def unit_slices(w, n, h):
    """(batch row, token slice) of logical sequence n."""
    if w.cu_seqlens is None:
        return n, slice(0, w.T)
    cu = w.cu_seqlens.tolist()
    return 0, slice(cu[n], cu[n + 1])


def oracle_unit(w, n, h):
    """float64 oracle output [L, V] and final state [K, V] of one (sequence, head) unit,
    computed from that unit's slice of the inputs only."""
    import oracle

    b, sl = unit_slices(w, n, h)
    hs = slice(h, h + 1)

    def cut(x):
        return x[b:b + 1, sl, hs].contiguous()

    S0 = None if w.initial_state is None else w.initial_state[n:n + 1, hs].contiguous()
    o, st = oracle.forward(cut(w.q), cut(w.k), cut(w.v), cut(w.g), cut(w.beta),
                           None if w.A_log is None else w.A_log[hs],
                           None if w.dt_bias is None else w.dt_bias[hs],
                           w.mode, w.lower_bound, S0)
    return o[0, :, 0], st[0, 0]


def check_units(w, o_gpu, st_gpu, units):
    for n, h in units:
        b, sl = unit_slices(w, n, h)
        o_ref, s_ref = oracle_unit(w, n, h)
        if o_ref.shape[0]:
            check_o(o_gpu[b, sl, h], o_ref, w.q.dtype, what=f"o[{n},{h}]")
        if st_gpu is not None:
            check_state(st_gpu[n, h], s_ref, w.q.dtype, what=f"state[{n},{h}]")
