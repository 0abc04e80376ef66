"""CPU float64 oracle for the Kimi Delta Attention (KDA) forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product package
(``chunked_kda_gb300``) never imports it and shares no code with it.

Two independent restatements live here:

* ``kda_oracle.c`` (loaded through ctypes): the token-by-token float64
  recurrence, the definition every result is checked against.
* ``chunked.py``: a float64 numpy restatement of the chunked (WY) form that
  exposes the per-chunk intermediates (G, Akk, Aqk, (I+Akk)^-1, w, u, v_new,
  h).  It is pinned to the recurrence by brute force on small inputs.

Inputs are taken exactly as the GPU sees them: bf16 or fp32 values widened to
float64 before the call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_libs = {}

GATE_PRE = 0
GATE_SAFE = 1
GATE_NONSAFE = 2  # -exp(A_log) * softplus(g + dt_bias)
GATE_LOG2 = 3     # the recurrent entry point's per-token log2 decay


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the C oracle with gcc (OpenMP when available). Returns the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", out, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return out


def load(path: str | None = None):
    """ctypes handle of the oracle library (the built one, or another build of the source)."""
    with _lock:
        key = path or _LIB
        if key not in _libs:
            lib = ctypes.CDLL(path or build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.kda_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_double,
                                           dp, dp, dp, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp,
                                           ctypes.c_double, ctypes.c_double, ctypes.c_int, ip,
                                           ctypes.c_int, ctypes.c_int]
            lib.kda_oracle_fwd.restype = ctypes.c_int
            lib.kda_oracle_gate.argtypes = [dp, dp, dp, ctypes.c_int, ctypes.c_double, ip,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, dp]
            lib.kda_oracle_gate.restype = ctypes.c_int
            lib.kda_oracle_gate_act.argtypes = [ctypes.c_double] * 3 + [ctypes.c_int, ctypes.c_double]
            lib.kda_oracle_gate_act.restype = ctypes.c_double
            lib.kda_oracle_max_threads.argtypes = []
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            _libs[key] = lib
    return _libs[key]


def _load(lib=None):
    return lib if lib is not None else load()


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly (bf16 -> fp32 -> f64 is exact)
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def max_threads(lib=None) -> int:
    return int(_load(lib).kda_oracle_max_threads())


def gate_act(g: float, A_log: float, dt_bias: float, mode: int, lb: float, lib=None) -> float:
    """Scalar gate activation in natural-log units (FLA skill "fla-kda", "Gate modes")."""
    return float(_load(lib).kda_oracle_gate_act(g, A_log, dt_bias, mode, lb))


def gate(g, A_log=None, dt_bias=None, mode=GATE_SAFE, lower_bound=-5.0, cu_seqlens=None,
         chunk_size=64, lib=None):
    """Chunk-local cumulative gate in log2 units, [B, T, H, K] float64.

    Positions outside every sequence are returned as NaN (the oracle does not
    write them).
    """
    g = _f64(g)
    B, T, H, K = g.shape
    cu = _i32(cu_seqlens)
    out = np.full(g.shape, np.nan, dtype=np.float64)
    al, db = _f64(A_log), _f64(dt_bias)
    n_seqs = 0 if cu is None else len(cu) - 1
    rc = _load(lib).kda_oracle_gate(_dptr(g), _dptr(al), _dptr(db), int(mode), float(lower_bound),
                                 _iptr(cu), n_seqs, B, T, H, K, int(chunk_size), _dptr(out))
    if rc != 0:
        raise ValueError(f"kda_oracle_gate failed ({rc})")
    return out


Q_L2NORM_EPS = 1e-6  # eps floor of the optional query l2 normalisation


def forward(q, k, v, g, beta, A_log=None, dt_bias=None, mode=GATE_SAFE, lower_bound=-5.0,
            initial_state=None, cu_seqlens=None, units=None, nthreads=0, lib=None,
            q_l2norm=False, k_l2norm=False, beta_logits=False):
    """Token-by-token float64 KDA forward.

    ``q_l2norm``: each query row is first replaced by q / sqrt(sum q^2 + Q_L2NORM_EPS)
    (attention-gym PR #345 "Fuse q l2norm into the chunk_kda output kernel"); ``k_l2norm``
    the same for the key rows; ``beta_logits``: beta holds logits, sigmoid(beta) is used
    (the decode-side preprocessing of the recurrent path).
    Returns (o [B,T,H,V] float64, final_state [N,H,K,V] float64).  Rows of o
    outside every sequence (and rows of units not listed in ``units``) are NaN.
    """
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    B, T, Hk, K = q.shape
    H = v.shape[2]  # value heads; the query / key heads Hk divide them
    V = v.shape[-1]
    cu = _i32(cu_seqlens)
    N = B if cu is None else len(cu) - 1
    S0 = _f64(initial_state)
    ST = np.full((N, H, K, V), np.nan, dtype=np.float64)
    o = np.full((B, T, H, V), np.nan, dtype=np.float64)
    al, db = _f64(A_log), _f64(dt_bias)
    un = None
    if units is not None:
        un = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    rc = _load(lib).kda_oracle_fwd(_dptr(q), _dptr(k), _dptr(v), _dptr(g), _dptr(al), _dptr(db),
                                int(mode), float(lower_bound), _dptr(beta), _dptr(S0), _dptr(ST),
                                _iptr(cu), 0 if cu is None else N, B, T, H, Hk, K, V, _dptr(o),
                                float(Q_L2NORM_EPS if q_l2norm else -1.0),
                                float(Q_L2NORM_EPS if k_l2norm else -1.0), int(bool(beta_logits)),
                                _iptr(un), 0 if un is None else un.shape[0], int(nthreads))
    if rc != 0:
        raise ValueError(f"kda_oracle_fwd failed ({rc})")
    return o, ST
