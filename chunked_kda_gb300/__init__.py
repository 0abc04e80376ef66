"""Thin Python binding of libkda_gb300.so, the sm_103a KDA forward library.

The functions here carry the C ABI's names (include/kda.h) and only marshal
arguments: they check dtypes, devices and contiguity, allocate outputs with
torch when the caller passes none, and pass raw device pointers plus the
current CUDA stream.  Every step of the computation runs in the library's
CUDA kernels; there is no other code path, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["kda_gate_fwd", "kda_chunk_workspace_bytes", "kda_chunk_workspace_bytes_ex",
           "kda_fused_wait_timeouts", "kda_chunk_fwd_launches", "kda_test_hooks",
           "kda_chunk_fwd", "kda_chunk_fwd_ex",
           "kda_chunk_fwd_noalloc", "kda_recurrent_fwd", "KdaError", "GATE_PRE", "GATE_SAFE",
           "GATE_NONSAFE", "GATE_LOG2", "FLAG_K_L2NORM", "FLAG_BETA_LOGITS", "kda_recurrent_fwd_ex",
           "FLAG_Q_L2NORM", "NOALLOC_SCRATCH_BYTES", "library_path", "load_library"]

GATE_PRE = 0
GATE_SAFE = 1
GATE_NONSAFE = 2  # -exp(A_log) * softplus(g + dt_bias); fused kernel for bf16 K = V = 128, else stages
GATE_LOG2 = 3     # the per-token log2 decay (the recurrent entry points' gate)
NOALLOC_SCRATCH_BYTES = 16 << 20  # KDA_NOALLOC_SCRATCH_BYTES in include/kda.h
FLAG_Q_L2NORM = 1  # KDA_FLAG_Q_L2NORM
FLAG_K_L2NORM = 2  # KDA_FLAG_K_L2NORM
FLAG_BETA_LOGITS = 4  # KDA_FLAG_BETA_LOGITS
_F32, _BF16 = 0, 1
_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    """A non-OK kda_status, with the library's detail message."""

    def __init__(self, fn, status, detail):
        super().__init__(f"{fn} failed: status {status} ({detail})")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libkda_gb300.so")


def load_library():
    """Load libkda_gb300.so (built in-tree by ``_build.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -c 'import "
                               "__graft_entry__ as g; g.build()'` (needs nvcc)")
        lib = ctypes.CDLL(path)
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.kda_gate_fwd.argtypes = [vp, i32, vp, vp, i32, f32, vp, i32, i32, i32, i32, i32, i32,
                                     vp, vp]
        lib.kda_chunk_workspace_bytes.argtypes = [i32] * 8
        lib.kda_chunk_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_chunk_workspace_bytes_ex.argtypes = [i32] * 9
        lib.kda_chunk_workspace_bytes_ex.restype = ctypes.c_size_t
        lib.kda_chunk_fwd_launches.argtypes = [i32] * 10
        lib.kda_chunk_fwd_launches.restype = i32
        lib.kda_fused_wait_timeouts.argtypes = [vp, i32]
        lib.kda_fused_wait_timeouts.restype = i32
        lib.kda_chunk_fwd.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp, vp, vp,
                                      i32, i32, i32, i32, i32, i32, i32, vp, i32, vp,
                                      ctypes.c_size_t, vp]
        lib.kda_chunk_fwd_ex.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp, vp,
                                         vp, i32, i32, i32, i32, i32, i32, i32, vp, i32, vp,
                                         ctypes.c_size_t, i32, ctypes.c_uint, vp, vp]
        lib.kda_chunk_fwd_ex.restype = ctypes.c_int
        lib.kda_test_hooks.argtypes = [i32, i32, i32, i32]
        lib.kda_test_hooks.restype = i32
        lib.kda_recurrent_fwd_ex.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp, vp,
                                             vp, i32, i32, i32, i32, i32, i32, vp, i32, i32,
                                             ctypes.c_uint, vp]
        lib.kda_recurrent_fwd_ex.restype = ctypes.c_int
        lib.kda_recurrent_fwd.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                          i32, i32, vp, i32, vp]
        lib.kda_chunk_fwd_noalloc.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp,
                                              vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, i32,
                                              vp]
        lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        for fn in (lib.kda_gate_fwd, lib.kda_chunk_fwd, lib.kda_recurrent_fwd):
            fn.restype = ctypes.c_int
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_last_error.argtypes = []
        lib.kda_last_error.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _check(fn, status):
    if status != 0:
        lib = load_library()
        raise KdaError(fn, lib.kda_status_string(status).decode(), lib.kda_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dt(t, name):
    if t.dtype == torch.float32:
        return _F32
    if t.dtype == torch.bfloat16:
        return _BF16
    raise TypeError(f"{name}: dtype {t.dtype} is not float32 or bfloat16")


def _cuda(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.requires_grad:
        raise ValueError(f"{name} requires grad: this library is forward-only (inference)")
    return t


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _seqs(cu_seqlens, B):
    if cu_seqlens is None:
        return 0
    _cuda(cu_seqlens, "cu_seqlens", torch.int32)
    if B != 1:
        raise ValueError("packed mode (cu_seqlens given) needs B == 1")
    return cu_seqlens.numel() - 1


def kda_gate_fwd(g, A_log=None, dt_bias=None, mode=GATE_SAFE, lower_bound=-5.0,
                 cu_seqlens=None, chunk_size=64, out=None, stream=None):
    """Gate activation + chunk-local cumsum in log2 units; returns float32 [B, T, H, K]."""
    _cuda(g, "g")
    B, T, H, K = g.shape
    if out is None:
        out = torch.empty(g.shape, device=g.device, dtype=torch.float32)
    _cuda(out, "out", torch.float32)
    _cuda(A_log, "A_log", torch.float32)
    _cuda(dt_bias, "dt_bias", torch.float32)
    n = _seqs(cu_seqlens, B)
    lib = load_library()
    _check("kda_gate_fwd", lib.kda_gate_fwd(_ptr(g), _dt(g, "g"), _ptr(A_log), _ptr(dt_bias), mode,
                                            lower_bound, _ptr(cu_seqlens), n, B, T, H, K,
                                            chunk_size, _ptr(out), _stream(stream)))
    return out


def kda_chunk_workspace_bytes(dtype, B, T, H, K, V, chunk_size, n_seqs=0, mode=None) -> int:
    """Scratch bytes of kda_chunk_fwd; ``mode`` (a gate mode) selects kda_chunk_workspace_bytes_ex."""
    code = _F32 if dtype == torch.float32 else _BF16
    lib = load_library()
    if mode is None:
        return int(lib.kda_chunk_workspace_bytes(code, B, T, H, K, V, chunk_size, n_seqs))
    return int(lib.kda_chunk_workspace_bytes_ex(code, B, T, H, K, V, chunk_size, n_seqs, mode))


def kda_chunk_workspace_bytes_ex(dtype, B, T, H, K, V, chunk_size, n_seqs, mode) -> int:
    return kda_chunk_workspace_bytes(dtype, B, T, H, K, V, chunk_size, n_seqs, mode)


def kda_chunk_fwd_launches(dtype, B, T, H, K, V, chunk_size, n_seqs=0, mode=GATE_SAFE,
                           o_dtype=None) -> int:
    """Kernel launches of one kda_chunk_fwd call with these sizes on the current device (-1 for
    invalid sizes)."""
    code = _F32 if dtype == torch.float32 else _BF16
    ocode = code if o_dtype is None else (_F32 if o_dtype == torch.float32 else _BF16)
    lib = load_library()
    return int(lib.kda_chunk_fwd_launches(code, ocode, B, T, H, K, V, chunk_size, n_seqs, mode))


def kda_test_hooks(wait_timeout_chunk=-1, sm_count=0, one_launch=False, two_pass_d128=False) -> None:
    """The tensor-core paths' test hooks (kda_test_hooks in kda.h), process-wide; the defaults
    turn them off."""
    _check("kda_test_hooks", load_library().kda_test_hooks(int(wait_timeout_chunk), int(sm_count),
                                                           1 if one_launch else 0,
                                                           1 if two_pass_d128 else 0))


def kda_fused_wait_timeouts(reset=False) -> int:
    """Fused-kernel mbarrier waits that gave up on the current device (0 after normal runs);
    synchronises with the device."""
    lib = load_library()
    n = ctypes.c_uint(0)
    _check("kda_fused_wait_timeouts", lib.kda_fused_wait_timeouts(ctypes.byref(n), 1 if reset else 0))
    return int(n.value)


def kda_chunk_fwd(q, k, v, g, beta, A_log=None, dt_bias=None, mode=GATE_SAFE, lower_bound=-5.0,
                  initial_state=None, output_final_state=False, cu_seqlens=None, chunk_size=64,
                  o=None, final_state=None, workspace=None, stream=None, o_dtype=None,
                  q_l2norm=False, status=None):
    """Chunked KDA forward; returns (o, final_state or None).

    ``o_dtype`` is the dtype of q (default) or torch.float32.

    ``q_l2norm``: use every query row as q / sqrt(|q|^2 + 1e-6) without a separate pass
    over q (kda_chunk_fwd_ex with KDA_FLAG_Q_L2NORM); forward only.

    Grouped value heads: q and k may have fewer heads than v (a divisor of them); value
    head h then reads query / key head h / (H / Hk).

    ``status``: an int32 CUDA tensor of one element (kda_chunk_fwd_ex's status word); bit 0
    is set on the device when a fused-kernel CTA gave up a bounded wait.  The caller zeroes
    it and reads it after synchronising.

    ``final_state`` may be passed (and may be ``initial_state`` itself) to
    write the final state in place; otherwise it is allocated when
    ``output_final_state`` is true.  ``workspace`` is a uint8 CUDA tensor of at
    least ``kda_chunk_workspace_bytes`` bytes (allocated here when omitted).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _cuda(t, name)
    B, T, Hk, K = q.shape
    H, V = v.shape[2], v.shape[3]  # value heads; q, k may have fewer (grouped value heads)
    if k.shape != q.shape or H % Hk != 0:
        raise ValueError("k must have q's shape and the q/k heads must divide v's heads")
    dt = _dt(q, "q")
    if k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise TypeError("q, k, v and beta must share one dtype")
    _cuda(A_log, "A_log", torch.float32)
    _cuda(dt_bias, "dt_bias", torch.float32)
    _cuda(initial_state, "initial_state", torch.float32)
    n = _seqs(cu_seqlens, B)
    if o is None:
        o = torch.empty((B, T, H, V), device=q.device, dtype=o_dtype or q.dtype)
    _cuda(o, "o")
    if final_state is None and output_final_state:
        N = n if cu_seqlens is not None else B
        final_state = torch.empty((N, H, K, V), device=q.device, dtype=torch.float32)
    _cuda(final_state, "final_state", torch.float32)
    need = kda_chunk_workspace_bytes(q.dtype, B, T, H, K, V, chunk_size, n, mode)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load_library()
    args = (_ptr(q), _ptr(k), _ptr(v), dt, _ptr(g), _dt(g, "g"), _ptr(A_log), _ptr(dt_bias), mode,
            lower_bound, _ptr(beta), _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), n,
            B, T, H, K, V, chunk_size, _ptr(o), _dt(o, "o"), _ptr(workspace), ws_bytes)
    if status is not None:
        _cuda(status, "status", torch.int32)
        if status.numel() < 1:
            raise ValueError("status needs one int32 element")
    if q_l2norm or Hk != H or status is not None:
        _check("kda_chunk_fwd_ex", lib.kda_chunk_fwd_ex(
            *args, Hk, FLAG_Q_L2NORM if q_l2norm else 0, _ptr(status), _stream(stream)))
    else:
        _check("kda_chunk_fwd", lib.kda_chunk_fwd(*args, _stream(stream)))
    return o, final_state


def kda_chunk_fwd_ex(*args, flags=0, **kwargs):
    """kda_chunk_fwd with option bits (``FLAG_Q_L2NORM``); other arguments as kda_chunk_fwd."""
    if flags & ~FLAG_Q_L2NORM:
        raise ValueError(f"unknown flag bits {flags:#x}")
    return kda_chunk_fwd(*args, q_l2norm=bool(flags & FLAG_Q_L2NORM), **kwargs)


def kda_chunk_fwd_noalloc(q, k, v, g, beta, A_log=None, dt_bias=None, mode=GATE_SAFE,
                          lower_bound=-5.0, initial_state=None, cu_seqlens=None, chunk_size=64,
                          o=None, final_state=None, stream=None):
    """The chunked forward without a workspace, for callers that cannot allocate device
    memory: the library's fixed scratch array (NOALLOC_SCRATCH_BYTES per device) stands in
    for it.  ``o`` and ``final_state`` must be passed preallocated (so this call allocates
    nothing); ``final_state`` may be None.  Returns (o, final_state)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("o", o)):
        if t is None:
            raise ValueError(f"{name} is required")
        _cuda(t, name)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise TypeError("q, k, v and beta must share one dtype")
    _cuda(A_log, "A_log", torch.float32)
    _cuda(dt_bias, "dt_bias", torch.float32)
    _cuda(initial_state, "initial_state", torch.float32)
    _cuda(final_state, "final_state", torch.float32)
    n = _seqs(cu_seqlens, B)
    lib = load_library()
    _check("kda_chunk_fwd_noalloc", lib.kda_chunk_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _dt(q, "q"), _ptr(g), _dt(g, "g"), _ptr(A_log), _ptr(dt_bias),
        mode, lower_bound, _ptr(beta), _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens),
        n, B, T, H, K, V, chunk_size, _ptr(o), _dt(o, "o"), _stream(stream)))
    return o, final_state


def kda_recurrent_fwd(q, k, v, gate, beta, initial_state=None, output_final_state=False,
                      cu_seqlens=None, o=None, final_state=None, stream=None, o_dtype=None):
    """Token-sequential KDA forward with a per-token log2 gate; returns (o, final_state or None).

    ``final_state`` may be ``initial_state`` itself (in-place decode).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta)):
        _cuda(t, name)
    _cuda(gate, "gate", torch.float32)
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = _dt(q, "q")
    if k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise TypeError("q, k, v and beta must share one dtype")
    _cuda(initial_state, "initial_state", torch.float32)
    n = _seqs(cu_seqlens, B)
    if o is None:
        o = torch.empty((B, T, H, V), device=q.device, dtype=o_dtype or q.dtype)
    _cuda(o, "o")
    if final_state is None and output_final_state:
        N = n if cu_seqlens is not None else B
        final_state = torch.empty((N, H, K, V), device=q.device, dtype=torch.float32)
    _cuda(final_state, "final_state", torch.float32)
    lib = load_library()
    _check("kda_recurrent_fwd", lib.kda_recurrent_fwd(
        _ptr(q), _ptr(k), _ptr(v), dt, _ptr(gate), _ptr(beta), _ptr(initial_state),
        _ptr(final_state), _ptr(cu_seqlens), n, B, T, H, K, V, _ptr(o), _dt(o, "o"),
        _stream(stream)))
    return o, final_state


def kda_recurrent_fwd_ex(q, k, v, g, beta, A_log=None, dt_bias=None, mode=GATE_LOG2,
                         lower_bound=-5.0, initial_state=None, output_final_state=False,
                         cu_seqlens=None, o=None, final_state=None, stream=None, o_dtype=None,
                         flags=0):
    """Token-sequential KDA forward with the decode-side preprocessing in the kernel: ``g`` is
    read according to ``mode`` (GATE_LOG2 per-token log2 decay, GATE_PRE natural-log decay,
    GATE_SAFE / GATE_NONSAFE raw gate with A_log, dt_bias); ``flags`` combines FLAG_Q_L2NORM,
    FLAG_K_L2NORM and FLAG_BETA_LOGITS.  Returns (o, final_state or None)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        _cuda(t, name)
    B, T, Hk, K = q.shape
    H, V = v.shape[2], v.shape[3]  # value heads; q, k may have fewer (grouped value heads)
    if k.shape != q.shape or H % Hk != 0:
        raise ValueError("k must have q's shape and the q/k heads must divide v's heads")
    dt = _dt(q, "q")
    if k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise TypeError("q, k, v and beta must share one dtype")
    _cuda(A_log, "A_log", torch.float32)
    _cuda(dt_bias, "dt_bias", torch.float32)
    _cuda(initial_state, "initial_state", torch.float32)
    n = _seqs(cu_seqlens, B)
    if o is None:
        o = torch.empty((B, T, H, V), device=q.device, dtype=o_dtype or q.dtype)
    _cuda(o, "o")
    if final_state is None and output_final_state:
        N = n if cu_seqlens is not None else B
        final_state = torch.empty((N, H, K, V), device=q.device, dtype=torch.float32)
    _cuda(final_state, "final_state", torch.float32)
    lib = load_library()
    _check("kda_recurrent_fwd_ex", lib.kda_recurrent_fwd_ex(
        _ptr(q), _ptr(k), _ptr(v), dt, _ptr(g), _dt(g, "g"), _ptr(A_log), _ptr(dt_bias), mode,
        lower_bound, _ptr(beta), _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), n, B,
        T, H, K, V, _ptr(o), _dt(o, "o"), Hk, flags, _stream(stream)))
    return o, final_state
