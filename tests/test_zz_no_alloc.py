"""kda_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate device
memory (for instance a plugin that only receives input and output pointers from a host
framework that owns all device memory).  It runs on the library's fixed scratch array
instead of a workspace.

Checked here against the float64 oracle on several calls in a row with different sizes, so
that a call never depends on what the previous one left in the shared array; against
kda_chunk_fwd bit for bit where that call takes the same stage-by-stage kernels (float32
inputs, head dims other than 128); and across a cudaDeviceReset in a separate process, after
which the array lives at a new device address.  This file is collected last on purpose."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from chunked_kda_gb300 import workloads
from parity import check_o, check_state, to_device, valid_mask

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_kda_gb300

    return chunked_kda_gb300


def _run_noalloc(kda, w):
    t = to_device(w)
    o = torch.full((w.B, w.T, w.H, w.V), 777.0, device="cuda", dtype=w.q.dtype)
    st = torch.full((w.n_seqs, w.H, w.K, w.V), 777.0, device="cuda")
    kda.kda_chunk_fwd_noalloc(t["q"], t["k"], t["v"], t["g"], t["beta"], A_log=t["A_log"],
                              dt_bias=t["dt_bias"], mode=w.mode, lower_bound=w.lower_bound,
                              initial_state=t["initial_state"], cu_seqlens=t["cu_seqlens"],
                              chunk_size=w.chunk_size, o=o, final_state=st)
    torch.cuda.synchronize()
    return o, st


def _run_with_workspace(kda, w):
    t = to_device(w)
    o, st = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], A_log=t["A_log"],
                              dt_bias=t["dt_bias"], mode=w.mode, lower_bound=w.lower_bound,
                              initial_state=t["initial_state"], output_final_state=True,
                              cu_seqlens=t["cu_seqlens"], chunk_size=w.chunk_size)
    torch.cuda.synchronize()
    return o, st


def _against_oracle(w, o, st):
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, w.mode,
                                  w.lower_bound, w.initial_state, w.cu_seqlens)
    check_o(o, o_ref, w.q.dtype, valid_mask(w), what=f"o {w.name}")
    check_state(st, s_ref, w.q.dtype, what=f"state {w.name}")
    if w.cu_seqlens is not None:  # the capacity tail is not written
        end = int(w.cu_seqlens[-1])
        assert torch.equal(o[:, end:], torch.full_like(o[:, end:], 777.0))


def _cases():
    # float32 and bf16 inputs, dense and packed with empty slots, different sizes per call
    yield workloads.make_dense("a", 1, 128, 2, 64, 64, 64, torch.float32, 501, state_std=0.05)
    yield workloads.make_varlen("b", [0, 70, 1, 0, 100], 200, 2, 128, 128, 32, torch.bfloat16, 502)
    yield workloads.make_dense("c", 2, 300, 2, 128, 128, 64, torch.bfloat16, 503, state_std=0.05)
    yield workloads.make_dense("d", 1, 97, 2, 256, 64, 32, torch.float32, 504, state_std=0.05)
    yield workloads.make_dense("a", 1, 128, 2, 64, 64, 64, torch.float32, 501, state_std=0.05)


def _same_kernels_as_kda_chunk_fwd(w):
    """kda_chunk_fwd runs the same stage-by-stage kernels for these inputs (it takes the fused
    tensor-core kernel only for bf16 with K = V = 128 and a bounded gate)."""
    return w.q.dtype == torch.float32 or w.K != 128 or w.V != 128


def test_noalloc_matches_the_oracle_on_consecutive_calls(kda):
    for w in _cases():
        o, st = _run_noalloc(kda, w)
        _against_oracle(w, o, st)
        if _same_kernels_as_kda_chunk_fwd(w):
            o2, st2 = _run_with_workspace(kda, w)
            m = torch.from_numpy(valid_mask(w)).cuda()
            assert torch.equal(o[m], o2[m]) and torch.equal(st, st2), w.name


def test_noalloc_repeat_after_a_larger_call_is_bitwise_the_same(kda):
    """A float32 call, a call of other sizes that writes more of the shared array, and the
    first call again: the two results of the first call are bitwise equal (nothing depends on
    what the array held) and both match the oracle at rel-L2 <= 1e-4."""
    a = workloads.make_dense("a", 1, 150, 2, 64, 64, 64, torch.float32, 511, state_std=0.05)
    big = workloads.make_dense("big", 2, 400, 3, 128, 64, 32, torch.float32, 512, state_std=0.05)
    o1, s1 = _run_noalloc(kda, a)
    ob, sb = _run_noalloc(kda, big)
    o2, s2 = _run_noalloc(kda, a)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    _against_oracle(a, o1, s1)
    _against_oracle(big, ob, sb)


_RESET_SCRIPT = r"""
import ctypes, sys
import numpy as np
lib_path, npz, out = sys.argv[1:4]
lib = ctypes.CDLL(lib_path)
rt = ctypes.CDLL("libcudart.so.13")  # the runtime the library already loaded
vp = ctypes.c_void_p
d = dict(np.load(npz))
B, T, H, K, V = (int(x) for x in d["dims"])

def upload(a):
    p = vp()
    assert rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(a.nbytes)) == 0
    assert rt.cudaMemcpy(p, a.ctypes.data_as(vp), ctypes.c_size_t(a.nbytes), 1) == 0
    return p

def download(p, shape):
    a = np.empty(shape, np.float32)
    assert rt.cudaMemcpy(a.ctypes.data_as(vp), p, ctypes.c_size_t(a.nbytes), 2) == 0
    return a

lib.kda_chunk_fwd_noalloc.argtypes = [vp, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, vp,
                                      ctypes.c_int, ctypes.c_float, vp, vp, vp, vp] + \
                                     [ctypes.c_int] * 7 + [vp, ctypes.c_int, vp]
res = {}
for rep in range(2):
    p = {n: upload(np.ascontiguousarray(d[n], dtype=np.float32))
         for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0")}
    p["o"] = upload(np.zeros((B, T, H, V), np.float32))
    p["hT"] = upload(np.zeros((B, H, K, V), np.float32))
    st = lib.kda_chunk_fwd_noalloc(p["q"], p["k"], p["v"], 0, p["g"], 0, p["A_log"], p["dt_bias"],
                                   1, -5.0, p["beta"], p["h0"], p["hT"], None, 0, B, T, H, K, V,
                                   64, p["o"], 0, None)
    assert st == 0, st
    assert rt.cudaDeviceSynchronize() == 0
    res[f"o{rep}"] = download(p["o"], (B, T, H, V))
    res[f"s{rep}"] = download(p["hT"], (B, H, K, V))
    if rep == 0:
        assert rt.cudaDeviceReset() == 0  # ends this process's context only
np.savez(out, **res)
"""


def test_noalloc_after_device_reset(kda, tmp_path):
    """In a process of its own (a reset would end the test process's context): one call,
    cudaDeviceReset, then another call on newly allocated buffers.  The scratch array lives
    at a new address in the new context; both calls match the oracle and each other."""
    w = workloads.make_dense("r", 1, 150, 2, 64, 64, 64, torch.float32, 521, state_std=0.05)
    npz = tmp_path / "in.npz"
    out = tmp_path / "out.npz"
    np.savez(npz, dims=np.array([w.B, w.T, w.H, w.K, w.V]), q=w.q.numpy(), k=w.k.numpy(),
             v=w.v.numpy(), g=w.g.numpy(), beta=w.beta.numpy(), A_log=w.A_log.numpy(),
             dt_bias=w.dt_bias.numpy(), h0=w.initial_state.numpy())
    r = subprocess.run([sys.executable, "-c", _RESET_SCRIPT, kda.library_path(), str(npz),
                        str(out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    res = np.load(out)
    assert np.array_equal(res["o0"], res["o1"]) and np.array_equal(res["s0"], res["s1"])
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, w.mode,
                                  w.lower_bound, w.initial_state)
    check_o(res["o0"], o_ref, torch.float32, what="o after reset")
    check_state(torch.from_numpy(res["s1"]), s_ref, torch.float32, what="state after reset")


def test_noalloc_rejects_sizes_beyond_the_scratch(kda):
    # B=1, T=8192, H=4, K=V=128 needs about 3.8 KB per token and head, far above 16 MiB
    dev = "cuda"
    q = torch.zeros((1, 8192, 4, 128), device=dev, dtype=torch.bfloat16)
    beta = torch.zeros((1, 8192, 4), device=dev, dtype=torch.bfloat16)
    A_log = torch.zeros((4, 128), device=dev)
    o = torch.empty_like(q)
    with pytest.raises(kda.KdaError, match="KDA_NOALLOC_SCRATCH_BYTES"):
        kda.kda_chunk_fwd_noalloc(q, q, q, q, beta, A_log=A_log, o=o)
