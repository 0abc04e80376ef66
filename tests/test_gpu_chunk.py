"""kda_chunk_fwd (C ABI, through the binding) against the float64 oracle, element by
element on small inputs spanning several chunks and ragged tails, and on sampled
(sequence, head) units of the full-size workloads."""
import math

import numpy as np
import pytest
import torch

import oracle
from chunked_kda_gb300 import workloads
from parity import check_o, check_state, check_units, to_device, valid_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def kda():
    import chunked_kda_gb300

    return chunked_kda_gb300


def run_gpu(w, **kw):
    t = to_device(w)
    args = dict(A_log=t["A_log"], dt_bias=t["dt_bias"], mode=w.mode, lower_bound=w.lower_bound,
                initial_state=t["initial_state"], output_final_state=True,
                cu_seqlens=t["cu_seqlens"], chunk_size=w.chunk_size)
    args.update(kw)
    o, st = kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], **args)
    torch.cuda.synchronize()
    return o, st


def run_oracle(w):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, w.mode, w.lower_bound,
                          w.initial_state, w.cu_seqlens)


def compare(w, o, st):
    o_ref, s_ref = run_oracle(w)
    check_o(o, o_ref, w.q.dtype, valid_mask(w))
    if st is not None:
        check_state(st, s_ref, w.q.dtype)


def test_tiny_fp32_workload():
    w = workloads.make("tiny_fp32_b1_t128_h2_d64")
    o, st = run_gpu(w)
    compare(w, o, st)


@pytest.mark.parametrize("dtype,o_dtype", [(torch.float32, None), (torch.bfloat16, None),
                                           (torch.bfloat16, torch.float32)],
                         ids=["f32", "bf16", "bf16-f32out"])
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("T", [1, 17, 64, 65, 130, 200])
@pytest.mark.parametrize("D", [64, 128])
def test_dense_small(dtype, o_dtype, C, T, D):
    w = workloads.make_dense("t", 2, T, 2, D, D, C, dtype, 11 + T + D, state_std=0.05)
    o, st = run_gpu(w, o_dtype=o_dtype)
    assert o.dtype == (o_dtype or dtype)
    compare(w, o, st)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("K,V", [(256, 256), (64, 128), (256, 64)])
def test_dense_head_dims(dtype, K, V):
    w = workloads.make_dense("t", 1, 97, 2, K, V, 64, dtype, 5 + K + V, state_std=0.05)
    o, st = run_gpu(w)
    compare(w, o, st)


# bf16 inputs with the output in bf16 (checked under the bf16-storage allowance) and in float32
# (held to the plain max-abs bound), and float32 inputs
DTYPES_OUT = [(torch.float32, None), (torch.bfloat16, None), (torch.bfloat16, torch.float32)]
DTYPES_OUT_IDS = ["f32", "bf16", "bf16-f32out"]


@pytest.mark.parametrize("dtype,o_dtype", DTYPES_OUT, ids=DTYPES_OUT_IDS)
@pytest.mark.parametrize("C", [32, 64])
def test_pre_gated(dtype, o_dtype, C):
    w = workloads.make_dense("t", 2, 150, 2, 128, 128, C, dtype, 21, state_std=0.05,
                             mode=workloads.GATE_PRE)
    o, st = run_gpu(w, o_dtype=o_dtype)
    assert o.dtype == (o_dtype or dtype)
    compare(w, o, st)


@pytest.mark.parametrize("o_dtype", [None, torch.float32], ids=["bf16out", "f32out"])
@pytest.mark.parametrize("lb,g_std", [(-5.0, 10.0), (-0.01, 1.0), (-1e-4, 3.0), (-5.0, 0.01)])
def test_gate_extremes(lb, g_std, o_dtype):
    """lb = -5 with large +-(g + dt_bias), lb close to 0, long cumulative decay
    (FLA skill "fla-kda", correctness checklist: gate numerical extremes)."""
    w = workloads.make_dense("t", 1, 300, 2, 128, 128, 64, torch.bfloat16, 31, g_std=g_std,
                             state_std=0.05, lower_bound=lb)
    w.A_log = w.A_log * 3.0  # exp(A_log) up to 4096: saturates the sigmoid
    o, st = run_gpu(w, o_dtype=o_dtype)
    compare(w, o, st)


@pytest.mark.parametrize("mode", [workloads.GATE_PRE, workloads.GATE_SAFE], ids=["pre", "safe"])
@pytest.mark.parametrize("T", [64, 150])
def test_float32_gate_with_bf16_inputs(mode, T):
    """bf16 q, k, v, beta with a float32 gate: the fused kernel reads g from global memory
    instead of a bf16 TMA tile.  A float32 gate holding the bf16 gate's values gives the
    same activations, so the results are bitwise those of the bf16-gate call (and match
    the oracle)."""
    w = workloads.make_dense("t", 2, T, 2, 128, 128, 64, torch.bfloat16, 23, state_std=0.05,
                             mode=mode)
    o16, st16 = run_gpu(w)
    w.g = w.g.float()
    o32, st32 = run_gpu(w)
    assert torch.equal(o32, o16) and torch.equal(st32, st16)
    compare(w, o32, st32)


def test_float32_gate_varlen():
    cap = sum([0, 37, 64, 1, 0, 130]) + 23
    w = workloads.make_varlen("t", [0, 37, 64, 1, 0, 130], cap, 2, 128, 128, 64, torch.bfloat16,
                              43, mode=workloads.GATE_SAFE)
    o16, st16 = run_gpu(w)
    w.g = w.g.float()
    o32, st32 = run_gpu(w)
    end = int(w.cu_seqlens[-1])
    assert torch.equal(o32[:, :end], o16[:, :end]) and torch.equal(st32, st16)
    compare(w, o32, st32)


VARLEN_LENGTHS = [0, 37, 64, 1, 0, 0, 130, 65, 16, 0]


@pytest.mark.parametrize("dtype,o_dtype", DTYPES_OUT, ids=DTYPES_OUT_IDS)
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("mode", [workloads.GATE_PRE, workloads.GATE_SAFE, workloads.GATE_NONSAFE],
                         ids=["pre", "safe", "nonsafe"])
def test_varlen_contract(dtype, o_dtype, C, mode):
    """Packed sequences with empty slots (first, interior, consecutive, last) and a
    NaN-poisoned capacity tail (attention-gym PR #317, Agent note)."""
    cap = sum(VARLEN_LENGTHS) + 23
    w = workloads.make_varlen("t", VARLEN_LENGTHS, cap, 2, 128, 128, C, dtype, 41, mode=mode)
    t = to_device(w)
    sentinel = torch.full((1, cap, 2, 128), 12345.0, device="cuda", dtype=o_dtype or dtype)
    o, st = run_gpu(w, o=sentinel)
    compare(w, o, st)
    end = int(w.cu_seqlens[-1])
    # the tail beyond the last offset is not written (bitwise)
    assert torch.equal(o[:, end:], torch.full_like(o[:, end:], 12345.0))
    # empty slots pass their state through bit for bit
    for n, L in enumerate(VARLEN_LENGTHS):
        if L == 0:
            assert torch.equal(st[n], t["initial_state"][n])
    # each packed sequence equals the same sequence run alone (same chunk alignment)
    cu = w.cu_seqlens.tolist()
    for n, L in enumerate(VARLEN_LENGTHS):
        if L == 0:
            continue
        sl = slice(cu[n], cu[n + 1])
        wd = workloads.Workload("d", 1, L, 2, 128, 128, C, mode, w.lower_bound,
                                w.q[:, sl].contiguous(), w.k[:, sl].contiguous(),
                                w.v[:, sl].contiguous(), w.g[:, sl].contiguous(),
                                w.beta[:, sl].contiguous(), w.A_log, w.dt_bias,
                                w.initial_state[n:n + 1].contiguous())
        od, sd = run_gpu(wd, o_dtype=o_dtype)
        assert torch.equal(od[0], o[0, sl]), f"sequence {n}: packed != alone"
        assert torch.equal(sd[0], st[n])


# lengths crossing 32-token boundaries (31, 32, 33, 63, 65, 95, 97) and a packed tail
C32_LENGTHS = [31, 0, 32, 33, 63, 65, 95, 97, 1]


@pytest.mark.parametrize("mode", [workloads.GATE_PRE, workloads.GATE_SAFE], ids=["pre", "safe"])
def test_chunk_size_32_on_the_fused_path(mode):
    """Helion PR #3290: chunk sizes 32 and 64.  The chunked form computes the same function for
    every chunk size (the chunk size only blocks the recurrence; the oracle pins C = 1, 16, 32,
    64 against the token recurrence), and the bf16 tensor-core path runs chunk_size = 32 as
    64-token chunks.  Pinned here: on sequences crossing 32-token boundaries, packed and dense,
    chunk_size = 32 and 64 give bitwise the same o and final state on that path, both within
    the tolerance of the oracle."""
    cap = sum(C32_LENGTHS) + 9
    w = workloads.make_varlen("t", C32_LENGTHS, cap, 2, 128, 128, 32, torch.bfloat16, 71, mode=mode)
    assert kda().kda_chunk_fwd_launches(torch.bfloat16, 1, cap, 2, 128, 128, 32, len(C32_LENGTHS),
                                        mode) == 1
    o32, s32 = run_gpu(w, o_dtype=torch.float32)
    o64, s64 = run_gpu(w, o_dtype=torch.float32, chunk_size=64)
    end = int(w.cu_seqlens[-1])
    assert torch.equal(o32[:, :end], o64[:, :end]) and torch.equal(s32, s64)
    compare(w, o32, s32)
    wd = workloads.make_dense("t", 2, 97, 2, 128, 128, 32, torch.bfloat16, 72, state_std=0.05,
                              mode=mode)
    a, sa = run_gpu(wd)
    b, sb = run_gpu(wd, chunk_size=64)
    assert torch.equal(a, b) and torch.equal(sa, sb)
    compare(wd, a, sa)


def test_no_initial_state_equals_zeros_and_no_final_state():
    w = workloads.make_dense("t", 2, 100, 2, 128, 128, 64, torch.bfloat16, 51)
    o1, s1 = run_gpu(w)
    t = to_device(w)
    zeros = torch.zeros((2, 2, 128, 128), device="cuda")
    o2, s2 = run_gpu(w, initial_state=zeros)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    o3, s3 = run_gpu(w, output_final_state=False)
    assert s3 is None and torch.equal(o1, o3)


def test_final_state_in_place():
    w = workloads.make_dense("t", 2, 100, 2, 128, 128, 64, torch.bfloat16, 52, state_std=0.05)
    o1, s1 = run_gpu(w)
    t = to_device(w)
    S = t["initial_state"].clone()
    o2, _ = kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"],
                                t["dt_bias"], w.mode, w.lower_bound, S, True, None, 64,
                                final_state=S)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, S)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_linear_in_v_and_state_exactly(dtype):
    """(v, S0) -> (o, S_T) is linear, and scaling by 2 is exact in floating point."""
    w = workloads.make_dense("t", 1, 130, 2, 128, 128, 64, dtype, 53, state_std=0.05)
    o1, s1 = run_gpu(w)
    w.v = (w.v.float() * 2).to(dtype)
    w.initial_state = w.initial_state * 2
    o2, s2 = run_gpu(w)
    assert torch.equal(o2.float(), 2 * o1.float()) and torch.equal(s2, 2 * s1)


def test_state_carry():
    """Two calls chained through the state equal one call (within tolerance: the chunk
    boundaries differ)."""
    w = workloads.make_dense("t", 1, 200, 2, 128, 128, 64, torch.bfloat16, 54, state_std=0.05)
    o, st = run_gpu(w)
    t1 = 77
    parts = []
    S = w.initial_state
    for sl in (slice(0, t1), slice(t1, 200)):
        wp = workloads.Workload("p", 1, sl.stop - sl.start, 2, 128, 128, 64, w.mode,
                                w.lower_bound, w.q[:, sl].contiguous(), w.k[:, sl].contiguous(),
                                w.v[:, sl].contiguous(), w.g[:, sl].contiguous(),
                                w.beta[:, sl].contiguous(), w.A_log, w.dt_bias, S)
        op, sp = run_gpu(wp)
        parts.append(op)
        S = sp.cpu()
    oc = torch.cat(parts, dim=1)
    o_ref, s_ref = run_oracle(w)
    check_o(oc, o_ref, torch.bfloat16)
    check_state(S, s_ref, torch.bfloat16)


def _sample_units(w, k=4, seed=0):
    r = np.random.default_rng(seed)
    N = w.n_seqs
    units = {(0, 0), (N - 1, w.H - 1)}
    while len(units) < k:
        units.add((int(r.integers(N)), int(r.integers(w.H))))
    if w.cu_seqlens is not None:
        cu = w.cu_seqlens.tolist()
        units = {(n, h) for n, h in units if cu[n + 1] > cu[n]} | {
            (n, 0) for n in range(N) if cu[n + 1] == cu[n]}
    return sorted(units)


@pytest.mark.parametrize("name", ["dense_bf16_b4_t2048_h16_d128",
                                  "varlen_bf16_n16_cap20480_h32_d128_c32",
                                  "dense_bf16_b1_t8192_h96_d128",
                                  "dense_bf16_b4_t4096_h64_d128",
                                  "dense_bf16_b8_t2048_h32_d256",
                                  "dense_bf16_b4_t4096_h64_d128_nonsafe"])
def test_full_size_sampled(name):
    """The full workloads, in the configuration bench.py times (bf16 o), and with a
    float32 o, checked on sampled (sequence, head) units the oracle computes one by one."""
    w = workloads.make(name, device="cpu")
    units = _sample_units(w)
    for o_dtype in (None, torch.float32):
        o, st = run_gpu(w, o_dtype=o_dtype)
        assert torch.isfinite(o[torch.from_numpy(valid_mask(w)).cuda()]).all()
        check_units(w, o, st, units)
        del o, st


@pytest.mark.parametrize("dtype,o_dtype", DTYPES_OUT, ids=DTYPES_OUT_IDS)
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("g_std", [1.0, 30.0], ids=["g1", "g30"])
def test_nonsafe_gate(dtype, o_dtype, C, g_std):
    """The non-safe in-kernel gate -exp(A_log) softplus(g + dt_bias) (FLA skill "fla-kda",
    "Gate modes"): with raw g ~ N(0, 30) single tokens decay by e^-1000 and more; the result
    stays finite and matches the oracle.  bf16 runs the fused kernel (first-row anchors off the
    diagonal, per-pair factors on the diagonal 16 x 16 blocks), float32 the stage path."""
    w = workloads.make_dense("t", 2, 150, 2, 128, 128, C, dtype, 300 + C, state_std=0.05,
                             g_std=g_std, mode=workloads.GATE_NONSAFE)
    want = 1 if dtype == torch.bfloat16 else 6
    assert kda().kda_chunk_fwd_launches(dtype, 2, 150, 2, 128, 128, C, 0, workloads.GATE_NONSAFE,
                                        o_dtype) == want
    o, st = run_gpu(w, o_dtype=o_dtype)
    assert torch.isfinite(o).all() and torch.isfinite(st).all()
    compare(w, o, st)


def test_nonsafe_gate_varlen():
    lens = workloads.varlen_lengths(6, 200, 1000, empty_slots=(1,), seed=31)
    w = workloads.make_varlen("t", lens, 1100, 2, 128, 128, 64, torch.bfloat16, 31,
                              mode=workloads.GATE_NONSAFE)
    o, st = run_gpu(w)
    compare(w, o, st)


def grouped(w, hk):
    """Keep the first hk query / key heads: value head h then reads head h / (H / hk)."""
    w.q = w.q[:, :, :hk].contiguous()
    w.k = w.k[:, :, :hk].contiguous()
    return w


@pytest.mark.parametrize("dtype,C", [(torch.bfloat16, 64), (torch.bfloat16, 32), (torch.float32, 64)],
                         ids=["fused", "stagewise-c32", "stagewise-f32"])
@pytest.mark.parametrize("hk", [1, 2])
@pytest.mark.parametrize("o_dtype", [None, torch.float32], ids=["out-in-dtype", "f32out"])
def test_grouped_value_heads(dtype, C, hk, o_dtype):
    """GVA (FLA skill "fla-kda", "Correctness checklist": HV > H): 4 value heads over 1 or 2
    query / key heads, against the oracle, and equal to the multi-head call on q and k with
    their heads repeated."""
    w = grouped(workloads.make_dense("t", 2, 130, 4, 128, 128, C, dtype, 600 + C + hk,
                                     state_std=0.05), hk)
    o, st = run_gpu(w, o_dtype=o_dtype)
    compare(w, o, st)
    t = to_device(w)
    r = 4 // hk
    q4 = t["q"].repeat_interleave(r, dim=2)
    k4 = t["k"].repeat_interleave(r, dim=2)
    o2, st2 = kda().kda_chunk_fwd(q4, k4, t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                                  w.mode, w.lower_bound, t["initial_state"], True, None, C,
                                  o_dtype=o_dtype)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(st, st2)


# ---- degenerate inputs and a long sequence

@pytest.mark.parametrize("dtype,o_dtype", DTYPES_OUT, ids=DTYPES_OUT_IDS)
def test_beta_zero_reads_the_decayed_state(dtype, o_dtype):
    """beta = 0: the state is only decayed, o_t = S_t^T q_t / sqrt(K) with S_t the initial state
    decayed through token t (a closed form; the oracle pins the same case)."""
    w = workloads.make_dense("t", 1, 70, 2, 128, 128, 64, dtype, 801, state_std=0.05,
                             mode=workloads.GATE_PRE)
    w.beta = torch.zeros_like(w.beta)
    w.g = (w.g.float() * 0.02).to(dtype)  # decay mild enough that S_0 is still visible at the end
    o, st = run_gpu(w, o_dtype=o_dtype)
    a = w.g.double()[0].cumsum(0)                       # [T, H, K] natural-log decay so far
    S0 = w.initial_state.double()[0]                    # [H, K, V]
    q = w.q.double()[0]                                 # [T, H, K]
    ref = torch.einsum("thk,hkv->thv", q * torch.exp(a), S0) / math.sqrt(128)
    check_o(o, ref.unsqueeze(0).numpy(), dtype)
    check_state(st, (torch.exp(a[-1])[..., None] * S0).unsqueeze(0).numpy(), dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_zero_queries_and_single_tokens(dtype):
    """All-zero query rows give zero output rows exactly; sequences of one token match the
    oracle (the chunk is one valid row and 63 masked ones)."""
    w = workloads.make_dense("t", 3, 1, 2, 128, 128, 64, dtype, 802, state_std=0.05)
    o, st = run_gpu(w)
    compare(w, o, st)
    w2 = workloads.make_dense("t", 1, 90, 2, 128, 128, 64, dtype, 803, state_std=0.05)
    w2.q[:, 10:30] = 0
    o2, _ = run_gpu(w2)
    assert (o2[:, 10:30] == 0).all()


@pytest.mark.slow
def test_long_sequence_carry_is_bitwise():
    """2^17 tokens through the fused kernel: the first 4096 outputs against the oracle, and
    two calls split at a chunk boundary and chained through the state equal one call bit
    for bit (the chunks, hence the arithmetic, are the same)."""
    T, H = 1 << 17, 2
    w = workloads.make_dense("t", 1, T, H, 128, 128, 64, torch.bfloat16, 804, state_std=0.05)
    o, st = run_gpu(w)
    n = 4096
    wp = workloads.Workload("p", 1, n, H, 128, 128, 64, w.mode, w.lower_bound, w.q[:, :n],
                            w.k[:, :n], w.v[:, :n], w.g[:, :n], w.beta[:, :n], w.A_log,
                            w.dt_bias, w.initial_state)
    o_ref, _ = run_oracle(wp)
    check_o(o[:, :n], o_ref, torch.bfloat16)
    t1 = 64 * 1000
    S = w.initial_state
    outs = []
    for sl in (slice(0, t1), slice(t1, T)):
        ws = workloads.Workload("p", 1, sl.stop - sl.start, H, 128, 128, 64, w.mode,
                                w.lower_bound, w.q[:, sl].contiguous(), w.k[:, sl].contiguous(),
                                w.v[:, sl].contiguous(), w.g[:, sl].contiguous(),
                                w.beta[:, sl].contiguous(), w.A_log, w.dt_bias, S)
        op, sp = run_gpu(ws)
        outs.append(op)
        S = sp.cpu()
    assert torch.equal(torch.cat(outs, dim=1), o) and torch.equal(S.cuda(), st)
