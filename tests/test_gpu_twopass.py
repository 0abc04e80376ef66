"""The two-pass tensor-core path of kda_chunk_fwd (bf16, K in {128, 256}, V a multiple of 128):
pass 1 per (chunk, head) writes T diag(beta), Aqk and the chain's operands into the workspace,
pass 2 per (sequence, head, 128 value channels) runs the state chain.  K = V = 256 and K != V
take it by default; K = V = 128 takes it under the library's test hook (the fused kernel is the
default there).  Checked
against the float64 oracle element by element, with the varlen contract's bitwise parts, on
small inputs spanning several chunks and ragged tails."""
import contextlib

import pytest
import torch

import oracle
from chunked_kda_gb300 import workloads
from parity import check_o, check_state, to_device, valid_mask
from test_gpu_chunk import compare, grouped, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def kda():
    import chunked_kda_gb300

    return chunked_kda_gb300


@contextlib.contextmanager
def two_pass(D):
    """K = V = D on the two-pass path (a hook for D = 128, the default for D = 256)."""
    if D == 128:
        kda().kda_test_hooks(two_pass_d128=True)
    try:
        yield
    finally:
        kda().kda_test_hooks()


def _launches(w):
    n = 0 if w.cu_seqlens is None else w.n_seqs
    return kda().kda_chunk_fwd_launches(w.q.dtype, w.B, w.T, w.H, w.K, w.V, w.chunk_size, n, w.mode)


@pytest.mark.parametrize("o_dtype", [None, torch.float32], ids=["bf16out", "f32out"])
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("T", [1, 17, 64, 65, 130, 200])
@pytest.mark.parametrize("D", [128, 256])
def test_two_pass_dense_small(D, T, C, o_dtype):
    w = workloads.make_dense("t", 2, T, 2, D, D, C, torch.bfloat16, 901 + T + D, state_std=0.05)
    with two_pass(D):
        assert _launches(w) == 2
        o, st = run_gpu(w, o_dtype=o_dtype)
    compare(w, o, st)


VARLEN_LENGTHS = [0, 37, 64, 1, 0, 0, 130, 65, 16, 0]


@pytest.mark.parametrize("mode", [workloads.GATE_PRE, workloads.GATE_SAFE, workloads.GATE_NONSAFE],
                         ids=["pre", "safe", "nonsafe"])
@pytest.mark.parametrize("D", [128, 256])
def test_two_pass_varlen_contract(D, mode):
    """Packed sequences with empty slots first, interior, consecutive and last, and a
    NaN-poisoned capacity tail (attention-gym PR #317, Agent note): the tail is not written,
    empty slots pass their state through and each packed sequence equals the same sequence run
    alone, bit for bit."""
    if D == 128 and mode == workloads.GATE_NONSAFE:
        pytest.skip("K = V = 128 takes the fused kernel for the non-safe gate")
    cap = sum(VARLEN_LENGTHS) + 23
    w = workloads.make_varlen("t", VARLEN_LENGTHS, cap, 2, D, D, 64, torch.bfloat16, 941, mode=mode)
    t = to_device(w)
    with two_pass(D):
        sentinel = torch.full((1, cap, 2, D), 12345.0, device="cuda", dtype=torch.bfloat16)
        o, st = run_gpu(w, o=sentinel)
        end = int(w.cu_seqlens[-1])
        assert torch.equal(o[:, end:], torch.full_like(o[:, end:], 12345.0))
        for n, L in enumerate(VARLEN_LENGTHS):
            if L == 0:
                assert torch.equal(st[n], t["initial_state"][n])
        cu = w.cu_seqlens.tolist()
        for n, L in enumerate(VARLEN_LENGTHS):
            if L == 0:
                continue
            sl = slice(cu[n], cu[n + 1])
            wd = workloads.Workload("d", 1, L, 2, D, D, 64, mode, w.lower_bound,
                                    w.q[:, sl].contiguous(), w.k[:, sl].contiguous(),
                                    w.v[:, sl].contiguous(), w.g[:, sl].contiguous(),
                                    w.beta[:, sl].contiguous(), w.A_log, w.dt_bias,
                                    w.initial_state[n:n + 1].contiguous())
            od, sd = run_gpu(wd)
            assert torch.equal(od[0], o[0, sl]), f"sequence {n}: packed != alone"
            assert torch.equal(sd[0], st[n])
    compare(w, o, st)


@pytest.mark.parametrize("o_dtype", [None, torch.float32], ids=["bf16out", "f32out"])
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("g_std", [1.0, 30.0], ids=["g1", "g30"])
def test_two_pass_nonsafe_gate(g_std, C, o_dtype):
    """The non-safe gate -exp(A_log) softplus(g + dt_bias) (FLA skill "fla-kda", "Gate modes") on
    the K = V = 256 two-pass path: first-row anchors off the diagonal, per-pair factors on the
    diagonal 16 x 16 blocks.  With raw g ~ N(0, 30) single tokens decay by e^-1000 and more."""
    w = workloads.make_dense("t", 2, 150, 2, 256, 256, C, torch.bfloat16, 1101 + C, state_std=0.05,
                             g_std=g_std, mode=workloads.GATE_NONSAFE)
    assert _launches(w) == 2
    o, st = run_gpu(w, o_dtype=o_dtype)
    assert torch.isfinite(o).all() and torch.isfinite(st).all()
    compare(w, o, st)


@pytest.mark.parametrize("o_dtype", [None, torch.float32], ids=["bf16out", "f32out"])
@pytest.mark.parametrize("mode,g_std", [(workloads.GATE_SAFE, 1.0), (workloads.GATE_NONSAFE, 30.0)],
                         ids=["safe", "nonsafe"])
@pytest.mark.parametrize("K,V", [(128, 256), (256, 128)])
def test_two_pass_k_not_v(K, V, mode, g_std, o_dtype):
    """K != V (FLA skill "fla-kda", "Correctness checklist": D != Dv): pass 1 works on the K key
    channels, pass 2 on V / 128 value blocks with a [128 v][K] state each."""
    w = workloads.make_dense("t", 2, 150, 2, K, V, 64, torch.bfloat16, 1201 + K + V, state_std=0.05,
                             g_std=g_std, mode=mode)
    assert _launches(w) == 2
    o, st = run_gpu(w, o_dtype=o_dtype)
    compare(w, o, st)


@pytest.mark.parametrize("K,V", [(128, 256), (256, 128)])
def test_two_pass_k_not_v_varlen(K, V):
    cap = sum(VARLEN_LENGTHS) + 23
    w = workloads.make_varlen("t", VARLEN_LENGTHS, cap, 2, K, V, 64, torch.bfloat16, 1211 + K,
                              mode=workloads.GATE_SAFE)
    o, st = run_gpu(w)
    compare(w, o, st)
    end = int(w.cu_seqlens[-1])
    t = to_device(w)
    for n, L in enumerate(VARLEN_LENGTHS):
        if L == 0:
            assert torch.equal(st[n], t["initial_state"][n])


@pytest.mark.parametrize("lb,g_std", [(-5.0, 10.0), (-1e-4, 3.0)])
def test_two_pass_gate_extremes(lb, g_std):
    """lb = -5 with a saturated sigmoid, and lb close to 0 (FLA skill "fla-kda", correctness
    checklist: gate numerical extremes), with a float32 o held to the plain bound."""
    w = workloads.make_dense("t", 1, 300, 2, 256, 256, 64, torch.bfloat16, 951, g_std=g_std,
                             state_std=0.05, lower_bound=lb)
    w.A_log = w.A_log * 3.0
    o, st = run_gpu(w, o_dtype=torch.float32)
    compare(w, o, st)


@pytest.mark.parametrize("hk", [1, 2])
def test_two_pass_grouped_value_heads(hk):
    """GVA: 4 value heads over 1 or 2 query / key heads, against the oracle and bitwise equal to
    the multi-head call on repeated q and k heads."""
    w = grouped(workloads.make_dense("t", 2, 130, 4, 256, 256, 64, torch.bfloat16, 960 + hk,
                                     state_std=0.05), hk)
    o, st = run_gpu(w)
    compare(w, o, st)
    t = to_device(w)
    r = 4 // hk
    o2, st2 = kda().kda_chunk_fwd(t["q"].repeat_interleave(r, dim=2), t["k"].repeat_interleave(r, dim=2),
                                  t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"], w.mode,
                                  w.lower_bound, t["initial_state"], True, None, 64)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(st, st2)


@pytest.mark.parametrize("D", [128, 256])
def test_two_pass_float32_gate_is_bitwise_the_bf16_gate(D):
    w = workloads.make_dense("t", 2, 150, 2, D, D, 64, torch.bfloat16, 971, state_std=0.05)
    with two_pass(D):
        o16, s16 = run_gpu(w)
        w.g = w.g.float()
        o32, s32 = run_gpu(w)
    assert torch.equal(o16, o32) and torch.equal(s16, s32)
    compare(w, o32, s32)


@pytest.mark.parametrize("D", [128, 256])
def test_two_pass_q_l2norm(D):
    """The deferred q l2norm (attention-gym PR #345) on query rows scaled by 10^U(-3, 3) with
    an all-zero row, against the oracle with the same option."""
    w = workloads.make_dense("t", 1, 150, 2, D, D, 64, torch.bfloat16, 981, state_std=0.05)
    g = torch.Generator().manual_seed(982)
    sc = torch.pow(10.0, torch.rand((1, 150, 2, 1), generator=g) * 6 - 3)
    sc[:, 70] = 0.0
    w.q = (w.q.float() * sc).to(w.q.dtype)
    with two_pass(D):
        o, st = run_gpu(w, q_l2norm=True, o_dtype=torch.float32)
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, w.mode,
                                  w.lower_bound, w.initial_state, None, q_l2norm=True)
    check_o(o, o_ref, torch.bfloat16)
    check_state(st, s_ref, torch.bfloat16)


def test_two_pass_status_word_stays_clear():
    w = workloads.make_dense("t", 1, 200, 2, 256, 256, 64, torch.bfloat16, 991, state_std=0.05)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda().kda_fused_wait_timeouts(reset=True)
    o, st = run_gpu(w, status=status)
    assert int(status.item()) == 0 and kda().kda_fused_wait_timeouts() == 0
    compare(w, o, st)


def test_two_pass_no_initial_state_and_in_place_state():
    w = workloads.make_dense("t", 2, 100, 2, 256, 256, 64, torch.bfloat16, 992)
    o1, s1 = run_gpu(w)
    zeros = torch.zeros((2, 2, 256, 256), device="cuda")
    o2, s2 = run_gpu(w, initial_state=zeros)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    w2 = workloads.make_dense("t", 2, 100, 2, 256, 256, 64, torch.bfloat16, 993, state_std=0.05)
    oa, sa = run_gpu(w2)
    t = to_device(w2)
    S = t["initial_state"].clone()
    ob, _ = kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                                w2.mode, w2.lower_bound, S, True, None, 64, final_state=S)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob) and torch.equal(sa, S)


# ---- the balanced schedule of pass 2 (dense inputs whose (sequence, head) units leave the last
# wave of a one-CTA-per-unit grid part-empty): one cooperative launch, the value blocks of a head
# on a group of CTAs side by side, each group running an equal share of the units' chunks laid
# end to end; a unit cut at a group boundary runs its first chunks on one group and the rest on
# the previous one, the FP32 state crossing through the workspace behind a flag.  The chunks are
# computed from the FP32 state and their images alone, so the two schedules agree bitwise.

def _chain_cuts(N, H, T, groups):
    """Chunk-times per group and, per cut unit u = n + N h, the chunks of its first part (the
    library's plan restated: boundaries at multiples of ceil(U nt / groups))."""
    import math

    nt, U = math.ceil(T / 64), N * H
    cm = math.ceil(U * nt / groups)
    cuts = {}
    for i in range(1, groups):
        b = i * cm
        if b < U * nt and b % nt:
            cuts[b // nt] = (b // nt + 1) * nt - b
    return cm, cuts


def _balanced_shape():
    """About 2.1 waves of (sequence, head) units of 16 chunks on the device's groups of two SMs
    (160 units on 76 groups of a 152-SM GB300)."""
    S = torch.cuda.get_device_properties(0).multi_processor_count
    return 4, max(1, round(2.1 * (S // 2) / 4)), S // 2


def _ws(w):
    return kda().kda_chunk_workspace_bytes(w.q.dtype, w.B, w.T, w.H, w.K, w.V, w.chunk_size, 0, w.mode)


@pytest.mark.parametrize("mode,o_dtype,state", [
    (workloads.GATE_SAFE, None, True),
    (workloads.GATE_NONSAFE, None, False),
    (workloads.GATE_PRE, torch.float32, True),
], ids=["safe-bf16o-state", "nonsafe-bf16o", "pre-f32o-state"])
def test_two_pass_balanced_chain_equals_plain_grid(mode, o_dtype, state):
    from parity import check_units

    B, H, groups = _balanced_shape()
    T = 1000  # 16 chunks, the last one ragged
    w = workloads.make_dense("t", B, T, H, 256, 256, 64, torch.bfloat16, 950 + mode,
                             state_std=0.05 if state else None, mode=mode,
                             g_std=2.0 if mode == workloads.GATE_NONSAFE else 1.0)
    cm, cuts = _chain_cuts(B, H, T, groups)
    assert cuts and min(cuts.values()) >= 1 and max(cuts.values()) < 16
    ws_bal = _ws(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda().kda_fused_wait_timeouts(reset=True)
    o1, s1 = run_gpu(w, o_dtype=o_dtype, status=status)
    assert int(status.item()) == 0 and kda().kda_fused_wait_timeouts() == 0
    kda().kda_test_hooks(one_launch=True)  # one CTA per (value block, sequence, head)
    try:
        assert _ws(w) < ws_bal, "the balanced schedule applies to these sizes"
        o2, s2 = run_gpu(w, o_dtype=o_dtype)
    finally:
        kda().kda_test_hooks()
    assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)
    U = B * H
    pick = {0, U - 1, min(cuts), min(cuts, key=lambda u: cuts[u]), max(cuts, key=lambda u: cuts[u])}
    check_units(w, o1, s1, sorted({(u % B, u // B) for u in pick}))


def test_two_pass_balanced_chain_in_a_cuda_graph():
    """The flag reset and the cooperative launch are captured; a replay with new inputs written
    in place matches an eager call bitwise."""
    B, H, _ = _balanced_shape()
    ws = [workloads.make_dense("t", B, 1000, H, 256, 256, 64, torch.bfloat16, 960 + i, state_std=0.05)
          for i in range(2)]
    t = to_device(ws[0])
    S0, S_fin = t["initial_state"].clone(), torch.empty_like(t["initial_state"])
    o = torch.empty((B, 1000, H, 256), device="cuda", dtype=torch.bfloat16)
    work = torch.empty(_ws(ws[0]), device="cuda", dtype=torch.uint8)

    def call():
        kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                            ws[0].mode, ws[0].lower_bound, S0, True, None, 64, o=o,
                            final_state=S_fin, workspace=work)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    for w in ws[::-1]:
        src = to_device(w)
        for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias"):
            t[name].copy_(src[name])
        S0.copy_(src["initial_state"])
        graph.replay()
        torch.cuda.synchronize()
        o_g, s_g = o.clone(), S_fin.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_g, o) and torch.equal(s_g, S_fin)
