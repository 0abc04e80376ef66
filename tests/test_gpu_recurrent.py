"""kda_recurrent_fwd and kda_gate_fwd against the float64 oracle, and the chunked form
against the recurrent form on the same inputs (attention-gym PR #317, Test Plan:
cross-check vs chunk_kda via bounded_gate_cumsum(chunk_size=1 vs 64))."""
import math

import numpy as np
import pytest
import torch

import oracle
from chunked_kda_gb300 import workloads
from parity import check_o, check_state, rel_l2, to_device, to_np, valid_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def kda():
    import chunked_kda_gb300

    return chunked_kda_gb300


def log2_gate(shape, seed):
    gen = torch.Generator().manual_seed(seed)
    return -(torch.rand(shape, generator=gen) * 4.99 + 0.01) / math.log(2.0)


def run_rec(q, k, v, gate, beta, S0, cu=None, **kw):
    dev = "cuda"
    o, st = kda().kda_recurrent_fwd(q.to(dev), k.to(dev), v.to(dev), gate.to(dev), beta.to(dev),
                                    None if S0 is None else S0.to(dev), True,
                                    None if cu is None else cu.to(dev), **kw)
    torch.cuda.synchronize()
    return o, st


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("K,V", [(64, 64), (128, 128), (256, 256), (64, 128), (128, 256),
                                 (256, 64)])
@pytest.mark.parametrize("T", [1, 7, 33])
def test_recurrent_dense(dtype, K, V, T):
    w = workloads.make_dense("r", 2, T, 3, K, V, 64, dtype, 60 + T, state_std=0.05)
    gate = log2_gate((2, T, 3, K), 61 + T)
    o, st = run_rec(w.q, w.k, w.v, gate, w.beta, w.initial_state)
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, gate, w.beta, None, None, oracle.GATE_LOG2, 0.0,
                                  w.initial_state)
    check_o(o, o_ref, dtype)
    check_state(st, s_ref, torch.float32 if dtype == torch.float32 else dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_recurrent_packed(dtype):
    lens = [0, 5, 1, 0, 0, 40, 17, 0]
    cap = sum(lens) + 9
    w = workloads.make_varlen("r", lens, cap, 2, 128, 128, 64, dtype, 70)
    gate = log2_gate((1, cap, 2, 128), 71)
    gate[:, sum(lens):] = float("nan")
    sentinel = torch.full((1, cap, 2, 128), -777.0, device="cuda", dtype=dtype)
    o, st = run_rec(w.q, w.k, w.v, gate, w.beta, w.initial_state, w.cu_seqlens, o=sentinel)
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, gate, w.beta, None, None, oracle.GATE_LOG2, 0.0,
                                  w.initial_state, w.cu_seqlens)
    check_o(o, o_ref, dtype, valid_mask(w))
    check_state(st, s_ref, dtype)
    end = sum(lens)
    assert torch.equal(o[:, end:], torch.full_like(o[:, end:], -777.0))
    S0 = w.initial_state.cuda()
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.equal(st[n], S0[n])


def test_decode_in_place_256_steps():
    """512 packed one-token sequences, H=32, K=V=128, bf16, FP32 states updated in place
    over 256 steps with fresh inputs; sampled units followed by the oracle step by step."""
    n, H, K, V, steps = 512, 32, 128, 128, 256
    cu = workloads.decode_cu_seqlens(n, device="cuda")
    S = workloads.decode_state(n, H, K, V, device="cpu")
    units = [(0, 0), (511, 31), (137, 5), (300, 17)]
    ref = {u: S[u[0], u[1]].double().numpy().copy() for u in units}
    S_dev = S.cuda()
    for step in range(steps):
        st = workloads.decode_step(step, n, H, K, V, device="cuda")
        o, _ = kda().kda_recurrent_fwd(st.q, st.k, st.v, st.gate, st.beta, S_dev, True, cu,
                                       final_state=S_dev)
        if step in (0, steps - 1):
            torch.cuda.synchronize()
            o_np = to_np(o)
        for (sn, h) in units:
            sl = slice(sn, sn + 1)
            hs = slice(h, h + 1)
            o_ref, s_new = oracle.forward(st.q[:, sl, hs].cpu(), st.k[:, sl, hs].cpu(),
                                          st.v[:, sl, hs].cpu(), st.gate[:, sl, hs].cpu(),
                                          st.beta[:, sl, hs].cpu(), None, None,
                                          oracle.GATE_LOG2, 0.0,
                                          ref[(sn, h)].reshape(1, 1, K, V))
            ref[(sn, h)] = s_new[0, 0]
            if step in (0, steps - 1):
                check_o(o_np[0, sn, h], o_ref[0, 0, 0], torch.bfloat16, what=f"o step {step}")
    torch.cuda.synchronize()
    for (sn, h) in units:
        e = rel_l2(to_np(S_dev[sn, h]), ref[(sn, h)])
        assert e <= 1e-4, f"state[{sn},{h}] after {steps} steps: rel-L2 {e:.2e}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("C", [1, 16, 32, 64])
@pytest.mark.parametrize("mode", [workloads.GATE_PRE, workloads.GATE_SAFE, workloads.GATE_NONSAFE],
                         ids=["pre", "safe", "nonsafe"])
def test_gate_fwd(dtype, C, mode):
    lens = [0, 70, 1, 0, 64, 33]
    cap = sum(lens) + 11
    w = workloads.make_varlen("g", lens, cap, 3, 128, 128, 64, dtype, 80, mode=mode)
    out = torch.full((1, cap, 3, 128), 4242.0, device="cuda")
    t = to_device(w)
    kda().kda_gate_fwd(t["g"], t["A_log"], t["dt_bias"], mode, w.lower_bound, t["cu_seqlens"], C,
                       out=out)
    torch.cuda.synchronize()
    ref = oracle.gate(w.g, w.A_log, w.dt_bias, mode, w.lower_bound, w.cu_seqlens, C)
    end = sum(lens)
    got = to_np(out)[0, :end]
    assert np.allclose(got, ref[0, :end], rtol=1e-5, atol=1e-5), np.abs(got - ref[0, :end]).max()
    assert torch.equal(out[:, end:], torch.full_like(out[:, end:], 4242.0))
    if mode == workloads.GATE_SAFE and C == 1:
        nat = got * math.log(2.0)
        assert (nat <= 0).all() and (nat >= w.lower_bound * (1 + 1e-6)).all()


@pytest.mark.parametrize("K", [128, 12])
def test_gate_fwd_vector_and_scalar_kernels(K):
    """Rows of H * K channels that are a multiple of 8 with 16-byte aligned g and out take the
    vectorised kernel; others (K = 12 with H = 3, or an output offset by one element) take the
    scalar one.  Both match the oracle."""
    lens = [0, 70, 1, 0, 64, 33]
    cap = sum(lens) + 11
    w = workloads.make_varlen("g", lens, cap, 3, K, K, 64, torch.bfloat16, 81, mode=workloads.GATE_SAFE)
    t = to_device(w)
    ref = oracle.gate(w.g, w.A_log, w.dt_bias, workloads.GATE_SAFE, w.lower_bound, w.cu_seqlens, 64)
    end = sum(lens)
    buf = torch.full((1 + cap * 3 * K,), 4242.0, device="cuda")
    for off in (0, 1):  # aligned, then one float past it
        out = buf[off:off + cap * 3 * K].view(1, cap, 3, K)
        kda().kda_gate_fwd(t["g"], t["A_log"], t["dt_bias"], workloads.GATE_SAFE, w.lower_bound,
                           t["cu_seqlens"], 64, out=out)
        torch.cuda.synchronize()
        got = to_np(out)[0, :end]
        assert np.allclose(got, ref[0, :end], rtol=1e-5, atol=1e-5), np.abs(got - ref[0, :end]).max()


def test_gate_half_point():
    """g + dt_bias = 0 gives sigmoid(0) = 1/2, so the activation is lower_bound / 2."""
    H, K = 2, 128
    dt_bias = torch.linspace(-3, 3, H * K).reshape(H, K)
    g = (-dt_bias).reshape(1, 1, H, K).contiguous()
    A_log = torch.full((H, K), 1.7)
    out = kda().kda_gate_fwd(g.cuda(), A_log.cuda(), dt_bias.cuda(), workloads.GATE_SAFE, -3.0,
                             None, 1)
    torch.cuda.synchronize()
    want = -1.5 / math.log(2.0)
    assert torch.allclose(out.cpu(), torch.full_like(out.cpu(), want), rtol=1e-6, atol=0)


@pytest.mark.parametrize("C", [32, 64])
def test_chunk_vs_recurrent(C):
    """Same inputs through both forms: the log2 gate from kda_gate_fwd(chunk_size=1) feeds
    the recurrent form; the chunked form applies the gate in-kernel."""
    w = workloads.make_dense("x", 2, 150, 2, 128, 128, C, torch.bfloat16, 90, state_std=0.05)
    t = to_device(w)
    gate = kda().kda_gate_fwd(t["g"], t["A_log"], t["dt_bias"], w.mode, w.lower_bound, None, 1)
    o_r, s_r = kda().kda_recurrent_fwd(t["q"], t["k"], t["v"], gate, t["beta"],
                                       t["initial_state"], True)
    o_c, s_c = kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"],
                                   t["dt_bias"], w.mode, w.lower_bound, t["initial_state"], True,
                                   None, C)
    torch.cuda.synchronize()
    assert rel_l2(to_np(o_c), to_np(o_r)) <= 2e-2
    assert rel_l2(to_np(s_c), to_np(s_r)) <= 2e-2


# ---- non-power-of-two head sizes and the decode-side preprocessing (kda_recurrent_fwd_ex)

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("K,V", [(40, 24), (96, 80), (100, 130), (200, 256), (256, 7), (1, 1)])
def test_recurrent_masked_head_dims(dtype, K, V):
    """K and V that are not 64, 128 or 256 (attention-gym PR #317 test plan: non-power-of-two
    K/V masking): dense and packed, against the oracle."""
    w = workloads.make_dense("r", 2, 9, 3, K, V, 64, dtype, 500 + K + V, state_std=0.05)
    gate = log2_gate((2, 9, 3, K), 501 + K)
    o, st = run_rec(w.q, w.k, w.v, gate, w.beta, w.initial_state)
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, gate, w.beta, None, None, oracle.GATE_LOG2, 0.0,
                                  w.initial_state)
    check_o(o, o_ref, dtype)
    check_state(st, s_ref, dtype)
    lens = [3, 0, 11]
    wp = workloads.make_varlen("r", lens, 16, 2, K, V, 64, dtype, 502 + K)
    gp = log2_gate((1, 16, 2, K), 503 + K)
    o, st = run_rec(wp.q, wp.k, wp.v, gp, wp.beta, wp.initial_state, wp.cu_seqlens)
    o_ref, s_ref = oracle.forward(wp.q, wp.k, wp.v, gp, wp.beta, None, None, oracle.GATE_LOG2,
                                  0.0, wp.initial_state, wp.cu_seqlens)
    check_o(o, o_ref, dtype, valid_mask(wp))
    check_state(st, s_ref, dtype)


def run_rec_ex(w, g, mode, flags, beta=None):
    t = to_device(w)
    o, st = kda().kda_recurrent_fwd_ex(t["q"], t["k"], t["v"], g.cuda(), t["beta"] if beta is None
                                       else beta.cuda(), t["A_log"], t["dt_bias"], mode,
                                       w.lower_bound, t["initial_state"], True, t["cu_seqlens"],
                                       flags=flags)
    torch.cuda.synchronize()
    return o, st


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("mode", [workloads.GATE_PRE, workloads.GATE_SAFE, workloads.GATE_NONSAFE],
                         ids=["pre", "safe", "nonsafe"])
def test_recurrent_in_kernel_gate(dtype, mode):
    """The raw gate activated inside the recurrent kernel equals the oracle with the same gate
    mode, and the explicit path (kda_gate_fwd with chunk_size 1, then kda_recurrent_fwd)."""
    lens = [0, 40, 1, 0, 23]
    w = workloads.make_varlen("r", lens, 70, 2, 128, 128, 64, dtype, 520 + mode, mode=mode)
    o, st = run_rec_ex(w, w.g, mode, 0)
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, mode,
                                  w.lower_bound, w.initial_state, w.cu_seqlens)
    check_o(o, o_ref, dtype, valid_mask(w))
    check_state(st, s_ref, dtype)
    t = to_device(w)
    gate = kda().kda_gate_fwd(t["g"], t["A_log"], t["dt_bias"], mode, w.lower_bound,
                              t["cu_seqlens"], 1)
    o2, st2 = run_rec(w.q, w.k, w.v, gate, w.beta, w.initial_state, w.cu_seqlens)
    end = sum(lens)
    assert rel_l2(to_np(o)[:, :end], to_np(o2)[:, :end]) < 1e-5
    assert rel_l2(to_np(st), to_np(st2)) < 1e-5


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("flags", [1, 2, 4, 7], ids=["q", "k", "beta", "all"])
def test_recurrent_preprocessing_flags(dtype, flags):
    """q / k l2norm and beta logits inside the kernel: rows scaled by 1e-3 .. 1e3 and a zero
    row, against the oracle with the same options."""
    w = workloads.make_dense("r", 2, 21, 3, 128, 128, 64, dtype, 540 + flags, state_std=0.05)
    gen = torch.Generator().manual_seed(541 + flags)
    sq = torch.pow(10.0, torch.rand((2, 21, 3, 1), generator=gen) * 6 - 3)
    sk = torch.pow(10.0, torch.rand((2, 21, 3, 1), generator=gen) * 6 - 3)
    sq[:, 4] = 0.0
    if flags & 1:
        w.q = (w.q.float() * sq).to(dtype)
    if flags & 2:
        w.k = (w.k.float() * sk).to(dtype)
    beta = w.beta
    if flags & 4:
        beta = (torch.randn((2, 21, 3), generator=gen) * 2).to(dtype)  # logits
    gate = log2_gate((2, 21, 3, 128), 542 + flags)
    w2 = w
    o, st = run_rec_ex(w2, gate, kda().GATE_LOG2, flags, beta=beta)
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, gate, beta, None, None, oracle.GATE_LOG2, 0.0,
                                  w.initial_state, q_l2norm=bool(flags & 1),
                                  k_l2norm=bool(flags & 2), beta_logits=bool(flags & 4))
    check_o(o, o_ref, dtype)
    check_state(st, s_ref, dtype)
    if flags & 1:
        assert (to_np(o)[:, 4] == 0).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_recurrent_grouped_value_heads(dtype):
    """GVA in the recurrent form: 6 value heads over 2 query / key heads."""
    w = workloads.make_dense("r", 2, 17, 6, 128, 128, 64, dtype, 640, state_std=0.05)
    w.q = w.q[:, :, :2].contiguous()
    w.k = w.k[:, :, :2].contiguous()
    gate = log2_gate((2, 17, 6, 128), 641)
    t = to_device(w)
    o, st = kda().kda_recurrent_fwd_ex(t["q"], t["k"], t["v"], gate.cuda(), t["beta"],
                                       initial_state=t["initial_state"], output_final_state=True)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.forward(w.q, w.k, w.v, gate, w.beta, None, None, oracle.GATE_LOG2, 0.0,
                                  w.initial_state)
    check_o(o, o_ref, dtype)
    check_state(st, s_ref, dtype)
