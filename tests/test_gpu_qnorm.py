"""Deferred query l2 normalisation (kda_chunk_fwd_ex with KDA_FLAG_Q_L2NORM, attention-gym
PR #345 "Fuse q l2norm into the chunk_kda output kernel"): against the float64 oracle with
the same option, on query rows scaled by 1e-3 .. 1e3 and on all-zero rows, through the fused
bf16 kernel and the float32 stage-by-stage path, and against the explicit path (q normalised
before the call)."""
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


def scaled_rows(w, seed):
    """q rows times 10^U(-3, 3), two all-zero rows, in the workload's dtype."""
    g = torch.Generator().manual_seed(seed)
    B, T, H, _ = w.q.shape
    sc = torch.pow(10.0, torch.rand((B, T, H, 1), generator=g) * 6 - 3)
    sc[:, T // 3] = 0.0
    sc[0, -1, -1] = 0.0
    w.q = (w.q.float() * sc).to(w.q.dtype)
    return w


def run(w, q_l2norm, q=None, **kw):
    t = to_device(w)
    o, st = kda().kda_chunk_fwd(t["q"] if q is None else q, t["k"], t["v"], t["g"], t["beta"],
                                A_log=t["A_log"], dt_bias=t["dt_bias"], mode=w.mode,
                                lower_bound=w.lower_bound, initial_state=t["initial_state"],
                                output_final_state=True, cu_seqlens=t["cu_seqlens"],
                                chunk_size=w.chunk_size, q_l2norm=q_l2norm, **kw)
    torch.cuda.synchronize()
    return o, st


def ref(w):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, w.mode, w.lower_bound,
                          w.initial_state, w.cu_seqlens, q_l2norm=True)


@pytest.mark.parametrize("dtype,C,o_dtype", [(torch.bfloat16, 64, None),
                                             (torch.bfloat16, 64, torch.float32),
                                             (torch.bfloat16, 32, None),
                                             (torch.float32, 64, None)],
                         ids=["fused-bf16", "fused-f32out", "stagewise-c32", "stagewise-f32"])
@pytest.mark.parametrize("T", [17, 130, 200])
def test_q_l2norm_against_oracle(dtype, C, o_dtype, T):
    w = scaled_rows(workloads.make_dense("t", 2, T, 3, 128, 128, C, dtype, 71 + T,
                                         state_std=0.05), 5 + T)
    o, st = run(w, True, o_dtype=o_dtype)
    o_ref, s_ref = ref(w)
    check_o(o, o_ref, dtype, valid_mask(w))
    check_state(st, s_ref, dtype)
    zero = to_np(o)[:, T // 3]
    assert (zero == 0).all() and (to_np(o)[0, -1, -1] == 0).all()


def test_q_l2norm_varlen_packed():
    lens = workloads.varlen_lengths(6, 300, 1500, empty_slots=(2,), seed=3)
    w = workloads.make_varlen("t", lens, 1600, 2, 128, 128, 64, torch.bfloat16, 3, poison_tail=False)
    w = scaled_rows(w, 9)
    o, st = run(w, True)
    o_ref, s_ref = ref(w)
    check_o(o, o_ref, torch.bfloat16, valid_mask(w))
    check_state(st, s_ref, torch.bfloat16)


def test_q_l2norm_state_does_not_see_q():
    """The final state is the same with and without the option, bit for bit."""
    w = scaled_rows(workloads.make_dense("t", 2, 150, 2, 128, 128, 64, torch.bfloat16, 91,
                                         state_std=0.05), 13)
    _, s1 = run(w, False)
    _, s2 = run(w, True)
    assert torch.equal(s1, s2)


def test_q_l2norm_matches_explicit_path():
    """Normalising q before the call (in float32, then rounded to bf16 as a separate pass
    would) gives the same output within the bf16 tolerance."""
    w = scaled_rows(workloads.make_dense("t", 2, 190, 2, 128, 128, 64, torch.bfloat16, 97,
                                         state_std=0.05), 17)
    o_fused, _ = run(w, True, o_dtype=torch.float32)
    qd = w.q.float().cuda()
    qn = (qd * torch.rsqrt((qd * qd).sum(-1, keepdim=True) + oracle.Q_L2NORM_EPS)).to(w.q.dtype)
    o_expl, _ = run(w, False, q=qn, o_dtype=torch.float32)
    assert rel_l2(to_np(o_fused), to_np(o_expl)) < 2e-2


def test_flag_bits_through_binding():
    w = workloads.make_dense("t", 1, 64, 2, 128, 128, 64, torch.bfloat16, 1)
    t = to_device(w)
    with pytest.raises(ValueError):
        kda().kda_chunk_fwd_ex(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"],
                               t["dt_bias"], flags=4)
    o1, _ = kda().kda_chunk_fwd_ex(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"],
                                   t["dt_bias"], flags=kda().FLAG_Q_L2NORM)
    o2, _ = run(w, True)
    assert torch.equal(o1, o2)
