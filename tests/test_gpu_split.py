"""The fused kernel's split schedule for dense batches of a little more than one wave of
(sequence, head) units: a first launch runs the leading chunks of one wave of units, a second
runs the other units whole and finishes the first ones from the FP32 state they left in their
own output rows.  Every chunk of the chunked form is computed from the FP32 state and the
chunk's inputs alone, so the two schedules agree bitwise; the split one is also checked
against the oracle on sampled units (split units and whole units of the second launch)."""
import pytest
import torch

from chunked_kda_gb300 import workloads
from parity import check_units, to_device
from test_gpu_chunk import kda, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def split_shape():
    """(B, H): B H = 1.5 S units on S SMs (the last wave half full, the second pieces then take
    two rounds on the SMs the whole units leave free)."""
    S = torch.cuda.get_device_properties(0).multi_processor_count
    return 2, (S + S // 2) // 2, S


T_SPLIT = 720  # 12 chunks, the last one ragged; the second pieces hold 272 tokens


def _units(B, H, S):
    """A few units u = n + B h: the first and last split unit, the first and last whole one."""
    U = B * H
    return sorted({(u % B, u // B) for u in (0, S - 1, S, U - 1)})


def _launches(w, o_dtype=None):
    return kda().kda_chunk_fwd_launches(w.q.dtype, w.B, w.T, w.H, w.K, w.V, w.chunk_size, 0,
                                        w.mode, o_dtype)


@pytest.mark.parametrize("mode,o_dtype,state", [
    (workloads.GATE_SAFE, None, True),
    (workloads.GATE_PRE, None, False),
    (workloads.GATE_SAFE, torch.float32, False),
], ids=["safe-bf16o-state", "pre-bf16o", "safe-f32o"])
def test_split_equals_one_launch(mode, o_dtype, state):
    B, H, S = split_shape()
    w = workloads.make_dense("t", B, T_SPLIT, H, 128, 128, 64, torch.bfloat16, 71 + mode,
                             state_std=0.05 if state else None, mode=mode)
    assert _launches(w, o_dtype) == 2
    o1, s1 = run_gpu(w, o_dtype=o_dtype)
    kda().kda_test_hooks(one_launch=True)
    try:
        assert _launches(w, o_dtype) == 1
        o2, s2 = run_gpu(w, o_dtype=o_dtype)
    finally:
        kda().kda_test_hooks()
    assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)
    check_units(w, o1, s1, _units(B, H, S))


def test_split_state_in_place_and_q_l2norm():
    """final_state aliasing initial_state (each unit's slot is read by its first piece before
    its last piece writes it), with the deferred q l2norm."""
    B, H, S = split_shape()
    w = workloads.make_dense("t", B, T_SPLIT, H, 128, 128, 64, torch.bfloat16, 77, state_std=0.05)
    t = to_device(w)

    def run():
        S0 = t["initial_state"].clone()
        o, st = kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"],
                                    t["dt_bias"], w.mode, w.lower_bound, S0, True, None, 64,
                                    final_state=S0, q_l2norm=True)
        torch.cuda.synchronize()
        assert st.data_ptr() == S0.data_ptr()
        return o, st

    o1, s1 = run()
    kda().kda_test_hooks(one_launch=True)
    try:
        o2, s2 = run()
    finally:
        kda().kda_test_hooks()
    assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)


def test_no_split_when_the_second_pieces_are_too_short():
    """A second piece must hold the state in its output rows (256 bf16 rows): short sequences
    keep one launch."""
    B, H, S = split_shape()
    assert kda().kda_chunk_fwd_launches(torch.bfloat16, B, 320, H, 128, 128, 64, 0) == 1
    assert kda().kda_chunk_fwd_launches(torch.bfloat16, B, T_SPLIT, H, 128, 128, 64, 0) == 2
    # whole waves, fewer units than SMs, or a last wave more than half full: one launch
    assert kda().kda_chunk_fwd_launches(torch.bfloat16, 1, 4096, S + S // 2 + 2, 128, 128, 64, 0) == 1
    assert kda().kda_chunk_fwd_launches(torch.bfloat16, 1, 4096, S, 128, 128, 64, 0) == 1
    assert kda().kda_chunk_fwd_launches(torch.bfloat16, 1, 4096, S - 1, 128, 128, 64, 0) == 1
    # packed inputs keep their heads-fastest grid
    assert kda().kda_chunk_fwd_launches(torch.bfloat16, 1, 8192, H, 128, 128, 64, B) == 1


def test_split_schedule_in_a_cuda_graph():
    """Both launches of the split schedule are captured; replays with new inputs written in
    place match eager calls bitwise."""
    B, H, S = split_shape()
    ws = [workloads.make_dense("t", B, T_SPLIT, H, 128, 128, 64, torch.bfloat16, 80 + i,
                               state_std=0.05) for i in range(2)]
    t = to_device(ws[0])
    S0, S_fin = t["initial_state"].clone(), torch.empty_like(t["initial_state"])
    o = torch.empty((B, T_SPLIT, H, 128), device="cuda", dtype=torch.bfloat16)

    def call():
        kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                            ws[0].mode, ws[0].lower_bound, S0, True, None, 64, o=o,
                            final_state=S_fin)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        call()  # warm-up outside the capture
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
