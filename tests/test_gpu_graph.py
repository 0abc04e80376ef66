"""CUDA-graph capture and replay (attention-gym PR #317 test plan: CUDA-graph replay with
mutated boundaries and history).  Every entry point only enqueues work on the caller's
stream and never reads cu_seqlens on the host, so one captured call replays correctly after
the device-side offsets, inputs and states it points at are rewritten in place."""
import math

import numpy as np
import pytest
import torch

import oracle
from chunked_kda_gb300 import workloads
from parity import check_o, check_state, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def kda():
    import chunked_kda_gb300

    return chunked_kda_gb300


def _log2_gate(shape, seed):
    gen = torch.Generator().manual_seed(seed)
    return -(torch.rand(shape, generator=gen) * 4.99 + 0.01) / math.log(2.0)


def test_recurrent_graph_replay_mutated_boundaries_and_history():
    cap, H, K, V, N = 48, 2, 128, 128, 4
    dev = "cuda"
    q = torch.empty((1, cap, H, K), device=dev, dtype=torch.bfloat16)
    k, v = torch.empty_like(q), torch.empty((1, cap, H, V), device=dev, dtype=torch.bfloat16)
    gate = torch.empty((1, cap, H, K), device=dev)
    beta = torch.empty((1, cap, H), device=dev, dtype=torch.bfloat16)
    cu = torch.zeros(N + 1, device=dev, dtype=torch.int32)
    S = torch.empty((N, H, K, V), device=dev)
    o = torch.zeros((1, cap, H, V), device=dev, dtype=torch.bfloat16)

    def fill(lens, seed):
        w = workloads.make_varlen("g", lens, cap, H, K, V, 64, torch.bfloat16, seed)
        g2 = _log2_gate((1, cap, H, K), seed + 1)
        q.copy_(w.q.nan_to_num(0.0)); k.copy_(w.k.nan_to_num(0.0)); v.copy_(w.v.nan_to_num(0.0))
        beta.copy_(w.beta.nan_to_num(0.0)); gate.copy_(g2); cu.copy_(w.cu_seqlens)
        S.copy_(w.initial_state)
        return w, g2

    w, g2 = fill([5, 0, 17, 9], 700)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kda().kda_recurrent_fwd(q, k, v, gate, beta, S, True, cu, o=o, final_state=S)
    for lens, seed in (([5, 0, 17, 9], 700), ([0, 30, 1, 0], 710), ([12, 12, 12, 12], 720)):
        w, g2 = fill(lens, seed)
        S0 = w.initial_state.clone()
        graph.replay()
        torch.cuda.synchronize()
        o_ref, s_ref = oracle.forward(w.q.nan_to_num(0.0), w.k.nan_to_num(0.0), w.v.nan_to_num(0.0),
                                      g2, w.beta.nan_to_num(0.0), None, None, oracle.GATE_LOG2,
                                      0.0, S0, w.cu_seqlens)
        end = sum(lens)
        check_o(o[:, :end], o_ref[:, :end], torch.bfloat16)
        check_state(S, s_ref, torch.bfloat16)
        # history: replaying again continues from the state the last replay left in place
        S1 = S.clone()
        graph.replay()
        torch.cuda.synchronize()
        _, s_ref2 = oracle.forward(w.q.nan_to_num(0.0), w.k.nan_to_num(0.0), w.v.nan_to_num(0.0),
                                   g2, w.beta.nan_to_num(0.0), None, None, oracle.GATE_LOG2, 0.0,
                                   S1.cpu(), w.cu_seqlens)
        check_state(S, s_ref2, torch.bfloat16)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 128), (torch.bfloat16, 256)],
                         ids=["fused", "stagewise", "two-pass"])
def test_chunk_graph_replay_mutated_boundaries(dtype, D):
    cap, H, K, V, N = 300, 2, D, D, 3
    dev = "cuda"
    lens0 = [100, 0, 150]
    w = workloads.make_varlen("g", lens0, cap, H, K, V, 64, dtype, 730, poison_tail=False)
    t = {n: (x.to(dev) if x is not None else None) for n, x in w.tensors().items()}
    o = torch.zeros((1, cap, H, V), device=dev, dtype=dtype)
    S_out = torch.empty((N, H, K, V), device=dev)
    need = kda().kda_chunk_workspace_bytes(dtype, 1, cap, H, K, V, 64, N)
    ws = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kda().kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], None, None, w.mode,
                            w.lower_bound, t["initial_state"], True, t["cu_seqlens"], 64, o=o,
                            final_state=S_out, workspace=ws)
    for lens, seed in ((lens0, 730), ([0, 260, 33], 740), ([64, 64, 64], 750)):
        w2 = workloads.make_varlen("g", lens, cap, H, K, V, 64, dtype, seed, poison_tail=False)
        for n in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens"):
            t[n].copy_(getattr(w2, n))
        graph.replay()
        torch.cuda.synchronize()
        o_ref, s_ref = oracle.forward(w2.q, w2.k, w2.v, w2.g, w2.beta, None, None, w2.mode,
                                      w2.lower_bound, w2.initial_state, w2.cu_seqlens)
        end = sum(lens)
        check_o(o[:, :end], o_ref[:, :end], dtype)
        check_state(S_out, s_ref, dtype)
