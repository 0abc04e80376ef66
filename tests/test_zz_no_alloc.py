"""kda_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate device
memory (for instance a plugin that only receives input and output pointers from a host
framework that owns all device memory).  It runs on the library's fixed scratch array
instead of a workspace.  Checked here against kda_chunk_fwd on several calls in a row,
so that a call never depends on what the previous one left in the shared array.
This file is collected last on purpose."""
import pytest
import torch

from chunked_kda_gb300 import workloads
from parity import check_o, check_state, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_kda_gb300

    return chunked_kda_gb300


def _cases():
    # float32 and bf16 inputs, dense and packed with empty slots, different sizes per call
    yield workloads.make_dense("a", 1, 128, 2, 64, 64, 64, torch.float32, 501, state_std=0.05)
    w = workloads.make_varlen("b", [0, 70, 1, 0, 100], 200, 2, 128, 128, 32, torch.bfloat16, 502)
    yield w
    yield workloads.make_dense("c", 2, 300, 2, 128, 128, 64, torch.bfloat16, 503, state_std=0.05)
    yield workloads.make_dense("a", 1, 128, 2, 64, 64, 64, torch.float32, 501, state_std=0.05)


def test_noalloc_matches_kda_chunk_fwd_on_consecutive_calls(kda):
    for w in _cases():
        t = to_device(w)
        common = dict(A_log=t["A_log"], dt_bias=t["dt_bias"], mode=w.mode,
                      lower_bound=w.lower_bound, initial_state=t["initial_state"],
                      cu_seqlens=t["cu_seqlens"], chunk_size=w.chunk_size)
        o_ref, s_ref = kda.kda_chunk_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"],
                                         output_final_state=True, **common)
        o = torch.full_like(o_ref, 777.0)
        st = torch.full_like(s_ref, 777.0)
        kda.kda_chunk_fwd_noalloc(t["q"], t["k"], t["v"], t["g"], t["beta"], o=o, final_state=st,
                                  **common)
        torch.cuda.synchronize()
        if w.cu_seqlens is not None:
            end = int(w.cu_seqlens[-1])
            assert torch.equal(o[:, end:], torch.full_like(o[:, end:], 777.0))
            o, o_ref = o[:, :end], o_ref[:, :end]
        check_o(o, o_ref.double().cpu().numpy(), w.q.dtype, what=f"o {w.name}")
        check_state(st, s_ref.double().cpu().numpy(), w.q.dtype, what=f"state {w.name}")


def test_noalloc_rejects_sizes_beyond_the_scratch(kda):
    # B=1, T=8192, H=4, K=V=128 needs about 3.8 KB per token and head, far above 16 MiB
    dev = "cuda"
    q = torch.zeros((1, 8192, 4, 128), device=dev, dtype=torch.bfloat16)
    beta = torch.zeros((1, 8192, 4), device=dev, dtype=torch.bfloat16)
    A_log = torch.zeros((4, 128), device=dev)
    o = torch.empty_like(q)
    with pytest.raises(kda.KdaError, match="KDA_NOALLOC_SCRATCH_BYTES"):
        kda.kda_chunk_fwd_noalloc(q, q, q, q, beta, A_log=A_log, o=o)
