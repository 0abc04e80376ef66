"""The tensor-core kernels' bounded waits (the fused kernel and the two-pass state chain): a
wait that nothing completes gives up after its limit, the other waits of the CTA stop (at once
in the fused kernel, at their own limits in the chain), the launch takes its abort path (no MMAs or copies left in flight, TMEM freed), the host reads
the count, and the CUDA context stays usable.  The failure is made by the kernels' test hook
(an mbarrier that nothing arrives on), never by a fault, trap or hang."""
import pytest
import torch

from chunked_kda_gb300 import workloads
from test_gpu_chunk import compare, kda, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def test_normal_runs_count_no_timeouts():
    w = workloads.make_dense("t", 1, 200, 2, 128, 128, 64, torch.bfloat16, 61, state_std=0.05)
    kda().kda_fused_wait_timeouts(reset=True)
    o, st = run_gpu(w)
    assert kda().kda_fused_wait_timeouts() == 0
    compare(w, o, st)


@pytest.mark.parametrize("chunk", [0, 2])
def test_wait_gives_up_and_the_context_stays_usable(chunk):
    """The give-up reaches the caller without a host synchronisation in the library: the
    status word of kda_chunk_fwd_ex gets bit 0 on the device, read after the caller's own
    stream sync; the per-device counter agrees."""
    w = workloads.make_dense("t", 1, 260, 2, 128, 128, 64, torch.bfloat16, 62, state_std=0.05)
    kda().kda_fused_wait_timeouts(reset=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda().kda_test_hooks(wait_timeout_chunk=chunk)
    try:
        run_gpu(w, status=status)  # the launch itself succeeds; its outputs are not valid
    finally:
        kda().kda_test_hooks()
    assert int(status.item()) & 1 == 1
    assert kda().kda_fused_wait_timeouts(reset=True) >= 2  # both CTAs gave up a wait
    status.zero_()
    o, st = run_gpu(w, status=status)  # the same context: a normal call matches the oracle
    assert int(status.item()) == 0
    assert kda().kda_fused_wait_timeouts() == 0
    compare(w, o, st)


@pytest.mark.parametrize("chunk", [0, 3])
def test_two_pass_wait_gives_up_and_the_context_stays_usable(chunk):
    """The same on the K = V = 256 two-pass path: the chain's issuing warp gives up at the
    chunk, every chain CTA (2 heads x 2 value blocks) counts one give-up, and a normal call in
    the same context matches the oracle."""
    w = workloads.make_dense("t", 1, 300, 2, 256, 256, 64, torch.bfloat16, 63, state_std=0.05)
    kda().kda_fused_wait_timeouts(reset=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda().kda_test_hooks(wait_timeout_chunk=chunk)
    try:
        run_gpu(w, status=status)
    finally:
        kda().kda_test_hooks()
    assert int(status.item()) & 1 == 1
    assert kda().kda_fused_wait_timeouts(reset=True) >= 4
    status.zero_()
    o, st = run_gpu(w, status=status)
    assert int(status.item()) == 0
    assert kda().kda_fused_wait_timeouts() == 0
    compare(w, o, st)
