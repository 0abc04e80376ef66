"""Host arithmetic of bench.py (CPU): the per-head-token algorithmic bytes and flops behind the
roofline fraction, and the comment-blind code digest that keeps a DRAM-traffic figure tied to
the kernel source it was captured from."""
import math

import bench


def test_algorithmic_bytes_per_head_token():
    # bf16 q, k, g (K each) and v (V) in, beta in, o (V) out
    assert bench.algorithmic_bytes_per_head_token(128, 128) == 3 * 256 + 256 + 2 + 256 == 1282
    assert bench.algorithmic_bytes_per_head_token(256, 256) == 2562
    # float32 inputs and gate
    assert bench.algorithmic_bytes_per_head_token(64, 64, 4, 4) == 4 * (2 * 64 + 64) + 4 * 64 + 4 + 4 * 64


def test_algorithmic_flops_per_head_token():
    # 6KV + 2K(C+16) + CK + CV + (C+1)V + C^2/3: 144,853 / 123,349 / 484,949 as tabulated for
    # K = V = 128 at C = 64 and 32, and K = V = 256 at C = 64
    assert math.floor(bench.algorithmic_flops_per_head_token(128, 128, 64)) == 144853
    assert math.floor(bench.algorithmic_flops_per_head_token(128, 128, 32)) == 123349
    assert math.floor(bench.algorithmic_flops_per_head_token(256, 256, 64)) == 484949


def test_code_digest_ignores_comments_only(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void f(float* x) {\n    x[0] = 1.f;  // one\n}\n")
    d0 = bench.kernel_code_digest(str(src))
    src.write_text("// a new header line\n__global__ void f(float* x) {\n\n    x[0] = 1.f;  // changed\n}\n")
    assert bench.kernel_code_digest(str(src)) == d0
    src.write_text("__global__ void f(float* x) {\n    x[0] = 2.f;\n}\n")
    assert bench.kernel_code_digest(str(src)) != d0


def test_traffic_only_for_its_workload():
    assert bench.fused_traffic_bytes("dense_bf16_b4_t2048_h16_d128") is None


def test_roofline_of_takes_the_slower_bound():
    import types

    class T:
        def __init__(self, n, es):
            self.n, self.es = n, es

        def numel(self):
            return self.n

        def element_size(self):
            return self.es

    w = types.SimpleNamespace(K=128, V=128, chunk_size=64, initial_state=None,
                              q=T(0, 2), g=T(0, 2), head_tokens=lambda: 1 << 20)
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    nbytes = 1282 * (1 << 20)
    flops = bench.algorithmic_flops_per_head_token(128, 128, 64) * (1 << 20)
    t = 1e-3
    r = bench.roofline_of(w, t, peaks)
    assert r["bytes"] == nbytes and r["bound"] == "hbm"
    assert math.isclose(r["frac"], nbytes / 6800e9 / t)
    assert math.isclose(r["tflops"], flops / t / 1e12)
    # with a much lower tensor peak the flops bound the time instead
    r2 = bench.roofline_of(w, t, {"hbm_gbs": 6800.0, "bf16_tflops": 10.0})
    assert r2["bound"] == "tensor" and math.isclose(r2["frac"], flops / 10e12 / t)
    # initial and final states count once each
    w.initial_state = T(4 * 128 * 128, 4)
    assert bench.roofline_of(w, t, peaks)["bytes"] == nbytes + 2 * 4 * 128 * 128 * 4


def test_path_of_follows_the_dispatch_rule():
    import types

    import torch

    def w(dtype, K, V, mode):
        return types.SimpleNamespace(q=torch.empty(0, dtype=dtype), K=K, V=V, mode=mode)

    assert bench.path_of(w(torch.bfloat16, 128, 128, 1)) == "fused"
    assert bench.path_of(w(torch.bfloat16, 128, 128, 2)) == "fused"
    assert bench.path_of(w(torch.bfloat16, 256, 256, 0)) == "two-pass"
    assert bench.path_of(w(torch.bfloat16, 256, 256, 2)) == "two-pass"
    assert bench.path_of(w(torch.bfloat16, 128, 256, 1)) == "two-pass"
    assert bench.path_of(w(torch.bfloat16, 64, 128, 1)) == "stage-by-stage"
    assert bench.path_of(w(torch.float32, 128, 128, 1)) == "stage-by-stage"
