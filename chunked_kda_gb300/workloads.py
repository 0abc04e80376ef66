"""Seeded synthetic KDA forward workloads.

This module only draws random inputs; it holds none of the method's
arithmetic, so both the product side (bench.py, the binding's examples) and
the test side (the oracle comparisons) can take their inputs from it.

Recipes (every tensor is drawn in float32 from a ``torch.Generator`` seeded
with ``1000 + workload id`` on the requested device, then cast):

* q, k ~ N(0, 1), then divided by max(||row||, 1e-6) per (token, head) row;
  v ~ N(0, 1); beta = sigmoid(N(0, 1)) in the dtype of q.
* safe in-kernel gate: raw g ~ N(0, sigma_g) in the dtype of q,
  A_log ~ U(0, ln 16) and dt_bias ~ N(0, 0.5) as float32 [H, K], lower_bound -5.
* pre-gated: g = -U(0.01, 5) per token and channel (natural-log decay).
* non-safe in-kernel gate: g, A_log, dt_bias drawn as for the safe gate.
* recurrent decode: per-token log2 gate = log2(e) * (-U(0.01, 5)) in float32.
* initial states (where drawn): N(0, 0.05) float32 [N, H, K, V].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

GATE_PRE = 0
GATE_SAFE = 1
GATE_NONSAFE = 2


@dataclass
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    chunk_size: int
    mode: int
    lower_bound: float
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    A_log: Optional[torch.Tensor] = None
    dt_bias: Optional[torch.Tensor] = None
    initial_state: Optional[torch.Tensor] = None
    cu_seqlens: Optional[torch.Tensor] = None
    output_final_state: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def n_seqs(self) -> int:
        return self.B if self.cu_seqlens is None else int(self.cu_seqlens.numel()) - 1

    def head_tokens(self) -> int:
        """B*T*H for dense inputs, (sum of valid lengths)*H for packed ones."""
        if self.cu_seqlens is None:
            return self.B * self.T * self.H
        return int(self.cu_seqlens[-1].item()) * self.H

    def tensors(self):
        return {n: getattr(self, n) for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias",
                                              "initial_state", "cu_seqlens")}


# name -> (workload id, description); the ids seed the generators
WORKLOADS = {
    "tiny_fp32_b1_t128_h2_d64": 0,
    "dense_bf16_b4_t2048_h16_d128": 1,
    "varlen_bf16_n16_cap20480_h32_d128_c32": 2,
    "dense_bf16_b1_t8192_h96_d128": 3,
    "dense_bf16_b4_t4096_h64_d128": 3,
    "dense_bf16_b8_t2048_h32_d256": 4,
    # a smaller case of the dense workload for profiler captures: one CTA per SM
    # (152 sequence-heads), inputs (318 MB) still larger than L2
    "dense_bf16_b1_t2048_h152_d128": 6,
}


def _gen(device, seed):
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return gen


def _randn(shape, gen, device, std=1.0):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def _rand(shape, gen, device, lo, hi):
    return torch.rand(shape, generator=gen, device=device, dtype=torch.float32) * (hi - lo) + lo


def _unit_rows(x):
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)


def _qkvb(B, T, H, K, V, gen, device, dtype):
    q = _unit_rows(_randn((B, T, H, K), gen, device)).to(dtype)
    k = _unit_rows(_randn((B, T, H, K), gen, device)).to(dtype)
    v = _randn((B, T, H, V), gen, device).to(dtype)
    beta = torch.sigmoid(_randn((B, T, H), gen, device)).to(dtype)
    return q, k, v, beta


def make_dense(name, B, T, H, K, V, chunk_size, dtype, seed, device="cpu", g_std=1.0,
               state_std=None, mode=GATE_SAFE, lower_bound=-5.0, output_final_state=True):
    gen = _gen(device, seed)
    q, k, v, beta = _qkvb(B, T, H, K, V, gen, device, dtype)
    A_log = dt_bias = None
    if mode in (GATE_SAFE, GATE_NONSAFE):
        g = _randn((B, T, H, K), gen, device, g_std).to(dtype)
        A_log = _rand((H, K), gen, device, 0.0, math.log(16.0))
        dt_bias = _randn((H, K), gen, device, 0.5)
    else:
        g = (-_rand((B, T, H, K), gen, device, 0.01, 5.0)).to(dtype)
    S0 = None if state_std is None else _randn((B, H, K, V), gen, device, state_std)
    return Workload(name, B, T, H, K, V, chunk_size, mode, lower_bound, q, k, v, g, beta,
                    A_log, dt_bias, S0, None, output_final_state)


def varlen_lengths(n_slots, max_len, capacity, empty_slots, seed):
    """Lengths U[1, max_len] for the non-empty slots, redrawn until their sum < capacity."""
    gen = torch.Generator().manual_seed(seed)
    while True:
        lens = torch.randint(1, max_len + 1, (n_slots,), generator=gen)
        for e in empty_slots:
            lens[e] = 0
        if int(lens.sum()) < capacity:
            return [int(x) for x in lens]


def make_varlen(name, lengths, capacity, H, K, V, chunk_size, dtype, seed, device="cpu",
                mode=GATE_PRE, state_std=0.05, lower_bound=-5.0, poison_tail=True):
    """Packed layout [1, capacity, H, *]; the tail beyond the last offset is NaN-poisoned."""
    gen = _gen(device, seed)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    assert cu[-1] <= capacity
    q, k, v, beta = _qkvb(1, capacity, H, K, V, gen, device, dtype)
    A_log = dt_bias = None
    if mode in (GATE_SAFE, GATE_NONSAFE):
        g = _randn((1, capacity, H, K), gen, device).to(dtype)
        A_log = _rand((H, K), gen, device, 0.0, math.log(16.0))
        dt_bias = _randn((H, K), gen, device, 0.5)
    else:
        g = (-_rand((1, capacity, H, K), gen, device, 0.01, 5.0)).to(dtype)
    S0 = None if state_std is None else _randn((len(lengths), H, K, V), gen, device, state_std)
    if poison_tail and cu[-1] < capacity:
        for t in (q, k, v, g, beta):
            t[:, cu[-1]:] = float("nan")
    cu_t = torch.tensor(cu, dtype=torch.int32, device=device)
    return Workload(name, 1, capacity, H, K, V, chunk_size, mode, lower_bound, q, k, v, g, beta,
                    A_log, dt_bias, S0, cu_t, True)


def make(name, device="cpu"):
    """The named workloads (sizes in the name)."""
    if name == "tiny_fp32_b1_t128_h2_d64":
        return make_dense(name, 1, 128, 2, 64, 64, 64, torch.float32, 1000, device)
    if name == "dense_bf16_b4_t2048_h16_d128":
        return make_dense(name, 4, 2048, 16, 128, 128, 64, torch.bfloat16, 1001, device,
                          state_std=0.05)
    if name == "varlen_bf16_n16_cap20480_h32_d128_c32":
        lens = varlen_lengths(16, 2048, 20480, empty_slots=(0, 7), seed=1002)
        return make_varlen(name, lens, 20480, 32, 128, 128, 32, torch.bfloat16, 1002, device)
    if name == "dense_bf16_b1_t8192_h96_d128":
        return make_dense(name, 1, 8192, 96, 128, 128, 64, torch.bfloat16, 1003, device,
                          g_std=2.0)
    if name == "dense_bf16_b4_t4096_h64_d128":
        return make_dense(name, 4, 4096, 64, 128, 128, 64, torch.bfloat16, 1003, device,
                          g_std=2.0)
    if name == "dense_bf16_b4_t4096_h64_d128_nonsafe":
        return make_dense(name, 4, 4096, 64, 128, 128, 64, torch.bfloat16, 1003, device,
                          g_std=2.0, mode=GATE_NONSAFE)
    if name == "dense_bf16_b1_t2048_h152_d128":
        return make_dense(name, 1, 2048, 152, 128, 128, 64, torch.bfloat16, 1006, device,
                          g_std=2.0)
    if name == "dense_bf16_b1_t2048_h152_d128_nonsafe":
        return make_dense(name, 1, 2048, 152, 128, 128, 64, torch.bfloat16, 1006, device,
                          g_std=2.0, mode=GATE_NONSAFE)
    if name == "dense_bf16_b2_t2048_h32_d256":  # a quarter of the D = 256 workload (profiling)
        return make_dense(name, 2, 2048, 32, 256, 256, 64, torch.bfloat16, 1007, device,
                          g_std=2.0)
    if name == "dense_bf16_b8_t2048_h32_d256_nonsafe":
        return make_dense(name, 8, 2048, 32, 256, 256, 64, torch.bfloat16, 1004, device,
                          g_std=2.0, mode=GATE_NONSAFE)
    if name == "dense_bf16_b8_t2048_h32_d256":
        return make_dense(name, 8, 2048, 32, 256, 256, 64, torch.bfloat16, 1004, device,
                          g_std=2.0)
    raise KeyError(name)


@dataclass
class DecodeStep:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    gate: torch.Tensor
    beta: torch.Tensor


def decode_state(n_seqs=512, H=32, K=128, V=128, device="cpu", seed=1005):
    gen = _gen(device, seed)
    return _randn((n_seqs, H, K, V), gen, device, 0.05)


def decode_step(step, n_seqs=512, H=32, K=128, V=128, dtype=torch.bfloat16, device="cpu",
                seed=1005):
    """Fresh packed one-token-per-sequence inputs for decode step ``step``."""
    gen = _gen(device, seed * 100003 + step + 1)
    q, k, v, beta = _qkvb(1, n_seqs, H, K, V, gen, device, dtype)
    gate = -_rand((1, n_seqs, H, K), gen, device, 0.01, 5.0) * (1.0 / math.log(2.0))
    return DecodeStep(q, k, v, gate, beta)


def decode_cu_seqlens(n_seqs=512, device="cpu"):
    return torch.arange(n_seqs + 1, dtype=torch.int32, device=device)
