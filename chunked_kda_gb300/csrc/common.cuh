// Device helpers shared by the KDA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// log2(e): converts the natural-log decay to base 2 before exp2 (FLA skill
// "fla-kda", "Safe gate numerical note": the RCP_LN2 conversion).
constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Natural-log per-token decay from the gate input (FLA skill "fla-kda",
// "Gate modes").  mode 0: pre-gated, a = g.  mode 1: safe in-kernel,
// a = lb * sigmoid(expA * (g + dt_bias)).  mode 2: in-kernel without the safe
// gate, a = -expA * softplus(g + dt_bias), unbounded below.  expA = exp(A_log)
// precomputed.
__device__ __forceinline__ float softplus_f(float x) {  // ln(1 + e^x) without overflow
    return x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}
__device__ __forceinline__ float gate_act(float g, float expA, float dtb, int mode, float lb) {
    if (mode == 0) return g;
    if (mode == 2) return -expA * softplus_f(g + dtb);
    float z = expA * (g + dtb);
    return lb / (1.0f + expf(-z));
}

// Where chunk slot `x` lives.  Chunks start at every sequence start and every C
// tokens after it.  Dense mode (cu == nullptr): slot = b * ceil(T / C) + c.
// Packed mode: slot = floor(bos_n / C) + n + c, an injective numbering
// (floor(b/C) + ceil(l/C) <= floor((b+l)/C) + 1), so a grid of
// floor(T_cap / C) + N + 1 slots covers every chunk without reading the
// offsets on the host.
struct ChunkMap {
    const int32_t* cu;
    int N;  // logical sequences (B in dense mode)
    int T;  // tokens per row (dense) or capacity (packed)
    int C;

    __host__ __device__ int n_slots() const {
        return cu ? (T / C + N + 1) : N * ((T + C - 1) / C);
    }
    // fills (n, first token, valid length); false if slot x is not a chunk
    __device__ bool map(int x, int& n, int& t0, int& len, int& bos, int& eos) const {
        if (!cu) {
            int per = (T + C - 1) / C;
            n = x / per;
            int c = x - n * per;
            bos = n * T;
            eos = bos + T;
            t0 = bos + c * C;
            len = min(C, eos - t0);
            return n < N && len > 0;
        }
        // largest n with floor(cu[n]/C) + n <= x
        int lo = 0, hi = N - 1, best = -1;
        while (lo <= hi) {
            int mid = (lo + hi) >> 1;
            int f = __ldg(cu + mid) / C + mid;
            if (f <= x) { best = mid; lo = mid + 1; } else { hi = mid - 1; }
        }
        if (best < 0) return false;
        n = best;
        bos = __ldg(cu + n);
        eos = __ldg(cu + n + 1);
        int c = x - (bos / C + n);
        t0 = bos + c * C;
        len = min(C, eos - t0);
        return len > 0;
    }
    // first slot of sequence n
    __device__ int first_slot(int n, int bos) const {
        return cu ? (bos / C + n) : n * ((T + C - 1) / C);
    }
};

}  // namespace kda
