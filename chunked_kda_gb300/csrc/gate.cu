// K1 standalone: gate activation + chunk-local inclusive cumsum in log2 units.
//
// FLA skill "fla-kda", "Gate modes" (pre-gated, safe and non-safe in-kernel
// activations) and "Safe gate numerical note" (RCP_LN2 conversion before
// exp2); attention-gym PR #317, Agent note (bounded_gate_cumsum with
// chunk_size = 1 is the per-token log2 gate of the recurrent entry point).
//
// One block per (chunk slot, 1024 consecutive (head, channel) pairs): each thread owns 8
// consecutive channels, loads them as one 16-byte vector (bf16; two for float32) per token and
// stores their sums as two 16-byte vectors, so a warp moves 256 channels of a token with fully
// used 128-byte lines.  The chunk's tokens are walked in order, four at a time with their loads
// issued together.  A row of H * K channels that is not a multiple of 8 takes the scalar kernel
// (one channel per thread).  The chunked forward fuses this step into its own kernels; this
// entry point serves standalone callers and the recurrent path.
#include "common.cuh"
#include "kda_internal.h"

namespace kda {

// 8 values of g from one token row (16-byte aligned)
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <typename InT>
__global__ void __launch_bounds__(128) gate_cumsum_vec8_kernel(
    const InT* __restrict__ g, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
    int mode, float lb, ChunkMap cm, int HK, float* __restrict__ out) {
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int c0 = 8 * (blockIdx.y * 128 + threadIdx.x);  // the thread's first channel
    if (c0 >= HK) return;
    float expA[8], dtb[8], acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        expA[e] = (mode != 0) ? expf(__ldg(A_log + c0 + e)) : 0.f;
        dtb[e] = (mode != 0 && dt_bias) ? __ldg(dt_bias + c0 + e) : 0.f;
        acc[e] = 0.f;
    }
    const size_t base = (size_t)t0 * HK + c0;
    auto emit = [&](int i, const float (&x)[8]) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            acc[e] += gate_act(x[e], expA[e], dtb[e], mode, lb);
            y[e] = acc[e] * kLog2e;
        }
        float4* o = reinterpret_cast<float4*>(out + base + (size_t)i * HK);
        o[0] = make_float4(y[0], y[1], y[2], y[3]);
        o[1] = make_float4(y[4], y[5], y[6], y[7]);
    };
    int i = 0;
    for (; i + 4 <= len; i += 4) {
        float x[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) load8(g + base + (size_t)(i + u) * HK, x[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) emit(i + u, x[u]);
    }
    for (; i < len; ++i) {
        float x[8];
        load8(g + base + (size_t)i * HK, x);
        emit(i, x);
    }
}

template <typename InT>
__global__ void __launch_bounds__(128) gate_cumsum_kernel(
    const InT* __restrict__ g, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
    int mode, float lb, ChunkMap cm, int HK, float* __restrict__ out) {
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    int hk = blockIdx.y * 128 + threadIdx.x;
    if (hk >= HK) return;
    float expA = (mode != 0) ? expf(__ldg(A_log + hk)) : 0.f;
    float dtb = (mode != 0 && dt_bias) ? __ldg(dt_bias + hk) : 0.f;
    float acc = 0.f;
    size_t idx = (size_t)t0 * HK + hk;
    for (int i = 0; i < len; ++i, idx += HK) {
        acc += gate_act(to_f32(g[idx]), expA, dtb, mode, lb);
        out[idx] = acc * kLog2e;
    }
}

cudaError_t launch_gate(const GateArgs& a) {
    ChunkMap cm{a.cu, a.N, a.T, a.C};
    const int HK = a.H * a.K;
    if (cm.n_slots() == 0) return cudaSuccess;
    const bool aligned = ((uintptr_t)a.g & 15u) == 0 && ((uintptr_t)a.out & 15u) == 0;
    if (HK % 8 == 0 && aligned) {  // 16-byte vectors of 8 channels
        const dim3 grid(cm.n_slots(), (HK / 8 + 127) / 128);
        if (a.g_bf16)
            gate_cumsum_vec8_kernel<__nv_bfloat16><<<grid, 128, 0, a.stream>>>(
                (const __nv_bfloat16*)a.g, a.A_log, a.dt_bias, a.mode, a.lb, cm, HK, a.out);
        else
            gate_cumsum_vec8_kernel<float><<<grid, 128, 0, a.stream>>>(
                (const float*)a.g, a.A_log, a.dt_bias, a.mode, a.lb, cm, HK, a.out);
        return cudaGetLastError();
    }
    const dim3 grid(cm.n_slots(), (HK + 127) / 128);
    if (a.g_bf16)
        gate_cumsum_kernel<__nv_bfloat16><<<grid, 128, 0, a.stream>>>(
            (const __nv_bfloat16*)a.g, a.A_log, a.dt_bias, a.mode, a.lb, cm, HK, a.out);
    else
        gate_cumsum_kernel<float><<<grid, 128, 0, a.stream>>>(
            (const float*)a.g, a.A_log, a.dt_bias, a.mode, a.lb, cm, HK, a.out);
    return cudaGetLastError();
}

}  // namespace kda
