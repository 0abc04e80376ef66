// K1 standalone: gate activation + chunk-local inclusive cumsum in log2 units.
//
// FLA skill "fla-kda", "Gate modes" (pre-gated, safe and non-safe in-kernel
// activations) and "Safe gate numerical note" (RCP_LN2 conversion before
// exp2); attention-gym PR #317, Agent note (bounded_gate_cumsum with
// chunk_size = 1 is the per-token log2 gate of the recurrent entry point).
//
// One block per (chunk slot, 128 consecutive (head, channel) pairs).  Each
// thread walks the chunk's tokens in order; for every token the block reads
// 128 consecutive channels, so loads and stores are coalesced.  The chunked
// forward fuses this step into its own kernel; this entry point serves
// standalone callers and the recurrent path.
#include "common.cuh"
#include "kda_internal.h"

namespace kda {

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
    int HK = a.H * a.K;
    dim3 grid(cm.n_slots(), (HK + 127) / 128);
    if (grid.x == 0) return cudaSuccess;
    if (a.g_bf16)
        gate_cumsum_kernel<__nv_bfloat16><<<grid, 128, 0, a.stream>>>(
            (const __nv_bfloat16*)a.g, a.A_log, a.dt_bias, a.mode, a.lb, cm, HK, a.out);
    else
        gate_cumsum_kernel<float><<<grid, 128, 0, a.stream>>>(
            (const float*)a.g, a.A_log, a.dt_bias, a.mode, a.lb, cm, HK, a.out);
    return cudaGetLastError();
}

}  // namespace kda
