// K7: token-sequential KDA forward (decode / short prefill).
//
// attention-gym PR #317 "Add fused recurrent_kda for decode and inference
// prefill", Agent note: one program per (sequence, head, value block) scans the
// tokens in order with its [K, BV] FP32 state block in registers and computes
// in FP32 whatever the input dtype; the gate is the per-token log2 decay.
//
// Per token t (rows d of S are key channels):
//   S[d, :] *= 2^gate_t[d];  r = S^T k_t;  S += beta_t k_t (v_t - r)^T;
//   o_t = S^T q_t / sqrt(K).
//
// Block = 8 warps.  Warp w owns rows [w*K/8, (w+1)*K/8); lane l owns BV/32
// consecutive value columns, so every state row is read and written with
// coalesced vector accesses.  The two reductions over d (r and o) are partial
// sums per thread, then across the 8 warps through shared memory.
#include "common.cuh"
#include "kda_internal.h"

namespace kda {

template <int VPT>
struct VecF;
template <>
struct VecF<1> { using T = float; };
template <>
struct VecF<2> { using T = float2; };
template <>
struct VecF<4> { using T = float4; };

template <int VPT>
__device__ __forceinline__ void ld_vec(const float* p, float* r) {
    if constexpr (VPT == 4) {
        float4 x = *reinterpret_cast<const float4*>(p);
        r[0] = x.x; r[1] = x.y; r[2] = x.z; r[3] = x.w;
    } else if constexpr (VPT == 2) {
        float2 x = *reinterpret_cast<const float2*>(p);
        r[0] = x.x; r[1] = x.y;
    } else {
        r[0] = *p;
    }
}

template <int VPT>
__device__ __forceinline__ void st_vec(float* p, const float* r) {
    if constexpr (VPT == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(r[0], r[1], r[2], r[3]);
    } else if constexpr (VPT == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(r[0], r[1]);
    } else {
        *p = r[0];
    }
}

template <typename InT, typename OutT, int K, int BV>
__global__ void __launch_bounds__(256) recurrent_kernel(
    const InT* __restrict__ q, const InT* __restrict__ k, const InT* __restrict__ v,
    const float* __restrict__ gate, const InT* __restrict__ beta, const float* h0, float* hT,
    const int32_t* __restrict__ cu, int T, int H, int V, OutT* __restrict__ o) {
    constexpr int RPW = K / 8;    // state rows per warp
    constexpr int VPT = BV / 32;  // value columns per lane
    __shared__ float s_q[K], s_k[K], s_dec[K];
    __shared__ float s_v[BV];
    __shared__ float s_red[8][BV];
    __shared__ float s_beta;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * BV;
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    long bos, eos;
    if (cu) { bos = __ldg(cu + n); eos = __ldg(cu + n + 1); }
    else    { bos = (long)n * T; eos = bos + T; }

    const size_t st_base = ((size_t)n * H + h) * (size_t)K * V;
    const int col = v0 + lane * VPT;
    float S[RPW][VPT];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        int d = warp * RPW + r;
        if (h0) ld_vec<VPT>(h0 + st_base + (size_t)d * V + col, S[r]);
        else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) S[r][j] = 0.f;
        }
    }
    const float scale = rsqrtf((float)K);

    for (long t = bos; t < eos; ++t) {
        __syncthreads();  // previous token's readers of s_* are done
        const size_t qk_off = ((size_t)t * H + h) * K;
        for (int i = tid; i < K; i += 256) {
            s_q[i] = to_f32(q[qk_off + i]);
            s_k[i] = to_f32(k[qk_off + i]);
            s_dec[i] = exp2f(__ldg(gate + qk_off + i));
        }
        const size_t v_off = ((size_t)t * H + h) * V + v0;
        for (int i = tid; i < BV; i += 256) s_v[i] = to_f32(v[v_off + i]);
        if (tid == 0) s_beta = to_f32(beta[(size_t)t * H + h]);
        __syncthreads();

        // decay, then partial r = S^T k over this warp's rows
        float part[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) part[j] = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int d = warp * RPW + r;
            const float dec = s_dec[d], kd = s_k[d];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                S[r][j] *= dec;
                part[j] = fmaf(S[r][j], kd, part[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) s_red[warp][lane * VPT + j] = part[j];
        __syncthreads();
        float u[VPT];
        const float bt = s_beta;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float rr = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) rr += s_red[w][lane * VPT + j];
            u[j] = bt * (s_v[lane * VPT + j] - rr);
        }
        __syncthreads();  // s_red is reused below

        // delta update, then partial o = S^T q
        float op[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) op[j] = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int d = warp * RPW + r;
            const float kd = s_k[d], qd = s_q[d];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                S[r][j] = fmaf(kd, u[j], S[r][j]);
                op[j] = fmaf(S[r][j], qd, op[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) s_red[warp][lane * VPT + j] = op[j];
        __syncthreads();
        for (int i = tid; i < BV; i += 256) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += s_red[w][i];
            o[v_off + i] = from_f32<OutT>(acc * scale);
        }
    }

    if (hT) {
        // every thread of this program has read its whole block (above), and no
        // other program touches these addresses, so hT may alias h0
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            int d = warp * RPW + r;
            st_vec<VPT>(hT + st_base + (size_t)d * V + col, S[r]);
        }
    }
}

template <typename InT, int K, int BV>
static cudaError_t launch_rec_t(const RecArgs& a) {
    dim3 grid(a.V / BV, a.H, a.N);
    if (a.o_f32)
        recurrent_kernel<InT, float, K, BV><<<grid, 256, 0, a.stream>>>(
            (const InT*)a.q, (const InT*)a.k, (const InT*)a.v, a.gate, (const InT*)a.beta, a.h0,
            a.hT, a.cu, a.T, a.H, a.V, (float*)a.o);
    else
        recurrent_kernel<InT, InT, K, BV><<<grid, 256, 0, a.stream>>>(
            (const InT*)a.q, (const InT*)a.k, (const InT*)a.v, a.gate, (const InT*)a.beta, a.h0,
            a.hT, a.cu, a.T, a.H, a.V, (InT*)a.o);
    return cudaGetLastError();
}

template <typename InT>
static cudaError_t launch_rec_k(const RecArgs& a) {
    // value block: at most 64 state floats per thread (K * BV / 256)
    switch (a.K) {
        case 64:
            return a.V >= 128 ? launch_rec_t<InT, 64, 128>(a) : launch_rec_t<InT, 64, 64>(a);
        case 128:
            return a.V >= 128 ? launch_rec_t<InT, 128, 128>(a) : launch_rec_t<InT, 128, 64>(a);
        case 256:
            return launch_rec_t<InT, 256, 64>(a);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_recurrent(const RecArgs& a) {
    if (a.N == 0) return cudaSuccess;
    return a.qkv_bf16 ? launch_rec_k<__nv_bfloat16>(a) : launch_rec_k<float>(a);
}

}  // namespace kda
