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
// Block = 8 warps.  Warp w owns rows [w*KP/8, (w+1)*KP/8) (KP = K rounded up
// to 64, 128 or 256, rows beyond K masked); lane l owns BV/32 consecutive value
// columns (columns beyond V masked), so every state row is read and written
// with coalesced vector accesses.  The two reductions over d (r and o) are
// partial sums per thread, then across the 8 warps through shared memory.
//
// Decode-side preprocessing (attention-gym PR #317 test plan; FLA skill
// "fla-kda", "Correctness checklist"): the gate may be given raw and activated
// here (pre-gated, safe or non-safe mode, as in the chunked path), the q and k
// rows may be l2-normalised here and beta may be given as logits.
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

// flags of the preprocessing (the values of KDA_FLAG_Q_L2NORM, KDA_FLAG_K_L2NORM and
// KDA_FLAG_BETA_LOGITS in include/kda.h)
constexpr unsigned kRecQNorm = 1u, kRecKNorm = 2u, kRecBetaLogits = 4u;

// KP: K rounded up to 64, 128 or 256 (rows d >= K are masked); BV: value columns per program
// (columns >= V are masked).  MASKED = false when K == KP and BV divides V: no row or column
// checks, whole-vector state accesses.  PREP = false: the gate is the per-token log2 decay
// and no flag is set (the plain decode step), so no activation or normalisation code.
// mode: 0 pre-gated natural-log decay, 1 safe, 2 non-safe, 3 the per-token log2 decay.
template <typename InT, typename GT, typename OutT, int KP, int BV, bool MASKED, bool PREP>
__global__ void __launch_bounds__(256, 2) recurrent_kernel(  // two programs per SM keep HBM busy
    const InT* __restrict__ q, const InT* __restrict__ k, const InT* __restrict__ v,
    const GT* __restrict__ gate, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
    int mode, float lb, const InT* __restrict__ beta, const float* h0, float* hT,
    const int32_t* __restrict__ cu, int T, int H, int hr, int K, int V, unsigned flags,
    OutT* __restrict__ o) {
    constexpr int RPW = KP / 8;   // state rows per warp
    constexpr int VPT = BV / 32;  // value columns per lane
    static_assert(KP <= 256, "one element of q, k per thread");
    __shared__ float s_q[KP], s_k[KP], s_dec[KP], s_expA[KP], s_dtb[KP];
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

    if (PREP && tid < KP) {
        const bool in = tid < K && (mode == 1 || mode == 2);
        s_expA[tid] = in ? expf(__ldg(A_log + (size_t)h * K + tid)) : 0.f;
        s_dtb[tid] = (in && dt_bias) ? __ldg(dt_bias + (size_t)h * K + tid) : 0.f;
    }
    const size_t st_base = ((size_t)n * H + h) * (size_t)K * V;
    const int Hq = H / hr, hq = h / hr;  // query / key heads, and the one of this value head
    const int col = v0 + lane * VPT;
    // whole vectors of VPT columns when the rows allow it, else one column at a time
    const bool vec = !MASKED || ((V % VPT) == 0 && col + VPT <= V);
    float S[RPW][VPT];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int d = warp * RPW + r;
        if constexpr (!MASKED) {
            if (h0) ld_vec<VPT>(h0 + st_base + (size_t)d * V + col, S[r]);
            else {
#pragma unroll
                for (int j = 0; j < VPT; ++j) S[r][j] = 0.f;
            }
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) S[r][j] = 0.f;
            if (h0 && d < K) {
                const float* src = h0 + st_base + (size_t)d * V + col;
                if (vec) ld_vec<VPT>(src, S[r]);
                else {
#pragma unroll
                    for (int j = 0; j < VPT; ++j)
                        if (col + j < V) S[r][j] = src[j];
                }
            }
        }
    }
    const float scale = rsqrtf((float)K);

    for (long t = bos; t < eos; ++t) {
        __syncthreads();  // previous token's readers of s_* are done
        const size_t qk_off = ((size_t)t * Hq + hq) * K;  // query / key head h / hr
        const size_t g_off = ((size_t)t * H + h) * K;
        float qv = 0.f, kv = 0.f;
        if (tid < KP) {
            float dec = 1.f;
            if (tid < K) {
                qv = to_f32(q[qk_off + tid]);
                kv = to_f32(k[qk_off + tid]);
                const float gv = to_f32(gate[g_off + tid]);
                if constexpr (PREP)
                    dec = (mode == 3) ? exp2f(gv) : expf(gate_act(gv, s_expA[tid], s_dtb[tid], mode, lb));
                else
                    dec = exp2f(gv);
            }
            s_dec[tid] = dec;
        }
        if (PREP && (flags & (kRecQNorm | kRecKNorm))) {  // sums of squares of the q and k rows
            float sq = qv * qv, sk = kv * kv;
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, m);
                sk += __shfl_xor_sync(0xffffffffu, sk, m);
            }
            if (lane == 0) { s_red[warp][0] = sq; s_red[warp][1] = sk; }
            __syncthreads();
            float tq = 0.f, tk = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) { tq += s_red[w][0]; tk += s_red[w][1]; }
            if (flags & kRecQNorm) qv *= rsqrtf(tq + kQNormEps);
            if (flags & kRecKNorm) kv *= rsqrtf(tk + kQNormEps);
        }
        if (tid < KP) { s_q[tid] = qv; s_k[tid] = kv; }
        const size_t v_off = ((size_t)t * H + h) * V + v0;
        for (int i = tid; i < BV; i += 256) s_v[i] = (!MASKED || v0 + i < V) ? to_f32(v[v_off + i]) : 0.f;
        if (tid == 0) {
            const float b = to_f32(beta[(size_t)t * H + h]);
            s_beta = (PREP && (flags & kRecBetaLogits)) ? 1.f / (1.f + expf(-b)) : b;
        }
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
            if (!MASKED || v0 + i < V) o[v_off + i] = from_f32<OutT>(acc * scale);
        }
    }

    if (hT) {
        // every thread of this program has read its whole block (above), and no
        // other program touches these addresses, so hT may alias h0
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int d = warp * RPW + r;
            if (MASKED && d >= K) continue;
            float* dst = hT + st_base + (size_t)d * V + col;
            if (vec) st_vec<VPT>(dst, S[r]);
            else {
#pragma unroll
                for (int j = 0; j < VPT; ++j)
                    if (col + j < V) dst[j] = S[r][j];
            }
        }
    }
}

template <typename InT, typename GT, typename OutT, int KP, int BV, bool MASKED, bool PREP>
static cudaError_t launch_rec_p(const RecArgs& a) {
    dim3 grid((a.V + BV - 1) / BV, a.H, a.N);
    recurrent_kernel<InT, GT, OutT, KP, BV, MASKED, PREP><<<grid, 256, 0, a.stream>>>(
        (const InT*)a.q, (const InT*)a.k, (const InT*)a.v, (const GT*)a.gate, a.A_log, a.dt_bias,
        a.mode, a.lb, (const InT*)a.beta, a.h0, a.hT, a.cu, a.T, a.H, a.Hk > 0 ? a.H / a.Hk : 1, a.K,
        a.V, a.flags, (OutT*)a.o);
    return cudaGetLastError();
}

template <typename InT, typename GT, typename OutT, int KP, int BV, bool MASKED>
static cudaError_t launch_rec_m(const RecArgs& a) {
    if (a.mode == 3 && a.flags == 0) return launch_rec_p<InT, GT, OutT, KP, BV, MASKED, false>(a);
    return launch_rec_p<InT, GT, OutT, KP, BV, MASKED, true>(a);
}

template <typename InT, typename GT, int KP, int BV>
static cudaError_t launch_rec_t(const RecArgs& a) {
    const bool masked = a.K != KP || a.V % BV != 0;
    if (a.o_f32)
        return masked ? launch_rec_m<InT, GT, float, KP, BV, true>(a)
                      : launch_rec_m<InT, GT, float, KP, BV, false>(a);
    return masked ? launch_rec_m<InT, GT, InT, KP, BV, true>(a)
                  : launch_rec_m<InT, GT, InT, KP, BV, false>(a);
}

template <typename InT, typename GT>
static cudaError_t launch_rec_k(const RecArgs& a) {
    // value block: at most 64 state floats per thread (KP * BV / 256)
    if (a.K <= 64) return a.V > 64 ? launch_rec_t<InT, GT, 64, 128>(a) : launch_rec_t<InT, GT, 64, 64>(a);
    if (a.K <= 128) return a.V > 64 ? launch_rec_t<InT, GT, 128, 128>(a) : launch_rec_t<InT, GT, 128, 64>(a);
    if (a.K <= 256) return launch_rec_t<InT, GT, 256, 64>(a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_recurrent(const RecArgs& a) {
    if (a.N == 0) return cudaSuccess;
    if (a.qkv_bf16)
        return a.gate_bf16 ? launch_rec_k<__nv_bfloat16, __nv_bfloat16>(a) : launch_rec_k<__nv_bfloat16, float>(a);
    return a.gate_bf16 ? launch_rec_k<float, __nv_bfloat16>(a) : launch_rec_k<float, float>(a);
}

}  // namespace kda
