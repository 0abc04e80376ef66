// Chunked KDA forward, float32 stage-by-stage path, one kernel per step.
//
// This path computes every step in FP32 with FFMA, so it meets float32-input
// accuracy (tensor-core bf16/tf32 operands would not), and it serves as the
// stage-by-stage form of the chunked algorithm.  The exceptions: with bf16 inputs
// the safe gate's scores, the WY step and the output step run their products on
// the tensor cores with tf32 operands (10-bit mantissa, FP32 accumulation), far
// inside the bf16-input tolerance.  Steps and their sources:
//   a1 gate + chunk-local log2 cumsum   FLA skill "fla-kda", "Gate modes" and
//                                       "Safe gate numerical note" (RCP_LN2)
//   a2 causal scores Akk, Aqk           Helion PR #3290 "Read only the causal
//                                       columns in chunk_fwd_A_diag_anchored"
//   a3 T = (I + Akk)^-1                 FLA skill "fla-kda", "Safe gate
//                                       numerical note" (masked lower-triangular
//                                       solve)
//   a4 w = T (beta k 2^G), u = T (beta v)   FLA skill "fla-kda", "Public code
//                                       map" (recompute_w_u_fwd)
//   a5 v_new = u - w h; h <- 2^Glast h + (k 2^(Glast-G))^T v_new  (state scan)
//   a6 o = s (q 2^G) h + Aqk v_new      attention-gym PR #345 (output kernel)
// Every exp2 here has a non-positive argument (G is non-increasing inside a
// chunk under the bounded-gate contract), so no offsets are needed: each
// decay factor 2^(G_i - G_j), j <= i, is evaluated directly.
//
// Workspace (float32, token-indexed like the inputs; T_tot = B * T):
//   G [T_tot,H,K] | Akk [T_tot,H,C] | Aqk [T_tot,H,C] | Tm [T_tot,H,C] |
//   w [T_tot,H,K] | u [T_tot,H,V] | v_new [T_tot,H,V] | h [slots,H,K,V]
#include <type_traits>

#include "common.cuh"
#include "kda_internal.h"
#include "sm100.cuh"

namespace kda {

// row of query / key head for value head h at token t: Hk = H / hr query / key heads, value
// head h reads head h / hr (grouped value heads; hr = 1 is multi-head)
__device__ __forceinline__ size_t qk_row(long t, int h, int H, int hr) {
    return (size_t)t * (size_t)(H / hr) + (size_t)(h / hr);
}
namespace {

constexpr int DT = 32;  // channel tile

struct PreciseWs {
    float *G, *Akk, *Aqk, *Tm, *w, *u, *vn, *hc;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PreciseWs carve(void* base, int B, int T, int H, int K, int V, int C, int slots, size_t* total) {
    size_t tt = (size_t)B * T * H;
    size_t sizes[8] = {tt * K, tt * C, tt * C, tt * C, tt * K, tt * V, tt * V,
                       (size_t)slots * H * K * V};
    float* ptrs[8];
    size_t off = 0;
    for (int i = 0; i < 8; ++i) {
        ptrs[i] = base ? (float*)((char*)base + off) : nullptr;
        off += align256(sizes[i] * sizeof(float));
    }
    if (total) *total = off;
    return PreciseWs{ptrs[0], ptrs[1], ptrs[2], ptrs[3], ptrs[4], ptrs[5], ptrs[6], ptrs[7]};
}

// a2: Akk[i,j] = beta_i sum_d k_i k_j 2^(G_i-G_j) (j<i); Aqk[i,j] = s sum_d q_i k_j 2^(G_i-G_j) (j<=i)
template <typename InT, int C>
__global__ void __launch_bounds__(256) scores_kernel(const InT* __restrict__ q,
                                                     const InT* __restrict__ k,
                                                     const InT* __restrict__ beta,
                                                     const float* __restrict__ G, ChunkMap cm,
                                                     int H, int hr, int K, float* __restrict__ Akk,
                                                     float* __restrict__ Aqk) {
    constexpr int PM = C * C / 256;
    __shared__ float qs[C][DT + 1], ks[C][DT + 1], gs[C][DT + 1];
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, tid = threadIdx.x;
    float akk[PM], aqk[PM];
#pragma unroll
    for (int m = 0; m < PM; ++m) akk[m] = aqk[m] = 0.f;
    for (int d0 = 0; d0 < K; d0 += DT) {
        __syncthreads();
        for (int idx = tid; idx < C * DT; idx += 256) {
            int i = idx / DT, dd = idx % DT;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (i < len) {
                size_t off = ((size_t)(t0 + i) * H + h) * K + d0 + dd;
                size_t qo = qk_row(t0 + i, h, H, hr) * K + d0 + dd;
                qv = to_f32(q[qo]);
                kv = to_f32(k[qo]);
                gv = G[off];
            }
            qs[i][dd] = qv;
            ks[i][dd] = kv;
            gs[i][dd] = gv;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < PM; ++m) {
            int p = tid + 256 * m, i = p / C, j = p % C;
            if (j <= i && i < len) {
                float a1 = 0.f, a2 = 0.f;
#pragma unroll 8
                for (int dd = 0; dd < DT; ++dd) {
                    float e = exp2f(gs[i][dd] - gs[j][dd]);
                    float kj = ks[j][dd] * e;
                    a1 = fmaf(ks[i][dd], kj, a1);
                    a2 = fmaf(qs[i][dd], kj, a2);
                }
                akk[m] += a1;
                aqk[m] += a2;
            }
        }
    }
    const float scale = rsqrtf((float)K);
#pragma unroll
    for (int m = 0; m < PM; ++m) {
        int p = tid + 256 * m, i = p / C, j = p % C;
        if (i < len) {
            size_t off = ((size_t)(t0 + i) * H + h) * C + j;
            float bi = to_f32(beta[(size_t)(t0 + i) * H + h]);
            Akk[off] = (j < i) ? bi * akk[m] : 0.f;
            Aqk[off] = (j <= i) ? scale * aqk[m] : 0.f;
        }
    }
}

// a2 for the safe gate, whose per-token decay is bounded (lb >= -5: at most 5 / ln 2 in log2
// units per token): the pairwise factor 2^(G_i - G_j) split at the midpoint m of row i's
// 16-row sub-block, as in the fused kernel (Helion PR #3290, "chunk_fwd_A_diag_anchored"):
// rows k_i 2^(G_i - G_m), q_i 2^(G_i - G_m) (|exponent| <= 16 * 5 / ln 2), columns
// k_j 2^(G_m - G_j) per sub-block anchor; then plain products.  Thread: column j, rows
// r0 + RS m (their sub-block is known at compile time); the scaled row tiles are read as
// float4, broadcast to the warp.
template <typename InT, int C>
__global__ void __launch_bounds__(256) scores_anchored_kernel(const InT* __restrict__ q,
                                                              const InT* __restrict__ k,
                                                              const InT* __restrict__ beta,
                                                              const float* __restrict__ G,
                                                              ChunkMap cm, int H, int hr, int K,
                                                              float* __restrict__ Akk,
                                                              float* __restrict__ Aqk) {
    constexpr int NB = C / 16, DA = 16, PM = C * C / 256, RS = 256 / C;
    static_assert(RS * PM == C && 16 % RS == 0, "pair layout");
    __shared__ __align__(16) float krs[C][DA];
    __shared__ __align__(16) float qrs[C][DA];
    __shared__ float ksm[C][DA + 1], gsm[C][DA + 1];
    __shared__ float kcs[NB][C][DA + 1];
    __shared__ float gm[NB][DA];
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, tid = threadIdx.x;
    const int j = tid % C, r0 = tid / C;
    float a1[PM], a2[PM];
#pragma unroll
    for (int m = 0; m < PM; ++m) a1[m] = a2[m] = 0.f;
    for (int d0 = 0; d0 < K; d0 += DA) {
        __syncthreads();
        for (int idx = tid; idx < C * DA; idx += 256) {
            const int i = idx / DA, dd = idx % DA;
            float kv = 0.f, qv = 0.f, gv = 0.f;
            if (i < len) {
                const size_t qo = qk_row(t0 + i, h, H, hr) * K + d0 + dd;
                kv = to_f32(k[qo]);
                qv = to_f32(q[qo]);
                gv = G[((size_t)(t0 + i) * H + h) * K + d0 + dd];
            }
            ksm[i][dd] = kv;
            gsm[i][dd] = gv;
            qrs[i][dd] = qv;
        }
        __syncthreads();
        if (tid < NB * DA) {  // anchors: the sub-block's midpoint row, or its last valid row
            const int b = tid / DA, dd = tid % DA;
            gm[b][dd] = (16 * b < len) ? gsm[min(16 * b + 8, len - 1)][dd] : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < C * DA; idx += 256) {
            const int i = idx / DA, dd = idx % DA;
            const float e = (i < len) ? exp2f(gsm[i][dd] - gm[i / 16][dd]) : 0.f;
            krs[i][dd] = ksm[i][dd] * e;
            qrs[i][dd] *= e;
        }
        for (int idx = tid; idx < NB * C * DA; idx += 256) {
            const int b = idx / (C * DA), jj = (idx / DA) % C, dd = idx % DA;
            kcs[b][jj][dd] = (jj < 16 * (b + 1) && jj < len)
                                 ? ksm[jj][dd] * exp2f(gm[b][dd] - gsm[jj][dd]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int dd = 0; dd < DA; dd += 4) {
            float kc[NB][4];
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) kc[b][e] = kcs[b][j][dd + e];
#pragma unroll
            for (int m = 0; m < PM; ++m) {
                const int i = r0 + RS * m, b = (RS * m) / 16;
                const float4 kr = *reinterpret_cast<const float4*>(&krs[i][dd]);
                const float4 qr = *reinterpret_cast<const float4*>(&qrs[i][dd]);
                a1[m] = fmaf(kr.x, kc[b][0], a1[m]);
                a1[m] = fmaf(kr.y, kc[b][1], a1[m]);
                a1[m] = fmaf(kr.z, kc[b][2], a1[m]);
                a1[m] = fmaf(kr.w, kc[b][3], a1[m]);
                a2[m] = fmaf(qr.x, kc[b][0], a2[m]);
                a2[m] = fmaf(qr.y, kc[b][1], a2[m]);
                a2[m] = fmaf(qr.z, kc[b][2], a2[m]);
                a2[m] = fmaf(qr.w, kc[b][3], a2[m]);
            }
        }
    }
    const float scale = rsqrtf((float)K);
#pragma unroll
    for (int m = 0; m < PM; ++m) {
        const int i = r0 + RS * m;
        if (i < len) {
            const size_t off = ((size_t)(t0 + i) * H + h) * C + j;
            const float bi = to_f32(beta[(size_t)(t0 + i) * H + h]);
            Akk[off] = (j < i) ? bi * a1[m] : 0.f;
            Aqk[off] = (j <= i) ? scale * a2[m] : 0.f;
        }
    }
}

// a4 for bf16 inputs: [w | u] = T [beta k 2^G | beta v] with m16n8k8 tf32 MMAs (FP32
// accumulation).  One block of 256 threads per (chunk slot, head); T (rows past the end zero)
// stays in shared memory and in the A fragments of each warp; the K + V columns go in passes of
// NB, each staged as rows of beta k 2^G or beta v (zero past the end).  Warp w owns rows
// 16 (w % WM) .. + 15 and NB / WN columns of each pass.  Fragment layout as in out_tc_kernel.
template <int C>
__global__ void __launch_bounds__(256) wu_tc_kernel(const __nv_bfloat16* __restrict__ k,
                                                    const __nv_bfloat16* __restrict__ v,
                                                    const __nv_bfloat16* __restrict__ beta,
                                                    const float* __restrict__ G,
                                                    const float* __restrict__ Tm, ChunkMap cm, int H,
                                                    int hr, int K, int V, float* __restrict__ w,
                                                    float* __restrict__ u) {
    using namespace sm100;
    constexpr int WM = C / 16, WN = 8 / WM, NB = 64, NT = NB / (8 * WN);
    constexpr int LA = C + 4, LB = NB + 8;
    __shared__ __align__(16) float Ts[C][LA];
    __shared__ __align__(16) float Xs[C][LB];
    __shared__ float bs[C];
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, tid = threadIdx.x, wp = tid >> 5, l = tid & 31;
    const int g = l >> 2, t = l & 3;
    const int r0 = 16 * (wp % WM), c0 = (wp / WM) * (NB / WN);
    for (int idx = tid; idx < C * C; idx += 256) {
        const int i = idx / C, j = idx % C;
        Ts[i][j] = (i < len) ? Tm[((size_t)(t0 + i) * H + h) * C + j] : 0.f;
    }
    for (int i = tid; i < C; i += 256) bs[i] = (i < len) ? __bfloat162float(beta[(size_t)(t0 + i) * H + h]) : 0.f;
    __syncthreads();
    uint32_t a[C / 8][4];
#pragma unroll
    for (int ks = 0; ks < C / 8; ++ks) {
        const int k0 = 8 * ks;
        a[ks][0] = to_tf32(Ts[r0 + g][k0 + t]);
        a[ks][1] = to_tf32(Ts[r0 + g + 8][k0 + t]);
        a[ks][2] = to_tf32(Ts[r0 + g][k0 + t + 4]);
        a[ks][3] = to_tf32(Ts[r0 + g + 8][k0 + t + 4]);
    }
#pragma unroll 1
    for (int col0 = 0; col0 < K + V; col0 += NB) {  // K is a multiple of NB: no pass straddles it
        const bool isk = col0 < K;
        __syncthreads();  // the previous pass is consumed
        for (int idx = tid; idx < C * NB; idx += 256) {
            const int j = idx / NB, c = idx % NB;
            float val = 0.f;
            if (j < len) {
                if (isk) {
                    const size_t off = ((size_t)(t0 + j) * H + h) * K + col0 + c;
                    val = bs[j] * __bfloat162float(k[qk_row(t0 + j, h, H, hr) * K + col0 + c]) * exp2f(G[off]);
                } else {
                    val = bs[j] * __bfloat162float(v[((size_t)(t0 + j) * H + h) * V + (col0 - K) + c]);
                }
            }
            Xs[j][c] = val;
        }
        __syncthreads();
        float acc[NT][4];
#pragma unroll
        for (int jt = 0; jt < NT; ++jt) acc[jt][0] = acc[jt][1] = acc[jt][2] = acc[jt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks) {
#pragma unroll
            for (int jt = 0; jt < NT; ++jt) {
                const int cb = c0 + 8 * jt + g;
                const uint32_t b[2] = {to_tf32(Xs[8 * ks + t][cb]), to_tf32(Xs[8 * ks + t + 4][cb])};
                mma_tf32_16x8x8(acc[jt], a[ks], b);
            }
        }
#pragma unroll
        for (int jt = 0; jt < NT; ++jt) {
            const int col = col0 + c0 + 8 * jt + 2 * t;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int i = r0 + g + 8 * half;
                if (i < len) {
                    float* dst = isk ? w + ((size_t)(t0 + i) * H + h) * K + col
                                     : u + ((size_t)(t0 + i) * H + h) * V + (col - K);
                    dst[0] = acc[jt][2 * half];
                    dst[1] = acc[jt][2 * half + 1];
                }
            }
        }
    }
}

// a2 for the safe gate with bf16 inputs: the anchored products of scores_anchored_kernel as
// m16n8k8 tf32 MMAs (FP32 accumulation).  Per channel slab of DA: rows k_i 2^(G_i - G_m) and
// q_i 2^(G_i - G_m) (A operands, anchor m of row i's sub-block), and for each sub-block b the
// causal columns k_j 2^(G_m(b) - G_j), j < 16 (b + 1) (B operands).  The output tiles of
// 16 rows x 8 columns are (sub-block b, k or q rows, column tile nt < 2 (b + 1)): 40 for
// C = 64, dealt round-robin to the eight warps; entries above the diagonal are dropped by
// selection (never multiplied), the columns right of the causal ones written as zeros.
// Fragment layout as in out_tc_kernel; the row length DA + 4 keeps both fragment loads on
// 32 different banks.
template <int C>
__global__ void __launch_bounds__(256) scores_tc_kernel(const __nv_bfloat16* __restrict__ q,
                                                        const __nv_bfloat16* __restrict__ k,
                                                        const __nv_bfloat16* __restrict__ beta,
                                                        const float* __restrict__ G, ChunkMap cm,
                                                        int H, int hr, int K, float* __restrict__ Akk,
                                                        float* __restrict__ Aqk) {
    using namespace sm100;
    constexpr int NB = C / 16, DA = 16, LD = DA + 4;
    constexpr int NTILE = 2 * NB * (NB + 1), TPW = (NTILE + 7) / 8;
    __shared__ __align__(16) float krs[C][LD];
    __shared__ __align__(16) float qrs[C][LD];
    __shared__ float gsm[C][DA + 1];
    __shared__ __align__(16) float kcs[NB][C][LD];
    __shared__ float gm[NB][DA];
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, tid = threadIdx.x, wp = tid >> 5, l = tid & 31;
    const int g = l >> 2, t = l & 3;
    // the warp's tiles T = wp + 8 s: sub-block tb, rows tk (0: k, 1: q), column tile tn
    int tb[TPW], tk[TPW], tn[TPW];
#pragma unroll
    for (int s = 0; s < TPW; ++s) {
        int rem = wp + 8 * s, b = 0;
        tb[s] = -1;
        tk[s] = tn[s] = 0;
        for (; b < NB; ++b) {
            const int per = 2 * (b + 1);  // column tiles of sub-block b
            if (rem < 2 * per) {
                tb[s] = b;
                tk[s] = rem / per;
                tn[s] = rem % per;
                break;
            }
            rem -= 2 * per;
        }
    }
    float acc[TPW][4];
#pragma unroll
    for (int s = 0; s < TPW; ++s) acc[s][0] = acc[s][1] = acc[s][2] = acc[s][3] = 0.f;
    for (int d0 = 0; d0 < K; d0 += DA) {
        __syncthreads();  // the previous slab is consumed
        for (int idx = tid; idx < C * DA; idx += 256) {
            const int i = idx / DA, dd = idx % DA;
            float kv = 0.f, qv = 0.f, gv = 0.f;
            if (i < len) {
                const size_t qo = qk_row(t0 + i, h, H, hr) * K + d0 + dd;
                kv = __bfloat162float(k[qo]);
                qv = __bfloat162float(q[qo]);
                gv = G[((size_t)(t0 + i) * H + h) * K + d0 + dd];
            }
            krs[i][dd] = kv;  // raw k until the columns below are built
            qrs[i][dd] = qv;
            gsm[i][dd] = gv;
        }
        __syncthreads();
        if (tid < NB * DA) {  // anchors: the sub-block's midpoint row, or its last valid row
            const int b = tid / DA, dd = tid % DA;
            gm[b][dd] = (16 * b < len) ? gsm[min(16 * b + 8, len - 1)][dd] : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < NB * C * DA; idx += 256) {
            const int b = idx / (C * DA), jj = (idx / DA) % C, dd = idx % DA;
            kcs[b][jj][dd] = (jj < 16 * (b + 1) && jj < len)
                                 ? krs[jj][dd] * exp2f(gm[b][dd] - gsm[jj][dd]) : 0.f;
        }
        __syncthreads();  // the columns have read the raw k rows
        for (int idx = tid; idx < C * DA; idx += 256) {
            const int i = idx / DA, dd = idx % DA;
            const float e = (i < len) ? exp2f(gsm[i][dd] - gm[i / 16][dd]) : 0.f;
            krs[i][dd] *= e;
            qrs[i][dd] *= e;
        }
        __syncthreads();
#pragma unroll
        for (int k0 = 0; k0 < DA; k0 += 8) {
#pragma unroll
            for (int s = 0; s < TPW; ++s) {
                if (tb[s] < 0) continue;
                const float (*A)[LD] = tk[s] ? qrs : krs;
                const int r = 16 * tb[s], cb = 8 * tn[s] + g;
                const uint32_t a[4] = {to_tf32(A[r + g][k0 + t]), to_tf32(A[r + g + 8][k0 + t]),
                                       to_tf32(A[r + g][k0 + t + 4]), to_tf32(A[r + g + 8][k0 + t + 4])};
                const uint32_t bb[2] = {to_tf32(kcs[tb[s]][cb][k0 + t]), to_tf32(kcs[tb[s]][cb][k0 + t + 4])};
                mma_tf32_16x8x8(acc[s], a, bb);
            }
        }
    }
    const float scale = rsqrtf((float)K);
#pragma unroll
    for (int s = 0; s < TPW; ++s) {
        if (tb[s] < 0) continue;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int i = 16 * tb[s] + g + 8 * half;
            if (i >= len) continue;
            const float bi = __bfloat162float(beta[(size_t)(t0 + i) * H + h]);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = 8 * tn[s] + 2 * t + e;
                const float val = acc[s][2 * half + e];
                const size_t off = ((size_t)(t0 + i) * H + h) * C + j;
                if (tk[s] == 0) Akk[off] = (j < i) ? bi * val : 0.f;
                else            Aqk[off] = (j <= i) ? scale * val : 0.f;
            }
        }
    }
    for (int idx = tid; idx < C * C; idx += 256) {  // right of the causal columns
        const int i = idx / C, j = idx % C;
        if (i < len && j >= 16 * (i / 16 + 1)) {
            const size_t off = ((size_t)(t0 + i) * H + h) * C + j;
            Akk[off] = 0.f;
            Aqk[off] = 0.f;
        }
    }
}

// a3: T = (I + Akk)^-1 by forward substitution, one thread per column of T
template <int C>
__global__ void __launch_bounds__(C) solve_kernel(const float* __restrict__ Akk, ChunkMap cm,
                                                  int H, float* __restrict__ Tm) {
    __shared__ float A[C][C + 1];
    __shared__ float X[C][C + 1];
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, col = threadIdx.x;
    for (int i = 0; i < len; ++i) A[i][col] = Akk[((size_t)(t0 + i) * H + h) * C + col];
    __syncthreads();
    for (int i = 0; i < len; ++i) {
        float val = (i == col) ? 1.f : 0.f;
        for (int j = col; j < i; ++j) val = fmaf(-A[i][j], X[j][col], val);
        X[i][col] = (i < col) ? 0.f : val;
    }
    for (int i = 0; i < len; ++i) Tm[((size_t)(t0 + i) * H + h) * C + col] = X[i][col];
}

// a4: w = T (beta k 2^G) [C,K], u = T (beta v) [C,V]; one thread per output column, four
// rows at a time (four independent sums; T read as float4, broadcast to the warp)
template <typename InT, int C>
__global__ void __launch_bounds__(256, 2) wu_kernel(const InT* __restrict__ k,
                                                 const InT* __restrict__ v,
                                                 const InT* __restrict__ beta,
                                                 const float* __restrict__ G,
                                                 const float* __restrict__ Tm, ChunkMap cm, int H,
                                                 int hr, int K, int V, float* __restrict__ w,
                                                 float* __restrict__ u) {
    __shared__ __align__(16) float Ts[C][C];
    __shared__ float bs[C];
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, tid = threadIdx.x;
    for (int idx = tid; idx < C * C; idx += 256) {
        int i = idx / C, j = idx % C;
        Ts[i][j] = (i < len) ? Tm[((size_t)(t0 + i) * H + h) * C + j] : 0.f;
    }
    for (int i = tid; i < C; i += 256) bs[i] = (i < len) ? to_f32(beta[(size_t)(t0 + i) * H + h]) : 0.f;
    __syncthreads();
    for (int col = tid; col < K + V; col += 256) {
        float x[C];
        const bool isk = col < K;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            float val = 0.f;
            if (j < len) {
                if (isk) {
                    size_t off = ((size_t)(t0 + j) * H + h) * K + col;
                    val = bs[j] * to_f32(k[qk_row(t0 + j, h, H, hr) * K + col]) * exp2f(G[off]);
                } else {
                    val = bs[j] * to_f32(v[((size_t)(t0 + j) * H + h) * V + (col - K)]);
                }
            }
            x[j] = val;
        }
        // T is unit lower triangular and stored with zeros above the diagonal (and in the
        // rows past the end), so the full row product equals the causal one; x stays in
        // registers (static indices)
#pragma unroll 1
        for (int i0 = 0; i0 < len; i0 += 4) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < C; j += 4) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float4 t4 = *reinterpret_cast<const float4*>(&Ts[min(i0 + r, C - 1)][j]);
                    acc[r] = fmaf(t4.x, x[j], acc[r]);
                    acc[r] = fmaf(t4.y, x[j + 1], acc[r]);
                    acc[r] = fmaf(t4.z, x[j + 2], acc[r]);
                    acc[r] = fmaf(t4.w, x[j + 3], acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + r;
                if (i < len) {
                    if (isk) w[((size_t)(t0 + i) * H + h) * K + col] = acc[r];
                    else u[((size_t)(t0 + i) * H + h) * V + (col - K)] = acc[r];
                }
            }
        }
    }
}

// a5: sequential state scan over the chunks of one sequence, 32 value columns per block.
// v_new = u - w h: the w rows of the chunk are staged 32 channels at a time and every
// thread accumulates a register tile of C / 16 rows x 2 columns.  h <- 2^Glast h + kd^T v_new:
// every thread owns CPT consecutive columns of one state row d in registers and adds
// kd[i][d] v_new[i][.] over the chunk's rows, kd = k 2^(Glast - G) read coalesced over d.
template <typename InT, int C, int K>
__global__ void __launch_bounds__(256, 3) scan_kernel(const InT* __restrict__ k,
                                                   const float* __restrict__ G,
                                                   const float* __restrict__ w,
                                                   const float* __restrict__ u, const float* h0,
                                                   float* hT, ChunkMap cm, int H, int hr, int V,
                                                   float* __restrict__ hc,
                                                   float* __restrict__ vn) {
    constexpr int BV = 32, DW = 32;       // value columns per block, channels per w tile
    constexpr int RPT = C / 16;           // v_new rows per thread (16 row groups x 16 column pairs)
    constexpr int TPR = 256 / K;          // threads per state row in the update
    constexpr int CPT = BV / TPR;         // state columns per thread in the update
    static_assert(K * TPR == 256 && CPT % 4 == 0, "state tiling");
    __shared__ __align__(16) float hs[K][BV];
    __shared__ __align__(16) float vns[C][BV];
    __shared__ float wt[C][DW + 1];
    const int tid = threadIdx.x;
    const int v0 = blockIdx.x * BV, h = blockIdx.y, n = blockIdx.z;
    long bos, eos;
    if (cm.cu) { bos = __ldg(cm.cu + n); eos = __ldg(cm.cu + n + 1); }
    else       { bos = (long)n * cm.T; eos = bos + cm.T; }
    const size_t st = ((size_t)n * H + h) * (size_t)K * V;
    for (int idx = tid; idx < K * BV; idx += 256) {
        int d = idx / BV, vv = idx % BV;
        hs[d][vv] = h0 ? h0[st + (size_t)d * V + v0 + vv] : 0.f;
    }
    const int rg = tid >> 4, cp = tid & 15;          // v_new: rows rg*RPT.., columns 2cp, 2cp+1
    const int dr = tid / TPR, c0 = (tid % TPR) * CPT;  // update: row dr, columns c0..c0+CPT
    const int slot0 = cm.first_slot(n, (int)bos);
    const int nt = (int)((eos - bos + C - 1) / C);
    for (int c = 0; c < nt; ++c) {
        const long t0 = bos + (long)c * C;
        const int len = (int)min((long)C, eos - t0);
        __syncthreads();
        const size_t hoff = ((size_t)(slot0 + c) * H + h) * (size_t)K * V;
        for (int idx = tid; idx < K * BV; idx += 256) {
            int d = idx / BV, vv = idx % BV;
            hc[hoff + (size_t)d * V + v0 + vv] = hs[d][vv];
        }
        // v_new = u - w h
        float acc[RPT][2];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int i = rg * RPT + r;
            const size_t row = (size_t)(t0 + i) * H + h;
            acc[r][0] = (i < len) ? u[row * V + v0 + 2 * cp] : 0.f;
            acc[r][1] = (i < len) ? u[row * V + v0 + 2 * cp + 1] : 0.f;
        }
        // the w tiles are software-pipelined: tile d0 + DW is loaded into registers while the
        // products of tile d0 run
        constexpr int WPT = C * DW / 256;  // w elements per thread and tile
        float wreg[WPT];
        auto load_w = [&](int d0) {
#pragma unroll
            for (int e = 0; e < WPT; ++e) {
                const int idx = tid + 256 * e, i = idx / DW, dd = idx % DW;
                wreg[e] = (i < len) ? w[((size_t)(t0 + i) * H + h) * K + d0 + dd] : 0.f;
            }
        };
        load_w(0);
        for (int d0 = 0; d0 < K; d0 += DW) {
            __syncthreads();  // the previous w tile is consumed
#pragma unroll
            for (int e = 0; e < WPT; ++e) {
                const int idx = tid + 256 * e;
                wt[idx / DW][idx % DW] = wreg[e];
            }
            __syncthreads();
            if (d0 + DW < K) load_w(d0 + DW);
#pragma unroll 8
            for (int dd = 0; dd < DW; ++dd) {
                const float2 hv = *reinterpret_cast<const float2*>(&hs[d0 + dd][2 * cp]);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const float wv = wt[rg * RPT + r][dd];
                    acc[r][0] = fmaf(-wv, hv.x, acc[r][0]);
                    acc[r][1] = fmaf(-wv, hv.y, acc[r][1]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int i = rg * RPT + r;
            vns[i][2 * cp] = acc[r][0];
            vns[i][2 * cp + 1] = acc[r][1];
            if (i < len) {
                const size_t row = (size_t)(t0 + i) * H + h;
                vn[row * V + v0 + 2 * cp] = acc[r][0];
                vn[row * V + v0 + 2 * cp + 1] = acc[r][1];
            }
        }
        __syncthreads();
        // h <- 2^Glast h + (k 2^(Glast - G))^T v_new
        const float gl = G[((size_t)(t0 + len - 1) * H + h) * K + dr];
        float hrow[CPT];
        {
            const float gam = exp2f(gl);
#pragma unroll
            for (int j = 0; j < CPT; j += 4) {
                const float4 x = *reinterpret_cast<const float4*>(&hs[dr][c0 + j]);
                hrow[j] = gam * x.x; hrow[j + 1] = gam * x.y; hrow[j + 2] = gam * x.z; hrow[j + 3] = gam * x.w;
            }
        }
#pragma unroll 8
        for (int i = 0; i < len; ++i) {
            const size_t off = ((size_t)(t0 + i) * H + h) * K + dr;
            const float kd = to_f32(k[qk_row(t0 + i, h, H, hr) * K + dr]) * exp2f(gl - G[off]);
#pragma unroll
            for (int j = 0; j < CPT; j += 4) {
                const float4 x = *reinterpret_cast<const float4*>(&vns[i][c0 + j]);
                hrow[j] = fmaf(kd, x.x, hrow[j]);
                hrow[j + 1] = fmaf(kd, x.y, hrow[j + 1]);
                hrow[j + 2] = fmaf(kd, x.z, hrow[j + 2]);
                hrow[j + 3] = fmaf(kd, x.w, hrow[j + 3]);
            }
        }
        __syncthreads();  // every thread has read hs and vns
#pragma unroll
        for (int j = 0; j < CPT; j += 4)
            *reinterpret_cast<float4*>(&hs[dr][c0 + j]) = make_float4(hrow[j], hrow[j + 1], hrow[j + 2], hrow[j + 3]);
    }
    __syncthreads();
    if (hT) {
        for (int idx = tid; idx < K * BV; idx += 256) {
            int d = idx / BV, vv = idx % BV;
            hT[st + (size_t)d * V + v0 + vv] = hs[d][vv];
        }
    }
}

// a6: o = s (q 2^G) h_c + Aqk v_new; one thread per value column, all C rows (the q 2^G and
// Aqk tiles read as float4, broadcast to the warp, four channels / columns per step).  With
// qnorm, row i is finally scaled by 1 / sqrt(|q_i|^2 + eps): every q-dependent term of the
// row is linear in q_i (attention-gym PR #345, deferred q l2norm).
template <typename InT, typename OutT, int C>
__global__ void __launch_bounds__(256) out_kernel(const InT* __restrict__ q,
                                                  const float* __restrict__ G,
                                                  const float* __restrict__ Aqk,
                                                  const float* __restrict__ hc,
                                                  const float* __restrict__ vn, ChunkMap cm,
                                                  int H, int hr, int K, int V, int qnorm,
                                                  OutT* __restrict__ o) {
    __shared__ __align__(16) float qg[C][DT];
    __shared__ __align__(16) float As[C][C];
    __shared__ float rs[C];
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, tid = threadIdx.x, nthr = blockDim.x;
    const float scale = rsqrtf((float)K);
    for (int i = tid; i < C; i += nthr) {
        float r = 1.f;
        if (qnorm && i < len) {
            float ss = 0.f;
            const InT* qi = q + qk_row(t0 + i, h, H, hr) * K;
            for (int d = 0; d < K; ++d) ss = fmaf(to_f32(qi[d]), to_f32(qi[d]), ss);
            r = rsqrtf(ss + kQNormEps);
        }
        rs[i] = r;
    }
    for (int idx = tid; idx < C * C; idx += nthr) {
        int i = idx / C, j = idx % C;
        As[i][j] = (i < len) ? Aqk[((size_t)(t0 + i) * H + h) * C + j] : 0.f;
    }
    const int vcol = tid;  // blockDim.x == V
    const size_t hoff = ((size_t)blockIdx.x * H + h) * (size_t)K * V;
    float acc[C];
#pragma unroll
    for (int i = 0; i < C; ++i) acc[i] = 0.f;
    for (int d0 = 0; d0 < K; d0 += DT) {
        __syncthreads();
        for (int idx = tid; idx < C * DT; idx += nthr) {
            int i = idx / DT, dd = idx % DT;
            float val = 0.f;
            if (i < len) {
                size_t off = ((size_t)(t0 + i) * H + h) * K + d0 + dd;
                val = scale * to_f32(q[qk_row(t0 + i, h, H, hr) * K + d0 + dd]) * exp2f(G[off]);
            }
            qg[i][dd] = val;
        }
        __syncthreads();
        for (int dd = 0; dd < DT; dd += 4) {
            float hv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) hv[e] = hc[hoff + (size_t)(d0 + dd + e) * V + vcol];
#pragma unroll
            for (int i = 0; i < C; ++i) {
                const float4 g4 = *reinterpret_cast<const float4*>(&qg[i][dd]);
                acc[i] = fmaf(g4.x, hv[0], acc[i]);
                acc[i] = fmaf(g4.y, hv[1], acc[i]);
                acc[i] = fmaf(g4.z, hv[2], acc[i]);
                acc[i] = fmaf(g4.w, hv[3], acc[i]);
            }
        }
    }
    __syncthreads();
    // Aqk is zero above the diagonal and in the rows past the end; v_new rows past the end
    // are not read (they may hold anything)
    for (int j = 0; j < len; j += 4) {
        float vj[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) vj[e] = (j + e < len) ? vn[((size_t)(t0 + j + e) * H + h) * V + vcol] : 0.f;
#pragma unroll
        for (int i = 0; i < C; ++i) {
            const float4 a4 = *reinterpret_cast<const float4*>(&As[i][j]);
            acc[i] = fmaf(a4.x, vj[0], acc[i]);
            acc[i] = fmaf(a4.y, vj[1], acc[i]);
            acc[i] = fmaf(a4.z, vj[2], acc[i]);
            acc[i] = fmaf(a4.w, vj[3], acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < C; ++i)
        if (i < len) o[((size_t)(t0 + i) * H + h) * V + vcol] = from_f32<OutT>(acc[i] * rs[i]);
}

// a6 for bf16 inputs: the same o = s (q 2^G) h_c + Aqk v_new with m16n8k8 tf32 MMAs (FP32
// accumulation).  One block of 256 threads per (chunk slot, head); warp w owns the 16 rows
// 16 (w % WM) .. and the V / WN columns from (w / WM) V / WN on, as NT tiles of 8 columns.
// The K (then C) dimension goes through shared memory in slabs of KS: rows of s q 2^G (then
// of Aqk) and rows of h_c (then of v_new, zero past the end of the chunk, where it may hold
// anything).  The h_c slabs are double-buffered: slab s + 1 is copied asynchronously while
// the MMAs of slab s run.  Fragments (g = lane / 4, t = lane % 4): a = A[g][t], A[g+8][t], A[g][t+4],
// A[g+8][t+4]; b = B[t][g], B[t+4][g]; c = C[g][2t], C[g][2t+1], C[g+8][2t], C[g+8][2t+1].
// The padded row lengths make both fragment loads hit 32 different banks.
template <int C, int V, typename OutT>
__global__ void __launch_bounds__(256) out_tc_kernel(const __nv_bfloat16* __restrict__ q,
                                                     const float* __restrict__ G,
                                                     const float* __restrict__ Aqk,
                                                     const float* __restrict__ hc,
                                                     const float* __restrict__ vn, ChunkMap cm,
                                                     int H, int hr, int K, int qnorm,
                                                     OutT* __restrict__ o) {
    using namespace sm100;
    constexpr int WM = C / 16, WN = 8 / WM, NT = V / (8 * WN), KS = 32;
    constexpr int LA = KS + 4, LB = V + 8;
    extern __shared__ __align__(16) float out_tc_smem[];
    float (*As)[LA] = reinterpret_cast<float (*)[LA]>(out_tc_smem);                  // [C][LA]
    float (*Bb)[KS][LB] = reinterpret_cast<float (*)[KS][LB]>(out_tc_smem + C * LA);  // [2][KS][LB]
    float* rs = out_tc_smem + C * LA + 2 * KS * LB;                                   // [C]
    int n, t0, len, bos, eos;
    if (!cm.map(blockIdx.x, n, t0, len, bos, eos)) return;
    const int h = blockIdx.y, tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int g = l >> 2, t = l & 3;
    const int r0 = 16 * (w % WM), c0 = (w / WM) * (V / WN);
    const float scale = rsqrtf((float)K);
    for (int i = tid; i < C; i += 256) {
        float r = 1.f;
        if (qnorm && i < len) {
            float ss = 0.f;
            const __nv_bfloat16* qi = q + qk_row(t0 + i, h, H, hr) * K;
            for (int d = 0; d < K; ++d) ss = fmaf(__bfloat162float(qi[d]), __bfloat162float(qi[d]), ss);
            r = rsqrtf(ss + kQNormEps);
        }
        rs[i] = r;
    }
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    auto mma_slab = [&](const float (*Bs)[LB]) {
#pragma unroll
        for (int k0 = 0; k0 < KS; k0 += 8) {
            const uint32_t a[4] = {to_tf32(As[r0 + g][k0 + t]), to_tf32(As[r0 + g + 8][k0 + t]),
                                   to_tf32(As[r0 + g][k0 + t + 4]), to_tf32(As[r0 + g + 8][k0 + t + 4])};
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int cb = c0 + 8 * j + g;
                const uint32_t b[2] = {to_tf32(Bs[k0 + t][cb]), to_tf32(Bs[k0 + t + 4][cb])};
                mma_tf32_16x8x8(acc[j], a, b);
            }
        }
    };
    // s (q 2^G) h_c
    const size_t hoff = ((size_t)blockIdx.x * H + h) * (size_t)K * V;
    auto load_h = [&](int d0, int buf) {
        for (int idx = tid; idx < KS * (V / 4); idx += 256) {
            const int dd = idx / (V / 4), c4 = idx % (V / 4);
            cp_async16(smem_u32(&Bb[buf][dd][4 * c4]), hc + hoff + (size_t)(d0 + dd) * V + 4 * c4);
        }
        cp_async_commit();
    };
    load_h(0, 0);
    for (int d0 = 0, buf = 0; d0 < K; d0 += KS, buf ^= 1) {
        __syncthreads();  // the previous slab is consumed
        if (d0 + KS < K) load_h(d0 + KS, buf ^ 1);
        else cp_async_commit();  // an empty group keeps the count below uniform
        for (int idx = tid; idx < C * KS; idx += 256) {
            const int i = idx / KS, dd = idx % KS;
            float val = 0.f;
            if (i < len) {
                const size_t off = ((size_t)(t0 + i) * H + h) * K + d0 + dd;
                val = scale * __bfloat162float(q[qk_row(t0 + i, h, H, hr) * K + d0 + dd]) * exp2f(G[off]);
            }
            As[i][dd] = val;
        }
        cp_async_wait_groups<1>();  // this slab's copy (the next one may still be in flight)
        __syncthreads();
        mma_slab(Bb[buf]);
    }
    cp_async_wait_groups<0>();
    // + Aqk v_new (Aqk is zero above the diagonal; both operands are zero past the end)
    for (int j0 = 0; j0 < C; j0 += KS) {
        __syncthreads();
        for (int idx = tid; idx < C * KS; idx += 256) {
            const int i = idx / KS, jj = idx % KS;
            As[i][jj] = (i < len) ? Aqk[((size_t)(t0 + i) * H + h) * C + j0 + jj] : 0.f;
        }
        for (int idx = tid; idx < KS * (V / 4); idx += 256) {
            const int jj = idx / (V / 4), c4 = idx % (V / 4);
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j0 + jj < len)
                x = *reinterpret_cast<const float4*>(vn + ((size_t)(t0 + j0 + jj) * H + h) * V + 4 * c4);
            *reinterpret_cast<float4*>(&Bb[0][jj][4 * c4]) = x;
        }
        __syncthreads();
        mma_slab(Bb[0]);
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int col = c0 + 8 * j + 2 * t;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int i = r0 + g + 8 * half;
            if (i < len) {
                OutT* orow = o + ((size_t)(t0 + i) * H + h) * V + col;
                orow[0] = from_f32<OutT>(acc[j][2 * half] * rs[i]);
                orow[1] = from_f32<OutT>(acc[j][2 * half + 1] * rs[i]);
            }
        }
    }
}

template <int C, int V, typename OutT>
cudaError_t launch_out_tc_v(const FwdArgs& a, const PreciseWs& ws, const ChunkMap& cm, int slots, int hr) {
    constexpr size_t smem = sizeof(float) * (C * (32 + 4) + 2 * 32 * (V + 8) + C);
    auto kern = out_tc_kernel<C, V, OutT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(slots, a.H), 256, smem, a.stream>>>((const __nv_bfloat16*)a.q, ws.G, ws.Aqk, ws.hc, ws.vn,
                                                     cm, a.H, hr, a.K, a.q_l2norm, (OutT*)a.o);
    return cudaSuccess;
}

template <int C, typename OutT>
cudaError_t launch_out_tc(const FwdArgs& a, const PreciseWs& ws, const ChunkMap& cm, int slots, int hr) {
    switch (a.V) {
        case 64: return launch_out_tc_v<C, 64, OutT>(a, ws, cm, slots, hr);
        case 128: return launch_out_tc_v<C, 128, OutT>(a, ws, cm, slots, hr);
        case 256: return launch_out_tc_v<C, 256, OutT>(a, ws, cm, slots, hr);
        default: return cudaErrorInvalidValue;
    }
}

template <typename InT, int C>
cudaError_t run(const FwdArgs& a, const PreciseWs& ws) {
    ChunkMap cm{a.cu, a.N, a.T, C};
    const int slots = cm.n_slots();
    const int hr = a.Hk > 0 ? a.H / a.Hk : 1;  // value heads per query / key head
    GateArgs ga{a.g, a.g_bf16, a.A_log, a.dt_bias, a.mode, a.lb, a.cu, a.N,
                a.B, a.T, a.H, a.K, C, ws.G, a.stream};
    cudaError_t e = launch_gate(ga);
    if (e != cudaSuccess) return e;
    const InT* q = (const InT*)a.q;
    const InT* k = (const InT*)a.k;
    const InT* v = (const InT*)a.v;
    const InT* beta = (const InT*)a.beta;
    if (slots > 0) {
        dim3 g2(slots, a.H);
        if (a.mode == 1 && std::is_same<InT, __nv_bfloat16>::value)  // safe gate, tensor cores
            scores_tc_kernel<C><<<g2, 256, 0, a.stream>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                                          (const __nv_bfloat16*)beta, ws.G, cm, a.H, hr, a.K,
                                                          ws.Akk, ws.Aqk);
        else if (a.mode == 1)  // safe gate: bounded decay, anchored products
            scores_anchored_kernel<InT, C><<<g2, 256, 0, a.stream>>>(q, k, beta, ws.G, cm, a.H, hr, a.K,
                                                                     ws.Akk, ws.Aqk);
        else
            scores_kernel<InT, C><<<g2, 256, 0, a.stream>>>(q, k, beta, ws.G, cm, a.H, hr, a.K, ws.Akk,
                                                            ws.Aqk);
        solve_kernel<C><<<g2, C, 0, a.stream>>>(ws.Akk, cm, a.H, ws.Tm);
        if (std::is_same<InT, __nv_bfloat16>::value)
            wu_tc_kernel<C><<<g2, 256, 0, a.stream>>>((const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
                                                      (const __nv_bfloat16*)beta, ws.G, ws.Tm, cm, a.H, hr,
                                                      a.K, a.V, ws.w, ws.u);
        else
            wu_kernel<InT, C><<<g2, 256, 0, a.stream>>>(k, v, beta, ws.G, ws.Tm, cm, a.H, hr, a.K, a.V,
                                                        ws.w, ws.u);
    }
    dim3 g5(a.V / 32, a.H, a.N);
    switch (a.K) {
        case 64:
            scan_kernel<InT, C, 64><<<g5, 256, 0, a.stream>>>(k, ws.G, ws.w, ws.u, a.h0, a.hT, cm,
                                                              a.H, hr, a.V, ws.hc, ws.vn);
            break;
        case 128:
            scan_kernel<InT, C, 128><<<g5, 256, 0, a.stream>>>(k, ws.G, ws.w, ws.u, a.h0, a.hT, cm,
                                                               a.H, hr, a.V, ws.hc, ws.vn);
            break;
        case 256:
            scan_kernel<InT, C, 256><<<g5, 256, 0, a.stream>>>(k, ws.G, ws.w, ws.u, a.h0, a.hT, cm,
                                                               a.H, hr, a.V, ws.hc, ws.vn);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    if (slots > 0 && std::is_same<InT, __nv_bfloat16>::value) {
        e = a.o_f32 ? launch_out_tc<C, float>(a, ws, cm, slots, hr)
                    : launch_out_tc<C, __nv_bfloat16>(a, ws, cm, slots, hr);
        if (e != cudaSuccess) return e;
    } else if (slots > 0) {
        if (a.o_f32)
            out_kernel<InT, float, C><<<dim3(slots, a.H), a.V, 0, a.stream>>>(
                q, ws.G, ws.Aqk, ws.hc, ws.vn, cm, a.H, hr, a.K, a.V, a.q_l2norm, (float*)a.o);
        else
            out_kernel<InT, InT, C><<<dim3(slots, a.H), a.V, 0, a.stream>>>(
                q, ws.G, ws.Aqk, ws.hc, ws.vn, cm, a.H, hr, a.K, a.V, a.q_l2norm, (InT*)a.o);
    }
    return cudaGetLastError();
}

}  // namespace

size_t precise_workspace_bytes(int B, int T, int H, int K, int V, int C, int N, bool packed) {
    ChunkMap cm{packed ? (const int32_t*)1 : nullptr, N, T, C};
    size_t total = 0;
    carve(nullptr, B, T, H, K, V, C, cm.n_slots(), &total);
    return total;
}

cudaError_t launch_chunk_precise(const FwdArgs& a) {
    ChunkMap cm{a.cu, a.N, a.T, a.C};
    size_t total = 0;
    PreciseWs ws = carve(a.ws, a.B, a.T, a.H, a.K, a.V, a.C, cm.n_slots(), &total);
    if (a.ws_bytes < total) return cudaErrorInvalidValue;
    if (a.C == 64)
        return a.qkv_bf16 ? run<__nv_bfloat16, 64>(a, ws) : run<float, 64>(a, ws);
    return a.qkv_bf16 ? run<__nv_bfloat16, 32>(a, ws) : run<float, 32>(a, ws);
}

}  // namespace kda
