// Fused chunked KDA forward for bf16 inputs, K = V = 128, C = 64 (sm_103a).
//
// One CTA per (sequence, head) walks the sequence chunk by chunk; the FP32
// state stays on chip for the whole sequence, so HBM sees only q, k, v, g,
// beta, o and the states.  Per chunk of 64 tokens (all steps of the chunked
// form, FLA skill "fla-kda", "Public code map"):
//   a1 gate activation + chunk-local cumsum in log2 units (FLA skill "fla-kda",
//      "Gate modes", "Safe gate numerical note": RCP_LN2 before exp2)
//   a2 causal scores on 16-token sub-blocks, one tcgen05 MMA of N = 160: the
//      rows are k_i and q_i scaled by 2^(G_i - G_m) with m the midpoint of the
//      row's own sub-block, the columns k_j scaled by 2^(G_m - G_j), for the
//      causal columns j < 16 (b + 1) of sub-block b only (Helion PR #3290 "Read
//      only the causal columns in chunk_fwd_A_diag_anchored": C(NC+1)/2 = 160
//      columns instead of NC * C = 256).  In the diagonal blocks each factor
//      spans half a sub-block (|exponent| <= 8 * 5 / ln 2); off the diagonal
//      the column factor is the paired product 2^(G_m(row) - G_m(col)) *
//      2^(G_m(col) - G_j), whose first term is <= 1 (FLA skill "fla-kda",
//      "Safe gate numerical note").
//   a3 T = (I + Akk)^-1 in FP32: 16 x 16 diagonal blocks by forward
//      substitution, then the off-diagonal blocks level by level
//   a4/a5 the WY terms and the state step as tcgen05 MMAs, with the state
//      transposed (TMEM lane = value channel v):
//        Y^T   = h^T (k 2^G)^T                      [V x C]
//        vn^T  = v^T (T diag beta)^T - Y^T (T diag beta)^T      (v_new)
//        dH^T  = vn^T (k 2^(Glast - G))             [V x K]
//        h^T  <- h^T Diag(2^Glast) + dH^T           (FP32, registers)
//   a6 o^T = h^T (s q 2^G)^T + vn^T Aqk^T           [V x C]
// Rows beyond the end of a sequence are masked to zero before any product.
//
// Precision: every product runs on bf16 operands with FP32 accumulation; the
// operands whose rounding dominates the output error are carried as a bf16
// pair x = hi + lo (hi = bf16(x), lo = bf16(x - hi), about 16 significant
// bits) and multiplied as hi*B + lo*B (+ A*lo): the score rows, v_new and Aqk.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kda_internal.h"
#include "sm100.cuh"

namespace kda {

__device__ unsigned int g_fused_timeouts = 0;  // mbarrier waits that gave up

namespace fused {

using namespace sm100;

constexpr int C = 64, KD = 128, VD = 128, NTHR = 256;
// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_V = 0;         // v tile (TMA) = MN-major A of v^T            16 KB
constexpr uint32_t OFF_SAH = 16384;   // score rows hi [128 ch][128 rows] MN-major    32 KB
constexpr uint32_t OFF_SAL = 49152;   // score rows lo                                32 KB
constexpr uint32_t OFF_SB = 81920;    // score cols [160][128 ch] K-major             40 KB
constexpr uint32_t OFF_AQKH = 16384;  //   after the scores: Aqk hi [64][64]  (alias)  8 KB
constexpr uint32_t OFF_AQKL = 24576;  //   Aqk lo                            (alias)  8 KB
constexpr uint32_t OFF_TP = 32768;    //   T diag(beta) bf16 [64][64]        (alias)  8 KB
constexpr uint32_t OFF_YA = 40960;    //   Y^T, then v_new^T hi [128][64]    (alias) 16 KB
constexpr uint32_t OFF_VNL = 57344;   //   v_new^T lo                        (alias) 16 KB
constexpr uint32_t OFF_AS = 73728;    //   Akk fp32 [64][65]                 (alias)
constexpr uint32_t OFF_TF = 90368;    //   T fp32 [64][65]                   (alias)
constexpr uint32_t OFF_XS = 107008;   //   block products fp32 [3][16][17]   (alias)
constexpr uint32_t OFF_KG = 122880;   // k 2^G        [128 ch][64 tok]                 16 KB
constexpr uint32_t OFF_QG = 139264;   // s q 2^G      [128 ch][64 tok]                 16 KB
constexpr uint32_t OFF_KD = 155648;   // k 2^(Gl-G)   [128 ch][64 tok]                 16 KB
constexpr uint32_t OFF_HA = 172032;   // h^T bf16 [128 v][128 ch] K-major              32 KB
constexpr uint32_t OFF_XCH = 204800;  // fp32 [4][128] per-sub-block sums of the gate
constexpr uint32_t OFF_GM = 206848;   // fp32 [4][128] G at the sub-block midpoints
constexpr uint32_t OFF_GL = 208896;   // fp32 [128] G at the last row
constexpr uint32_t OFF_GAM = 209408;  // fp32 [128] 2^G at the last row
constexpr uint32_t OFF_BETA = 209920; // fp32 [64]
constexpr uint32_t OFF_BAR = 210176;  // 2 mbarriers
constexpr uint32_t OFF_MISC = 210192; // tmem base, abort flag
constexpr uint32_t SMEM_BYTES = 210208 + 1024;  // + alignment slack
constexpr int LD = 65;                // fp32 row stride of the solve matrices

// TMEM columns
constexpr uint32_t TM_S = 0, TM_Y = 160, TM_O = 224, TM_VN = 288, TM_DH = 352, TM_COLS = 512;
constexpr int SB_ROWS = 160;                     // score columns (causal only)
__host__ __device__ constexpr int sb_off(int b) { return 8 * b * (b + 1); }  // 0, 16, 48, 96

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }

__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
// x = hi + lo: hi = bf16(x), lo = bf16(x - hi), for the pair (a, b)
__device__ __forceinline__ void pack_split(float a, float b, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
    float2 hf = __bfloat1622float2(h2);
    hi = *reinterpret_cast<uint32_t*>(&h2);
    lo = pack_bf16(a - hf.x, b - hf.y);
}
template <typename OT>
__device__ __forceinline__ OT to_out(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
__device__ __forceinline__ void st_s32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_s128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
__device__ __forceinline__ uint32_t ld_s32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

template <typename GT>
struct GatePair;
template <>
struct GatePair<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float& a, float& b) {
        uint32_t x = __ldg(reinterpret_cast<const unsigned int*>(p));
        a = bf_lo(x);
        b = bf_hi(x);
    }
};
template <>
struct GatePair<float> {
    static __device__ __forceinline__ void load(const float* p, float& a, float& b) {
        float2 x = __ldg(reinterpret_cast<const float2*>(p));
        a = x.x;
        b = x.y;
    }
};

// per-token decay in log2 units
__device__ __forceinline__ float gate_log2(float g, float expA, float dtb, int mode, float lb) {
    if (mode == 0) return g * kLog2e;
    float z = expA * (g + dtb);
    return (lb * kLog2e) * __frcp_rn(1.0f + __expf(-z));
}

struct Params {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* beta;
    const void* g;
    const float* A_log;
    const float* dt_bias;
    const float* h0;
    float* hT;
    const int32_t* cu;
    void* o;
    int mode;
    float lb;
    int T, H;
};

template <typename GT, typename OT>
__global__ void __launch_bounds__(NTHR, 1)
chunk_fused_kernel(const __grid_constant__ CUtensorMap tm_v, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    float* xch = reinterpret_cast<float*>(smem + OFF_XCH);
    float* gmid = reinterpret_cast<float*>(smem + OFF_GM);
    float* glast = reinterpret_cast<float*>(smem + OFF_GL);
    float* gam = reinterpret_cast<float*>(smem + OFF_GAM);
    float* bsm = reinterpret_cast<float*>(smem + OFF_BETA);
    float* As = reinterpret_cast<float*>(smem + OFF_AS);
    float* Tf = reinterpret_cast<float*>(smem + OFF_TF);
    float* Xs = reinterpret_cast<float*>(smem + OFF_XS);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC);
    const uint32_t bar_tma = sb + OFF_BAR, bar_mma = sb + OFF_BAR + 8;

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int h = blockIdx.y, n = blockIdx.x;
    const int H = p.H;
    long bos, eos;
    if (p.cu) { bos = __ldg(p.cu + n); eos = __ldg(p.cu + n + 1); }
    else      { bos = (long)n * p.T; eos = bos + p.T; }
    const int nt = (int)((eos - bos + C - 1) / C);

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        misc[1] = 0;
        prefetch_tmap(&tm_v);
    }
    if (w == 0) tmem_alloc(sb + OFF_MISC, TM_COLS);

    // ---- state: thread owns value channel v (TMEM lane) and key channels [64 ch, 64 ch + 64)
    const int vlane = 32 * (w & 3) + l;
    const int hch = w >> 2;
    const size_t st_off = ((size_t)n * H + h) * (size_t)KD * VD;
    float hs[64];
#pragma unroll
    for (int j = 0; j < 64; ++j)
        hs[j] = p.h0 ? __ldg(p.h0 + st_off + (size_t)(64 * hch + j) * VD + vlane) : 0.f;

    // ---- prep mapping: channel pair (d0, d0 + 1), sub-block rq (rows 16 rq .. 16 rq + 15)
    const int cbp = w & 1;
    const int d0 = 2 * (32 * cbp + l);
    const int rq = w >> 1;
    float expA0 = 0.f, expA1 = 0.f, dtb0 = 0.f, dtb1 = 0.f;
    if (p.mode == 1) {
        expA0 = expf(__ldg(p.A_log + h * KD + d0));
        expA1 = expf(__ldg(p.A_log + h * KD + d0 + 1));
        if (p.dt_bias) {
            dtb0 = __ldg(p.dt_bias + h * KD + d0);
            dtb1 = __ldg(p.dt_bias + h * KD + d0 + 1);
        }
    }
    const float scale = rsqrtf((float)KD);
    const GT* gptr = reinterpret_cast<const GT*>(p.g);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    uint32_t mma_phase = 0;
    bool abort_ = false;

    // write h^T (bf16) into the K-major A operand
    auto write_hA = [&]() {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            uint32_t a = sb + OFF_HA + hch * 16384 + sw128(vlane, c8);
            st_s128(a, pack_bf16(hs[8 * c8 + 0], hs[8 * c8 + 1]), pack_bf16(hs[8 * c8 + 2], hs[8 * c8 + 3]),
                    pack_bf16(hs[8 * c8 + 4], hs[8 * c8 + 5]), pack_bf16(hs[8 * c8 + 6], hs[8 * c8 + 7]));
        }
    };
    write_hA();

    for (int c = 0; c < nt && !abort_; ++c) {
        const long t0 = bos + (long)c * C;
        const int len = (int)min((long)C, eos - t0);

        // ---------------- phase 0: TMA v tile; gate of own rows meanwhile
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_tma, 16384);
            for (int cb = 0; cb < 2; ++cb)
                tma_load_3d(sb + OFF_V + cb * 8192, &tm_v, 64 * cb, h, (int)t0, bar_tma);
        }
        // gate of own rows while the tiles land (global loads)
        float G0[16], G1[16];
        {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * rq + i;
                float a0 = 0.f, a1 = 0.f;
                if (r < len) {
                    float g0, g1;
                    GatePair<GT>::load(gptr + ((size_t)(t0 + r) * H + h) * KD + d0, g0, g1);
                    a0 = gate_log2(g0, expA0, dtb0, p.mode, p.lb);
                    a1 = gate_log2(g1, expA1, dtb1, p.mode, p.lb);
                }
                acc0 += a0;
                acc1 += a1;
                G0[i] = acc0;
                G1[i] = acc1;
            }
            xch[rq * 128 + d0] = acc0;
            xch[rq * 128 + d0 + 1] = acc1;
        }
        if (tid < C) bsm[tid] = (tid < len) ? __bfloat162float(p.beta[(size_t)(t0 + tid) * H + h]) : 0.f;
        if (!mbar_wait(bar_tma, c & 1)) { atomicAdd(&g_fused_timeouts, 1u); misc[1] = 1; }
        __syncthreads();
        if (misc[1]) { abort_ = true; break; }
        {
            float c0 = 0.f, c1 = 0.f;
            for (int q2 = 0; q2 < rq; ++q2) {
                c0 += xch[q2 * 128 + d0];
                c1 += xch[q2 * 128 + d0 + 1];
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) { G0[i] += c0; G1[i] += c1; }
            gmid[rq * 128 + d0] = G0[8];
            gmid[rq * 128 + d0 + 1] = G1[8];
            if (rq == 3) { glast[d0] = G0[15]; glast[d0 + 1] = G1[15]; }
        }
        // zero the v rows beyond the end of the sequence (they may hold the next
        // sequence's data or NaN padding; T's zero columns would not cancel NaN)
        if (len < C) {
            for (int idx = tid; idx < (C - len) * 16; idx += NTHR) {
                int r = len + idx / 16, cbk = (idx / 8) & 1, ch = idx & 7;
                st_s128(sb + OFF_V + cbk * 8192 + sw128(r, ch), 0, 0, 0, 0);
            }
        }
        __syncthreads();

        // ---------------- phase 1: operands
        {
            const float gm0 = G0[8], gm1 = G1[8];
            const float gl0 = glast[d0], gl1 = glast[d0 + 1];
            const float P0 = exp2f(gm0), P1 = exp2f(gm1);              // 2^G at the midpoint
            const float L0 = exp2f(gl0 - gm0), L1 = exp2f(gl1 - gm1);  // 2^(Glast - Gmid) <= 1
            if (rq == 3) { gam[d0] = exp2f(gl0); gam[d0 + 1] = exp2f(gl1); }
            // paired offsets for the later sub-blocks bi > rq: 2^(G_m(bi) - G_m(rq)) <= 1
            float R0[4], R1[4];
#pragma unroll
            for (int bi = 0; bi < 4; ++bi) {
                R0[bi] = (bi > rq) ? exp2f(gmid[bi * 128 + d0] - gm0) : 1.f;
                R1[bi] = (bi > rq) ? exp2f(gmid[bi * 128 + d0 + 1] - gm1) : 1.f;
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t ch = 2 * rq + half;
                uint32_t ak0[4], ak1[4], aq0[4], aq1[4], g_k0[4], g_k1[4], g_q0[4], g_q1[4], dk0[4], dk1[4];
                uint32_t lk0[4], lk1[4], lq0[4], lq1[4];
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
                    float kv0[2], kv1[2], qv0[2], qv1[2], e0[2], e1[2], f0[2], f1[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int i = 8 * half + 2 * pr + u, r = 16 * rq + i;
                        uint32_t kr = 0u, qr = 0u;
                        if (r < len) {
                            const size_t off = ((size_t)(t0 + r) * H + h) * KD + d0;
                            kr = __ldg(reinterpret_cast<const unsigned int*>(p.k + off));
                            qr = __ldg(reinterpret_cast<const unsigned int*>(p.q + off));
                        }
                        kv0[u] = bf_lo(kr); kv1[u] = bf_hi(kr);
                        qv0[u] = scale * bf_lo(qr); qv1[u] = scale * bf_hi(qr);
                        e0[u] = exp2f(G0[i] - gm0); e1[u] = exp2f(G1[i] - gm1);
                        f0[u] = exp2f(gm0 - G0[i]); f1[u] = exp2f(gm1 - G1[i]);
                        // score columns, K-major [n][channel]: sub-block bi >= rq sees row r as
                        // column j = r with anchor m_bi: k_j 2^(G_m(bi) - G_j) = k_j F_j R(bi)
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi) {
                            if (bi < rq) continue;
                            const int nrow = sb_off(bi) + r;
                            st_s32(sb + OFF_SB + cbp * (SB_ROWS * 128) + sw128(nrow, (d0 & 63) >> 3) + (d0 & 7) * 2,
                                   pack_bf16(kv0[u] * f0[u] * R0[bi], kv1[u] * f1[u] * R1[bi]));
                        }
                    }
                    pack_split(kv0[0] * e0[0], kv0[1] * e0[1], ak0[pr], lk0[pr]);
                    pack_split(kv1[0] * e1[0], kv1[1] * e1[1], ak1[pr], lk1[pr]);
                    pack_split(qv0[0] * e0[0], qv0[1] * e0[1], aq0[pr], lq0[pr]);
                    pack_split(qv1[0] * e1[0], qv1[1] * e1[1], aq1[pr], lq1[pr]);
                    g_k0[pr] = pack_bf16(kv0[0] * e0[0] * P0, kv0[1] * e0[1] * P0);
                    g_k1[pr] = pack_bf16(kv1[0] * e1[0] * P1, kv1[1] * e1[1] * P1);
                    g_q0[pr] = pack_bf16(qv0[0] * e0[0] * P0, qv0[1] * e0[1] * P0);
                    g_q1[pr] = pack_bf16(qv1[0] * e1[0] * P1, qv1[1] * e1[1] * P1);
                    dk0[pr] = pack_bf16(kv0[0] * f0[0] * L0, kv0[1] * f0[1] * L0);
                    dk1[pr] = pack_bf16(kv1[0] * f1[0] * L1, kv1[1] * f1[1] * L1);
                }
                // MN-major [channel][row] operands: one 16-byte chunk of 8 rows per channel
                const uint32_t r0 = sw128(d0, ch), r1 = sw128(d0 + 1, ch);
                st_s128(sb + OFF_SAH + r0, ak0[0], ak0[1], ak0[2], ak0[3]);
                st_s128(sb + OFF_SAH + r1, ak1[0], ak1[1], ak1[2], ak1[3]);
                st_s128(sb + OFF_SAH + 16384 + r0, aq0[0], aq0[1], aq0[2], aq0[3]);
                st_s128(sb + OFF_SAH + 16384 + r1, aq1[0], aq1[1], aq1[2], aq1[3]);
                st_s128(sb + OFF_SAL + r0, lk0[0], lk0[1], lk0[2], lk0[3]);
                st_s128(sb + OFF_SAL + r1, lk1[0], lk1[1], lk1[2], lk1[3]);
                st_s128(sb + OFF_SAL + 16384 + r0, lq0[0], lq0[1], lq0[2], lq0[3]);
                st_s128(sb + OFF_SAL + 16384 + r1, lq1[0], lq1[1], lq1[2], lq1[3]);
                st_s128(sb + OFF_KG + r0, g_k0[0], g_k0[1], g_k0[2], g_k0[3]);
                st_s128(sb + OFF_KG + r1, g_k1[0], g_k1[1], g_k1[2], g_k1[3]);
                st_s128(sb + OFF_QG + r0, g_q0[0], g_q0[1], g_q0[2], g_q0[3]);
                st_s128(sb + OFF_QG + r1, g_q1[0], g_q1[1], g_q1[2], g_q1[3]);
                st_s128(sb + OFF_KD + r0, dk0[0], dk0[1], dk0[2], dk0[3]);
                st_s128(sb + OFF_KD + r1, dk1[0], dk1[1], dk1[2], dk1[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---------------- phase 2: scores, Y^T = h^T kg^T, o^T = h^T qg^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_s = idesc_bf16(128, SB_ROWS, 1, 0);
            const uint32_t id_y = idesc_bf16(128, 64, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint64_t b = umma_desc(sb + OFF_SB + (kk >> 2) * (SB_ROWS * 128) + (kk & 3) * 32, 16, 1024);
                uint64_t ah = umma_desc(sb + OFF_SAH + kk * 2048, 16384, 1024);
                uint64_t al = umma_desc(sb + OFF_SAL + kk * 2048, 16384, 1024);
                umma_bf16(tmem + TM_S, ah, b, id_s, kk > 0);
                umma_bf16(tmem + TM_S, al, b, id_s, 1);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint64_t a = umma_desc(sb + OFF_HA + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                uint64_t bk = umma_desc(sb + OFF_KG + kk * 2048, 16384, 1024);
                uint64_t bq = umma_desc(sb + OFF_QG + kk * 2048, 16384, 1024);
                umma_bf16(tmem + TM_Y, a, bk, id_y, kk > 0);
                umma_bf16(tmem + TM_O, a, bq, id_y, kk > 0);
            }
            umma_commit(bar_mma);
        }
        if (!mbar_wait(bar_mma, mma_phase)) { atomicAdd(&g_fused_timeouts, 1u); misc[1] = 1; }
        mma_phase ^= 1;
        tc_fence_after();

        // ---------------- phase 3: read scores (warps 0-3) and Y^T (warps 4-7)
        if (w < 4) {
            const int row = 32 * w + l;       // TMEM lane
            const int i = row & 63;           // chunk row
            const bool is_q = row >= 64;
            const int bi = i >> 4;
            // the 32 lanes of this warp hold two sub-blocks (bmin, bmin + 1); every lane
            // loads the columns of both (warp-collective loads), then keeps its own
            const int bmin = 2 * (w & 1);
            float sv[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) sv[j] = 0.f;
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int bb = bmin + sub;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    if (t <= bb) {
                        float tmp[16];
                        tmem_ld16(tmem + ((uint32_t)(32 * w) << 16) + TM_S + sb_off(bb) + 16 * t, tmp);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (bi == bb) sv[16 * t + e] = tmp[e];
                    }
                }
            }
            if (!is_q) {
                const float bi_beta = bsm[i];
#pragma unroll
                for (int j = 0; j < 64; ++j) As[i * LD + j] = (j < i && j < 16 * (bi + 1)) ? bi_beta * sv[j] : 0.f;
            } else {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint32_t pk[4], pl[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        int j0 = 8 * c8 + 2 * e, j1 = j0 + 1;
                        float x0 = (j0 <= i && j0 < 16 * (bi + 1)) ? sv[j0] : 0.f;
                        float x1 = (j1 <= i && j1 < 16 * (bi + 1)) ? sv[j1] : 0.f;
                        pack_split(x0, x1, pk[e], pl[e]);
                    }
                    st_s128(sb + OFF_AQKH + sw128(i, c8), pk[0], pk[1], pk[2], pk[3]);
                    st_s128(sb + OFF_AQKL + sw128(i, c8), pl[0], pl[1], pl[2], pl[3]);
                }
            }
        } else {
            float yv[64];
#pragma unroll
            for (int t = 0; t < 4; ++t) tmem_ld16(tmem + ((uint32_t)(32 * (w & 3)) << 16) + TM_Y + 16 * t, yv + 16 * t);
            tmem_wait_ld();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
                st_s128(sb + OFF_YA + sw128(vlane, c8), pack_bf16(yv[8 * c8], yv[8 * c8 + 1]),
                        pack_bf16(yv[8 * c8 + 2], yv[8 * c8 + 3]), pack_bf16(yv[8 * c8 + 4], yv[8 * c8 + 5]),
                        pack_bf16(yv[8 * c8 + 6], yv[8 * c8 + 7]));
        }
        __syncthreads();

        // ---------------- phase 4: T = (I + Akk)^-1 (FP32), then T diag(beta) in bf16
        if (tid < 64) {
            const int b = tid >> 4, cc = tid & 15;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float val = (i == cc) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) val = fmaf(-As[(16 * b + i) * LD + 16 * b + j], x[j], val);
                x[i] = (i < cc) ? 0.f : val;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tf[(16 * b + i) * LD + 16 * b + cc] = x[i];
        }
        for (int idx = tid; idx < 64 * 64; idx += NTHR) {
            int i = idx >> 6, j = idx & 63;
            if ((j >> 4) > (i >> 4)) Tf[i * LD + j] = 0.f;
        }
        __syncthreads();
#pragma unroll 1
        for (int lev = 1; lev < 4; ++lev) {
            const int nb = 4 - lev;  // blocks (b + lev, b), b < nb
            const int i = tid >> 4, j = tid & 15;
            for (int b = 0; b < nb; ++b) {
                float acc = 0.f;
                for (int t = 0; t < 16 * lev; ++t)
                    acc = fmaf(As[(16 * (b + lev) + i) * LD + 16 * b + t], Tf[(16 * b + t) * LD + 16 * b + j], acc);
                Xs[(b * 16 + i) * 17 + j] = acc;
            }
            __syncthreads();
            for (int b = 0; b < nb; ++b) {
                float acc = 0.f;
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    acc = fmaf(Tf[(16 * (b + lev) + i) * LD + 16 * (b + lev) + t], Xs[(b * 16 + t) * 17 + j], acc);
                Tf[(16 * (b + lev) + i) * LD + 16 * b + j] = -acc;
            }
            __syncthreads();
        }
        for (int idx = tid; idx < 64 * 8; idx += NTHR) {
            const int i = idx >> 3, c8 = idx & 7;
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int j0 = 8 * c8 + 2 * e;
                pk[e] = pack_bf16(Tf[i * LD + j0] * bsm[j0], Tf[i * LD + j0 + 1] * bsm[j0 + 1]);
            }
            st_s128(sb + OFF_TP + sw128(i, c8), pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---------------- phase 5: vn^T = v^T T'^T - Y^T T'^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_v = idesc_bf16(128, 64, 1, 0);
            const uint32_t id_y = idesc_bf16(128, 64, 0, 0, 1, 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint64_t a = umma_desc(sb + OFF_V + kk * 2048, 8192, 1024);
                uint64_t b = umma_desc(sb + OFF_TP + kk * 32, 16, 1024);
                umma_bf16(tmem + TM_VN, a, b, id_v, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint64_t a = umma_desc(sb + OFF_YA + kk * 32, 16, 1024);
                uint64_t b = umma_desc(sb + OFF_TP + kk * 32, 16, 1024);
                umma_bf16(tmem + TM_VN, a, b, id_y, 1);
            }
            umma_commit(bar_mma);
        }
        if (!mbar_wait(bar_mma, mma_phase)) { atomicAdd(&g_fused_timeouts, 1u); misc[1] = 1; }
        mma_phase ^= 1;
        tc_fence_after();

        // ---------------- phase 6: v_new^T -> bf16 A operand (overwrites Y^T)
        {
            float vv[32];
            const int half = w >> 2;
#pragma unroll
            for (int t = 0; t < 2; ++t)
                tmem_ld16(tmem + ((uint32_t)(32 * (w & 3)) << 16) + TM_VN + 32 * half + 16 * t, vv + 16 * t);
            tmem_wait_ld();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) pack_split(vv[8 * c4 + 2 * e], vv[8 * c4 + 2 * e + 1], hi[e], lo[e]);
                st_s128(sb + OFF_YA + sw128(vlane, 4 * half + c4), hi[0], hi[1], hi[2], hi[3]);
                st_s128(sb + OFF_VNL + sw128(vlane, 4 * half + c4), lo[0], lo[1], lo[2], lo[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---------------- phase 7: o^T += vn^T Aqk^T; dH^T = vn^T kd
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_o = idesc_bf16(128, 64, 0, 0);
            const uint32_t id_h = idesc_bf16(128, 128, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint64_t ah = umma_desc(sb + OFF_YA + kk * 32, 16, 1024);
                uint64_t al = umma_desc(sb + OFF_VNL + kk * 32, 16, 1024);
                uint64_t boh = umma_desc(sb + OFF_AQKH + kk * 32, 16, 1024);
                uint64_t bol = umma_desc(sb + OFF_AQKL + kk * 32, 16, 1024);
                uint64_t bh = umma_desc(sb + OFF_KD + kk * 32, 16, 1024);
                umma_bf16(tmem + TM_O, ah, boh, id_o, 1);
                umma_bf16(tmem + TM_O, al, boh, id_o, 1);
                umma_bf16(tmem + TM_O, ah, bol, id_o, 1);
                umma_bf16(tmem + TM_DH, ah, bh, id_h, kk > 0);
                umma_bf16(tmem + TM_DH, al, bh, id_h, 1);
            }
            umma_commit(bar_mma);
        }
        if (!mbar_wait(bar_mma, mma_phase)) { atomicAdd(&g_fused_timeouts, 1u); misc[1] = 1; }
        mma_phase ^= 1;
        tc_fence_after();

        // ---------------- phase 8: state update, o out
        {
            float dh[64];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                tmem_ld16(tmem + ((uint32_t)(32 * (w & 3)) << 16) + TM_DH + 64 * hch + 16 * t, dh + 16 * t);
            float ov[32];
#pragma unroll
            for (int t = 0; t < 2; ++t)
                tmem_ld16(tmem + ((uint32_t)(32 * (w & 3)) << 16) + TM_O + 32 * hch + 16 * t, ov + 16 * t);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 64; ++j) hs[j] = fmaf(gam[64 * hch + j], hs[j], dh[j]);
            write_hA();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int i = 32 * hch + j;
                if (i < len) reinterpret_cast<OT*>(p.o)[((size_t)(t0 + i) * H + h) * VD + vlane] = to_out<OT>(ov[j]);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (misc[1]) abort_ = true;
    }

    if (p.hT && !abort_) {
#pragma unroll
        for (int j = 0; j < 64; ++j) p.hT[st_off + (size_t)(64 * hch + j) * VD + vlane] = hs[j];
    }
    tc_fence_before();
    __syncthreads();
    if (w == 0) {
        if (abort_ && l == 0) {
            // let any MMA still in flight finish before the columns are released
            umma_commit(bar_mma);
            mbar_wait(bar_mma, mma_phase);
        }
        __syncwarp();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [tokens, H, D] bf16, box of 64 channels x 1 head x 64 tokens, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, long tokens, int H, int D) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace fused

bool fused_supported_dims(bool qkv_bf16, int K, int V, int C) {
    return qkv_bf16 && K == 128 && V == 128 && C == 64;
}

bool fused_supported(const FwdArgs& a) { return fused_supported_dims(a.qkv_bf16, a.K, a.V, a.C); }

template <typename GT, typename OT>
static cudaError_t launch_t(const FwdArgs& a, const CUtensorMap& mv, const fused::Params& p) {
    using namespace fused;
    auto kern = chunk_fused_kernel<GT, OT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.N, a.H), NTHR, SMEM_BYTES, a.stream>>>(mv, p);
    return cudaGetLastError();
}

cudaError_t launch_chunk_fused(const FwdArgs& a) {
    using namespace fused;
    CUtensorMap mv;
    const long tokens = (long)a.B * a.T;
    if (!make_map(&mv, a.v, tokens, a.H, VD)) return cudaErrorInvalidValue;
    Params p{(const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.beta, a.g,
             a.A_log, a.dt_bias, a.h0, a.hT, a.cu, a.o, a.mode, a.lb, a.T, a.H};
    if (a.g_bf16)
        return a.o_f32 ? launch_t<__nv_bfloat16, float>(a, mv, p) : launch_t<__nv_bfloat16, __nv_bfloat16>(a, mv, p);
    return a.o_f32 ? launch_t<float, float>(a, mv, p) : launch_t<float, __nv_bfloat16>(a, mv, p);
}

}  // namespace kda
