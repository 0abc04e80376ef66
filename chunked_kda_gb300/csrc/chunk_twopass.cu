// Two-pass chunked KDA forward for bf16 inputs with K = V in {128, 256} (sm_103a).
//
// A K = V = 256 head does not fit the single fused kernel: its FP32 state alone is 256 KB, all
// of TMEM.  The work is split where the chunked form allows it (FLA skill "fla-kda", "Public
// code map": the intra / solve stages depend only on the chunk's own inputs, the state scan is
// the one sequential stage):
//
//   pass 1, chunk_prep_kernel: persistent CTAs over the (chunk, head) items, every chunk in
//     parallel.  a1 gate
//     activation and chunk-local log2 cumsum, a2 the causal scores on 16-token sub-blocks as one
//     tcgen05 MMA of N = 160 causal columns per 128 key channels (Helion PR #3290, causal columns
//     only; midpoint anchors and paired offsets, FLA skill "fla-kda", "Safe gate numerical
//     note"), a3 T = (I + Akk)^-1.  It writes T diag(beta) (bf16) and Aqk (fp32) for the chunk,
//     as the byte images of the shared-memory operand tiles the second pass multiplies with.
//     It also writes the chain's operands k 2^G, s q 2^G, k 2^(Gl - G) and 2^Gl.  With the
//     non-safe gate the anchors sit at sub-block first rows and the diagonal 16 x 16 blocks take
//     per-pair factors (nonsafe_diag.cuh).
//   pass 2, chunk_chain_kernel: one CTA per (sequence, head, 128 value channels), the state chain
//     a4-a6 on tcgen05 with the FP32 state h^T [128 v x K] in TMEM:
//        [Y^T | o^T] = h^T [(k 2^G)^T | (s q 2^G)^T]
//        vn^T = (v - Y)^T (T diag beta)^T                          (v_new = u - w h)
//        o^T += vn^T Aqk^T  (tf32, A = the FP32 vn^T accumulator)
//        h^T <- h^T Diag(2^Gl) + vn^T (k 2^(Gl - G))
// Rows beyond the end of a sequence are zero in every operand.
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "kda_internal.h"
#include "nonsafe_diag.cuh"
#include "sm100.cuh"

namespace kda {
namespace twopass {

using namespace sm100;

constexpr int C = 64;
// Pass 1's output per (chunk slot, head) in the workspace: the byte images of the operand tiles
// pass 2 multiplies with, in the shared-memory layouts of its MMAs (128-byte swizzle)
template <int K>
struct Img {
    static constexpr uint32_t TP = 0;               // T diag(beta) bf16 [64][64] K-major
    static constexpr uint32_t AQK = 8192;           // Aqk fp32 [64 i][64 j] K-major, 2 x 32 columns
    static constexpr uint32_t HANDOFF = 24576;      //   (T diag(beta), Aqk: 24 KB)
    static constexpr uint32_t TILE = 64 * K * 2;    // [64 tok][K] bf16 in K / 64 boxes [64][64]
    static constexpr uint32_t KG = HANDOFF;         // k 2^G
    static constexpr uint32_t QG = KG + TILE;       // s q 2^G
    static constexpr uint32_t KD = QG + TILE;       // k 2^(Gl - G)
    static constexpr uint32_t GAM = KD + TILE;      // 2^Glast fp32 [K]
    static constexpr uint32_t QSS = GAM + K * 4;    // sums of q^2 per row fp32 [64]
    static constexpr uint32_t BYTES = QSS + 256;
    static_assert(BYTES % 256 == 0, "image size");
};
// the word of channel pair (d, d + 1), token r in a [64 tok][K] image of K / 64 swizzled boxes
__host__ __device__ __forceinline__ uint32_t pair_off(int r, int d) {
    return (uint32_t)(d >> 6) * 8192u + sm100::sw128((uint32_t)r, (uint32_t)((d & 63) >> 3)) + (uint32_t)(d & 7) * 2u;
}
constexpr int SB_ROWS = 160;            // causal score columns of a 64-token chunk
__host__ __device__ constexpr int sb_off(int b) { return 8 * b * (b + 1); }  // 0, 16, 48, 96
constexpr int LD = 68;                  // fp32 row stride of the solve matrices

__device__ unsigned int g_twopass_timeouts = 0;  // bounded waits that gave up

// ------------------------------------------------------------------ pass 1
namespace prep {
constexpr int NTHR = 256;
// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t OFF_SAH = 0;         // score rows [128 ch][128 rows] MN-major bf16 (k, q)
constexpr uint32_t OFF_SB = 32768;      // score cols [128 ch][160] MN-major, 3 x 16 KB
constexpr uint32_t OFF_AS = 0;          //   after the last score MMA: Akk^T fp32 [64][68]
constexpr uint32_t OFF_TF = 17408;      //   T fp32 [64][68]
constexpr uint32_t OFF_XS = 34816;      //   block products fp32 [4][16][24]
constexpr uint32_t OFF_TP = 40960;      //   T diag(beta) image, 8 KB
constexpr uint32_t OFF_AQK = 49152;     //   Aqk image, 16 KB
constexpr uint32_t OFF_GC = 81920;      // gate sums of the row quarters fp32 [4][128]
constexpr uint32_t OFF_GM = 83968;      // G at the sub-block midpoints fp32 [4][128]
constexpr uint32_t OFF_BETA = 86016;    // beta fp32 [64]
constexpr uint32_t OFF_QSS = 86272;     // partial sums of q^2 per row fp32 [4][64]
constexpr uint32_t OFF_BAR = 87296;     // mbarriers: score MMAs, drain after a give-up
constexpr uint32_t OFF_MISC = 87312;    // tmem base
constexpr uint32_t SMEM_END = 87328;
constexpr uint32_t SMEM_BYTES = SMEM_END + 1024;
static_assert(OFF_SB + 3 * 16384 <= OFF_GC && OFF_AQK + 16384 <= OFF_SB + 3 * 16384, "layout");
static_assert(OFF_XS + 4 * 16 * 24 * 4 <= OFF_TP && OFF_TF + 64 * LD * 4 <= OFF_XS, "layout");
static_assert(OFF_GC + 4 * 128 * 4 <= OFF_GM && OFF_GM + 4 * 128 * 4 <= OFF_BETA, "layout");
static_assert(OFF_BETA + 256 <= OFF_QSS && OFF_QSS + 4 * 64 * 4 <= OFF_BAR, "layout");

struct Params {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* beta;
    const void* g;
    const float* A_log;
    const float* dt_bias;
    int mode;
    float lb;
    int H, hr;  // value heads; value heads per query / key head
    ChunkMap cm;
    uint8_t* img;  // [slots][H][Img<K>::BYTES]
    int* status;   // optional caller word: bit 0 when a wait gives up
    int qnorm;     // write the sums of q^2 per row (deferred q l2norm)
};

// kNS: the non-safe gate (first-row anchors off the diagonal, per-pair diagonal blocks)
template <int K, typename GT, bool kNS>
__global__ void __launch_bounds__(NTHR, 2) chunk_prep_kernel(Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int H = p.H, Hk = H / p.hr;
    const int items = p.cm.n_slots() * H;  // (chunk slot, head) pairs, slot-major
    constexpr bool kGateBf16 = std::is_same<GT, __nv_bfloat16>::value;
    using GW = typename std::conditional<kGateBf16, uint32_t, float2>::type;  // a channel pair

    float* gcarry = reinterpret_cast<float*>(smem + OFF_GC);
    float* gmid = reinterpret_cast<float*>(smem + OFF_GM);
    float* bsm = reinterpret_cast<float*>(smem + OFF_BETA);
    float* As = reinterpret_cast<float*>(smem + OFF_AS);
    float* Tf = reinterpret_cast<float*>(smem + OFF_TF);
    float* Xs = reinterpret_cast<float*>(smem + OFF_XS);
    const uint32_t bar = sb + OFF_BAR;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC);

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 8, 1);
        fence_mbar_init();
    }
    if (w == 0) tmem_alloc(sb + OFF_MISC, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    bool ok = true;  // false (in every thread) once a bounded wait gave up: no further MMA
    uint32_t ph = 0;  // phases of the score-MMA barrier waited for so far (the same in every thread)

    // Thread: channel pair (d0, d0 + 1) of the 128-channel half, rows 16 rq .. 16 rq + 15 (one
    // sub-block); ch0 / ch1 is the pair in swapped order on lanes with bit 2 set, so a warp's
    // 16-byte stores to a channel-major tile cover all eight bank groups.
    const int cbp = w & 1, rq = w >> 1;
    const int d0 = 2 * (32 * cbp + l);
    const int swap = (l >> 2) & 1;
    const int ch0 = d0 + swap, ch1 = d0 + 1 - swap;
    const float scale = rsqrtf((float)K);
    const GT* gptr = reinterpret_cast<const GT*>(p.g);
    const float lbl2 = p.lb * kLog2e;
    // per-token factor into log2 units (the non-safe activation is in log2 units already)
    const float m = kNS ? 1.f : (p.mode == 1) ? lbl2 : kLog2e;

    // Persistent: the CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...; the warps idle
    // during an item's inverse send the next item's rows towards L2
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int slot = item / H, h = item - slot * H;
        int n, t0, len, bos, eos;
        if (!p.cm.map(slot, n, t0, len, bos, eos)) continue;  // not a chunk (the whole CTA)
        const int hq = h / p.hr;
        // beta of the chunk (its previous readers finished with the previous item)
        if (tid < C) bsm[tid] = (tid < len) ? __bfloat162float(p.beta[(size_t)(t0 + tid) * H + h]) : 0.f;
        float dg[4] = {0.f, 0.f, 0.f, 0.f};  // non-safe gate: the diagonal entries this thread holds

        for (int half = 0; half < K / 128; ++half) {
            const int cb = 128 * half;
            // the own rows: k, q pairs and the gate pair, all loads issued first
            uint32_t kr[16], qr[16];
            GW gw[16];
            {
                // row pointers of the sub-block's first row, advanced by one token per row (rows
                // past the end read the last row again: their k, q are zeroed, g adds nothing)
                const size_t tok0 = (size_t)(t0 + min(16 * rq, len - 1));
                const __nv_bfloat16* kp = p.k + (tok0 * Hk + hq) * K + cb + d0;
                const __nv_bfloat16* qp = p.q + (tok0 * Hk + hq) * K + cb + d0;
                const GT* gp = gptr + (tok0 * H + h) * K + cb + d0;
                const size_t sqk = (size_t)Hk * K, sg = (size_t)H * K;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const bool valid = 16 * rq + i < len;
                    kr[i] = valid ? __ldg(reinterpret_cast<const uint32_t*>(kp)) : 0u;
                    qr[i] = valid ? __ldg(reinterpret_cast<const uint32_t*>(qp)) : 0u;
                    gw[i] = __ldg(reinterpret_cast<const GW*>(gp));
                    if (16 * rq + i + 1 < len) {
                        kp += sqk;
                        qp += sqk;
                        gp += sg;
                    }
                }
            }
            // the next half's rows of the warp's 64 channels towards L2 (lane i: row 16 rq + i)
            if (half + 1 < K / 128 && l < 16 && 16 * rq + l < len) {
                const size_t tok = (size_t)(t0 + 16 * rq + l);
                const int cn = cb + 128 + 64 * cbp;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p.k + (tok * Hk + hq) * K + cn));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p.q + (tok * Hk + hq) * K + cn));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(gptr + (tok * H + h) * K + cn));
            }
            // a1: activation in log2 units and the sub-block's inclusive sums (f32x2 on the pair).
            // The bounded-gate instances sum in the thread's (ch0, ch1) order, so no row needs a
            // swap; the non-safe one sums in (d0, d0 + 1) order, which leaves it fewer live
            // registers.  Non-safe gate: -exp(A_log) softplus(g + dt_bias) in log2 units is
            // nA (max(y, 0) + log2(1 + 2^-|y|)), y = (g + dt_bias) log2(e), nA = -exp(A_log)
            constexpr bool kPairOrder = !kNS;
            const int c0 = kPairOrder ? ch0 : d0, c1 = kPairOrder ? ch1 : d0 + 1;
            float2 nA = make_float2(0.f, 0.f), nAd = make_float2(0.f, 0.f);
            if constexpr (kNS) {
                nA.x = -expf(__ldg(p.A_log + h * K + cb + c0));
                nA.y = -expf(__ldg(p.A_log + h * K + cb + c1));
                if (p.dt_bias) {
                    nAd.x = __ldg(p.dt_bias + h * K + cb + c0) * kLog2e;
                    nAd.y = __ldg(p.dt_bias + h * K + cb + c1) * kLog2e;
                }
            } else if (p.mode == 1) {
                nA.x = -expf(__ldg(p.A_log + h * K + cb + c0)) * kLog2e;
                nA.y = -expf(__ldg(p.A_log + h * K + cb + c1)) * kLog2e;
                if (p.dt_bias) {
                    nAd.x = nA.x * __ldg(p.dt_bias + h * K + cb + c0);
                    nAd.y = nA.y * __ldg(p.dt_bias + h * K + cb + c1);
                }
            }
            float2 gv[16], acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float2 a;
                if constexpr (kGateBf16 && kPairOrder) {
                    const uint32_t u0 = swap ? 0x3244u : 0x1044u, u1 = swap ? 0x1044u : 0x3244u;
                    a = make_float2(__uint_as_float(__byte_perm(gw[i], 0u, u0)),
                                    __uint_as_float(__byte_perm(gw[i], 0u, u1)));
                } else if constexpr (kGateBf16) {
                    a = make_float2(bf_lo(gw[i]), bf_hi(gw[i]));
                } else {
                    a = (kPairOrder && swap) ? make_float2(gw[i].y, gw[i].x) : gw[i];
                }
                if constexpr (kNS) {
                    const float2 y = __ffma2_rn(a, make_float2(kLog2e, kLog2e), nAd);
                    const float sp0 = fmaxf(y.x, 0.f) + lg2_fast(1.f + ex2_fast(-fabsf(y.x)));
                    const float sp1 = fmaxf(y.y, 0.f) + lg2_fast(1.f + ex2_fast(-fabsf(y.y)));
                    a = make_float2(nA.x * sp0, nA.y * sp1);
                } else if (p.mode == 1) {
                    float2 z = __ffma2_rn(nA, a, nAd);
                    z = __fadd2_rn(make_float2(ex2_fast(z.x), ex2_fast(z.y)), make_float2(1.f, 1.f));
                    a = make_float2(rcp_fast(z.x), rcp_fast(z.y));
                }
                const float mv = (16 * rq + i < len) ? m : 0.f;  // rows past the end add zero
                acc = __ffma2_rn(make_float2(mv, mv), a, acc);
                gv[i] = acc;
            }
            *reinterpret_cast<float2*>(gcarry + rq * 128 + d0) = acc;
            __syncthreads();  // carries out; the previous half's readers of gmid are done
            float2 cy = make_float2(0.f, 0.f), tot = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 t2 = *reinterpret_cast<const float2*>(gcarry + q * 128 + d0);
                if (q < rq) cy = __fadd2_rn(cy, t2);
                tot = __fadd2_rn(tot, t2);  // G of the chunk's last row (rows past the end add zero)
            }
            uint8_t* img = p.img + ((size_t)slot * H + h) * Img<K>::BYTES;
            if (rq == 0) {  // 2^Glast of the pair, in channel order
                const float e0 = ex2_fast(tot.x), e1 = ex2_fast(tot.y);
                *reinterpret_cast<float2*>(img + Img<K>::GAM + (cb + d0) * 4) =
                    (kPairOrder && swap) ? make_float2(e1, e0) : make_float2(e0, e1);
            }
            float G0[16], G1[16];  // in (ch0, ch1) order
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 g2 = __fadd2_rn(gv[i], cy);
                G0[i] = (kPairOrder || !swap) ? g2.x : g2.y;
                G1[i] = (kPairOrder || !swap) ? g2.y : g2.x;
            }
            // the sub-block anchors: the midpoint row (bounded gates), the first row (non-safe)
            gmid[rq * 128 + ch0] = kNS ? G0[0] : G0[8];
            gmid[rq * 128 + ch1] = kNS ? G1[0] : G1[8];
            // the previous half's score MMA has read the operand tiles (every thread waits; the
            // verdict is made the same in all of them)
            const bool w_ok = !(half > 0 && ok) || mbar_wait(bar, ph & 1u);
            if (ok && !__syncthreads_and(w_ok)) {  // midpoints out, operand tiles free
                if (tid == 0) {
                    atomicAdd(&g_twopass_timeouts, 1u);
                    if (p.status) atomicOr(p.status, 1);
                }
                ok = false;
            } else if (!ok) {
                __syncthreads();
            } else if (half > 0) {
                ++ph;
            }
            // non-safe gate: this half's channel sums of the diagonal blocks (nonsafe_diag.cuh)
            // through the operand area, free now
            if constexpr (kNS) {
                float2 al[16];
#pragma unroll
                for (int i = 1; i < 16; ++i)
                    al[i] = make_float2(ex2_fast(G0[i] - G0[i - 1]), ex2_fast(G1[i] - G1[i - 1]));
                const uint32_t s0 = swap ? 0x3244u : 0x1044u, s1 = swap ? 0x1044u : 0x3244u;
                auto bf_0 = [&](uint32_t x) { return __uint_as_float(__byte_perm(x, 0u, s0)); };
                auto bf_1 = [&](uint32_t x) { return __uint_as_float(__byte_perm(x, 0u, s1)); };
                nsdiag::pass(kr, qr, al, bf_0, bf_1, rq, 32 * cbp + l, tid, sb + OFF_SAH, 0u, dg);
            }

            // a2 operands, channel-major [128 ch][rows] tiles: rows k 2^(G - G_m(rq)), s q 2^(G - G_m(rq));
            // columns of sub-block bi >= rq: k 2^(G_m(rq) - G) 2^(G_m(bi) - G_m(rq)) (the second factor
            // <= 1: paired offsets)
            // (non-safe gate: rows anchored at the sub-block's first row, columns at the next
            // sub-block's first row, or the last row for rq = 3, so every factor is <= 1; the
            // diagonal blocks' own columns are zero, their entries come from the pass above)
            {
                const float gm0 = kNS ? G0[0] : G0[8], gm1 = kNS ? G1[0] : G1[8];  // row anchor
                // chain operands from the anchored products: k 2^G = (k 2^(G - Gm)) 2^Gm,
                // s q 2^G likewise, k 2^(Gl - G) = (k 2^(Gc - G)) 2^(Gl - Gc)
                const float Pm0 = ex2_fast(gm0), Pm1 = ex2_fast(gm1);
                const float tl0 = (kPairOrder || !swap) ? tot.x : tot.y;
                const float tl1 = (kPairOrder || !swap) ? tot.y : tot.x;
                const float gc0 = kNS ? (rq < 3 ? gmid[(rq + 1) * 128 + ch0] : tl0) : gm0;  // column anchor
                const float gc1 = kNS ? (rq < 3 ? gmid[(rq + 1) * 128 + ch1] : tl1) : gm1;
                const float Lm0 = ex2_fast(tl0 - gc0), Lm1 = ex2_fast(tl1 - gc1);
                float qsq[16];
                float R0[4], R1[4];
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) {
                    R0[bi] = (bi > rq) ? ex2_fast(gmid[bi * 128 + ch0] - gc0) : (kNS ? 0.f : 1.f);
                    R1[bi] = (bi > rq) ? ex2_fast(gmid[bi * 128 + ch1] - gc1) : (kNS ? 0.f : 1.f);
                }
                const uint32_t sel0 = swap ? 0x3244u : 0x1044u, sel1 = swap ? 0x1044u : 0x3244u;
                const uint32_t nat = swap ? 0x1032u : 0x3210u;  // (ch0, ch1) word -> (d0, d0 + 1) word
                // the image word of row 16 rq + i: pair_off(16 rq + i, cb + d0) =
                // pbase + 128 i + ((chunk ^ (i & 7)) << 4), the XOR with a constant per row
                const uint32_t pbase = (uint32_t)((cb + d0) >> 6) * 8192u + (uint32_t)rq * 2048u +
                                       (uint32_t)((cb + d0) & 7) * 2u;
                const uint32_t pchunk = (uint32_t)(((cb + d0) & 63) >> 3) << 4;
                uint8_t* const ikg = img + Img<K>::KG;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const uint32_t chk = 2 * rq + hf;
                    const uint32_t r0 = sw128(ch0, chk), r1 = sw128(ch1, chk);
                    uint32_t ak0[4], ak1[4], aq0[4], aq1[4];
                    float kf0[8], kf1[8];
#pragma unroll
                    for (int pr = 0; pr < 4; ++pr) {
                        float ke0[2], ke1[2], qe0[2], qe1[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int i = 8 * hf + 2 * pr + u;
                            const float e0 = ex2_fast(G0[i] - gm0), e1 = ex2_fast(G1[i] - gm1);
                            const float f0 = ex2_fast(gc0 - G0[i]), f1 = ex2_fast(gc1 - G1[i]);
                            const float kv0 = __uint_as_float(__byte_perm(kr[i], 0u, sel0));
                            const float kv1 = __uint_as_float(__byte_perm(kr[i], 0u, sel1));
                            const float qv0 = __uint_as_float(__byte_perm(qr[i], 0u, sel0));
                            const float qv1 = __uint_as_float(__byte_perm(qr[i], 0u, sel1));
                            ke0[u] = kv0 * e0;
                            ke1[u] = kv1 * e1;
                            qe0[u] = scale * qv0 * e0;
                            qe1[u] = scale * qv1 * e1;
                            kf0[2 * pr + u] = kv0 * f0;
                            kf1[2 * pr + u] = kv1 * f1;
                            if (p.qnorm) qsq[i] = fmaf(qv0, qv0, qv1 * qv1);
                            // the pair's words in natural channel order (d0 low, d0 + 1 high)
                            const uint32_t wkg = __byte_perm(pack_bf16(ke0[u] * Pm0, ke1[u] * Pm1), 0u, nat);
                            const uint32_t wqg = __byte_perm(pack_bf16(qe0[u] * Pm0, qe1[u] * Pm1), 0u, nat);
                            const uint32_t wkd =
                                __byte_perm(pack_bf16(kf0[2 * pr + u] * Lm0, kf1[2 * pr + u] * Lm1), 0u, nat);
                            uint32_t* const wp = reinterpret_cast<uint32_t*>(
                                ikg + (pbase + (uint32_t)i * 128u + (pchunk ^ ((uint32_t)(i & 7) << 4))));
                            wp[0] = wkg;                     // k 2^G
                            wp[Img<K>::TILE / 4] = wqg;      // s q 2^G
                            wp[2 * Img<K>::TILE / 4] = wkd;  // k 2^(Gl - G)
                        }
                        ak0[pr] = pack_bf16(ke0[0], ke0[1]);
                        ak1[pr] = pack_bf16(ke1[0], ke1[1]);
                        aq0[pr] = pack_bf16(qe0[0], qe0[1]);
                        aq1[pr] = pack_bf16(qe1[0], qe1[1]);
                    }
                    st_s128(sb + OFF_SAH + r0, ak0[0], ak0[1], ak0[2], ak0[3]);
                    st_s128(sb + OFF_SAH + r1, ak1[0], ak1[1], ak1[2], ak1[3]);
                    st_s128(sb + OFF_SAH + 16384 + r0, aq0[0], aq0[1], aq0[2], aq0[3]);
                    st_s128(sb + OFF_SAH + 16384 + r1, aq1[0], aq1[1], aq1[2], aq1[3]);
#pragma unroll
                    for (int bi = 0; bi < 4; ++bi) {
                        if (bi < rq) continue;
                        const uint32_t n0 = (uint32_t)(sb_off(bi) + 16 * rq + 8 * hf);
                        const uint32_t base = sb + OFF_SB + (n0 >> 6) * 16384u;
                        const uint32_t cn = (n0 & 63u) >> 3;
                        uint32_t s0[4], s1[4];
#pragma unroll
                        for (int pr = 0; pr < 4; ++pr) {
                            s0[pr] = pack_bf16(kf0[2 * pr] * R0[bi], kf0[2 * pr + 1] * R0[bi]);
                            s1[pr] = pack_bf16(kf1[2 * pr] * R1[bi], kf1[2 * pr + 1] * R1[bi]);
                        }
                        st_s128(base + sw128(ch0, cn), s0[0], s0[1], s0[2], s0[3]);
                        st_s128(base + sw128(ch1, cn), s1[0], s1[1], s1[2], s1[3]);
                    }
                }
                if (p.qnorm) {
                    // sum over the warp's 64 channels: butterfly over lane bits 4..1 leaves lane l with
                    // row (l >> 1) & 15, then the pair (l, l ^ 1) completes it
                    float v8[8], v4[4], v2[2];
                    const bool b4 = l & 16, b3 = l & 8, b2 = l & 4, b1 = l & 2;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v8[i] = (b4 ? qsq[8 + i] : qsq[i]) + __shfl_xor_sync(0xffffffffu, b4 ? qsq[i] : qsq[8 + i], 16);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        v4[i] = (b3 ? v8[4 + i] : v8[i]) + __shfl_xor_sync(0xffffffffu, b3 ? v8[i] : v8[4 + i], 8);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        v2[i] = (b2 ? v4[2 + i] : v4[i]) + __shfl_xor_sync(0xffffffffu, b2 ? v4[i] : v4[2 + i], 4);
                    float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
                    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
                    float* qss = reinterpret_cast<float*>(smem + OFF_QSS);
                    if ((l & 1) == 0) qss[(2 * half + cbp) * 64 + 16 * rq + ((l >> 1) & 15)] = v1;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0 && ok) {
                tc_fence_after();
                const uint32_t id_s = idesc_bf16(128, SB_ROWS, 1, 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    uint64_t b = desc_at(umma_desc(sb + OFF_SB, 16384, 1024), kk * 2048);
                    uint64_t a = desc_at(umma_desc(sb + OFF_SAH, 16384, 1024), kk * 2048);
                    umma_bf16(tmem, a, b, id_s, (half > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar);
            }
        }
        {
            const bool w_ok = !ok || mbar_wait(bar, ph & 1u);
            if (!__syncthreads_and(w_ok)) {
                if (tid == 0 && ok) {
                    atomicAdd(&g_twopass_timeouts, 1u);
                    if (p.status) atomicOr(p.status, 1);
                }
                ok = false;
            } else if (ok) {
                ++ph;
            }
        }
        tc_fence_after();

        // the strictly upper 16 x 16 blocks of T diag(beta) are zero
        for (int idx = tid; idx < 64 * 8; idx += NTHR) {
            const int i = idx >> 3, c8 = idx & 7;
            if ((c8 >> 1) > (i >> 4)) st_s128(sb + OFF_TP + sw128(i, c8), 0u, 0u, 0u, 0u);
        }
        // ---- read the scores: warps w and w + 4 share the TMEM lanes of quadrant w & 3 and take
        // alternate 16-column pieces.  Akk rows (lanes 0-63, beta-scaled, strictly lower) into the
        // solve matrix, Aqk rows (lanes 64-127) into the fp32 image.
        if (ok) {
            const int lq = w & 3, part = w >> 2;
            const int row = 32 * lq + l;
            const int i = row & 63;
            const bool is_q = row >= 64;
            const int bi = i >> 4;
            const int bmin = 2 * (lq & 1);
            const bool own_a = bi == bmin;
            const float b_i = bsm[i];
            const uint32_t tl = tmem + ((uint32_t)(32 * lq) << 16);
#pragma unroll 1
            for (int tt = 0; tt < 2; ++tt) {
                const int t = part + 2 * tt;
                float va[16], vb[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) { va[e] = 0.f; vb[e] = 0.f; }
                if (t <= bmin) tmem_ld16(tl + sb_off(bmin) + 16 * t, va);
                if (t <= bmin + 1) tmem_ld16(tl + sb_off(bmin + 1) + 16 * t, vb);
                if (t <= bmin + 1) tmem_wait_ld();
                float sv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) sv[e] = own_a ? va[e] : vb[e];
                if (!is_q) {
                    if (t < bi || (t == bi && !kNS)) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int j = 16 * t + e;
                            As[j * LD + i] = (j < i) ? b_i * sv[e] : 0.f;
                        }
                    }
                } else if (kNS && t == bi) {
                    // the diagonal block (non-safe gate): zeros above the diagonal here, the
                    // per-pair entries below
                    const uint32_t ab = sb + OFF_AQK + (uint32_t)(t >> 1) * 8192u;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int j = 16 * t + e;
                        if (j > i)
                            st_s32(ab + sw128(i, (uint32_t)(4 * (t & 1) + (e >> 2))) + (uint32_t)(e & 3) * 4u, 0u);
                    }
                } else {
                    const uint32_t ab = sb + OFF_AQK + (uint32_t)(t >> 1) * 8192u;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t x[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 16 * t + 4 * c4 + e;
                            x[e] = __float_as_uint((j <= i) ? sv[4 * c4 + e] : 0.f);
                        }
                        st_s128(ab + sw128(i, (uint32_t)(4 * (t & 1) + c4)), x[0], x[1], x[2], x[3]);
                    }
                }
            }
        }
        if constexpr (kNS) {  // the per-pair diagonal entries this thread holds (one per round)
            const float scale_q = rsqrtf((float)K);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                int rb, i, j;
                bool akk;
                nsdiag::entry(tid, q, rb, i, j, akk);
                const int I = 16 * rb + i, J = 16 * rb + j;
                if (akk) {
                    As[J * LD + I] = bsm[I] * dg[q];  // Akk^T, beta-scaled
                } else {
                    st_s32(sb + OFF_AQK + (uint32_t)(J >> 5) * 8192u + sw128(I, (uint32_t)((J & 31) >> 2)) +
                               (uint32_t)(J & 3) * 4u,
                           __float_as_uint(scale_q * dg[q]));
                }
            }
        }
        tc_fence_before();
        __syncthreads();

        // ---- warps 4-7: the next item's k, q and g rows towards L2 (one row of each per thread)
        if (w >= 4 && item + (int)gridDim.x < items) {
            const int nx = item + (int)gridDim.x, sl2 = nx / H, h2 = nx - sl2 * H;
            int n2, t2, len2, bos2, eos2;
            const int r = tid - 128;
            if (p.cm.map(sl2, n2, t2, len2, bos2, eos2) && r < len2) {
                const size_t tok = (size_t)(t2 + r);
                const int hq2 = h2 / p.hr;
                prefetch_l2(p.k + (tok * Hk + hq2) * K, K * 2);
                prefetch_l2(p.q + (tok * Hk + hq2) * K, K * 2);
                prefetch_l2(gptr + (tok * H + h2) * K, K * (uint32_t)sizeof(GT));
            }
        }
        // ---- a3 on warps 0-3: T = (I + Akk)^-1 into the bf16 T diag(beta) image.  Diagonal 16 x 16
        // blocks by forward substitution, one thread per column; then the off-diagonal blocks as a
        // 2 x 2 recursion on 32 x 32 blocks with m16n8k8 tf32 MMAs.
        if (w < 4 && ok) {
            if (w < 2) {
                const int b = 2 * w + (l >> 4), cc = l & 15;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = (i == cc) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < 15; ++j) {
                    const float4* col = reinterpret_cast<const float4*>(As + (16 * b + j) * LD + 16 * b);
#pragma unroll
                    for (int mq = (j + 1) / 4; mq < 4; ++mq) {
                        const float4 c4 = col[mq];
                        const float av[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * mq + e > j) x[4 * mq + e] = fmaf(-av[e], x[j], x[4 * mq + e]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) Tf[(16 * b + i) * LD + 16 * b + cc] = x[i];
                __syncwarp();
                const int i = 16 * b + cc;
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j0 = 16 * b + 2 * e;
                    pk[e] = pack_bf16(Tf[i * LD + j0] * bsm[j0], Tf[i * LD + j0 + 1] * bsm[j0 + 1]);
                }
                st_s128(sb + OFF_TP + sw128(i, 2 * b), pk[0], pk[1], pk[2], pk[3]);
                st_s128(sb + OFF_TP + sw128(i, 2 * b + 1), pk[4], pk[5], pk[6], pk[7]);
            }
            bar_sync(1, 128);
            const int gq = l >> 2, tq = l & 3;
            auto prod_A_T = [&](float (&acc)[2][4], int r0, int kc0, int nk, int n0) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    if (ks >= nk) break;
                    const int kc = kc0 + 8 * ks;
                    uint32_t a[4] = {to_tf32(As[(kc + tq) * LD + r0 + gq]), to_tf32(As[(kc + tq) * LD + r0 + gq + 8]),
                                     to_tf32(As[(kc + tq + 4) * LD + r0 + gq]),
                                     to_tf32(As[(kc + tq + 4) * LD + r0 + gq + 8])};
#pragma unroll
                    for (int n8 = 0; n8 < 2; ++n8) {
                        uint32_t bb[2] = {to_tf32(Tf[(kc + tq) * LD + n0 + 8 * n8 + gq]),
                                          to_tf32(Tf[(kc + tq + 4) * LD + n0 + 8 * n8 + gq])};
                        mma_tf32_16x8x8(acc[n8], a, bb);
                    }
                }
            };
            auto prod_T_X = [&](float (&acc)[2][4], int r0, int k0, const float* X) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int kc = k0 + 8 * ks;
                    uint32_t a[4] = {to_tf32(Tf[(r0 + gq) * LD + kc + tq]), to_tf32(Tf[(r0 + gq + 8) * LD + kc + tq]),
                                     to_tf32(Tf[(r0 + gq) * LD + kc + tq + 4]),
                                     to_tf32(Tf[(r0 + gq + 8) * LD + kc + tq + 4])};
#pragma unroll
                    for (int n8 = 0; n8 < 2; ++n8) {
                        uint32_t bb[2] = {to_tf32(X[(8 * ks + tq) * 24 + 8 * n8 + gq]),
                                          to_tf32(X[(8 * ks + tq + 4) * 24 + 8 * n8 + gq])};
                        mma_tf32_16x8x8(acc[n8], a, bb);
                    }
                }
            };
            auto store_X = [&](float* X, const float (&acc)[2][4]) {
#pragma unroll
                for (int n8 = 0; n8 < 2; ++n8) {
                    X[gq * 24 + 8 * n8 + 2 * tq] = acc[n8][0];
                    X[gq * 24 + 8 * n8 + 2 * tq + 1] = acc[n8][1];
                    X[(gq + 8) * 24 + 8 * n8 + 2 * tq] = acc[n8][2];
                    X[(gq + 8) * 24 + 8 * n8 + 2 * tq + 1] = acc[n8][3];
                }
            };
            auto store_T = [&](int r0, int c0, const float (&acc)[2][4], bool keep) {
#pragma unroll
                for (int n8 = 0; n8 < 2; ++n8) {
                    const int j = c0 + 8 * n8 + 2 * tq;
                    if (keep) {
                        Tf[(r0 + gq) * LD + j] = -acc[n8][0];
                        Tf[(r0 + gq) * LD + j + 1] = -acc[n8][1];
                        Tf[(r0 + gq + 8) * LD + j] = -acc[n8][2];
                        Tf[(r0 + gq + 8) * LD + j + 1] = -acc[n8][3];
                    }
                    const float b0 = -bsm[j], b1 = -bsm[j + 1];
                    const uint32_t o = sb + OFF_TP + (uint32_t)(j & 7) * 2;
                    st_s32(o + sw128(r0 + gq, j >> 3), pack_bf16(acc[n8][0] * b0, acc[n8][1] * b1));
                    st_s32(o + sw128(r0 + gq + 8, j >> 3), pack_bf16(acc[n8][2] * b0, acc[n8][3] * b1));
                }
            };
            if (w < 2) {  // T10 = -T11 (A10 T00), T32 = -T33 (A32 T22)
                const int r0 = 32 * w + 16, c0 = 32 * w;
                float xa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                prod_A_T(xa, r0, c0, 2, c0);
                float* X = Xs + w * (16 * 24);
                store_X(X, xa);
                __syncwarp();
                float ta[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                prod_T_X(ta, r0, r0, X);
                store_T(r0, c0, ta, true);
            }
            bar_sync(1, 128);
            const int rb = 2 + (w >> 1), cbk = w & 1;
            {  // X[r][c] = sum_t A[r][t] T[t][c], r = 2, 3; c = 0, 1
                float xa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                prod_A_T(xa, 16 * rb, 16 * cbk, 4 - 2 * cbk, 16 * cbk);
                store_X(Xs + w * (16 * 24), xa);
            }
            bar_sync(1, 128);
            {  // T[r][c] = -sum_{s=2..r} T[r][s] X[s][c]
                float ta[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 1
                for (int s = 2; s <= 3; ++s)
                    if (s <= rb) prod_T_X(ta, 16 * rb, 16 * s, Xs + (2 * (s - 2) + cbk) * (16 * 24));
                store_T(16 * rb, 16 * cbk, ta, false);
            }
        }
        __syncthreads();
        // the T diag(beta) and Aqk tile images out (24 KB), and the sums of q^2 per row
        {
            uint8_t* img = p.img + ((size_t)slot * H + h) * Img<K>::BYTES;
            uint4* dst = reinterpret_cast<uint4*>(img);
            const uint4* tp = reinterpret_cast<const uint4*>(smem + OFF_TP);
            const uint4* aq = reinterpret_cast<const uint4*>(smem + OFF_AQK);
            for (int x = tid; x < (int)(Img<K>::HANDOFF / 16); x += NTHR)
                dst[x] = x < 512 ? tp[x] : aq[x - 512];
            if (p.qnorm && tid < C) {
                const float* qss = reinterpret_cast<const float*>(smem + OFF_QSS);
                float ssum = 0.f;
#pragma unroll
                for (int j = 0; j < K / 64; ++j) ssum += qss[j * 64 + tid];
                reinterpret_cast<float*>(img + Img<K>::QSS)[tid] = ssum;
            }
        }
        __syncthreads();  // the item's shared buffers and TMEM columns are free for the next one
    }
    // a CTA that gave up a wait lets its MMAs in flight finish before it frees TMEM
    if (!ok && tid == 0) {
        umma_commit(bar + 8);
        mbar_wait(bar + 8, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (w == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}
}  // namespace prep

// ------------------------------------------------------------------ pass 2
namespace chain {
constexpr int NSIMT = 256;                  // 8 warps, two per TMEM lane quadrant
constexpr int NTHR = NSIMT + 32;            // and one that issues the MMAs and the copies
constexpr uint32_t BAR_CHAIN = 1;           // the 8 SIMT warps
// hand-offs from the SIMT warps (arrive) to the issuing warp (sync), all 9 warps: the bf16 state
// and the scaled state ready (HR), the bf16 Y^T tile and the v tile (YA), the bf16 v_new^T tile (VN)
constexpr uint32_t BAR_HR = 2, BAR_YA = 3, BAR_VN = 4;

// shared memory (bytes from a 1024-aligned base); K-dependent sizes
template <int K>
struct Smem {
    using I = Img<K>;
    // k 2^G and s q 2^G (image, bulk copies) interleaved by 64-channel panel: panel p holds the
    // 64 k rows then the 64 q rows, so one N = 128 MMA forms Y^T and o^T together
    static constexpr uint32_t KT = 0;                          // 2 TILE bytes
    static constexpr uint32_t QT = KT + I::TILE;
    static constexpr uint32_t KDB = (I::TILE + K * 4 + 1023) / 1024 * 1024;  // one kd buffer:
    static constexpr uint32_t KD = QT + I::TILE;               //   k 2^(Gl - G), then 2^Glast (one
    static constexpr uint32_t GAM = KD + I::TILE;              //   copy); two buffers (parity)
    static constexpr uint32_t V = KD + 2 * KDB;                // v tile [64 tok][128 v]
    static constexpr uint32_t IMG = V + 16384;                 // T diag(beta), Aqk: two buffers
    static constexpr uint32_t YA = IMG + 2 * I::HANDOFF;       // Y^T, then v_new^T, bf16 [128 v][64 tok]
    static constexpr uint32_t BAR = YA + 16384;                // mbarriers
    static constexpr uint32_t MISC = BAR + 128;                // tmem base, abort flag, loads issued
    static constexpr uint32_t END = MISC + 32;
    static constexpr uint32_t BYTES = END + 1024;
    static_assert(BYTES <= 232448, "shared memory of one CTA");
    static_assert(I::QG - I::KG == I::TILE && I::GAM - I::KD == GAM - KD, "copy layout");
    static_assert(KDB % 1024 == 0 && V % 1024 == 0, "align");
};
// TMEM columns: h^T fp32 [128 v][K], its bf16 copy (K / 2 columns), Y^T / v_new^T, o^T (right
// after Y^T: one N = 128 MMA writes both)
template <int K>
struct Tmem {
    static constexpr uint32_t H = 0, HA = K, Y = K + K / 2, O = Y + 64;
    static constexpr uint32_t COLS = 512;
    static_assert(O + 64 <= COLS, "TMEM");
};

enum { B_OPS = 0, B_KD0, B_KD1, B_YDONE, B_VFULL, B_IMG0, B_IMG1, B_VNDONE, B_OHDONE, B_DRAIN, B_STALL, NBAR };

struct Params {
    const float* h0;
    float* hT;
    const int32_t* cu;
    void* o;
    int T, H, V;
    int qnorm;           // scale each output row by 1 / sqrt(|q row|^2 + kQNormEps)
    ChunkMap cm;
    const uint8_t* img;  // pass 1's images [slots][H][Img<K>::BYTES]
    int* status;         // optional caller word: bit 0 when a wait gives up
    int stall_chunk;     // test hook (>= 0): at this chunk the issuing warp waits, with a short
                         // limit, on an mbarrier nothing arrives on, and gives up
    // Dense inputs, balanced schedule (chunk_chain_kernel<..., true>, one CTA per SM, all
    // resident at once): the (sequence, head) units u = n + N h, bal_nt chunks each, laid end to
    // end; the CTAs form groups of V / 128 (the value blocks of a head side by side), and group
    // m runs the chunk-times [m bal_cm, (m + 1) bal_cm) of that row.  A unit cut by the boundary
    // at m bal_cm runs its first chunks at the start of group m and its other chunks at the end
    // of group m - 1 (bal_cm > bal_nt: the first part ends before the second starts); the FP32
    // state of value block vb crosses in slot m (V / 128) + vb of bal_state ([K][128] words),
    // published by the flag of the same index (zero on entry).
    int N, bal_cm, bal_nt;
    float* bal_state;
    unsigned* bal_flag;
};

struct Sync {
    uint32_t bars;
    volatile uint32_t* abort_flag;
    int* status;
    __device__ __forceinline__ uint32_t bar(int i) const { return bars + 8u * i; }
    __device__ __forceinline__ void wait(int i, uint32_t parity) const {
        if (*abort_flag) return;
        // (the plain wait: the abort-aware one measured 2 % slower on this kernel; a give-up
        // reaches the other waits of the CTA through their own limits)
        if (!mbar_wait(bar(i), parity)) {
            atomicAdd(&g_twopass_timeouts, 1u);
            if (status) atomicOr(status, 1);
            *abort_flag = 1u;
        }
    }
    __device__ __forceinline__ bool aborted() const { return *abort_flag != 0u; }
    __device__ __forceinline__ void group_wait(int i, uint32_t parity, bool leader) const {
        if (leader) wait(i, parity);
        bar_sync(BAR_CHAIN, NSIMT);
    }
};

// a bulk copy of `bytes` (a multiple of 16) in pieces of at most 32 KB, completing on `bar`
__device__ __forceinline__ void bulk_copy(uint32_t dst, const uint8_t* src, uint32_t bytes, uint32_t bar) {
    mbar_arrive_expect_tx(bar, bytes);
    for (uint32_t o = 0; o < bytes; o += 32768u)
        bulk_load(dst + o, src + o, min(32768u, bytes - o), bar);
}

// One piece of a (sequence, head, value block vb) unit: its chunks [c0, c1).  head_slot >= 0:
// the piece ends before the unit does, and its final FP32 state goes to that slot of the
// balanced schedule; cont_slot >= 0: the piece starts after the unit does, and its initial
// state comes from that slot once its flag is set.
template <int K, typename OT>
__device__ __forceinline__ void chain_piece(const CUtensorMap& tm_v, const Params& p, uint8_t* smem,
                                            uint32_t sb, uint32_t tmem, const Sync& sy, int vb, int n,
                                            int h, int c0, int c1, int head_slot, int cont_slot) {
    using S = Smem<K>;
    using I = Img<K>;
    using TM = Tmem<K>;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + S::MISC);
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int H = p.H;
    long sbos, seos;  // the sequence
    if (p.cu) { sbos = __ldg(p.cu + n); seos = __ldg(p.cu + n + 1); }
    else      { sbos = (long)n * p.T; seos = sbos + p.T; }
    const long bos = sbos + (long)c0 * C, eos = min(sbos + (long)c1 * C, seos);
    const int nt = c1 - c0;
    const int slot0 = p.cm.first_slot(n, (int)sbos) + c0;
    auto image = [&](int c) { return p.img + ((size_t)(slot0 + c) * H + h) * I::BYTES; };
    volatile uint32_t* issued = misc + 2;

    const int lg = w & 3, hch = w >> 2;
    const int vlane = 32 * lg + l;                  // value channel within the block
    const int vch = 128 * vb + vlane;               // value channel
    const uint32_t lane_base = (uint32_t)(32 * lg) << 16;
    const size_t st_off = ((size_t)n * H + h) * (size_t)K * p.V;
    const uint32_t yab = sb + S::YA;
    // state columns of this thread: key channels hch * K / 2 .. + K / 2 - 1, in pieces of 32
    auto ld_h = [&](int s, float (&hv)[32]) {
        tmem_ld16(tmem + lane_base + TM::H + (K / 2) * hch + 32 * s, hv);
        tmem_ld16(tmem + lane_base + TM::H + (K / 2) * hch + 32 * s + 16, hv + 16);
    };
    auto st_h = [&](int s, const float (&hv)[32]) {
        tmem_st16(tmem + lane_base + TM::H + (K / 2) * hch + 32 * s, reinterpret_cast<const uint32_t*>(hv));
        tmem_st16(tmem + lane_base + TM::H + (K / 2) * hch + 32 * s + 16,
                  reinterpret_cast<const uint32_t*>(hv) + 16);
    };
    auto st_hA = [&](int s, const float (&hv)[32]) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = pack_bf16(hv[2 * e], hv[2 * e + 1]);
        tmem_st16(tmem + lane_base + TM::HA + (K / 4) * hch + 16 * s, r);
    };
    // the thread's 32 tokens (32 hch ..) of a [128 v][64 tok] fp32 accumulator row -> the bf16
    // K-major A tile (row = value channel, 128 bytes, 128-byte swizzle)
    auto acc_to_bf16_tile = [&](uint32_t col) {
        float x[32];
        tmem_ld16(tmem + lane_base + col + 32 * hch, x);
        tmem_ld16(tmem + lane_base + col + 32 * hch + 16, x + 16);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q)
            st_s128(yab + sw128((uint32_t)vlane, (uint32_t)(4 * hch + q)), pack_bf16(x[8 * q], x[8 * q + 1]),
                    pack_bf16(x[8 * q + 2], x[8 * q + 3]), pack_bf16(x[8 * q + 4], x[8 * q + 5]),
                    pack_bf16(x[8 * q + 6], x[8 * q + 7]));
    };
    // v - Y^T of the thread's value channel and 32 tokens (the v tile's rows past the end give
    // zero: they may hold the next sequence's tokens or NaN padding) -> the bf16 A tile of the
    // v_new MMA
    auto v_minus_y_tile = [&](int len) {
        float x[32];
        tmem_ld16(tmem + lane_base + TM::Y + 32 * hch, x);
        tmem_ld16(tmem + lane_base + TM::Y + 32 * hch + 16, x + 16);
        const uint32_t vrow = sb + S::V + (uint32_t)(vlane >> 6) * 8192u + (uint32_t)(vlane & 7) * 2u;
        const uint32_t vchk = (uint32_t)((vlane & 63) >> 3);
        float vv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) vv[j] = ld_s_bf16(vrow + sw128((uint32_t)(32 * hch + j), vchk));
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = (32 * hch + j < len) ? vv[j] - x[j] : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            st_s128(yab + sw128((uint32_t)vlane, (uint32_t)(4 * hch + q)), pack_bf16(x[8 * q], x[8 * q + 1]),
                    pack_bf16(x[8 * q + 2], x[8 * q + 3]), pack_bf16(x[8 * q + 4], x[8 * q + 5]),
                    pack_bf16(x[8 * q + 6], x[8 * q + 7]));
    };
    // copies of chunk c's image parts (issued by thread 0); the next chunk's parts are prefetched
    // to L2 along with them
    auto load_ops = [&](int c) {
        issued[0] = issued[0] + 1u;
        mbar_arrive_expect_tx(sy.bar(B_OPS), 2 * I::TILE);
        for (int pnl = 0; pnl < K / 64; ++pnl)
            for (int t = 0; t < 2; ++t)
                bulk_load(sb + S::KT + (uint32_t)pnl * 16384u + (uint32_t)t * 8192u,
                          image(c) + I::KG + (size_t)t * I::TILE + (size_t)pnl * 8192u, 8192u, sy.bar(B_OPS));
        if (c + 1 < nt) prefetch_l2(image(c + 1) + I::KG, 2 * I::TILE);
    };
    auto load_kd = [&](int c) {
        issued[1] = issued[1] + 1u;
        const int b = c & 1;
        bulk_copy(sb + S::KD + (uint32_t)b * S::KDB, image(c) + I::KD, I::TILE + K * 4, sy.bar(B_KD0 + b));
        if (c + 1 < nt) prefetch_l2(image(c + 1) + I::KD, I::TILE + K * 4);
    };
    auto load_img = [&](int c) {
        issued[3] = issued[3] + 1u;
        const int b = c & 1;
        bulk_copy(sb + S::IMG + (uint32_t)b * I::HANDOFF, image(c), I::HANDOFF, sy.bar(B_IMG0 + b));
    };
    auto load_v = [&](long t) {
        issued[2] = issued[2] + 1u;
        mbar_arrive_expect_tx(sy.bar(B_VFULL), 16384);
        for (int cb = 0; cb < 2; ++cb)
            tma_load_3d(sb + S::V + cb * 8192, &tm_v, 128 * vb + 64 * cb, h, (int)t, sy.bar(B_VFULL));
    };
    // o of chunk c (the thread's 32 rows of its value channel), stored while chunk c + 1's
    // MMAs run
    float ov[32];
    auto store_o = [&](int c) {
        const long tc = bos + (long)c * C;
        const int lc = (int)min((long)C, eos - tc);
        if (p.qnorm) {  // o row / sqrt(|q row|^2 + eps), the sums from pass 1
            const float* qss = reinterpret_cast<const float*>(image(c) + I::QSS) + 32 * hch;
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] *= rsqrtf(__ldg(qss + j) + kQNormEps);
        }
        OT* op = reinterpret_cast<OT*>(p.o) + ((size_t)(tc + 32 * hch) * H + h) * p.V + vch;
        const size_t ostride = (size_t)H * p.V;
        const int nvalid = lc - 32 * hch;
#pragma unroll
        for (int j = 0; j < 32; ++j, op += ostride)
            if (j < nvalid) *op = to_out<OT>(ov[j]);
    };
    // the bf16 copy of h^T: the next Y / o MMAs' A operand
    auto copy_hA = [&]() {
#pragma unroll 1
        for (int s = 0; s < K / 64; ++s) {
            float hv[32];
            ld_h(s, hv);
            tmem_wait_ld();
            st_hA(s, hv);
        }
    };
    // h^T <- h^T Diag(2^Glast) of chunk cs (the gamma row of that chunk's kd buffer) for its
    // state MMA; runs while that chunk's v_new MMA does
    auto scale_h = [&](int cs) {
        const float* gm = reinterpret_cast<const float*>(smem + S::KD + (uint32_t)(cs & 1) * S::KDB + I::TILE) +
                          (K / 2) * hch;
#pragma unroll 1
        for (int s = 0; s < K / 64; ++s) {
            float hv[32];
            ld_h(s, hv);
            float gv[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 g4 = *reinterpret_cast<const float4*>(gm + 32 * s + j);
                gv[j] = g4.x; gv[j + 1] = g4.y; gv[j + 2] = g4.z; gv[j + 3] = g4.w;
            }
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) hv[j] *= gv[j];
            st_h(s, hv);
        }
    };

    if (w == 8) {
        // ---- the issuing warp (lane 0): copies a chunk ahead, and every MMA
        if (l == 0 && nt > 0) {
            load_ops(0);
            load_kd(0);
            load_img(0);
            load_v(bos);
        }
        for (int c = 0; c < nt; ++c) {
            const long t0 = bos + (long)c * C;
            const uint32_t img = sb + S::IMG + (uint32_t)(c & 1) * I::HANDOFF;
            const uint32_t kdb = S::KD + (uint32_t)(c & 1) * S::KDB;
            if (c == p.stall_chunk && l == 0 && !sy.aborted() && !mbar_wait(sy.bar(B_STALL), 0, 1u << 10)) {
                atomicAdd(&g_twopass_timeouts, 1u);  // test hook: a bounded wait that gives up
                if (p.status) atomicOr(p.status, 1);
                *sy.abort_flag = 1u;
            }
            if (l == 0) sy.wait(B_OPS, (uint32_t)(c & 1));
            bar_sync(BAR_HR, NTHR);  // bf16 h^T of the state before chunk c; o^T of chunk c - 1 read
            // ---- [Y^T | o^T] = h^T [(k 2^G)^T | (s q 2^G)^T] (N = 128)
            if (l == 0 && !sy.aborted()) {
                tc_fence_after();
                if (c + 1 < nt) {  // their buffers' readers (chunk c - 1) are done
                    load_img(c + 1);
                    load_kd(c + 1);
                }
                const uint32_t id_y = idesc_bf16(128, 128, 0, 0);
#pragma unroll
                for (int kk = 0; kk < K / 16; ++kk) {
                    const uint32_t boff = (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u;
                    uint64_t bkq = desc_at(umma_desc(sb + S::KT, 16, 1024), boff);
                    umma_bf16_ta(tmem + TM::Y, tmem + TM::HA + 8 * kk, bkq, id_y, kk > 0);
                }
                umma_commit(sy.bar(B_YDONE));
            }
            if (l == 0) {
                sy.wait(B_YDONE, (uint32_t)(c & 1));
                if (c + 1 < nt && !sy.aborted()) load_ops(c + 1);  // the operand tiles are free
            }
            bar_sync(BAR_YA, NTHR);  // bf16 (v - Y)^T tile
            // ---- v_new^T = (v - Y)^T T'^T into the Y^T columns, then o^T += v_new^T Aqk^T
            // (tf32: A = the FP32 v_new^T accumulator)
            if (l == 0) {
                sy.wait(B_IMG0 + (c & 1), (uint32_t)((c >> 1) & 1));
                if (!sy.aborted()) {
                    tc_fence_after();
                    const uint32_t id_n = idesc_bf16(128, 64, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint64_t a = desc_at(umma_desc(yab, 16, 1024), kk * 32);
                        uint64_t b = desc_at(umma_desc(img + I::TP, 16, 1024), kk * 32);
                        umma_bf16(tmem + TM::Y, a, b, id_n, kk > 0);
                    }
                    umma_commit(sy.bar(B_VNDONE));
                }
                sy.wait(B_VNDONE, (uint32_t)(c & 1));
                if (c + 1 < nt && !sy.aborted()) load_v(t0 + C);
                if (!sy.aborted()) {
                    tc_fence_after();
                    const uint32_t id_o = idesc_tf32(128, 64);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        uint64_t bo = desc_at(umma_desc(img + I::AQK + (uint32_t)(kk >> 2) * 8192u, 16, 1024),
                                              (uint32_t)(kk & 3) * 32u);
                        umma_tf32_ta(tmem + TM::O, tmem + TM::Y + 8 * kk, bo, id_o, 1);
                    }
                }
            }
            bar_sync(BAR_VN, NTHR);  // bf16 v_new^T tile
            // ---- h^T += v_new^T (k 2^(Gl - G)) on the scaled state
            if (l == 0) {
                sy.wait(B_KD0 + (c & 1), (uint32_t)((c >> 1) & 1));
                if (!sy.aborted()) {
                    tc_fence_after();
                    const uint32_t id_h = idesc_bf16(128, K, 0, 1);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint64_t a = desc_at(umma_desc(yab, 16, 1024), kk * 32);
                        uint64_t b = desc_at(umma_desc(sb + kdb, 8192, 1024), kk * 2048);
                        umma_bf16(tmem + TM::H, a, b, id_h, 1);
                    }
                    umma_commit(sy.bar(B_OHDONE));
                }
                sy.wait(B_OHDONE, (uint32_t)(c & 1));  // the next copies reuse this chunk's buffers
            }
            __syncwarp();
        }
        // after a give-up: let the last copy of each kind land, and the MMAs in flight finish
        if (l == 0 && sy.aborted()) {
            if (issued[0] > 0) mbar_wait(sy.bar(B_OPS), (issued[0] - 1u) & 1u);
            const uint32_t nk = issued[1];
            if (nk > 0) mbar_wait(sy.bar(B_KD0 + ((nk - 1u) & 1u)), ((nk - 1u) >> 1) & 1u);
            if (issued[2] > 0) mbar_wait(sy.bar(B_VFULL), (issued[2] - 1u) & 1u);
            const uint32_t ni = issued[3];
            if (ni > 0) mbar_wait(sy.bar(B_IMG0 + ((ni - 1u) & 1u)), ((ni - 1u) >> 1) & 1u);
            umma_commit(sy.bar(B_DRAIN));
            mbar_wait(sy.bar(B_DRAIN), 0);
        }
    } else {
        // ---- the 8 SIMT warps.  The initial state (or zero, or the slot a previous piece of the
        // unit filled) into TMEM with its bf16 copy for the first Y / o MMAs
        if (cont_slot >= 0) {  // the CTA that ran the unit's first chunks publishes it (bounded)
            if (tid == 0 && !sy.aborted()) {
                bool ok = false;
                for (uint32_t i = 0; i < (1u << 22) && !ok; ++i) {
                    ok = ld_acquire_gpu(p.bal_flag + cont_slot) != 0u;
                    if (!ok) __nanosleep(256);
                }
                if (!ok) {
                    atomicAdd(&g_twopass_timeouts, 1u);
                    if (p.status) atomicOr(p.status, 1);
                    *sy.abort_flag = 1u;
                }
            }
            bar_sync(BAR_CHAIN, NSIMT);
            __threadfence();
        }
        if (nt > 0) {
#pragma unroll 1
            for (int s = 0; s < K / 64; ++s) {
                float hv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int kch = (K / 2) * hch + 32 * s + j;
                    hv[j] = cont_slot >= 0 ? __ldcg(p.bal_state + ((size_t)cont_slot * K + kch) * 128 + vlane)
                          : p.h0 ? __ldg(p.h0 + st_off + (size_t)kch * p.V + vch) : 0.f;
                }
                st_h(s, hv);
                st_hA(s, hv);
            }
            tmem_wait_st();
            tc_fence_before();
            bar_arrive(BAR_HR, NTHR);
        }
        for (int c = 0; c < nt; ++c) {
            const long t0 = bos + (long)c * C;
            const int len = (int)min((long)C, eos - t0);
            // the previous chunk's o out while the Y / o MMAs run
            if (c > 0) store_o(c - 1);
            sy.group_wait(B_YDONE, (uint32_t)(c & 1), w == 0);
            tc_fence_after();
            // ---- (v - Y)^T -> bf16 A tile
            sy.group_wait(B_VFULL, (uint32_t)(c & 1), w == 0);
            v_minus_y_tile(len);
            fence_proxy_async_smem();
            tc_fence_before();
            bar_arrive(BAR_YA, NTHR);
            // ---- h^T scaled by this chunk's 2^Glast while the v_new MMA runs
            sy.group_wait(B_KD0 + (c & 1), (uint32_t)((c >> 1) & 1), w == 0);
            scale_h(c);
            tmem_wait_st();
            // ---- v_new^T -> bf16 A tile for the state MMA
            sy.group_wait(B_VNDONE, (uint32_t)(c & 1), w == 0);
            tc_fence_after();
            acc_to_bf16_tile(TM::Y);
            fence_proxy_async_smem();
            tc_fence_before();
            bar_arrive(BAR_VN, NTHR);
            // ---- after the state MMA: bf16 h^T for the next chunk and o into registers (stored
            // during the next chunk)
            sy.group_wait(B_OHDONE, (uint32_t)(c & 1), w == 0);
            tc_fence_after();
            const bool more = c + 1 < nt;
            if (more) copy_hA();
            tmem_ld16(tmem + lane_base + TM::O + 32 * hch, ov);
            tmem_ld16(tmem + lane_base + TM::O + 32 * hch + 16, ov + 16);
            tmem_wait_ld();
            tmem_wait_st();
            tc_fence_before();
            if (more) bar_arrive(BAR_HR, NTHR);
        }
        if (nt > 0 && !sy.aborted()) store_o(nt - 1);
        if (head_slot >= 0) {  // the unit's first chunks: publish the state
            if (!sy.aborted()) {
#pragma unroll 1
                for (int s = 0; s < K / 64; ++s) {
                    float hv[32];
                    ld_h(s, hv);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        __stcg(p.bal_state + ((size_t)head_slot * K + (K / 2) * hch + 32 * s + j) * 128 + vlane, hv[j]);
                }
            }
            __threadfence();
            bar_sync(BAR_CHAIN, NSIMT);
            if (tid == 0 && !sy.aborted()) st_release_gpu(p.bal_flag + head_slot, 1u);
        } else if (p.hT && !sy.aborted()) {
#pragma unroll 1
            for (int s = 0; s < K / 64; ++s) {
                float hv[32];
                if (nt > 0) {
                    ld_h(s, hv);
                    tmem_wait_ld();
                } else {  // an empty sequence passes its state through
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        hv[j] = p.h0 ? __ldg(p.h0 + st_off + (size_t)((K / 2) * hch + 32 * s + j) * p.V + vch) : 0.f;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    p.hT[st_off + (size_t)((K / 2) * hch + 32 * s + j) * p.V + vch] = hv[j];
            }
        }
    }
}

// kBal: the balanced schedule of dense inputs (a cooperative launch: its CTAs wait on one
// another); else one CTA per (value block, sequence, head)
template <int K, typename OT, bool kBal>
__global__ void __launch_bounds__(NTHR, 1)
chunk_chain_kernel(const __grid_constant__ CUtensorMap tm_v, Params p) {
    using S = Smem<K>;
    using TM = Tmem<K>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + S::MISC);
    Sync sy{sb + S::BAR, misc + 1, p.status};
    const int tid = threadIdx.x, w = tid >> 5;
    auto init_bars = [&]() {  // fresh barriers and copy counts (operands, kd, v, images)
        for (int i = 0; i < NBAR; ++i) mbar_init(sy.bar(i), 1);
        fence_mbar_init();
        misc[2] = misc[3] = misc[4] = misc[5] = 0;
    };
    if (tid == 0) {
        init_bars();
        misc[1] = 0;
        prefetch_tmap(&tm_v);
    }
    if (w == 0) tmem_alloc(sb + S::MISC, TM::COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if constexpr (!kBal) {
        const int n = blockIdx.y;
        long bos, eos;
        if (p.cu) { bos = __ldg(p.cu + n); eos = __ldg(p.cu + n + 1); }
        else      { bos = (long)n * p.T; eos = bos + p.T; }
        chain_piece<K, OT>(tm_v, p, smem, sb, tmem, sy, blockIdx.x, n, blockIdx.z, 0,
                           (int)((eos - bos + C - 1) / C), -1, -1);
    } else {
        // the group's pieces in order: at most a unit's first chunks, whole units, at most a
        // unit's last chunks
        const int nvb = p.V / 128, m = (int)blockIdx.x / nvb, vb = (int)blockIdx.x % nvb;
        const int ntu = p.bal_nt;
        const long s0 = (long)m * p.bal_cm, e0 = min(s0 + (long)p.bal_cm, (long)p.N * p.H * ntu);
        const int u0 = (int)(s0 / ntu);
        const int npieces = s0 < e0 ? (int)((e0 - 1) / ntu) - u0 + 1 : 0;
        for (int k = 0; k < npieces; ++k) {
            const int u = u0 + k;
            const long ju = (long)u * ntu;
            const long pos = max(s0, ju), pe = min(e0, ju + ntu);
            int c0 = 0, c1 = ntu, head_slot = -1, cont_slot = -1;
            if (pos > ju) {  // cut at the group's start: the unit's first chunks
                c1 = (int)(pe - pos);
                head_slot = m * nvb + vb;
            } else if (pe < ju + ntu) {  // cut at its end: the unit's other chunks
                c0 = ntu - (int)(pe - pos);
                cont_slot = (m + 1) * nvb + vb;
            }
            if (k > 0) {  // every wait and copy of the previous piece ended
                if (tid == 0) {
                    for (int i = 0; i < NBAR; ++i) mbar_inval(sy.bar(i));
                    init_bars();
                }
                __syncthreads();
                tc_fence_after();
            }
            chain_piece<K, OT>(tm_v, p, smem, sb, tmem, sy, vb, u % p.N, u / p.N, c0, c1, head_slot, cont_slot);
            tc_fence_before();
            __syncthreads();
            if (sy.aborted()) break;  // the same verdict in every thread
        }
    }
    tc_fence_before();
    __syncthreads();
    if (w == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM::COLS);
    }
}
}  // namespace chain
}  // namespace twopass

// ------------------------------------------------------------------ host side
namespace fused {
bool make_map(CUtensorMap* m, const void* base, long tokens, int H, int D);
}

// bf16, K in {128, 256} and V a multiple of 128 (pass 1 depends on K only, pass 2 takes the
// value channels in blocks of 128), at most 65535 heads (a grid dimension); every gate mode
// except the non-safe gate at K = V = 128, which the fused kernel takes.  Both chunk sizes run
// as 64-token chunks, as on the fused path.
bool twopass_supported_dims(bool qkv_bf16, int K, int V, int mode, int H) {
    const bool dims_ok = (K == 128 || K == 256) && V >= 128 && V % 128 == 0;
    const bool gate_ok = mode == 0 || mode == 1 || (mode == 2 && !(K == 128 && V == 128));
    return qkv_bf16 && dims_ok && gate_ok && H <= 65535;
}

namespace {
// Balanced schedule of pass 2 for dense inputs.  One CTA per (value block, sequence, head) puts
// U = N H units of nt chunks on M = S / (V / 128) groups of SMs: U = f M + r take f + 1
// unit-lengths, the last wave r / M full.  Laid end to end the U nt chunks fill M groups of
// cm = ceil(U nt / M) chunk-times each: the wrap-around rule for preemptive scheduling on
// identical machines (McNaughton, 1959), a unit cut at a group boundary running its first part
// at the start of the later group, before its second part at the end of the earlier one
// (cm > nt).  A group runs a few pieces, each paying about a chunk-time to start and end; kept
// only for a clear gain.  cm = 0: one CTA per unit.
struct ChainPlan {
    int cm, nt, groups;
};
ChainPlan chain_plan(int T, int H, int V, int N, bool packed) {
    ChainPlan pl{0, 0, 0};
    const int nvb = V / 128;
    if (packed || hook_one_launch() || nvb <= 0) return pl;
    const int M = planned_sm_count() / nvb;
    const long U = (long)N * H;  // the kernel indexes units with an int
    const long nt = (T + twopass::C - 1) / twopass::C;
    if (M <= 0 || U <= M || U % M == 0 || nt <= 0 || U > 0x7fffffffL) return pl;
    const long cm = (U * nt + M - 1) / M;
    const long f = U / M;
    if (20L * (cm + 2) > 19L * (f + 1) * nt || cm > 0x7fffffffL) return pl;
    pl.cm = (int)cm;
    pl.nt = (int)nt;
    pl.groups = M;
    return pl;
}
size_t images_bytes(int T, int H, int K, int N, bool packed) {
    ChunkMap cm{packed ? reinterpret_cast<const int32_t*>(1) : nullptr, N, T, twopass::C};
    const size_t per = K == 256 ? twopass::Img<256>::BYTES : twopass::Img<128>::BYTES;
    return (size_t)cm.n_slots() * (size_t)H * per;
}
// the balanced schedule's flags (one per slot, rounded to 256 bytes) and FP32 [K][128] slots
size_t flag_bytes(int slots) { return ((size_t)slots * 4 + 255) / 256 * 256; }
size_t slot_bytes(int K) { return (size_t)K * 128 * sizeof(float); }
}  // namespace

size_t twopass_workspace_bytes(int T, int H, int K, int V, int N, bool packed) {
    size_t bytes = images_bytes(T, H, K, N, packed);
    const ChainPlan pl = chain_plan(T, H, V, N, packed);
    if (pl.cm > 0) {
        const int slots = pl.groups * (V / 128);
        bytes += flag_bytes(slots) + (size_t)slots * slot_bytes(K);
    }
    return bytes;
}

cudaError_t read_twopass_timeouts(unsigned* count, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(count, twopass::g_twopass_timeouts, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(twopass::g_twopass_timeouts, &zero, sizeof(unsigned));
    }
    return e;
}

namespace {
// SMs of the current device, cached per device ordinal (0 if it cannot be read)
int device_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 64) cached[dev] = n;
    return n;
}

template <int K, typename GT, typename OT>
cudaError_t launch_k(const FwdArgs& a, const ChunkMap& cm, int slots) {
    using namespace twopass;
    const int Hk = a.Hk > 0 ? a.Hk : a.H;
    const int hr = a.H / Hk;
    // pass 1: every (chunk, head), two persistent CTAs per SM
    {
        auto kp = (a.mode == 2) ? prep::chunk_prep_kernel<K, GT, true> : prep::chunk_prep_kernel<K, GT, false>;
        cudaError_t e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, prep::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        prep::Params pp{(const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.beta,
                        a.g, a.A_log, a.dt_bias, a.mode, a.lb, a.H, hr, cm, (uint8_t*)a.ws, a.status,
                        a.q_l2norm ? 1 : 0};
        const long items = (long)slots * a.H;
        const int sms = device_sms();
        const int grid = (int)((sms > 0 && items > 2L * sms) ? 2L * sms : items);
        kp<<<dim3(grid), prep::NTHR, prep::SMEM_BYTES, a.stream>>>(pp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // pass 2: every (sequence, head, 128 value channels), the value blocks of a head side by
    // side so that they share their reads of the images in L2
    CUtensorMap mv;
    const long tokens = (long)a.B * a.T;
    if (!fused::make_map(&mv, a.v, tokens, a.H, a.V)) return cudaErrorInvalidValue;
    constexpr uint32_t smem = chain::Smem<K>::BYTES;
    chain::Params cp{a.h0, a.hT, a.cu, a.o, a.T, a.H, a.V, a.q_l2norm ? 1 : 0, cm, (const uint8_t*)a.ws,
                     a.status, hook_stall_chunk(), a.N, 0, 0, nullptr, nullptr};
    const int nvb = a.V / 128;
    const ChainPlan pl = chain_plan(a.T, a.H, a.V, a.N, a.cu != nullptr);
    // (a plan for more SMs than the device has keeps one CTA per unit: the balanced grid must
    // be resident at once)
    if (pl.cm > 0 && pl.groups * nvb <= device_sms()) {
        auto kb = chain::chunk_chain_kernel<K, OT, true>;
        cudaError_t e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const int slots = pl.groups * nvb;
        uint8_t* extra = reinterpret_cast<uint8_t*>(a.ws) + images_bytes(a.T, a.H, K, a.N, false);
        cp.bal_cm = pl.cm;
        cp.bal_nt = pl.nt;
        cp.bal_flag = reinterpret_cast<unsigned*>(extra);
        cp.bal_state = reinterpret_cast<float*>(extra + flag_bytes(slots));
        e = cudaMemsetAsync(extra, 0, flag_bytes(slots), a.stream);
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(slots);
        cfg.blockDim = dim3(chain::NTHR);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = a.stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kb, mv, cp);
    }
    auto kc = chain::chunk_chain_kernel<K, OT, false>;
    cudaError_t e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kc<<<dim3(nvb, a.N, a.H), chain::NTHR, smem, a.stream>>>(mv, cp);
    return cudaGetLastError();
}
template <int K>
cudaError_t launch_dims(const FwdArgs& a, const ChunkMap& cm, int slots) {
    if (a.g_bf16)
        return a.o_f32 ? launch_k<K, __nv_bfloat16, float>(a, cm, slots)
                       : launch_k<K, __nv_bfloat16, __nv_bfloat16>(a, cm, slots);
    return a.o_f32 ? launch_k<K, float, float>(a, cm, slots) : launch_k<K, float, __nv_bfloat16>(a, cm, slots);
}
}  // namespace

cudaError_t launch_chunk_twopass(const FwdArgs& a) {
    const ChunkMap cm{a.cu, a.N, a.T, twopass::C};
    const int slots = cm.n_slots();
    if (!a.ws || a.ws_bytes < twopass_workspace_bytes(a.T, a.H, a.K, a.V, a.N, a.cu != nullptr))
        return cudaErrorInvalidValue;
    return a.K == 256 ? launch_dims<256>(a, cm, slots) : launch_dims<128>(a, cm, slots);
}

}  // namespace kda
