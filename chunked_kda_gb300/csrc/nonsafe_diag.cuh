// The diagonal 16 x 16 blocks of the chunk scores under the non-safe gate (sm_103a), shared by
// the fused kernel's preparation group and pass 1 of the two-pass path.
//
// FLA skill "fla-kda", "Safe vs non-safe intra path": with an unbounded per-token decay the
// scores inside a 16-token sub-block take a factor 2^(G_i - G_j) per pair and channel (the
// token-parallel diagonal blocks), while the off-diagonal sub-blocks keep anchored products
// ("Safe gate numerical note": paired offsets, both non-positive).  Here every pair j <= i
// of a sub-block gets
//     Akk(i, j) = sum_c k_i[c] k_j[c] 2^(G_i[c] - G_j[c])     (j < i)
//     Aqk(i, j) = sum_c q_i[c] k_j[c] 2^(G_i[c] - G_j[c])     (j <= i, before the 1/sqrt(K))
// exactly for any decay: per column j the factor runs down the rows as a product of the
// per-token factors 2^(G_i - G_(i-1)) <= 1, so it can only underflow together with the score.
//
// Layout: 256 threads, thread = (sub-block rq, channel pair (ch0, ch1)) over the sub-block's
// 16 rows (the operand layout of both kernels).  Each thread forms its two-channel sums; four
// rounds of 64 entries per sub-block are summed over the 64 channel pairs through a 64 KB
// shared-memory area [4 sub-blocks][16 entry quads][64 channel pairs] of float4.  The thread
// with index t keeps entry e(t) = 4 qd + lq of sub-block rb = t >> 6 in each round (see
// ns_diag_entry), for the store after the caller's readback.
#pragma once

#include "sm100.cuh"

namespace kda {
namespace nsdiag {

using namespace sm100;

// the reducer coordinates of thread t: entry quad qd (lanes 8 lq + (qd & 7), so the eight lanes
// of each phase of a 16-byte load read eight distinct bank groups), part lq, sub-block rb
__device__ __forceinline__ int reducer_qd(int t) { return (t & 7) | (((t >> 5) & 1) << 3); }
__device__ __forceinline__ int reducer_lq(int t) { return (t >> 3) & 3; }

// Adds this call's channel sums of the four rounds to dg (the caller's channels: one 128-channel
// slice of K; call once per slice).  kr / qr: the rows' words holding the channel pair, bf0 / bf1
// extract ch0 / ch1 as fp32; al[i] = (2^(G_i - G_(i-1)) of ch0, of ch1), i = 1 .. 15.  scr: the
// 64 KB area; bar_id / nthr: the named barrier of the 256 threads.
template <typename BF0, typename BF1>
__device__ __forceinline__ void pass(const uint32_t (&kr)[16], const uint32_t (&qr)[16], const float2 (&al)[16],
                                     BF0 bf_0, BF1 bf_1, int rq, int ch64, int t, uint32_t scr,
                                     uint32_t bar_id, float (&dg)[4]) {
    const int rb = t >> 6, qd = reducer_qd(t), lq = reducer_lq(t);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        // entry order of round q: columns cp = 2q, 15 - 2q, 2q + 1, 14 - 2q; per column j:
        // Aqk(j, j), then Akk(i, j), Aqk(i, j) for i = j + 1 .. 15 (32 entries per column pair)
        float buf[4];
        int slot = 0;
        auto emit = [&](float v) {
            buf[slot & 3] = v;
            if ((slot & 3) == 3)
                st_s128(scr + ((uint32_t)((rq * 16 + (slot >> 2)) * 64 + ch64) << 4), __float_as_uint(buf[0]),
                        __float_as_uint(buf[1]), __float_as_uint(buf[2]), __float_as_uint(buf[3]));
            ++slot;
        };
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int cp = 2 * q + (u >> 1);
            const int j = (u & 1) ? 15 - cp : cp;
            float2 kj = make_float2(bf_0(kr[j]), bf_1(kr[j]));
            emit(fmaf(bf_0(qr[j]), kj.x, bf_1(qr[j]) * kj.y));
#pragma unroll
            for (int i = j + 1; i < 16; ++i) {
                kj = __fmul2_rn(kj, al[i]);
                emit(fmaf(bf_0(kr[i]), kj.x, bf_1(kr[i]) * kj.y));
                emit(fmaf(bf_0(qr[i]), kj.x, bf_1(qr[i]) * kj.y));
            }
        }
        bar_sync(bar_id, 256);
        // entry 4 qd + lq of sub-block rb: the 64 channel pairs in four parts of 16 (a rotated
        // start keeps the warp's loads on distinct bank groups), then the parts
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int ln = 16 * lq + ((k + qd) & 15);
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(scr + ((uint32_t)((rb * 16 + qd) * 64 + ln) << 4)));
            sum.x += __uint_as_float(x0);
            sum.y += __uint_as_float(x1);
            sum.z += __uint_as_float(x2);
            sum.w += __uint_as_float(x3);
        }
#pragma unroll
        for (int m = 8; m <= 16; m <<= 1) {
            sum.x += __shfl_xor_sync(0xffffffffu, sum.x, m);
            sum.y += __shfl_xor_sync(0xffffffffu, sum.y, m);
            sum.z += __shfl_xor_sync(0xffffffffu, sum.z, m);
            sum.w += __shfl_xor_sync(0xffffffffu, sum.w, m);
        }
        dg[q] += (lq == 0) ? sum.x : (lq == 1) ? sum.y : (lq == 2) ? sum.z : sum.w;
        bar_sync(bar_id, 256);  // the next round rewrites the area
    }
}

// The entry thread t holds from round q: sub-block rb, row i, column j, and whether it is an
// Akk entry (else Aqk).
__device__ __forceinline__ void entry(int t, int q, int& rb, int& i, int& j, bool& akk) {
    rb = t >> 6;
    const int e = 4 * reducer_qd(t) + reducer_lq(t);
    const int cp = 2 * q + (e >> 5), x0 = e & 31, len0 = 31 - 2 * cp;
    j = (x0 < len0) ? cp : 15 - cp;
    const int x = (x0 < len0) ? x0 : x0 - len0;
    i = j + ((x + 1) >> 1);
    akk = (x & 1) != 0;
}

}  // namespace nsdiag
}  // namespace kda
