/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library
 *          (libkda_gb300.so).
 *
 * The library computes the KDA forward: per head, a K x V FP32 state S that
 * decays per key channel and is updated by the delta rule,
 *
 *     S_t = Diag(exp(a_t)) S_{t-1};  S_t += beta_t k_t (v_t - S_t^T k_t)^T;
 *     o_t = S_t^T q_t / sqrt(K),
 *
 * in chunked (WY) form for prefill and token by token for decode.  Sources:
 *   - attention-gym PR #317 "Add fused recurrent_kda for decode and inference
 *     prefill", Agent note: call contract (q, k, v, gate, beta, initial_state,
 *     cu_seqlens, output_final_state), device-resident int32 offsets, repeated
 *     offsets as empty slots whose state passes through bitwise, a terminal
 *     offset below the physical capacity leaving the tail outside the
 *     contract, FP32 states with one leading entry per logical sequence, the
 *     recurrent gate as a per-token log2 decay, the 1/sqrt(K) query scale.
 *   - FLA skill page "fla-kda", sections "Gate modes" (pre-gated and safe
 *     in-kernel activations, -5 <= lower_bound < 0) and "Safe gate numerical
 *     note" (RCP_LN2 conversion to base 2, sub-chunk offsets before exp2).
 *   - Helion PR #3290 "Read only the causal columns in
 *     chunk_fwd_A_diag_anchored": chunk sizes 32 and 64, 16-row diagonal
 *     sub-blocks, causal columns only.
 *
 * Conventions for every entry point
 *   - All pointers are DEVICE pointers (cudaMalloc'd or equivalent), owned by
 *     the caller, contiguous in the stated layout, 16-byte aligned.  The
 *     library never allocates, never synchronises the stream and never reads
 *     cu_seqlens on the host; all work is enqueued on `stream`, so calls can be
 *     captured in a CUDA graph.
 *   - Sizes: B * T (tokens, or the packed capacity) below 2^31; B and n_seqs
 *     at most 65535.
 *   - Layout is token-major: q, k, g [B, T, H, K]; v, o [B, T, H, V];
 *     beta [B, T, H]; A_log, dt_bias [H, K] float32; states [N, H, K, V]
 *     float32 with N = n_seqs (packed) or B (dense).
 *   - Packed (varlen) mode: cu_seqlens != NULL, B must be 1, T is the physical
 *     capacity, cu_seqlens holds n_seqs + 1 non-decreasing int32 offsets with
 *     cu_seqlens[0] = 0 and cu_seqlens[n_seqs] <= T.  A repeated offset is an
 *     empty slot: its final state equals its initial state bit for bit (zeros
 *     when initial_state is NULL).  Rows of o at or beyond cu_seqlens[n_seqs]
 *     are neither read into any result nor written.  Offsets that break these
 *     rules are undefined behaviour (they live on the device and are not
 *     checked on the host).
 *   - Dense mode: cu_seqlens == NULL, n_seqs is ignored, B sequences of T.
 *   - initial_state == NULL means a zero initial state; final_state == NULL
 *     means the final state is not produced (output_final_state = False).
 *   - Every argument that the host can check is checked before any launch;
 *     a failed check returns KDA_ERR_INVALID_ARG or KDA_ERR_UNSUPPORTED and
 *     enqueues nothing.  A launch error returns KDA_ERR_CUDA.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* a cudaStream_t (NULL = the legacy default stream) */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad bound */
    KDA_ERR_UNSUPPORTED = 2, /* valid but not implemented (dtype, head dim, chunk size) */
    KDA_ERR_CUDA = 3         /* a CUDA launch or runtime call failed */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef enum {
    /* g already is the natural-log decay (FLA skill "fla-kda", "Gate modes",
       pre-gated mode); A_log, dt_bias and lower_bound are ignored.  The chunked
       bf16 kernel needs the bounded range -5 <= g <= 0 that attention-gym
       PR #345 calls the bounded-gate contract. */
    KDA_GATE_PRE = 0,
    /* safe in-kernel mode: a = lower_bound * sigmoid(exp(A_log) * (g + dt_bias)),
       A_log required, dt_bias optional, -5 <= lower_bound < 0 (FLA skill
       "fla-kda", "Gate modes") */
    KDA_GATE_SAFE = 1,
    /* in-kernel mode without the safe gate: a = -exp(A_log) * softplus(g + dt_bias),
       A_log required, dt_bias optional, lower_bound ignored; the decay is
       unbounded (same section).  The tensor-core paths anchor the off-diagonal
       scores at sub-block first rows (every factor <= 1) and compute the
       diagonal 16 x 16 blocks with per-pair factors 2^(G_i - G_j), j <= i; the
       float32 stage-by-stage path uses per-pair factors throughout. */
    KDA_GATE_NONSAFE = 2,
    /* the per-token log2 decay itself (S rows scale by 2^g): the gate of the
       recurrent entry points (attention-gym PR #317, Agent note); rejected by
       kda_gate_fwd and the chunked forward */
    KDA_GATE_LOG2 = 3
} kda_gate_mode;

/*
 * Gate activation followed by the chunk-local inclusive cumulative sum in
 * log2 units (FLA skill "fla-kda", "Safe gate numerical note": RCP_LN2
 * conversion; attention-gym PR #317: bounded_gate_cumsum, chunk_size = 1 gives
 * the recurrent entry point's per-token log2 gate).
 *
 *   g          [B, T, H, K], dtype g_dtype (KDA_F32 or KDA_BF16)
 *   A_log      [H, K] float32, required in the in-kernel modes (SAFE, NONSAFE)
 *   dt_bias    [H, K] float32 or NULL (= 0)
 *   chunk_size 1, 16, 32 or 64; chunks restart at every sequence start
 *   g_out      [B, T, H, K] float32: g_out[t] = (1/ln 2) * sum of the
 *              activation over the tokens of t's chunk up to and including t.
 *              Packed mode: rows at or beyond cu_seqlens[n_seqs] are not written.
 */
kda_status kda_gate_fwd(const void* g, kda_dtype g_dtype, const float* A_log,
                        const float* dt_bias, kda_gate_mode mode, float lower_bound,
                        const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                        int chunk_size, float* g_out, kda_stream_t stream);

/*
 * Bytes of device scratch memory kda_chunk_fwd needs for these sizes (0 when
 * the selected kernels need none).  n_seqs is the number of logical sequences
 * in packed mode and 0 in dense mode.  The caller allocates the scratch and
 * passes it to kda_chunk_fwd; its contents on entry do not matter.  Returns 0
 * as well for sizes kda_chunk_fwd would reject.
 */
size_t kda_chunk_workspace_bytes(kda_dtype qkv_dtype, int B, int T, int H, int K, int V,
                                 int chunk_size, int n_seqs);

/* The scratch size for a given gate mode: kda_chunk_workspace_bytes is this with
   KDA_GATE_SAFE (the pre-gated mode needs the same).  Every mode takes the same
   path for given dtypes and head sizes, so the sizes agree; the query exists for
   callers that pass the mode through. */
size_t kda_chunk_workspace_bytes_ex(kda_dtype qkv_dtype, int B, int T, int H, int K, int V,
                                    int chunk_size, int n_seqs, kda_gate_mode mode);

/*
 * Kernel launches one kda_chunk_fwd call with these sizes makes on the current device, for
 * profiling and launch accounting: 0 when there are no sequences, 6 on the stage-by-stage
 * path, 2 on the two-pass path, 1 on the fused path, 2 when the fused path uses its split
 * schedule.  n_seqs as for
 * kda_chunk_workspace_bytes (0 = dense).  Invalid sizes or enums: -1.  No device work.
 *
 * Split schedule (dense bf16 inputs, K = V = 128): one CTA per SM runs one (sequence, head)
 * unit, so U = f S + r units on S SMs take f + 1 unit-lengths with the last wave r / S full.
 * When that wave is at most half full, the call launches the fused kernel twice on
 * the stream: the first S units' leading chunks, then the other units whole together with
 * the first S units' remaining chunks, which fill the SMs the last whole units leave free.
 * The FP32 state crosses between the two launches through the unit's own rows of o (before
 * the second launch overwrites them), so the split needs no workspace and the results are
 * bitwise those of one launch.  kda_test_hooks can force one launch (for tests).
 */
int kda_chunk_fwd_launches(kda_dtype qkv_dtype, kda_dtype o_dtype, int B, int T, int H, int K, int V,
                           int chunk_size, int n_seqs, kda_gate_mode mode);

/*
 * Chunked KDA forward (prefill).  Steps: gate activation + chunk-local log2
 * cumsum; causal intra-chunk scores Akk (strictly lower, beta-scaled) and Aqk
 * (lower incl. diagonal, 1/sqrt(K)-scaled) on 16-token sub-blocks; the unit
 * lower-triangular solve T = (I + Akk)^-1; WY terms w = T (beta k 2^G),
 * u = T (beta v); the sequential inter-chunk state scan; the output
 * o = (1/sqrt(K)) (q 2^G) h + Aqk v_new.
 * Paths: bf16 inputs with K = V = 128 run the fused tensor-core kernel (one
 * launch, or two for the split schedule described with kda_chunk_fwd_launches;
 * no workspace); other bf16 inputs with K in {128, 256} and V a multiple of 128
 * run the two-pass tensor-core kernels (two launches: a parallel pass per chunk
 * and head that writes T diag(beta), Aqk and the state chain's operands into
 * the workspace, 121 KB per 64-token chunk and head at K = 256, then the state
 * chain per sequence, head and 128 value channels); every gate mode runs on
 * both.  Dense batches whose (sequence, head) units leave the state chain's last
 * wave part-empty run the chain as one cooperative launch of one CTA per SM
 * instead, the value blocks of a head on neighbouring SMs and the units' chunks
 * shared out evenly; a unit cut between two groups of SMs passes its FP32 state
 * through the workspace behind a flag (kda_chunk_workspace_bytes includes the
 * flags and S K x 128 FP32 slots, about 19 MB at K = 256 on 152 SMs; the call
 * zeroes the flags with cudaMemsetAsync on the stream).  The results are bitwise
 * those of one CTA per unit.  Everything else runs the stage-by-stage path (six launches, a workspace),
 * which computes in FP32 except that with bf16 inputs the safe-gate scores, the
 * WY terms and the output are tf32 tensor-core products with FP32 accumulation.
 *
 *   q, k       [B, T, H, K], dtype qkv_dtype; rows are used as given
 *   v          [B, T, H, V], dtype qkv_dtype
 *   g          [B, T, H, K], dtype g_dtype (raw gate in SAFE mode, the
 *              natural-log decay in PRE mode)
 *   beta       [B, T, H], dtype qkv_dtype, post-sigmoid
 *   o          [B, T, H, V], dtype o_dtype (output): the qkv dtype, or KDA_F32
 *              to keep the forward's FP32 result without the final rounding
 *   chunk_size 32 or 64 (Helion PR #3290: the two chunk sizes FLA's KDA accepts).
 *              The bf16 tensor-core paths (K = V = 128 or 256, pre-gated or safe
 *              gate) run both as 64-token chunks: the chunked form is exact for
 *              any chunk size, so only the rounding differs; the float32 path
 *              uses the size given.
 *   K, V       64, 128 or 256 (K == V on the bf16 tensor-core path; any pair
 *              of these on the float32 path)
 *   workspace  device scratch of at least kda_chunk_workspace_bytes(...) bytes,
 *              256-byte aligned; may be NULL when that size is 0.
 * initial_state and final_state may be the same buffer.
 */
kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                         const void* g, kda_dtype g_dtype, const float* A_log,
                         const float* dt_bias, kda_gate_mode mode, float lower_bound,
                         const void* beta, const float* initial_state, float* final_state,
                         const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                         int V, int chunk_size, void* o, kda_dtype o_dtype, void* workspace,
                         size_t workspace_bytes, kda_stream_t stream);

/* Option bits of kda_chunk_fwd_ex (Q_L2NORM) and kda_recurrent_fwd_ex (all three). */
#define KDA_FLAG_Q_L2NORM 1u    /* normalise every query row inside the forward */
#define KDA_FLAG_K_L2NORM 2u    /* normalise every key row inside the forward */
#define KDA_FLAG_BETA_LOGITS 4u /* beta holds logits; sigmoid(beta) is used */

/*
 * kda_chunk_fwd with options (attention-gym PR #345 "Fuse q l2norm into the
 * chunk_kda output kernel").  flags = 0 is kda_chunk_fwd.
 *
 *   KDA_FLAG_Q_L2NORM  each query row is used as q / sqrt(sum_d q[d]^2 + 1e-6)
 *                      (the eps floor of the callers' l2norm), without a
 *                      separate pass over q: an output row is linear in its
 *                      query row, so the scores are formed from q as given
 *                      and each finished output row is scaled once by that
 *                      row's 1/||q||.  Keys are used as given.  The final
 *                      state does not depend on q.  Forward only.
 *
 *   n_qk_heads         grouped value heads (FLA skill "fla-kda", "Correctness
 *                      checklist": HV > H): q and k are [B, T, n_qk_heads, K]
 *                      and value head h (of H) reads query / key head
 *                      h / (H / n_qk_heads); g, beta, v, o, A_log, dt_bias and
 *                      the states have H heads.  0 means H (multi-head); it
 *                      must divide H.
 *
 *   status             NULL, or a 4-byte aligned device int32 the caller owns:
 *                      the call ORs KDA_DEVICE_WAIT_GAVE_UP into it when a CTA
 *                      of the fused kernel gave up one of its bounded waits
 *                      (the outputs of that call are then not valid; the
 *                      context stays usable).  The library never clears it:
 *                      zero it before the call and read it once the caller's
 *                      stream has synchronised (no host synchronisation in
 *                      the library).  The stage-by-stage path has no waits
 *                      that can give up and leaves it untouched.
 *
 * Every other argument, the layouts and the errors are those of
 * kda_chunk_fwd; unknown flag bits return KDA_ERR_INVALID_ARG.
 */
kda_status kda_chunk_fwd_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                            const void* g, kda_dtype g_dtype, const float* A_log,
                            const float* dt_bias, kda_gate_mode mode, float lower_bound,
                            const void* beta, const float* initial_state, float* final_state,
                            const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                            int V, int chunk_size, void* o, kda_dtype o_dtype, void* workspace,
                            size_t workspace_bytes, int n_qk_heads, unsigned flags,
                            int32_t* status, kda_stream_t stream);

/* bit of kda_chunk_fwd_ex's status word: a fused-kernel CTA gave up a bounded wait */
#define KDA_DEVICE_WAIT_GAVE_UP 1

/*
 * Chunked forward for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point.  Some callers only
 * receive input and output pointers and may not call cudaMalloc: a plugin or
 * callback inside a host framework that owns all device memory, code running
 * under an allocator or capture mode that forbids new allocations, or an
 * embedded caller with a fixed memory budget.  kda_chunk_fwd needs a
 * caller-allocated workspace; this entry point instead runs the float32
 * stage-by-stage chunked path (for any input dtype) on a fixed scratch array
 * of KDA_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU
 * that loads the library holds until the process exits.  It allocates
 * nothing and calls no allocating routine.
 *
 *   Arguments, layouts and results: as for kda_chunk_fwd, without the
 *   workspace.  Sizes whose scratch would exceed KDA_NOALLOC_SCRATCH_BYTES
 *   (kda_chunk_workspace_bytes(KDA_F32, ...) of the same sizes, roughly 3.8 KB
 *   per token and head at K = V = 128, C = 64) are rejected with
 *   KDA_ERR_INVALID_ARG before anything is enqueued.
 *   Validation: the host checks of kda_chunk_fwd, the same code, run first
 *   (sizes below 2^31 tokens, dtypes, head dims, chunk size, gate, pointers).
 *   Set-up: every call looks up the scratch array's device address in the
 *   current context (cudaGetSymbolAddress, with the device current), so the
 *   address stays right after cudaDeviceReset or a new primary context.  The
 *   first call on a device may load the library's device code there; make
 *   that first call before any stream capture.
 *   Sharing: every call on a device uses the same scratch array and it keeps
 *   the last call's contents (each call writes every byte it reads, so nothing
 *   needs clearing); calls whose kernels overlap on the GPU, e.g. from two
 *   streams or two host threads, race on it and must be serialised.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (16u << 20)

kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                 const void* g, kda_dtype g_dtype, const float* A_log,
                                 const float* dt_bias, kda_gate_mode mode, float lower_bound,
                                 const void* beta, const float* initial_state, float* final_state,
                                 const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                                 int V, int chunk_size, void* o, kda_dtype o_dtype,
                                 kda_stream_t stream);

/*
 * Token-sequential KDA forward (decode and short prefill), attention-gym PR
 * #317: one program per (sequence, head, value block) scans the tokens with
 * its FP32 state block in registers and computes in FP32 for any input dtype.
 *
 *   gate       [B, T, H, K] float32: per-token LOG2 decay (S rows scale by
 *              2^gate), e.g. kda_gate_fwd(..., chunk_size = 1, ...)
 *   q, k, v, beta, o, o_dtype, states, cu_seqlens: as for kda_chunk_fwd.
 *   K, V       any value from 1 to 256 (rows and columns beyond them are masked
 *              inside the kernel; attention-gym PR #317 tests non-power-of-two
 *              K and V).
 * final_state may alias initial_state (in-place decode): each program reads
 * its whole state block before it writes any of it.
 */
kda_status kda_recurrent_fwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                             const float* gate, const void* beta, const float* initial_state,
                             float* final_state, const int32_t* cu_seqlens, int n_seqs, int B,
                             int T, int H, int K, int V, void* o, kda_dtype o_dtype,
                             kda_stream_t stream);

/*
 * kda_recurrent_fwd with the decode-side preprocessing inside the kernel (attention-gym
 * PR #317 test plan; FLA skill "fla-kda", "Correctness checklist": gate modes, raw beta
 * logits, qk l2norm in kernel), so a decode step needs no separate activation or
 * normalisation pass:
 *
 *   g, g_dtype  [B, T, H, K], KDA_F32 or KDA_BF16, read according to mode:
 *               KDA_GATE_LOG2 the per-token log2 decay (kda_recurrent_fwd's gate);
 *               KDA_GATE_PRE the natural-log decay; KDA_GATE_SAFE / KDA_GATE_NONSAFE
 *               the raw gate, activated per token as kda_gate_fwd does (A_log
 *               required, dt_bias optional, lower_bound as for kda_chunk_fwd)
 *   flags       KDA_FLAG_Q_L2NORM / KDA_FLAG_K_L2NORM: each q / k row is used as
 *               x / sqrt(sum x^2 + 1e-6); KDA_FLAG_BETA_LOGITS: beta holds logits
 *               and sigmoid(beta) is used.  Unknown bits return KDA_ERR_INVALID_ARG.
 *   n_qk_heads  grouped value heads, as for kda_chunk_fwd_ex (0 = H).
 * Every other argument is that of kda_recurrent_fwd; flags = 0 with KDA_GATE_LOG2, a
 * float32 g and n_qk_heads = 0 is kda_recurrent_fwd.
 */
kda_status kda_recurrent_fwd_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                const void* g, kda_dtype g_dtype, const float* A_log,
                                const float* dt_bias, kda_gate_mode mode, float lower_bound,
                                const void* beta, const float* initial_state, float* final_state,
                                const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                                int V, void* o, kda_dtype o_dtype, int n_qk_heads,
                                unsigned flags, kda_stream_t stream);

/* static, NUL-terminated description of a status code */
/*
 * Diagnostics of the tensor-core paths' bounded waits.  Every mbarrier wait of the fused
 * and two-pass chunked kernels gives up after a fixed number of polls; a CTA whose wait gave
 * up adds to a per-device counter, stops waiting, issuing MMAs and copies, lets the ones in
 * flight finish (bounded), frees its TMEM and returns, so the context stays usable but that
 * launch's outputs are not valid.  kda_fused_wait_timeouts writes the counters of the current
 * device to *count (their sum, 0 after normal runs) and zeroes them when reset != 0.  It copies from the device
 * and therefore synchronises with it: a diagnostic call, not for the hot path.  Null count:
 * KDA_ERR_INVALID_ARG; a failing copy: KDA_ERR_CUDA.
 */
kda_status kda_fused_wait_timeouts(unsigned int* count, int reset);

/*
 * Test hooks of the tensor-core paths, process-wide, all off by default and read by nothing
 * else (no environment variables).  For tests only; set them back to (-1, 0, 0, 0) afterwards.
 *   wait_timeout_chunk  >= 0: every CTA of later fused launches and of the two-pass state
 *                       chain waits, at that chunk and with a short limit, on an mbarrier
 *                       nothing completes, and takes the give-up path (counted by
 *                       kda_fused_wait_timeouts, flagged in the status word of
 *                       kda_chunk_fwd_ex); -1: off
 *   sm_count            > 0: plan the fused split schedule (kda_chunk_fwd_launches) and the
 *                       two-pass state chain's balanced schedule (kda_chunk_fwd) for this
 *                       many SMs instead of the device's (a chain plan for more SMs than the
 *                       device has runs one CTA per unit); 0: the device's
 *   one_launch          nonzero: never split a fused call into two launches, and run the
 *                       two-pass state chain as one CTA per unit
 *   two_pass_d128       nonzero: bf16 K = V = 128 calls run the two-pass kernels (with their
 *                       workspace, kda_chunk_workspace_bytes_ex) instead of the fused one
 * Always KDA_OK; no device work.
 */
kda_status kda_test_hooks(int wait_timeout_chunk, int sm_count, int one_launch, int two_pass_d128);

const char* kda_status_string(kda_status status);

/* the last error detail recorded by a failed call on this host thread ("" if none) */
const char* kda_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
