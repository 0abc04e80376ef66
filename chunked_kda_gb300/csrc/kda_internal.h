// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

struct GateArgs {
    const void* g;
    bool g_bf16;
    const float* A_log;
    const float* dt_bias;
    int mode;
    float lb;
    const int32_t* cu;
    int N;  // logical sequences (B when dense)
    int B, T, H, K, C;
    float* out;
    cudaStream_t stream;
};

struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    bool qkv_bf16;
    bool g_bf16;
    const float* A_log;
    const float* dt_bias;
    int mode;  // 0 pre-gated, 1 safe, 2 non-safe
    float lb;
    const float* h0;
    float* hT;
    const int32_t* cu;
    int N;  // logical sequences (B when dense)
    int B, T, H, K, V, C;
    void* o;
    bool o_f32;  // o is float32 (else the qkv dtype)
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
    bool q_l2norm = false;  // scale each output row by 1 / sqrt(|q row|^2 + kQNormEps)
    int Hk = 0;             // query / key heads (a divisor of H; value head h reads h / (H / Hk))
    int* status = nullptr;  // optional device word: bit 0 set when a fused CTA gives up a wait
};
constexpr float kQNormEps = 1e-6f;

struct RecArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* gate;  // the per-token log2 decay (mode 3) or the raw gate of modes 0-2
    const void* beta;
    bool qkv_bf16;
    const float* h0;
    float* hT;
    const int32_t* cu;
    int N;
    int B, T, H, K, V;
    void* o;
    bool o_f32;  // o is float32 (else the qkv dtype)
    cudaStream_t stream;
    bool gate_bf16 = false;
    int mode = 3;  // 0 pre-gated (natural log), 1 safe, 2 non-safe, 3 log2 decay
    float lb = 0.f;
    const float* A_log = nullptr;
    const float* dt_bias = nullptr;
    unsigned flags = 0;  // KDA_FLAG_Q_L2NORM, KDA_FLAG_K_L2NORM, KDA_FLAG_BETA_LOGITS
    int Hk = 0;          // query / key heads (a divisor of H; value head h reads h / (H / Hk))
};

cudaError_t launch_gate(const GateArgs& a);
cudaError_t launch_recurrent(const RecArgs& a);

// float32 SIMT chunked path: stage-by-stage kernels with a device workspace
size_t precise_workspace_bytes(int B, int T, int H, int K, int V, int C, int N, bool packed);
cudaError_t launch_chunk_precise(const FwdArgs& a);

// bf16 fused single-kernel path (tcgen05 / TMEM / TMA); needs no workspace (its split schedule
// hands the state over in the unit's own output rows)
bool fused_supported(const FwdArgs& a);
bool fused_supported_dims(bool qkv_bf16, int K, int V, int C, int mode);
cudaError_t launch_chunk_fused(const FwdArgs& a);
// kernel launches of the fused path for these sizes on the current device (1, or 2 for the
// split schedule of dense inputs)
int fused_launch_count(int N, int H, int T, bool packed, bool o_f32, int mode);
// fused-kernel mbarrier waits that gave up on the current device (synchronises), optional reset
cudaError_t read_fused_timeouts(unsigned* count, bool reset);
// bf16 two-pass path (K = V in {128, 256}): a parallel pass per (chunk, head) writes T diag(beta)
// and Aqk into the workspace, a chain pass per (sequence, head, 128 value channels) runs the state
// scan; tcgen05 / TMEM / TMA throughout
bool twopass_supported_dims(bool qkv_bf16, int K, int V, int mode, int H);
// the images of pass 1, and for the balanced schedule of pass 2 its flags and state slots
size_t twopass_workspace_bytes(int T, int H, int K, int V, int N, bool packed);
cudaError_t launch_chunk_twopass(const FwdArgs& a);
cudaError_t read_twopass_timeouts(unsigned* count, bool reset);
// the fused path's test hooks (kda_test_hooks)
void set_test_hooks(int stall_chunk, int sm_count, int one_launch, int two_pass_d128);
bool hook_two_pass_d128();
int hook_stall_chunk();  // the forced-give-up chunk of both tensor-core paths (-1: none)
bool hook_one_launch();  // the plain grids whatever the plan (no split or balanced schedule)
int planned_sm_count();  // the SM count the schedules are planned for (test hook, else device)

// Which kernels run a chunked forward: the fused kernel (bf16, K = V = 128, every gate mode), the
// two-pass tensor-core kernels (bf16, K in {128, 256} with V a multiple of 128 other than
// K = V = 128, every gate mode; K = V = 128 too under the test hook), or the stage-by-stage
// float32 kernels (everything else)
enum class Path { Fused, TwoPass, Precise };
inline Path select_path(bool qkv_bf16, int K, int V, int C, int mode, int H, bool q_l2norm) {
    (void)q_l2norm;  // every path supports the deferred q l2norm
    const bool two = twopass_supported_dims(qkv_bf16, K, V, mode, H);
    if (fused_supported_dims(qkv_bf16, K, V, C, mode) && !(two && hook_two_pass_d128())) return Path::Fused;
    if (two && (K != 128 || V != 128 || hook_two_pass_d128())) return Path::TwoPass;
    return Path::Precise;
}

// sets the message kda_last_error() returns on this host thread
void record_error(const char* msg);

// every host check of the chunked forward (layout and size limits, dtypes, head dims, chunk
// size, gate mode and bound, null and misaligned pointers), shared by kda_chunk_fwd_ex and
// kda_chunk_fwd_noalloc; records the error message and fills *N (logical sequences)
kda_status check_chunk_args(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                            const void* g, kda_dtype g_dtype, const float* A_log,
                            const float* dt_bias, kda_gate_mode mode, float lower_bound,
                            const void* beta, const float* initial_state, float* final_state,
                            const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                            int V, int chunk_size, void* o, kda_dtype o_dtype, int n_qk_heads,
                            unsigned flags, int* N);

}  // namespace kda
