// C ABI of libkda_gb300.so: host-side validation, workspace sizing and
// dispatch to the kernels.  Declarations and the contract: include/kda.h.
#include <stdio.h>

#include <string>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

thread_local std::string g_last_error;

kda_status fail(kda_status st, const char* msg) {
    g_last_error = msg;
    return st;
}

kda_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    g_last_error = std::string("CUDA: ") + cudaGetErrorString(e);
    return KDA_ERR_CUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

// checks shared by every entry point; fills N (logical sequences)
kda_status check_layout(const int32_t* cu, int n_seqs, int B, int T, int H, int* N) {
    if (B < 0 || T < 0 || H <= 0) return fail(KDA_ERR_INVALID_ARG, "B, T must be >= 0 and H > 0");
    if ((long long)B * T * H > (1ll << 40)) return fail(KDA_ERR_INVALID_ARG, "input too large");
    // token coordinates (TMA) and chunk-slot numbers are 32-bit
    if ((long long)B * T >= (1ll << 31)) return fail(KDA_ERR_INVALID_ARG, "B * T must be below 2^31");
    if (cu) {
        if (B != 1) return fail(KDA_ERR_INVALID_ARG, "packed mode (cu_seqlens != NULL) needs B == 1");
        if (n_seqs < 0 || n_seqs > 65535)
            return fail(KDA_ERR_INVALID_ARG, "n_seqs must be in [0, 65535]");
        if (((uintptr_t)cu & 3u) != 0) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens misaligned");
        *N = n_seqs;
    } else {
        if (B > 65535) return fail(KDA_ERR_INVALID_ARG, "B must be <= 65535");
        *N = B;
    }
    return KDA_OK;
}

// gate mode and its parameters (FLA skill "fla-kda", "Gate modes")
kda_status check_gate(kda_gate_mode mode, const float* A_log, float lower_bound) {
    if (mode != KDA_GATE_PRE && mode != KDA_GATE_SAFE && mode != KDA_GATE_NONSAFE)
        return fail(KDA_ERR_INVALID_ARG, "gate mode");
    if (mode != KDA_GATE_PRE && !A_log) return fail(KDA_ERR_INVALID_ARG, "in-kernel gate needs A_log");
    if (mode == KDA_GATE_SAFE && !(lower_bound >= -5.0f && lower_bound < 0.0f))
        return fail(KDA_ERR_INVALID_ARG, "safe gate needs -5 <= lower_bound < 0");
    return KDA_OK;
}

}  // namespace

namespace kda {
void record_error(const char* msg) { g_last_error = msg; }

// The host checks of the chunked forward, shared by kda_chunk_fwd_ex and kda_chunk_fwd_noalloc;
// fills *N (logical sequences)
kda_status check_chunk_args(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                            const void* g, kda_dtype g_dtype, const float* A_log,
                            const float* dt_bias, kda_gate_mode mode, float lower_bound,
                            const void* beta, const float* initial_state, float* final_state,
                            const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                            int V, int chunk_size, void* o, kda_dtype o_dtype, int n_qk_heads,
                            unsigned flags, int* N) {
    if (flags & ~KDA_FLAG_Q_L2NORM) return fail(KDA_ERR_INVALID_ARG, "unknown flag bits");
    if (n_qk_heads < 0 || (n_qk_heads > 0 && (H <= 0 || H % n_qk_heads != 0)))
        return fail(KDA_ERR_INVALID_ARG, "n_qk_heads must divide H");
    kda_status st = check_layout(cu_seqlens, n_seqs, B, T, H, N);
    if (st != KDA_OK) return st;
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16) return fail(KDA_ERR_UNSUPPORTED, "qkv dtype");
    if (g_dtype != KDA_F32 && g_dtype != KDA_BF16) return fail(KDA_ERR_UNSUPPORTED, "g dtype");
    if (o_dtype != qkv_dtype && o_dtype != KDA_F32)
        return fail(KDA_ERR_UNSUPPORTED, "o dtype must be the qkv dtype or float32");
    if (!head_dim_ok(K) || !head_dim_ok(V)) return fail(KDA_ERR_UNSUPPORTED, "K and V must be 64, 128 or 256");
    if (chunk_size != 32 && chunk_size != 64) return fail(KDA_ERR_UNSUPPORTED, "chunk_size must be 32 or 64");
    st = check_gate(mode, A_log, lower_bound);
    if (st != KDA_OK) return st;
    const bool any_tokens = (long long)B * T > 0 && *N > 0;
    if (any_tokens && (!q || !k || !v || !g || !beta || !o))
        return fail(KDA_ERR_INVALID_ARG, "null q, k, v, g, beta or o");
    const void* ptrs[] = {q, k, v, g, beta, o, initial_state, final_state, A_log, dt_bias};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    return KDA_OK;
}
}  // namespace kda

extern "C" {

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported configuration";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA error";
    }
    return "unknown kda_status";
}

const char* kda_last_error(void) { return g_last_error.c_str(); }

kda_status kda_gate_fwd(const void* g, kda_dtype g_dtype, const float* A_log,
                        const float* dt_bias, kda_gate_mode mode, float lower_bound,
                        const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                        int chunk_size, float* g_out, kda_stream_t stream) {
    g_last_error.clear();
    int N = 0;
    kda_status st = check_layout(cu_seqlens, n_seqs, B, T, H, &N);
    if (st != KDA_OK) return st;
    if (K <= 0) return fail(KDA_ERR_INVALID_ARG, "K must be > 0");
    if (g_dtype != KDA_F32 && g_dtype != KDA_BF16) return fail(KDA_ERR_UNSUPPORTED, "g dtype");
    if (chunk_size != 1 && chunk_size != 16 && chunk_size != 32 && chunk_size != 64)
        return fail(KDA_ERR_UNSUPPORTED, "chunk_size must be 1, 16, 32 or 64");
    st = check_gate(mode, A_log, lower_bound);
    if (st != KDA_OK) return st;
    if ((long long)B * T == 0 || N == 0) return KDA_OK;
    if (!g || !g_out) return fail(KDA_ERR_INVALID_ARG, "null g or g_out");
    kda::GateArgs a{g, g_dtype == KDA_BF16, A_log, dt_bias, (int)mode, lower_bound, cu_seqlens,
                    N, B, T, H, K, chunk_size, g_out, (cudaStream_t)stream};
    return cuda_status(kda::launch_gate(a));
}

size_t kda_chunk_workspace_bytes(kda_dtype qkv_dtype, int B, int T, int H, int K, int V,
                                 int chunk_size, int n_seqs) {
    return kda_chunk_workspace_bytes_ex(qkv_dtype, B, T, H, K, V, chunk_size, n_seqs, KDA_GATE_SAFE);
}

size_t kda_chunk_workspace_bytes_ex(kda_dtype qkv_dtype, int B, int T, int H, int K, int V,
                                    int chunk_size, int n_seqs, kda_gate_mode mode) {
    if (B < 0 || T < 0 || H <= 0 || !head_dim_ok(K) || !head_dim_ok(V)) return 0;
    if (chunk_size != 32 && chunk_size != 64) return 0;
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16) return 0;
    if (mode != KDA_GATE_PRE && mode != KDA_GATE_SAFE && mode != KDA_GATE_NONSAFE) return 0;
    bool packed = n_seqs > 0;
    int N = packed ? n_seqs : B;
    switch (kda::select_path(qkv_dtype == KDA_BF16, K, V, chunk_size, (int)mode, H, false)) {
        case kda::Path::Fused: return 0;
        case kda::Path::TwoPass: return kda::twopass_workspace_bytes(T, H, K, V, N, packed);
        default: return kda::precise_workspace_bytes(B, T, H, K, V, chunk_size, N, packed);
    }
}

int kda_chunk_fwd_launches(kda_dtype qkv_dtype, kda_dtype o_dtype, int B, int T, int H, int K, int V,
                           int chunk_size, int n_seqs, kda_gate_mode mode) {
    if (B < 0 || T < 0 || H <= 0 || n_seqs < 0 || !head_dim_ok(K) || !head_dim_ok(V)) return -1;
    if (chunk_size != 32 && chunk_size != 64) return -1;
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16) return -1;
    if (o_dtype != qkv_dtype && o_dtype != KDA_F32) return -1;
    if (mode != KDA_GATE_PRE && mode != KDA_GATE_SAFE && mode != KDA_GATE_NONSAFE) return -1;
    const bool packed = n_seqs > 0;
    if (packed && B != 1) return -1;
    const int N = packed ? n_seqs : B;
    if (N == 0) return 0;
    switch (kda::select_path(qkv_dtype == KDA_BF16, K, V, chunk_size, (int)mode, H, false)) {
        case kda::Path::Fused: return kda::fused_launch_count(N, H, T, packed, o_dtype == KDA_F32, (int)mode);
        case kda::Path::TwoPass: return 2;
        default: return 6;
    }
}

kda_status kda_test_hooks(int wait_timeout_chunk, int sm_count, int one_launch, int two_pass_d128) {
    g_last_error.clear();
    kda::set_test_hooks(wait_timeout_chunk, sm_count, one_launch, two_pass_d128);
    return KDA_OK;
}

kda_status kda_fused_wait_timeouts(unsigned int* count, int reset) {
    g_last_error.clear();
    if (!count) return fail(KDA_ERR_INVALID_ARG, "null count");
    unsigned a = 0, b = 0;
    kda_status st = cuda_status(kda::read_fused_timeouts(&a, reset != 0));
    if (st != KDA_OK) return st;
    st = cuda_status(kda::read_twopass_timeouts(&b, reset != 0));
    *count = a + b;
    return st;
}

kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                         const void* g, kda_dtype g_dtype, const float* A_log,
                         const float* dt_bias, kda_gate_mode mode, float lower_bound,
                         const void* beta, const float* initial_state, float* final_state,
                         const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                         int V, int chunk_size, void* o, kda_dtype o_dtype, void* workspace,
                         size_t workspace_bytes, kda_stream_t stream) {
    return kda_chunk_fwd_ex(q, k, v, qkv_dtype, g, g_dtype, A_log, dt_bias, mode, lower_bound, beta,
                            initial_state, final_state, cu_seqlens, n_seqs, B, T, H, K, V,
                            chunk_size, o, o_dtype, workspace, workspace_bytes, 0, 0u, nullptr,
                            stream);
}

kda_status kda_chunk_fwd_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                            const void* g, kda_dtype g_dtype, const float* A_log,
                            const float* dt_bias, kda_gate_mode mode, float lower_bound,
                            const void* beta, const float* initial_state, float* final_state,
                            const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                            int V, int chunk_size, void* o, kda_dtype o_dtype, void* workspace,
                            size_t workspace_bytes, int n_qk_heads, unsigned flags,
                            int32_t* status, kda_stream_t stream) {
    g_last_error.clear();
    int N = 0;
    kda_status st = kda::check_chunk_args(q, k, v, qkv_dtype, g, g_dtype, A_log, dt_bias, mode,
                                          lower_bound, beta, initial_state, final_state,
                                          cu_seqlens, n_seqs, B, T, H, K, V, chunk_size, o,
                                          o_dtype, n_qk_heads, flags, &N);
    if (st != KDA_OK) return st;
    if (N == 0) return KDA_OK;
    size_t need = kda_chunk_workspace_bytes_ex(qkv_dtype, B, T, H, K, V, chunk_size,
                                               cu_seqlens ? n_seqs : 0, mode);
    if (workspace_bytes < need || (need > 0 && !workspace))
        return fail(KDA_ERR_INVALID_ARG, "workspace smaller than kda_chunk_workspace_bytes_ex()");
    if (workspace && ((uintptr_t)workspace & 255u) != 0)
        return fail(KDA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (status && ((uintptr_t)status & 3u) != 0)
        return fail(KDA_ERR_INVALID_ARG, "status must be 4-byte aligned");
    kda::FwdArgs a{q, k, v, g, beta, qkv_dtype == KDA_BF16, g_dtype == KDA_BF16, A_log, dt_bias,
                   (int)mode, lower_bound, initial_state, final_state, cu_seqlens, N, B, T, H, K,
                   V, chunk_size, o, o_dtype == KDA_F32, workspace, workspace_bytes,
                   (cudaStream_t)stream, (flags & KDA_FLAG_Q_L2NORM) != 0,
                   n_qk_heads > 0 ? n_qk_heads : H, reinterpret_cast<int*>(status)};
    switch (kda::select_path(a.qkv_bf16, K, V, chunk_size, (int)mode, H, a.q_l2norm)) {
        case kda::Path::Fused: return cuda_status(kda::launch_chunk_fused(a));
        case kda::Path::TwoPass: return cuda_status(kda::launch_chunk_twopass(a));
        default: return cuda_status(kda::launch_chunk_precise(a));
    }
}

kda_status kda_recurrent_fwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                             const float* gate, const void* beta, const float* initial_state,
                             float* final_state, const int32_t* cu_seqlens, int n_seqs, int B,
                             int T, int H, int K, int V, void* o, kda_dtype o_dtype,
                             kda_stream_t stream) {
    return kda_recurrent_fwd_ex(q, k, v, qkv_dtype, gate, KDA_F32, nullptr, nullptr, KDA_GATE_LOG2,
                                0.0f, beta, initial_state, final_state, cu_seqlens, n_seqs, B, T,
                                H, K, V, o, o_dtype, 0, 0u, stream);
}

kda_status kda_recurrent_fwd_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                const void* g, kda_dtype g_dtype, const float* A_log,
                                const float* dt_bias, kda_gate_mode mode, float lower_bound,
                                const void* beta, const float* initial_state, float* final_state,
                                const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K,
                                int V, void* o, kda_dtype o_dtype, int n_qk_heads,
                                unsigned flags, kda_stream_t stream) {
    g_last_error.clear();
    if (n_qk_heads < 0 || (n_qk_heads > 0 && (H <= 0 || H % n_qk_heads != 0)))
        return fail(KDA_ERR_INVALID_ARG, "n_qk_heads must divide H");
    int N = 0;
    kda_status st = check_layout(cu_seqlens, n_seqs, B, T, H, &N);
    if (st != KDA_OK) return st;
    if (flags & ~(KDA_FLAG_Q_L2NORM | KDA_FLAG_K_L2NORM | KDA_FLAG_BETA_LOGITS))
        return fail(KDA_ERR_INVALID_ARG, "unknown flag bits");
    if (qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16) return fail(KDA_ERR_UNSUPPORTED, "qkv dtype");
    if (g_dtype != KDA_F32 && g_dtype != KDA_BF16) return fail(KDA_ERR_UNSUPPORTED, "g dtype");
    if (o_dtype != qkv_dtype && o_dtype != KDA_F32)
        return fail(KDA_ERR_UNSUPPORTED, "o dtype must be the qkv dtype or float32");
    if (K < 1 || K > 256 || V < 1 || V > 256)
        return fail(KDA_ERR_UNSUPPORTED, "K and V must be in [1, 256]");
    if (mode != KDA_GATE_LOG2) {
        st = check_gate(mode, A_log, lower_bound);
        if (st != KDA_OK) return st;
    }
    const bool any_tokens = (long long)B * T > 0 && N > 0;
    if (any_tokens && (!q || !k || !v || !g || !beta || !o))
        return fail(KDA_ERR_INVALID_ARG, "null q, k, v, gate, beta or o");
    const void* ptrs[] = {q, k, v, g, beta, o, initial_state, final_state, A_log, dt_bias};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (N == 0) return KDA_OK;
    kda::RecArgs a{q, k, v, g, beta, qkv_dtype == KDA_BF16, initial_state, final_state,
                   cu_seqlens, N, B, T, H, K, V, o, o_dtype == KDA_F32, (cudaStream_t)stream,
                   g_dtype == KDA_BF16, (int)mode, lower_bound, A_log, dt_bias, flags,
                   n_qk_heads > 0 ? n_qk_heads : H};
    return cuda_status(kda::launch_recurrent(a));
}

}  // extern "C"
