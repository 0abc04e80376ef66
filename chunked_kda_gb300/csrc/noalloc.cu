// kda_chunk_fwd_noalloc: the float32 stage-by-stage chunked forward with its
// scratch memory taken from a fixed array compiled into this library instead
// of a caller-provided workspace.  Declared and documented in include/kda.h.
//
// Who needs this: code that runs where device allocation is not allowed or
// not possible -- e.g. a callback or plugin that only receives input and
// output pointers from a host framework that owns all device memory, code
// running while a CUDA graph is being captured through an API that forbids
// cudaMalloc, or embedded callers with a fixed memory budget.  Such callers
// cannot call cudaMalloc for the workspace that kda_chunk_fwd needs.
#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

// The scratch area.  Every GPU that loads this library holds these bytes in
// device memory until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mu;
constexpr int kMaxDevices = 256;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device ordinal

// The address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the device address must come
// from cudaGetSymbolAddress, once per device, with that device current.
kda_status scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        kda::record_error("kda_chunk_fwd_noalloc: cudaGetDevice failed");
        return KDA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        kda::record_error("kda_chunk_fwd_noalloc: device ordinal out of range");
        return KDA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            kda::record_error("kda_chunk_fwd_noalloc: cudaGetSymbolAddress of the scratch failed");
            return KDA_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

bool hd_ok(int d) { return d == 64 || d == 128 || d == 256; }
bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(
    const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const void* g,
    kda_dtype g_dtype, const float* A_log, const float* dt_bias, kda_gate_mode mode,
    float lower_bound, const void* beta, const float* initial_state, float* final_state,
    const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K, int V, int chunk_size,
    void* o, kda_dtype o_dtype, kda_stream_t stream) {
    kda::record_error("");
    if (B < 0 || T < 0 || H <= 0 || (cu_seqlens && (B != 1 || n_seqs < 0 || n_seqs > 65535)) ||
        (!cu_seqlens && B > 65535)) {
        kda::record_error("kda_chunk_fwd_noalloc: bad B, T, H or n_seqs");
        return KDA_ERR_INVALID_ARG;
    }
    if ((qkv_dtype != KDA_F32 && qkv_dtype != KDA_BF16) || (g_dtype != KDA_F32 && g_dtype != KDA_BF16) ||
        (o_dtype != qkv_dtype && o_dtype != KDA_F32) || !hd_ok(K) || !hd_ok(V) ||
        (chunk_size != 32 && chunk_size != 64)) {
        kda::record_error("kda_chunk_fwd_noalloc: unsupported dtype, head dim or chunk size");
        return KDA_ERR_UNSUPPORTED;
    }
    if (mode != KDA_GATE_PRE && mode != KDA_GATE_SAFE && mode != KDA_GATE_NONSAFE) {
        kda::record_error("kda_chunk_fwd_noalloc: bad gate mode");
        return KDA_ERR_INVALID_ARG;
    }
    if (mode != KDA_GATE_PRE && !A_log) {
        kda::record_error("kda_chunk_fwd_noalloc: in-kernel gate needs A_log");
        return KDA_ERR_INVALID_ARG;
    }
    if (mode == KDA_GATE_SAFE && !(lower_bound >= -5.0f && lower_bound < 0.0f)) {
        kda::record_error("kda_chunk_fwd_noalloc: safe gate needs -5 <= lower_bound < 0");
        return KDA_ERR_INVALID_ARG;
    }
    const int N = cu_seqlens ? n_seqs : B;
    if ((long long)B * T > 0 && N > 0 && (!q || !k || !v || !g || !beta || !o)) {
        kda::record_error("kda_chunk_fwd_noalloc: null q, k, v, g, beta or o");
        return KDA_ERR_INVALID_ARG;
    }
    const void* ptrs[] = {q, k, v, g, beta, o, initial_state, final_state, A_log, dt_bias};
    for (const void* p : ptrs)
        if (p && !al16(p)) {
            kda::record_error("kda_chunk_fwd_noalloc: pointers must be 16-byte aligned");
            return KDA_ERR_INVALID_ARG;
        }
    if (((uintptr_t)cu_seqlens & 3u) != 0) {
        kda::record_error("kda_chunk_fwd_noalloc: cu_seqlens misaligned");
        return KDA_ERR_INVALID_ARG;
    }
    if (N == 0) return KDA_OK;
    // the scratch this call needs must fit in the static area; nothing is allocated
    const size_t need = kda::precise_workspace_bytes(B, T, H, K, V, chunk_size, N, cu_seqlens != nullptr);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) {
        kda::record_error(
            "kda_chunk_fwd_noalloc: these sizes need more scratch than the fixed "
            "KDA_NOALLOC_SCRATCH_BYTES area holds; use kda_chunk_fwd with a workspace");
        return KDA_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    kda_status st = scratch_on_current_device(&scratch);
    if (st != KDA_OK) return st;
    // Every region of the scratch is written before it is read within one call,
    // so nothing needs clearing between calls.
    kda::FwdArgs a{q, k, v, g, beta, qkv_dtype == KDA_BF16, g_dtype == KDA_BF16, A_log, dt_bias,
                   (int)mode, lower_bound, initial_state, final_state, cu_seqlens, N, B, T, H, K,
                   V, chunk_size, o, o_dtype == KDA_F32, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES,
                   (cudaStream_t)stream};
    cudaError_t e = kda::launch_chunk_precise(a);
    if (e != cudaSuccess) {
        kda::record_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}
