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
#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

// The scratch area.  Every GPU that loads this library holds these bytes in
// device memory until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

// The device address of g_noalloc_scratch in the current context.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, with the device current.  It is looked up on every call rather
// than cached: after cudaDeviceReset, or when the primary context is released and created
// again, the array lives at a new address, and a cached one would point at freed memory.
kda_status scratch_on_current_device(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        kda::record_error("kda_chunk_fwd_noalloc: cudaGetSymbolAddress of the scratch failed");
        return KDA_ERR_CUDA;
    }
    *out = p;
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(
    const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const void* g,
    kda_dtype g_dtype, const float* A_log, const float* dt_bias, kda_gate_mode mode,
    float lower_bound, const void* beta, const float* initial_state, float* final_state,
    const int32_t* cu_seqlens, int n_seqs, int B, int T, int H, int K, int V, int chunk_size,
    void* o, kda_dtype o_dtype, kda_stream_t stream) {
    kda::record_error("");
    // the same host checks as kda_chunk_fwd (sizes, dtypes, head dims, chunk size, gate,
    // null and misaligned pointers), before anything else
    int N = 0;
    kda_status st = kda::check_chunk_args(q, k, v, qkv_dtype, g, g_dtype, A_log, dt_bias, mode,
                                          lower_bound, beta, initial_state, final_state,
                                          cu_seqlens, n_seqs, B, T, H, K, V, chunk_size, o,
                                          o_dtype, 0, 0u, &N);
    if (st != KDA_OK) return st;
    if (N == 0) return KDA_OK;
    // the scratch this call needs must fit in the static area; nothing is allocated (the size
    // is computed in 64-bit arithmetic from sizes the checks above bounded)
    const size_t need = kda::precise_workspace_bytes(B, T, H, K, V, chunk_size, N, cu_seqlens != nullptr);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) {
        kda::record_error(
            "kda_chunk_fwd_noalloc: these sizes need more scratch than the fixed "
            "KDA_NOALLOC_SCRATCH_BYTES area holds; use kda_chunk_fwd with a workspace");
        return KDA_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    st = scratch_on_current_device(&scratch);
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
