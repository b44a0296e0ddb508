// isd_verify_noalloc: isd_verify with its scratch in a fixed, library-owned
// device array, for callers that cannot allocate device memory themselves.
//
// The array below is reserved when the library's module loads in a CUDA
// context and stays reserved until that context is destroyed.  Host code
// cannot use the array's name as a device address (on the host it names a
// host-side shadow), so the address is looked up by cudaGetSymbolAddress,
// with the device and context current, once per context, and cached under
// the context's unique id (cuCtxGetId: ids are never reused, so a context
// created later, after cudaDeviceReset for instance, never finds a stale
// address).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/isd.h"
#include "isd_internal.h"

namespace {

static_assert(ISD_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size is 256-byte granular");

static __device__ __align__(256) unsigned char g_verify_scratch[ISD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxContexts = 64;

struct ScratchEntry {
    unsigned long long ctx_id;
    void* ptr;
};

std::mutex g_setup_mutex;
ScratchEntry g_scratch[kMaxContexts];
int g_scratch_n = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Resolves the two driver calls through the runtime (no link-time driver
// dependency).
isd_status driver_calls() {
    if (g_ctx_get_current && g_ctx_get_id) return ISD_OK;
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult q0{}, q1{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &q0) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q0 != cudaDriverEntryPointSuccess || q1 != cudaDriverEntryPointSuccess || !f0 || !f1)
        return ISD_ERR_CUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f0);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f1);
    return ISD_OK;
}

// The device address of the scratch array in the current context, looked up
// on the first call in that context.
isd_status scratch_address(void** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    isd_status st = driver_calls();
    if (st != ISD_OK) return st;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return ISD_ERR_CUDA;
    void* fresh = nullptr;
    if (ctx == nullptr) {
        // No context yet: the runtime's first call makes the current
        // device's primary context current, and this lookup is that call.
        if (cudaGetSymbolAddress(&fresh, g_verify_scratch) != cudaSuccess || fresh == nullptr) return ISD_ERR_CUDA;
        if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return ISD_ERR_CUDA;
    }
    unsigned long long id = 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return ISD_ERR_CUDA;
    for (int k = 0; k < g_scratch_n; ++k)
        if (g_scratch[k].ctx_id == id) {
            *out = g_scratch[k].ptr;
            return ISD_OK;
        }
    if (fresh == nullptr &&
        (cudaGetSymbolAddress(&fresh, g_verify_scratch) != cudaSuccess || fresh == nullptr))
        return ISD_ERR_CUDA;
    // The table keeps the most recent contexts; the oldest entry makes room.
    if (g_scratch_n == kMaxContexts) {
        for (int k = 1; k < kMaxContexts; ++k) g_scratch[k - 1] = g_scratch[k];
        --g_scratch_n;
    }
    g_scratch[g_scratch_n++] = ScratchEntry{id, fresh};
    *out = fresh;
    return ISD_OK;
}

}  // namespace

extern "C" {

isd_status isd_verify_noalloc(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                              isd_dtype dtype, int vocab, const int32_t* tokens,
                              const int32_t* seq_offsets, int num_seqs, int total_positions,
                              const float* temperature, uint64_t seed, uint64_t offset,
                              int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                              void* stream) {
    // Every check isd_verify makes comes first: a refused call touches
    // neither the array nor the stream.
    const isd::VerifyOptions opts;
    const isd_status chk = isd::verify_check(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets,
                                             num_seqs, total_positions, temperature, accept_len, out_tokens,
                                             ratio, alpha, opts);
    if (chk != ISD_OK || num_seqs == 0) return chk;
    const size_t need = isd::verify_workspace(num_seqs, total_positions, vocab, dtype, false);
    if (need == 0) return ISD_ERR_INVALID_ARG;
    if (need > ISD_NOALLOC_SCRATCH_BYTES) return ISD_ERR_WORKSPACE;  // batch too large for the array
    void* scratch = nullptr;
    const isd_status st = scratch_address(&scratch);
    if (st != ISD_OK) return st;
    // The array keeps whatever the previous call left; start from zeros, as
    // isd_verify requires of a fresh workspace.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return ISD_ERR_CUDA;
    return isd::verify_run(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                           total_positions, temperature, seed, offset, accept_len, out_tokens, ratio, alpha, opts,
                           scratch, ISD_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
