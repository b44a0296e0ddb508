// isd_verify_noalloc: isd_verify with its scratch in a fixed, library-owned
// device array, for callers that cannot allocate device memory themselves.
//
// The array below is reserved when the library's module loads on a device
// and stays reserved on every device that loaded it until the process exits.
// Host code cannot use the array's name as a device address (on the host it
// names a host-side shadow), so each device's address is looked up once,
// with that device current, by cudaGetSymbolAddress and cached here.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/isd.h"

namespace {

static_assert(ISD_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size is 256-byte granular");

static __device__ __align__(256) unsigned char g_verify_scratch[ISD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// The device address of the scratch array on the current device, looked up
// on the first call per device.
isd_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ISD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ISD_ERR_UNSUPPORTED;
    void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr)
                return ISD_ERR_CUDA;
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
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
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 ||
        (dtype != ISD_DTYPE_BF16 && dtype != ISD_DTYPE_F32))
        return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    const size_t need = isd_verify_workspace_bytes(num_seqs, total_positions, vocab, dtype);
    if (need == 0) return ISD_ERR_INVALID_ARG;
    if (need > ISD_NOALLOC_SCRATCH_BYTES) return ISD_ERR_WORKSPACE;  // batch too large for the array
    void* scratch = nullptr;
    const isd_status st = scratch_address(&scratch);
    if (st != ISD_OK) return st;
    // The array keeps whatever the previous call left; start from zeros, as
    // isd_verify requires of a fresh workspace.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return ISD_ERR_CUDA;
    return isd_verify(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                      total_positions, temperature, seed, offset, accept_len, out_tokens, ratio, alpha,
                      scratch, ISD_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
