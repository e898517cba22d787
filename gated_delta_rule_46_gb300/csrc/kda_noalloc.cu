// kda_noalloc.cu -- kda_chunk_prefill_noalloc: the prefill entry point for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run a prefill:
// plugin code hosted by an application that owns all device memory and hands
// out no allocator, serving loops whose device-memory budget is fixed at
// start-up, and code paths that must not take the allocator's implicit device
// synchronisation.  This variant needs no workspace from them: its scratch
// (status word, work counter, longest-first schedule) lives in the file-scope
// device array below, which every GPU that loads this library holds until the
// process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {
cudaError_t launch_prefill_chunk_simt(const void *q, const void *k, const void *v, const void *z,
                                      const float *A, const float *beta, const int32_t *cu, int num_seqs,
                                      int64_t total, int H, int dk, int dv, bool bf16, const float *s0,
                                      float *s1, void *out, uint32_t *status, cudaStream_t st);
cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *z,
                              const float *A, const float *beta, const int32_t *cu,
                              int num_seqs, int64_t total, int H, const float *s0, float *s1,
                              void *out, void *workspace, size_t workspace_bytes, cudaStream_t st);
}  // namespace kda

namespace {

constexpr size_t kScratchBytes = kda::kWsOrder + sizeof(int32_t) * KDA_NOALLOC_MAX_SEQS;

// The scratch itself.  In host code this name is only a host-side stand-in;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  Outside a stream
// capture it is looked up on every call (with the device current): after a
// host-side device reset the library's module is loaded anew and the array
// may move, so a cached address could be stale.  During a capture (when a
// lookup that loads the module must not happen) the address cached by the
// last call outside a capture is used.
cudaError_t scratch_on_current_device(cudaStream_t st, void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(st, &cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" kda_status_t kda_chunk_prefill_noalloc(
    const void *q, const void *k, const void *v, const void *z, const float *A,
    const float *beta, const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens, int H,
    int dk, int dv, kda_dtype_t dtype, const float *initial_state, float *final_state, void *out,
    kda_stream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || dk <= 0 || dv <= 0)
        return KDA_ERR_INVALID_ARG;
    if (num_seqs > KDA_NOALLOC_MAX_SEQS) return KDA_ERR_UNSUPPORTED;   // scratch holds no more
    if ((dtype != KDA_F32 && dtype != KDA_BF16) || !dim_ok(dk) || !dim_ok(dv))
        return KDA_ERR_UNSUPPORTED;
    if (total_tokens >= (int64_t(1) << 31) || (int64_t)num_seqs * H >= (int64_t(1) << 31))
        return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!cu_seqlens || !A) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !z || !beta || !out)) return KDA_ERR_INVALID_ARG;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if (scratch_on_current_device(st, &scratch) != cudaSuccess) return KDA_ERR_CUDA;
    const bool tc = dtype == KDA_BF16 && dk == 128 && dv == 128 && total_tokens > 0 &&
                    aligned16(q) && aligned16(k) && aligned16(v) && aligned16(z) &&
                    aligned16(out);
    if (tc) {
        // the schedule kernel zeroes the work counter and status word in the scratch
        return kda::launch_prefill_tc(q, k, v, z, A, beta, cu_seqlens, num_seqs, total_tokens,
                                      H, initial_state, final_state, out, scratch, kScratchBytes, st) ==
                       cudaSuccess
                   ? KDA_OK
                   : KDA_ERR_CUDA;
    }
    uint32_t *status = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) + kda::kWsStatus);
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return KDA_ERR_CUDA;
    return kda::launch_prefill_chunk_simt(q, k, v, z, A, beta, cu_seqlens, num_seqs, total_tokens, H,
                                          dk, dv, dtype == KDA_BF16, initial_state, final_state, out,
                                          status, st) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}
