// kda_api.cu -- the extern "C" entry points declared in include/kda.h:
// argument validation on the host, kernel selection, launches on the caller's
// stream, and the device status word.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_testing.h"

namespace kda {
cudaError_t launch_gate(const void *z, bool bf16, const float *A, float *g, int64_t n_tokens,
                        int H, int dk, cudaStream_t st);
cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *z,
                          const float *A, const float *beta, float *state, void *out, int N,
                          int H, int dk, int dv, bool bf16, cudaStream_t st);
cudaError_t launch_prefill_serial(const void *q, const void *k, const void *v, const void *z,
                                  const float *A, const float *beta, const int32_t *cu,
                                  int num_seqs, int64_t total, int H, int dk, int dv, bool bf16,
                                  const float *s0, float *s1, void *out, uint32_t *status,
                                  cudaStream_t st, const float *g = nullptr);
cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *z,
                              const float *A, const float *beta, const int32_t *cu,
                              int num_seqs, int64_t total, int H, const float *s0, float *s1,
                              void *out, void *workspace, size_t workspace_bytes, cudaStream_t st);
cudaError_t launch_prefill_chunk_simt(const void *q, const void *k, const void *v, const void *z,
                                      const float *A, const float *beta, const int32_t *cu, int num_seqs,
                                      int64_t total, int H, int dk, int dv, bool bf16, const float *s0,
                                      float *s1, void *out, uint32_t *status, cudaStream_t st);
size_t prefill_tc_workspace_bytes(int64_t total, int num_seqs, int H);
size_t prefill_tc_logdecay_workspace_bytes(int64_t total, int num_seqs, int H);
cudaError_t launch_prefill_tc_logdecay(const void *q, const void *k, const void *v, const float *g,
                                       const float *beta, const int32_t *cu, int num_seqs,
                                       int64_t total, int H, const float *s0, float *s1, void *out,
                                       void *workspace, size_t workspace_bytes, cudaStream_t st);
int prefill_tc_launches(int64_t total, int num_seqs, int H, size_t workspace_bytes);
void set_test_expire(int mask);
size_t segment_map_workspace_bytes(int64_t total, int num_seqs, int H);
cudaError_t launch_segment_map(const void *q, const void *k, const void *v, const void *z,
                               const float *A, const float *beta, const int32_t *cu, int num_seqs,
                               int64_t total, int H, float *M_out, float *b_out, void *workspace,
                               size_t workspace_bytes, cudaStream_t st);
cudaError_t launch_state_compose(const float *M, const float *b, int n_maps, int N, int H, int dk,
                                 int dv, const float *init, float *states, cudaStream_t st);
cudaError_t launch_state_slots(float *pool, int pool_size, const int32_t *slots, float *states,
                               int N, int H, int dk, int dv, bool to_pool, uint32_t *status,
                               cudaStream_t st);
cudaError_t launch_decode_tokens(const void *q, const void *k, const void *v, const void *z,
                                 const float *A, const float *beta, float *pool, int pool_size,
                                 const int32_t *slots, void *out, int N, int n_tok, int H, int dk,
                                 int dv, bool bf16, uint32_t *status, cudaStream_t st);
cudaError_t launch_decode_tokens_tc(const void *q, const void *k, const void *v, const void *z, const float *A,
                                    const float *beta, float *pool, int pool_size, const int32_t *slots, void *out,
                                    int N, int n_tokens, int H, uint32_t *status, int sms, cudaStream_t st);
}  // namespace kda

namespace {

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
// from this many tokens per sequence kda_decode_tokens runs the chunked form
constexpr int kDecodeTcMinTokens = 4;
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool dtype_ok(kda_dtype_t t) { return t == KDA_F32 || t == KDA_BF16; }

kda_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// The tensor-core prefill covers bf16 with dk = dv = 128 and needs 16-byte
// aligned q/k/v/z (TMA descriptors) and out (16-byte stores).
bool use_tc(kda_dtype_t dt, int dk, int dv, const void *q, const void *k, const void *v,
            const void *z, const void *out, int64_t total) {
    return dt == KDA_BF16 && dk == 128 && dv == 128 && total > 0 && total < (int64_t(1) << 31) &&
           aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(z, 16) &&
           aligned(out, 16);
}

}  // namespace

extern "C" {

const char *kda_status_string(kda_status_t status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported shape or dtype";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA call or launch failed";
        case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT: device-side wait expired";
    }
    return "KDA_ERR_UNKNOWN";
}

kda_status_t kda_gate(const void *z, kda_dtype_t z_dtype, const float *A, float *g_out,
                      int64_t n_tokens, int H, int dk, kda_stream_t stream) {
    if (n_tokens < 0 || H <= 0 || dk <= 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(z_dtype)) return KDA_ERR_UNSUPPORTED;
    if (!dim_ok(dk)) return KDA_ERR_UNSUPPORTED;
    if (n_tokens == 0) return KDA_OK;
    if (!z || !A || !g_out) return KDA_ERR_INVALID_ARG;
    if (!aligned(z, 16) || !aligned(g_out, 16)) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_gate(z, z_dtype == KDA_BF16, A, g_out, n_tokens, H, dk,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t kda_prefill_workspace_size(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                  kda_dtype_t dtype) {
    if (num_seqs < 0) num_seqs = 0;
    size_t bytes = kda::kWsOrder + sizeof(int32_t) * (size_t)num_seqs;
    bytes = (bytes + 255) & ~size_t(255);
    // the tensor-core path can also use room for its split (few-chain) plan
    if (dtype == KDA_BF16 && dk == 128 && dv == 128 && H > 0 && total_tokens > 0 &&
        total_tokens < (int64_t(1) << 31)) {
        const size_t extra = kda::prefill_tc_workspace_bytes(total_tokens, num_seqs, H);
        if (extra > bytes) bytes = (extra + 255) & ~size_t(255);
    }
    return bytes;
}

size_t kda_prefill_logdecay_workspace_size(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                           kda_dtype_t dtype) {
    if (num_seqs < 0) num_seqs = 0;
    size_t bytes = kda::kWsOrder + sizeof(int32_t) * (size_t)num_seqs;
    bytes = (bytes + 255) & ~size_t(255);
    if (dtype == KDA_BF16 && dk == 128 && dv == 128 && H > 0 && total_tokens > 0 &&
        total_tokens < (int64_t(1) << 31)) {
        const size_t extra = kda::prefill_tc_logdecay_workspace_bytes(total_tokens, num_seqs, H);
        if (extra > bytes) bytes = (extra + 255) & ~size_t(255);
    }
    return bytes;
}

int kda_prefill_kernel_launches(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                kda_dtype_t dtype, size_t workspace_bytes) {
    if (num_seqs <= 0 || H <= 0) return 0;
    if (dtype == KDA_BF16 && dk == 128 && dv == 128 && total_tokens > 0 &&
        total_tokens < (int64_t(1) << 31))
        return kda::prefill_tc_launches(total_tokens, num_seqs, H, workspace_bytes);
    return 1;
}

kda_status_t kda_chunk_prefill(const void *q, const void *k, const void *v, const void *z,
                               const float *A, const float *beta, const int32_t *cu_seqlens,
                               int num_seqs, int64_t total_tokens, int H, int dk, int dv,
                               kda_dtype_t dtype, const float *initial_state,
                               float *final_state, void *out, void *workspace,
                               size_t workspace_bytes, kda_stream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || dk <= 0 || dv <= 0)
        return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (total_tokens >= (int64_t(1) << 31) || (int64_t)num_seqs * H >= (int64_t(1) << 31))
        return KDA_ERR_UNSUPPORTED;
    // the schedule area is required; room for the split plan is optional
    const size_t min_bytes = (kda::kWsOrder + sizeof(int32_t) * (size_t)num_seqs + 255) & ~size_t(255);
    if (!workspace || !aligned(workspace, 16) || workspace_bytes < min_bytes)
        return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return KDA_OK;
    if (!cu_seqlens || !A) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !z || !beta || !out)) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (use_tc(dtype, dk, dv, q, k, v, z, out, total_tokens)) {
        return from_cuda(kda::launch_prefill_tc(q, k, v, z, A, beta, cu_seqlens, num_seqs,
                                                total_tokens, H, initial_state, final_state, out,
                                                workspace, workspace_bytes, st));
    }
    // float32 inputs, dk or dv of 32 or 64 (or unaligned buffers): the chunkwise
    // algebra in float32 on the CUDA cores
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kda::kWsStatus);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    return from_cuda(kda::launch_prefill_chunk_simt(q, k, v, z, A, beta, cu_seqlens, num_seqs,
                                                    total_tokens, H, dk, dv, dtype == KDA_BF16,
                                                    initial_state, final_state, out, status, st));
}

kda_status_t kda_chunk_prefill_logdecay(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta,
                                        const int32_t *cu_seqlens, int num_seqs,
                                        int64_t total_tokens, int H, int dk, int dv,
                                        kda_dtype_t dtype, const float *initial_state,
                                        float *final_state, void *out, void *workspace,
                                        size_t workspace_bytes, kda_stream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || dk <= 0 || dv <= 0)
        return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (total_tokens >= (int64_t(1) << 31) || (int64_t)num_seqs * H >= (int64_t(1) << 31))
        return KDA_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 16) || workspace_bytes < 4) return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return KDA_OK;
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the chunked tensor-core path (bf16, 128 x 128 heads, few long chains) when
    // the workspace holds its plan; the token-serial kernel otherwise
    if (use_tc(dtype, dk, dv, q, k, v, g, out, total_tokens)) {
        const cudaError_t e = kda::launch_prefill_tc_logdecay(q, k, v, g, beta, cu_seqlens, num_seqs,
                                                              total_tokens, H, initial_state, final_state,
                                                              out, workspace, workspace_bytes, st);
        if (e != cudaErrorNotSupported) return from_cuda(e);
    }
    uint32_t *status = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + kda::kWsStatus);
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return KDA_ERR_CUDA;
    return from_cuda(kda::launch_prefill_serial(q, k, v, nullptr, nullptr, beta, cu_seqlens,
                                                num_seqs, total_tokens, H, dk, dv,
                                                dtype == KDA_BF16, initial_state, final_state, out,
                                                status, st, g));
}

kda_status_t kda_decode_step(const void *q, const void *k, const void *v, const void *z,
                             const float *A, const float *beta, float *state, void *out,
                             int N, int H, int dk, int dv, kda_dtype_t dtype,
                             kda_stream_t stream) {
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * H >= (int64_t(1) << 31)) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !z || !A || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned(state, 16)) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_decode(q, k, v, z, A, beta, state, out, N, H, dk, dv,
                                        dtype == KDA_BF16, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status_t kda_decode_tokens(const void *q, const void *k, const void *v, const void *z,
                               const float *A, const float *beta, float *state_pool,
                               int pool_size, const int32_t *slot_ids, void *out, int N,
                               int n_tokens, int H, int dk, int dv, kda_dtype_t dtype,
                               uint32_t *status, kda_stream_t stream) {
    if (N < 0 || n_tokens < 0 || pool_size < 0 || H <= 0 || dk <= 0 || dv <= 0)
        return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * n_tokens * H >= (int64_t(1) << 31) || (int64_t)N * H >= (int64_t(1) << 31))
        return KDA_ERR_UNSUPPORTED;
    if (N == 0 || n_tokens == 0) return KDA_OK;
    if (!slot_ids && pool_size < N) return KDA_ERR_INVALID_ARG;
    if (!q || !k || !v || !z || !A || !beta || !state_pool || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned(state_pool, 16)) return KDA_ERR_INVALID_ARG;
    // Several tokens per sequence, bf16, 128 x 128 heads: the chunked form on the
    // tensor cores (the tokens of a sequence as chunks of the fused prefill
    // kernel, the state from and back to its slot); one or a few tokens: the
    // token-serial kernel, which moves only the state.
    if (dtype == KDA_BF16 && dk == 128 && dv == 128 && n_tokens >= kDecodeTcMinTokens && aligned(q, 16) &&
        aligned(k, 16) && aligned(v, 16) && aligned(z, 16) && aligned(out, 16) && aligned(state_pool, 16)) {
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        return from_cuda(kda::launch_decode_tokens_tc(q, k, v, z, A, beta, state_pool, pool_size, slot_ids, out,
                                                      N, n_tokens, H, status, sms,
                                                      reinterpret_cast<cudaStream_t>(stream)));
    }
    return from_cuda(kda::launch_decode_tokens(q, k, v, z, A, beta, state_pool, pool_size, slot_ids,
                                               out, N, n_tokens, H, dk, dv, dtype == KDA_BF16,
                                               status, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status_t kda_state_slots_copy(float *state_pool, int pool_size, const int32_t *slot_ids,
                                  float *states, int N, int H, int dk, int dv, int to_pool,
                                  uint32_t *status, kda_stream_t stream) {
    if (N < 0 || pool_size < 0 || H <= 0 || dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (!state_pool || !slot_ids || !states) return KDA_ERR_INVALID_ARG;
    if (!aligned(state_pool, 16) || !aligned(states, 16)) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_state_slots(state_pool, pool_size, slot_ids, states, N, H, dk, dv,
                                             to_pool != 0, status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

void kda_testing_expire_next_wait(int kernels) { kda::set_test_expire(kernels); }

size_t kda_segment_map_workspace_size(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                      kda_dtype_t dtype) {
    if (dtype != KDA_BF16 || dk != 128 || dv != 128 || num_seqs <= 0 || H <= 0 || total_tokens <= 0 ||
        total_tokens >= (int64_t(1) << 31))
        return (kda::kWsOrder + sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 0) + 255) & ~size_t(255);
    return (kda::segment_map_workspace_bytes(total_tokens, num_seqs, H) + 255) & ~size_t(255);
}

kda_status_t kda_segment_map(const void *q, const void *k, const void *v, const void *z,
                             const float *A, const float *beta, const int32_t *cu_seqlens,
                             int num_seqs, int64_t total_tokens, int H, int dk, int dv,
                             kda_dtype_t dtype, float *M, float *b, void *workspace,
                             size_t workspace_bytes, kda_stream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (dtype != KDA_BF16 || dk != 128 || dv != 128) return KDA_ERR_UNSUPPORTED;
    if (total_tokens >= (int64_t(1) << 31) || (int64_t)num_seqs * H >= (int64_t(1) << 31))
        return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!cu_seqlens || !A || !M || !b || !workspace || !aligned(workspace, 16)) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (total_tokens == 0) {   // every map is the identity with no offset
        if (workspace_bytes < 4) return KDA_ERR_INVALID_ARG;
        if (cudaMemsetAsync(workspace, 0, 4, st) != cudaSuccess) return KDA_ERR_CUDA;
        kda::ComposeParams ident{};
        ident.init_identity = 1;
        ident.out_last = M;
        ident.last_prob = (int64_t)dk * dk;
        ident.R = 0;
        ident.ncols = dk;
        if (kda::launch_compose(ident, num_seqs * H, dk, st) != cudaSuccess) return KDA_ERR_CUDA;
        return from_cuda(cudaMemsetAsync(b, 0, sizeof(float) * (size_t)num_seqs * H * dk * dv, st));
    }
    if (!q || !k || !v || !z || !beta) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16)) return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < kda_segment_map_workspace_size(total_tokens, num_seqs, H, dk, dv, dtype))
        return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_segment_map(q, k, v, z, A, beta, cu_seqlens, num_seqs, total_tokens, H, M,
                                             b, workspace, workspace_bytes, st));
}

kda_status_t kda_state_compose(const float *M, const float *b, int n_maps, int num_seqs, int H, int dk,
                               int dv, const float *initial_state, float *states, kda_stream_t stream) {
    if (n_maps < 0 || num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * H >= (int64_t(1) << 31)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!states || (n_maps > 0 && (!M || !b))) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_state_compose(M, b, n_maps, num_seqs, H, dk, dv, initial_state, states,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

kda_status_t kda_check_device_status(const void *workspace, kda_stream_t stream) {
    if (!workspace) return KDA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, static_cast<const uint8_t *>(workspace) + kda::kWsStatus,
                        sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
    return static_cast<kda_status_t>(word);
}

}  // extern "C"
