// kda_common.cuh -- shared definitions of the CUDA kernels (not of the oracle).
//
// The KDA definitions restated here come from "Kimi K3 internals analysis"
// (molayo1419.me), section "Sequence mixing": the gate
// g = g_min * sigmoid(exp(A) * z) with g_min = -5, alpha = exp(g), and the
// delta-rule write into a fixed-size state after a channel-wise decay.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr float kGMin = -5.0f;

// Device status word values (kept in the caller's workspace).
constexpr uint32_t kDevOk = 0;
constexpr uint32_t kDevTimeout = KDA_ERR_DEVICE_TIMEOUT;
constexpr uint32_t kDevBadSeqlens = KDA_ERR_INVALID_ARG;

// Workspace layout of kda_chunk_prefill (offsets in bytes).
constexpr size_t kWsStatus = 0;      // uint32 device status
constexpr size_t kWsCounter = 16;    // uint32 dynamic work counter
constexpr size_t kWsOrder = 256;     // int32 [num_seqs] longest-first schedule

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Bounded gate: g = g_min * sigmoid(eA * z) with eA = exp(A) precomputed.
// Written as g_min / (1 + exp(-x)); for very negative x the exponential
// overflows to +inf and the quotient is -0, the correct limit.
__device__ __forceinline__ float gate_log_decay(float eA, float z) {
    const float x = eA * z;
    return kGMin / (1.0f + expf(-x));
}

// Records a device-side condition in the workspace status word (first one wins).
__device__ __forceinline__ void report_status(uint32_t *status, uint32_t code) {
    if (status) atomicCAS(status, kDevOk, code);
}

// Affine-map composition (kda_compose.cu): for P independent problems,
// X_0 = init (or zeros, or the identity), X_{r+1} = M_r X_r + B_r, with
// X [dk][ncols], M_r [dk][dk], B_r [dk][ncols] float32.
struct ComposeParams {
    const float *M;             // M_r of problem p at M + r m_step + p m_prob
    int64_t m_step, m_prob;
    const float *B;             // B_r of problem p at B + r b_step + p b_prob, or nullptr
    int64_t b_step, b_prob;
    const float *init;          // X_0 of problem p at init + p init_prob, or nullptr
    int64_t init_prob;
    int init_identity;          // with init == nullptr: X_0 = I (else zeros)
    float *out_all;             // X_r of problem p at out_all + r out_step + p out_prob (r = 0..R), or nullptr
    int64_t out_step, out_prob;
    float *out_last;            // X_R of problem p at out_last + p last_prob, or nullptr
    int64_t last_prob;
    int R;                      // steps of every problem, unless cu_seqlens is given
    int ncols;                  // columns of X (a multiple of 32)
    // per-problem step counts of a segment map: problem p = (sequence p / H,
    // head p % H) has ceil(ceil(len / 64) / seg_len) segments
    const int32_t *cu_seqlens;
    int H, seg_len;
    int64_t total;
    uint32_t *status;
};
cudaError_t launch_compose(const ComposeParams &p, int P, int dk, cudaStream_t st);

}  // namespace kda
