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

}  // namespace kda
