// kda_tc_util.cuh -- small device helpers shared by the tensor-core prefill
// kernels (kda_prefill_tc.cu, kda_prefill_c32.cu): the 128-byte-swizzled
// K-major operand layout, fast float32 exponentials, bf16 packing, chains of
// tcgen05.mma over K-blocks, and bulk copies between shared and global memory.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace tc {

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` of a K-major,
// 128B-swizzled operand (rows 128 B apart, chunk index XOR-ed with row % 8).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
// 8 floats -> one 16-byte chunk of bf16.
__device__ __forceinline__ void st_chunk(uint8_t *base, uint32_t off, const float *x) {
    uint4 v;
    v.x = pack_bf16(x[0], x[1]);
    v.y = pack_bf16(x[2], x[3]);
    v.z = pack_bf16(x[4], x[5]);
    v.w = pack_bf16(x[6], x[7]);
    *reinterpret_cast<uint4 *>(base + off) = v;
}
// one 16-byte chunk of bf16 -> 8 floats.
__device__ __forceinline__ void ld_chunk(const uint8_t *base, uint32_t off, float *x) {
    const uint4 v = *reinterpret_cast<const uint4 *>(base + off);
    const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void ld4(const float *p, float *x) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void ld8(const float *p, float *x) { ld4(p, x); ld4(p + 4, x + 4); }

// KSTEPS tcgen05 MMAs of K = 16 over K-major SW128 operands; K-blocks of 64
// elements are a_kblk / b_kblk bytes apart.
template <int KSTEPS>
__device__ __forceinline__ void mma_k(uint32_t d, uint32_t a_addr, uint32_t a_kblk, uint32_t b_addr,
                                      uint32_t b_kblk, uint32_t idesc, bool accumulate_first) {
    const uint64_t a0 = ptx::sdesc_kmajor_sw128(a_addr), b0 = ptx::sdesc_kmajor_sw128(b_addr);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        const uint64_t a = a0 + (uint64_t)(((ks >> 2) * a_kblk + (ks & 3) * 32u) >> 4);
        const uint64_t b = b0 + (uint64_t)(((ks >> 2) * b_kblk + (ks & 3) * 32u) >> 4);
        ptx::mma_bf16_ss(d, a, b, idesc, (ks > 0 || accumulate_first) ? 1u : 0u);
    }
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}

// Sequence bounds with the kernel's own bounds check: malformed offsets are
// reported and the sequence treated as empty.
__device__ __forceinline__ void seq_bounds(const int32_t *cu, int seq, int64_t total, uint32_t *status,
                                           int tid, int64_t &bos, int64_t &eos) {
    bos = cu[seq];
    eos = cu[seq + 1];
    if (bos < 0 || eos < bos || eos > total) {
        if (tid == 0) report_status(status, kDevBadSeqlens);
        bos = eos = 0;
    }
}

__device__ __forceinline__ void bulk_store(uint8_t *gdst, const uint8_t *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(gdst)),
                 "r"(ptx::smem_addr(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_copy_in(uint8_t *sdst, const uint8_t *gsrc, uint32_t bytes,
                                             uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            ptx::smem_addr(sdst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(ptx::smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_load(uint8_t *sdst, const uint8_t *gsrc, uint32_t bytes,
                                          uint64_t *bar) {
    ptx::mbar_arrive_expect_tx(bar, bytes);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            ptx::smem_addr(sdst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(ptx::smem_addr(bar))
        : "memory");
}

// The same copies with an L2 cache policy.
__device__ __forceinline__ void bulk_store_hint(uint8_t *gdst, const uint8_t *ssrc, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                     reinterpret_cast<uint64_t>(gdst)),
                 "r"(ptx::smem_addr(ssrc)), "r"(bytes), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void bulk_copy_in_hint(uint8_t *sdst, const uint8_t *gsrc, uint32_t bytes,
                                                  uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            ptx::smem_addr(sdst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(ptx::smem_addr(bar)), "l"(pol)
        : "memory");
}

}  // namespace tc
}  // namespace kda
