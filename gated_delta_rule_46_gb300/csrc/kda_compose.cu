// kda_compose.cu -- composition of affine state maps, the exchange step of
// KDA context parallelism ("Kimi K3 internals analysis", molayo1419.me,
// section "3T급 MoE를 위한 인프라" (infrastructure for the 3T-class MoE), the
// paragraph on KDA context parallelism): over a segment of tokens the state map
// is affine, S_out = M S_in + b, so the segments of one long sequence can run
// on different workers, each from a zero state, and be joined afterwards by
// composing the maps in order.
//
// compose_kernel runs, for P independent problems, the recurrence
//   X_0 = init (or zeros, or the identity),   X_{r+1} = M_r X_r + B_r
// with X [dk][ncols], M_r [dk][dk], B_r [dk][ncols] float32 (B_r may be
// absent: zero).  One CTA per (problem, block of 32 columns): the columns of X
// do not mix, so the blocks run independently; M_r is staged in shared memory
// (rows padded by one word), X's block stays there between steps.  This is a
// small, latency-bound kernel (a few steps of dk x dk x 32 products per CTA):
// plain float32 FMAs, no tensor cores.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"

namespace kda {

template <int DK>
__global__ void __launch_bounds__(256) compose_kernel(const ComposeParams p) {
    constexpr int TPR = 256 / DK;   // threads per row of X's block
    constexpr int CPT = 32 / TPR;   // columns per thread
    extern __shared__ float csm[];
    float *Ms = csm;                              // [DK][DK + 1]
    float *Xs = csm + DK * (DK + 1);              // [DK][32]
    const int prob = blockIdx.x, j0 = blockIdx.y * 32, tid = threadIdx.x;
    const int row = tid / TPR, col0 = (tid % TPR) * CPT;
    const int64_t nc = p.ncols;
    int R = p.R;
    if (p.cu_seqlens) {
        const int seq = prob / p.H;
        int64_t bos = p.cu_seqlens[seq], eos = p.cu_seqlens[seq + 1];
        if (bos < 0 || eos < bos || eos > p.total) {
            if (tid == 0 && blockIdx.y == 0) report_status(p.status, kDevBadSeqlens);
            bos = eos = 0;
        }
        const int64_t nch = (eos - bos + 63) / 64;
        R = (int)((nch + p.seg_len - 1) / p.seg_len);
    }
    for (int e = tid; e < DK * 32; e += 256) {
        const int c = e >> 5, j = e & 31;
        float v;
        if (p.init) v = p.init[(int64_t)prob * p.init_prob + c * nc + j0 + j];
        else v = (p.init_identity && c == j0 + j) ? 1.f : 0.f;
        Xs[c * 32 + j] = v;
        if (p.out_all) p.out_all[(int64_t)prob * p.out_prob + c * nc + j0 + j] = v;
    }
    for (int r = 0; r < R; ++r) {
        __syncthreads();   // X_r complete, M_{r-1} no longer read
        const float *Mr = p.M + (int64_t)r * p.m_step + (int64_t)prob * p.m_prob;
        for (int e = tid; e < DK * DK; e += 256) Ms[(e / DK) * (DK + 1) + (e % DK)] = Mr[e];
        __syncthreads();
        float acc[CPT];
        const float *Br = p.B ? p.B + (int64_t)r * p.b_step + (int64_t)prob * p.b_prob + row * nc + j0 + col0
                              : nullptr;
#pragma unroll
        for (int i = 0; i < CPT; ++i) acc[i] = Br ? Br[i] : 0.f;
        const float *mrow = Ms + row * (DK + 1);
#pragma unroll 4
        for (int c2 = 0; c2 < DK; ++c2) {
            const float m = mrow[c2];
            const float *xr = Xs + c2 * 32 + col0;
#pragma unroll
            for (int i = 0; i < CPT; ++i) acc[i] = fmaf(m, xr[i], acc[i]);
        }
        __syncthreads();   // every thread has read X_r
#pragma unroll
        for (int i = 0; i < CPT; ++i) Xs[row * 32 + col0 + i] = acc[i];
        if (p.out_all) {
            float *o = p.out_all + (int64_t)(r + 1) * p.out_step + (int64_t)prob * p.out_prob + row * nc + j0 + col0;
#pragma unroll
            for (int i = 0; i < CPT; ++i) o[i] = acc[i];
        }
    }
    __syncthreads();
    if (p.out_last) {
        for (int e = tid; e < DK * 32; e += 256) {
            const int c = e >> 5, j = e & 31;
            p.out_last[(int64_t)prob * p.last_prob + c * nc + j0 + j] = Xs[c * 32 + j];
        }
    }
}

// Launches compose_kernel for P problems with dk rows; returns
// cudaErrorInvalidValue for an unsupported dk or ncols.
cudaError_t launch_compose(const ComposeParams &p, int P, int dk, cudaStream_t st) {
    if (P <= 0) return cudaSuccess;
    if (p.ncols % 32 != 0 || p.ncols <= 0) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)P, (unsigned)(p.ncols / 32));
    const size_t smem = (size_t)dk * (dk + 1) * 4 + (size_t)dk * 32 * 4;
    cudaError_t e;
    switch (dk) {
        case 32:
            e = cudaFuncSetAttribute(compose_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            compose_kernel<32><<<grid, 256, smem, st>>>(p);
            break;
        case 64:
            e = cudaFuncSetAttribute(compose_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            compose_kernel<64><<<grid, 256, smem, st>>>(p);
            break;
        case 128:
            e = cudaFuncSetAttribute(compose_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            compose_kernel<128><<<grid, 256, smem, st>>>(p);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// kda_state_compose: states[0] = initial (or zeros), states[r + 1] = M_r states[r] + b_r
// for every (sequence, head), maps laid out [n_maps][N][H][dk][dk] and [n_maps][N][H][dk][dv].
cudaError_t launch_state_compose(const float *M, const float *b, int n_maps, int N, int H, int dk,
                                 int dv, const float *init, float *states, cudaStream_t st) {
    const int64_t P = (int64_t)N * H;
    ComposeParams p{};
    p.M = M;
    p.m_prob = (int64_t)dk * dk;
    p.m_step = P * p.m_prob;
    p.B = b;
    p.b_prob = (int64_t)dk * dv;
    p.b_step = P * p.b_prob;
    p.init = init;
    p.init_prob = (int64_t)dk * dv;
    p.init_identity = 0;
    p.out_all = states;
    p.out_prob = (int64_t)dk * dv;
    p.out_step = P * p.out_prob;
    p.out_last = nullptr;
    p.R = n_maps;
    p.ncols = dv;
    p.cu_seqlens = nullptr;
    return launch_compose(p, (int)P, dk, st);
}

}  // namespace kda
