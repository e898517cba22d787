// kda_chunk_simt.cu -- the chunkwise KDA prefill in float32 arithmetic on the
// CUDA cores, for the inputs the tensor-core path does not take: float32
// q/k/v/z (whose tolerance a bf16 operand cannot meet) and head sizes dk, dv in
// {32, 64} (and bf16 128 x 128 batches whose buffers are not 16-byte aligned).
//
// The same chunked algebra as the tensor-core prefill ("Kimi K3 internals
// analysis", molayo1419.me, section "Sequence mixing": the bounded gate
// g = -5 sigmoid(exp(A) z) and the delta-rule write after a channel-wise
// decay), with one 16-token decay tile per chunk.  Per (sequence, head) and
// chunk of C = 16 tokens with start state S0 and inclusive cumulative
// log-decay G_t (per key channel c):
//   K~ = k e^{G},  Q~ = q e^{G},  K^ = k e^{-G},  Kend = k e^{G_end - G}
//   L_ts = beta_t K~_t . K^_s  (s < t),   P_ts = Q~_t . K^_s  (s <= t)
//   T = (I + L)^{-1} Diag(beta)
//   U = T (V - K~ S0),   O = Q~ S0 + P U,   S1 = Diag(e^{G_end}) S0 + Kend^T U.
// The gate bounds every 16-token cumulative log-decay to (-80, 0], so e^{-G}
// stays below e^80 and every factor is finite in float32 (the tile bound of
// the same section); each L and P entry is a sum of products k_tc k_sc
// e^{G_tc - G_sc} with an exponent <= 0.
//
// One CTA of 256 threads per (sequence, head, block of JB value channels), JB
// = 32 when the batch gives at least two CTAs per SM, else 16 or 8 (more CTAs,
// fewer state rows per thread; the state-independent work of a chunk is then
// repeated per block); thread (j = tid % JB, row group rg = tid / JB) keeps
// rows rg DK/RG .. (rg + 1) DK/RG - 1 of state column j in registers, RG =
// 256 / JB.  Per chunk: stage the inputs (loaded into registers during the
// previous chunk), cumulative decay and the four operand tiles (one thread per
// key channel), L and P (one thread per (t, s) pair), the partial products
// K~ S0 and Q~ S0 over each row group, then the 16 x 16 forward substitution
// (one warp) beside the reduction of those partials into V - K~ S0 and Q~ S0,
// then U, then the output and the state update.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"

namespace kda {
namespace chunk_simt {

constexpr int C = 16;      // tokens per chunk (one 16-token decay tile)
constexpr int NT = 256;    // threads per CTA

template <int DK, int JB>
struct Smem {
    static constexpr int PK = DK + 1;   // padded row: column reads of the tiles are conflict-free
    static constexpr int RG = NT / JB;  // row groups
    float kt[C][PK], kh[C][PK], qt[C][PK], ke[C][PK];   // K~, K^, Q~, Kend (raw k, q, G while staging)
    float red[2][RG][C][JB + 1];                         // partial K~ S0 and Q~ S0 per row group
    float L[C][C + 1], P[C][C + 1], T[C][C + 1];
    float v[C][JB], rhs[C][JB + 1], qs[C][JB + 1], u[C][JB + 1];
    float eA[DK], gend[DK], beta[C];
};

template <typename T, int DK, int JB>
__global__ void __launch_bounds__(NT) prefill_chunk_simt_kernel(
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, const T *__restrict__ z,
    const float *__restrict__ A, const float *__restrict__ beta, const int32_t *__restrict__ cu_seqlens,
    int64_t total_tokens, int H, int dv, const float *__restrict__ initial_state,
    float *__restrict__ final_state, T *__restrict__ out, uint32_t *status) {
    constexpr int RG = NT / JB;    // row groups
    constexpr int RPT = DK / RG;   // state rows per thread
    static_assert(NT % JB == 0 && DK % RG == 0 && RPT >= 1, "value block");
    constexpr int KE = C * DK / NT;                 // staged k, q, z elements per thread
    constexpr int VE = (C * JB + NT - 1) / NT;      // staged v elements per thread
    extern __shared__ float4 smem_f4[];
    Smem<DK, JB> &sm = *reinterpret_cast<Smem<DK, JB> *>(smem_f4);

    const int sh = blockIdx.x;
    const int seq = sh / H, h = sh % H;
    const int j0 = blockIdx.y * JB;
    const int tid = threadIdx.x;
    const int j = tid % JB, rg = tid / JB;
    const int c0 = rg * RPT;

    int64_t bos = cu_seqlens[seq], eos = cu_seqlens[seq + 1];
    if (bos < 0 || eos < bos || eos > total_tokens) {
        if (tid == 0) report_status(status, kDevBadSeqlens);
        bos = eos = 0;
    }
    const int64_t sbase = ((int64_t)seq * H + h) * DK * dv;
    float S[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
        S[i] = initial_state ? initial_state[sbase + (int64_t)(c0 + i) * dv + j0 + j] : 0.f;
    for (int c = tid; c < DK; c += NT) sm.eA[c] = expf(A[h * DK + c]);

    // this thread's raw inputs of a chunk (element e = tid + NT i of the [C][DK]
    // and [C][JB] tiles; rows past the sequence end read as zero), loaded one
    // chunk ahead so that their latency is spent under the previous chunk
    float rk[KE], rq[KE], rz[KE], rv[VE], rb = 0.f;
    auto load_raw = [&](int64_t ta) {
        const int na = (int)((eos - ta) < C ? (eos - ta) : C);
#pragma unroll
        for (int i = 0; i < KE; ++i) {
            const int e = tid + NT * i, t = e / DK, c = e % DK;
            rk[i] = rq[i] = rz[i] = 0.f;
            if (t < na) {
                const int64_t idx = ((ta + t) * H + h) * DK + c;
                rk[i] = to_f32(k[idx]);
                rq[i] = to_f32(q[idx]);
                rz[i] = to_f32(z[idx]);
            }
        }
#pragma unroll
        for (int i = 0; i < VE; ++i) {
            const int e = tid + NT * i, t = e / JB, jj = e % JB;
            rv[i] = (e < C * JB && t < na) ? to_f32(v[((ta + t) * H + h) * (int64_t)dv + j0 + jj]) : 0.f;
        }
        rb = (tid < na) ? beta[(ta + tid) * H + h] : 0.f;
    };
    if (bos < eos) load_raw(bos);

    for (int64_t t0 = bos; t0 < eos; t0 += C) {
        const int nt = (int)((eos - t0) < C ? (eos - t0) : C);
        __syncthreads();   // the previous chunk is consumed (and eA is ready)
        // ---- stage: raw k and q, the gate's log-decay g (rows >= nt: zeros), v, beta
#pragma unroll
        for (int i = 0; i < KE; ++i) {
            const int e = tid + NT * i, t = e / DK, c = e % DK;
            sm.kh[t][c] = rk[i];
            sm.qt[t][c] = rq[i];
            sm.ke[t][c] = t < nt ? gate_log_decay(sm.eA[c], rz[i]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < VE; ++i) {
            const int e = tid + NT * i;
            if (e < C * JB) sm.v[e / JB][e % JB] = rv[i];
        }
        if (tid < C) sm.beta[tid] = rb;
        if (t0 + C < eos) load_raw(t0 + C);   // the next chunk's inputs, in flight meanwhile
        __syncthreads();
        // ---- cumulative decay and the operand tiles, one thread per key channel
        for (int c = tid; c < DK; c += NT) {
            float G = 0.f;
#pragma unroll
            for (int t = 0; t < C; ++t) {
                G += sm.ke[t][c];
                sm.ke[t][c] = G;
            }
            const float gend = expf(G);
            sm.gend[c] = gend;
#pragma unroll
            for (int t = 0; t < C; ++t) {
                const float Gt = sm.ke[t][c];
                const float kk = sm.kh[t][c], qq = sm.qt[t][c];
                const float eg = expf(Gt), ieg = expf(-Gt);
                sm.kt[t][c] = kk * eg;
                sm.qt[t][c] = qq * eg;
                sm.kh[t][c] = kk * ieg;
                sm.ke[t][c] = (kk * ieg) * gend;   // k e^{G_end - G_t}
            }
        }
        __syncthreads();
        // ---- L and P, one thread per (t, s) pair
        {
            const int t = tid / C, s = tid % C;
            float l = 0.f, p = 0.f;
            if (s <= t) {
#pragma unroll 8
                for (int c = 0; c < DK; ++c) {
                    const float kh = sm.kh[s][c];
                    l += sm.kt[t][c] * kh;
                    p += sm.qt[t][c] * kh;
                }
            }
            sm.L[t][s] = s < t ? sm.beta[t] * l : 0.f;
            sm.P[t][s] = s <= t ? p : 0.f;
        }
        // ---- partial K~ S0 and Q~ S0 over this thread's rows of column j
        {
            float ks[C], qs[C];
#pragma unroll
            for (int s = 0; s < C; ++s) { ks[s] = 0.f; qs[s] = 0.f; }
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float sv = S[i];
#pragma unroll
                for (int s = 0; s < C; ++s) {
                    ks[s] += sm.kt[s][c0 + i] * sv;
                    qs[s] += sm.qt[s][c0 + i] * sv;
                }
            }
#pragma unroll
            for (int s = 0; s < C; ++s) {
                sm.red[0][rg][s][j] = ks[s];
                sm.red[1][rg][s][j] = qs[s];
            }
        }
        __syncthreads();
        // ---- warp 0: T = (I + L)^{-1} Diag(beta) by forward substitution, one
        //      column per lane; warps 1-7: V - K~ S0 and Q~ S0 from the partials
        if (tid < 32) {
            if (tid < C) {
                const int s = tid;
                float y[C];
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    float acc = (t == s) ? 1.f : 0.f;
#pragma unroll
                    for (int m = 0; m < t; ++m) acc -= sm.L[t][m] * y[m];
                    y[t] = t >= s ? acc : 0.f;
                }
                const float bs = sm.beta[s];
#pragma unroll
                for (int t = 0; t < C; ++t) sm.T[t][s] = y[t] * bs;
            }
        } else {
            for (int e = tid - 32; e < C * JB; e += NT - 32) {
                const int s = e / JB, jj = e % JB;
                float ks = 0.f, qs = 0.f;
#pragma unroll
                for (int r = 0; r < RG; ++r) { ks += sm.red[0][r][s][jj]; qs += sm.red[1][r][s][jj]; }
                sm.rhs[s][jj] = sm.v[s][jj] - ks;
                sm.qs[s][jj] = qs;
            }
        }
        __syncthreads();
        // ---- U = T (V - K~ S0), two outputs per thread
        for (int e = tid; e < C * JB; e += NT) {
            const int t = e / JB, jj = e % JB;
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < C; ++s) acc += sm.T[t][s] * sm.rhs[s][jj];
            sm.u[t][jj] = acc;
        }
        __syncthreads();
        // ---- O = Q~ S0 + P U
        for (int e = tid; e < C * JB; e += NT) {
            const int t = e / JB, jj = e % JB;
            if (t < nt) {
                float acc = sm.qs[t][jj];
#pragma unroll
                for (int s = 0; s < C; ++s) acc += sm.P[t][s] * sm.u[s][jj];
                out[((t0 + t) * H + h) * (int64_t)dv + j0 + jj] = from_f32<T>(acc);
            }
        }
        // ---- S1 = Diag(e^{G_end}) S0 + Kend^T U on this thread's rows
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int c = c0 + i;
            float acc = sm.gend[c] * S[i];
#pragma unroll
            for (int s = 0; s < C; ++s) acc += sm.ke[s][c] * sm.u[s][j];
            S[i] = acc;
        }
    }
    if (final_state) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) final_state[sbase + (int64_t)(c0 + i) * dv + j0 + j] = S[i];
    }
}

template <typename T, int DK, int JB>
cudaError_t launch_jb(const void *q, const void *k, const void *v, const void *z, const float *A,
                      const float *beta, const int32_t *cu, int num_seqs, int64_t total, int H, int dv,
                      const float *s0, float *s1, void *out, uint32_t *status, cudaStream_t st) {
    const size_t smem = sizeof(Smem<DK, JB>);
    cudaError_t e = cudaFuncSetAttribute(prefill_chunk_simt_kernel<T, DK, JB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((int64_t)num_seqs * H), (unsigned)(dv / JB));
    prefill_chunk_simt_kernel<T, DK, JB><<<grid, NT, smem, st>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<const T *>(z), A, beta, cu, total, H, dv, s0, s1, static_cast<T *>(out), status);
    return cudaGetLastError();
}

// The value block: 32 channels when the batch gives at least two CTAs per SM,
// else 16 or 8 (each chain's chunks run one after another whatever the block,
// so a narrow block only adds CTAs and shortens each chunk's state work).
template <typename T, int DK>
cudaError_t launch_dk(const void *q, const void *k, const void *v, const void *z, const float *A,
                      const float *beta, const int32_t *cu, int num_seqs, int64_t total, int H, int dv,
                      const float *s0, float *s1, void *out, uint32_t *status, cudaStream_t st) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t chains = (int64_t)num_seqs * H;
    if (chains * (dv / 32) >= 2 * (int64_t)sms)
        return launch_jb<T, DK, 32>(q, k, v, z, A, beta, cu, num_seqs, total, H, dv, s0, s1, out, status, st);
    if (chains * (dv / 16) >= 2 * (int64_t)sms)
        return launch_jb<T, DK, 16>(q, k, v, z, A, beta, cu, num_seqs, total, H, dv, s0, s1, out, status, st);
    return launch_jb<T, DK, 8>(q, k, v, z, A, beta, cu, num_seqs, total, H, dv, s0, s1, out, status, st);
}

}  // namespace chunk_simt

// The chunkwise float32 prefill for every supported (dtype, dk, dv); dv a
// multiple of 32.
cudaError_t launch_prefill_chunk_simt(const void *q, const void *k, const void *v, const void *z,
                                      const float *A, const float *beta, const int32_t *cu, int num_seqs,
                                      int64_t total, int H, int dk, int dv, bool bf16, const float *s0,
                                      float *s1, void *out, uint32_t *status, cudaStream_t st) {
    using namespace chunk_simt;
    if (num_seqs <= 0) return cudaSuccess;
    if (dv % 32 != 0) return cudaErrorInvalidValue;
#define KDA_CHUNK_SIMT_CASE(TT, DKK)                                                                       \
    return launch_dk<TT, DKK>(q, k, v, z, A, beta, cu, num_seqs, total, H, dv, s0, s1, out, status, st)
    if (bf16) {
        if (dk == 32) KDA_CHUNK_SIMT_CASE(__nv_bfloat16, 32);
        if (dk == 64) KDA_CHUNK_SIMT_CASE(__nv_bfloat16, 64);
        if (dk == 128) KDA_CHUNK_SIMT_CASE(__nv_bfloat16, 128);
    } else {
        if (dk == 32) KDA_CHUNK_SIMT_CASE(float, 32);
        if (dk == 64) KDA_CHUNK_SIMT_CASE(float, 64);
        if (dk == 128) KDA_CHUNK_SIMT_CASE(float, 128);
    }
#undef KDA_CHUNK_SIMT_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
