// kda_simt.cu -- the bandwidth-bound and scalar kernels of the KDA library:
//   * the standalone bounded gate,
//   * the one-token decode step that streams the float32 state in place,
//   * the token-serial float32 prefill (float32 inputs and the head sizes the
//     tensor-core prefill does not cover),
//   * the longest-first schedule used by the tensor-core prefill.
//
// KDA ("Kimi K3 internals analysis", molayo1419.me, section "Sequence mixing"):
//   g = -5 sigmoid(exp(A) z), alpha = exp(g)          (channel-wise, over dk)
//   S' = Diag(alpha) S;  u = beta (v - S'^T k);  S = S' + k u^T;  o = S^T q
// and o = S^T q = S'^T q + u (k . q), which lets one pass over S' give both
// column reductions.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"

namespace kda {

// ---------------------------------------------------------------------------
// Gate: g[t, h, c] = -5 sigmoid(exp(A[h, c]) z[t, h, c]).  HBM-bound elementwise
// kernel: 8 elements per thread per iteration (16-byte loads for bf16), exp(A)
// staged once per block in shared memory.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) gate_kernel(const T *__restrict__ z,
                                                   const float *__restrict__ A,
                                                   float *__restrict__ g, int64_t n_vec8,
                                                   int H, int dk, int use_table) {
    extern __shared__ float s_eA[];
    const int HD = H * dk;
    if (use_table) {
        for (int i = threadIdx.x; i < HD; i += blockDim.x) s_eA[i] = expf(A[i]);
        __syncthreads();
    }
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec8;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e0 = v * 8;
        const int hc = (int)(e0 % HD);  // 8 consecutive channels of one head (dk % 8 == 0)
        float zz[8];
        if constexpr (sizeof(T) == 2) {
            uint4 raw = *reinterpret_cast<const uint4 *>(z + e0);
            const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
            for (int i = 0; i < 8; ++i) zz[i] = __bfloat162float(b[i]);
        } else {
            float4 a = *reinterpret_cast<const float4 *>(z + e0);
            float4 b = *reinterpret_cast<const float4 *>(z + e0 + 4);
            zz[0] = a.x; zz[1] = a.y; zz[2] = a.z; zz[3] = a.w;
            zz[4] = b.x; zz[5] = b.y; zz[6] = b.z; zz[7] = b.w;
        }
        float out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float eA = use_table ? s_eA[hc + i] : expf(A[hc + i]);
            out[i] = gate_log_decay(eA, zz[i]);
        }
        float4 *dst = reinterpret_cast<float4 *>(g + e0);
        dst[0] = make_float4(out[0], out[1], out[2], out[3]);
        dst[1] = make_float4(out[4], out[5], out[6], out[7]);
    }
}

// ---------------------------------------------------------------------------
// Decode step: one CTA per (sequence, head), 256 threads.  The dk x dv float32
// state is read once with 16-byte loads, held in registers, decayed, reduced
// over its rows (S'^T k and S'^T q) and written back once in place.
// ---------------------------------------------------------------------------
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(256) decode_kernel(
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ z, const float *__restrict__ A, const float *__restrict__ beta,
    float *__restrict__ state, T *__restrict__ out, int H) {
    constexpr int F = DV / 4;             // float4 per state row
    constexpr int ROWS_PER_PASS = 256 / F;
    constexpr int PASSES = DK / ROWS_PER_PASS;
    static_assert(DK % ROWS_PER_PASS == 0, "decode tiling");

    __shared__ float s_alpha[DK], s_k[DK], s_q[DK];
    __shared__ float s_red[2][ROWS_PER_PASS][DV + 1];
    __shared__ float s_u[DV];
    __shared__ float s_kq;

    const int nh = blockIdx.x;            // n * H + h
    const int h = nh % H;
    const int tid = threadIdx.x;
    const int64_t rowk = (int64_t)nh * DK, rowv = (int64_t)nh * DV;

    // issue the state loads first: they are the bytes that matter
    const int col4 = tid % F;
    const int r0 = tid / F;
    float4 *S4 = reinterpret_cast<float4 *>(state + (int64_t)nh * DK * DV);
    float4 s[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) s[p] = S4[(int64_t)(r0 + p * ROWS_PER_PASS) * F + col4];

    if (tid < DK) {
        const float zz = to_f32(z[rowk + tid]);
        s_alpha[tid] = expf(gate_log_decay(expf(A[h * DK + tid]), zz));
        s_k[tid] = to_f32(k[rowk + tid]);
        s_q[tid] = to_f32(q[rowk + tid]);
    }
    __syncthreads();
    if (tid < 32) {
        float acc = 0.f;
        for (int c = tid; c < DK; c += 32) acc += s_k[c] * s_q[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (tid == 0) s_kq = acc;
    }

    // S' = Diag(alpha) S ; partial column sums of S'^T k and S'^T q
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int c = r0 + p * ROWS_PER_PASS;
        const float a = s_alpha[c], kc = s_k[c], qc = s_q[c];
        s[p].x *= a; s[p].y *= a; s[p].z *= a; s[p].w *= a;
        pk.x += s[p].x * kc; pk.y += s[p].y * kc; pk.z += s[p].z * kc; pk.w += s[p].w * kc;
        pq.x += s[p].x * qc; pq.y += s[p].y * qc; pq.z += s[p].z * qc; pq.w += s[p].w * qc;
    }
    s_red[0][r0][4 * col4 + 0] = pk.x; s_red[0][r0][4 * col4 + 1] = pk.y;
    s_red[0][r0][4 * col4 + 2] = pk.z; s_red[0][r0][4 * col4 + 3] = pk.w;
    s_red[1][r0][4 * col4 + 0] = pq.x; s_red[1][r0][4 * col4 + 1] = pq.y;
    s_red[1][r0][4 * col4 + 2] = pq.z; s_red[1][r0][4 * col4 + 3] = pq.w;
    __syncthreads();
    if (tid < DV) {
        float kv = 0.f, sq = 0.f;
#pragma unroll 8
        for (int r = 0; r < ROWS_PER_PASS; ++r) { kv += s_red[0][r][tid]; sq += s_red[1][r][tid]; }
        const float u = beta[nh] * (to_f32(v[rowv + tid]) - kv);
        s_u[tid] = u;
        out[rowv + tid] = from_f32<T>(sq + u * s_kq);
    }
    __syncthreads();
    // S = S' + k u^T, written back in place
    const float u0 = s_u[4 * col4], u1 = s_u[4 * col4 + 1], u2 = s_u[4 * col4 + 2],
                u3 = s_u[4 * col4 + 3];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
        const int c = r0 + p * ROWS_PER_PASS;
        const float kc = s_k[c];
        s[p].x += kc * u0; s[p].y += kc * u1; s[p].z += kc * u2; s[p].w += kc * u3;
        S4[(int64_t)c * F + col4] = s[p];
    }
}

// ---------------------------------------------------------------------------
// Token-serial prefill in float32.  Grid (num_seqs * H, dv / 32); 128 threads
// own 32 state columns: warp w owns columns 8w..8w+7, lane = 8 * rg + col, and
// each thread keeps rows rg*DK/4 .. rg*DK/4 + DK/4 - 1 of its column in
// registers.  Per token the two column reductions are four-thread shuffles,
// so tokens advance without block barriers; inputs are staged TB tokens at a
// time.
// ---------------------------------------------------------------------------
template <typename T, int DK>
__global__ void __launch_bounds__(128) prefill_serial_kernel(
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ z, const float *__restrict__ A, const float *__restrict__ beta,
    const int32_t *__restrict__ cu_seqlens, int64_t total_tokens, int H, int dv,
    const float *__restrict__ initial_state, float *__restrict__ final_state,
    T *__restrict__ out, uint32_t *status, const float *__restrict__ g_direct) {
    constexpr int TB = 16;                 // tokens staged per round
    constexpr int RPT = DK / 4;            // state rows per thread
    constexpr int PAD = DK + DK / 32;      // padded row so the 4 row groups hit distinct banks
    __shared__ float s_a[TB][PAD], s_k[TB][PAD], s_q[TB][PAD];
    __shared__ float s_v[TB][32], s_b[TB], s_kq[TB];
    __shared__ float s_eA[DK];

    const int sh = blockIdx.x;
    const int seq = sh / H, h = sh % H;
    const int j0 = blockIdx.y * 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 3, colw = lane & 7;
    const int j = j0 + warp * 8 + colw;    // this thread's state column
    const int cbase = rg * RPT;

    int64_t bos = cu_seqlens[seq], eos = cu_seqlens[seq + 1];
    if (bos < 0 || eos < bos || eos > total_tokens) {
        if (tid == 0) report_status(status, kDevBadSeqlens);
        bos = eos = 0;
    }
    const int64_t sbase = ((int64_t)seq * H + h) * DK * dv;

    float S[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
        S[i] = initial_state ? initial_state[sbase + (int64_t)(cbase + i) * dv + j] : 0.f;
    if (!g_direct)
        for (int c = tid; c < DK; c += 128) s_eA[c] = expf(A[h * DK + c]);

    for (int64_t t0 = bos; t0 < eos; t0 += TB) {
        const int nt = (int)((eos - t0) < TB ? (eos - t0) : TB);
        __syncthreads();   // previous round fully consumed (and s_eA ready)
        for (int e = tid; e < nt * DK; e += 128) {
            const int tt = e / DK, c = e % DK;
            const int64_t idx = ((t0 + tt) * H + h) * DK + c;
            const int pc = c + c / 32;
            // alpha = exp(g): g from the bounded gate, or given directly (any value)
            s_a[tt][pc] = expf(g_direct ? g_direct[idx] : gate_log_decay(s_eA[c], to_f32(z[idx])));
            s_k[tt][pc] = to_f32(k[idx]);
            s_q[tt][pc] = to_f32(q[idx]);
        }
        for (int e = tid; e < nt * 32; e += 128) {
            const int tt = e / 32, jj = e % 32;
            s_v[tt][jj] = to_f32(v[((t0 + tt) * H + h) * (int64_t)dv + j0 + jj]);
        }
        if (tid < nt) s_b[tid] = beta[(t0 + tid) * H + h];
        __syncthreads();
        // k . q per staged token (one warp per token, round robin)
        for (int tt = warp; tt < nt; tt += 4) {
            float acc = 0.f;
            for (int c = lane; c < DK; c += 32) acc += s_k[tt][c + c / 32] * s_q[tt][c + c / 32];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) s_kq[tt] = acc;
        }
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            float kv = 0.f, sq = 0.f;
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int pc = cbase + i + (cbase + i) / 32;
                S[i] *= s_a[tt][pc];
                kv += S[i] * s_k[tt][pc];
                sq += S[i] * s_q[tt][pc];
            }
            kv += __shfl_xor_sync(0xffffffffu, kv, 8);
            kv += __shfl_xor_sync(0xffffffffu, kv, 16);
            sq += __shfl_xor_sync(0xffffffffu, sq, 8);
            sq += __shfl_xor_sync(0xffffffffu, sq, 16);
            const float u = s_b[tt] * (s_v[tt][warp * 8 + colw] - kv);
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int pc = cbase + i + (cbase + i) / 32;
                S[i] += s_k[tt][pc] * u;
            }
            if (rg == 0) out[((t0 + tt) * H + h) * (int64_t)dv + j] = from_f32<T>(sq + u * s_kq[tt]);
        }
    }
    if (final_state) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) final_state[sbase + (int64_t)(cbase + i) * dv + j] = S[i];
    }
}

// ---------------------------------------------------------------------------
// Schedule for the tensor-core prefill: sequence indices ordered by length,
// longest first (ties by index), plus a zeroed work counter and status word.
// One block; bitonic sort in shared memory for up to kSortMax sequences, the
// identity order beyond that.
// ---------------------------------------------------------------------------
constexpr int kSortMax = 4096;

__global__ void __launch_bounds__(1024) schedule_kernel(const int32_t *__restrict__ cu_seqlens,
                                                        int num_seqs, int32_t *order,
                                                        uint32_t *counter, uint32_t *status) {
    __shared__ int64_t s_key[kSortMax];
    const int tid = threadIdx.x;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the prefill kernel may start its setup
    if (tid == 0) { *counter = 0u; *status = kDevOk; }
    if (num_seqs > kSortMax) {
        for (int i = tid; i < num_seqs; i += blockDim.x) order[i] = i;
        return;
    }
    int n = 1;
    while (n < num_seqs) n <<= 1;
    for (int i = tid; i < n; i += blockDim.x) {
        int64_t key;
        if (i < num_seqs) {
            int64_t len = (int64_t)cu_seqlens[i + 1] - cu_seqlens[i];
            if (len < 0) len = 0;
            // descending length, ascending index: sort ascending on (-len, i)
            key = ((int64_t)(0x7fffffff - (len > 0x7ffffffe ? 0x7ffffffe : len)) << 32) | (uint32_t)i;
        } else {
            key = INT64_MAX;
        }
        s_key[i] = key;
    }
    __syncthreads();
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n; i += blockDim.x) {
                const int p = i ^ stride;
                if (p > i) {
                    const bool up = ((i & size) == 0);
                    const int64_t a = s_key[i], b = s_key[p];
                    if ((a > b) == up) { s_key[i] = b; s_key[p] = a; }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < num_seqs; i += blockDim.x) order[i] = (int32_t)(s_key[i] & 0xffffffff);
}

// ---------------------------------------------------------------------------
// Host-side launchers (internal ABI between the translation units).
// ---------------------------------------------------------------------------
cudaError_t launch_gate(const void *z, bool bf16, const float *A, float *g, int64_t n_tokens,
                        int H, int dk, cudaStream_t st) {
    const int64_t n = n_tokens * H * dk;
    if (n == 0) return cudaSuccess;
    const int64_t nv = n / 8;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (nv + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    const int use_table = (H * dk <= 8192) ? 1 : 0;
    const size_t smem = use_table ? sizeof(float) * H * dk : 0;
    if (bf16)
        gate_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, smem, st>>>(
            (const __nv_bfloat16 *)z, A, g, nv, H, dk, use_table);
    else
        gate_kernel<float><<<(unsigned)blocks, 256, smem, st>>>((const float *)z, A, g, nv, H, dk,
                                                                use_table);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t decode_dispatch(const void *q, const void *k, const void *v, const void *z,
                                   const float *A, const float *beta, float *state, void *out,
                                   int N, int H, int dk, int dv, cudaStream_t st) {
    const unsigned grid = (unsigned)N * (unsigned)H;
#define KDA_DECODE_CASE(DK_, DV_)                                                              \
    if (dk == DK_ && dv == DV_) {                                                              \
        decode_kernel<T, DK_, DV_><<<grid, 256, 0, st>>>((const T *)q, (const T *)k,           \
                                                         (const T *)v, (const T *)z, A, beta, \
                                                         state, (T *)out, H);                  \
        return cudaGetLastError();                                                             \
    }
    KDA_DECODE_CASE(32, 32) KDA_DECODE_CASE(32, 64) KDA_DECODE_CASE(32, 128)
    KDA_DECODE_CASE(64, 32) KDA_DECODE_CASE(64, 64) KDA_DECODE_CASE(64, 128)
    KDA_DECODE_CASE(128, 32) KDA_DECODE_CASE(128, 64) KDA_DECODE_CASE(128, 128)
#undef KDA_DECODE_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *z,
                          const float *A, const float *beta, float *state, void *out, int N,
                          int H, int dk, int dv, bool bf16, cudaStream_t st) {
    if ((int64_t)N * H == 0) return cudaSuccess;
    return bf16 ? decode_dispatch<__nv_bfloat16>(q, k, v, z, A, beta, state, out, N, H, dk, dv, st)
                : decode_dispatch<float>(q, k, v, z, A, beta, state, out, N, H, dk, dv, st);
}

template <typename T>
static cudaError_t serial_dispatch(const void *q, const void *k, const void *v, const void *z,
                                   const float *A, const float *beta, const int32_t *cu,
                                   int num_seqs, int64_t total, int H, int dk, int dv,
                                   const float *s0, float *s1, void *out, uint32_t *status,
                                   const float *g, cudaStream_t st) {
    dim3 grid((unsigned)num_seqs * (unsigned)H, (unsigned)(dv / 32));
#define KDA_SERIAL_CASE(DK_)                                                                   \
    if (dk == DK_) {                                                                           \
        prefill_serial_kernel<T, DK_><<<grid, 128, 0, st>>>(                                   \
            (const T *)q, (const T *)k, (const T *)v, (const T *)z, A, beta, cu, total, H, dv, \
            s0, s1, (T *)out, status, g);                                                      \
        return cudaGetLastError();                                                             \
    }
    KDA_SERIAL_CASE(32) KDA_SERIAL_CASE(64) KDA_SERIAL_CASE(128)
#undef KDA_SERIAL_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_serial(const void *q, const void *k, const void *v, const void *z,
                                  const float *A, const float *beta, const int32_t *cu,
                                  int num_seqs, int64_t total, int H, int dk, int dv, bool bf16,
                                  const float *s0, float *s1, void *out, uint32_t *status,
                                  cudaStream_t st, const float *g) {
    if ((int64_t)num_seqs * H == 0) return cudaSuccess;
    return bf16 ? serial_dispatch<__nv_bfloat16>(q, k, v, z, A, beta, cu, num_seqs, total, H, dk,
                                                 dv, s0, s1, out, status, g, st)
                : serial_dispatch<float>(q, k, v, z, A, beta, cu, num_seqs, total, H, dk, dv, s0,
                                         s1, out, status, g, st);
}

cudaError_t launch_schedule(const int32_t *cu, int num_seqs, int32_t *order, uint32_t *counter,
                            uint32_t *status, cudaStream_t st) {
    schedule_kernel<<<1, 1024, 0, st>>>(cu, num_seqs, order, counter, status);
    return cudaGetLastError();
}

}  // namespace kda
