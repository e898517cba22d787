// kda_decode_pool.cu -- decode over a pool of recurrent states: several new
// tokens per sequence in one launch, each sequence's state found through a
// slot id.
//
// KDA ("Kimi K3 internals analysis", molayo1419.me, section "Sequence
// mixing"): per token, with the channel-wise decay alpha = exp(g),
// g = -5 sigmoid(exp(A) z),
//   S' = Diag(alpha) S;  u = beta (v - S'^T k);  S = S' + k u^T;  o = S^T q,
// and o = S'^T q + u (k . q) lets one pass over S' give both column
// reductions.  The state is the fixed-size memory that replaces a KV cache; a
// serving engine keeps one per live sequence in a pool and steps a batch of
// them.  Here the dk x dv float32 state is read once, kept in registers for
// all n tokens of the call and written back once, so the state traffic per
// token drops by the factor n.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"

namespace kda {

// One CTA per (sequence, head, block of DVB value channels), 256 threads: the
// recurrence is separable over the value channels (columns of S), so a state
// splits exactly into column blocks.  Thread (r0, col4) holds rows
// r0 + p * ROWS_PER_PASS of its four columns in registers for the whole call.
// The tokens' inputs are staged in shared memory TG at a time (the gate and
// k . q computed there, off the per-token path), so a token costs two block
// barriers and no global-memory latency.
template <typename T, int DK, int DV, int DVB>
__global__ void __launch_bounds__(256) decode_tokens_kernel(
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ z, const float *__restrict__ A, const float *__restrict__ beta,
    float *__restrict__ pool, int pool_size, const int32_t *__restrict__ slots,
    T *__restrict__ out, int n_tok, int H, uint32_t *status) {
    constexpr int F = DVB / 4;            // float4 per state row of this block
    constexpr int ROWS_PER_PASS = 256 / F;
    constexpr int PASSES = DK / ROWS_PER_PASS;
    constexpr int TG = 8;                 // tokens staged at a time
    static_assert(DK % ROWS_PER_PASS == 0 && DV % DVB == 0, "decode tiling");

    __shared__ float s_alpha[TG][DK], s_k[TG][DK], s_q[TG][DK], s_v[TG][DVB];
    __shared__ float s_beta[TG], s_kq[TG];
    __shared__ float s_red[2][ROWS_PER_PASS][DVB + 1];
    __shared__ float s_u[DVB];

    const int nh = blockIdx.x;            // sequence * H + head
    const int n = nh / H, h = nh % H;
    const int j0 = blockIdx.y * DVB;      // first value channel of this block
    const int tid = threadIdx.x;
    int slot = slots ? slots[n] : n;
    if (slot >= pool_size) {              // bad id: reported, row treated as padding
        if (tid == 0 && blockIdx.y == 0) report_status(status, KDA_ERR_INVALID_ARG);
        slot = -1;
    }
    if (slot < 0) {                       // padding row: zero outputs, no state access
        for (int i = tid; i < n_tok * DVB; i += blockDim.x) {
            const int t = i / DVB, j = i % DVB;
            out[(((int64_t)n * n_tok + t) * H + h) * DV + j0 + j] = from_f32<T>(0.f);
        }
        return;
    }

    const int col4 = tid % F;
    const int r0 = tid / F;
    constexpr int RS = DV / 4;            // float4 per full state row
    float4 *S4 = reinterpret_cast<float4 *>(pool + ((int64_t)slot * H + h) * DK * DV + j0);
    float4 s[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) s[p] = S4[(int64_t)(r0 + p * ROWS_PER_PASS) * RS + col4];

    for (int t0 = 0; t0 < n_tok; t0 += TG) {
        const int tn = (n_tok - t0) < TG ? (n_tok - t0) : TG;
        // stage tokens t0 .. t0 + tn - 1
        for (int i = tid; i < tn * DK; i += blockDim.x) {
            const int t = i / DK, c = i % DK;
            const int64_t rk = (((int64_t)n * n_tok + t0 + t) * H + h) * DK + c;
            s_alpha[t][c] = expf(gate_log_decay(expf(A[h * DK + c]), to_f32(z[rk])));
            s_k[t][c] = to_f32(k[rk]);
            s_q[t][c] = to_f32(q[rk]);
        }
        for (int i = tid; i < tn * DVB; i += blockDim.x) {
            const int t = i / DVB, j = i % DVB;
            s_v[t][j] = to_f32(v[(((int64_t)n * n_tok + t0 + t) * H + h) * DV + j0 + j]);
        }
        if (tid < tn) s_beta[tid] = beta[((int64_t)n * n_tok + t0 + tid) * H + h];
        __syncthreads();
        {   // k . q of every staged token: one warp per token
            const int w = tid >> 5, l = tid & 31;
            for (int t = w; t < tn; t += 8) {
                float acc = 0.f;
                for (int c = l; c < DK; c += 32) acc += s_k[t][c] * s_q[t][c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (l == 0) s_kq[t] = acc;
            }
        }
        for (int t = 0; t < tn; ++t) {
            // S' = Diag(alpha) S ; partial column sums of S'^T k and S'^T q
            float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
            for (int p = 0; p < PASSES; ++p) {
                const int c = r0 + p * ROWS_PER_PASS;
                const float a = s_alpha[t][c], kc = s_k[t][c], qc = s_q[t][c];
                s[p].x *= a; s[p].y *= a; s[p].z *= a; s[p].w *= a;
                pk.x += s[p].x * kc; pk.y += s[p].y * kc; pk.z += s[p].z * kc; pk.w += s[p].w * kc;
                pq.x += s[p].x * qc; pq.y += s[p].y * qc; pq.z += s[p].z * qc; pq.w += s[p].w * qc;
            }
            s_red[0][r0][4 * col4 + 0] = pk.x; s_red[0][r0][4 * col4 + 1] = pk.y;
            s_red[0][r0][4 * col4 + 2] = pk.z; s_red[0][r0][4 * col4 + 3] = pk.w;
            s_red[1][r0][4 * col4 + 0] = pq.x; s_red[1][r0][4 * col4 + 1] = pq.y;
            s_red[1][r0][4 * col4 + 2] = pq.z; s_red[1][r0][4 * col4 + 3] = pq.w;
            __syncthreads();   // (also orders s_kq, written above, before its use)
            if (tid < DVB) {
                float kv = 0.f, sq = 0.f;
#pragma unroll 8
                for (int r = 0; r < ROWS_PER_PASS; ++r) { kv += s_red[0][r][tid]; sq += s_red[1][r][tid]; }
                const float u = s_beta[t] * (s_v[t][tid] - kv);
                s_u[tid] = u;
                out[(((int64_t)n * n_tok + t0 + t) * H + h) * DV + j0 + tid] = from_f32<T>(sq + u * s_kq[t]);
            }
            __syncthreads();
            // S = S' + k u^T
            const float u0 = s_u[4 * col4], u1 = s_u[4 * col4 + 1], u2 = s_u[4 * col4 + 2],
                        u3 = s_u[4 * col4 + 3];
#pragma unroll
            for (int p = 0; p < PASSES; ++p) {
                const float kc = s_k[t][r0 + p * ROWS_PER_PASS];
                s[p].x += kc * u0; s[p].y += kc * u1; s[p].z += kc * u2; s[p].w += kc * u3;
            }
        }
        __syncthreads();   // the staged tokens are consumed before the next group overwrites them
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) S4[(int64_t)(r0 + p * ROWS_PER_PASS) * RS + col4] = s[p];
}

template <typename T>
static cudaError_t tokens_dispatch(const void *q, const void *k, const void *v, const void *z,
                                   const float *A, const float *beta, float *pool, int pool_size,
                                   const int32_t *slots, void *out, int N, int n_tok, int H,
                                   int dk, int dv, uint32_t *status, cudaStream_t st) {
#define KDA_TOKENS_CASE(DK_, DV_)                                                               \
    if (dk == DK_ && dv == DV_) {                                                               \
        constexpr int DVB = DV_ < 64 ? DV_ : 64;                                                \
        const dim3 grid((unsigned)N * (unsigned)H, DV_ / DVB);                                  \
        decode_tokens_kernel<T, DK_, DV_, DVB><<<grid, 256, 0, st>>>(                           \
            (const T *)q, (const T *)k, (const T *)v, (const T *)z, A, beta, pool, pool_size,   \
            slots, (T *)out, n_tok, H, status);                                                 \
        return cudaGetLastError();                                                              \
    }
    KDA_TOKENS_CASE(32, 32) KDA_TOKENS_CASE(32, 64) KDA_TOKENS_CASE(32, 128)
    KDA_TOKENS_CASE(64, 32) KDA_TOKENS_CASE(64, 64) KDA_TOKENS_CASE(64, 128)
    KDA_TOKENS_CASE(128, 32) KDA_TOKENS_CASE(128, 64) KDA_TOKENS_CASE(128, 128)
#undef KDA_TOKENS_CASE
    return cudaErrorInvalidValue;
}

// Prefill -> decode handoff: N contiguous states [N, H, dk, dv] to or from
// their pool slots.  One CTA per (row, head), float4 copies; a negative slot
// skips the row (on a gather its states are zeroed), a slot >= pool_size is
// reported in *status and treated the same way.
__global__ void __launch_bounds__(256) state_slots_kernel(float *__restrict__ pool, int pool_size,
                                                          const int32_t *__restrict__ slots,
                                                          float *__restrict__ states, int H,
                                                          int64_t per_head, bool to_pool,
                                                          uint32_t *status) {
    const int i = blockIdx.x, h = blockIdx.y;
    int slot = slots[i];
    if (slot >= pool_size) {
        if (threadIdx.x == 0 && h == 0) report_status(status, KDA_ERR_INVALID_ARG);
        slot = -1;
    }
    float4 *row = reinterpret_cast<float4 *>(states + ((int64_t)i * H + h) * per_head);
    const int64_t n4 = per_head / 4;
    if (slot < 0) {
        if (!to_pool)
            for (int64_t e = threadIdx.x; e < n4; e += blockDim.x) row[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    float4 *cell = reinterpret_cast<float4 *>(pool + ((int64_t)slot * H + h) * per_head);
    if (to_pool)
        for (int64_t e = threadIdx.x; e < n4; e += blockDim.x) cell[e] = row[e];
    else
        for (int64_t e = threadIdx.x; e < n4; e += blockDim.x) row[e] = cell[e];
}

cudaError_t launch_state_slots(float *pool, int pool_size, const int32_t *slots, float *states,
                               int N, int H, int dk, int dv, bool to_pool, uint32_t *status,
                               cudaStream_t st) {
    if ((int64_t)N * H == 0) return cudaSuccess;
    state_slots_kernel<<<dim3((unsigned)N, (unsigned)H), 256, 0, st>>>(
        pool, pool_size, slots, states, H, (int64_t)dk * dv, to_pool, status);
    return cudaGetLastError();
}

cudaError_t launch_decode_tokens(const void *q, const void *k, const void *v, const void *z,
                                 const float *A, const float *beta, float *pool, int pool_size,
                                 const int32_t *slots, void *out, int N, int n_tok, int H, int dk,
                                 int dv, bool bf16, uint32_t *status, cudaStream_t st) {
    if ((int64_t)N * H == 0 || n_tok == 0) return cudaSuccess;
    return bf16 ? tokens_dispatch<__nv_bfloat16>(q, k, v, z, A, beta, pool, pool_size, slots, out,
                                                 N, n_tok, H, dk, dv, status, st)
                : tokens_dispatch<float>(q, k, v, z, A, beta, pool, pool_size, slots, out, N,
                                         n_tok, H, dk, dv, status, st);
}

}  // namespace kda
