// kda_prefill_tc.cu -- chunkwise KDA prefill on the sm_103a tensor cores
// (tcgen05.mma with TMEM accumulators, TMA tile loads, mbarriers).
//
// Method ("Kimi K3 internals analysis", molayo1419.me, section "Sequence
// mixing"): the gate g = -5 sigmoid(exp(A) z) bounds every per-token log-decay
// to (-5, 0), so the cumulative log-decay of any 16-token tile stays inside
// (-80, 0) and its exponential and reciprocal both fit the float32/bf16
// exponent range.  That is what lets the diagonal 16-token tiles of the
// intra-chunk products use the same dense tensor-core path as the
// off-diagonal ones.
//
// Algebra, per (sequence, head) and 64-token chunk with start state S0 and
// inclusive chunk-local cumulative log-decay G_t (per key channel c):
//   L_ts = beta_t sum_c k_tc k_sc e^{G_tc - G_sc}    (s < t)
//   P_ts =        sum_c q_tc k_sc e^{G_tc - G_sc}    (s <= t)
//   T    = (I + L)^{-1} Diag(beta)
//   U    = T (V - K~ S0),            K~ = k * e^{G}
//   O    = Q~ S0 + P U,              Q~ = q * e^{G}
//   S1   = Diag(e^{G_end}) S0 + (k * e^{G_end - G})^T U
// which is the token recurrence S' = Diag(alpha) S, S = S' + beta k (v - S'^T k)^T,
// o = S^T q unrolled over the chunk.
//
// Tile factorisation of e^{G_t - G_s} (the 16-token bound at work): with
// R_a = G at the end of tile a-1 (R_0 = 0), a row t of tile a uses the left
// factor e^{G_t - R_a} in (e^-80, 1] and a column s <= end of tile a uses the
// right factor e^{R_a - G_s}, which is in [1, e^80) inside tile a and <= 1 for
// earlier tiles.  Both factors are finite in float32 and bf16, so one dense
// MMA per row tile covers its diagonal and off-diagonal blocks.
//
// One CTA (256 threads, 8 warps) per SM, persistent over (sequence, head)
// chains taken longest-first from a device work counter.  Per chunk:
//   A  SIMT: gate, cumulative decay, operand tiles (bf16, 128B-swizzled)
//      MMA: Gram/P tiles [Q^;K^] x B_a^T (4 tiles) and S^T x [K~;Q~]^T
//   B  SIMT: mask P and L from TMEM, RHS^T = V^T - (K~S0)^T, blocked
//      forward substitution for T
//      MMA: U^T = RHS^T T^T
//   C  SIMT: U^T -> bf16 operand
//      MMA: O^T += U^T P^T ; dS^T = U^T Kend^T
//   D  SIMT: S^T = S^T Diag(e^{G_end}) + dS^T (float32 master in registers),
//      bf16 copy of S^T for the next chunk, O stored to global memory
// The state is kept transposed (rows = value channels) so every accumulator
// has M = 128 rows, one per TMEM lane.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace tc {

constexpr int C = 64;      // chunk length (tokens)
constexpr int D = 128;     // dk = dv
constexpr int NT = 512;    // threads per CTA (16 warps)

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kGMin2 = -5.0f * 1.4426950408889634f;   // g_min in log2 units

// ---- shared memory map (bytes from a 1024-aligned base) ---------------------
// q and k arrive by TMA interleaved so that together they form the 128-row
// K-major operand [q; k] (K-block 0 = q ch 0-63, k ch 0-63; K-block 1 = the
// rest); the left-factor operand [Q^; K^] of the Gram/P MMA is built in place.
constexpr uint32_t OFF_QK = 0;         // [Q^; K^] 128 x 128 bf16 (32 KB)
constexpr uint32_t OFF_V = 32768;      // v tile: 64 rows x 128 ch, two boxes
constexpr uint32_t OFF_Z = 49152;      // z tile
constexpr uint32_t OFF_VT = 65536;     // V^T [j][s] 128 x 64 bf16 (masked rows zeroed)
constexpr uint32_t OFF_OST = 81920;    // output tile: two 64-channel boxes in the TMA 128B-swizzle layout
constexpr uint32_t OFF_PB = 81920;     // P [t][s]: 64 x 64 bf16 (phases B-C, before the output tile)
constexpr uint32_t OFF_GB = 98304;     // right factors: 160 rows (tile a at row 16a(a+1)/2) x 128
constexpr uint32_t GB_KBLK = 160 * 128;
constexpr uint32_t OFF_B1 = 139264;    // [K~; Q~] 128 x 128 bf16 (B of the state MMA)
// reused once the Gram/P and state MMAs have completed:
constexpr int LSTR = 68;               // float32 row stride of L and Y (16-byte multiple)
constexpr uint32_t OFF_L = 98304;      // L [64][LSTR] float32
constexpr uint32_t OFF_Y = OFF_L + 64 * LSTR * 4;      // Y = (I + L)^{-1}
constexpr uint32_t OFF_W = OFF_Y + 64 * LSTR * 4;      // W_am = Y_aa L_am, 6 blocks of 16 x 16
constexpr uint32_t OFF_TB = 139264;    // T [t][s]: 64 x 64 bf16 (after the state MMA)
constexpr uint32_t OFF_RU = 155648;    // RHS^T, then U^T: 128 x 64 bf16 (after the state MMA)
constexpr uint32_t OFF_KE = 172032;    // Kend^T [c][s] 128 x 64 bf16
constexpr uint32_t OFF_ST = 188416;    // S^T [j][c] 128 x 128 bf16 (A of the state MMA)
constexpr uint32_t OFF_MISC = 221184;
constexpr uint32_t OFF_BETA = OFF_MISC;              // 64 float
constexpr uint32_t OFF_EAN = OFF_BETA + 256;         // 128 float: -exp(A) log2(e)
constexpr uint32_t OFF_R = OFF_EAN + 512;            // [4][128]: R1, R2, R3, G_end (log2 units)
constexpr uint32_t OFF_E = OFF_R + 2048;             // [4][128]: 2^(R_{a+1} - R_a)
constexpr uint32_t OFF_RHO = OFF_E + 2048;           // [4][128]: 2^(R_a)
constexpr uint32_t OFF_TAIL = OFF_RHO + 2048;        // [4][128]: prod_{a' > a} E_a'
constexpr uint32_t OFF_GAMMA = OFF_TAIL + 2048;      // 128 float: 2^(G_end)
constexpr uint32_t OFF_BAR = OFF_GAMMA + 512;        // mbarriers
constexpr uint32_t OFF_SLOT = OFF_BAR + 64;          // TMEM base, work item, abort flag
constexpr uint32_t SMEM_USED = OFF_SLOT + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;    // slack to align the base to 1024 B
static_assert(OFF_GB + 2 * GB_KBLK <= OFF_B1, "right-factor tiles overlap");
static_assert(OFF_W + 6 * 256 * 4 <= OFF_TB, "solve scratch overlaps");
static_assert(OFF_RU + 16384 <= OFF_KE, "RU overlaps");
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// ---- tensor memory map (columns; 128 lanes each) ----------------------------
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t TM_G = 0;           // Gram/P tiles, N = 160 (tile a at column 16a(a+1)/2)
constexpr uint32_t TM_D1 = 192;        // [(K~S0)^T | (Q~S0 + P U)^T]  128 x 128
constexpr uint32_t TM_D2 = 320;        // U^T 128 x 64
constexpr uint32_t TM_D3 = 384;        // dS^T 128 x 128

constexpr long long kWaitBudget = 2000000000LL;   // cycles (about one second)

// first row (and TMEM column) of right-factor tile a: 0, 16, 48, 96
__device__ __forceinline__ int tile_off(int a) { return 8 * a * (a + 1); }

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

// One level of the blocked inverse: Y_ab = -sum_{m=b}^{a-1} W_am Y_mb for the
// blocks with a - b = dist, where W_am = Y_aa L_am.  One output per task.
__device__ __forceinline__ void solve_level(int dist, float *Ym, const float *Wm, int tid) {
    const int ntask = (4 - dist) * 256;
    for (int task = tid; task < ntask; task += NT) {
        const int b = task >> 8, a = b + dist, i = (task >> 4) & 15, j = task & 15;
        float acc0 = 0.f, acc1 = 0.f;
        for (int m = b; m < a; ++m) {
            const float *w = Wm + ((a * (a - 1)) / 2 + m) * 256 + i * 16;
            float wr[16];
            ld8(w, wr); ld8(w + 8, wr + 8);
            const float *y = Ym + (16 * m) * LSTR + 16 * b + j;
#pragma unroll
            for (int n = 0; n < 16; n += 2) {
                acc0 += wr[n] * y[n * LSTR];
                acc1 += wr[n + 1] * y[(n + 1) * LSTR];
            }
        }
        Ym[(16 * a + i) * LSTR + 16 * b + j] = -(acc0 + acc1);
    }
}

struct Params {
    const float *A;            // [H, 128]
    const float *beta;         // [T, H]
    const int32_t *cu_seqlens; // [N + 1]
    const float *initial_state;
    float *final_state;
    __nv_bfloat16 *out;        // [T, H, 128]
    const int32_t *order;      // [N] longest first
    uint32_t *counter;
    uint32_t *status;
    int64_t total_tokens;
    int num_seqs;
    int H;
};

__device__ __forceinline__ void tma_qk(uint8_t *sm, const CUtensorMap *tq, const CUtensorMap *tk,
                                       int hx, int y, uint64_t *bar) {
    ptx::mbar_arrive_expect_tx(bar, 32768);
    ptx::tma_load_2d(sm + OFF_QK, tq, hx, y, bar);
    ptx::tma_load_2d(sm + OFF_QK + 8192, tk, hx, y, bar);
    ptx::tma_load_2d(sm + OFF_QK + 16384, tq, hx + 64, y, bar);
    ptx::tma_load_2d(sm + OFF_QK + 24576, tk, hx + 64, y, bar);
}
__device__ __forceinline__ void tma_2box(uint8_t *dst, const CUtensorMap *tm, int hx, int y,
                                         uint64_t *bar) {
    ptx::mbar_arrive_expect_tx(bar, 16384);
    ptx::tma_load_2d(dst, tm, hx, y, bar);
    ptx::tma_load_2d(dst + 8192, tm, hx + 64, y, bar);
}

__global__ void __launch_bounds__(NT, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_z,
                  const __grid_constant__ CUtensorMap tm_o, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(sm);
    float *s_beta = reinterpret_cast<float *>(sm + OFF_BETA);
    float *s_eAn = reinterpret_cast<float *>(sm + OFF_EAN);
    float *s_R = reinterpret_cast<float *>(sm + OFF_R);
    float *s_E = reinterpret_cast<float *>(sm + OFF_E);
    float *s_rho = reinterpret_cast<float *>(sm + OFF_RHO);
    float *s_tail = reinterpret_cast<float *>(sm + OFF_TAIL);
    float *s_gamma = reinterpret_cast<float *>(sm + OFF_GAMMA);
    uint64_t *bar_qk = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_z = bar_qk + 1;
    uint64_t *bar_v = bar_qk + 2;
    uint64_t *bar_g = bar_qk + 3;      // Gram/P MMA done
    uint64_t *bar_s = bar_qk + 4;      // state MMA done
    uint64_t *bar_m = bar_qk + 5;      // U MMA, then output/state MMAs done
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + OFF_SLOT);
    volatile int *s_work = reinterpret_cast<volatile int *>(sm + OFF_SLOT + 4);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + OFF_SLOT + 8);
    float *Lm = reinterpret_cast<float *>(sm + OFF_L);
    float *Ym = reinterpret_cast<float *>(sm + OFF_Y);
    float *Wm = reinterpret_cast<float *>(sm + OFF_W);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // phases B-D: value channel j == TMEM lane, 16/32-column group cg
    const int qw = warp & 3;           // TMEM lane quarter this warp may access
    const int cg = warp >> 2;          // 0..3
    const int ch = 32 * qw + lane;
    // phase A: 8 key channels per warp, rows lane and lane + 32 per lane (rows
    // 8 apart land on distinct swizzled bank groups)
    const int cw = 8 * warp;
    const int kb = warp >> 3;          // K-block (64 channels) of these channels
    const int chk = warp & 7;          // their 16-byte chunk inside the 128-byte row
    const int H = p.H;
    const int64_t rowstride = (int64_t)H * D;

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) ptx::mbar_init(bar_qk + i, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_z);
        ptx::prefetch_tensormap(&tm_o);
        *s_abort = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(s_tmem, TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * qw) << 16);

    // issue / completion counters of the barriers (uniform across threads);
    // a barrier's next expected phase parity is (done & 1)
    uint32_t qk_issued = 0, qk_done = 0, z_issued = 0, z_done = 0, v_issued = 0, v_done = 0;
    uint32_t g_issued = 0, g_done = 0, s_issued = 0, s_done = 0, m_issued = 0, m_done = 0;
    const int n_work = p.num_seqs * H;

    for (;;) {
        if (tid == 0) *s_work = (int)atomicAdd(p.counter, 1u);
        __syncthreads();
        const int w = *s_work;
        if (w >= n_work || *s_abort) break;
        const int seq = p.order[w / H];
        const int h = w % H;
        int64_t bos = p.cu_seqlens[seq], eos = p.cu_seqlens[seq + 1];
        if (bos < 0 || eos < bos || eos > p.total_tokens) {
            if (tid == 0) report_status(p.status, kDevBadSeqlens);
            bos = eos = 0;
        }
        const int nchunks = (int)((eos - bos + C - 1) / C);
        const int64_t sidx = ((int64_t)seq * H + h) * D * D;
        const int hx = h * D;   // column of this head in the [T, H*D] view

        if (nchunks > 0 && tid == 0) {
            tma_qk(sm, &tm_q, &tm_k, hx, (int)bos, bar_qk);
            tma_2box(sm + OFF_Z, &tm_z, hx, (int)bos, bar_z);
            tma_2box(sm + OFF_V, &tm_v, hx, (int)bos, bar_v);
        }
        if (nchunks > 0) { ++qk_issued; ++z_issued; ++v_issued; }

        // ---- start state: float32 master S^T[j][c] lives in TMEM (the dS accumulator),
        // its bf16 copy in smem; this thread holds c in [32 cg, 32 cg + 32) of row j
        {
            float Sm[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 32 * cg + i;
                Sm[i] = p.initial_state ? p.initial_state[sidx + (int64_t)c * D + ch] : 0.f;
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                st_chunk(sm + OFF_ST + (cg >> 1) * 16384, swz(ch, 4 * (cg & 1) + q4), &Sm[8 * q4]);
            ptx::tmem_st32(lane_base + TM_D3 + 32 * cg, Sm);
            ptx::tmem_st_wait();
        }
        if (tid < D) s_eAn[tid] = -expf(p.A[h * D + tid]) * kLog2e;
        float beta_next = 0.f;
        if (tid < C && nchunks > 0) beta_next = (bos + tid < eos) ? p.beta[(bos + tid) * H + h] : 0.f;
        __syncthreads();   // s_eAn visible

        for (int cidx = 0; cidx < nchunks; ++cidx) {
            const int64_t row0 = bos + (int64_t)cidx * C;
            const int nvalid = (int)((eos - row0) < C ? (eos - row0) : C);
            const bool has_next = (cidx + 1 < nchunks);
            const int64_t next_row = row0 + C;

            // =============================== phase A: gate, cumulative decay, operands
            if (tid < C) s_beta[tid] = beta_next;
            if (ptx::mbar_wait(bar_z, z_done & 1, kWaitBudget)) ++z_done; else *s_abort = 1;
            float G0[8], G1[8];   // log2-domain cumulative log-decay of rows lane, lane + 32
            {
                float z0[8], z1[8], eAn[8];
                const uint8_t *zt = sm + OFF_Z + kb * 8192;
                ld_chunk(zt, swz(lane, chk), z0);
                ld_chunk(zt, swz(lane + 32, chk), z1);
                ld8(s_eAn + cw, eAn);
                const bool ok0 = lane < nvalid, ok1 = lane + 32 < nvalid;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    // g = g_min sigmoid(exp(A) z) = g_min / (1 + 2^(-exp(A) z log2 e))
                    float a0 = ok0 ? kGMin2 * rcp(1.f + ex2(eAn[i] * z0[i])) : 0.f;
                    float a1 = ok1 ? kGMin2 * rcp(1.f + ex2(eAn[i] * z1[i])) : 0.f;
                    // inclusive scans over the lanes: rows 0..31, then rows 32..63
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float t0 = __shfl_up_sync(0xffffffffu, a0, off);
                        const float t1 = __shfl_up_sync(0xffffffffu, a1, off);
                        if (lane >= off) { a0 += t0; a1 += t1; }
                    }
                    G0[i] = a0;
                    G1[i] = a1 + __shfl_sync(0xffffffffu, a0, 31);
                }
            }
            // tile references: rows 15, 31, 47, 63 live in lanes 15 (G0), 31 (G0), 15 (G1), 31 (G1)
            if ((lane & 15) == 15) {
                float *d0 = s_R + (lane >> 4) * 128 + cw;          // R1 or R2
                float *d1 = s_R + (2 + (lane >> 4)) * 128 + cw;    // R3 or G_end
                *reinterpret_cast<float4 *>(d0) = make_float4(G0[0], G0[1], G0[2], G0[3]);
                *reinterpret_cast<float4 *>(d0 + 4) = make_float4(G0[4], G0[5], G0[6], G0[7]);
                *reinterpret_cast<float4 *>(d1) = make_float4(G1[0], G1[1], G1[2], G1[3]);
                *reinterpret_cast<float4 *>(d1 + 4) = make_float4(G1[4], G1[5], G1[6], G1[7]);
            }
            __syncwarp();
            if (lane < 8) {
                const int c = cw + lane;
                const float R1 = s_R[c], R2 = s_R[128 + c], R3 = s_R[256 + c], Ge = s_R[384 + c];
                const float E0 = ex2(R1), E1 = ex2(R2 - R1), E2 = ex2(R3 - R2), E3 = ex2(Ge - R3);
                s_E[c] = E0; s_E[128 + c] = E1; s_E[256 + c] = E2; s_E[384 + c] = E3;
                s_rho[c] = 1.f; s_rho[128 + c] = ex2(R1); s_rho[256 + c] = ex2(R2);
                s_rho[384 + c] = ex2(R3);
                s_tail[c] = E1 * E2 * E3; s_tail[128 + c] = E2 * E3; s_tail[256 + c] = E3;
                s_tail[384 + c] = 1.f;
                s_gamma[c] = ex2(Ge);
            }
            if (ptx::mbar_wait(bar_qk, qk_done & 1, kWaitBudget)) ++qk_done; else *s_abort = 1;
            __syncwarp();
            {
                const uint32_t kbo = kb * 16384;
                const uint32_t gbk = OFF_GB + kb * GB_KBLK;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = lane + 32 * rr;
                    const int ta = r >> 4;                       // 16-token tile of this row
                    const bool ok = r < nvalid;
                    float Rb[8], rho[8], E[8], tl[8];
                    if (ta == 0) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) Rb[i] = 0.f;
                    } else {
                        ld8(s_R + (ta - 1) * 128 + cw, Rb);
                    }
                    ld8(s_rho + ta * 128 + cw, rho);
                    ld8(s_E + ta * 128 + cw, E);
                    ld8(s_tail + ta * 128 + cw, tl);
                    float qv[8], kv[8];
                    ld_chunk(sm + OFF_QK + kbo, swz(r, chk), qv);
                    ld_chunk(sm + OFF_QK + kbo, swz(64 + r, chk), kv);
                    float qe[8], ke[8], f[8], tk[8], tq[8], kend[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float x = (rr ? G1[i] : G0[i]) - Rb[i];   // in (-115.4, 0]
                        const float el = ok ? ex2(x) : 0.f;              // left factor
                        const float dd = ok ? ex2(-x) : 0.f;             // right factor
                        qe[i] = qv[i] * el;
                        ke[i] = kv[i] * el;
                        f[i] = kv[i] * dd;
                        tk[i] = ke[i] * rho[i];
                        tq[i] = qe[i] * rho[i];
                        kend[i] = (f[i] * E[i]) * tl[i];                 // k 2^(G_end - G_r)
                    }
                    st_chunk(sm + OFF_QK + kbo, swz(r, chk), qe);        // in place: [Q^; K^]
                    st_chunk(sm + OFF_QK + kbo, swz(64 + r, chk), ke);
                    st_chunk(sm + OFF_B1 + kbo, swz(r, chk), tk);
                    st_chunk(sm + OFF_B1 + kbo, swz(64 + r, chk), tq);
                    // Kend^T [c][s]
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int c = cw + i;
                        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_KE + swz(c, r >> 3) + (r & 7) * 2) =
                            __float2bfloat16_rn(kend[i]);
                    }
                    // right factors for the Gram/P tiles a2 >= ta: k 2^(R_a2 - G_r)
                    for (int a2 = ta; a2 < 4; ++a2) {
                        st_chunk(sm + gbk, swz(tile_off(a2) + r, chk), f);
                        if (a2 < 3) {   // next tile: multiply by E_a2 = 2^(R_{a2+1} - R_a2)
                            float en[8];
                            if (a2 == ta) {
#pragma unroll
                                for (int i = 0; i < 8; ++i) en[i] = E[i];
                            } else {
                                ld8(s_E + a2 * 128 + cw, en);
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) f[i] *= en[i];
                        }
                    }
                }
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                ptx::bulk_wait_read();   // the previous output tile has left OST (P goes there next)
                // every thread has read its z rows: prefetch the next chunk's
                if (has_next) tma_2box(sm + OFF_Z, &tm_z, hx, (int)next_row, bar_z);
                // Gram/P: D[r][tile_off(a) + s] = [Q^;K^][r] . B[tile_off(a) + s], all four tiles
                mma_k<8>(tmem + TM_G, sbase + OFF_QK, 16384u, sbase + OFF_GB, GB_KBLK,
                         ptx::idesc_bf16_f32(128, 160), false);
                ptx::mma_commit(bar_g);
                // state product: D1[j][s|t] = S^T[j] . [K~;Q~][s|t]
                mma_k<8>(tmem + TM_D1, sbase + OFF_ST, 16384u, sbase + OFF_B1, 16384u,
                         ptx::idesc_bf16_f32(128, 128), false);
                ptx::mma_commit(bar_s);
            }
            ++g_issued; ++s_issued;
            if (has_next) ++z_issued;

            // =============================== phase B: P, L, V^T, T, RHS
            if (ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done; else *s_abort = 1;
            if (tid == 0 && has_next) tma_qk(sm, &tm_q, &tm_k, hx, (int)next_row, bar_qk);
            if (has_next) ++qk_issued;
            if (ptx::mbar_wait(bar_v, v_done & 1, kWaitBudget)) ++v_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            {
                // P (TMEM rows 0..63) and L (rows 64..127): 16 columns per thread
                const int r = 32 * qw + lane;
                const int t = r & 63;
                const bool isL = r >= 64;
                const int m = qw & 1;                 // this warp sees tiles 2m, 2m+1
                const int a = 2 * m + (lane >> 4);
                const int colbase = 16 * cg;
                float X[16], Y[16];
                const bool loadX = cg <= 2 * m, loadY = cg <= 2 * m + 1;   // warp-uniform
                if (loadX) ptx::tmem_ld16(lane_base + TM_G + tile_off(2 * m) + colbase, X);
                if (loadY) ptx::tmem_ld16(lane_base + TM_G + tile_off(2 * m + 1) + colbase, Y);
                ptx::tmem_ld_wait();
                const bool have = cg <= a;
                const float bt = s_beta[t];
                float vals[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int s = colbase + i;
                    const float d = have ? ((lane < 16) ? X[i] : Y[i]) : 0.f;
                    vals[i] = isL ? ((s < t) ? bt * d : 0.f) : ((s <= t) ? d : 0.f);
                }
                if (isL) {
                    float4 *dst = reinterpret_cast<float4 *>(Lm + t * LSTR + colbase);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(vals[4 * i], vals[4 * i + 1], vals[4 * i + 2], vals[4 * i + 3]);
                } else {
                    st_chunk(sm + OFF_PB, swz(t, 2 * cg), &vals[0]);
                    st_chunk(sm + OFF_PB, swz(t, 2 * cg + 1), &vals[8]);
                }
            }
            __syncthreads();
            if (warp < 4) {
                // diagonal 16 x 16 blocks of (I + L)^{-1} by forward substitution, one column per lane
                if (lane < 16) {
                    const int b0 = 16 * warp;
                    float y[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float lr[16];
                        const float *src = Lm + (b0 + i) * LSTR + b0;
                        ld8(src, lr); ld8(src + 8, lr + 8);
                        float a0 = (i == lane) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
                        for (int mm = 0; mm < i; ++mm) {
                            if (mm & 1) a1 -= lr[mm] * y[mm]; else a0 -= lr[mm] * y[mm];
                        }
                        y[i] = a0 + a1;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) Ym[(b0 + i) * LSTR + b0 + lane] = y[i];
                }
            } else {
                // meanwhile: V^T [j][s] (rows past the sequence end zeroed); a warp
                // transposes one 8-channel chunk, lane = rows lane and lane + 32
                for (int cc = warp - 4; cc < 16; cc += 12) {
                    float v0[8], v1[8];
                    const uint8_t *vt = sm + OFF_V + (cc >> 3) * 8192;
                    ld_chunk(vt, swz(lane, cc & 7), v0);
                    ld_chunk(vt, swz(lane + 32, cc & 7), v1);
                    const bool ok0 = lane < nvalid, ok1 = lane + 32 < nvalid;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int j = 8 * cc + i;
                        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_VT + swz(j, lane >> 3) + (lane & 7) * 2) =
                            __float2bfloat16_rn(ok0 ? v0[i] : 0.f);
                        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_VT + swz(j, 4 + (lane >> 3)) + (lane & 7) * 2) =
                            __float2bfloat16_rn(ok1 ? v1[i] : 0.f);
                    }
                }
            }
            __syncthreads();
            if (tid == 0 && has_next) tma_2box(sm + OFF_V, &tm_v, hx, (int)next_row, bar_v);
            if (has_next) ++v_issued;
            // W_am = Y_aa L_am for the six blocks below the diagonal (1 x 4 outputs per task)
            for (int task = tid; task < 6 * 64; task += NT) {
                const int blk = task >> 6, i = (task >> 2) & 15, jj = task & 3;
                const int a = blk < 1 ? 1 : (blk < 3 ? 2 : 3);
                const int m = blk - (a * (a - 1)) / 2;
                float yr[16];
                const float *src = Ym + (16 * a + i) * LSTR + 16 * a;
                ld8(src, yr); ld8(src + 8, yr + 8);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    float lv[4];
                    ld4(Lm + (16 * a + n) * LSTR + 16 * m + 4 * jj, lv);
                    acc[0] += yr[n] * lv[0]; acc[1] += yr[n] * lv[1];
                    acc[2] += yr[n] * lv[2]; acc[3] += yr[n] * lv[3];
                }
                *reinterpret_cast<float4 *>(Wm + blk * 256 + i * 16 + 4 * jj) =
                    make_float4(acc[0], acc[1], acc[2], acc[3]);
            }
            __syncthreads();
            solve_level(1, Ym, Wm, tid);
            __syncthreads();
            solve_level(2, Ym, Wm, tid);
            __syncthreads();
            solve_level(3, Ym, Wm, tid);
            __syncthreads();
            // the state MMA (still reading B1, where T and RHS go) overlapped the solve
            if (ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            {
                // T = Y Diag(beta), lower triangle, bf16; 8 columns per thread
                const int t = tid >> 3, q8 = tid & 7;
                float tv[8], yr[8], bv[8];
                ld8(Ym + t * LSTR + 8 * q8, yr);
                ld8(s_beta + 8 * q8, bv);
#pragma unroll
                for (int i = 0; i < 8; ++i) tv[i] = (8 * q8 + i <= t) ? yr[i] * bv[i] : 0.f;
                st_chunk(sm + OFF_TB, swz(t, q8), tv);
            }
            {
                // RHS^T[j][s] = V^T[j][s] - (K~ S0)^T[j][s], 16 columns per thread
                float KS[16], vt[16];
                ptx::tmem_ld16(lane_base + TM_D1 + 16 * cg, KS);
                ld_chunk(sm + OFF_VT, swz(ch, 2 * cg), vt);
                ld_chunk(sm + OFF_VT, swz(ch, 2 * cg + 1), vt + 8);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) vt[i] -= KS[i];
                st_chunk(sm + OFF_RU, swz(ch, 2 * cg), vt);
                st_chunk(sm + OFF_RU, swz(ch, 2 * cg + 1), vt + 8);
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                // U^T = RHS^T T^T
                mma_k<4>(tmem + TM_D2, sbase + OFF_RU, 0u, sbase + OFF_TB, 0u,
                         ptx::idesc_bf16_f32(128, 64), false);
                ptx::mma_commit(bar_m);
            }
            ++m_issued;
            if (tid < C && has_next)
                beta_next = (next_row + tid < eos) ? p.beta[(next_row + tid) * H + h] : 0.f;

            // =============================== phase C: U^T to smem, output and state MMAs
            if (ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            {
                float U[16], Sx[32], gm[32];
                ptx::tmem_ld16(lane_base + TM_D2 + 16 * cg, U);
                ptx::tmem_ld32(lane_base + TM_D3 + 32 * cg, Sx);
                ld8(s_gamma + 32 * cg, gm); ld8(s_gamma + 32 * cg + 8, gm + 8);
                ld8(s_gamma + 32 * cg + 16, gm + 16); ld8(s_gamma + 32 * cg + 24, gm + 24);
                ptx::tmem_ld_wait();
                st_chunk(sm + OFF_RU, swz(ch, 2 * cg), U);
                st_chunk(sm + OFF_RU, swz(ch, 2 * cg + 1), U + 8);
                // S^T <- S^T Diag(2^G_end); the dS MMA then accumulates onto it
#pragma unroll
                for (int i = 0; i < 32; ++i) Sx[i] *= gm[i];
                ptx::tmem_st32(lane_base + TM_D3 + 32 * cg, Sx);
                ptx::tmem_st_wait();
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                // O^T += U^T P^T  (onto the Q~S0 half of D1)
                mma_k<4>(tmem + TM_D1 + 64, sbase + OFF_RU, 0u, sbase + OFF_PB, 0u,
                         ptx::idesc_bf16_f32(128, 64), true);
                // S^T += U^T Kend
                mma_k<4>(tmem + TM_D3, sbase + OFF_RU, 0u, sbase + OFF_KE, 0u,
                         ptx::idesc_bf16_f32(128, 128), true);
                ptx::mma_commit(bar_m);
            }
            ++m_issued;

            // =============================== phase D: state update, output
            if (ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            {
                float X[32], O[16];
                ptx::tmem_ld32(lane_base + TM_D3 + 32 * cg, X);
                ptx::tmem_ld16(lane_base + TM_D1 + 64 + 16 * cg, O);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    st_chunk(sm + OFF_ST + (cg >> 1) * 16384, swz(ch, 4 * (cg & 1) + q4), &X[8 * q4]);
                // O tile staged in the TMA layout: box j/64, row t, 16-byte chunk XOR t % 8
                const uint32_t obox = OFF_OST + (ch >> 6) * 8192;
                const int jc = (ch & 63) >> 3, jin = (ch & 7) * 2;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = 16 * cg + i;
                    *reinterpret_cast<__nv_bfloat16 *>(sm + obox + swz(t, jc) + jin) = __float2bfloat16_rn(O[i]);
                }
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            if (nvalid == C) {
                if (tid == 0) {
                    ptx::tma_store_2d(&tm_o, hx, (int)row0, sm + OFF_OST);
                    ptx::tma_store_2d(&tm_o, hx + 64, (int)row0, sm + OFF_OST + 8192);
                    ptx::bulk_commit();
                }
            } else {
                // ragged last chunk: only rows < nvalid may be written
                const int t = tid >> 3, part = tid & 7;
                if (t < nvalid) {
                    __nv_bfloat16 *dst = p.out + (row0 + t) * rowstride + hx;
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int cc = 2 * part + k2;     // 16-byte chunk of the 256-byte row
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            sm + OFF_OST + (cc >> 3) * 8192 + swz(t, cc & 7));
                        *reinterpret_cast<uint4 *>(dst + cc * 8) = v;
                    }
                }
            }
        }
        if (*s_abort) break;
        if (p.final_state) {
            float X[32];
            ptx::tmem_ld32(lane_base + TM_D3 + 32 * cg, X);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) p.final_state[sidx + (int64_t)(32 * cg + i) * D + ch] = X[i];
        }
        ptx::tc_fence_before_sync();
        __syncthreads();
    }

    // ---- teardown: let in-flight copies and MMAs land before the CTA exits
    __syncthreads();
    if (*s_abort) {
        if (tid == 0) report_status(p.status, kDevTimeout);
        // wait (bounded) for every copy / MMA still in flight before leaving
        while (qk_done < qk_issued && ptx::mbar_wait(bar_qk, qk_done & 1, kWaitBudget)) ++qk_done;
        while (z_done < z_issued && ptx::mbar_wait(bar_z, z_done & 1, kWaitBudget)) ++z_done;
        while (v_done < v_issued && ptx::mbar_wait(bar_v, v_done & 1, kWaitBudget)) ++v_done;
        while (g_done < g_issued && ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done;
        while (s_done < s_issued && ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done;
        while (m_done < m_issued && ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done;
    }
    if (tid == 0) ptx::bulk_wait_all();   // output stores done before shared memory goes away
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// Host launcher.
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [T, H*128] bf16 viewed as a 2-D tensor; 64 x 64 boxes, 128-byte swizzle,
// rows beyond T read as zeros.
static bool make_map(CUtensorMap *m, const void *base, int64_t T, int H) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)H * 128, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)H * 128 * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_schedule(const int32_t *cu, int num_seqs, int32_t *order, uint32_t *counter,
                            uint32_t *status, cudaStream_t st);

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *z,
                              const float *A, const float *beta, const int32_t *cu,
                              int num_seqs, int64_t total, int H, const float *s0, float *s1,
                              void *out, void *workspace, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mz, mo;
    if (!make_map(&mq, q, total, H) || !make_map(&mk, k, total, H) ||
        !make_map(&mv, v, total, H) || !make_map(&mz, z, total, H) ||
        !make_map(&mo, out, total, H))
        return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kWsStatus);
    uint32_t *counter = reinterpret_cast<uint32_t *>(ws + kWsCounter);
    int32_t *order = reinterpret_cast<int32_t *>(ws + kWsOrder);
    cudaError_t e = launch_schedule(cu, num_seqs, order, counter, status, st);
    if (e != cudaSuccess) return e;

    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = cudaFuncSetAttribute(tc::prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const int64_t n_work = (int64_t)num_seqs * H;
    const int grid = (int)(n_work < sms ? n_work : sms);
    tc::Params prm;
    prm.A = A; prm.beta = beta; prm.cu_seqlens = cu; prm.initial_state = s0;
    prm.final_state = s1; prm.out = static_cast<__nv_bfloat16 *>(out); prm.order = order;
    prm.counter = counter; prm.status = status; prm.total_tokens = total;
    prm.num_seqs = num_seqs; prm.H = H;
    tc::prefill_tc_kernel<<<grid, tc::NT, tc::SMEM_ALLOC, st>>>(mq, mk, mv, mz, mo, prm);
    return cudaGetLastError();
}

}  // namespace kda
