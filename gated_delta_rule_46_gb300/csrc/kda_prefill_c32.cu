// kda_prefill_c32.cu -- the one-kernel chunkwise prefill for batches whose
// (sequence, head) chains fill the GPU, laid out so that TWO CTAs fit on every
// SM: 32-token chunks (two 16-token decay tiles), 256 threads, 112 KB of shared
// memory and 256 TMEM columns per CTA.
//
// Method ("Kimi K3 internals analysis", molayo1419.me, section "Sequence
// mixing"): the bounded gate g = -5 sigmoid(exp(A) z) keeps the cumulative
// log-decay of every 16-token tile inside (-80, 0), so the intra-chunk
// products split into bounded left and right factors and run as dense
// tensor-core tiles, the diagonal tiles included.  Per (sequence, head) and
// chunk, with start state S0 and chunk-local inclusive log-decay G:
//   L_ts = beta_t sum_c k_tc k_sc e^{G_tc - G_sc} (s < t),  P_ts = sum_c q_tc k_sc e^{G_tc - G_sc} (s <= t)
//   T = (I + L)^{-1} Diag(beta),  U = T (V - K~ S0),  O = Q~ S0 + P U,
//   S1 = Diag(e^{G_end}) S0 + Kend^T U,   K~ = k e^{G}, Q~ = q e^{G}, Kend = k e^{G_end - G}.
//
// Why two CTAs per SM: the per-chunk work is a chain of phases separated by
// block barriers and tensor-core round trips; with one CTA per SM the SIMT
// phases issue at full rate but every barrier and MMA wait leaves the SM idle.
// Two independent CTAs fill each other's idle phases.  A 32-token chunk keeps
// the working set small enough: [Q^; K^] 16 KB, the right factors of the two
// row tiles 48 rows (12 KB), [K~; Q~] 16 KB, Kend^T 16 KB, the bf16 state
// operand 32 KB; the small intermediates (L, Y, T, P, RHS/U, the output tile)
// reuse regions whose data is consumed (see the map below).
//
// Per chunk: A gate, decay, operands (SIMT) | MMA Gram/P (N = 48) and
// [K~S | Q~S] (N = 64) | RHS^T = V^T - (K~S)^T | P, L out of TMEM | the inverse:
// two diagonal 16 x 16 blocks by float32 forward substitution and the block
// below them as two 16 x 16 products on warp-level tf32 MMAs | U^T = RHS^T T^T (MMA, while the
// master state is scaled by e^{G_end}) | O^T += U^T P^T, S^T += U^T Kend (MMA) |
// the bf16 state copy and the output tile (TMA store).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_tc_util.cuh"
#include "kda_testing.h"
#include "sm100_ptx.cuh"

namespace kda {
namespace c32 {

using namespace tc;

constexpr int C = 32;      // chunk length (tokens): two 16-token decay tiles
constexpr int D = 128;     // dk = dv
constexpr int NT = 256;    // threads per CTA (8 warps)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kGMin2 = -5.0f * 1.4426950408889634f;   // g_min in log2 units
constexpr long long kWaitBudget = 2000000000LL;        // cycles (about one second)
constexpr long long kTestWaitBudget = 1LL << 21;

// ---- shared memory (bytes from a 1024-aligned base) -------------------------
// Operand tiles are K-major, 128-byte rows with the 16-byte chunk index XOR-ed
// with (row & 7) (the TMA 128B swizzle), 8-row groups 1024 B apart.
constexpr uint32_t R_QK = 0;           // [Q^ (rows 0-31); K^ (rows 32-63)], two K-blocks of 8 KB.  The
                                       // Gram MMA reads 128 rows per K-block; rows 64-127 are garbage lanes
constexpr uint32_t R_GB = 16384;       // right factors: tile 0 rows 0-15, tile 1 rows 16-47; K-blocks 6 KB
constexpr uint32_t GB_KB = 48 * 128;
constexpr int LS = 36;                 // float32 row stride of L and Y (after the Gram MMA, in R_GB)
constexpr uint32_t R_L = R_GB;
constexpr uint32_t R_Y = R_GB + C * LS * 4;
constexpr uint32_t R_OST = R_GB;       // output tile (after the inverse): two 64-channel boxes of 32 rows
constexpr uint32_t R_Z = 28672;        // z: two boxes of 64 channels x 32 rows
constexpr uint32_t R_V = 36864;        // v: two boxes; after the RHS, P [t][s] and T [t][s]
constexpr uint32_t R_P = R_V;
constexpr uint32_t R_T = R_V + 4096;
constexpr uint32_t R_B1 = 45056;       // [K~ (rows 0-31); Q~ (rows 32-63)], K-blocks 8 KB; after the state
constexpr uint32_t R_RU = R_B1;        // MMA: RHS^T, then U^T [j][s] (128 rows, K = 32)
constexpr uint32_t R_KE = 61440;       // Kend^T [c][s] (128 rows, K = 32)
constexpr uint32_t R_ST = 77824;       // S^T bf16 [j][c], two K-blocks of 16 KB
constexpr uint32_t R_BETA = 110592;    // 32 float
constexpr uint32_t R_EAN = R_BETA + 128;     // 128 float: -exp(A) log2(e)
constexpr uint32_t R_HT = R_EAN + 512;       // [4][128] float: sums of the log2 decay per 8-token group
constexpr uint32_t R_GAMMA = R_HT + 2048;    // 128 float: 2^(G_end)
constexpr uint32_t R_BAR = R_GAMMA + 512;    // 16 mbarriers
constexpr uint32_t R_SLOT = R_BAR + 128;     // TMEM base, work item, abort flag
constexpr uint32_t SMEM_USED = R_SLOT + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;   // slack to align the base to 1024 B
static_assert(R_GB + 2 * GB_KB <= R_Z && R_Y + C * LS * 4 <= R_Z && R_OST + 8192 <= R_Z, "R_GB region");
static_assert(R_T + 4096 <= R_B1 && R_KE + 16384 <= R_ST && R_ST + 32768 <= R_BETA, "regions");
static_assert(2 * (SMEM_ALLOC + 1024) <= 233472, "two CTAs per SM");

// ---- tensor memory (256 columns, 128 lanes) ---------------------------------
constexpr uint32_t TM_COLS = 256;
constexpr uint32_t TM_S = 0;           // S^T master, float32 [j][c]
constexpr uint32_t TM_D1 = 128;        // [(K~S0)^T | (Q~S0 + P U)^T], 32 + 32 columns
constexpr uint32_t TM_G = 192;         // Gram/P, 48 columns (lanes 0-31 P rows, 32-63 L rows)
constexpr uint32_t TM_U = 192;         // U^T, 32 columns (after P and L are out)

// first row of right-factor tile a (and its first TMEM column)
__device__ __forceinline__ int toff(int a) { return 16 * a; }

struct Params {
    const float *A;
    const float *beta;
    const int32_t *cu_seqlens;
    const float *initial_state;
    float *final_state;
    __nv_bfloat16 *out;
    const int32_t *order;
    uint32_t *counter;
    uint32_t *status;
    int64_t total_tokens;
    int num_seqs;
    int H;
    int test_expire;
    // state-pool mode (kda_decode_tokens) when pool != nullptr: sequence i is
    // tokens [i L, (i + 1) L), L = uniform_len, and its state is pool slot
    // slots[i] (or i), read and written in place; a negative slot is a padding
    // row (zero outputs, no state), a slot >= pool_size is reported and padded.
    // Chains are taken in order, CTA b the chains b, b + grid, ...
    float *pool;
    const int32_t *slots;
    int pool_size;
    int uniform_len;
};

struct Ctx {
    uint8_t *sm;
    float *s_beta, *s_eAn, *s_ht, *s_gamma;
    int tid, warp, lane, qw, half, ch;
    uint32_t lane_base;
};

__device__ __forceinline__ Ctx make_ctx(uint8_t *sm, uint32_t tmem) {
    Ctx x;
    x.sm = sm;
    x.s_beta = reinterpret_cast<float *>(sm + R_BETA);
    x.s_eAn = reinterpret_cast<float *>(sm + R_EAN);
    x.s_ht = reinterpret_cast<float *>(sm + R_HT);
    x.s_gamma = reinterpret_cast<float *>(sm + R_GAMMA);
    x.tid = threadIdx.x;
    x.warp = x.tid >> 5;
    x.lane = x.tid & 31;
    x.qw = x.warp & 3;                   // TMEM lane quarter
    x.half = x.warp >> 2;                // which half of the columns this warp takes
    x.ch = 32 * x.qw + x.lane;           // TMEM lane = value channel j
    x.lane_base = tmem + ((uint32_t)(32 * x.qw) << 16);
    return x;
}

// ---- state --------------------------------------------------------------------
// Master S^T [j][c] into TMEM and its bf16 copy into the state operand tile; this
// thread holds c in [64 half, 64 half + 64) of row j.  src == nullptr: zeros.
// The same from the float32 state [c][j] that a chain start bulk-copied into
// shared memory (rows 0-63 over the [K~; Q~] and Kend regions, rows 64-127
// over the state operand tile): every thread reads its 64 values first, then
// the bf16 copy overwrites the second half (a block barrier between).
__device__ __forceinline__ void load_state_staged(const Ctx &x) {
    const float *rows = reinterpret_cast<const float *>(x.sm + (x.half ? R_ST : R_B1));
    float Sm[2][32];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < 32; ++i) Sm[m][i] = rows[(32 * m + i) * D + x.ch];
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            st_chunk(x.sm + R_ST + x.half * 16384, swz(x.ch, 4 * m + q4), &Sm[m][8 * q4]);
        ptx::tmem_st32(x.lane_base + TM_S + 64 * x.half + 32 * m, Sm[m]);
    }
    ptx::tmem_st_wait();
}
__device__ __forceinline__ void load_state(const Ctx &x, const float *src) {
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
        float Sm[32];
        const int c0 = 64 * x.half + 32 * m;
#pragma unroll
        for (int i = 0; i < 32; ++i) Sm[i] = src ? src[(int64_t)(c0 + i) * D + x.ch] : 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            st_chunk(x.sm + R_ST + x.half * 16384, swz(x.ch, 4 * m + q4), &Sm[8 * q4]);
        ptx::tmem_st32(x.lane_base + TM_S + c0, Sm);
    }
    ptx::tmem_st_wait();
}
__device__ __forceinline__ void save_state(const Ctx &x, float *dst) {
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
        float X[32];
        const int c0 = 64 * x.half + 32 * m;
        ptx::tmem_ld32(x.lane_base + TM_S + c0, X);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[(int64_t)(c0 + i) * D + x.ch] = X[i];
    }
}
// S^T <- S^T Diag(2^G_end) on columns [c_lo, c_lo + 32 n) of this warp's lane
// quarter (the master only; the MMAs accumulate onto it)
__device__ __forceinline__ void scale_state(const Ctx &x, int c_lo, int n) {
#pragma unroll 1
    for (int m = 0; m < n; ++m) {
        float X[32], g[32];
        const int c0 = c_lo + 32 * m;
        ptx::tmem_ld32(x.lane_base + TM_S + c0, X);
#pragma unroll
        for (int i = 0; i < 32; i += 8) ld8(x.s_gamma + c0 + i, g + i);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) X[i] *= g[i];
        ptx::tmem_st32(x.lane_base + TM_S + c0, X);
    }
    ptx::tmem_st_wait();
}

// ---- phase A: gate, cumulative decay, operand tiles --------------------------
// Thread (warp w, lane l) owns key channels c = 64 (w >> 2) + 2l, c + 1 of the
// eight rows 8h .. 8h + 7, h = w & 3 (16-token tile h / 2).  The chunk-local log2
// decay is summed in registers; the four group sums per channel are exchanged
// through shared memory.  Writes [Q^; K^] in place, [K~; Q~], the right factors
// of the two Gram/P row tiles, Kend^T and 2^(G_end).  one_tile (at most 16 valid
// rows, every later product restricted to rows and columns 0-15): the rows of
// tile 1 and the tile-1 right factors are left as they are, as nothing reads
// what they feed.
__device__ __forceinline__ void phase_a(const Ctx &x, int nvalid, bool one_tile, uint64_t *bar_z,
                                        uint32_t &z_done, uint64_t *bar_qk, uint32_t &qk_done,
                                        volatile int *s_abort) {
    uint8_t *sm = x.sm;
    const int lane = x.lane, h = x.warp & 3, kb = x.warp >> 2;
    const int ta = h >> 1;
    const int c = 64 * kb + 2 * lane;
    const uint32_t cb = (uint32_t)(lane >> 2), co = (uint32_t)(lane & 3) * 4u;
    const float2 ea = *reinterpret_cast<const float2 *>(x.s_eAn + c);
    if (ptx::mbar_wait(bar_z, z_done & 1, kWaitBudget)) ++z_done; else *s_abort = 1;
    // a group of rows wholly past the chunk's valid rows (a short decode chunk,
    // a ragged tail) only writes zero operand rows (warp-uniform)
    const bool empty = 8 * h >= nvalid;
    float g0[8], g1[8];
    if (empty) {
#pragma unroll
        for (int i = 0; i < 8; ++i) g0[i] = g1[i] = 0.f;
        *reinterpret_cast<float2 *>(x.s_ht + h * 128 + c) = make_float2(0.f, 0.f);
    } else {
        const uint8_t *zt = sm + R_Z + kb * 4096;
        float run0 = 0.f, run1 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * h + i;
            const bool ok = t < nvalid;
            const float2 zz = bf2_to_f2(*reinterpret_cast<const uint32_t *>(zt + swz(t, cb) + co));
            run0 += ok ? kGMin2 * rcp(1.f + ex2(ea.x * zz.x)) : 0.f;
            run1 += ok ? kGMin2 * rcp(1.f + ex2(ea.y * zz.y)) : 0.f;
            g0[i] = run0;
            g1[i] = run1;
        }
        *reinterpret_cast<float2 *>(x.s_ht + h * 128 + c) = make_float2(run0, run1);
    }
    // the right-factor rows go over the previous chunk's output tile: it must have
    // been read by its TMA store
    if (x.tid == 0) ptx::bulk_wait_read();
    __syncthreads();
    // R_1 (end of tile 0), R_2 = G_end, and the first group of this tile when h is odd
    float R10, R11, R20, R21, hp0 = 0.f, hp1 = 0.f;
    {
        const float2 v0 = *reinterpret_cast<const float2 *>(x.s_ht + 0 * 128 + c);
        const float2 v1 = *reinterpret_cast<const float2 *>(x.s_ht + 1 * 128 + c);
        const float2 v2 = *reinterpret_cast<const float2 *>(x.s_ht + 2 * 128 + c);
        const float2 v3 = *reinterpret_cast<const float2 *>(x.s_ht + 3 * 128 + c);
        R10 = v0.x + v1.x; R11 = v0.y + v1.y;
        R20 = R10 + v2.x + v3.x; R21 = R11 + v2.y + v3.y;
        if (h == 1) { hp0 = v0.x; hp1 = v0.y; }
        if (h == 3) { hp0 = v2.x; hp1 = v2.y; }
    }
    const float Rt0 = ta ? R10 : 0.f, Rt1 = ta ? R11 : 0.f;
    if (h == 0) *reinterpret_cast<float2 *>(x.s_gamma + c) = make_float2(ex2(R20), ex2(R21));
    const float rho0 = ex2(Rt0), rho1 = ex2(Rt1);                   // 2^(R_ta)
    const float ke0 = ex2(R20 - Rt0), ke1 = ex2(R21 - Rt1);         // 2^(G_end - R_ta)
    const float f0 = ex2(R10), f1 = ex2(R11);                       // 2^(R_1 - R_0) (tile 0 rows only)
    if (ptx::mbar_wait(bar_qk, qk_done & 1, kWaitBudget)) ++qk_done; else *s_abort = 1;
    if (one_tile && ta == 1) return;
    uint8_t *qk = sm + R_QK + kb * 8192;
    uint8_t *b1 = sm + R_B1 + kb * 8192;
    uint8_t *gb = sm + R_GB + kb * GB_KB;
    float kr0[8], kr1[8];
    if (empty) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * h + i;
            const uint32_t oq = swz(t, cb) + co, okk = swz(32 + t, cb) + co;
            *reinterpret_cast<uint32_t *>(qk + oq) = 0u;
            *reinterpret_cast<uint32_t *>(qk + okk) = 0u;
            *reinterpret_cast<uint32_t *>(b1 + oq) = 0u;
            *reinterpret_cast<uint32_t *>(b1 + okk) = 0u;
            *reinterpret_cast<uint32_t *>(gb + swz(toff(ta) + t, cb) + co) = 0u;
            if (ta == 0 && !one_tile) *reinterpret_cast<uint32_t *>(gb + swz(toff(1) + t, cb) + co) = 0u;
            kr0[i] = kr1[i] = 0.f;
        }
        st_chunk(sm + R_KE, swz(c, h), kr0);
        st_chunk(sm + R_KE, swz(c + 1, h), kr1);
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = 8 * h + i;
        const bool ok = t < nvalid;
        const uint32_t oq = swz(t, cb) + co, okk = swz(32 + t, cb) + co;
        const float2 qv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qk + oq));
        const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qk + okk));
        const float x0 = hp0 + g0[i], x1 = hp1 + g1[i];             // G_t - R_ta
        const float el0 = ok ? ex2(x0) : 0.f, el1 = ok ? ex2(x1) : 0.f;
        const float dd0 = ok ? ex2(-x0) : 0.f, dd1 = ok ? ex2(-x1) : 0.f;
        const float qe0 = qv.x * el0, qe1 = qv.y * el1, kh0 = kv.x * el0, kh1 = kv.y * el1;
        const uint32_t pq = pack_bf16(qe0, qe1), pk = pack_bf16(kh0, kh1);
        *reinterpret_cast<uint32_t *>(qk + oq) = pq;                           // Q^
        *reinterpret_cast<uint32_t *>(qk + okk) = pk;                          // K^
        if (ta == 0) {   // R_0 = 0: K~ = K^ and Q~ = Q^
            *reinterpret_cast<uint32_t *>(b1 + oq) = pk;
            *reinterpret_cast<uint32_t *>(b1 + okk) = pq;
        } else {
            *reinterpret_cast<uint32_t *>(b1 + oq) = pack_bf16(kh0 * rho0, kh1 * rho1);    // K~
            *reinterpret_cast<uint32_t *>(b1 + okk) = pack_bf16(qe0 * rho0, qe1 * rho1);   // Q~
        }
        const float fr0 = kv.x * dd0, fr1 = kv.y * dd1;                        // k 2^(R_ta - G_t)
        kr0[i] = fr0 * ke0;
        kr1[i] = fr1 * ke1;
        *reinterpret_cast<uint32_t *>(gb + swz(toff(ta) + t, cb) + co) = pack_bf16(fr0, fr1);
        if (ta == 0 && !one_tile)   // tile 0 tokens also appear in tile 1's block: k 2^(R_1 - G_t)
            *reinterpret_cast<uint32_t *>(gb + swz(toff(1) + t, cb) + co) = pack_bf16(fr0 * f0, fr1 * f1);
    }
    st_chunk(sm + R_KE, swz(c, h), kr0);
    st_chunk(sm + R_KE, swz(c + 1, h), kr1);
}

// RHS^T [j][s] = V^T - (K~S0)^T into the RU tile; this thread: row j, s in
// [16 half, 16 half + 16).  Rows past the sequence end read as zero values.
__device__ __forceinline__ void phase_rhs(const Ctx &x, int nvalid) {
    float KS[16];
    ptx::tmem_ld16(x.lane_base + TM_D1 + 16 * x.half, KS);
    const int j = x.ch;
    const uint8_t *vb = x.sm + R_V + (j >> 6) * 4096;
    const uint32_t jc = (uint32_t)((j & 63) >> 3), jo = (uint32_t)(j & 7) * 2u;
    float r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int s = 16 * x.half + i;
        const float vv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(vb + swz(s, jc) + jo));
        r[i] = s < nvalid ? vv : 0.f;
    }
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] -= KS[i];
    st_chunk(x.sm + R_RU, swz(j, 2 * x.half), r);
    st_chunk(x.sm + R_RU, swz(j, 2 * x.half + 1), r + 8);
}

// P (lanes 0-31) and L (lanes 32-63) out of TMEM, masked: P into its bf16
// tile [t][s], L (times beta) in float32 [t][s].  Warps with lane quarter 0 or
// 1; half 0 takes s < 16, half 1 s >= 16.  Row t of tile a uses the block of
// tile a (columns 16a .. 16a + 16(a + 1) - 1, absolute s).
__device__ __forceinline__ void phase_extract(const Ctx &x) {
    if (x.qw >= 2) return;
    const bool isL = x.qw == 1;
    const int t = x.lane, a = t >> 4;
    float X[16], Y[16];
    // half 0: s = 0..15 sits in column 0.. (tile 0) or 16.. (tile 1); half 1: s = 16..31 in column 32..
    ptx::tmem_ld16(x.lane_base + TM_G + (x.half ? 32 : 0), X);
    ptx::tmem_ld16(x.lane_base + TM_G + 16, Y);
    ptx::tmem_ld_wait();
    const float bt = x.s_beta[t];
    float vals[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int s = 16 * x.half + i;
        float d;
        if (x.half == 0) d = a == 0 ? X[i] : Y[i];
        else d = a == 1 ? X[i] : 0.f;
        vals[i] = isL ? (s < t ? bt * d : 0.f) : (s <= t ? d : 0.f);
    }
    if (isL) {
        float4 *dst = reinterpret_cast<float4 *>(x.sm + R_L + (t * LS + 16 * x.half) * 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(vals[4 * i], vals[4 * i + 1], vals[4 * i + 2], vals[4 * i + 3]);
    } else {
        st_chunk(x.sm + R_P, swz(t, 2 * x.half), vals);
        st_chunk(x.sm + R_P, swz(t, 2 * x.half + 1), vals + 8);
    }
}

// Warps 0 and 1 (lanes 0-15): the diagonal blocks D_a = (I + L_aa)^{-1} by
// forward substitution in float32, one column per lane, into Y.
__device__ __forceinline__ void phase_diag(const Ctx &x, int nblocks = 2) {
    if (x.warp >= nblocks || x.lane >= 16) return;
    const float *Lm = reinterpret_cast<const float *>(x.sm + R_L);
    float *Ym = reinterpret_cast<float *>(x.sm + R_Y);
    const int b0 = 16 * x.warp;
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float lr[16];
        const float *src = Lm + (b0 + i) * LS + b0;
        ld8(src, lr);
        ld8(src + 8, lr + 8);
        float a0 = (i == x.lane) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < i; ++m) {
            if (m & 1) a1 -= lr[m] * y[m]; else a0 -= lr[m] * y[m];
        }
        y[i] = a0 + a1;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Ym[(b0 + i) * LS + b0 + x.lane] = y[i];
}

// A barrier of warps 0 and 1 only (named barrier 1), so that the other warps
// run on meanwhile.
__device__ __forceinline__ void sync_w01() { asm volatile("bar.sync 1, 64;" ::: "memory"); }

// tf32 of a float32 (round to nearest, ties away)
__device__ __forceinline__ uint32_t to_tf32(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}
// d += a b for one m16n8k8 tile, tf32 inputs, float32 accumulation.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// acc (16 x 16, two n-tiles) = A (16 x 16 at Am, row stride LS) B (16 x 16 at
// Bm), one warp; fragment layouts of m16n8k8 (g = lane / 4, q = lane % 4).
__device__ __forceinline__ void warp_mm16(float (&acc)[2][4], const float *Am, const float *Bm, int lane) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4];
        a[0] = to_tf32(Am[g * LS + 8 * ks + q]);
        a[1] = to_tf32(Am[(g + 8) * LS + 8 * ks + q]);
        a[2] = to_tf32(Am[g * LS + 8 * ks + q + 4]);
        a[3] = to_tf32(Am[(g + 8) * LS + 8 * ks + q + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b0 = to_tf32(Bm[(8 * ks + q) * LS + 8 * nt + g]);
            const uint32_t b1 = to_tf32(Bm[(8 * ks + q + 4) * LS + 8 * nt + g]);
            mma_tf32(acc[nt], a, b0, b1);
        }
    }
}

// Warps 0 and 1: the block below the diagonal, Y_10 = -D_1 L_10 D_0, on warp 0's
// tf32 tensor-core MMAs (float32 accumulation; the diagonal blocks, solved
// before in float32, carry the precision), then T = Y Diag(beta) into its bf16
// tile by both warps.
__device__ __forceinline__ void phase_offdiag_T(const Ctx &x) {
    float *Lm = reinterpret_cast<float *>(x.sm + R_L);
    float *Ym = reinterpret_cast<float *>(x.sm + R_Y);
    if (x.warp == 0) {
        const int g = x.lane >> 2, q = x.lane & 3;
        float acc[2][4];
        warp_mm16(acc, Lm + 16 * LS, Ym, x.lane);            // X = L_10 D_0
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {                      // X into the unused upper-right block of L
            Lm[g * LS + 16 + 8 * nt + 2 * q] = acc[nt][0];
            Lm[g * LS + 16 + 8 * nt + 2 * q + 1] = acc[nt][1];
            Lm[(g + 8) * LS + 16 + 8 * nt + 2 * q] = acc[nt][2];
            Lm[(g + 8) * LS + 16 + 8 * nt + 2 * q + 1] = acc[nt][3];
        }
        __syncwarp();
        warp_mm16(acc, Ym + 16 * LS + 16, Lm + 16, x.lane);  // D_1 X
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {                      // Y_10 = -D_1 X
            Ym[(16 + g) * LS + 8 * nt + 2 * q] = -acc[nt][0];
            Ym[(16 + g) * LS + 8 * nt + 2 * q + 1] = -acc[nt][1];
            Ym[(24 + g) * LS + 8 * nt + 2 * q] = -acc[nt][2];
            Ym[(24 + g) * LS + 8 * nt + 2 * q + 1] = -acc[nt][3];
        }
    }
    sync_w01();
    const int u = x.tid;                       // 0 .. 63
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {   // T [t][s] = Y [t][s] beta_s (s <= block of t), zero above
        const int e = u + 64 * rep;             // one 8-column chunk of a row
        const int t = e >> 2, p = e & 3;
        const int a = t >> 4;
        float v[8], bt[8];
        ld8(Ym + t * LS + 8 * p, v);
        ld8(x.s_beta + 8 * p, bt);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (8 * p + i < 16 * (a + 1)) ? v[i] * bt[i] : 0.f;
        st_chunk(x.sm + R_T, swz(t, p), v);
    }
}

// A chunk with at most 16 valid rows: its second tile is empty (zero L rows,
// zero beta), so T = D_0 Diag(beta) in the first 16 x 16 block and zero
// elsewhere.  Warps 0 and 1, after warp 0 has solved D_0 (phase_diag with one
// block).
__device__ __forceinline__ void phase_T_single(const Ctx &x) {
    const float *Ym = reinterpret_cast<const float *>(x.sm + R_Y);
    const int u = x.tid;                       // 0 .. 63
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
        const int e = u + 64 * rep;             // one 8-column chunk of a row
        const int t = e >> 2, p = e & 3;
        float v[8];
        if (t < 16 && p < 2) {
            float bt[8];
            ld8(Ym + t * LS + 8 * p, v);
            ld8(x.s_beta + 8 * p, bt);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= bt[i];
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        st_chunk(x.sm + R_T, swz(t, p), v);
    }
}

// U^T out of TMEM into the RU tile (over RHS^T, read by the finished U MMA):
// row j, t in [16 half, 16 half + 16).
__device__ __forceinline__ void phase_u_out(const Ctx &x) {
    float U[16];
    ptx::tmem_ld16(x.lane_base + TM_U + 16 * x.half, U);
    ptx::tmem_ld_wait();
    st_chunk(x.sm + R_RU, swz(x.ch, 2 * x.half), U);
    st_chunk(x.sm + R_RU, swz(x.ch, 2 * x.half + 1), U + 8);
}

// The new state's bf16 copy into the state operand tile, and O^T (t in [16 half,
// 16 half + 16)) into the output tile [t][j] (two 64-channel TMA boxes).
__device__ __forceinline__ void phase_state_out(const Ctx &x) {
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
        float X[32];
        ptx::tmem_ld32(x.lane_base + TM_S + 64 * x.half + 32 * m, X);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
            st_chunk(x.sm + R_ST + x.half * 16384, swz(x.ch, 4 * m + q4), &X[8 * q4]);
    }
    float O[16];
    ptx::tmem_ld16(x.lane_base + TM_D1 + 32 + 16 * x.half, O);
    ptx::tmem_ld_wait();
    const int j = x.ch;
    const uint32_t obox = R_OST + (uint32_t)(j >> 6) * 4096u;
    const uint32_t jc = (uint32_t)((j & 63) >> 3), jo = (uint32_t)(j & 7) * 2u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int t = 16 * x.half + i;
        *reinterpret_cast<__nv_bfloat16 *>(x.sm + obox + swz(t, jc) + jo) = __float2bfloat16_rn(O[i]);
    }
}
// Only O^T into the output tile (the last chunk of a chain in state-pool
// mode: nobody reads the bf16 state copy, its region receives the next
// chain's start state).
__device__ __forceinline__ void phase_o_out(const Ctx &x) {
    float O[16];
    ptx::tmem_ld16(x.lane_base + TM_D1 + 32 + 16 * x.half, O);
    ptx::tmem_ld_wait();
    const int j = x.ch;
    const uint32_t obox = R_OST + (uint32_t)(j >> 6) * 4096u;
    const uint32_t jc = (uint32_t)((j & 63) >> 3), jo = (uint32_t)(j & 7) * 2u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int t = 16 * x.half + i;
        *reinterpret_cast<__nv_bfloat16 *>(x.sm + obox + swz(t, jc) + jo) = __float2bfloat16_rn(O[i]);
    }
}

// The staged output tile to global memory (after a block barrier): one TMA
// store per 64-channel box for a full chunk, 16-byte stores of the rows <
// nvalid otherwise.
__device__ __forceinline__ void store_output(const Ctx &x, const CUtensorMap *tm_o, __nv_bfloat16 *out,
                                             int64_t row0, int nvalid, int hx, int64_t rowstride) {
    if (nvalid == C) {
        if (x.tid == 0) {
            ptx::tma_store_2d(tm_o, hx, (int)row0, x.sm + R_OST);
            ptx::tma_store_2d(tm_o, hx + 64, (int)row0, x.sm + R_OST + 4096);
            ptx::bulk_commit();
        }
    } else {
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
            const int e = x.tid + NT * rep;          // 32 rows x 16 chunks of 16 bytes
            const int t = e >> 4, cc = e & 15;
            if (t < nvalid) {
                const uint4 v = *reinterpret_cast<const uint4 *>(x.sm + R_OST + (cc >> 3) * 4096 + swz(t, cc & 7));
                *reinterpret_cast<uint4 *>(out + (row0 + t) * rowstride + hx + cc * 8) = v;
            }
        }
    }
}

__device__ __forceinline__ void tma_2box(uint8_t *dst, const CUtensorMap *tm, int hx, int y, uint64_t *bar) {
    ptx::mbar_arrive_expect_tx(bar, 8192);
    ptx::tma_load_2d(dst, tm, hx, y, bar);
    ptx::tma_load_2d(dst + 4096, tm, hx + 64, y, bar);
}
__device__ __forceinline__ void tma_qk(uint8_t *sm, const CUtensorMap *tq, const CUtensorMap *tk, int hx, int y,
                                       uint64_t *bar) {
    ptx::mbar_arrive_expect_tx(bar, 16384);
    ptx::tma_load_2d(sm + R_QK, tq, hx, y, bar);                // q rows 0-31, channels 0-63
    ptx::tma_load_2d(sm + R_QK + 4096, tk, hx, y, bar);         // k rows 32-63
    ptx::tma_load_2d(sm + R_QK + 8192, tq, hx + 64, y, bar);    // channels 64-127
    ptx::tma_load_2d(sm + R_QK + 12288, tk, hx + 64, y, bar);
}

// POOL: the state-pool mode (kda_decode_tokens); the prefill instantiation
// carries none of its code.
template <bool POOL>
__global__ void __launch_bounds__(NT, 2)
prefill_c32_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_z,
                   const __grid_constant__ CUtensorMap tm_o, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(sm);
    uint64_t *bar_qk = reinterpret_cast<uint64_t *>(sm + R_BAR);
    uint64_t *bar_z = bar_qk + 1;
    uint64_t *bar_v = bar_qk + 2;
    uint64_t *bar_g = bar_qk + 3;      // Gram/P MMA done
    uint64_t *bar_s = bar_qk + 4;      // state MMA done
    uint64_t *bar_m = bar_qk + 5;      // U MMA, then the output MMA done
    uint64_t *bar_m2 = bar_qk + 6;     // the state update MMA done (thread 32)
    uint64_t *bar_never = bar_qk + 7;  // test support: nothing arrives here
    uint64_t *bar_st = bar_qk + 8;     // a chain's start state bulk-copied into shared memory
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + R_SLOT);
    volatile int *s_work = reinterpret_cast<volatile int *>(sm + R_SLOT + 4);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + R_SLOT + 8);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = p.H;
    const int64_t rowstride = (int64_t)H * D;

    if (tid == 0) {
        for (int i = 0; i < 9; ++i) ptx::mbar_init(bar_qk + i, 1);
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
    const Ctx x = make_ctx(sm, tmem);
    ptx::pdl_wait();                 // the schedule kernel's order, counter and status
    ptx::pdl_launch_dependents();

    uint32_t qk_issued = 0, qk_done = 0, z_issued = 0, z_done = 0, v_issued = 0, v_done = 0;
    uint32_t g_issued = 0, g_done = 0, s_issued = 0, s_done = 0, m_issued = 0, m_done = 0;
    uint32_t m2_issued = 0, m2_done = 0, st_issued = 0, st_done = 0;
    const int n_work = p.num_seqs * H;
    bool first = true;

    constexpr bool pool_mode = POOL;
    int next_static = blockIdx.x;
    const float *pre_init = nullptr;   // a start state whose bulk copy the previous chain issued
    for (;;) {
        if (pool_mode) {
            if (tid == 0) *s_work = next_static;
            next_static += gridDim.x;
        } else if (tid == 0) {
            *s_work = (int)atomicAdd(p.counter, 1u);
        }
        __syncthreads();
        const int w = *s_work;
        if (w >= n_work || *s_abort) break;
        const int seq = pool_mode ? w / H : p.order[w / H];
        const int h = w % H;
        const int hx = h * D;
        int64_t bos, eos;
        const float *s_init;
        float *s_fin;
        if (pool_mode) {
            bos = (int64_t)seq * p.uniform_len;
            eos = bos + p.uniform_len;
            const int slot = p.slots ? p.slots[seq] : seq;
            if (slot < 0 || slot >= p.pool_size) {   // padding row: zero outputs, no state
                if (slot >= p.pool_size && tid == 0) report_status(p.status, kDevBadSeqlens);
                for (int e = tid; e < p.uniform_len * 16; e += NT)
                    *reinterpret_cast<uint4 *>(p.out + (bos + e / 16) * rowstride + hx + (e % 16) * 8) =
                        make_uint4(0u, 0u, 0u, 0u);
                __syncthreads();   // (*s_work is rewritten by the next item)
                continue;
            }
            s_init = s_fin = p.pool + ((size_t)slot * H + h) * D * D;
        } else {
            seq_bounds(p.cu_seqlens, seq, p.total_tokens, p.status, tid, bos, eos);
            const int64_t sidx = ((int64_t)seq * H + h) * D * D;
            s_init = p.initial_state ? p.initial_state + sidx : nullptr;
            s_fin = p.final_state ? p.final_state + sidx : nullptr;
        }
        const int nchunks = (int)((eos - bos + C - 1) / C);

        // the start state by two bulk copies (the copy engine keeps all 64 KB in
        // flight; per-thread loads of the columns would wait several memory round
        // trips), when it is 16-byte aligned
        const bool staged = s_init && (reinterpret_cast<uintptr_t>(s_init) & 15) == 0;
        const bool pre = staged && s_init == pre_init;   // already in flight
        pre_init = nullptr;
        if (tid == 0) {
            if (staged && !pre) {
                ptx::mbar_arrive_expect_tx(bar_st, 65536);
                bulk_copy_in(sm + R_B1, reinterpret_cast<const uint8_t *>(s_init), 32768, bar_st);
                bulk_copy_in(sm + R_ST, reinterpret_cast<const uint8_t *>(s_init + 64 * D), 32768, bar_st);
            }
            if (nchunks > 0) {
                tma_qk(sm, &tm_q, &tm_k, hx, (int)bos, bar_qk);
                tma_2box(sm + R_Z, &tm_z, hx, (int)bos, bar_z);
                tma_2box(sm + R_V, &tm_v, hx, (int)bos, bar_v);
            }
        }
        if (nchunks > 0) { ++qk_issued; ++z_issued; ++v_issued; }
        if (staged) {
            if (!pre) ++st_issued;
            if (ptx::mbar_wait(bar_st, st_done & 1, kWaitBudget)) ++st_done; else *s_abort = 1;
            load_state_staged(x);
        } else {
            load_state(x, s_init);
        }
        if (pool_mode) {   // the next chain's state into L2 while this one runs (64 KB, 512 lines)
            const int wn = w + (int)gridDim.x;
            if (wn < n_work) {
                const int sn = p.slots ? p.slots[wn / H] : wn / H;
                if (sn >= 0 && sn < p.pool_size) {
                    const uint8_t *nx = reinterpret_cast<const uint8_t *>(p.pool + ((size_t)sn * H + wn % H) * D * D);
                    for (int i = tid; i < D * D * 4 / 128; i += NT) ptx::prefetch_l2(nx + (size_t)i * 128);
                }
            }
        }
        if (tid < D) x.s_eAn[tid] = -expf(p.A[h * D + tid]) * kLog2e;
        float beta_next = 0.f;
        if (tid < C && bos + tid < eos) beta_next = p.beta[(bos + tid) * H + h];
        __syncthreads();

        for (int cidx = 0; cidx < nchunks; ++cidx) {
            const int64_t row0 = bos + (int64_t)cidx * C;
            const int nvalid = (int)((eos - row0) < C ? (eos - row0) : C);
            const bool has_next = (cidx + 1 < nchunks);
            const int64_t next_row = row0 + C;

            // ===== A: gate, cumulative decay, operands
            if (tid < C) x.s_beta[tid] = beta_next;
            if (first && (p.test_expire & KDA_TESTING_FUSED) && blockIdx.x == 0 &&
                !ptx::mbar_wait(bar_never, 0, kTestWaitBudget))
                *s_abort = 1;
            first = false;
            phase_a(x, nvalid, pool_mode && nvalid <= 16, bar_z, z_done, bar_qk, qk_done, s_abort);
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            // One thread issues a tcgen05.mma only about every 100 cycles, so the
            // two independent products go to two issuing threads.
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                if (has_next) tma_2box(sm + R_Z, &tm_z, hx, (int)next_row, bar_z);   // z is read
                // Gram/P: D[r][16a + s] = [Q^;K^][r] . B[16a + s], both row tiles
                mma_k<8>(tmem + TM_G, sbase + R_QK, 8192u, sbase + R_GB, GB_KB, ptx::idesc_bf16_f32(128, 48),
                         false);
                ptx::mma_commit(bar_g);
            } else if (tid == 32) {
                ptx::tc_fence_after_sync();
                // state product: D1[j][s | t] = S^T[j] . [K~; Q~][s | t]
                mma_k<8>(tmem + TM_D1, sbase + R_ST, 16384u, sbase + R_B1, 8192u, ptx::idesc_bf16_f32(128, 64),
                         false);
                ptx::mma_commit(bar_s);
            }
            ++g_issued; ++s_issued;
            if (has_next) ++z_issued;

            // ===== RHS^T = V^T - (K~S0)^T (over [K~; Q~], read by the finished state MMA)
            if (ptx::mbar_wait(bar_v, v_done & 1, kWaitBudget)) ++v_done; else *s_abort = 1;
            if (ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            // (a state-pool chunk of at most 16 valid rows: the U product takes one K
            // step, token columns 0-15, so the warps of columns 16-31 skip)
            if (!(pool_mode && nvalid <= 16 && x.half)) phase_rhs(x, nvalid);
            // ===== P and L out of TMEM (P goes over v, read above)
            if (ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            __syncthreads();
            if (tid == 0 && has_next) tma_qk(sm, &tm_q, &tm_k, hx, (int)next_row, bar_qk);   // [Q^;K^] read
            if (has_next) ++qk_issued;
            // (columns s >= 16 of P and L feed neither the one-tile inverse nor the
            // one-K-step output product)
            if (!(pool_mode && nvalid <= 16 && x.half)) phase_extract(x);
            __syncthreads();
            // ===== warps 0-1: the inverse T = (I + L)^{-1} Diag(beta); warps 2-7
            // meanwhile: S^T <- S^T Diag(2^G_end) (warps 4 and 5 take the two lane
            // quarters of warps 0 and 1 in full, warps 2, 3, 6, 7 half of theirs)
            if (warp < 2) {
                if (nvalid <= 16) {   // one 16-token tile (a short decode chunk, a ragged tail)
                    phase_diag(x, 1);
                    sync_w01();
                    phase_T_single(x);
                } else {
                    phase_diag(x);
                    sync_w01();
                    phase_offdiag_T(x);
                }
            } else if (warp == 4 || warp == 5) {
                scale_state(x, 0, 4);
            } else {
                scale_state(x, 64 * x.half, 2);
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                // U^T = RHS^T T^T
                // (at most 16 valid rows: the tokens past 16 contribute zeros, one K step)
                if (nvalid <= 16)
                    mma_k<1>(tmem + TM_U, sbase + R_RU, 0u, sbase + R_T, 0u, ptx::idesc_bf16_f32(128, 32), false);
                else
                    mma_k<2>(tmem + TM_U, sbase + R_RU, 0u, sbase + R_T, 0u, ptx::idesc_bf16_f32(128, 32), false);
                ptx::mma_commit(bar_m);
            }
            ++m_issued;
            if (tid < C && has_next) {
                beta_next = 0.f;
                if (next_row + tid < eos) beta_next = p.beta[(next_row + tid) * H + h];
            }
            if (ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            if (!(pool_mode && nvalid <= 16 && x.half)) phase_u_out(x);
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                // O^T += U^T P^T (onto the Q~S0 half of D1)
                if (nvalid <= 16)
                    mma_k<1>(tmem + TM_D1 + 32, sbase + R_RU, 0u, sbase + R_P, 0u, ptx::idesc_bf16_f32(128, 32), true);
                else
                    mma_k<2>(tmem + TM_D1 + 32, sbase + R_RU, 0u, sbase + R_P, 0u, ptx::idesc_bf16_f32(128, 32), true);
                ptx::mma_commit(bar_m);
            } else if (tid == 32) {
                ptx::tc_fence_after_sync();
                // S^T += U^T Kend
                if (nvalid <= 16)
                    mma_k<1>(tmem + TM_S, sbase + R_RU, 0u, sbase + R_KE, 0u, ptx::idesc_bf16_f32(128, 128), true);
                else
                    mma_k<2>(tmem + TM_S, sbase + R_RU, 0u, sbase + R_KE, 0u, ptx::idesc_bf16_f32(128, 128), true);
                ptx::mma_commit(bar_m2);
            }
            ++m_issued;
            ++m2_issued;
            if (ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done; else *s_abort = 1;
            if (ptx::mbar_wait(bar_m2, m2_done & 1, kWaitBudget)) ++m2_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            if (tid == 0 && has_next) tma_2box(sm + R_V, &tm_v, hx, (int)next_row, bar_v);   // P, T are read
            if (has_next) ++v_issued;
            if (pool_mode && !has_next) {
                // the chain's last products are done, so its staging regions are free:
                // the next chain's start state starts arriving now, during the output
                // and the state save, instead of at the next chain's start
                const int wn = w + (int)gridDim.x;
                if (wn < n_work) {
                    const int sn = p.slots ? p.slots[wn / H] : wn / H;
                    if (sn >= 0 && sn < p.pool_size) {
                        pre_init = p.pool + ((size_t)sn * H + wn % H) * D * D;
                        if (tid == 0) {
                            ptx::mbar_arrive_expect_tx(bar_st, 65536);
                            bulk_copy_in(sm + R_B1, reinterpret_cast<const uint8_t *>(pre_init), 32768, bar_st);
                            bulk_copy_in(sm + R_ST, reinterpret_cast<const uint8_t *>(pre_init + 64 * D), 32768,
                                         bar_st);
                        }
                        ++st_issued;
                    }
                }
            }
            if (pre_init) {
                if (!(nvalid <= 16 && x.half)) phase_o_out(x);   // rows >= 16 are not stored
            } else {
                phase_state_out(x);
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            store_output(x, &tm_o, p.out, row0, nvalid, hx, rowstride);
        }
        if (*s_abort) break;
        if (s_fin) save_state(x, s_fin);
        ptx::tc_fence_before_sync();
        __syncthreads();
    }

    __syncthreads();
    if (*s_abort) {
        if (tid == 0) report_status(p.status, kDevTimeout);
        while (qk_done < qk_issued && ptx::mbar_wait(bar_qk, qk_done & 1, kWaitBudget)) ++qk_done;
        while (z_done < z_issued && ptx::mbar_wait(bar_z, z_done & 1, kWaitBudget)) ++z_done;
        while (v_done < v_issued && ptx::mbar_wait(bar_v, v_done & 1, kWaitBudget)) ++v_done;
        while (g_done < g_issued && ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done;
        while (s_done < s_issued && ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done;
        while (m_done < m_issued && ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done;
        while (m2_done < m2_issued && ptx::mbar_wait(bar_m2, m2_done & 1, kWaitBudget)) ++m2_done;
        while (st_done < st_issued && ptx::mbar_wait(bar_st, st_done & 1, kWaitBudget)) ++st_done;
    }
    if (tid == 0) ptx::bulk_wait_all();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace c32
}  // namespace kda

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace kda {

bool make_map_bf16(CUtensorMap *m, const void *base, int64_t T, int H, int box_rows);

// The fused plan with the two-CTAs-per-SM kernel: persistent CTAs (two per
// SM) walk the (sequence, head) chains longest-first from the counter the
// schedule kernel reset.
cudaError_t launch_prefill_c32(const void *q, const void *k, const void *v, const void *z, const float *A,
                               const float *beta, const int32_t *cu, int num_seqs, int64_t total, int H,
                               const float *s0, float *s1, void *out, int32_t *order, uint32_t *counter,
                               uint32_t *status, int test_expire, int sms, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mz, mo;
    if (!make_map_bf16(&mq, q, total, H, c32::C) || !make_map_bf16(&mk, k, total, H, c32::C) ||
        !make_map_bf16(&mv, v, total, H, c32::C) || !make_map_bf16(&mz, z, total, H, c32::C) ||
        !make_map_bf16(&mo, out, total, H, c32::C))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(c32::prefill_c32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)c32::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    c32::Params prm;
    prm.A = A; prm.beta = beta; prm.cu_seqlens = cu; prm.initial_state = s0; prm.final_state = s1;
    prm.out = static_cast<__nv_bfloat16 *>(out); prm.order = order; prm.counter = counter;
    prm.status = status; prm.total_tokens = total; prm.num_seqs = num_seqs; prm.H = H;
    prm.test_expire = test_expire;
    prm.pool = nullptr; prm.slots = nullptr; prm.pool_size = 0; prm.uniform_len = 0;
    const int64_t chains = (int64_t)num_seqs * H;
    const int64_t cap = 2 * (int64_t)sms;
    const unsigned grid = (unsigned)(chains < cap ? chains : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(c32::NT);
    cfg.dynamicSmemBytes = c32::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, c32::prefill_c32_kernel<false>, mq, mk, mv, mz, mo, prm);
}

// kda_decode_tokens on the tensor cores (bf16, dk = dv = 128): the n tokens of
// every sequence are one or more chunks of the one-kernel prefill, its state
// read from and written back to its pool slot.
cudaError_t launch_decode_tokens_tc(const void *q, const void *k, const void *v, const void *z, const float *A,
                                    const float *beta, float *pool, int pool_size, const int32_t *slots, void *out,
                                    int N, int n_tokens, int H, uint32_t *status, int sms, cudaStream_t st) {
    const int64_t total = (int64_t)N * n_tokens;
    CUtensorMap mq, mk, mv, mz, mo;
    if (!make_map_bf16(&mq, q, total, H, c32::C) || !make_map_bf16(&mk, k, total, H, c32::C) ||
        !make_map_bf16(&mv, v, total, H, c32::C) || !make_map_bf16(&mz, z, total, H, c32::C) ||
        !make_map_bf16(&mo, out, total, H, c32::C))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(c32::prefill_c32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)c32::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    c32::Params prm{};
    prm.A = A; prm.beta = beta; prm.cu_seqlens = nullptr; prm.initial_state = nullptr; prm.final_state = nullptr;
    prm.out = static_cast<__nv_bfloat16 *>(out); prm.order = nullptr; prm.counter = nullptr;
    prm.status = status; prm.total_tokens = total; prm.num_seqs = N; prm.H = H; prm.test_expire = 0;
    prm.pool = pool; prm.slots = slots; prm.pool_size = pool_size; prm.uniform_len = n_tokens;
    const int64_t chains = (int64_t)N * H;
    const int64_t cap = 2 * (int64_t)sms;
    const unsigned grid = (unsigned)(chains < cap ? chains : cap);
    c32::prefill_c32_kernel<true><<<grid, c32::NT, c32::SMEM_ALLOC, st>>>(mq, mk, mv, mz, mo, prm);
    return cudaGetLastError();
}

}  // namespace kda
