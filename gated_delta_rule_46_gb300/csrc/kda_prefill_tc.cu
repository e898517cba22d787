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
// Every kernel here runs 512 threads (16 warps) per CTA, one CTA per SM, with
// bf16 operands in 128-byte-swizzled K-major shared-memory tiles and float32
// accumulators in TMEM.  Per 64-token chunk:
//   A    SIMT: gate, cumulative decay, operand tiles (phase_gate_operands)
//   MMA  Gram/P tiles [Q^;K^] x B_a^T (one N = 160 chain)
//   B    P and L out of TMEM, the inverse T = (I + L)^{-1} Diag(beta): diagonal
//        blocks in float32 SIMT, the rest on warp-level tf32 MMAs
//   then the state pass: U, O = Q~S0 + PU and the new state on tcgen05.
// The state is kept transposed (rows = value channels) so every state
// accumulator has M = 128 rows, one per TMEM lane.  Plans (host code at the
// end): the fused persistent kernel for batches whose chains fill the GPU; for
// few chains the state-independent work runs chunk-parallel in
// prefill_intra_kernel and the state pass either window by window or as a
// segment scan (pass 1, scan, pass 2).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kda_common.cuh"
#include "kda_tc_util.cuh"
#include "kda_testing.h"
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
constexpr uint32_t OFF_TB = 139264;    // T [t][s]: 64 x 64 bf16 (after the state MMA)
constexpr uint32_t OFF_RU = 155648;    // RHS^T, then U^T: 128 x 64 bf16 (after the state MMA)
constexpr uint32_t OFF_KE = 172032;    // Kend^T [c][s] 128 x 64 bf16
constexpr uint32_t OFF_ST = 188416;    // S^T [j][c] 128 x 128 bf16 (A of the state MMA)
constexpr uint32_t OFF_KT = OFF_ST + 8192;   // intra kernel only: K~^T [c][s] 128 x 64 bf16
constexpr uint32_t OFF_MISC = 221184;
constexpr uint32_t OFF_BETA = OFF_MISC;              // 64 float
constexpr uint32_t OFF_EAN = OFF_BETA + 256;         // 128 float: -exp(A) log2(e)
constexpr uint32_t OFF_HT = OFF_EAN + 512;           // [8][128]: half-tile sums of the log2 decay
constexpr uint32_t OFF_GAMMA = OFF_HT + 4096;        // 128 float: 2^(G_end)
constexpr uint32_t OFF_BAR = OFF_GAMMA + 512;        // mbarriers
constexpr uint32_t OFF_SLOT = OFF_BAR + 64;          // TMEM base, work item, abort flag
constexpr uint32_t OFF_CU = OFF_SLOT + 64;           // intra kernel: cu_seqlens cache (CU_CACHE entries)
constexpr int CU_CACHE = 256;
constexpr uint32_t SMEM_USED = OFF_CU + 4 * CU_CACHE;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;    // slack to align the base to 1024 B
static_assert(OFF_GB + 2 * GB_KBLK <= OFF_B1, "right-factor tiles overlap");
static_assert(OFF_Y + 64 * LSTR * 4 <= OFF_TB, "solve scratch overlaps");
static_assert(OFF_RU + 16384 <= OFF_KE, "RU overlaps");
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// ---- tensor memory map (columns; 128 lanes each) ----------------------------
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t TM_G = 0;           // Gram/P tiles, N = 160 (tile a at column 16a(a+1)/2)
constexpr uint32_t TM_D1 = 192;        // [(K~S0)^T | (Q~S0 + P U)^T]  128 x 128
constexpr uint32_t TM_D2 = 320;        // U^T 128 x 64
constexpr uint32_t TM_D3 = 384;        // dS^T 128 x 128

constexpr long long kWaitBudget = 2000000000LL;   // cycles (about one second)

// Test support (kda_testing_expire_next_wait): CTA 0 of the kernels named by a
// bit of `test_expire` makes one bounded wait on an mbarrier that nothing ever
// arrives at, with this short budget, before its first chunk.  The wait runs
// out like one whose copy never landed, and the kernel takes its ordinary
// timeout path: record KDA_ERR_DEVICE_TIMEOUT, let the copies and MMAs in
// flight land, free TMEM, return.
constexpr long long kTestWaitBudget = 1LL << 21;   // cycles (about a millisecond)
enum : int {
    kExpireFused = KDA_TESTING_FUSED, kExpireIntra = KDA_TESTING_INTRA, kExpireSeg = KDA_TESTING_SEGMENT,
    kExpireScan = KDA_TESTING_SCAN, kExpireState = KDA_TESTING_STATE
};
__device__ __forceinline__ bool test_wait_expires(int mask, int bit, uint64_t *bar_never) {
    return (mask & bit) && blockIdx.x == 0 && !ptx::mbar_wait(bar_never, 0, kTestWaitBudget);
}

// first row (and TMEM column) of right-factor tile a: 0, 16, 48, 96
__device__ __forceinline__ int tile_off(int a) { return 8 * a * (a + 1); }

// Per-thread view of the CTA: shared-memory pointers and the thread's roles.
struct Ctx {
    uint8_t *sm;
    float *s_beta, *s_eAn, *s_ht, *s_gamma, *Lm, *Ym;
    int tid, warp, lane;
    int qw, cg, ch;        // phases B-D: TMEM lane quarter, column group, value channel j
    uint32_t lane_base;    // TMEM address of this warp's lane quarter
};

__device__ __forceinline__ Ctx make_ctx(uint8_t *sm, uint32_t tmem) {
    Ctx x;
    x.sm = sm;
    x.s_beta = reinterpret_cast<float *>(sm + OFF_BETA);
    x.s_eAn = reinterpret_cast<float *>(sm + OFF_EAN);
    x.s_ht = reinterpret_cast<float *>(sm + OFF_HT);
    x.s_gamma = reinterpret_cast<float *>(sm + OFF_GAMMA);
    x.Lm = reinterpret_cast<float *>(sm + OFF_L);
    x.Ym = reinterpret_cast<float *>(sm + OFF_Y);
    x.tid = threadIdx.x;
    x.warp = x.tid >> 5;
    x.lane = x.tid & 31;
    x.qw = x.warp & 3;
    x.cg = x.warp >> 2;
    x.ch = 32 * x.qw + x.lane;
    x.lane_base = tmem + ((uint32_t)(32 * x.qw) << 16);
    return x;
}

// Phase A of a chunk: bounded gate, log2-domain cumulative decay and the
// operand tiles.  Thread (warp w, lane l) owns key channels c = 64 (w >> 3) + 2l
// and c + 1 of the eight rows 8h .. 8h + 7, h = w & 7 (the first or second half
// of 16-token tile h / 2): the scan runs in registers, the eight half-tile sums
// per channel are exchanged through shared memory, and every operand row is
// written with 4-byte stores (one 128-byte row segment per warp).  Builds
// [Q^; K^] in place over the q/k tiles, the right factors of the four Gram/P
// tiles, [K~; Q~] and Kend^T, and 2^(G_end).  Waits for the z and q/k tiles
// itself.
//
// UNB: the log-decay g is given directly, unbounded below ("Kimi K3 internals
// analysis", section "Sequence mixing": the prior design's gate), as float32
// in four 32-channel TMA boxes (g_box_off).  The tile factorisation then holds only
// off the diagonal: every factor is formed as one power 2^(e) with e <= 0
// (left 2^(G_t - R_ta), right 2^(R_a2 - G_t) for a2 > ta, Kend 2^(G_end - G_t)),
// the diagonal tiles' right factors are zero, and those tiles are added
// position pair by position pair in the extraction (diag_tiles_kernel).
// Shared-memory offset of g box b (channels 32 b .. 32 b + 31) in the unbounded
// mode: the z region, then the K~ halves of B1, which the intra-chunk kernel
// (KT) does not use, or the V^T tile, which the fused kernel fills only after
// phase A.
template <bool KT>
__device__ __forceinline__ uint32_t g_box_off(int b) {
    return b < 2 ? OFF_Z + 8192u * (uint32_t)b
                 : (KT ? OFF_B1 + 16384u * (uint32_t)(b - 2) : OFF_VT + 8192u * (uint32_t)(b - 2));
}

template <bool KT, bool UNB = false>
__device__ __forceinline__ void phase_gate_operands(const Ctx &x, int nvalid, uint64_t *bar_z,
                                                    uint32_t &z_done, uint64_t *bar_qk,
                                                    uint32_t &qk_done, volatile int *s_abort) {
    uint8_t *sm = x.sm;
    const int lane = x.lane, h = x.warp & 7, kb = x.warp >> 3;
    const int ta = h >> 1;                          // 16-token tile of these rows
    const int c = 64 * kb + 2 * lane;               // first of the two key channels
    const uint32_t cb = (uint32_t)(lane >> 2);      // 16-byte chunk of the channels in a row
    const uint32_t co = (uint32_t)(lane & 3) * 4u;  // byte offset inside that chunk
    float *s_ht = x.s_ht;                           // [8][128] half-tile sums (log2 units)
    const float2 ea = *reinterpret_cast<const float2 *>(x.s_eAn + c);
    if (ptx::mbar_wait(bar_z, z_done & 1, kWaitBudget)) ++z_done; else *s_abort = 1;
    // g = g_min sigmoid(exp(A) z) = g_min / (1 + 2^(-exp(A) z log2 e)), rows past the end 0;
    // inclusive sums over this thread's eight rows
    float g0[8], g1[8];
    {
        const uint8_t *zt = sm + OFF_Z + kb * 8192;
        float run0 = 0.f, run1 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * h + i;
            const bool ok = t < nvalid;
            if (UNB) {
                // channels c, c + 1 sit in box 2 kb + (lane >> 4), columns 2 (lane & 15), + 1
                const uint8_t *gb = sm + g_box_off<KT>(2 * kb + (lane >> 4));
                const float2 gg = *reinterpret_cast<const float2 *>(
                    gb + swz(t, (lane & 15) >> 1) + 8u * (uint32_t)(lane & 1));
                run0 += ok ? fmaxf(gg.x, -100.f) * kLog2e : 0.f;
                run1 += ok ? fmaxf(gg.y, -100.f) * kLog2e : 0.f;
            } else {
                const float2 zz = bf2_to_f2(*reinterpret_cast<const uint32_t *>(zt + swz(t, cb) + co));
                run0 += ok ? kGMin2 * rcp(1.f + ex2(ea.x * zz.x)) : 0.f;
                run1 += ok ? kGMin2 * rcp(1.f + ex2(ea.y * zz.y)) : 0.f;
            }
            g0[i] = run0;
            g1[i] = run1;
        }
        *reinterpret_cast<float2 *>(s_ht + h * 128 + c) = make_float2(run0, run1);
    }
    __syncthreads();
    // R_a (start of tile a), G_end = R_4, and the first half of this tile when h is odd
    float R0[5], R1[5], hp0 = 0.f, hp1 = 0.f;
    {
        float acc0 = 0.f, acc1 = 0.f;
        R0[0] = 0.f;
        R1[0] = 0.f;
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            const float2 v = *reinterpret_cast<const float2 *>(s_ht + hh * 128 + c);
            if (hh + 1 == h && (h & 1)) { hp0 = v.x; hp1 = v.y; }
            acc0 += v.x;
            acc1 += v.y;
            if (hh & 1) { R0[(hh >> 1) + 1] = acc0; R1[(hh >> 1) + 1] = acc1; }
        }
    }
    const float Rt0 = ta == 0 ? 0.f : ta == 1 ? R0[1] : ta == 2 ? R0[2] : R0[3];
    const float Rt1 = ta == 0 ? 0.f : ta == 1 ? R1[1] : ta == 2 ? R1[2] : R1[3];
    if (h == 0) *reinterpret_cast<float2 *>(x.s_gamma + c) = make_float2(ex2(R0[4]), ex2(R1[4]));
    const float rho0 = ex2(Rt0), rho1 = ex2(Rt1);                 // 2^(R_ta)
    const float ke0 = ex2(R0[4] - Rt0), ke1 = ex2(R1[4] - Rt1);   // 2^(G_end - R_ta)
    float f0[4], f1[4];                                           // 2^(R_a2 - R_ta), a2 >= ta
#pragma unroll
    for (int a2 = 0; a2 < 4; ++a2) {
        f0[a2] = a2 > ta ? ex2(R0[a2] - Rt0) : 1.f;
        f1[a2] = a2 > ta ? ex2(R1[a2] - Rt1) : 1.f;
    }
    if (ptx::mbar_wait(bar_qk, qk_done & 1, kWaitBudget)) ++qk_done; else *s_abort = 1;
    uint8_t *qk = sm + OFF_QK + kb * 16384;
    uint8_t *b1 = sm + OFF_B1 + kb * 16384;
    uint8_t *gb = sm + OFF_GB + kb * GB_KBLK;
    float kr0[8], kr1[8];   // Kend^T rows c and c + 1, columns 8h .. 8h + 7
    float kt0[8], kt1[8];   // K~^T rows c and c + 1 (KT only)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = 8 * h + i;
        const bool ok = t < nvalid;
        const uint32_t oq = swz(t, cb) + co, okk = swz(64 + t, cb) + co;
        const float2 qv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qk + oq));
        const float2 kv = bf2_to_f2(*reinterpret_cast<const uint32_t *>(qk + okk));
        const float x0 = hp0 + g0[i], x1 = hp1 + g1[i];   // G_t - R_ta, in (-115.4, 0] when bounded
        const float el0 = ok ? ex2(x0) : 0.f, el1 = ok ? ex2(x1) : 0.f;     // left factors
        const float dd0 = (ok && !UNB) ? ex2(-x0) : 0.f, dd1 = (ok && !UNB) ? ex2(-x1) : 0.f;   // right factors
        const float qe0 = qv.x * el0, qe1 = qv.y * el1, kh0 = kv.x * el0, kh1 = kv.y * el1;
        *reinterpret_cast<uint32_t *>(qk + oq) = pack_bf16(qe0, qe1);        // [Q^; K^] in place
        *reinterpret_cast<uint32_t *>(qk + okk) = pack_bf16(kh0, kh1);
        kt0[i] = kh0 * rho0;
        kt1[i] = kh1 * rho1;
        if (!KT) *reinterpret_cast<uint32_t *>(b1 + oq) = pack_bf16(kt0[i], kt1[i]);   // K~ (KT: as K~^T)
        *reinterpret_cast<uint32_t *>(b1 + okk) = pack_bf16(qe0 * rho0, qe1 * rho1);   // Q~
        if (UNB) {
            // every factor as one power with a non-positive exponent
            kr0[i] = ok ? kv.x * ex2((R0[4] - Rt0) - x0) : 0.f;             // k 2^(G_end - G_t)
            kr1[i] = ok ? kv.y * ex2((R1[4] - Rt1) - x1) : 0.f;
#pragma unroll
            for (int a2 = 0; a2 < 4; ++a2)
                if (a2 >= ta) {
                    const float r0 = (a2 > ta && ok) ? kv.x * ex2((R0[a2] - Rt0) - x0) : 0.f;
                    const float r1 = (a2 > ta && ok) ? kv.y * ex2((R1[a2] - Rt1) - x1) : 0.f;
                    *reinterpret_cast<uint32_t *>(gb + swz(tile_off(a2) + t, cb) + co) = pack_bf16(r0, r1);
                }
        } else {
            const float fr0 = kv.x * dd0, fr1 = kv.y * dd1;                 // k 2^(R_ta - G_t)
            kr0[i] = fr0 * ke0;                                             // k 2^(G_end - G_t)
            kr1[i] = fr1 * ke1;
            // right factors for the Gram/P tiles a2 >= ta: k 2^(R_a2 - G_t)
#pragma unroll
            for (int a2 = 0; a2 < 4; ++a2)
                if (a2 >= ta)
                    *reinterpret_cast<uint32_t *>(gb + swz(tile_off(a2) + t, cb) + co) =
                        pack_bf16(fr0 * f0[a2], fr1 * f1[a2]);
        }
    }
    st_chunk(sm + OFF_KE, swz(c, h), kr0);
    st_chunk(sm + OFF_KE, swz(c + 1, h), kr1);
    if (KT) {
        st_chunk(sm + OFF_KT, swz(c, h), kt0);
        st_chunk(sm + OFF_KT, swz(c + 1, h), kt1);
    }
}

// P (TMEM rows 0..63 of the Gram/P accumulator) and L (rows 64..127), masked
// to the causal pattern: P into its bf16 operand tile, L (times beta) in float32.
// diag (optional): the four diagonal 16 x 16 tiles computed position pair by
// position pair, [L without beta | P][tile][t][s] float32, added where the
// Gram/P MMA left them zero.
__device__ __forceinline__ void phase_extract_PL(const Ctx &x, uint32_t off_pb,
                                                 const float *diag = nullptr) {
    uint8_t *sm = x.sm;
    const int lane = x.lane, qw = x.qw, cg = x.cg;
    const uint32_t lane_base = x.lane_base;
    float *s_beta = x.s_beta;
    float *Lm = x.Lm;
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
        float dg[16];
        if (diag && cg == a) {   // this thread's columns are the row's own tile
            const float4 *src = reinterpret_cast<const float4 *>(diag + ((isL ? 0 : 4) + a) * 256 + (t & 15) * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v4 = src[i];
                dg[4 * i] = v4.x; dg[4 * i + 1] = v4.y; dg[4 * i + 2] = v4.z; dg[4 * i + 3] = v4.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) dg[i] = 0.f;
        }
        float vals[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int s = colbase + i;
            const float d = (have ? ((lane < 16) ? X[i] : Y[i]) : 0.f) + dg[i];
            vals[i] = isL ? ((s < t) ? bt * d : 0.f) : ((s <= t) ? d : 0.f);
        }
        if (isL) {
            float4 *dst = reinterpret_cast<float4 *>(Lm + t * LSTR + colbase);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[i] = make_float4(vals[4 * i], vals[4 * i + 1], vals[4 * i + 2], vals[4 * i + 3]);
        } else {
            st_chunk(sm + off_pb, swz(t, 2 * cg), &vals[0]);
            st_chunk(sm + off_pb, swz(t, 2 * cg + 1), &vals[8]);
        }
    }
}

// Warps 0-3: the four diagonal 16 x 16 blocks of (I + L)^{-1} by forward
// substitution in float32 (one column per lane).
__device__ __forceinline__ void phase_diag(const Ctx &x) {
    const int warp = x.warp, lane = x.lane;
    float *Lm = x.Lm;
    float *Ym = x.Ym;
    if (warp < 4 && lane < 16) {
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
}

// Warps 1-15 (warp 0 issues the MMAs meanwhile): V^T [j][s] from the v tile,
// rows past the sequence end zeroed; a warp transposes one 8-channel chunk, lane
// = rows lane and lane + 32.
__device__ __forceinline__ void phase_vt(const Ctx &x, int nvalid) {
    uint8_t *sm = x.sm;
    const int lane = x.lane;
    for (int cc = x.warp - 1; cc >= 0 && cc < 16; cc += 15) {
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

// ---- off-diagonal blocks of the inverse on warp-level tf32 MMAs -------------
// With D_a = (I + L_aa)^{-1} (the diagonal 16 x 16 blocks, solved before in
// float32), the blocks below the diagonal follow block column by block column,
//   Y_ab = -D_a sum_{m=b}^{a-1} L_am Y_mb,   Y_bb = D_b,
// computed here transposed, Z_ab = Y_ab^T = -(sum_m Z_mb L_am^T) D_a^T, so that
// every product's accumulator is the next product's left operand.  Warp b
// (0-2) walks a = b+1..3 with m16n8k8 tf32 MMAs (float32 accumulation) and
// keeps its column's blocks in registers.  The accumulator holds columns
// 2q, 2q+1 of a k-step where the left operand wants q, q+4, so the reduction
// index of every product is permuted that way (k <-> 2k, k+4 <-> 2k+1 within
// each k-step) and the right operands, read from shared memory, use the same
// order.
__device__ __forceinline__ uint32_t to_tf32(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}
// d += a b for one 16 x 8 x 8 tile.
__device__ __forceinline__ void mma_tf32(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Right operand of k-step ks, n-tile nt, for B[k][n] = M[r0 + 8 nt + n][c0 + k] (a
// transposed 16 x 16 block of a float32 matrix with row stride LSTR), permuted k.
__device__ __forceinline__ void frag_bt(const float *M, int r0, int c0, int nt, int ks, int g,
                                        int q, uint32_t &b0, uint32_t &b1) {
    const float2 v = *reinterpret_cast<const float2 *>(M + (r0 + 8 * nt + g) * LSTR + c0 + 8 * ks + 2 * q);
    b0 = to_tf32(v.x);
    b1 = to_tf32(v.y);
}
// 16 x 16 accumulator (two n-tiles) -> left operand of both k-steps, permuted k.
__device__ __forceinline__ void acc_to_a(const float (*c)[4], uint32_t (*a)[4]) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        a[ks][0] = to_tf32(c[ks][0]);
        a[ks][1] = to_tf32(c[ks][2]);
        a[ks][2] = to_tf32(c[ks][1]);
        a[ks][3] = to_tf32(c[ks][3]);
    }
}
// acc += Z A-operand x (L_{ar} block)^T, for both n-tiles.
__device__ __forceinline__ void mma_zlt(float (*acc)[4], const uint32_t (*za)[4], const float *Lm,
                                        int a, int m, int g, int q) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t b0, b1;
            frag_bt(Lm, 16 * a, 16 * m, nt, ks, g, q, b0, b1);
            mma_tf32(acc[nt], za[ks], b0, b1);
        }
}

// Warps 0-2: T_ab = Y_ab Diag(beta) for the blocks below the diagonal in block
// column b = warp, straight into the bf16 T tile [t][s].
__device__ __forceinline__ void solve_chain(const Ctx &x, uint32_t off_tb) {
    const int lane = x.lane, g = lane >> 2, q = lane & 3;
    const int b = x.warp;
    const float *Lm = x.Lm, *Ym = x.Ym;
    uint32_t za[3][2][4];     // left operands of Z_{b+e, b}, e = 0..2
    float acc[3][2][4];       // sum_m Z_mb L_am^T for a = b+1..b+3
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {   // Z_bb = D_b^T
        const float *p = Ym + (16 * b + 8 * ks + 2 * q) * LSTR + 16 * b + g;
        za[0][ks][0] = to_tf32(p[0]);
        za[0][ks][1] = to_tf32(p[8]);
        za[0][ks][2] = to_tf32(p[LSTR]);
        za[0][ks][3] = to_tf32(p[LSTR + 8]);
    }
#pragma unroll
    for (int d = 0; d < 3; ++d)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[d][nt][i] = 0.f;
#pragma unroll
    for (int d = 1; d <= 3; ++d)
        if (b + d <= 3) mma_zlt(acc[d - 1], za[0], Lm, b + d, b, g, q);
    const float bt0 = x.s_beta[16 * b + g], bt1 = x.s_beta[16 * b + g + 8];
#pragma unroll
    for (int d = 1; d <= 3; ++d) {
        const int a = b + d;
        if (a > 3) break;
        // Z_ab = -acc D_a^T
        uint32_t xa[2][4];
        acc_to_a(acc[d - 1], xa);
        float z[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) z[nt][i] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t b0, b1;
                frag_bt(Ym, 16 * a, 16 * a, nt, ks, g, q, b0, b1);
                mma_tf32(z[nt], xa[ks], b0, b1);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) z[nt][i] = -z[nt][i];
        }
        // T[16a + 8nt + 2q (+1)][16b + g (+8)] = Z[g (+8)][8nt + 2q (+1)] beta
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int t = 16 * a + 8 * nt + 2 * q;
            uint8_t *tb = x.sm + off_tb;
            *reinterpret_cast<__nv_bfloat16 *>(tb + swz(t, 2 * b) + 2 * g) = __float2bfloat16_rn(z[nt][0] * bt0);
            *reinterpret_cast<__nv_bfloat16 *>(tb + swz(t + 1, 2 * b) + 2 * g) = __float2bfloat16_rn(z[nt][1] * bt0);
            *reinterpret_cast<__nv_bfloat16 *>(tb + swz(t, 2 * b + 1) + 2 * g) = __float2bfloat16_rn(z[nt][2] * bt1);
            *reinterpret_cast<__nv_bfloat16 *>(tb + swz(t + 1, 2 * b + 1) + 2 * g) = __float2bfloat16_rn(z[nt][3] * bt1);
        }
        if (d < 3) {
            acc_to_a(z, za[d]);
#pragma unroll
            for (int d2 = d + 1; d2 <= 3; ++d2)
                if (b + d2 <= 3) mma_zlt(acc[d2 - 1], za[d], Lm, b + d2, a, g, q);
        }
    }
}

// Warps 3-4 (one row t each): the diagonal blocks T_aa = D_a Diag(beta) and the
// zero blocks above the diagonal of the bf16 T tile.
__device__ __forceinline__ void solve_diag_T(const Ctx &x, uint32_t off_tb) {
    const int t = x.tid - 3 * 32;
    const int a = t >> 4;
    float yr[16], bt[16];
    const float *src = x.Ym + t * LSTR + 16 * a;
    ld8(src, yr); ld8(src + 8, yr + 8);
    ld8(x.s_beta + 16 * a, bt); ld8(x.s_beta + 16 * a + 8, bt + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) yr[i] *= bt[i];
    st_chunk(x.sm + off_tb, swz(t, 2 * a), yr);
    st_chunk(x.sm + off_tb, swz(t, 2 * a + 1), yr + 8);
    for (int c = 2 * a + 2; c < 8; ++c)
        *reinterpret_cast<uint4 *>(x.sm + off_tb + swz(t, c)) = make_uint4(0u, 0u, 0u, 0u);
}

// Warps 8-15: RHS^T[j][s] = V^T[j][s] - (K~ S0)^T[j][s], 32 columns per thread.
__device__ __forceinline__ void phase_rhs_w8(const Ctx &x, uint32_t tm_ks, uint32_t off_vt,
                                             uint32_t off_ru) {
    const int half = (x.warp >> 2) & 1;
    float KS[32], vt[32];
    ptx::tmem_ld32(x.lane_base + tm_ks + 32 * half, KS);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) ld_chunk(x.sm + off_vt, swz(x.ch, 4 * half + c4), vt + 8 * c4);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) vt[i] -= KS[i];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) st_chunk(x.sm + off_ru, swz(x.ch, 4 * half + c4), vt + 8 * c4);
}

// After the diagonal blocks: T (warps 0-4) and, in the fused kernel, RHS (warps 8-15).
__device__ __forceinline__ void solve_T(const Ctx &x, uint32_t off_tb, bool rhs, uint32_t tm_ks,
                                        uint32_t off_vt, uint32_t off_ru) {
    if (x.warp < 3) solve_chain(x, off_tb);
    else if (x.warp < 5) solve_diag_T(x, off_tb);
    else if (rhs && x.warp >= 8) phase_rhs_w8(x, tm_ks, off_vt, off_ru);
}

// ---- state-pass pieces shared by the fused and the state-only kernels ------

// Start state: float32 master S^T[j][c] into TMEM (the dS accumulator) and its
// bf16 copy into the state operand tile; src == nullptr means zeros.  This
// thread holds c in [32 cg, 32 cg + 32) of row j.
__device__ __forceinline__ void load_state(const Ctx &x, const float *src, uint32_t tm_s,
                                           uint32_t off_st) {
    float Sm[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) Sm[i] = src ? src[(int64_t)(32 * x.cg + i) * D + x.ch] : 0.f;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        st_chunk(x.sm + off_st + (x.cg >> 1) * 16384, swz(x.ch, 4 * (x.cg & 1) + q4), &Sm[8 * q4]);
    ptx::tmem_st32(x.lane_base + tm_s + 32 * x.cg, Sm);
    ptx::tmem_st_wait();
}

// Master state out of TMEM into dst [dk][dv] (row c, column j).
__device__ __forceinline__ void save_state(const Ctx &x, float *dst, uint32_t tm_s) {
    float X[32];
    ptx::tmem_ld32(x.lane_base + tm_s + 32 * x.cg, X);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) dst[(int64_t)(32 * x.cg + i) * D + x.ch] = X[i];
}

// RHS^T[j][s] = V^T[j][s] - (K~ S0)^T[j][s], 16 columns per thread.
__device__ __forceinline__ void phase_rhs(const Ctx &x, uint32_t tm_ks, uint32_t off_vt,
                                          uint32_t off_ru) {
    float KS[16], vt[16];
    ptx::tmem_ld16(x.lane_base + tm_ks + 16 * x.cg, KS);
    ld_chunk(x.sm + off_vt, swz(x.ch, 2 * x.cg), vt);
    ld_chunk(x.sm + off_vt, swz(x.ch, 2 * x.cg + 1), vt + 8);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) vt[i] -= KS[i];
    st_chunk(x.sm + off_ru, swz(x.ch, 2 * x.cg), vt);
    st_chunk(x.sm + off_ru, swz(x.ch, 2 * x.cg + 1), vt + 8);
}

// S^T <- S^T Diag(2^G_end) in TMEM (the dS MMA then accumulates onto it).  It
// touches only the master state, so it can run while an MMA that does not
// write the master (the U product) is in flight.
__device__ __forceinline__ void scale_state_cols(const Ctx &x, uint32_t tm_s, const float *gamma, int cg) {
    float Sx[32], gm[32];
    ptx::tmem_ld32(x.lane_base + tm_s + 32 * cg, Sx);
    const float *g = gamma + 32 * cg;
    ld8(g, gm); ld8(g + 8, gm + 8); ld8(g + 16, gm + 16); ld8(g + 24, gm + 24);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) Sx[i] *= gm[i];
    ptx::tmem_st32(x.lane_base + tm_s + 32 * cg, Sx);
    ptx::tmem_st_wait();
}
__device__ __forceinline__ void scale_state(const Ctx &x, uint32_t tm_s, const float *gamma) {
    scale_state_cols(x, tm_s, gamma, x.cg);
}
// U^T out of TMEM into its bf16 operand tile.
__device__ __forceinline__ void u_out(const Ctx &x, uint32_t tm_u, uint32_t off_ru) {
    float U[16];
    ptx::tmem_ld16(x.lane_base + tm_u + 16 * x.cg, U);
    ptx::tmem_ld_wait();
    st_chunk(x.sm + off_ru, swz(x.ch, 2 * x.cg), U);
    st_chunk(x.sm + off_ru, swz(x.ch, 2 * x.cg + 1), U + 8);
}

// New state's bf16 copy into the state operand tile; O^T out of TMEM into the
// output staging tile (two 64-channel boxes in the TMA 128B-swizzle layout).
__device__ __forceinline__ void phase_state_out(const Ctx &x, uint32_t tm_s, uint32_t tm_o,
                                                uint32_t off_st, uint32_t off_ost) {
    float X[32], O[16];
    ptx::tmem_ld32(x.lane_base + tm_s + 32 * x.cg, X);
    ptx::tmem_ld16(x.lane_base + tm_o + 16 * x.cg, O);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        st_chunk(x.sm + off_st + (x.cg >> 1) * 16384, swz(x.ch, 4 * (x.cg & 1) + q4), &X[8 * q4]);
    const uint32_t obox = off_ost + (x.ch >> 6) * 8192;
    const int jc = (x.ch & 63) >> 3, jin = (x.ch & 7) * 2;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int t = 16 * x.cg + i;
        *reinterpret_cast<__nv_bfloat16 *>(x.sm + obox + swz(t, jc) + jin) = __float2bfloat16_rn(O[i]);
    }
}

// The staged output tile to global memory (after a block barrier): one TMA
// tile store per 64-channel box for a full chunk, plain 16-byte stores of the
// rows < nvalid for the ragged last chunk of a sequence.
__device__ __forceinline__ void store_output(const Ctx &x, const CUtensorMap *tm_o, uint32_t off_ost,
                                             __nv_bfloat16 *out, int64_t row0, int nvalid, int hx,
                                             int64_t rowstride) {
    if (nvalid == C) {
        if (x.tid == 0) {
            ptx::tma_store_2d(tm_o, hx, (int)row0, x.sm + off_ost);
            ptx::tma_store_2d(tm_o, hx + 64, (int)row0, x.sm + off_ost + 8192);
            ptx::bulk_commit();
        }
    } else {
        const int t = x.tid >> 3, part = x.tid & 7;
        if (t < nvalid) {
            __nv_bfloat16 *dst = out + (row0 + t) * rowstride + hx;
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int cc = 2 * part + k2;     // 16-byte chunk of the 256-byte row
                const uint4 v = *reinterpret_cast<const uint4 *>(x.sm + off_ost + (cc >> 3) * 8192 + swz(t, cc & 7));
                *reinterpret_cast<uint4 *>(dst + cc * 8) = v;
            }
        }
    }
}

// Slot of chunk c of sequence seq (first token bos), head h, in the diagonal-tile
// store of the unbounded mode (see diag_tiles_kernel).
__host__ __device__ __forceinline__ int64_t diag_slot(int64_t stride, int h, int64_t bos, int seq, int c) {
    return (int64_t)h * stride + (bos >> 6) + seq + c;
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
    const float *diag;         // unbounded mode: diagonal tiles per chunk (diag_slot)
    int64_t diag_stride;
    int test_expire;           // kExpire* bits (test support), 0 otherwise
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
// The same with an L2 cache policy (the chunk-parallel kernel reads its inputs
// with evict_first, so that the per-chunk records it writes stay in L2).
__device__ __forceinline__ void tma_qk_h(uint8_t *sm, const CUtensorMap *tq, const CUtensorMap *tk,
                                         int hx, int y, uint64_t *bar, uint64_t pol) {
    ptx::mbar_arrive_expect_tx(bar, 32768);
    ptx::tma_load_2d_hint(sm + OFF_QK, tq, hx, y, bar, pol);
    ptx::tma_load_2d_hint(sm + OFF_QK + 8192, tk, hx, y, bar, pol);
    ptx::tma_load_2d_hint(sm + OFF_QK + 16384, tq, hx + 64, y, bar, pol);
    ptx::tma_load_2d_hint(sm + OFF_QK + 24576, tk, hx + 64, y, bar, pol);
}
__device__ __forceinline__ void tma_2box_h(uint8_t *dst, const CUtensorMap *tm, int hx, int y,
                                           uint64_t *bar, uint64_t pol) {
    ptx::mbar_arrive_expect_tx(bar, 16384);
    ptx::tma_load_2d_hint(dst, tm, hx, y, bar, pol);
    ptx::tma_load_2d_hint(dst + 8192, tm, hx + 64, y, bar, pol);
}

// Fused kernel: one CTA per SM, persistent over (sequence, head) chains taken
// longest-first; every chunk runs phases A-D above.  Used when the batch has
// enough chains to fill the GPU.  UNB: the log-decay is given (tm_z maps g as
// float32 32-channel boxes: two in the z region, two in the V^T tile) and the
// diagonal tiles come from diag_tiles_kernel; see phase_gate_operands.
template <bool UNB>
__global__ void __launch_bounds__(NT, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_z,
                  const __grid_constant__ CUtensorMap tm_o, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(sm);
    uint64_t *bar_qk = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_z = bar_qk + 1;
    uint64_t *bar_v = bar_qk + 2;
    uint64_t *bar_g = bar_qk + 3;      // Gram/P MMA done
    uint64_t *bar_s = bar_qk + 4;      // state MMA done
    uint64_t *bar_m = bar_qk + 5;      // U MMA, then output/state MMAs done
    uint64_t *bar_d = bar_qk + 6;      // UNB: the chunk's diagonal tiles staged (behind P)
    uint64_t *bar_never = bar_qk + 7;  // test support: nothing arrives here
    constexpr uint32_t OFF_DG = OFF_OST + 8192;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + OFF_SLOT);
    volatile int *s_work = reinterpret_cast<volatile int *>(sm + OFF_SLOT + 4);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + OFF_SLOT + 8);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = p.H;
    const int64_t rowstride = (int64_t)H * D;

    if (tid == 0) {
        for (int i = 0; i < 8; ++i) ptx::mbar_init(bar_qk + i, 1);
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

    // issue / completion counters of the barriers (uniform across threads);
    // a barrier's next expected phase parity is (done & 1)
    uint32_t qk_issued = 0, qk_done = 0, z_issued = 0, z_done = 0, v_issued = 0, v_done = 0;
    uint32_t g_issued = 0, g_done = 0, s_issued = 0, s_done = 0, m_issued = 0, m_done = 0;
    uint32_t d_issued = 0, d_done = 0;
    const int n_work = p.num_seqs * H;

    for (;;) {
        if (tid == 0) *s_work = (int)atomicAdd(p.counter, 1u);
        __syncthreads();
        const int w = *s_work;
        if (w >= n_work || *s_abort) break;
        const int seq = p.order[w / H];
        const int h = w % H;
        int64_t bos, eos;
        seq_bounds(p.cu_seqlens, seq, p.total_tokens, p.status, tid, bos, eos);
        const int nchunks = (int)((eos - bos + C - 1) / C);
        const int64_t sidx = ((int64_t)seq * H + h) * D * D;
        const int hx = h * D;   // column of this head in the [T, H*D] view

        if (nchunks > 0 && tid == 0) {
            tma_qk(sm, &tm_q, &tm_k, hx, (int)bos, bar_qk);
            if (UNB) {
                ptx::mbar_arrive_expect_tx(bar_z, 32768);
                for (int b = 0; b < 4; ++b)
                    ptx::tma_load_2d(sm + g_box_off<false>(b), &tm_z, hx + 32 * b, (int)bos, bar_z);
            } else {
                tma_2box(sm + OFF_Z, &tm_z, hx, (int)bos, bar_z);
            }
            tma_2box(sm + OFF_V, &tm_v, hx, (int)bos, bar_v);
        }
        if (nchunks > 0) { ++qk_issued; ++z_issued; ++v_issued; }
        load_state(x, p.initial_state ? p.initial_state + sidx : nullptr, TM_D3, OFF_ST);
        if (!UNB && tid < D) x.s_eAn[tid] = -expf(p.A[h * D + tid]) * kLog2e;
        float beta_next = 0.f;
        if (tid < C && bos + tid < eos) beta_next = p.beta[(bos + tid) * H + h];
        __syncthreads();   // s_eAn visible

        for (int cidx = 0; cidx < nchunks; ++cidx) {
            const int64_t row0 = bos + (int64_t)cidx * C;
            const int nvalid = (int)((eos - row0) < C ? (eos - row0) : C);
            const bool has_next = (cidx + 1 < nchunks);
            const int64_t next_row = row0 + C;

            // =============================== phase A: gate, cumulative decay, operands
            if (tid < C) x.s_beta[tid] = beta_next;
            if (cidx == 0 && test_wait_expires(p.test_expire, kExpireFused, bar_never)) *s_abort = 1;
            phase_gate_operands<false, UNB>(x, nvalid, bar_z, z_done, bar_qk, qk_done, s_abort);
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            if (tid == 0) {
                ptx::tc_fence_after_sync();
                ptx::bulk_wait_read();   // the previous output tile has left OST (P goes there next)
                // every thread has read its z rows: prefetch the next chunk's (UNB: the
                // two g boxes of the z region now, the two in V^T once the RHS read it)
                if (has_next) {
                    if (UNB) {
                        ptx::mbar_arrive_expect_tx(bar_z, 32768);
                        for (int b = 0; b < 2; ++b)
                            ptx::tma_load_2d(sm + g_box_off<false>(b), &tm_z, hx + 32 * b, (int)next_row, bar_z);
                    } else {
                        tma_2box(sm + OFF_Z, &tm_z, hx, (int)next_row, bar_z);
                    }
                }
                if (UNB)   // this chunk's diagonal tiles, behind P
                    bulk_load(sm + OFF_DG, reinterpret_cast<const uint8_t *>(
                                  p.diag + diag_slot(p.diag_stride, h, bos, seq, cidx) * 2048),
                              8192, bar_d);
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
            if (UNB) ++d_issued;
            // while the MMAs run: V^T
            if (ptx::mbar_wait(bar_v, v_done & 1, kWaitBudget)) ++v_done; else *s_abort = 1;
            phase_vt(x, nvalid);

            // =============================== phase B: P, L, T, RHS
            if (ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done; else *s_abort = 1;
            if (tid == 0 && has_next) tma_qk(sm, &tm_q, &tm_k, hx, (int)next_row, bar_qk);
            if (has_next) ++qk_issued;
            if (UNB) {
                if (ptx::mbar_wait(bar_d, d_done & 1, kWaitBudget)) ++d_done; else *s_abort = 1;
            }
            ptx::tc_fence_after_sync();
            phase_extract_PL(x, OFF_PB, UNB ? reinterpret_cast<const float *>(sm + OFF_DG) : nullptr);
            __syncthreads();
            // warps 0-3: the diagonal blocks of the inverse; warps 8-15 meanwhile the
            // RHS, once the state MMA (reading B1, where RHS goes) has completed
            if (warp < 4) {
                phase_diag(x);
            } else if (warp >= 8) {
                if (ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done; else *s_abort = 1;
                ptx::tc_fence_after_sync();
                phase_rhs_w8(x, TM_D1, OFF_VT, OFF_RU);
            }
            __syncthreads();
            if (tid == 0 && has_next) tma_2box(sm + OFF_V, &tm_v, hx, (int)next_row, bar_v);
            if (has_next) ++v_issued;
            if (warp < 8) {   // (warps 8-15 have waited already)
                if (ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done; else *s_abort = 1;
            }
            ptx::tc_fence_after_sync();
            solve_T(x, OFF_TB, false, TM_D1, OFF_VT, OFF_RU);
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
                if (UNB && has_next)   // the RHS has read V^T: the next chunk's other two g boxes
                    for (int b = 2; b < 4; ++b)
                        ptx::tma_load_2d(sm + g_box_off<false>(b), &tm_z, hx + 32 * b, (int)next_row, bar_z);
            }
            ++m_issued;
            // (loaded into the register untouched: the load latency hides behind phases C-D)
            if (tid < C && has_next) {
                beta_next = 0.f;
                if (next_row + tid < eos) beta_next = p.beta[(next_row + tid) * H + h];
            }

            // S^T <- S^T Diag(2^G_end) while the U MMA runs (it does not touch the master)
            scale_state(x, TM_D3, x.s_gamma);

            // =============================== phase C: U^T to smem, output and state MMAs
            if (ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            u_out(x, TM_D2, OFF_RU);
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
            phase_state_out(x, TM_D3, TM_D1 + 64, OFF_ST, OFF_OST);
            ptx::fence_async_smem();
            ptx::tc_fence_before_sync();
            __syncthreads();
            if (*s_abort) break;
            store_output(x, &tm_o, OFF_OST, p.out, row0, nvalid, hx, rowstride);
        }
        if (*s_abort) break;
        if (p.final_state) save_state(x, p.final_state + sidx, TM_D3);
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
        while (d_done < d_issued && ptx::mbar_wait(bar_d, d_done & 1, kWaitBudget)) ++d_done;
    }
    if (tid == 0) ptx::bulk_wait_all();   // output stores done before shared memory goes away
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, TM_COLS);
    }
}

// ---- split path for batches with few chains ---------------------------------
// With fewer (sequence, head) chains than about half the SMs, most of the GPU
// would idle while each chain walks its chunks.  The state-independent work of
// every chunk is then done by prefill_intra_kernel, over all chunks of a window
// in parallel: gate, operands, Gram/P, the inverse T, and W = T K~ and
// U~ = T V on the tensor cores; it exports one record per chunk.
// prefill_state_kernel (one CTA per chain) streams the records and runs the
// state-dependent part in two MMA round trips per chunk:
//   [U | Q~S0]^T = [U~ | 0]^T + S0^T [-W; Q~]^T,
//   O^T = (Q~S0)^T + U^T P^T,   S1^T = S0^T Diag(e^{G_end}) + U^T Kend.
// The host runs the state kernel of window k on the caller's stream while the
// intra kernel of window k+1 runs on a side stream (records double-buffered,
// ordered by events only).

// Exported record of one chunk (bf16 operand tiles in their smem layout).
constexpr uint32_t REC_B1 = 0;         // [-W; Q~] 128 x 128
constexpr uint32_t REC_KE = 32768;     // Kend^T [c][s] 128 x 64
constexpr uint32_t REC_PB = 49152;     // P [t][s] 64 x 64
constexpr uint32_t REC_UT = 57344;     // U~^T [j][t] 128 x 64
constexpr uint32_t REC_G = 73728;      // 2^(G_end), 128 float
constexpr uint32_t REC_BYTES = 74240;
constexpr uint32_t OFF_TB_INTRA = OFF_ST;   // the intra kernel keeps T where the state tile would be
constexpr uint32_t OFF_UT_INTRA = OFF_PB;   // U~^T staging: P (exported by then) and the unused 8 KB after it
constexpr uint32_t OFF_NW_INTRA = OFF_VT;   // -W staging (two 64-row K-block halves), over V^T once the MMAs ran
constexpr uint32_t TM_W = 0, TM_UT = 128;   // intra kernel: W [t][c] (N = 128) and U~^T (N = 64)
static_assert(OFF_KT + 16384 <= OFF_MISC, "K~^T tile overlaps");
static_assert(OFF_TB_INTRA + 8192 == OFF_KT, "the W MMA reads 128 rows from the T tile on");
static_assert(OFF_UT_INTRA + 16384 <= OFF_GB && OFF_NW_INTRA + 16384 <= OFF_PB, "staging overlaps");

struct SplitParams {
    const float *A;
    const float *beta;
    const int32_t *cu_seqlens;
    const float *initial_state;
    float *final_state;
    __nv_bfloat16 *out;
    uint8_t *records;          // [chains][W] records of this window
    float *states;             // [chains][128][128] state carried between windows
    uint32_t *status;
    int64_t total_tokens;
    int num_seqs;
    int H;
    int w0;                    // first chunk index of the window
    int wn;                    // chunks in the window
    int W;                     // record slots per chain
    // segment mode (the segment scan): the state and transition kernels run
    // one CTA per (chain, segment), blockIdx = chain * segs + segment
    int segs;                  // segments per chain; <= 1 means window mode
    int seg_len;               // chunks per segment
    uint8_t *seg_out;          // [chains][segs] cells of SEG_CELL bytes: S0 (from a zero state, float32
                               // [c][j]) and M (bf16 tile M[c'][c], the scan's B operand layout)
    float *seg_in;             // [chains][segs][128][128]: the state each segment starts from
    // unbounded log-decay (kda_chunk_prefill_logdecay): the diagonal tiles of
    // every chunk ([L | P][tile][16][16] float32), at diag_slot()
    const float *diag;
    int64_t diag_stride;
    int test_expire;           // kExpire* bits (test support), 0 otherwise
    // segment-map mode (kda_segment_map): every segment's map, the last one's
    // too, as float32 S0 and M per (chain, segment) cell of MAP_CELL bytes;
    // records then sit at the compact slots h rec_stride + (bos >> 6) + seq + c
    uint8_t *map_out;
    int64_t rec_stride;        // 0: records at chain W + (c - w0)
    // the records of the whole call fit in L2: they are written and read with
    // an evict-last policy, and the state pass drops them from L2 after use
    int rec_in_l2;
};


struct ItemInfo {
    int chain, h, c;
    int64_t row0;
    int nvalid;
};

// Work item `it` of a window: chain it / wn, chunk w0 + it % wn; false when
// that chunk lies past the end of its sequence.
__device__ __forceinline__ bool item_info(const SplitParams &p, const int32_t *cu, int it, ItemInfo &r) {
    const int chain = it / p.wn;
    const int c = p.w0 + it % p.wn;
    const int seq = chain / p.H;
    int64_t bos = cu[seq], eos = cu[seq + 1];
    if (bos < 0 || eos < bos || eos > p.total_tokens) return false;
    const int64_t row0 = bos + (int64_t)c * C;
    if (row0 >= eos) return false;
    r.chain = chain;
    r.h = chain % p.H;
    r.c = c;
    r.row0 = row0;
    r.nvalid = (int)((eos - row0) < C ? (eos - row0) : C);
    return true;
}

// ---- diagonal tiles for an unbounded log-decay -------------------------------
// With no bound on g a diagonal 16-token tile cannot be split into bounded left
// and right factors, so its entries are summed position pair by position pair:
//   L'_ts = sum_c k_tc k_sc 2^(G_tc - G_sc),  P_ts = sum_c q_tc k_sc 2^(G_tc - G_sc),
// s <= t in the same tile (L' without beta and only for s < t), with G the
// tile-local inclusive log2 decay, so every power is <= 1.  Rows past the
// sequence end count as zero keys and queries.
//
// Storage: 2048 floats per (head, chunk), at slot h S + (bos >> 6) + seq + c
// for chunk c of sequence seq starting at token bos, S = (T >> 6) + N + 1:
// sequences never share a slot and the slots of a head fit in S.
struct DiagParams {
    const __nv_bfloat16 *q, *k;
    const float *g;
    const int32_t *cu_seqlens;
    int64_t total_tokens;
    int num_seqs;
    int H;
    float *diag;
    int64_t stride;            // S
};
constexpr int DG_P = 129;   // padded row of the staged tiles
constexpr uint32_t SMEM_DIAG = 3 * 64 * DG_P * 4;

// One CTA per slot, persistent over slots; a slot's sequence is the last one
// whose base (bos >> 6) + seq is <= the slot (bases increase), found by all
// threads at once: one load each and a maximum, not a chain of dependent loads.
__global__ void __launch_bounds__(256)
diag_tiles_kernel(const DiagParams p) {
    extern __shared__ float dsm[];
    __shared__ int s_seq;
    float *Kt = dsm, *Qt = dsm + 64 * DG_P, *Gt = dsm + 2 * 64 * DG_P;
    const int tid = threadIdx.x;
    const int64_t n_slots = (int64_t)p.H * p.stride;
    for (int64_t it = blockIdx.x; it < n_slots; it += gridDim.x) {
        const int h = (int)(it / p.stride);
        const int64_t sl = it - (int64_t)h * p.stride;
        __syncthreads();                         // the previous slot's tiles and s_seq are consumed
        if (tid == 0) s_seq = 0;
        __syncthreads();
        int best = 0;
        for (int i = tid; i < p.num_seqs; i += 256)
            if ((int64_t)(p.cu_seqlens[i] >> 6) + i <= sl) best = i;
        best = __reduce_max_sync(0xffffffffu, best);
        if ((tid & 31) == 0 && best > 0) atomicMax(&s_seq, best);
        __syncthreads();
        const int seq = s_seq;
        int64_t bos = p.cu_seqlens[seq], eos = p.cu_seqlens[seq + 1];
        if (bos < 0 || eos < bos || eos > p.total_tokens) continue;   // reported by the main kernel
        const int64_t c = sl - ((bos >> 6) + seq);
        const int64_t nch = (eos - bos + C - 1) / C;
        if (c < 0 || c >= nch) continue;   // uniform over the CTA
        ItemInfo cur;
        cur.h = h;
        cur.row0 = bos + c * C;
        cur.nvalid = (int)((eos - cur.row0) < C ? (eos - cur.row0) : C);
        const int64_t rs = (int64_t)p.H * D;     // row stride of q, k, g
        for (int e = tid; e < 64 * D; e += 256) {
            const int t = e >> 7, cc = e & (D - 1);
            const bool ok = t < cur.nvalid;
            const int64_t gi = (cur.row0 + t) * rs + (int64_t)cur.h * D + cc;
            Kt[t * DG_P + cc] = ok ? __bfloat162float(p.k[gi]) : 0.f;
            Qt[t * DG_P + cc] = ok ? __bfloat162float(p.q[gi]) : 0.f;
            Gt[t * DG_P + cc] = ok ? fmaxf(p.g[gi], -100.f) * kLog2e : 0.f;
        }
        __syncthreads();
        for (int e = tid; e < 4 * D; e += 256) {   // tile-local inclusive sums, per (tile, channel)
            const int a = e >> 7, cc = e & (D - 1);
            float run = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                run += Gt[(16 * a + i) * DG_P + cc];
                Gt[(16 * a + i) * DG_P + cc] = run;
            }
        }
        __syncthreads();
        float *out = p.diag + it * 2048;
        // the 136 pairs s <= t of each tile, numbered r = t (t + 1) / 2 + s, all
        // lanes busy; the diagonal (factor 1) through the same expression
        for (int e = tid; e < 4 * 136; e += 256) {
            const int a = e / 136, r = e - 136 * a;
            int t = (int)((sqrtf(8.f * (float)r + 1.f) - 1.f) * 0.5f);
            while ((t + 1) * (t + 2) / 2 <= r) ++t;
            while (t * (t + 1) / 2 > r) --t;
            const int s_ = r - t * (t + 1) / 2;
            const float *kt = Kt + (16 * a + t) * DG_P, *qt = Qt + (16 * a + t) * DG_P;
            const float *ks = Kt + (16 * a + s_) * DG_P;
            const float *gt = Gt + (16 * a + t) * DG_P, *gs = Gt + (16 * a + s_) * DG_P;
            // four channels per step into independent partial sums (no long
            // dependence chain through one accumulator)
            float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f, p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll 2
            for (int c = 0; c < D; c += 4) {
                const float f0 = ks[c] * ex2(gt[c] - gs[c]);
                const float f1 = ks[c + 1] * ex2(gt[c + 1] - gs[c + 1]);
                const float f2 = ks[c + 2] * ex2(gt[c + 2] - gs[c + 2]);
                const float f3 = ks[c + 3] * ex2(gt[c + 3] - gs[c + 3]);
                l0 += kt[c] * f0; l1 += kt[c + 1] * f1; l2 += kt[c + 2] * f2; l3 += kt[c + 3] * f3;
                p0 += qt[c] * f0; p1 += qt[c + 1] * f1; p2 += qt[c + 2] * f2; p3 += qt[c + 3] * f3;
            }
            const float l = (l0 + l1) + (l2 + l3), pp = (p0 + p1) + (p2 + p3);
            out[a * 256 + t * 16 + s_] = s_ < t ? l : 0.f;
            out[1024 + a * 256 + t * 16 + s_] = pp;
        }
        for (int e = tid; e < 1024; e += 256) {   // the upper triangles
            const int t = (e >> 4) & 15, s_ = e & 15;
            if (s_ > t) { out[e] = 0.f; out[1024 + e] = 0.f; }
        }
    }
}

// W and U~^T out of TMEM into their staging tiles: -W [t][c] as the two 64-row
// K-block halves of the [-W; Q~] operand (lanes t < 64, 32 columns per
// thread), U~^T [j][t] (all lanes, 16 columns per thread).
__device__ __forceinline__ void phase_wu_out(const Ctx &x) {
    if (x.qw < 2) {
        float Wr[32];
        ptx::tmem_ld32(x.lane_base + TM_W + 32 * x.cg, Wr);   // W[t][32 cg + i], t = ch
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) Wr[i] = -Wr[i];
        uint8_t *nw = x.sm + OFF_NW_INTRA + (x.cg >> 1) * 8192;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) st_chunk(nw, swz(x.ch, 4 * (x.cg & 1) + q4), Wr + 8 * q4);
    }
    float Ut[16];
    ptx::tmem_ld16(x.lane_base + TM_UT + 16 * x.cg, Ut);   // U~^T[j][16 cg + i], j = ch
    ptx::tmem_ld_wait();
    st_chunk(x.sm + OFF_UT_INTRA, swz(x.ch, 2 * x.cg), Ut);
    st_chunk(x.sm + OFF_UT_INTRA, swz(x.ch, 2 * x.cg + 1), Ut + 8);
}

// UNB: the log-decay is given (tm_z maps g, float32, in 32-channel boxes) and
// the diagonal tiles come from diag_tiles_kernel; see phase_gate_operands.
template <bool UNB>
__global__ void __launch_bounds__(NT, 1)
prefill_intra_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_z,
                     const SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(sm);
    uint64_t *bar_qk = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_z = bar_qk + 1;
    uint64_t *bar_v = bar_qk + 2;
    uint64_t *bar_g = bar_qk + 3;      // Gram/P MMA, then the W MMA done
    uint64_t *bar_g2 = bar_qk + 5;     // the U~ MMA done (issued by thread 32)
    uint64_t *bar_d = bar_qk + 4;      // UNB: the item's diagonal tiles staged
    uint64_t *bar_never = bar_qk + 7;  // test support: nothing arrives here
    // UNB: the diagonal tiles are staged behind P (free until U~^T is staged)
    constexpr uint32_t OFF_DG = OFF_PB + 8192;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + OFF_SLOT);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + OFF_SLOT + 8);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = p.H;

    if (tid == 0) {
        for (int i = 0; i < 8; ++i) ptx::mbar_init(bar_qk + i, 1);
        ptx::fence_mbar_init();
        *s_abort = 0;
    }
    // the sequence offsets, read once into shared memory when they fit (the
    // next item's bounds are then not a global-memory round trip on every
    // item's critical path); the inputs were complete before the previous
    // kernel of the call started, so this may precede the dependency wait
    int32_t *s_cu = reinterpret_cast<int32_t *>(sm + OFF_CU);
    const bool cu_cached = p.num_seqs < CU_CACHE;
    if (cu_cached)
        for (int i = tid; i <= p.num_seqs; i += NT) s_cu[i] = p.cu_seqlens[i];
    const int32_t *cu = cu_cached ? s_cu : p.cu_seqlens;
    if (warp == 0) {
        ptx::tmem_alloc(s_tmem, 256);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    const Ctx x = make_ctx(sm, tmem);

    uint32_t qk_issued = 0, qk_done = 0, z_issued = 0, z_done = 0, v_issued = 0, v_done = 0;
    uint32_t g_issued = 0, g_done = 0, d_issued = 0, d_done = 0, g2_issued = 0, g2_done = 0;
    // inputs are read once (evict first); the records are read back by the next
    // kernels of the call (evict last), and the last reader discards them
    // (only when the records of the call fit in L2; plain copies otherwise)
    const bool hint = p.rec_in_l2 != 0;
    const uint64_t pol_in = ptx::policy_evict_first(), pol_rec = ptx::policy_evict_last();
    auto load_qk = [&](int hx, int row) {
        if (hint) tma_qk_h(sm, &tm_q, &tm_k, hx, row, bar_qk, pol_in);
        else tma_qk(sm, &tm_q, &tm_k, hx, row, bar_qk);
    };
    auto load_v = [&](int hx, int row) {
        if (hint) tma_2box_h(sm + OFF_V, &tm_v, hx, row, bar_v, pol_in);
        else tma_2box(sm + OFF_V, &tm_v, hx, row, bar_v);
    };
    auto export_rec = [&](uint8_t *gdst, const uint8_t *ssrc, uint32_t bytes) {
        if (hint) bulk_store_hint(gdst, ssrc, bytes, pol_rec);
        else bulk_store(gdst, ssrc, bytes);
    };
    auto load_gz = [&](int hx, int row) {   // z tile, or the four g boxes
        if (UNB) {
            ptx::mbar_arrive_expect_tx(bar_z, 32768);
            for (int b = 0; b < 4; ++b) {
                if (hint) ptx::tma_load_2d_hint(sm + g_box_off<true>(b), &tm_z, hx + 32 * b, row, bar_z, pol_in);
                else ptx::tma_load_2d(sm + g_box_off<true>(b), &tm_z, hx + 32 * b, row, bar_z);
            }
        } else {
            if (hint) tma_2box_h(sm + OFF_Z, &tm_z, hx, row, bar_z, pol_in);
            else tma_2box(sm + OFF_Z, &tm_z, hx, row, bar_z);
        }
    };
    const int n_items = p.num_seqs * H * p.wn;
    ItemInfo cur, nxt;
    int it = blockIdx.x;
    while (it < n_items && !item_info(p, cu, it, cur)) it += gridDim.x;
    // this thread's entry of A and beta for the coming item, raw: loaded one item
    // ahead and not used until that item starts, so the load latency is hidden
    float a_cur = 0.f, beta_cur = 0.f;
    // The inputs were complete before the previous kernel of the call started,
    // so the first item's tiles are fetched before waiting on that kernel;
    // nothing is written to global memory before the wait.
    if (it < n_items) {
        if (!UNB && tid < D) a_cur = p.A[cur.h * D + tid];   // (no gate constants for a given g)
        if (tid < cur.nvalid) beta_cur = p.beta[(cur.row0 + tid) * H + cur.h];
        if (tid == 0) {
            const int hx = cur.h * D;
            load_qk(hx, (int)cur.row0);
            load_gz(hx, (int)cur.row0);
            load_v(hx, (int)cur.row0);
        }
        ++qk_issued; ++z_issued; ++v_issued;
    }
    ptx::pdl_wait();                 // the previous kernel's status word (and, windowed, nothing else)
    ptx::pdl_launch_dependents();
    // bad sequence offsets are reported once, by the first CTA
    if (blockIdx.x == 0 && tid < p.num_seqs) {
        const int64_t b = p.cu_seqlens[tid], e = p.cu_seqlens[tid + 1];
        if (b < 0 || e < b || e > p.total_tokens) report_status(p.status, kDevBadSeqlens);
    }
    bool first_item = true;
    while (it < n_items) {
        int nit = it + gridDim.x;
        while (nit < n_items && !item_info(p, cu, nit, nxt)) nit += gridDim.x;
        const bool has_next = nit < n_items;
        const int nhx = has_next ? nxt.h * D : 0;
        const int nvalid = cur.nvalid;
        const size_t slot = p.rec_stride
            ? (size_t)((int64_t)cur.h * p.rec_stride + ((cur.row0 - (int64_t)cur.c * C) >> 6) + cur.chain / H + cur.c)
            : (size_t)cur.chain * p.W + (cur.c - p.w0);
        uint8_t *rec = p.records + slot * REC_BYTES;

        if (tid < D) x.s_eAn[tid] = -expf(a_cur) * kLog2e;
        if (tid < C) x.s_beta[tid] = beta_cur;
        // every export but the previous item's last group (-W, U~^T) has left smem
        if (tid == 0) ptx::bulk_wait_read_but1();
        __syncthreads();
        // the next item's gate constants and beta, loaded while this one runs
        if (has_next) {
            if (!UNB && tid < D) a_cur = p.A[nxt.h * D + tid];
            beta_cur = 0.f;
            if (tid < nxt.nvalid) beta_cur = p.beta[(nxt.row0 + tid) * H + nxt.h];
        }

        if (first_item && test_wait_expires(p.test_expire, kExpireIntra, bar_never)) *s_abort = 1;
        first_item = false;
        phase_gate_operands<true, UNB>(x, nvalid, bar_z, z_done, bar_qk, qk_done, s_abort);
        if (tid == 0) ptx::bulk_wait_read();   // -W and U~^T staging free for this item
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (*s_abort) break;
        if (tid == 0) {
            ptx::tc_fence_after_sync();
            if (has_next) load_gz(nhx, (int)nxt.row0);
            if (UNB)   // this item's diagonal tiles, into the space behind P
                bulk_load(sm + OFF_DG, reinterpret_cast<const uint8_t *>(
                              p.diag + diag_slot(p.diag_stride, cur.h, cur.row0 - (int64_t)cur.c * C,
                                                 cur.chain / H, cur.c) * 2048),
                          8192, bar_d);
            mma_k<8>(tmem + TM_G, sbase + OFF_QK, 16384u, sbase + OFF_GB, GB_KBLK,
                     ptx::idesc_bf16_f32(128, 160), false);
            ptx::mma_commit(bar_g);
            export_rec(rec + REC_KE, sm + OFF_KE, 16384);
            export_rec(rec + REC_G, reinterpret_cast<const uint8_t *>(x.s_gamma), 512);
            export_rec(rec + REC_B1 + 8192, sm + OFF_B1 + 8192, 8192);                 // Q~, K-block 0
            export_rec(rec + REC_B1 + 16384 + 8192, sm + OFF_B1 + 16384 + 8192, 8192); // Q~, K-block 1
            ptx::bulk_commit();
        }
        ++g_issued;
        if (has_next) ++z_issued;
        if (UNB) ++d_issued;
        if (ptx::mbar_wait(bar_v, v_done & 1, kWaitBudget)) ++v_done; else *s_abort = 1;
        phase_vt(x, nvalid);

        if (ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done; else *s_abort = 1;
        if (tid == 0 && has_next) load_qk(nhx, (int)nxt.row0);
        if (has_next) ++qk_issued;
        if (UNB) {
            if (ptx::mbar_wait(bar_d, d_done & 1, kWaitBudget)) ++d_done; else *s_abort = 1;
        }
        ptx::tc_fence_after_sync();
        phase_extract_PL(x, OFF_PB, UNB ? reinterpret_cast<const float *>(sm + OFF_DG) : nullptr);
        ptx::fence_async_smem();
        __syncthreads();
        phase_diag(x);
        __syncthreads();
        if (tid == 0) {
            if (has_next) load_v(nhx, (int)nxt.row0);
            export_rec(rec + REC_PB, sm + OFF_PB, 8192);
            ptx::bulk_commit();
        }
        if (has_next) ++v_issued;
        solve_T(x, OFF_TB_INTRA, false, 0, 0, 0);
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (*s_abort) break;
        // the two products from two issuing threads (one thread issues a
        // tcgen05.mma only about every 100 cycles)
        if (tid == 0) {
            ptx::tc_fence_after_sync();
            ptx::bulk_wait_read();   // P has left its tile (U~^T staging goes there)
            // W[t][c] = T[t] . K~^T[c] (rows t >= 64 of the left operand run over
            // the next tile and are discarded)
            mma_k<4>(tmem + TM_W, sbase + OFF_TB_INTRA, 0u, sbase + OFF_KT, 0u,
                     ptx::idesc_bf16_f32(128, 128), false);
            ptx::mma_commit(bar_g);
        } else if (tid == 32) {
            ptx::tc_fence_after_sync();
            // U~^T[j][t] = V^T[j] . T[t]
            mma_k<4>(tmem + TM_UT, sbase + OFF_VT, 0u, sbase + OFF_TB_INTRA, 0u,
                     ptx::idesc_bf16_f32(128, 64), false);
            ptx::mma_commit(bar_g2);
        }
        ++g_issued;
        ++g2_issued;
        if (ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done; else *s_abort = 1;
        if (ptx::mbar_wait(bar_g2, g2_done & 1, kWaitBudget)) ++g2_done; else *s_abort = 1;
        ptx::tc_fence_after_sync();
        phase_wu_out(x);
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (*s_abort) break;
        if (tid == 0) {
            export_rec(rec + REC_B1, sm + OFF_NW_INTRA, 8192);                  // -W, K-block 0
            export_rec(rec + REC_B1 + 16384, sm + OFF_NW_INTRA + 8192, 8192);   // -W, K-block 1
            export_rec(rec + REC_UT, sm + OFF_UT_INTRA, 16384);
            ptx::bulk_commit();
        }
        it = nit;
        cur = nxt;
    }

    __syncthreads();
    if (*s_abort) {
        if (tid == 0) report_status(p.status, kDevTimeout);
        while (qk_done < qk_issued && ptx::mbar_wait(bar_qk, qk_done & 1, kWaitBudget)) ++qk_done;
        while (z_done < z_issued && ptx::mbar_wait(bar_z, z_done & 1, kWaitBudget)) ++z_done;
        while (v_done < v_issued && ptx::mbar_wait(bar_v, v_done & 1, kWaitBudget)) ++v_done;
        while (g_done < g_issued && ptx::mbar_wait(bar_g, g_done & 1, kWaitBudget)) ++g_done;
        while (g2_done < g2_issued && ptx::mbar_wait(bar_g2, g2_done & 1, kWaitBudget)) ++g2_done;
        while (d_done < d_issued && ptx::mbar_wait(bar_d, d_done & 1, kWaitBudget)) ++d_done;
    }
    if (tid == 0) ptx::bulk_wait_all();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, 256);
    }
}

// ---- state-only kernel: shared memory map ------------------------------------
constexpr uint32_t SB_STAGE = 74752;            // record stage stride (1024-aligned)
constexpr uint32_t SB_ST = 2 * SB_STAGE;        // S^T bf16 (A of the first MMA)
constexpr uint32_t SB_RU = SB_ST + 32768;       // U^T, then the output tile
constexpr uint32_t SB_BAR = SB_RU + 16384;      // mbarriers and slots
constexpr uint32_t SMEM_STATE = SB_BAR + 128 + 1024;
static_assert(REC_BYTES <= SB_STAGE && SB_STAGE % 1024 == 0, "record stage");
static_assert(SMEM_STATE <= 232448, "shared memory budget");
constexpr uint32_t TS_D1 = 0;     // two buffers of 128 columns: [U^T | (Q~S0 + PU)^T]
constexpr uint32_t TS_D3 = 256;   // float32 master S^T

// [U~^T | 0] of a chunk into a D1 buffer: column groups 0-1 copy U~^T, 2-3 zero.
// Warp 0 is busy issuing MMAs when this runs, so warp 8 (the same TMEM lane
// quarter) also takes its share.
__device__ __forceinline__ void preload_u(const Ctx &x, uint32_t tm_d1, const uint8_t *ut) {
    if (x.warp == 0) return;
    float v[32];
    if (x.warp == 8) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) ld_chunk(ut, swz(x.ch, c4), v + 8 * c4);
        ptx::tmem_st32(x.lane_base + tm_d1, v);
    }
    if (x.cg < 2) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) ld_chunk(ut, swz(x.ch, 4 * x.cg + c4), v + 8 * c4);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
    }
    ptx::tmem_st32(x.lane_base + tm_d1 + 32 * x.cg, v);
    ptx::tmem_st_wait();
}

// SPLIT: each record stage is refetched in two parts, each as soon as its own
// readers are done (the windowed plan, whose records stream from DRAM);
// otherwise whole after its chunk (the segment plans, whose records sit in L2).
template <bool SPLIT>
__global__ void __launch_bounds__(NT, 1)
prefill_state_kernel(const __grid_constant__ CUtensorMap tm_o, const SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(sm);
    // With SPLIT a record stage arrives in two parts: [-W; Q~], U~^T and 2^G_end
    // (read by the first product, the preload and the state scaling) on bar_st,
    // Kend^T and P (read by the state and output products) on bar_kp, so that
    // each part of a stage is refetched as soon as its own readers are done;
    // otherwise the whole record arrives on bar_st
    uint64_t *bar_st = reinterpret_cast<uint64_t *>(sm + SB_BAR);   // [2] per stage
    uint64_t *bar_s = bar_st + 2;
    uint64_t *bar_m = bar_st + 3;      // the state update (thread 0)
    uint64_t *bar_m2 = bar_st + 4;     // the output product (thread 32: one thread issues a
                                       // tcgen05.mma only about every 100 cycles)
    uint64_t *bar_kp = bar_st + 5;     // [2] second parts (Kend^T, P) of the stages
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + SB_BAR + 64);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + SB_BAR + 72);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = p.H;
    // window mode: chain = blockIdx, chunks [w0, w0 + wn), records from chunk w0,
    // state carried in `states`; segment mode: one segment of a chain, records
    // from chunk 0, incoming state from the scan
    int chain, w0, wn, rec_c0;
    const float *carried;
    if (p.segs > 1) {
        chain = blockIdx.x / p.segs;
        const int sg = blockIdx.x % p.segs;
        w0 = sg * p.seg_len;
        wn = p.seg_len;
        rec_c0 = 0;
        carried = p.seg_in + ((size_t)chain * p.segs + sg) * D * D;
    } else {
        chain = blockIdx.x;
        w0 = p.w0;
        wn = p.wn;
        rec_c0 = p.w0;
        carried = p.states + (size_t)chain * D * D;
    }
    const int seq = chain / H, h = chain % H;
    const int hx = h * D;
    const int64_t rowstride = (int64_t)H * D;
    const int64_t sidx = (int64_t)chain * D * D;
    int64_t bos = p.cu_seqlens[seq], eos = p.cu_seqlens[seq + 1];
    if (bos < 0 || eos < bos || eos > p.total_tokens) bos = eos = 0;   // reported by the intra kernel
    const int nchunks = (int)((eos - bos + C - 1) / C);
    const int c_end = (w0 + wn < nchunks) ? w0 + wn : nchunks;
    const bool first = w0 == 0;
    const bool last = w0 + wn >= nchunks;
    if (w0 >= c_end && !(first && nchunks == 0)) return;   // nothing to do here (uniform per CTA)

    uint64_t *bar_never = bar_st + 7;   // test support: nothing arrives here
    if (tid == 0) {
        for (int i = 0; i < 8; ++i) ptx::mbar_init(bar_st + i, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&tm_o);
        *s_abort = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(s_tmem, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    Ctx x = make_ctx(sm, tmem);
    ptx::pdl_wait();                 // records, incoming states of the previous kernels
    ptx::pdl_launch_dependents();
    const uint8_t *recs = p.records + (size_t)chain * p.W * REC_BYTES;
    // this kernel is the last reader of the records: they are fetched with
    // evict_first and, once in shared memory, dropped from L2 without a write-back
    const uint64_t pol_rec = ptx::policy_evict_first();
    // byte ranges of the two parts in a record (and in its stage)
    static_assert(REC_B1 == 0 && REC_KE == 32768 && REC_PB == REC_KE + 16384 && REC_UT == REC_PB + 8192 &&
                  REC_G == REC_UT + 16384 && REC_BYTES == REC_G + 512, "record layout");
    auto copy_part = [&](int k, const uint8_t *r, uint32_t off, uint32_t bytes, uint64_t *bar) {
        if (p.rec_in_l2) bulk_copy_in_hint(sm + k * SB_STAGE + off, r + off, bytes, bar, pol_rec);
        else bulk_copy_in(sm + k * SB_STAGE + off, r + off, bytes, bar);
    };
    auto fetch_first = [&](int k, int c) {   // [-W; Q~], then U~^T and 2^G_end
        const uint8_t *r = recs + (size_t)(c - rec_c0) * REC_BYTES;
        ptx::mbar_arrive_expect_tx(bar_st + k, REC_KE + (REC_BYTES - REC_UT));
        copy_part(k, r, REC_B1, REC_KE, bar_st + k);
        copy_part(k, r, REC_UT, REC_BYTES - REC_UT, bar_st + k);
    };
    auto fetch_second = [&](int k, int c) {   // Kend^T and P
        const uint8_t *r = recs + (size_t)(c - rec_c0) * REC_BYTES;
        ptx::mbar_arrive_expect_tx(bar_kp + k, REC_UT - REC_KE);
        copy_part(k, r, REC_KE, REC_UT - REC_KE, bar_kp + k);
    };
    constexpr bool split_fetch = SPLIT;
    auto fetch_whole = [&](int k, int c) {
        const uint8_t *r = recs + (size_t)(c - rec_c0) * REC_BYTES;
        ptx::mbar_arrive_expect_tx(bar_st + k, REC_BYTES);
        copy_part(k, r, 0, REC_BYTES, bar_st + k);
    };
    // (only once both parts of the record are in shared memory)
    auto discard = [&](int c) {
        if (!p.rec_in_l2) return;
        const uint8_t *r = recs + (size_t)(c - rec_c0) * REC_BYTES;
        for (int i = tid; i < (int)(REC_BYTES / 128); i += NT) ptx::discard_l2(r + (size_t)i * 128);
    };

    uint32_t st_issued[2] = {0, 0}, st_done[2] = {0, 0}, kp_issued[2] = {0, 0}, kp_done[2] = {0, 0};
    uint32_t s_issued = 0, s_done = 0, m_issued = 0, m_done = 0, m2_done = 0;
    const int c0 = w0;
    if (tid == 0) {
        for (int k = 0; k < 2; ++k) {
            if (c0 + k >= c_end) continue;
            if (split_fetch) { fetch_first(k, c0 + k); fetch_second(k, c0 + k); }
            else fetch_whole(k, c0 + k);
        }
    }
    for (int k = 0; k < 2; ++k)
        if (c0 + k < c_end) { ++st_issued[k]; if (split_fetch) ++kp_issued[k]; }
    const float *src = first ? (p.initial_state ? p.initial_state + sidx : nullptr) : carried;
    load_state(x, src, TS_D3, SB_ST);
    if (c0 < c_end) {
        if (ptx::mbar_wait(bar_st, st_done[0] & 1, kWaitBudget)) ++st_done[0]; else *s_abort = 1;
        preload_u(x, TS_D1, sm + REC_UT);
    }
    if (test_wait_expires(p.test_expire, kExpireState, bar_never)) *s_abort = 1;
    ptx::fence_async_smem();
    ptx::tc_fence_before_sync();
    __syncthreads();

    for (int c = c0; c < c_end; ++c) {
        if (*s_abort) break;
        const int k = (c - c0) & 1;
        uint8_t *stg = sm + k * SB_STAGE;
        const uint32_t sstg = sbase + k * SB_STAGE;
        const uint32_t d1 = TS_D1 + 128 * k;
        const int64_t row0 = bos + (int64_t)c * C;
        const int nvalid = (int)((eos - row0) < C ? (eos - row0) : C);
        if (tid == 0) {
            ptx::tc_fence_after_sync();
            // D1 = [U~ | 0]^T + S^T [-W; Q~]^T
            mma_k<8>(tmem + d1, sbase + SB_ST, 16384u, sstg + REC_B1, 16384u,
                     ptx::idesc_bf16_f32(128, 128), true);
            ptx::mma_commit(bar_s);
            ptx::bulk_wait_read();   // the previous output tile has left RU
        }
        ++s_issued;
        // the master state is not touched by that MMA: scale it meanwhile.  Warp 0
        // is issuing, so warp 8 (the same TMEM lane quarter) scales its columns
        // too; the block barrier after the scaling orders the previous output
        // tile's read of RU before U is written there
        ptx::tc_fence_after_sync();
        {
            const float *gamma = reinterpret_cast<const float *>(stg + REC_G);
            if (warp != 0) scale_state(x, TS_D3, gamma);
            if (warp == 8) scale_state_cols(x, TS_D3, gamma, 0);
        }
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done; else *s_abort = 1;
        ptx::tc_fence_after_sync();
        u_out(x, d1, SB_RU);
        // this record's second part, fetched two chunks ago
        if (split_fetch) {
            if (ptx::mbar_wait(bar_kp + k, kp_done[k] & 1, kWaitBudget)) ++kp_done[k]; else *s_abort = 1;
        }
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (*s_abort) break;
        if (tid == 0) {
            ptx::tc_fence_after_sync();
            // S^T += U^T Kend
            mma_k<4>(tmem + TS_D3, sbase + SB_RU, 0u, sstg + REC_KE, 0u, ptx::idesc_bf16_f32(128, 128), true);
            ptx::mma_commit(bar_m);
        } else if (tid == 32) {
            ptx::tc_fence_after_sync();
            // O^T += U^T P^T
            mma_k<4>(tmem + d1 + 64, sbase + SB_RU, 0u, sstg + REC_PB, 0u, ptx::idesc_bf16_f32(128, 64), true);
            ptx::mma_commit(bar_m2);
        }
        ++m_issued;
        // the first part of stage k has been read (the first product, the scaling,
        // the preload a chunk ago): the record two chunks ahead goes there now, from
        // thread 0, whose warp has no share of the preload
        if (split_fetch && c + 2 < c_end) {
            if (tid == 0) fetch_first(k, c + 2);
            ++st_issued[k];
        }
        discard(c);   // both parts of this record are in shared memory: its L2 lines go
        // meanwhile: the next chunk's [U~ | 0] into the other D1 buffer
        if (c + 1 < c_end) {
            if (ptx::mbar_wait(bar_st + (k ^ 1), st_done[k ^ 1] & 1, kWaitBudget)) ++st_done[k ^ 1];
            else *s_abort = 1;
            preload_u(x, TS_D1 + 128 * (k ^ 1), sm + (k ^ 1) * SB_STAGE + REC_UT);
        }
        if (ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done; else *s_abort = 1;
        if (ptx::mbar_wait(bar_m2, m2_done & 1, kWaitBudget)) ++m2_done; else *s_abort = 1;
        // the second part of stage k has been read by those products
        if (split_fetch && c + 2 < c_end) {
            if (tid == 0) fetch_second(k, c + 2);
            ++kp_issued[k];
        }
        ptx::tc_fence_after_sync();
        phase_state_out(x, TS_D3, d1 + 64, SB_ST, SB_RU);
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (*s_abort) break;
        store_output(x, &tm_o, SB_RU, p.out, row0, nvalid, hx, rowstride);
        if (!split_fetch && c + 2 < c_end) {   // stage k has been consumed
            if (tid == 0) fetch_whole(k, c + 2);
            ++st_issued[k];
        }
    }
    if (!*s_abort) {
        if (last) {
            if (p.final_state) save_state(x, p.final_state + sidx, TS_D3);
        } else if (p.segs <= 1) {
            save_state(x, p.states + sidx, TS_D3);
        }
    }
    __syncthreads();
    if (*s_abort) {
        if (tid == 0) report_status(p.status, kDevTimeout);
        for (int k = 0; k < 2; ++k) {
            while (st_done[k] < st_issued[k] && ptx::mbar_wait(bar_st + k, st_done[k] & 1, kWaitBudget)) ++st_done[k];
            while (kp_done[k] < kp_issued[k] && ptx::mbar_wait(bar_kp + k, kp_done[k] & 1, kWaitBudget)) ++kp_done[k];
        }
        while (s_done < s_issued && ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done;
        while (m_done < m_issued && ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done;
        while (m2_done < m_issued && ptx::mbar_wait(bar_m2, m2_done & 1, kWaitBudget)) ++m2_done;
    }
    if (tid == 0) ptx::bulk_wait_all();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ---- segment scan for few chains with many chunks ----------------------------
// The pages' context-parallel form of the state pass ("Kimi K3 internals
// analysis", section on infrastructure for the 3T-class MoE: KDA context
// parallelism by an affine prefix scan over segments), here across the SMs of
// one GPU.  Over a segment of chunks the state map is affine,
//   S_out = M S_in + S0,   M = prod_chunks (Diag(e^{G_end}) - Kend^T W),
// where S0 is the segment run from a zero state.  Pass 1 (prefill_seg_kernel)
// runs every segment from S0 = 0 and M = I in parallel, propagating M as a
// second state with U~ = 0; prefill_scan_kernel composes the segments of a
// chain in order; pass 2 is prefill_state_kernel in segment mode, every segment
// again in parallel from its incoming state, writing the outputs.

// pass 1: record pieces it needs per chunk (-W, Kend^T, U~^T, 2^G_end)
constexpr uint32_t SG_NW = 0;          // -W, two 64-row K-block halves
constexpr uint32_t SG_KE = 16384;
constexpr uint32_t SG_UT = 32768;
constexpr uint32_t SG_G = 49152;
constexpr uint32_t SG_REC = 49664;     // bytes per stage
constexpr uint32_t SG_STAGE = 50176;
constexpr uint32_t SG_ST = 2 * SG_STAGE;       // S0^T bf16
constexpr uint32_t SG_MT = SG_ST + 32768;      // M^T bf16
constexpr uint32_t SG_RU = SG_MT + 32768;      // U^T bf16 of S0
constexpr uint32_t SG_RUM = SG_RU + 16384;     // U^T bf16 of M
constexpr uint32_t SG_BAR = SG_RUM + 16384;
constexpr uint32_t SMEM_SEG = SG_BAR + 128 + 1024;
static_assert(SG_REC <= SG_STAGE && SMEM_SEG <= 232448, "segment kernel shared memory");
constexpr uint32_t TG_S = 0, TG_M = 128, TG_U = 256, TG_UM = 320;   // TMEM columns
constexpr size_t SEG_S0 = 0, SEG_MT = 65536, SEG_CELL = 98304;       // bytes per (chain, segment)
constexpr size_t MAP_CELL = 2 * 65536;   // segment-map mode: float32 S0, then float32 M

// M (held transposed in TMEM, lane m, column c -> M[c][m]) as the bf16 tile
// B[c'][k] = M[c'][k] of the scan's MMA, written to global memory.
__device__ __forceinline__ void save_m_tile(const Ctx &x, uint8_t *dst, uint32_t tm_m) {
    float X[32];
    ptx::tmem_ld32(x.lane_base + tm_m + 32 * x.cg, X);
    ptx::tmem_ld_wait();
    const int m = x.ch;
    uint8_t *kb = dst + (m >> 6) * 16384;
    const uint32_t mc = (uint32_t)((m & 63) >> 3), mo = (uint32_t)(m & 7) * 2u;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        *reinterpret_cast<__nv_bfloat16 *>(kb + swz(32 * x.cg + i, mc) + mo) = __float2bfloat16_rn(X[i]);
}

// (the records are read again by the state pass: when they fit, their lines
// are kept in L2)
__device__ __forceinline__ void load_stage_seg(uint8_t *stg, const uint8_t *rec, uint64_t *bar, bool keep) {
    ptx::mbar_arrive_expect_tx(bar, SG_REC);
    const uint32_t dst[5] = {SG_NW, SG_NW + 8192, SG_KE, SG_UT, SG_G};
    const uint32_t src[5] = {REC_B1, REC_B1 + 16384, REC_KE, REC_UT, REC_G};
    const uint32_t len[5] = {8192, 8192, 16384, 16384, 512};
    const uint64_t pol = ptx::policy_evict_last();
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        if (keep) bulk_copy_in_hint(stg + dst[i], rec + src[i], len[i], bar, pol);
        else bulk_copy_in(stg + dst[i], rec + src[i], len[i], bar);
    }
}

// The identity as a transposed state: TMEM float32 and its bf16 operand copy.
__device__ __forceinline__ void load_identity(const Ctx &x, uint32_t tm_s, uint32_t off_st) {
    float Sm[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) Sm[i] = (32 * x.cg + i == x.ch) ? 1.f : 0.f;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        st_chunk(x.sm + off_st + (x.cg >> 1) * 16384, swz(x.ch, 4 * (x.cg & 1) + q4), &Sm[8 * q4]);
    ptx::tmem_st32(x.lane_base + tm_s + 32 * x.cg, Sm);
    ptx::tmem_st_wait();
}

// Warps 8-15: U~^T (64 columns) of a chunk into TMEM.
__device__ __forceinline__ void preload_u64(const Ctx &x, uint32_t tm_u, const uint8_t *ut) {
    if (x.warp < 8) return;
    const int half = (x.warp >> 2) & 1;
    float v[32];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) ld_chunk(ut, swz(x.ch, 4 * half + c4), v + 8 * c4);
    ptx::tmem_st32(x.lane_base + tm_u + 32 * half, v);
    ptx::tmem_st_wait();
}

// bf16 operand copy of a transposed state held in TMEM.
__device__ __forceinline__ void state_to_bf16(const Ctx &x, uint32_t tm_s, uint32_t off_st) {
    float X[32];
    ptx::tmem_ld32(x.lane_base + tm_s + 32 * x.cg, X);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
        st_chunk(x.sm + off_st + (x.cg >> 1) * 16384, swz(x.ch, 4 * (x.cg & 1) + q4), &X[8 * q4]);
}

__global__ void __launch_bounds__(NT, 1)
prefill_seg_kernel(const SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(sm);
    uint64_t *bar_st = reinterpret_cast<uint64_t *>(sm + SG_BAR);   // [2] stages
    // the S0 chain's products are issued by thread 0, the M chain's by thread
    // 32 (two issuing threads keep the tensor core about twice as busy)
    uint64_t *bar_s = bar_st + 2;      // U products (thread 0: S0)
    uint64_t *bar_m = bar_st + 3;      // state products (thread 0: S0)
    uint64_t *bar_s2 = bar_st + 4;     // U product (thread 32: M)
    uint64_t *bar_m2 = bar_st + 5;     // state product (thread 32: M)
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + SG_BAR + 64);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + SG_BAR + 72);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int chain = blockIdx.x / p.segs, sg = blockIdx.x % p.segs;
    const int seq = chain / p.H;
    int64_t bos = p.cu_seqlens[seq], eos = p.cu_seqlens[seq + 1];
    if (bos < 0 || eos < bos || eos > p.total_tokens) bos = eos = 0;   // reported by the intra kernel
    const int nchunks = (int)((eos - bos + C - 1) / C);
    const int c0 = sg * p.seg_len;
    const int c_end = (c0 + p.seg_len < nchunks) ? c0 + p.seg_len : nchunks;
    // empty, or the last segment of the scan plan (nobody needs its map there)
    if (c0 >= c_end || (c_end >= nchunks && !p.map_out)) return;

    uint64_t *bar_never = bar_st + 7;   // test support: nothing arrives here
    if (tid == 0) {
        for (int i = 0; i < 8; ++i) ptx::mbar_init(bar_st + i, 1);
        ptx::fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        ptx::tmem_alloc(s_tmem, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    const Ctx x = make_ctx(sm, tmem);
    ptx::pdl_wait();                 // the intra kernel's records
    ptx::pdl_launch_dependents();
    const size_t rec0 = p.rec_stride
        ? (size_t)((int64_t)(chain % p.H) * p.rec_stride + (bos >> 6) + seq)
        : (size_t)chain * p.W;
    const uint8_t *recs = p.records + rec0 * REC_BYTES;

    uint32_t st_issued[2] = {0, 0}, st_done[2] = {0, 0};
    uint32_t s_issued = 0, s_done = 0, m_issued = 0, m_done = 0;
    uint32_t s2_done = 0, m2_done = 0;   // (issued with s, m)
    if (tid == 0) {
        for (int k = 0; k < 2; ++k)
            if (c0 + k < c_end) load_stage_seg(sm + k * SG_STAGE, recs + (size_t)(c0 + k) * REC_BYTES, bar_st + k, p.rec_in_l2);
    }
    for (int k = 0; k < 2; ++k)
        if (c0 + k < c_end) ++st_issued[k];
    load_state(x, nullptr, TG_S, SG_ST);    // S0 = 0
    load_identity(x, TG_M, SG_MT);          // M = I
    if (ptx::mbar_wait(bar_st, st_done[0] & 1, kWaitBudget)) ++st_done[0]; else *s_abort = 1;
    preload_u64(x, TG_U, sm + SG_UT);
    if (test_wait_expires(p.test_expire, kExpireSeg, bar_never)) *s_abort = 1;
    ptx::fence_async_smem();
    ptx::tc_fence_before_sync();
    __syncthreads();

    for (int c = c0; c < c_end; ++c) {
        if (*s_abort) break;
        const int k = (c - c0) & 1;
        uint8_t *stg = sm + k * SG_STAGE;
        const uint32_t sstg = sbase + k * SG_STAGE;
        if (tid == 0) {
            ptx::tc_fence_after_sync();
            // U^T = U~^T + S0^T (-W)^T
            mma_k<8>(tmem + TG_U, sbase + SG_ST, 16384u, sstg + SG_NW, 8192u,
                     ptx::idesc_bf16_f32(128, 64), true);
            ptx::mma_commit(bar_s);
        } else if (tid == 32) {
            ptx::tc_fence_after_sync();
            // U_M^T = M^T (-W)^T
            mma_k<8>(tmem + TG_UM, sbase + SG_MT, 16384u, sstg + SG_NW, 8192u,
                     ptx::idesc_bf16_f32(128, 64), false);
            ptx::mma_commit(bar_s2);
        }
        ++s_issued;
        // the two master states are not touched by those MMAs: scale them meanwhile.
        // Warps 0 and 1 are issuing, so warps 8 and 12 (lane quarter 0) and 9 and
        // 13 (quarter 1) scale their columns of S0 and of M as well
        const float *gamma = reinterpret_cast<const float *>(stg + SG_G);
        ptx::tc_fence_after_sync();
        if (warp >= 2) {
            scale_state(x, TG_S, gamma);
            scale_state(x, TG_M, gamma);
        }
        if (warp == 8 || warp == 9) scale_state_cols(x, TG_S, gamma, 0);
        if (warp == 12 || warp == 13) scale_state_cols(x, TG_M, gamma, 0);
        if (ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done; else *s_abort = 1;
        if (ptx::mbar_wait(bar_s2, s2_done & 1, kWaitBudget)) ++s2_done; else *s_abort = 1;
        ptx::tc_fence_after_sync();
        u_out(x, TG_U, SG_RU);
        u_out(x, TG_UM, SG_RUM);
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (*s_abort) break;
        if (tid == 0) {
            ptx::tc_fence_after_sync();
            // S0^T += U^T Kend
            mma_k<4>(tmem + TG_S, sbase + SG_RU, 0u, sstg + SG_KE, 0u, ptx::idesc_bf16_f32(128, 128), true);
            ptx::mma_commit(bar_m);
        } else if (tid == 32) {
            ptx::tc_fence_after_sync();
            // M^T += U_M^T Kend
            mma_k<4>(tmem + TG_M, sbase + SG_RUM, 0u, sstg + SG_KE, 0u, ptx::idesc_bf16_f32(128, 128), true);
            ptx::mma_commit(bar_m2);
        }
        ++m_issued;
        if (c + 1 < c_end) {   // meanwhile: the next chunk's U~^T
            if (ptx::mbar_wait(bar_st + (k ^ 1), st_done[k ^ 1] & 1, kWaitBudget)) ++st_done[k ^ 1];
            else *s_abort = 1;
            preload_u64(x, TG_U, sm + (k ^ 1) * SG_STAGE + SG_UT);
        }
        if (ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done; else *s_abort = 1;
        if (ptx::mbar_wait(bar_m2, m2_done & 1, kWaitBudget)) ++m2_done; else *s_abort = 1;
        ptx::tc_fence_after_sync();
        state_to_bf16(x, TG_S, SG_ST);
        state_to_bf16(x, TG_M, SG_MT);
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();
        if (*s_abort) break;
        if (tid == 0 && c + 2 < c_end)
            load_stage_seg(stg, recs + (size_t)(c + 2) * REC_BYTES, bar_st + k, p.rec_in_l2);
        if (c + 2 < c_end) ++st_issued[k];
    }
    if (!*s_abort) {
        if (p.map_out) {   // float32 S0 [c][j] and M [c][c']
            uint8_t *cell = p.map_out + ((size_t)chain * p.segs + sg) * MAP_CELL;
            save_state(x, reinterpret_cast<float *>(cell), TG_S);
            save_state(x, reinterpret_cast<float *>(cell + MAP_CELL / 2), TG_M);
        } else {
            uint8_t *cell = p.seg_out + ((size_t)chain * p.segs + sg) * SEG_CELL;
            save_state(x, reinterpret_cast<float *>(cell + SEG_S0), TG_S);
            save_m_tile(x, cell + SEG_MT, TG_M);
        }
    }
    __syncthreads();
    if (*s_abort) {
        if (tid == 0) report_status(p.status, kDevTimeout);
        for (int k = 0; k < 2; ++k)
            while (st_done[k] < st_issued[k] && ptx::mbar_wait(bar_st + k, st_done[k] & 1, kWaitBudget)) ++st_done[k];
        while (s_done < s_issued && ptx::mbar_wait(bar_s, s_done & 1, kWaitBudget)) ++s_done;
        while (s2_done < s_issued && ptx::mbar_wait(bar_s2, s2_done & 1, kWaitBudget)) ++s2_done;
        while (m_done < m_issued && ptx::mbar_wait(bar_m, m_done & 1, kWaitBudget)) ++m_done;
        while (m2_done < m_issued && ptx::mbar_wait(bar_m2, m2_done & 1, kWaitBudget)) ++m2_done;
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// The scan: per chain, S_in(g + 1) = M_g S_in(g) + S0_g for the segments g
// before the last non-empty one.  The value channels (columns j of S) do not
// mix, so each chain is split over SCAN_SPLIT CTAs of SCAN_JB columns: one CTA
// keeps S_in[:, j0 .. j0 + 31] and runs, per segment, one M = 128, N = 32 MMA
//   D[c][j] = S0_g[c][j] + sum_c' M_g[c][c'] S_in(g)[c'][j]
// (A = M_g as written by the segment kernel, B = the bf16 block S_in^T[j][c']).
// Thread c owns row c (TMEM lane c).  The 128 x 32 float32 blocks of S0 (two
// segments ahead) and of S_in move as single TMA tiles (128-byte swizzle), so
// only the MMA and the bf16 copy of its result are on the chain of a step.
constexpr int SCAN_JB = 32, SCAN_SPLIT = D / SCAN_JB, SCAN_NT = 128;
constexpr uint32_t SCAN_BLK = 128 * SCAN_JB * 4;     // bytes of one float32 block
constexpr int SEG_CELL_ROWS = (int)(SEG_CELL / (D * 4));   // 512-byte rows per (chain, segment) cell
constexpr uint32_t SC_MB = 0, SC_SB = 65536;         // M tiles: two buffers of 32 KB; B tile 8 KB
constexpr uint32_t SC_S0 = SC_SB + 8192;             // two S0 blocks
constexpr uint32_t SC_OUT = SC_S0 + 2 * SCAN_BLK;    // S_in block going out (and the start's transpose)
constexpr uint32_t SC_BAR = SC_OUT + SCAN_BLK;
constexpr uint32_t SMEM_SCAN = SC_BAR + 64 + 1024;
static_assert(SC_S0 % 1024 == 0 && SC_OUT % 1024 == 0 && SEG_CELL % (D * 4) == 0, "scan layout");

// Byte offset of element (row r, column j) of a 128 x 32 float32 block in the
// 128-byte-swizzled TMA layout.
__device__ __forceinline__ uint32_t scan_off(int r, int j) {
    return swz(r, j >> 2) + (uint32_t)(j & 3) * 4u;
}

// This thread's row c of an f32 [c][j] state block into the bf16 B tile S^T[j][c]
// (32 rows j, K = c in two 64-element blocks of 4 KB).
__device__ __forceinline__ void scan_block_to_bf16(uint8_t *tile, int c, const float *X) {
    uint8_t *kb = tile + (c >> 6) * 4096;
    const uint32_t cc = (uint32_t)((c & 63) >> 3), co = (uint32_t)(c & 7) * 2u;
#pragma unroll
    for (int j = 0; j < SCAN_JB; ++j)
        *reinterpret_cast<__nv_bfloat16 *>(kb + swz(j, cc) + co) = __float2bfloat16_rn(X[j]);
}

__global__ void __launch_bounds__(SCAN_NT, 1)
prefill_scan_kernel(const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_sin,
                    const SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(sm);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + SC_BAR);   // MMA done
    uint64_t *bar_mb = bar + 1;                                  // [2] M tile arrived
    uint64_t *bar_s0 = bar + 3;                                  // [2] S0 block arrived
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + SC_BAR + 48);
    volatile int *s_abort = reinterpret_cast<volatile int *>(sm + SC_BAR + 56);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chain = blockIdx.x / SCAN_SPLIT, j0 = (blockIdx.x % SCAN_SPLIT) * SCAN_JB;
    const int seq = chain / p.H;
    int64_t bos = p.cu_seqlens[seq], eos = p.cu_seqlens[seq + 1];
    if (bos < 0 || eos < bos || eos > p.total_tokens) bos = eos = 0;
    const int nchunks = (int)((eos - bos + C - 1) / C);
    const int nseg = (nchunks + p.seg_len - 1) / p.seg_len;
    if (nseg <= 1) return;   // only the first segment runs, from the initial state

    uint64_t *bar_never = bar + 5;                               // test support: nothing arrives here
    if (tid == 0) {
        for (int i = 0; i < 6; ++i) ptx::mbar_init(bar + i, 1);
        ptx::fence_mbar_init();
        *s_abort = 0;
        ptx::prefetch_tensormap(&tm_s0);
        ptx::prefetch_tensormap(&tm_sin);
    }
    if (warp == 0) {
        ptx::tmem_alloc(s_tmem, 2 * SCAN_JB);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    const int c = tid;               // row of S (TMEM lane)
    ptx::pdl_wait();                 // the segment maps
    ptx::pdl_launch_dependents();
    const int cell0 = chain * p.segs;   // this chain's first (chain, segment) cell
    const uint8_t *cells = p.seg_out + (size_t)cell0 * SEG_CELL;
    uint32_t issued = 0, done = 0, mb_issued[2] = {0, 0}, mb_done[2] = {0, 0};
    uint32_t s0_issued[2] = {0, 0}, s0_done[2] = {0, 0};
    auto issue_s0 = [&](int g, int b) {   // S0_g block into staging buffer b
        if (tid == 0) {
            ptx::mbar_arrive_expect_tx(bar_s0 + b, SCAN_BLK);
            ptx::tma_load_2d(sm + SC_S0 + b * SCAN_BLK, &tm_s0, j0, (cell0 + g) * SEG_CELL_ROWS, bar_s0 + b);
        }
        ++s0_issued[b];
    };
    auto read_row = [&](uint32_t off, float (&Y)[SCAN_JB]) {   // row c of a swizzled block
#pragma unroll
        for (int i = 0; i < SCAN_JB / 4; ++i) {
            const float4 v = *reinterpret_cast<const float4 *>(sm + off + swz(c, i));
            Y[4 * i] = v.x; Y[4 * i + 1] = v.y; Y[4 * i + 2] = v.z; Y[4 * i + 3] = v.w;
        }
    };
    auto save = [&](int g, uint32_t buf, float (&Y)[SCAN_JB]) {   // S_in(g) block out of TMEM buffer buf
        ptx::tmem_ld32(lane_base + buf, Y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < SCAN_JB / 4; ++i)
            *reinterpret_cast<float4 *>(sm + SC_OUT + swz(c, i)) =
                make_float4(Y[4 * i], Y[4 * i + 1], Y[4 * i + 2], Y[4 * i + 3]);
        ptx::fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            ptx::tma_store_2d(&tm_sin, j0, (cell0 + g) * D, sm + SC_OUT);
            ptx::bulk_commit();
        }
    };
    if (tid == 0) {
        for (int k = 0; k < 2 && k + 1 < nseg; ++k)
            bulk_load(sm + SC_MB + k * 32768, cells + (size_t)k * SEG_CELL + SEG_MT, 32768, bar_mb + k);
    }
    for (int k = 0; k < 2 && k + 1 < nseg; ++k) ++mb_issued[k];
    for (int k = 0; k < 2 && k + 1 < nseg; ++k) issue_s0(k, k);
    float X[SCAN_JB];
    {   // S_in(0): the initial state (or zeros) as the first B operand; warp w loads
        // rows 32w .. 32w + 31 a row per instruction, turned through the out tile
        const float *src = p.initial_state ? p.initial_state + (int64_t)chain * D * D +
                                                 (int64_t)(32 * warp) * D + j0 + lane
                                           : nullptr;
#pragma unroll
        for (int i = 0; i < SCAN_JB; ++i) X[i] = src ? src[(int64_t)i * D] : 0.f;   // all loads in flight at once
#pragma unroll
        for (int i = 0; i < SCAN_JB; ++i) *reinterpret_cast<float *>(sm + SC_OUT + scan_off(32 * warp + i, lane)) = X[i];
        __syncwarp();
        read_row(SC_OUT, X);
        scan_block_to_bf16(sm + SC_SB, c, X);
    }
    if (ptx::mbar_wait(bar_s0, s0_done[0] & 1, kWaitBudget)) ++s0_done[0]; else *s_abort = 1;
    read_row(SC_S0, X);
    ptx::tmem_st32(lane_base, X);   // accumulator 0 = S0_0 block
    ptx::tmem_st_wait();
    if (test_wait_expires(p.test_expire, kExpireScan, bar_never)) *s_abort = 1;
    // Step g accumulates S_in(g + 1) in TMEM buffer g & 1 (32 columns each);
    // writing S_in(g) out and staging S0_(g+1) into the other buffer overlap it.
    for (int g = 0; g + 1 < nseg; ++g) {
        const int k = g & 1;
        const uint32_t dk = (uint32_t)(SCAN_JB * k), dn = (uint32_t)(SCAN_JB * (k ^ 1));
        if (tid == 0) ptx::bulk_wait_read();   // the last S_in block has left the out tile
        ptx::fence_async_smem();
        ptx::tc_fence_before_sync();
        __syncthreads();   // also: S0 block k has been read by every thread
        if (*s_abort) break;
        if (tid == 0) {
            if (ptx::mbar_wait(bar_mb + k, mb_done[k] & 1, kWaitBudget)) ++mb_done[k]; else *s_abort = 1;
            ptx::tc_fence_after_sync();
            mma_k<8>(tmem + dk, sbase + SC_MB + k * 32768, 16384u, sbase + SC_SB, 4096u,
                     ptx::idesc_bf16_f32(128, SCAN_JB), true);
            ptx::mma_commit(bar);
        }
        ++issued;
        if (g + 2 < nseg - 1) issue_s0(g + 2, k);
        ptx::tc_fence_after_sync();
        if (g >= 1) save(g, dn, X);   // S_in(g), from the last step
        if (g + 2 < nseg) {           // the other buffer = S0_(g+1) block
            if (ptx::mbar_wait(bar_s0 + (k ^ 1), s0_done[k ^ 1] & 1, kWaitBudget)) ++s0_done[k ^ 1];
            else *s_abort = 1;
            read_row(SC_S0 + (k ^ 1) * SCAN_BLK, X);
            ptx::tmem_st32(lane_base + dn, X);
            ptx::tmem_st_wait();
        }
        if (ptx::mbar_wait(bar, done & 1, kWaitBudget)) ++done; else *s_abort = 1;
        ptx::tc_fence_after_sync();
        // this M buffer is free again: fetch the tile two steps ahead into it
        if (tid == 0 && g + 3 < nseg)
            bulk_load(sm + SC_MB + k * 32768, cells + (size_t)(g + 2) * SEG_CELL + SEG_MT, 32768, bar_mb + k);
        if (g + 3 < nseg) ++mb_issued[k];
        ptx::tmem_ld32(lane_base + dk, X);   // S_in(g + 1): the next step's operand
        ptx::tmem_ld_wait();
        scan_block_to_bf16(sm + SC_SB, c, X);
    }
    if (tid == 0) ptx::bulk_wait_read();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (!*s_abort) {
        ptx::tc_fence_after_sync();
        save(nseg - 1, (uint32_t)(SCAN_JB * ((nseg - 2) & 1)), X);
    } else {
        if (tid == 0) report_status(p.status, kDevTimeout);
        while (done < issued && ptx::mbar_wait(bar, done & 1, kWaitBudget)) ++done;
        for (int k = 0; k < 2; ++k) {
            while (mb_done[k] < mb_issued[k] && ptx::mbar_wait(bar_mb + k, mb_done[k] & 1, kWaitBudget)) ++mb_done[k];
            while (s0_done[k] < s0_issued[k] && ptx::mbar_wait(bar_s0 + k, s0_done[k] & 1, kWaitBudget)) ++s0_done[k];
        }
    }
    if (tid == 0) ptx::bulk_wait_all();   // the S_in blocks are out before the CTA ends
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, 2 * SCAN_JB);
    }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// Host side.
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

// A float32 [rows][128] buffer as a 2-D tensor with 32 x 128 boxes (128-byte
// swizzle): the scan's state blocks.
static bool make_map_state(CUtensorMap *m, const void *base, int64_t rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)tc::D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)tc::D * 4};
    cuuint32_t box[2] = {(cuuint32_t)tc::SCAN_JB, 128};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The log-decay g, [T, H*128] float32, as a 2-D tensor with 32 x 64 boxes
// (128-byte rows, 128-byte swizzle); rows beyond T read as zeros.
static bool make_map_g(CUtensorMap *m, const float *base, int64_t T, int H) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)H * 128, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)H * 128 * 4};
    cuuint32_t box[2] = {32, 64};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T, H*128] bf16 viewed as a 2-D tensor; boxes of 64 channels x box_rows
// tokens, 128-byte swizzle, rows beyond T read as zeros.
bool make_map_bf16(CUtensorMap *m, const void *base, int64_t T, int H, int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)H * 128, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)H * 128 * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
static bool make_map(CUtensorMap *m, const void *base, int64_t T, int H) {
    return make_map_bf16(m, base, T, H, 64);
}

// Bytes of L2 on the current device.
static size_t l2_bytes() {
    int dev = 0, b = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&b, cudaDevAttrL2CacheSize, dev);
    return (size_t)b;
}
// Whether `bytes` of per-chunk records can stay in L2 beside the streamed
// inputs (at most three quarters of it).
static int records_fit_l2(size_t bytes) { return bytes <= l2_bytes() / 4 * 3 ? 1 : 0; }

static int sm_count() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

// Split-path plan: used when the chains fill at most half the SMs and the
// sequences average at least 8 chunks.  The chunks are taken in windows of W
// per chain; workspace after the schedule area: the states carried between
// windows, then two record buffers of W slots per chain (window k uses buffer
// k % 2, so the intra kernel of window k + 1 can run beside the state kernel of
// window k).
struct SplitPlan {
    bool ok;
    int W, windows;
    int64_t max_chunks;
    size_t states_off, records_off, window_bytes, bytes;
};

static SplitPlan plan_split(int64_t total, int num_seqs, int H) {
    SplitPlan s{};
    const int64_t chains = (int64_t)num_seqs * H;
    s.max_chunks = (total + tc::C - 1) / tc::C;
    s.ok = chains > 0 && 2 * chains <= sm_count() && total >= (int64_t)8 * tc::C * num_seqs;
    if (!s.ok) return s;
    int64_t W = (s.max_chunks + 3) / 4;   // about four windows, 8..256 chunks each
    W = W < 8 ? 8 : (W > 256 ? 256 : W);
    s.W = (int)W;
    s.windows = (int)((s.max_chunks + W - 1) / W);
    const size_t base = (kWsOrder + sizeof(int32_t) * (size_t)num_seqs + 1023) & ~size_t(1023);
    s.states_off = base;
    s.records_off = base + (size_t)chains * tc::D * tc::D * sizeof(float);
    s.window_bytes = (size_t)chains * s.W * tc::REC_BYTES;
    s.bytes = s.records_off + 2 * s.window_bytes;
    return s;
}

// Segment-scan plan: when the chains fill at most a third of the SMs, each
// chain's chunks are cut into `segs` segments of `seg_len` chunks (at most one
// CTA per segment on the GPU, at least 4 chunks each).  Workspace after the
// schedule area: a record for every chunk, then per (chain, segment) the
// segment's map (S0 and M) and its incoming state.
struct ScanPlan {
    bool ok;
    int segs, seg_len;
    int64_t max_chunks;
    size_t rec_off, seg_out_off, seg_in_off, bytes;
};
constexpr size_t kScanRecordLimit = size_t(1) << 31;   // records of every chunk at once

static ScanPlan plan_scan(int64_t total, int num_seqs, int H) {
    ScanPlan s{};
    const int64_t chains = (int64_t)num_seqs * H;
    const int sms = sm_count();
    s.max_chunks = (total + tc::C - 1) / tc::C;
    if (chains <= 0 || 3 * chains > sms || total < (int64_t)8 * tc::C * num_seqs) return s;
    int64_t segs = sms / chains;
    if (segs > 64) segs = 64;
    int64_t len = (s.max_chunks + segs - 1) / segs;
    if (len < 4) len = 4;
    segs = (s.max_chunks + len - 1) / len;
    const size_t records = (size_t)chains * s.max_chunks * tc::REC_BYTES;
    if (segs < 3 || records > kScanRecordLimit) return s;
    s.ok = true;
    s.segs = (int)segs;
    s.seg_len = (int)len;
    s.rec_off = (kWsOrder + sizeof(int32_t) * (size_t)num_seqs + 1023) & ~size_t(1023);
    s.seg_out_off = s.rec_off + records;
    s.seg_in_off = s.seg_out_off + (size_t)chains * segs * tc::SEG_CELL;
    s.bytes = s.seg_in_off + (size_t)chains * segs * tc::D * tc::D * sizeof(float);
    return s;
}

// Extra workspace bytes the tensor-core prefill can use for these sizes (0
// when the fused kernel alone is planned).
size_t prefill_tc_workspace_bytes(int64_t total, int num_seqs, int H) {
    const ScanPlan c = plan_scan(total, num_seqs, H);
    const SplitPlan s = plan_split(total, num_seqs, H);
    size_t b = s.ok ? s.bytes : 0;
    if (c.ok && c.bytes > b) b = c.bytes;
    return b;
}

// Kernels one tensor-core prefill launches: the schedule kernel, then either
// the fused kernel or an intra and a state kernel per window.
// The chunked path for a given (unbounded) log-decay: the segment-scan plan
// plus the diagonal tiles of every chunk; 0 when that plan does not apply.
static int64_t diag_stride(int64_t total, int num_seqs) { return (total >> 6) + num_seqs + 1; }

static cudaError_t launch_diag_tiles(const void *q, const void *k, const float *g, const int32_t *cu,
                                     int64_t total, int num_seqs, int H, float *diag, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(tc::diag_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tc::SMEM_DIAG);
    if (e != cudaSuccess) return e;
    tc::DiagParams dp;
    dp.q = static_cast<const __nv_bfloat16 *>(q);
    dp.k = static_cast<const __nv_bfloat16 *>(k);
    dp.g = g;
    dp.cu_seqlens = cu;
    dp.total_tokens = total;
    dp.num_seqs = num_seqs;
    dp.H = H;
    dp.diag = diag;
    dp.stride = diag_stride(total, num_seqs);
    const int64_t slots = (int64_t)H * dp.stride;
    const int64_t grid = 4 * (int64_t)sm_count();
    // a plain launch: it waits for the schedule (status word) like any kernel
    tc::diag_tiles_kernel<<<(unsigned)(slots < grid ? slots : grid), 256, tc::SMEM_DIAG, st>>>(dp);
    return cudaGetLastError();
}

// The chunked paths for a given (unbounded) log-decay: the segment-scan plan
// when it applies, else the fused kernel; both plus the diagonal tiles of
// every chunk.
static size_t diag_bytes(int64_t total, int num_seqs, int H) {
    return (size_t)H * (size_t)diag_stride(total, num_seqs) * 8192;
}
size_t prefill_tc_logdecay_workspace_bytes(int64_t total, int num_seqs, int H) {
    const ScanPlan c = plan_scan(total, num_seqs, H);
    const size_t base = c.ok ? c.bytes : kWsOrder + sizeof(int32_t) * (size_t)num_seqs;
    return ((base + 255) & ~size_t(255)) + diag_bytes(total, num_seqs, H);
}

int prefill_tc_launches(int64_t total, int num_seqs, int H, size_t workspace_bytes) {
    const ScanPlan c = plan_scan(total, num_seqs, H);
    if (c.ok && workspace_bytes >= c.bytes) return 5;
    const SplitPlan s = plan_split(total, num_seqs, H);
    return 1 + ((s.ok && workspace_bytes >= s.bytes) ? 2 * s.windows : 1);
}

// The split plan's side stream and events, one set per device, created on
// first use and kept until the process exits.  The mutex also keeps the
// event bookkeeping of calls from several host threads apart.
struct SideStream {
    cudaStream_t s;
    cudaEvent_t fork, intra[2], state[2];
};
constexpr int kMaxDevices = 64;
static std::mutex g_side_mu;
static SideStream g_side[kMaxDevices];

static cudaError_t side_stream(SideStream **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    SideStream &ss = g_side[dev];
    if (!ss.s) {
        SideStream n{};
        e = cudaStreamCreateWithFlags(&n.s, cudaStreamNonBlocking);
        cudaEvent_t *evs[5] = {&n.fork, &n.intra[0], &n.intra[1], &n.state[0], &n.state[1]};
        for (int i = 0; i < 5 && e == cudaSuccess; ++i)
            e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        ss = n;
    }
    *out = &ss;
    return cudaSuccess;
}

cudaError_t launch_schedule(const int32_t *cu, int num_seqs, int32_t *order, uint32_t *counter,
                            uint32_t *status, cudaStream_t st);
cudaError_t launch_prefill_c32(const void *q, const void *k, const void *v, const void *z, const float *A,
                               const float *beta, const int32_t *cu, int num_seqs, int64_t total, int H,
                               const float *s0, float *s1, void *out, int32_t *order, uint32_t *counter,
                               uint32_t *status, int test_expire, int sms, cudaStream_t st);

// Test support: the kExpire* bits the next tensor-core prefill call passes to
// its kernels (kda_testing_expire_next_wait); taken, and cleared, by that call.
static std::atomic<int> g_test_expire{0};
void set_test_expire(int mask) { g_test_expire.store(mask); }

// Launches a kernel with programmatic stream serialization: it may start
// while the previous kernel of the stream finishes and waits for that
// kernel's results in ptx::pdl_wait().
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, unsigned smem,
                              cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Prefill with the log-decay g given (any value): schedule, the diagonal
// tiles' pre-pass, the intra-chunk kernel in its unbounded mode, then the
// segment maps, the scan and the state pass of the segment-scan plan.  Returns
// cudaErrorNotSupported when that plan does not apply or the workspace is too
// small (the caller then runs the token-serial kernel).
cudaError_t launch_prefill_tc_logdecay(const void *q, const void *k, const void *v, const float *g,
                                       const float *beta, const int32_t *cu, int num_seqs,
                                       int64_t total, int H, const float *s0, float *s1, void *out,
                                       void *workspace, size_t workspace_bytes, cudaStream_t st) {
    const ScanPlan scan = plan_scan(total, num_seqs, H);
    const size_t need = prefill_tc_logdecay_workspace_bytes(total, num_seqs, H);
    if (workspace_bytes < need) return cudaErrorNotSupported;
    const int test_expire = g_test_expire.exchange(0);
    CUtensorMap mq, mk, mv, mg, mo;
    if (!make_map(&mq, q, total, H) || !make_map(&mk, k, total, H) ||
        !make_map(&mv, v, total, H) || !make_map_g(&mg, g, total, H) ||
        !make_map(&mo, out, total, H))
        return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kWsStatus);
    uint32_t *counter = reinterpret_cast<uint32_t *>(ws + kWsCounter);
    int32_t *order = reinterpret_cast<int32_t *>(ws + kWsOrder);
    cudaError_t e = launch_schedule(cu, num_seqs, order, counter, status, st);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    const int64_t chains = (int64_t)num_seqs * H;
    if (!scan.ok) {   // the fused kernel in its unbounded mode
        float *diag = reinterpret_cast<float *>(
            ws + ((kWsOrder + sizeof(int32_t) * (size_t)num_seqs + 255) & ~size_t(255)));
        if ((e = launch_diag_tiles(q, k, g, cu, total, num_seqs, H, diag, st)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(tc::prefill_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)tc::SMEM_ALLOC)) != cudaSuccess)
            return e;
        tc::Params prm;
        prm.A = nullptr; prm.beta = beta; prm.cu_seqlens = cu; prm.initial_state = s0;
        prm.final_state = s1; prm.out = static_cast<__nv_bfloat16 *>(out); prm.order = order;
        prm.counter = counter; prm.status = status; prm.total_tokens = total;
        prm.num_seqs = num_seqs; prm.H = H; prm.diag = diag; prm.diag_stride = diag_stride(total, num_seqs);
        prm.test_expire = test_expire;
        const int grid = (int)(chains < sms ? chains : sms);
        return launch_pdl(tc::prefill_tc_kernel<true>, (unsigned)grid, tc::NT, tc::SMEM_ALLOC, st, mq, mk, mv,
                          mg, mo, prm);
    }
    const void *kernels[4] = {(const void *)tc::prefill_intra_kernel<true>, (const void *)tc::prefill_seg_kernel,
                              (const void *)tc::prefill_scan_kernel, (const void *)tc::prefill_state_kernel<false>};
    const uint32_t smem[4] = {tc::SMEM_ALLOC, tc::SMEM_SEG, tc::SMEM_SCAN, tc::SMEM_STATE};
    for (int i = 0; i < 4; ++i)
        if ((e = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem[i])) != cudaSuccess)
            return e;
    tc::SplitParams sp;
    sp.A = nullptr; sp.beta = beta; sp.cu_seqlens = cu; sp.initial_state = s0; sp.final_state = s1;
    sp.out = static_cast<__nv_bfloat16 *>(out);
    sp.records = ws + scan.rec_off;
    sp.states = nullptr;
    sp.status = status; sp.total_tokens = total; sp.num_seqs = num_seqs; sp.H = H;
    sp.w0 = 0;
    sp.wn = (int)scan.max_chunks;
    sp.W = (int)scan.max_chunks;
    sp.segs = 1;
    sp.seg_len = scan.seg_len;
    sp.seg_out = ws + scan.seg_out_off;
    sp.seg_in = reinterpret_cast<float *>(ws + scan.seg_in_off);
    sp.diag = reinterpret_cast<float *>(ws + ((scan.bytes + 255) & ~size_t(255)));
    sp.diag_stride = diag_stride(total, num_seqs);
    sp.test_expire = test_expire;
    sp.map_out = nullptr; sp.rec_stride = 0;
    sp.rec_in_l2 = records_fit_l2((size_t)chains * scan.max_chunks * tc::REC_BYTES);
    const int64_t items = chains * scan.max_chunks;
    if ((e = launch_diag_tiles(q, k, g, cu, total, num_seqs, H, const_cast<float *>(sp.diag), st)) != cudaSuccess)
        return e;
    if ((e = launch_pdl(tc::prefill_intra_kernel<true>, (unsigned)(items < sms ? items : sms),
                        tc::NT, tc::SMEM_ALLOC, st, mq, mk, mv, mg, sp)) != cudaSuccess)
        return e;
    sp.segs = scan.segs;
    const unsigned cells = (unsigned)(chains * scan.segs);
    if ((e = launch_pdl(tc::prefill_seg_kernel, cells, tc::NT, tc::SMEM_SEG, st, sp)) != cudaSuccess) return e;
    CUtensorMap ms0, msin;
    if (!make_map_state(&ms0, sp.seg_out, chains * scan.segs * tc::SEG_CELL_ROWS) ||
        !make_map_state(&msin, sp.seg_in, chains * scan.segs * tc::D))
        return cudaErrorInvalidValue;
    if ((e = launch_pdl(tc::prefill_scan_kernel, (unsigned)(chains * tc::SCAN_SPLIT), tc::SCAN_NT,
                        tc::SMEM_SCAN, st, ms0, msin, sp)) != cudaSuccess)
        return e;
    return launch_pdl(tc::prefill_state_kernel<false>, cells, tc::NT, tc::SMEM_STATE, st, mo, sp);
}

// ---- segment maps (kda_segment_map) ------------------------------------------
// For every (sequence, head) the affine map of the whole sequence, S_out =
// M S_in + b: the intra kernel writes the records of every chunk (at compact
// slots, so a batch of many sequences needs no more than ~T/64 + N slots per
// head), the segment kernel in its map mode runs every segment of every chain
// from S = 0 and M = I in parallel and writes float32 (S0, M) per segment, and
// two compositions fold each chain's segments in order: M = M_last ... M_0 and
// b = the segments' S0 carried through the later maps.
struct MapPlan {
    bool ok;
    int segs, seg_len;
    int64_t max_chunks, stride;
    size_t rec_off, cell_off, bytes;
};

static MapPlan plan_map(int64_t total, int num_seqs, int H) {
    MapPlan m{};
    const int64_t chains = (int64_t)num_seqs * H;
    if (chains <= 0 || total <= 0) return m;
    m.max_chunks = (total + tc::C - 1) / tc::C;
    int64_t segs = sm_count() / chains;
    segs = segs < 1 ? 1 : (segs > 64 ? 64 : segs);
    int64_t len = (m.max_chunks + segs - 1) / segs;
    if (len < 1) len = 1;
    m.segs = (int)((m.max_chunks + len - 1) / len);
    m.seg_len = (int)len;
    m.stride = diag_stride(total, num_seqs);
    m.rec_off = (kWsOrder + sizeof(int32_t) * (size_t)num_seqs + 1023) & ~size_t(1023);
    m.cell_off = m.rec_off + (size_t)H * (size_t)m.stride * tc::REC_BYTES;
    m.bytes = m.cell_off + (size_t)chains * (size_t)m.segs * tc::MAP_CELL;
    m.ok = true;
    return m;
}

size_t segment_map_workspace_bytes(int64_t total, int num_seqs, int H) {
    const MapPlan m = plan_map(total, num_seqs, H);
    return m.ok ? m.bytes : 0;
}

cudaError_t launch_segment_map(const void *q, const void *k, const void *v, const void *z,
                               const float *A, const float *beta, const int32_t *cu, int num_seqs,
                               int64_t total, int H, float *M_out, float *b_out, void *workspace,
                               size_t workspace_bytes, cudaStream_t st) {
    const MapPlan m = plan_map(total, num_seqs, H);
    if (!m.ok) return cudaErrorInvalidValue;
    if (workspace_bytes < m.bytes) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv, mz;
    if (!make_map(&mq, q, total, H) || !make_map(&mk, k, total, H) ||
        !make_map(&mv, v, total, H) || !make_map(&mz, z, total, H))
        return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + kWsStatus);
    cudaError_t e = launch_schedule(cu, num_seqs, reinterpret_cast<int32_t *>(ws + kWsOrder),
                                    reinterpret_cast<uint32_t *>(ws + kWsCounter), status, st);
    if (e != cudaSuccess) return e;
    const void *kernels[2] = {(const void *)tc::prefill_intra_kernel<false>, (const void *)tc::prefill_seg_kernel};
    const uint32_t smem[2] = {tc::SMEM_ALLOC, tc::SMEM_SEG};
    for (int i = 0; i < 2; ++i)
        if ((e = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem[i])) != cudaSuccess)
            return e;
    const int sms = sm_count();
    const int64_t chains = (int64_t)num_seqs * H;
    tc::SplitParams sp{};
    sp.A = A; sp.beta = beta; sp.cu_seqlens = cu; sp.initial_state = nullptr; sp.final_state = nullptr;
    sp.out = nullptr;
    sp.records = ws + m.rec_off;
    sp.states = nullptr;
    sp.status = status; sp.total_tokens = total; sp.num_seqs = num_seqs; sp.H = H;
    sp.w0 = 0;
    sp.wn = (int)m.max_chunks;
    sp.W = (int)m.max_chunks;
    sp.segs = 1;
    sp.seg_len = m.seg_len;
    sp.seg_out = nullptr; sp.seg_in = nullptr;
    sp.diag = nullptr; sp.diag_stride = 0;
    sp.test_expire = 0;
    sp.map_out = ws + m.cell_off;
    sp.rec_stride = m.stride;
    sp.rec_in_l2 = records_fit_l2((size_t)H * (size_t)m.stride * tc::REC_BYTES);   // (kept for the segment kernel)
    const int64_t items = chains * m.max_chunks;
    if ((e = launch_pdl(tc::prefill_intra_kernel<false>, (unsigned)(items < sms ? items : sms), tc::NT,
                        tc::SMEM_ALLOC, st, mq, mk, mv, mz, sp)) != cudaSuccess)
        return e;
    sp.segs = m.segs;
    if ((e = launch_pdl(tc::prefill_seg_kernel, (unsigned)(chains * m.segs), tc::NT, tc::SMEM_SEG, st, sp)) !=
        cudaSuccess)
        return e;
    // fold each chain's segments: M = M_last ... M_0 (from I), b (from 0, adding each S0)
    const float *cells = reinterpret_cast<const float *>(ws + m.cell_off);
    const int64_t cell_f = (int64_t)(tc::MAP_CELL / 4);
    ComposeParams cp{};
    cp.M = cells + cell_f / 2;
    cp.m_step = cell_f;
    cp.m_prob = (int64_t)m.segs * cell_f;
    cp.B = nullptr;
    cp.init = nullptr;
    cp.init_identity = 1;
    cp.out_all = nullptr;
    cp.out_last = M_out;
    cp.last_prob = (int64_t)tc::D * tc::D;
    cp.ncols = tc::D;
    cp.cu_seqlens = cu;
    cp.H = H;
    cp.seg_len = m.seg_len;
    cp.total = total;
    cp.status = status;
    if ((e = launch_compose(cp, (int)chains, tc::D, st)) != cudaSuccess) return e;
    cp.B = cells;
    cp.b_step = cell_f;
    cp.b_prob = (int64_t)m.segs * cell_f;
    cp.init_identity = 0;
    cp.out_last = b_out;
    return launch_compose(cp, (int)chains, tc::D, st);
}

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *z,
                              const float *A, const float *beta, const int32_t *cu,
                              int num_seqs, int64_t total, int H, const float *s0, float *s1,
                              void *out, void *workspace, size_t workspace_bytes, cudaStream_t st) {
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
    const int sms = sm_count();
    const int64_t chains = (int64_t)num_seqs * H;
    const int test_expire = g_test_expire.exchange(0);

    const ScanPlan scan = plan_scan(total, num_seqs, H);
    if (scan.ok && workspace_bytes >= scan.bytes) {
        const void *kernels[4] = {(const void *)tc::prefill_intra_kernel<false>, (const void *)tc::prefill_seg_kernel,
                                  (const void *)tc::prefill_scan_kernel, (const void *)tc::prefill_state_kernel<false>};
        const uint32_t smem[4] = {tc::SMEM_ALLOC, tc::SMEM_SEG, tc::SMEM_SCAN, tc::SMEM_STATE};
        for (int i = 0; i < 4; ++i)
            if ((e = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem[i])) != cudaSuccess)
                return e;
        tc::SplitParams sp;
        sp.A = A; sp.beta = beta; sp.cu_seqlens = cu; sp.initial_state = s0; sp.final_state = s1;
        sp.out = static_cast<__nv_bfloat16 *>(out);
        sp.records = ws + scan.rec_off;
        sp.states = nullptr;
        sp.status = status; sp.total_tokens = total; sp.num_seqs = num_seqs; sp.H = H;
        sp.w0 = 0;
        sp.wn = (int)scan.max_chunks;
        sp.W = (int)scan.max_chunks;
        sp.segs = 1;
        sp.seg_len = scan.seg_len;
        sp.seg_out = ws + scan.seg_out_off;
        sp.seg_in = reinterpret_cast<float *>(ws + scan.seg_in_off);
        sp.diag = nullptr; sp.diag_stride = 0;
        sp.test_expire = test_expire;
        sp.map_out = nullptr; sp.rec_stride = 0;
        sp.rec_in_l2 = records_fit_l2((size_t)chains * scan.max_chunks * tc::REC_BYTES);
        const int64_t items = chains * scan.max_chunks;
        if ((e = launch_pdl(tc::prefill_intra_kernel<false>, (unsigned)(items < sms ? items : sms),
                            tc::NT, tc::SMEM_ALLOC, st, mq, mk, mv, mz, sp)) != cudaSuccess)
            return e;
        sp.segs = scan.segs;
        const unsigned cells = (unsigned)(chains * scan.segs);
        if ((e = launch_pdl(tc::prefill_seg_kernel, cells, tc::NT, tc::SMEM_SEG, st, sp)) != cudaSuccess) return e;
        CUtensorMap ms0, msin;
        if (!make_map_state(&ms0, sp.seg_out, chains * scan.segs * tc::SEG_CELL_ROWS) ||
            !make_map_state(&msin, sp.seg_in, chains * scan.segs * tc::D))
            return cudaErrorInvalidValue;
        if ((e = launch_pdl(tc::prefill_scan_kernel, (unsigned)(chains * tc::SCAN_SPLIT), tc::SCAN_NT,
                            tc::SMEM_SCAN, st, ms0, msin, sp)) != cudaSuccess)
            return e;
        return launch_pdl(tc::prefill_state_kernel<false>, cells, tc::NT, tc::SMEM_STATE, st, mo, sp);
    }

    const SplitPlan plan = plan_split(total, num_seqs, H);
    if (plan.ok && workspace_bytes >= plan.bytes) {
        e = cudaFuncSetAttribute(tc::prefill_intra_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::prefill_state_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::SMEM_STATE);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(g_side_mu);
        SideStream *ss = nullptr;
        e = side_stream(&ss);
        if (e != cudaSuccess) return e;
        tc::SplitParams sp;
        sp.A = A; sp.beta = beta; sp.cu_seqlens = cu; sp.initial_state = s0; sp.final_state = s1;
        sp.out = static_cast<__nv_bfloat16 *>(out);
        sp.states = reinterpret_cast<float *>(ws + plan.states_off);
        sp.status = status; sp.total_tokens = total; sp.num_seqs = num_seqs; sp.H = H;
        sp.W = plan.W;
        sp.segs = 1; sp.seg_len = 0; sp.seg_out = nullptr; sp.seg_in = nullptr;
        sp.diag = nullptr; sp.diag_stride = 0;
        sp.test_expire = test_expire;
        sp.map_out = nullptr; sp.rec_stride = 0;
        sp.rec_in_l2 = records_fit_l2(2 * plan.window_bytes);
        // fork: the side stream starts after everything already on `st`
        if ((e = cudaEventRecord(ss->fork, st)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(ss->s, ss->fork, 0)) != cudaSuccess) return e;
        for (int wi = 0; wi < plan.windows; ++wi) {
            const int buf = wi & 1;
            const int64_t w0 = (int64_t)wi * plan.W;
            sp.w0 = (int)w0;
            sp.wn = (int)((plan.max_chunks - w0) < plan.W ? (plan.max_chunks - w0) : plan.W);
            sp.records = ws + plan.records_off + buf * plan.window_bytes;
            // buffer `buf` was last read by the state kernel of window wi - 2
            if (wi >= 2 && (e = cudaStreamWaitEvent(ss->s, ss->state[buf], 0)) != cudaSuccess) return e;
            const int64_t items = chains * sp.wn;
            const int64_t cap = wi == 0 ? sms : sms - chains;   // leave room for the state kernel
            const int grid = (int)(items < cap ? items : cap);
            tc::prefill_intra_kernel<false><<<grid, tc::NT, tc::SMEM_ALLOC, ss->s>>>(mq, mk, mv, mz, sp);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            if ((e = cudaEventRecord(ss->intra[buf], ss->s)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(st, ss->intra[buf], 0)) != cudaSuccess) return e;
            tc::prefill_state_kernel<true><<<(unsigned)chains, tc::NT, tc::SMEM_STATE, st>>>(mo, sp);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            if ((e = cudaEventRecord(ss->state[buf], st)) != cudaSuccess) return e;
        }
        return cudaGetLastError();
    }

    return launch_prefill_c32(q, k, v, z, A, beta, cu, num_seqs, total, H, s0, s1, out, order, counter, status,
                              test_expire, sms, st);
}

}  // namespace kda
