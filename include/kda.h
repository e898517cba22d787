/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * Kimi Delta Attention (KDA) is the recurrent sequence mixer of the Kimi K3
 * hybrid stack ("Kimi K3 internals analysis", molayo1419.me, section
 * "Sequence mixing"): a fixed-size per-head state S (dk x dv, rows = key
 * channels) replaces the KV cache and is written by the delta rule, after a
 * channel-wise retention factor has decayed the old state:
 *
 *     g_t   = g_min * sigmoid(exp(A) * z_t),  g_min = -5,  alpha_t = exp(g_t)
 *     S'    = Diag(alpha_t) S_{t-1}
 *     S_t   = S' + beta_t k_t (v_t - S'^T k_t)^T
 *     o_t   = S_t^T q_t
 *
 * The bounded gate keeps the cumulative log-decay of any 16 consecutive tokens
 * inside (-80, 0) (same section), which is what lets the chunked prefill use
 * dense tensor-core tiles on the diagonal blocks too.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers, allocated and owned by the
 *     caller.  The library allocates no device memory in any call.
 *   - Every call is asynchronous on the caller's stream `stream` (0 = the
 *     legacy default stream).  Argument errors are detected on the host,
 *     before anything is launched, and returned as KDA_ERR_INVALID_ARG or
 *     KDA_ERR_UNSUPPORTED; nothing is written in that case.  A failed launch
 *     returns KDA_ERR_CUDA.  Conditions found on the device (a bounded wait
 *     that expired) are recorded in a status word inside the caller's
 *     workspace and read with kda_check_device_status().  No call traps.
 *   - Layouts are dense row-major ("packed"): tokens of all sequences are
 *     concatenated along the first axis, sequence i owning rows
 *     [cu_seqlens[i], cu_seqlens[i+1]).  Per-token tensors are [T, H, d].
 *   - q and k are used as given (callers normalise them; there is no 1/sqrt(dk)
 *     scale).  beta is a scalar per (token, head), already in (0, 1).
 *   - A, beta, g and every state are float32.  q, k, v, z and the output share
 *     one element type, kda_dtype_t.
 *   - Supported head dimensions: dk, dv in {32, 64, 128}.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t / CUstream). */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,    /* null pointer, negative size, misaligned buffer */
    KDA_ERR_UNSUPPORTED = 2,    /* valid but unsupported shape or dtype */
    KDA_ERR_CUDA = 3,           /* a CUDA runtime/driver call or launch failed */
    KDA_ERR_DEVICE_TIMEOUT = 4  /* a device-side bounded wait expired */
} kda_status_t;

typedef enum {
    KDA_F32 = 0,
    KDA_BF16 = 1
} kda_dtype_t;

/* Human-readable name of a status code (static string, never NULL). */
const char *kda_status_string(kda_status_t status);

/*
 * kda_gate -- the bounded gate ("Sequence mixing": g = g_min * sigmoid(exp(A) z),
 * g_min = -5).
 *   z      [n_tokens, H, dk], element type z_dtype
 *   A      [H, dk] float32
 *   g_out  [n_tokens, H, dk] float32 (written)
 * g_out lies in [-5, 0): in float32 the sigmoid rounds to exactly 1 once
 * exp(A) z exceeds about 16.6, so the open bound of the exact formula closes.
 */
kda_status_t kda_gate(const void *z, kda_dtype_t z_dtype, const float *A, float *g_out,
                      int64_t n_tokens, int H, int dk, kda_stream_t stream);

/*
 * kda_prefill_workspace_size -- bytes of device workspace that let
 * kda_chunk_prefill use its fastest plan for these sizes.  The minimum it
 * accepts is 256 + 4 * num_seqs bytes (rounded up to 256): a status word, a
 * work counter and a schedule.  For bf16, dk = dv = 128 batches with few
 * (sequence, head) chains (at most half the SM count) the returned size also
 * holds the chunk-parallel plan's per-chunk records (72.5 KB per chunk, two
 * buffers of a window of 8 to 256 chunks per chain) and one carried state per
 * chain; with less than that the call falls back to the one-kernel plan.  The
 * workspace holds no data between calls except the status word, which every
 * call clears on entry.
 */
size_t kda_prefill_workspace_size(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                  kda_dtype_t dtype);

/*
 * kda_chunk_prefill -- KDA over a packed batch of variable-length sequences
 * ("Sequence mixing"; the state is the fixed-size memory of the same section).
 *   q, k, z        [total_tokens, H, dk], element type dtype
 *   v              [total_tokens, H, dv], element type dtype
 *   A              [H, dk] float32
 *   beta           [total_tokens, H] float32
 *   cu_seqlens     [num_seqs + 1] int32, device; cu_seqlens[0] = 0, non-decreasing,
 *                  cu_seqlens[num_seqs] = total_tokens (not checked on the host:
 *                  reading it would synchronise)
 *   initial_state  [num_seqs, H, dk, dv] float32, or NULL for zeros
 *   final_state    [num_seqs, H, dk, dv] float32 (written), or NULL; it may be
 *                  the same buffer as initial_state
 *   out            [total_tokens, H, dv], element type dtype (written)
 *   workspace      device buffer, 16-byte aligned, of at least the minimum above
 *                  (kda_prefill_workspace_size() bytes enable every plan)
 * Length-0 sequences copy their initial state (or zeros) to final_state.
 * bf16 inputs with dk = dv = 128 run the chunkwise tensor-core path (64-token
 * chunks, 16-token decay tiles): one persistent kernel over the chains when
 * they fill the GPU, else, window by window, a chunk-parallel kernel for the
 * state-independent work and a per-chain state-pass kernel.  That split plan
 * runs the chunk-parallel kernel of the next window on an internal stream
 * (one per device, created on the first such call and kept until exit,
 * joined back to `stream` with events), so the call stays ordered on
 * `stream` as a whole; calls from several host threads take turns on it.
 * Every other supported case runs the token-serial float32 kernel.
 */
kda_status_t kda_chunk_prefill(const void *q, const void *k, const void *v, const void *z,
                               const float *A, const float *beta, const int32_t *cu_seqlens,
                               int num_seqs, int64_t total_tokens, int H, int dk, int dv,
                               kda_dtype_t dtype, const float *initial_state,
                               float *final_state, void *out, void *workspace,
                               size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_prefill_logdecay -- the same prefill with the per-channel
 * log-decay g given directly instead of through the bounded gate, so alpha =
 * exp(g) with g unbounded below (intended range g <= 0; the chunked path takes
 * values below -100 as -100, where exp(g) is already below the float32 normal
 * range).  "Kimi K3 internals
 * analysis", section "Sequence mixing": before K3 the log-decay had no lower
 * bound, the reciprocal cumulative decay of a chunk could overflow, and the
 * diagonal 16-token tiles needed a special position-pair path instead of the
 * dense tensor-core one.  That is what this call does for bf16 with dk = dv =
 * 128 when the workspace holds kda_prefill_logdecay_workspace_size() bytes:
 * the diagonal tiles of every chunk are summed pair by pair in a pre-pass and
 * every other factor is formed with a non-positive exponent, in the
 * segment-scan plan for batches of few long sequences and in the fused kernel
 * otherwise.  With a smaller workspace, or another dtype or head size, it runs
 * the token-serial kernel (a 4-byte workspace suffices).  Both are exact for
 * any decay; the measure of what the bound buys.
 *   g          [total_tokens, H, dk] float32 (replaces z and A), 16-byte aligned
 *   workspace  16-byte aligned; at least 4 bytes (the status word)
 * All other arguments as for kda_chunk_prefill.
 */
/* Workspace for kda_chunk_prefill_logdecay's chunked path (the kda_chunk_prefill
 * minimum when that path does not apply to these sizes). */
size_t kda_prefill_logdecay_workspace_size(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                           kda_dtype_t dtype);

kda_status_t kda_chunk_prefill_logdecay(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta,
                                        const int32_t *cu_seqlens, int num_seqs,
                                        int64_t total_tokens, int H, int dk, int dv,
                                        kda_dtype_t dtype, const float *initial_state,
                                        float *final_state, void *out, void *workspace,
                                        size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_prefill_kernel_launches -- how many kernels one kda_chunk_prefill call
 * with these sizes and this workspace size launches (q, k, v, z and out
 * assumed 16-byte aligned); 0 for an empty batch.  For instrumentation, e.g. a
 * benchmark that reports its kernel launches.  Pure host computation: no
 * device call, no error status.
 */
int kda_prefill_kernel_launches(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                kda_dtype_t dtype, size_t workspace_bytes);

/*
 * kda_chunk_prefill_noalloc -- kda_chunk_prefill for callers that cannot
 * allocate device memory.  The pages have no counterpart to this call: it is
 * a library convenience, not part of the method.
 *
 * Some callers cannot call cudaMalloc when they run a prefill: plugin code in
 * a host application that owns the device memory and offers no allocator,
 * serving loops whose device-memory budget is fixed at start-up, and code that
 * must not take the allocator's implicit device synchronisation.  This call
 * takes the same arguments as kda_chunk_prefill except the workspace, and
 * allocates nothing: its scratch is a fixed device array inside the library
 * (KDA_NOALLOC_MAX_SEQS * 4 + 256 bytes, about 64 KiB), which every GPU that
 * loads the library holds until the process exits.
 *   - num_seqs above KDA_NOALLOC_MAX_SEQS returns KDA_ERR_UNSUPPORTED, before
 *     anything is launched.
 *   - Each call looks up the scratch's device address (cudaGetSymbolAddress,
 *     with the caller's current device) and caches it per device; a call made
 *     during a stream capture uses the cached address, so make a first call
 *     on each device before any stream capture.
 *   - Every call on a device shares the one scratch array.  Each call resets
 *     the parts that must start at zero, but calls that overlap on the GPU
 *     (concurrent streams, or other host threads) race on it: serialise them.
 *   - Device-side conditions (malformed offsets, an expired wait) are recorded
 *     in that shared scratch and are not reported by this call; use
 *     kda_chunk_prefill with a workspace and kda_check_device_status to see
 *     them.
 *   - The scratch has room only for the one-kernel (fused) plan of the
 *     tensor-core path, never for the few-chain plans.  The results are
 *     therefore bit-identical to kda_chunk_prefill's when that call also runs
 *     the fused plan (always, given the minimum workspace; for batches of
 *     many chains also with kda_prefill_workspace_size() bytes).  For few
 *     long sequences kda_chunk_prefill with its full workspace sums in another
 *     order: the two agree within the parity tolerance, not bit for bit, and
 *     this call is slower there.
 *   - The lookup is repeated on every call made outside a capture, since the
 *     address changes if the host resets the device and the library's module
 *     is loaded anew.
 */
#define KDA_NOALLOC_MAX_SEQS 16384
kda_status_t kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v,
                                       const void *z, const float *A, const float *beta,
                                       const int32_t *cu_seqlens, int num_seqs,
                                       int64_t total_tokens, int H, int dk, int dv,
                                       kda_dtype_t dtype, const float *initial_state,
                                       float *final_state, void *out, kda_stream_t stream);

/*
 * kda_decode_step -- one new token for each of N sequences; the recurrent
 * state is read and updated IN PLACE (the fixed-size state that replaces the
 * KV cache, "Sequence mixing").
 *   q, k, z   [N, H, dk], element type dtype
 *   v         [N, H, dv], element type dtype
 *   A         [H, dk] float32
 *   beta      [N, H] float32
 *   state     [N, H, dk, dv] float32, read and overwritten
 *   out       [N, H, dv], element type dtype (written)
 */
kda_status_t kda_decode_step(const void *q, const void *k, const void *v, const void *z,
                             const float *A, const float *beta, float *state, void *out,
                             int N, int H, int dk, int dv, kda_dtype_t dtype,
                             kda_stream_t stream);

/*
 * kda_decode_tokens -- n_tokens new tokens for each of N sequences whose
 * recurrent states live in a pool, as a serving engine keeps them (the
 * fixed-size state that replaces the KV cache, "Sequence mixing": one state
 * per live sequence, stepped in batches).  Sequence i applies its tokens in
 * order to state_pool[slot_ids[i]], updated in place; every token gets its
 * output.  With n_tokens > 1 the state is read and written once per call, not
 * once per token.  kda_decode_step is the case n_tokens = 1, slot i = i.
 *   q, k, z     [N, n_tokens, H, dk], element type dtype
 *   v           [N, n_tokens, H, dv], element type dtype
 *   A           [H, dk] float32
 *   beta        [N, n_tokens, H] float32
 *   state_pool  [pool_size, H, dk, dv] float32, 16-byte aligned, read and
 *               overwritten at the slots named
 *   slot_ids    [N] int32, device, or NULL for slot i = sequence i (then
 *               pool_size >= N).  A negative id marks a padding row: its
 *               outputs are written as zeros and no state is touched.  An id
 *               >= pool_size is recorded in *status (KDA_ERR_INVALID_ARG) and
 *               its row is treated as padding.  Two rows of one call naming
 *               the same slot race; give each live sequence its own slot.
 *   out         [N, n_tokens, H, dv], element type dtype (written)
 *   status      device uint32, or NULL; e.g. the first word of a prefill
 *               workspace, then read with kda_check_device_status()
 * Supported: dk, dv in {32, 64, 128}, any n_tokens >= 0.
 * With bf16 inputs, dk = dv = 128, n_tokens >= 4 and 16-byte aligned q, k, v,
 * z, out and state_pool, the tokens of a sequence are processed in the chunked form on the
 * tensor cores (as kda_chunk_prefill does: results agree with the token-serial
 * form to bf16 rounding, not bit for bit); otherwise token by token in
 * float32.
 */
kda_status_t kda_decode_tokens(const void *q, const void *k, const void *v, const void *z,
                               const float *A, const float *beta, float *state_pool,
                               int pool_size, const int32_t *slot_ids, void *out, int N,
                               int n_tokens, int H, int dk, int dv, kda_dtype_t dtype,
                               uint32_t *status, kda_stream_t stream);

/*
 * kda_state_slots_copy -- the prefill -> decode handoff of a serving engine:
 * moves N recurrent states between a contiguous buffer (the final_state or
 * initial_state of kda_chunk_prefill) and their slots of a decode state pool
 * (kda_decode_tokens).  "Kimi K3 internals analysis", section "Sequence
 * mixing": the fixed-size state is what a sequence carries from prefill into
 * decode.
 *   state_pool  [pool_size, H, dk, dv] float32, 16-byte aligned
 *   slot_ids    [N] int32, device.  A negative id skips the row (when copying
 *               from the pool its states are written as zeros); an id >=
 *               pool_size is recorded in *status (KDA_ERR_INVALID_ARG) and
 *               skipped the same way.
 *   states      [N, H, dk, dv] float32, 16-byte aligned
 *   to_pool     nonzero: states -> pool slots; zero: pool slots -> states
 *   status      device uint32 or NULL, as for kda_decode_tokens
 * Supported: dk, dv in {32, 64, 128}.  Asynchronous on `stream`.
 */
kda_status_t kda_state_slots_copy(float *state_pool, int pool_size, const int32_t *slot_ids,
                                  float *states, int N, int H, int dk, int dv, int to_pool,
                                  uint32_t *status, kda_stream_t stream);

/*
 * Context parallelism: one long sequence split over several workers ("Kimi K3
 * internals analysis", section "3T급 MoE를 위한 인프라" (infrastructure for the
 * 3T-class MoE), the KDA context-parallelism paragraph).  Over any segment of
 * tokens the state map is affine,
 *     S_out = M S_in + b,    M [dk, dk],  b [dk, dv]  (S rows = key channels),
 * b being the segment run from a zero state and M the product of
 * (I - beta_t k_t k_t^T) Diag(alpha_t) over its tokens t, the last on the left.  Each worker computes the map of
 * its own segment (kda_segment_map), the workers exchange the maps (fixed size,
 * whatever the segment length), each composes the maps of the segments before
 * its own into its true incoming state (kda_state_compose) and runs its
 * segment from that state (kda_chunk_prefill with initial_state).
 *
 * kda_segment_map -- for every sequence of a packed batch (each one a segment
 * of some longer sequence) and every head, the map (M, b) of that sequence.
 *   q, k, v, z, A, beta, cu_seqlens, num_seqs, total_tokens, H, dk, dv, dtype:
 *                  as for kda_chunk_prefill; bf16 with dk = dv = 128 only
 *                  (KDA_ERR_UNSUPPORTED otherwise), q/k/v/z 16-byte aligned
 *   M              [num_seqs, H, dk, dk] float32 (written); I for an empty sequence
 *   b              [num_seqs, H, dk, dv] float32 (written); 0 for an empty sequence
 *   workspace      16-byte aligned, kda_segment_map_workspace_size() bytes:
 *                  the status word (kda_check_device_status), the per-chunk
 *                  records of every chunk (72.5 KB per 64-token chunk and head)
 *                  and a 128 KB cell per (sequence, head, segment)
 * Runs the chunk-parallel kernel of the prefill, the segment kernel in a mode
 * that keeps float32 maps for every segment of every (sequence, head), and a
 * float32 composition of each chain's segments in order.  The maps are meant
 * for batches of a few long sequences (one per worker and head); M's columns
 * are those of a state, so its rounding is that of a state carried through the
 * bf16 tensor-core products of the prefill.
 */
size_t kda_segment_map_workspace_size(int64_t total_tokens, int num_seqs, int H, int dk, int dv,
                                      kda_dtype_t dtype);
kda_status_t kda_segment_map(const void *q, const void *k, const void *v, const void *z,
                             const float *A, const float *beta, const int32_t *cu_seqlens,
                             int num_seqs, int64_t total_tokens, int H, int dk, int dv,
                             kda_dtype_t dtype, float *M, float *b, void *workspace,
                             size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_state_compose -- composes affine state maps in order, for every
 * (sequence, head): states[0] = initial_state (or zeros when NULL) and
 *     states[r + 1] = M_r states[r] + b_r,   r = 0 .. n_maps - 1,
 * so states[r] is the state with which segment r starts when segment 0
 * starts from initial_state, and states[n_maps] the state after the last.
 *   M              [n_maps, num_seqs, H, dk, dk] float32 (maps in segment order)
 *   b              [n_maps, num_seqs, H, dk, dv] float32
 *   initial_state  [num_seqs, H, dk, dv] float32, or NULL
 *   states         [n_maps + 1, num_seqs, H, dk, dv] float32 (written)
 * Plain float32 products (no tensor cores); n_maps = 0 copies the start state.
 * All pointers are device pointers; M and b may be a gathered copy of other
 * workers' maps, but must be in this device's memory.
 */
kda_status_t kda_state_compose(const float *M, const float *b, int n_maps, int num_seqs, int H,
                               int dk, int dv, const float *initial_state, float *states,
                               kda_stream_t stream);

/*
 * kda_check_device_status -- synchronises `stream`, reads the status word that
 * kda_chunk_prefill (or kda_chunk_prefill_logdecay) keeps in `workspace`, and
 * returns the first device-side condition the last call recorded:
 *   KDA_OK                  nothing recorded;
 *   KDA_ERR_INVALID_ARG     malformed cu_seqlens (an offset below 0, above
 *                           total_tokens, or below the previous one; that
 *                           sequence was treated as empty), or, for a status
 *                           word passed to kda_decode_tokens or
 *                           kda_state_slots_copy, a slot id >= pool_size;
 *   KDA_ERR_DEVICE_TIMEOUT  a bounded wait inside a kernel expired (the kernel
 *                           let its copies in flight land and returned; that
 *                           call's outputs are incomplete).
 * Returns KDA_ERR_CUDA if the copy or the synchronisation itself fails.
 */
kda_status_t kda_check_device_status(const void *workspace, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
