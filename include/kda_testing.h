/*
 * kda_testing.h -- test support of the GB300 KDA library.  The pages have no
 * counterpart to anything here: it exists so that a test can exercise the
 * library's failure handling without faulting, trapping or hanging a GPU.
 */
#ifndef KDA_GB300_TESTING_H
#define KDA_GB300_TESTING_H

#ifdef __cplusplus
extern "C" {
#endif

/* Bits of kda_testing_expire_next_wait(): the kernels of the tensor-core
 * prefill whose first CTA is to see a wait run out. */
#define KDA_TESTING_FUSED 1        /* one-kernel plan (many chains) */
#define KDA_TESTING_INTRA 2        /* chunk-parallel kernel of the few-chain plans */
#define KDA_TESTING_SEGMENT 4      /* segment maps of the segment-scan plan */
#define KDA_TESTING_SCAN 8         /* the scan over segments */
#define KDA_TESTING_STATE 16       /* state pass of the few-chain plans */

/*
 * kda_testing_expire_next_wait -- arms a simulated wait expiry for the next
 * bf16 d = 128 kda_chunk_prefill or kda_chunk_prefill_logdecay call in this
 * process (any thread, any device), which consumes and clears it.  In each
 * kernel named by `kernels` (a mask of the bits above) that the call
 * launches, CTA 0 waits, with a budget of about a millisecond, on a barrier
 * that nothing arrives at, before its first chunk.  The wait runs out and the
 * kernel takes the same path as a real expired wait: it records
 * KDA_ERR_DEVICE_TIMEOUT in the call's status word, lets its copies and
 * tensor-core operations in flight complete, frees its tensor memory and
 * returns, leaving that call's outputs incomplete and the CUDA context
 * usable.  kernels = 0 disarms.  Not for production use.
 */
void kda_testing_expire_next_wait(int kernels);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_TESTING_H */
