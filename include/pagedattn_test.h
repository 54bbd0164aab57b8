/*
 * pagedattn_test: test and tuning hooks of libpagedattn.so.
 *
 * These are exported by the same library as include/pagedattn.h but are not
 * part of the production interface: they change how the calling host
 * thread's next calls run (an injected wait that must time out, or the
 * choice of prefill kernel), for the library's own failure-detection tests
 * and kernel comparisons. Production callers include pagedattn.h only.
 */
#ifndef PAGEDATTN_TEST_H
#define PAGEDATTN_TEST_H

#include "pagedattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Test support for failure detection. The next call made by the calling
 * host thread that runs the split-KV kernel (pa_decode, pa_decode_noalloc,
 * pa_decode_dense, pa_attention routed to decode) runs one extra wait, in
 * its first block, on a barrier that nothing ever arrives at. That wait runs
 * out after its bounded limit (about one second), records PA_DEVERR_TIMEOUT
 * in the device error word, and the
 * kernel then finishes normally with the correct result. Nothing faults or
 * hangs; the CUDA context stays usable.
 */
void pa_debug_arm_wait_timeout(void);

/*
 * Test and tuning support: which tensor-core prefill kernel the calling host
 * thread's pa_prefill / pa_attention calls use (head_dim 128 and pages of 8
 * tokens or more; head_dim 64 and smaller pages always take the two-head
 * kernel).
 *   0  automatic (the default): as 2, except that a group size that is odd
 *      with fewer (request, head pair, query tile) items than SMs takes 1;
 *   1  one query head per block;
 *   2  two query heads of one KV group per block when the group size
 *      (num_q_heads / num_kv_heads) is at least 2; with an odd group size
 *      the last pair of each group computes its last head twice and writes
 *      it once. A group of 1 takes 1;
 *   4  as 2 on a grid of two thirds of the (request, head pair, query
 *      tile) items, so that a third of the blocks hold one item and the rest
 *      two; pa_attention given a prefill workspace then balances them with
 *      tail pieces (a block runs the last tiles of another's second item
 *      first and leaves their state, which that block merges), as it does by
 *      itself with 1 to 2 items per SM. For tests of the pieces on small
 *      shapes;
 *   5  as 4, with the receiving blocks running the piece after their own
 *      item, so that the donors usually finish first and the receiving
 *      blocks write the merged rows (the path taken when a receiving block
 *      starts late).
 * Settings 1 and 2 also hold for pa_prefill_split and for pa_attention given
 * a prefill workspace (the workspace is then not used). Any other value is
 * taken as 0. Returns the previous setting. Results agree
 * with the oracle under every setting; only the speed differs.
 */
int pa_debug_prefill_variant(int variant);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_TEST_H */
