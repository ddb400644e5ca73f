/*
 * pa_alloc.h -- host-side block allocator for the paged KV pool.
 *
 * The router hands out fixed-size KV-cache blocks with a block allocator and
 * keeps count of the blocks in use (TGI architecture wiki, data-sketchers.com,
 * section "The Router"; Blitzscale docs, section on the decode replica's
 * "used blocks" accounting); blocks go back to the free list when a request
 * finishes or is filtered out of the batch (text-generation-inference
 * Router/Webserver deep dive, section "Simple continuous batching").
 *
 * This allocator produces the index inputs of the device calls in pa.h:
 * block_table rows and slot_mapping.  It is plain host code (no CUDA calls),
 * not thread-safe (one owner, like the router's scheduling loop).
 *
 * Free list: a stack.  Never-used blocks are handed out in `initial_order`
 * (NULL = 0, 1, 2, ...); a released sequence pushes its blocks in table
 * order, so the block it owned last is the first to be reused.
 */
#ifndef PA_ALLOC_H_
#define PA_ALLOC_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_allocator pa_block_allocator;

/* NULL on bad arguments (num_blocks <= 0, block_size <= 0, initial_order not
 * a permutation of [0, num_blocks)) or out of host memory. */
pa_block_allocator *pa_alloc_create(int num_blocks, int block_size,
                                    const int32_t *initial_order);
void pa_alloc_destroy(pa_block_allocator *a);

/* Make sequence seq_id own ceil(num_tokens / block_size) blocks, taking the
 * missing ones from the free list (nothing changes on failure).
 * Returns PA_OK, PA_ERR_NO_BLOCKS or PA_ERR_INVALID_ARG. */
int pa_alloc_ensure(pa_block_allocator *a, int64_t seq_id, int num_tokens);

/* Return all blocks of seq_id to the free list.  PA_ERR_INVALID_ARG if the
 * sequence owns nothing. */
int pa_alloc_release(pa_block_allocator *a, int64_t seq_id);

int pa_alloc_num_free(const pa_block_allocator *a);
/* Blocks owned by seq_id (0 if unknown). */
int pa_alloc_num_blocks_of(const pa_block_allocator *a, int64_t seq_id);

/* table_out[r][j] = j-th block of seq_ids[r] for j < its block count, `fill`
 * after that; width columns per row (row-major int32).  PA_ERR_INVALID_ARG if
 * a sequence is unknown or owns more than `width` blocks. */
int pa_alloc_block_table(const pa_block_allocator *a, const int64_t *seq_ids,
                         int num_seqs, int width, int32_t fill,
                         int32_t *table_out);

/* Slots of the new tokens of one step: sequence seq_ids[r] gets n_new[r]
 * tokens at positions total_after[r] - n_new[r] .. total_after[r] - 1, packed
 * in order; slot = block * block_size + position % block_size.
 * PA_ERR_INVALID_ARG if a position is not covered by the sequence's blocks. */
int pa_alloc_slot_mapping(const pa_block_allocator *a, const int64_t *seq_ids,
                          const int32_t *n_new, const int32_t *total_after,
                          int num_seqs, int32_t *slots_out);

#ifdef __cplusplus
}
#endif

#endif /* PA_ALLOC_H_ */
