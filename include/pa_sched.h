/*
 * pa_sched.h -- the host continuous-batching scheduler that drives the
 * device calls of pa.h step by step.
 *
 * What it follows (text-generation-inference Router/Webserver deep dive,
 * section "Scheduling loop from the source"; its launcher defaults in the TGI
 * architecture wiki, section "Router"): the loop keeps taking the next batch
 * from a FIFO queue, with a token budget for the running batch and a token
 * budget for one prefill; "max_waiting_tokens" forces admission once that
 * many steps have passed without one, however small the new batch;
 * "waiting_served_ratio" sets the least number of waiting requests worth
 * pausing the running batch for (running size x ratio); with prefill
 * chunking those two are ignored and new prompts are concatenated with the
 * running batch's step and prefilled together, a prompt split over steps
 * when it does not fit.
 *
 * One step here is one pa_mixed_step: every running request whose prompt is
 * done decodes one token (its last generated token is appended), and
 * admitted prompts (or chunks) are prefilled in the same launch.  Readings
 * where the pages are silent:
 *   - a request's reservation against max_batch_total_tokens is the
 *     block-aligned size of prompt + max_new_tokens;
 *   - admission takes queued requests strictly in order and stops at the
 *     first that does not fit (no skipping);
 *   - without chunking a request's whole prompt is one prefill, and the
 *     batch admitted must have at least min_size requests (unless the wait
 *     is exceeded or nothing is running);
 *   - with chunking, a step's prefill rows plus its decode rows stay within
 *     max_batch_prefill_tokens; partially prefilled prompts go first;
 *   - a request produces its first token when its prompt is done and leaves
 *     when it has produced max_new_tokens (the last one is never appended).
 *
 * Host code, no CUDA calls, not thread-safe (one owner).  Every function
 * returns PA_OK or a PA_ERR_* code of pa.h.
 */
#ifndef PA_SCHED_H_
#define PA_SCHED_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int max_batch_prefill_tokens; /* rows one step may prefill (default 4096)        */
    int max_batch_total_tokens;   /* running batch's reservation cap (0: the pool)   */
    int max_waiting_tokens;       /* steps without admission before it is forced (20) */
    float waiting_served_ratio;   /* least admitted batch = running x ratio (1.2)     */
    int max_batch_size;           /* running requests cap (0: none)                   */
    int chunking;                 /* 1: prompts may be split over steps               */
    int max_input_tokens;         /* request validation (1024)                        */
    int max_total_tokens;         /* prompt + max_new_tokens limit (2048)             */
} pa_sched_params;

typedef struct pa_scheduler pa_scheduler;

/* NULL on bad arguments.  The scheduler owns a block allocator over
 * num_blocks blocks of block_size tokens (handed out 0, 1, 2, ... first). */
pa_scheduler *pa_sched_create(const pa_sched_params *params, int num_blocks, int block_size);
void pa_sched_destroy(pa_scheduler *s);

/* Queue a request: input_tokens prompt rows, up to max_new_tokens generated.
 * PA_ERR_INVALID_ARG for an id already known, input_tokens < 1,
 * max_new_tokens < 1, sizes past max_input_tokens / max_total_tokens, a
 * reservation past max_batch_total_tokens, or (without chunking) a prompt
 * longer than max_batch_prefill_tokens. */
int pa_sched_submit(pa_scheduler *s, int64_t request_id, int input_tokens, int max_new_tokens);

/* The client left: drop the request from the queue or the running batch and
 * free its blocks.  PA_ERR_INVALID_ARG if unknown. */
int pa_sched_cancel(pa_scheduler *s, int64_t request_id);

/* Plan the next step into caller buffers: seq_ids[S], q_start_loc[S+1],
 * seq_lens[S] (context after the step's append), block_table [S][width]
 * (-1 past a sequence's blocks), slot_mapping[T]; the first *num_decode
 * sequences have one row each.  *num_seqs = 0: nothing to run.  Sizes past
 * max_seqs / max_tokens / width give PA_ERR_INVALID_ARG and change nothing.
 * A planned step must be committed before the next plan. */
int pa_sched_plan(pa_scheduler *s, int max_seqs, int max_tokens, int width, int64_t *seq_ids,
                  int32_t *q_start_loc, int32_t *seq_lens, int32_t *block_table, int32_t *slot_mapping,
                  int *num_seqs, int *num_decode, int *num_tokens);

/* The planned step ran: advance every planned request; the ones that have
 * produced all their tokens leave (blocks freed) and are listed in
 * finished_out (up to max_finished; *num_finished counts all). */
int pa_sched_commit(pa_scheduler *s, int64_t *finished_out, int max_finished, int *num_finished);

/* Queue length, running requests, free blocks, steps since the last admission. */
int pa_sched_stats(const pa_scheduler *s, int *queued, int *running, int *free_blocks, int *waiting_steps);

#ifdef __cplusplus
}
#endif

#endif /* PA_SCHED_H_ */
