/*
 * pa.h -- libpagedattn: paged KV-cache attention for continuously batched LLM
 * serving, on one GB300 (sm_103a).
 *
 * The problem, as the pages state it (no kernel API is printed there):
 *  - A router batches requests continuously: new requests join and finished
 *    ones leave between forward steps (text-generation-inference
 *    Router/Webserver deep dive, xxmr.cn, sections "Continuous batching" and
 *    "Simple continuous batching").
 *  - Each request's past keys and values are cached; the first pass over a
 *    prompt ("prefill") computes the full causal attention matrix, every later
 *    pass ("decode") only the new token's attention (same page, section
 *    "Prefill, Decode and past key values").  Prompts may be chunked and
 *    concatenated with the running batch (same page, section "the scheduling
 *    loop from the source").
 *  - The cache is paged: the router's block allocator hands out fixed-size
 *    blocks (TGI architecture wiki, data-sketchers.com, section "The Router";
 *    the v3 schema adds "paged attention support", section "Call Flow").
 *  - Servers pass ragged batches with index-pointer arrays (Blitzscale docs,
 *    section "Model": ragged_indptr buffers).
 *  - Warmup fixes the maximum sizes before serving (TGI architecture wiki,
 *    section "Call Flow": warmup(max_input_tokens, max_batch_prefill_tokens,
 *    max_total_tokens, max_batch_size)); pa_workspace_size plays that role.
 *
 * Attention is textbook scaled dot-product softmax attention (the plainest
 * reading; the pages give no formula): query head h reads KV head
 * h / (Hq / Hkv); scale defaults to 1/sqrt(head_dim).
 *
 * ---------------------------------------------------------------------------
 * Conventions shared by every call
 * ---------------------------------------------------------------------------
 *  - Pointers named q, k*, v*, out, *_pool, workspace and every int32 index
 *    array are DEVICE pointers (except the host-side planners:
 *    pa_mixed_prefill_pairs here, and pa_alloc.h / pa_sched.h, whose arrays
 *    are host memory); the caller owns all of them.  The library
 *    calls no cudaMalloc.  The state it does keep, all process-wide:
 *      - the validation flag, the decode split override and the prefill
 *        CTA-pair override (pa_set_validation, pa_set_decode_split,
 *        pa_set_prefill_pairs);
 *      - a thread-local message for the last error;
 *      - per device, created on first use and held until exit: the device
 *        error word and the split-K scratch of pa_decode_noalloc (static
 *        device arrays of the library, 4 bytes and 16 MiB), the side stream
 *        and its two events that pa_mixed_step forks its prefill onto, and
 *        the kernels' shared-memory opt-ins.
 *  - bf16 everywhere for q, k, v, pools and out; indices are int32.
 *  - Layouts (row-major, contiguous):
 *        q        [T][Hq][d]            packed query rows
 *        k_new    [T][Hkv][d]           packed new keys (values alike)
 *        k_pool   [N][Hkv][B][d]        block pool ("HND"); v_pool alike
 *        out      [T][Hq][d]
 *        block_table [S][max_blocks_per_seq]; entries past a sequence's last
 *                 block are never read (any value is allowed there)
 *    Token p of sequence s lives in block block_table[s][p / B], row p % B.
 *  - d (head_dim) in {64, 128}; B (block_size) in {16, 32}; Hq % Hkv == 0;
 *    Hq / Hkv <= 16.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) except pa_check_device_error, and returns PA_OK or an
 *    error code.  Arguments are checked on the host before anything is
 *    enqueued; on an error nothing is enqueued and pa_last_error() describes
 *    it.  Indices read on the device (block_table entries, slots, lengths)
 *    are range-checked by the kernels: an out-of-range value is never
 *    dereferenced, the affected output is left unspecified and a device error
 *    word is set, which pa_check_device_error() reports.
 * ---------------------------------------------------------------------------
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_OK 0
#define PA_ERR_INVALID_ARG 1   /* null pointer, negative size, bad shape */
#define PA_ERR_UNSUPPORTED 2   /* head_dim, block_size or head ratio not built */
#define PA_ERR_WORKSPACE 3     /* workspace missing or smaller than required */
#define PA_ERR_CUDA 4          /* a CUDA call or kernel launch failed */
#define PA_ERR_BAD_INDEX 5     /* device saw an out-of-range block, slot or length */
#define PA_ERR_NO_BLOCKS 6     /* allocator: free list exhausted */
#define PA_ERR_TIMEOUT 7       /* a bounded device wait gave up */

typedef struct {
    int num_q_heads;   /* Hq */
    int num_kv_heads;  /* Hkv; Hq % Hkv == 0 */
    int head_dim;      /* d: 64 or 128 */
    int block_size;    /* B: tokens per block, 16 or 32 */
    int num_blocks;    /* N: blocks in the pool */
    float scale;       /* softmax scale; 0 means 1/sqrt(head_dim) */
} pa_shape_t;

/* Library version (major*10000 + minor*100 + patch). */
int pa_version(void);

/*
 * Workspace bytes needed by pa_decode / pa_decode_append / pa_decode_fp8 /
 * pa_mixed_step for batches of at most max_seqs sequences whose lengths
 * (after the step's append) are at most max_seq_len.  The workspace holds the
 * decode plan (the batch's work items, one per sequence, KV head and split,
 * its counters, 8 bytes per sequence and, when a sequence can split, a merge
 * count per sequence and KV head) and the split-K partial results (fp32); it
 * is owned by
 * the caller, its contents need no initialisation, and two calls whose
 * kernels may overlap on the GPU need two workspaces.  Writes *bytes.
 */
int pa_workspace_size(const pa_shape_t *shape, int max_seqs, int max_seq_len,
                      size_t *bytes);

/*
 * Split-K plan of a decode batch (host side, first step of the path): the
 * tokens per split (a multiple of block_size) and the number of splits of the
 * longest sequence, for num_seqs sequences of at most max_seq_len tokens on
 * the current device (its SM count enters the choice).  This is the finest
 * split the decode uses: its plan launch, which sees the batch's lengths,
 * takes split_tokens * 2^k (k <= 5) instead -- no split at all when even the
 * longest sequence is at most 3/5 of a decode CTA's share of the batch's KV
 * blocks, else the largest k that still leaves at least six work items per
 * decode CTA and no item longer than half of a CTA's share (fewer, longer
 * items cost less while the CTAs stay evenly loaded).  pa_workspace_size
 * covers every such choice.  Sequence s then uses
 * ceil(seq_lens[s] / split) splits (1 if it is empty), one fewer when the
 * last would hold at most split / 8 tokens (they join the split before),
 * never more than max_splits; a sequence with one split writes its output directly; for the
 * others, the split of each (sequence, KV head) that finishes last merges
 * all of its splits' partials, inside the decode kernel.  With
 * pa_set_decode_split in effect the split is exactly the override.
 */
int pa_decode_plan(const pa_shape_t *shape, int num_seqs, int max_seq_len,
                   int *split_tokens, int *max_splits);

/*
 * KV append (router's slot_mapping contract): for every new token i with
 * slot = slot_mapping[i] >= 0, copy k_new[i][h][:] to k_pool[slot/B][h][slot%B][:]
 * and v_new likewise, for all h.  slot < 0 means padding (skipped).  A pure
 * bit copy.  Slots must be distinct (a repeated slot leaves that row
 * unspecified); slot >= N*B is skipped and sets the device error word.
 */
int pa_kv_append(const pa_shape_t *shape, const void *k_new, const void *v_new,
                 const int32_t *slot_mapping, int num_tokens, void *k_pool,
                 void *v_pool, void *stream);

/*
 * Decode attention: one query row per sequence (q [S][Hq][d]) against that
 * sequence's seq_lens[s] cached tokens (counted after the step's append),
 * read through block_table.  out [S][Hq][d].  seq_lens[s] == 0 gives zeros.
 * Long contexts are split into chunks (split-K) whose partial softmax states
 * are merged in the same kernel, by the chunk of each (sequence, KV head)
 * that finishes last; the split is chosen from max_seq_len, which must bound
 * every seq_lens[s] (a longer sequence sets the device error word).  The
 * output is bitwise repeatable: for the same inputs and split it does not
 * depend on the order or the CTA in which the work items run.
 * workspace: at least pa_workspace_size(shape, num_seqs, max_seq_len) bytes.
 */
int pa_decode(const pa_shape_t *shape, const void *q, const void *k_pool,
              const void *v_pool, const int32_t *block_table,
              int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
              int max_seq_len, void *out, void *workspace, size_t ws_bytes,
              void *stream);

/*
 * Decode step with its append fused in: exactly
 *     pa_kv_append(k_new, v_new, slot_mapping, num_seqs rows)
 *     followed by pa_decode(...)
 * (the pages' decode step: the new token's key and value join the cache and
 * the new token attends to all of it, text-generation-inference
 * Router/Webserver deep dive, section "Prefill, Decode and past key
 * values"), in fewer launches: the decode's planning launch (which lists the
 * batch's work items) copies the rows too.  Sequence s brings one new row,
 * k_new[s] / v_new[s] ([S][Hkv][d]), whose slot is slot_mapping[s] (< 0:
 * none; slots distinct, as for pa_kv_append).  A slot past the pool sets the
 * error word and is skipped.  Arguments, workspace, errors and asynchrony as
 * pa_decode and pa_kv_append; bf16 pools only.
 */
int pa_decode_append(const pa_shape_t *shape, const void *q, const void *k_new,
                     const void *v_new, const int32_t *slot_mapping, void *k_pool,
                     void *v_pool, const int32_t *block_table, int max_blocks_per_seq,
                     const int32_t *seq_lens, int num_seqs, int max_seq_len, void *out,
                     void *workspace, size_t ws_bytes, void *stream);

/*
 * Causal prefill over packed prompts: rows [cu_seqlens_q[s], cu_seqlens_q[s+1])
 * of q belong to sequence s.  Row i of sequence s sits at absolute position
 * p0 + i and attends to keys 0 .. p0 + i (bottom-right causal alignment).
 *  - block_table == NULL: dense form.  k, v are the packed new keys/values
 *    [T][Hkv][d]; key j of sequence s is row cu_seqlens_q[s] + j; prefix_lens
 *    must be NULL (p0 = 0).
 *  - block_table != NULL: paged form.  k, v are the pools; every key of the
 *    sequence, prefix and new rows alike, is read through block_table (the
 *    caller appended the new rows first); p0 = prefix_lens[s] (NULL = 0).
 * num_tokens is the number of rows of q and out (and of k, v in the dense
 * form); cu_seqlens_q[num_seqs] must not exceed it.  max_q_len bounds every
 * prompt length (a longer one sets the error word and is not computed).
 * Runs on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
 */
int pa_prefill(const pa_shape_t *shape, const void *q, const void *k,
               const void *v, const int32_t *cu_seqlens_q,
               const int32_t *prefix_lens, const int32_t *block_table,
               int max_blocks_per_seq, int num_seqs, int num_tokens,
               int max_q_len, void *out, void *stream);

/*
 * One continuous-batching step (prefill chunks merged into the running batch):
 *   1. append all num_tokens new rows (k_new/v_new) at slot_mapping;
 *   2. decode attention for sequences [0, num_decode), which own exactly one
 *      query row each (q_start_loc[s+1] - q_start_loc[s] == 1);
 *   3. causal prefill (paged form, prefix = seq_lens[s] - n_s) for sequences
 *      [num_decode, num_seqs).
 * Steps 2 and 3 run concurrently: the decode rows' append goes with the
 * decode (as pa_decode_append) on `stream`; the prompt rows' append and the
 * prefill go to a higher-priority stream owned by the library (one per
 * device, created on first use), forked from `stream` and joined back into it
 * with events, so work enqueued on `stream` afterwards sees the whole step.
 * Blocks that one sequence writes in the step must not be read by another
 * (the allocator's ownership rule).
 * q_start_loc [num_seqs+1] packs the rows of q/k_new/v_new/out; seq_lens counts
 * tokens after the append.  max_seq_len bounds seq_lens, max_q_len bounds the
 * prefill rows per sequence.  workspace as for pa_decode.
 */
int pa_mixed_step(const pa_shape_t *shape, const void *q, const void *k_new,
                  const void *v_new, const int32_t *q_start_loc,
                  const int32_t *seq_lens, const int32_t *slot_mapping,
                  const int32_t *block_table, int max_blocks_per_seq,
                  int num_seqs, int num_decode, int num_tokens, int max_seq_len,
                  int max_q_len, void *k_pool, void *v_pool, void *out,
                  void *workspace, size_t ws_bytes, void *stream);

/*
 * pa_mixed_step with the GPU divided between its two halves (no counterpart
 * in the pages, which leave the placement of a mixed batch's work to the
 * hardware).  The prefill runs on prefill_pairs CTA pairs (2 * prefill_pairs
 * SMs) and the decode on the SMs left over, so both start at once and neither
 * waits for the other to drain.  prefill_pairs == 0 is exactly pa_mixed_step
 * (both halves spread over the whole GPU, the prefill placed first).  The
 * split applies only when both halves have work, the prefill runs the
 * tensor-core pair kernel (head_dim 128) and 2 * prefill_pairs is below the
 * device's SM count; otherwise the step runs as pa_mixed_step.  The appended
 * pools and the prefill rows are bit for bit pa_mixed_step's (a prefill work
 * unit is summed the same way on any pair); so are the decode rows when both
 * use the same split-K factor (pa_set_decode_split), and otherwise they agree
 * within the decode's tolerance: the plan chooses the factor for the SMs the
 * decode gets.
 * A negative count is PA_ERR_INVALID_ARG.  pa_mixed_prefill_pairs gives a
 * count for a step.
 */
int pa_mixed_step_split(const pa_shape_t *shape, const void *q, const void *k_new,
                        const void *v_new, const int32_t *q_start_loc,
                        const int32_t *seq_lens, const int32_t *slot_mapping,
                        const int32_t *block_table, int max_blocks_per_seq,
                        int num_seqs, int num_decode, int num_tokens,
                        int max_seq_len, int max_q_len, void *k_pool,
                        void *v_pool, void *out, void *workspace,
                        size_t ws_bytes, void *stream, int prefill_pairs);

/*
 * The prefill pair count for pa_mixed_step_split, chosen from host-known
 * lengths so that the two halves take about the same time: decode_lens
 * [num_decode] are the decode sequences' lengths after the append,
 * prompt_rows [num_prompts] the new rows of each prompt and prefix_lens
 * [num_prompts] (NULL = 0) the tokens already cached before them.  The cost
 * model (fit to timings on GB300): a prefill work unit costs about 1 us plus
 * 2 us per 128-key tile on one CTA pair; the decode streams about 50 GB/s of
 * K/V per SM.  num_sms <= 0 takes the current device's SM count (and then
 * needs a device); a positive value is used as given (no device needed).
 * Writes 0 to *pairs (no split) when either half is empty or head_dim is not
 * 128, else a count in [1, num_sms / 2 - 1].  All arrays are host memory.
 */
int pa_mixed_prefill_pairs(const pa_shape_t *shape, const int32_t *decode_lens,
                           int num_decode, const int32_t *prompt_rows,
                           const int32_t *prefix_lens, int num_prompts,
                           int num_sms, int *pairs);

/*
 * Decode without a caller workspace (no counterpart in the pages: an addition
 * for callers that cannot allocate device memory, e.g. code running inside a
 * pre-planned serving loop whose memory is fixed at start-up, or a host that
 * forbids allocation after warm-up).  Same computation, arguments and layouts
 * as pa_decode minus the workspace: the split-K partials go to a buffer that
 * lives inside this library, PA_NOALLOC_SCRATCH_BYTES (16 MiB) of device
 * memory on every GPU that loads it, held until the process exits.
 *  - Calls nothing that allocates (no cudaMalloc, no cudaFree).
 *  - The first call on a device looks up that device's copy of the buffer
 *    (cudaGetSymbolAddress, with the device current); make that first call
 *    before any stream capture.
 *  - A batch whose partials need more than the buffer holds is rejected
 *    with PA_ERR_WORKSPACE before anything is enqueued; use pa_decode then.
 *    The exact need, with max_splits from pa_decode_plan(shape, num_seqs,
 *    max_seq_len), is P + num_seqs * (max_splits * Hkv * 16 + 8) + 16 + C
 *    bytes, where P = num_seqs * Hq * max_splits * (d + 2) * 4 rounded up to
 *    a multiple of 16 and C = num_seqs * Hkv * 4 (P = C = 0 when max_splits
 *    is 1).  pa_workspace_size(shape, num_seqs,
 *    max_seq_len) is an upper bound of that need (it assumes the shortest
 *    split), so a batch with pa_workspace_size <= PA_NOALLOC_SCRATCH_BYTES is
 *    always accepted, and larger ones often are.
 *  - All calls share the one buffer and nothing in it needs clearing (every
 *    partial is written before it is read, and each call's plan launch sets
 *    its merge counts to zero); calls whose kernels overlap on the GPU
 *    (different streams, no ordering) race on it.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
int pa_decode_noalloc(const pa_shape_t *shape, const void *q, const void *k_pool,
                      const void *v_pool, const int32_t *block_table,
                      int max_blocks_per_seq, const int32_t *seq_lens,
                      int num_seqs, int max_seq_len, void *out, void *stream);

/*
 * fp8 KV cache: pools of e4m3 codes (OCP FP8 "e4m3fn": 1 sign, 4 exponent
 * bits with bias 7, 3 significand bits, largest finite 448, no infinities),
 * same [N][Hkv][B][d] layout with one byte per element, and one float scale
 * per KV head for K and one for V (device arrays [Hkv]): a value x of KV head
 * h is stored as the code of x / scale[h] (float division, nearest even,
 * saturating at +-448) and read as code * scale[h].  The pages name fp8 only
 * as a serving option (flashinfer's FP8 switch; a quantize flag), so this is
 * the plainest reading of an fp8 cache with per-head scales.
 *
 * pa_kv_append_fp8: pa_kv_append into fp8 pools (same slot rules and error
 * behaviour).
 * pa_decode_fp8: pa_decode over fp8 pools (head_dim 64 or 128); same
 * workspace (pa_workspace_size), split-K plan, errors and asynchrony.  q and
 * out stay bf16.
 */
int pa_kv_append_fp8(const pa_shape_t *shape, const void *k_new, const void *v_new,
                     const int32_t *slot_mapping, int num_tokens, const float *k_scale,
                     const float *v_scale, void *k_pool, void *v_pool, void *stream);
int pa_decode_fp8(const pa_shape_t *shape, const void *q, const void *k_pool, const void *v_pool,
                  const float *k_scale, const float *v_scale, const int32_t *block_table,
                  int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs, int max_seq_len,
                  void *out, void *workspace, size_t ws_bytes, void *stream);

/*
 * Rotary position embedding of a step's new tokens, fused with their KV
 * append (the position-encoding mode the pages' flashinfer build compiles in,
 * Blitzscale docs, section "Build"; the rotation of RoFormer with the Llama /
 * GPT-NeoX pairing): for token t at position p = positions[t], every query
 * head row and key head row x (length d) becomes, for i < d/2 and
 * f_i = theta^(-2i/d),
 *     y[i] = x[i] cos(p f_i) - x[i+d/2] sin(p f_i),
 *     y[i+d/2] = x[i+d/2] cos(p f_i) + x[i] sin(p f_i)   (rounded to bf16).
 * q [T][Hq][d] -> q_out [T][Hq][d] (q_out == q rotates in place); the rotated
 * k [T][Hkv][d] and v (unchanged) go to slot_mapping[t] of the pools exactly
 * as pa_kv_append writes them (slot < 0: no append for that token; its query
 * is still rotated).  Decode and prefill then take q_out and the pools as
 * usual.  rope_theta: 0 means 10000.  A negative position or a slot past the
 * pool sets the error word and that token (resp. its append) is skipped.
 * Returns PA_ERR_INVALID_ARG for NULL / misaligned pointers, num_tokens < 0
 * or a negative or infinite rope_theta; asynchronous on `stream`; the caller owns every
 * buffer.
 */
int pa_rope_append(const pa_shape_t *shape, const void *q, const void *k_new, const void *v_new,
                   const int32_t *positions, const int32_t *slot_mapping, int num_tokens,
                   float rope_theta, void *q_out, void *k_pool, void *v_pool, void *stream);

/*
 * Copy whole KV blocks between two pools of the same shape (num_kv_heads,
 * block_size, head_dim; shape->num_blocks is not used here):
 *     dst_k[dst_ids[i]] = src_k[src_ids[i]],  dst_v alike,  0 <= i < num_pairs
 * (K and V, every KV head of the block).  The cache's GPU region and CPU region
 * and the migration of a batch's cache between replicas (Blitzscale docs,
 * sections "CacheManager" and "migration_queue") need this: within one pool it
 * forks a sequence (copy-on-write), between device pools it migrates blocks,
 * and with one side in pinned host memory (cudaHostAlloc, torch pin_memory) it
 * swaps blocks out and back in -- the GPU reads or writes that memory through
 * its device alias.  src_num_blocks / dst_num_blocks are the pools' sizes in
 * blocks; an id outside them sets the device error word and that pair is
 * skipped.  The id arrays are device memory.  A destination block must not
 * also be a source, nor appear twice, in one call (the copies run in no fixed
 * order).  Pools must be 16-byte aligned.  Returns PA_ERR_INVALID_ARG for a
 * NULL, misaligned or pageable (not GPU-visible) pointer or a negative size,
 * PA_ERR_UNSUPPORTED for a shape the library does not take; num_pairs == 0 is
 * a no-op.  Asynchronous on `stream`; the caller owns every buffer.
 */
int pa_copy_blocks(const pa_shape_t *shape, const void *src_k, const void *src_v,
                   int src_num_blocks, void *dst_k, void *dst_v, int dst_num_blocks,
                   const int32_t *src_ids, const int32_t *dst_ids, int num_pairs,
                   void *stream);

/*
 * Validation mode (off by default, process-wide).  When on, each call first
 * runs a bounds-checking pass over block_table/slot_mapping/lengths; if it
 * finds a bad index it sets the device error word and the call's other
 * kernels return without touching their outputs.
 */
int pa_set_validation(int on);

/*
 * Synchronises `stream`, reads and clears the device error word of the
 * current device.  Returns PA_OK, PA_ERR_BAD_INDEX, PA_ERR_TIMEOUT or
 * PA_ERR_CUDA.
 */
int pa_check_device_error(void *stream);

/* Message for the last error returned on the calling thread ("" if none). */
const char *pa_last_error(void);

/*
 * Decode split override (tokens per split; a multiple of block_size), for
 * tests comparing split and unsplit results: the decode then uses exactly this
 * split.  0 restores the automatic choice.
 */
int pa_set_decode_split(int tokens);

/*
 * Prefill CTA-pair count override, for tests: with few pairs each pair walks
 * many work units in turn, so the hand-offs between consecutive units (Q
 * buffers, K/V ring stages, output staging) are exercised on every launch.
 * pairs = 0 restores the automatic choice (one pair per two SMs, at most one
 * per work unit); larger values are capped at that.  Returns PA_OK, or
 * PA_ERR_INVALID_ARG for pairs < 0.  Applies to pa_prefill and the prefill
 * part of pa_mixed_step.
 */
int pa_set_prefill_pairs(int pairs);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
