// pa_internal.h -- host-side declarations shared by the libpagedattn sources.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace pa {

// Dynamic shared memory above 48 KB needs an opt-in per kernel and per
// device (function attributes belong to the device's context).  `done` holds
// one bit per device ordinal (< 64) already opted in; a higher ordinal is
// set on every launch.  Concurrent first launches may both set the attribute,
// which is idempotent.
inline cudaError_t opt_in_smem(const void *kernel, int bytes, std::atomic<unsigned long long> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// ------------------------------------------------------------- decode ------
struct DecodeArgs {
    const __nv_bfloat16 *q;      // [S][Hq][d]
    const int32_t *block_table;  // [S][max_blocks]
    const int32_t *seq_lens;     // [S], tokens after the append
    __nv_bfloat16 *out;          // [S][Hq][d]
    float *part_acc;             // [S][Hq][max_splits][d], unnormalised sums
    float *part_ml;              // [S][Hq][max_splits][2]: (max, sum) in log2 units
    int *err;                    // device error word
    int num_seqs, num_q_heads, num_kv_heads, group, num_blocks, max_blocks;
    int split_tokens, max_splits, max_seq_len;
    // split_adapt: the plan launch may take split_tokens * 2^k instead (never
    // more splits than max_splits allows), from the batch's actual lengths;
    // the split it uses is plan_count[1].  num_ctas: the decode kernel's grid.
    int split_adapt, num_ctas;
    int check_err_first;         // validation mode: skip work if *err != 0
    float scale_log2;            // softmax scale * log2(e)
    const float *k_scale, *v_scale;  // fp8 pools: [Hkv] scales (value = code * scale); else null
    // Fused append (pa_decode_append; null otherwise): row s of k_new / v_new
    // [S][Hkv][d] goes to slot_mapping[s] of the pools, in the plan launch.
    const __nv_bfloat16 *k_new, *v_new;
    const int32_t *slot_mapping;
    __nv_bfloat16 *k_pool, *v_pool;
    long long num_slots;
    // The plan (first step of the path): decode_plan_kernel writes the work
    // items -- (sequence, KV head, split, length) -- into the workspace,
    // plan_count[0] = their number and plan_count[1] = the tokens per split.
    int4 *plan_items;
    int *plan_count;
    int2 *plan_seq;  // the plan's per-sequence scratch
    // [S][Hkv] splits of each (sequence, KV head) done (null when nothing can
    // split): set to zero by the plan launch; the split that brings it to the
    // sequence's split count merges the partials.
    int *merge_cnt;
};

// Tokens per split-K chunk chosen for a decode batch (multiple of block_size).
int decode_split_tokens(int num_seqs, int num_kv_heads, int max_seq_len, int block_size,
                        int num_sms, int override_tokens);
int decode_max_splits(int max_seq_len, int split_tokens);
// Workspace of one decode call: split partials (when any sequence splits),
// the plan's work items and its two counters.
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_splits);
// Where the plan lives inside that workspace.
void decode_plan_layout(void *ws, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_splits,
                        int4 **items, int **count, int2 **seq, int **merge_cnt);

// The plan launch (with the fused append's CTAs), then the persistent decode
// kernel (which also merges the splits), both on `stream`.
// tm_q: q as rows [S * Hq][d] bf16, boxes of 64 columns x G rows, 128-byte swizzle.
cudaError_t launch_decode(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          const DecodeArgs &a, int head_dim, int block_size, int num_sms, cudaStream_t stream,
                          bool fp8 = false);

// ------------------------------------------------------------- append ------
cudaError_t launch_kv_append(const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new,
                             const int32_t *slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, __nv_bfloat16 *k_pool,
                             __nv_bfloat16 *v_pool, int *err, int check_err_first, int num_sms,
                             cudaStream_t stream);

// Whole-block copies between pools (device or pinned host memory).
// Append with quantisation to e4m3 codes (one scale per KV head).
cudaError_t launch_kv_append_fp8(const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new,
                                 const int32_t *slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, const float *k_scale, const float *v_scale,
                                 uint8_t *k_pool, uint8_t *v_pool, int *err, int check_err_first,
                                 cudaStream_t stream);

// Rotary embedding of a step's new tokens fused with their KV append.
struct RopeArgs {
    const __nv_bfloat16 *q, *k_new, *v_new;
    const int32_t *positions, *slot_mapping;
    __nv_bfloat16 *q_out, *k_pool, *v_pool;
    int *err;
    int num_tokens, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
    int check_err_first;
    // turn[i]: f_i / (2 pi) as a 64-bit fixed-point fraction of a turn, with
    // f_i = theta^(-2i/d), i < d/2; position p's angle is p * turn[i] mod 2^64
    unsigned long long turn[64];
};
cudaError_t launch_rope_append(const RopeArgs &a, int num_sms, cudaStream_t stream);

cudaError_t launch_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int32_t *src_ids, const int32_t *dst_ids, int num_pairs,
                               long long block_bytes, int src_blocks, int dst_blocks, int num_sms, int *err,
                               int check_err_first, cudaStream_t stream);

// ------------------------------------------------------------ prefill ------
struct PrefillArgs {
    const int32_t *cu_seqlens;   // [S+1] query rows of each sequence (in q/out)
    const int32_t *prefix_lens;  // [S] or null (0)
    const int32_t *block_table;  // paged form: [S][max_blocks]; null = dense form
    const int32_t *seq_lens;     // mixed step: [S] tokens after append (prefix = len - n); or null
    __nv_bfloat16 *out;          // [T][Hq][d]
    int *err;
    int num_seqs, num_q_heads, num_kv_heads, group, num_blocks, max_blocks;
    int num_tokens;              // rows of q/out (and of packed k/v in the dense form)
    int max_q_len, num_q_tiles;
    int check_err_first;
    float scale_log2;
    int num_sms;                 // persistent kernels size their grid from it
};

cudaError_t launch_prefill(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                           const CUtensorMap &tm_v, const PrefillArgs &a, int head_dim,
                           int block_size, cudaStream_t stream);

// head_dim 128 on CTA pairs (M = 256 tcgen05.mma).  Dense form: tm_k boxes
// are 64 rows (each CTA of the pair loads half of a 128-key tile).
// tm_o: out as rows [T][Hq][d], boxes of 64 columns x 1 head x 32 rows.
cudaError_t launch_prefill_pair(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                const CUtensorMap &tm_v, const CUtensorMap &tm_o, const PrefillArgs &a,
                                int block_size, cudaStream_t stream);

// --------------------------------------------------------- validation ------
struct CheckArgs {
    const int32_t *slot_mapping;  // [T] or null
    int num_tokens;
    const int32_t *block_table;   // [S][max_blocks] or null
    const int32_t *seq_lens;      // [S] or null
    const int32_t *cu_seqlens;    // [S+1] or null
    const int32_t *prefix_lens;   // [S] or null
    int num_seqs, max_blocks, block_size, num_blocks, max_seq_len, max_q_len;
    int decode_rows;              // mixed step: sequences [0, decode_rows) own query row s
    int *err;
};
cudaError_t launch_index_check(const CheckArgs &a, cudaStream_t stream);

}  // namespace pa
