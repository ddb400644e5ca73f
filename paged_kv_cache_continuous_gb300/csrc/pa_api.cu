// pa_api.cu -- the C ABI of libpagedattn: argument checks, TMA tensor maps,
// split planning and kernel launches.  Nothing here allocates device memory;
// the caller owns every buffer (see include/pa.h for the contract).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

using namespace pa;

// A named NVTX range around each public call that enqueues GPU work, so a
// profiler's timeline shows which library call launched which kernels (free
// when no tool is attached: NVTX is header-only and calls into a tool only
// when one is injected).
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};

thread_local std::string t_last_error;
std::atomic<int> g_validation{0};
std::atomic<int> g_split_override{0};
std::atomic<int> g_pairs_override{0};  // prefill CTA pairs (0: automatic)

// Device error word: kernels record PA_ERR_BAD_INDEX / PA_ERR_TIMEOUT here
// instead of trapping; pa_check_device_error reads and clears it.
__device__ int g_error_word;

int fail(int code, const std::string &msg) {
    t_last_error = msg;
    return code;
}

int ok() {
    t_last_error.clear();
    return PA_OK;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(PA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct DevState {
    int *err = nullptr;
    int num_sms = 0;
    bool init = false;
};
std::mutex g_mu;
DevState g_dev[64];

int dev_state(DevState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PA_ERR_CUDA, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DevState &d = g_dev[dev];
    if (!d.init) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        d.err = static_cast<int *>(p);
        d.init = true;
    }
    *out = &d;
    return PA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const pa_shape_t *sh) {
    if (!sh) return fail(PA_ERR_INVALID_ARG, "shape is NULL");
    if (sh->num_q_heads <= 0 || sh->num_kv_heads <= 0 || sh->num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "head counts and num_blocks must be positive");
    if (sh->head_dim != 64 && sh->head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (sh->block_size != 16 && sh->block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 16 or 32");
    if (sh->num_q_heads % sh->num_kv_heads != 0)
        return fail(PA_ERR_UNSUPPORTED, "num_q_heads must be a multiple of num_kv_heads");
    if (sh->num_q_heads / sh->num_kv_heads > 16)
        return fail(PA_ERR_UNSUPPORTED, "at most 16 query heads per KV head");
    if (sh->num_kv_heads > 65535 || sh->num_q_heads > 65535)
        return fail(PA_ERR_UNSUPPORTED, "too many heads");
    if (!(sh->scale >= 0.f) || std::isinf(sh->scale))
        return fail(PA_ERR_INVALID_ARG, "scale must be finite and >= 0");
    const long long rows = (long long)sh->num_blocks * sh->num_kv_heads * sh->block_size;
    if (rows > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "pool too large (rows exceed 2^31)");
    return PA_OK;
}

float scale_log2(const pa_shape_t *sh) {
    const double sc = sh->scale > 0.f ? (double)sh->scale : 1.0 / std::sqrt((double)sh->head_dim);
    return (float)(sc * 1.4426950408889634);  // log2(e)
}

// ------------------------------------------------------------ tensor maps --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Pool viewed as [N*Hkv*B rows][d] bf16; box = 64 columns x B rows (one KV
// block of one head, one 128-byte half of each row), 128-byte swizzle.
int make_pool_map(CUtensorMap *m, const void *pool, const pa_shape_t *sh) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)sh->head_dim,
                                (cuuint64_t)sh->num_blocks * sh->num_kv_heads * sh->block_size};
    const cuuint64_t strides[1] = {(cuuint64_t)sh->head_dim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)sh->block_size};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(pool) failed");
    return PA_OK;
}

// fp8 pool [N][Hkv][B][d] of e4m3 codes as 2-D rows of d bytes; box = d
// bytes (one 128-byte swizzle row for d = 128) x one block.
int make_pool_map_u8(CUtensorMap *m, const void *pool, const pa_shape_t *sh) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    // Rows of 128 codes: one token's row for d = 128, two tokens' rows for
    // d = 64 (the decode kernel addresses token t at row t / 2, half t % 2).
    const int per_row = 128 / sh->head_dim;
    const cuuint64_t dims[2] = {128, (cuuint64_t)sh->num_blocks * sh->num_kv_heads * sh->block_size / per_row};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, (cuuint32_t)(sh->block_size / per_row)};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(fp8 pool) failed");
    return PA_OK;
}

// Packed rows [T][H][d] bf16; box = 64 columns x 1 head x box_rows rows.
int make_rows_map(CUtensorMap *m, const void *base, int head_dim, int heads, long long rows,
                  int box_rows = 128) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(rows) failed");
    return PA_OK;
}

// q of a decode batch as rows [S * Hq][d] bf16; box = 64 columns x G rows
// (the query heads of one KV head), 128-byte swizzle.
int make_qgroup_map(CUtensorMap *m, const void *q, const pa_shape_t *sh, int num_seqs) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)sh->head_dim, (cuuint64_t)num_seqs * sh->num_q_heads};
    const cuuint64_t strides[1] = {(cuuint64_t)sh->head_dim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(sh->num_q_heads / sh->num_kv_heads)};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed");
    return PA_OK;
}

int split_min_tokens(int block_size) {
    const int ov = g_split_override.load();
    const int base = ov > 0 ? ov : 256;
    return ((base + block_size - 1) / block_size) * block_size;
}

// ---------------------------------------------------------- the three ops --
int do_append(const pa_shape_t *sh, const void *k_new, const void *v_new, const int32_t *slots,
              int num_tokens, void *k_pool, void *v_pool, cudaStream_t st, DevState *d, int check_first) {
    if ((long long)num_tokens * sh->num_kv_heads * (sh->head_dim / 8) > 0x7fffffffLL - 4096)
        return fail(PA_ERR_UNSUPPORTED, "append: num_tokens * num_kv_heads * head_dim / 8 must be below 2^31");
    cudaError_t e = launch_kv_append(static_cast<const __nv_bfloat16 *>(k_new),
                                     static_cast<const __nv_bfloat16 *>(v_new), slots, num_tokens,
                                     sh->num_kv_heads, sh->head_dim, sh->block_size, sh->num_blocks,
                                     static_cast<__nv_bfloat16 *>(k_pool), static_cast<__nv_bfloat16 *>(v_pool),
                                     d->err, check_first, d->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    return PA_OK;
}

int do_decode(const pa_shape_t *sh, const void *q, const void *k_pool, const void *v_pool,
              const int32_t *block_table, int max_blocks, const int32_t *seq_lens, int num_seqs,
              int max_seq_len, void *out, void *ws, size_t ws_bytes, cudaStream_t st, DevState *d,
              int check_first, const float *k_scale = nullptr, const float *v_scale = nullptr,
              int split_planned = 0, const void *k_new = nullptr, const void *v_new = nullptr,
              const int32_t *slot_mapping = nullptr, int decode_sms = 0) {
    const bool fp8 = k_scale != nullptr;
    const int sms = decode_sms > 0 ? std::min(decode_sms, d->num_sms) : d->num_sms;  // SMs the decode may fill
    // split_planned > 0: the caller has already planned the split (and sized
    // its scratch from it); the override is not read a second time.
    const int override_tokens = g_split_override.load();
    const int split = split_planned > 0 ? split_planned
                                        : decode_split_tokens(num_seqs, sh->num_kv_heads, max_seq_len,
                                                              sh->block_size, sms, override_tokens);
    const int max_splits = decode_max_splits(max_seq_len, split);
    const size_t need = decode_workspace_bytes(num_seqs, sh->num_q_heads, sh->num_kv_heads, sh->head_dim,
                                               max_splits);
    if (ws == nullptr || ws_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace smaller than " + std::to_string(need) + " bytes");
    if (!aligned16(ws)) return fail(PA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    if ((long long)num_seqs * sh->num_q_heads > 0x7fffffffLL ||
        (long long)num_seqs * sh->num_kv_heads * max_splits > 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "decode batch too large");
    CUtensorMap tq, tk, tv;
    int rc = make_qgroup_map(&tq, q, sh, num_seqs);
    if (rc) return rc;
    rc = fp8 ? make_pool_map_u8(&tk, k_pool, sh) : make_pool_map(&tk, k_pool, sh);
    if (rc) return rc;
    rc = fp8 ? make_pool_map_u8(&tv, v_pool, sh) : make_pool_map(&tv, v_pool, sh);
    if (rc) return rc;
    DecodeArgs a{};
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.part_acc = max_splits > 1 ? static_cast<float *>(ws) : nullptr;
    a.part_ml = max_splits > 1
                    ? static_cast<float *>(ws) + (size_t)num_seqs * sh->num_q_heads * max_splits * sh->head_dim
                    : nullptr;
    decode_plan_layout(ws, num_seqs, sh->num_q_heads, sh->num_kv_heads, sh->head_dim, max_splits, &a.plan_items,
                       &a.plan_count, &a.plan_seq, &a.merge_cnt);
    a.err = d->err;
    a.num_seqs = num_seqs;
    a.num_q_heads = sh->num_q_heads;
    a.num_kv_heads = sh->num_kv_heads;
    a.group = sh->num_q_heads / sh->num_kv_heads;
    a.num_blocks = sh->num_blocks;
    a.max_blocks = max_blocks;
    a.split_tokens = split;
    a.split_adapt = override_tokens > 0 ? 0 : 1;  // an override (tests) is taken exactly
    a.max_splits = max_splits;
    a.max_seq_len = max_seq_len;
    a.check_err_first = check_first;
    a.scale_log2 = scale_log2(sh);
    if (k_new) {
        a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
        a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
        a.slot_mapping = slot_mapping;
        a.k_pool = static_cast<__nv_bfloat16 *>(const_cast<void *>(k_pool));
        a.v_pool = static_cast<__nv_bfloat16 *>(const_cast<void *>(v_pool));
        a.num_slots = (long long)sh->num_blocks * sh->block_size;
    }
    cudaError_t e = launch_decode(tq, tk, tv, a, sh->head_dim, sh->block_size, sms, st, fp8);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return PA_OK;
}

int do_prefill(const pa_shape_t *sh, const void *q, const void *k, const void *v, const int32_t *cu,
               const int32_t *prefix_lens, const int32_t *seq_lens, const int32_t *block_table,
               int max_blocks, int num_seqs, int num_tokens, int max_q_len, void *out, cudaStream_t st,
               DevState *d, int check_first, int pairs = 0) {
    CUtensorMap tq, tk, tv;
    int rc = make_rows_map(&tq, q, sh->head_dim, sh->num_q_heads, num_tokens);
    if (rc) return rc;
    if (block_table) {
        rc = make_pool_map(&tk, k, sh);
        if (!rc) rc = make_pool_map(&tv, v, sh);
    } else {
        const int kbox = sh->head_dim == 128 ? 64 : 128;  // CTA pairs load half-tiles of K
        rc = make_rows_map(&tk, k, sh->head_dim, sh->num_kv_heads, num_tokens, kbox);
        if (!rc) rc = make_rows_map(&tv, v, sh->head_dim, sh->num_kv_heads, num_tokens);
    }
    if (rc) return rc;
    PrefillArgs a{};
    a.cu_seqlens = cu;
    a.prefix_lens = prefix_lens;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = d->err;
    a.num_seqs = num_seqs;
    a.num_q_heads = sh->num_q_heads;
    a.num_kv_heads = sh->num_kv_heads;
    a.group = sh->num_q_heads / sh->num_kv_heads;
    a.num_blocks = sh->num_blocks;
    a.max_blocks = max_blocks;
    a.num_tokens = num_tokens;
    a.max_q_len = max_q_len;
    a.num_q_tiles = (max_q_len + 127) / 128;
    a.check_err_first = check_first;
    a.scale_log2 = scale_log2(sh);
    {
        const int ov = pairs > 0 ? pairs : g_pairs_override.load();
        a.num_sms = ov > 0 ? std::min(2 * ov, d->num_sms) : d->num_sms;
    }
    cudaError_t e;
    if (sh->head_dim == 128) {
        CUtensorMap to;
        if ((rc = make_rows_map(&to, out, sh->head_dim, sh->num_q_heads, num_tokens, 32))) return rc;
        e = launch_prefill_pair(tq, tk, tv, to, a, sh->block_size, st);
    } else {
        e = launch_prefill(tq, tk, tv, a, sh->head_dim, sh->block_size, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return PA_OK;
}

// Split-K scratch for pa_decode_noalloc: a fixed buffer inside the library,
// one copy per device, so that callers who cannot allocate device memory can
// still run decode.  Host code must not use the symbol itself as a device
// address; each device's address is looked up once and cached.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];
std::mutex g_scratch_mu;
void *g_scratch_ptr[64];

int noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PA_ERR_CUDA, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

// Mixed step: the prefill half runs on a second, higher-priority stream of
// the library's own, forked from and joined back into the caller's stream
// with events, so the tensor-bound prefill CTAs and the HBM-bound decode CTAs
// share the GPU instead of running back to back.  One side stream and one
// event pair per device, created on first use; the mutex keeps concurrent
// callers' fork/join sequences from interleaving.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, appended = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

int side_stream(SideStream **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PA_ERR_CUDA, "device ordinal out of range");
    SideStream &s = g_side[dev];
    if (!s.stream) {
        int lo = 0, hi = 0;
        e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&s.stream, cudaStreamNonBlocking, hi);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.appended, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "creating the mixed-step side stream");
    }
    *out = &s;
    return PA_OK;
}

int run_check(const CheckArgs &ca, cudaStream_t st) {
    cudaError_t e = launch_index_check(ca, st);
    if (e != cudaSuccess) return cuda_fail(e, "index check launch");
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_version(void) { return 100; }

int pa_workspace_size(const pa_shape_t *shape, int max_seqs, int max_seq_len, size_t *bytes) {
    int rc = check_shape(shape);
    if (rc) return rc;
    if (!bytes) return fail(PA_ERR_INVALID_ARG, "bytes is NULL");
    if (max_seqs < 0 || max_seq_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    const int split = split_min_tokens(shape->block_size);
    *bytes = decode_workspace_bytes(max_seqs, shape->num_q_heads, shape->num_kv_heads, shape->head_dim,
                                    decode_max_splits(max_seq_len, split));
    return ok();
}

int pa_decode_plan(const pa_shape_t *shape, int num_seqs, int max_seq_len, int *split_tokens,
                   int *max_splits) {
    int rc = check_shape(shape);
    if (rc) return rc;
    if (!split_tokens || !max_splits) return fail(PA_ERR_INVALID_ARG, "NULL output pointer");
    if (num_seqs < 0 || max_seq_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    *split_tokens = decode_split_tokens(num_seqs, shape->num_kv_heads, max_seq_len, shape->block_size,
                                        d->num_sms, g_split_override.load());
    *max_splits = decode_max_splits(max_seq_len, *split_tokens);
    return ok();
}

int pa_kv_append(const pa_shape_t *shape, const void *k_new, const void *v_new, const int32_t *slot_mapping,
                 int num_tokens, void *k_pool, void *v_pool, void *stream) {
    Range range_("pa_kv_append");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return ok();
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return fail(PA_ERR_INVALID_ARG, "k/v and pools must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.slot_mapping = slot_mapping;
        ca.num_tokens = num_tokens;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    if ((rc = do_append(shape, k_new, v_new, slot_mapping, num_tokens, k_pool, v_pool, st, d, val))) return rc;
    return ok();
}

int pa_rope_append(const pa_shape_t *shape, const void *q, const void *k_new, const void *v_new,
                   const int32_t *positions, const int32_t *slot_mapping, int num_tokens, float rope_theta,
                   void *q_out, void *k_pool, void *v_pool, void *stream) {
    Range range_("pa_rope_append");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (!(rope_theta >= 0.f) || std::isinf(rope_theta)) return fail(PA_ERR_INVALID_ARG, "rope_theta must be finite, >= 0");
    if (num_tokens == 0) return ok();
    if (!q || !k_new || !v_new || !positions || !slot_mapping || !q_out || !k_pool || !v_pool)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_out) || !aligned16(k_pool) ||
        !aligned16(v_pool))
        return fail(PA_ERR_INVALID_ARG, "q, k/v, q_out and pools must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.slot_mapping = slot_mapping;
        ca.num_tokens = num_tokens;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    RopeArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.positions = positions;
    a.slot_mapping = slot_mapping;
    a.q_out = static_cast<__nv_bfloat16 *>(q_out);
    a.k_pool = static_cast<__nv_bfloat16 *>(k_pool);
    a.v_pool = static_cast<__nv_bfloat16 *>(v_pool);
    a.err = d->err;
    a.num_tokens = num_tokens;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.head_dim = shape->head_dim;
    a.block_size = shape->block_size;
    a.num_blocks = shape->num_blocks;
    a.check_err_first = val;
    const double theta = rope_theta == 0.f ? 10000.0 : (double)rope_theta;
    for (int i = 0; i < shape->head_dim / 2; ++i) {
        // the frequency in turns per position, its fractional part as 64-bit fixed point
        double q = pow(theta, -2.0 * i / shape->head_dim) / 6.283185307179586;
        q -= std::floor(q);
        a.turn[i] = q >= 1.0 ? 0ull : (unsigned long long)std::ldexp(q, 64);
    }
    cudaError_t e = launch_rope_append(a, d->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "rope_append launch");
    return ok();
}

int pa_copy_blocks(const pa_shape_t *shape, const void *src_k, const void *src_v, int src_num_blocks,
                   void *dst_k, void *dst_v, int dst_num_blocks, const int32_t *src_ids,
                   const int32_t *dst_ids, int num_pairs, void *stream) {
    Range range_("pa_copy_blocks");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_pairs < 0 || src_num_blocks < 0 || dst_num_blocks < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_pairs == 0) return ok();
    if (!src_k || !src_v || !dst_k || !dst_v || !src_ids || !dst_ids) return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
        return fail(PA_ERR_INVALID_ARG, "pools must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    // Every pointer must be GPU-visible: device memory, or pinned host memory
    // (read and written through its device alias).
    const void *ptrs[6] = {src_k, src_v, dst_k, dst_v, src_ids, dst_ids};
    void *dev_ptrs[6];
    for (int i = 0; i < 6; ++i) {
        cudaPointerAttributes at{};
        cudaError_t pe = cudaPointerGetAttributes(&at, ptrs[i]);
        if (pe != cudaSuccess) return cuda_fail(pe, "copy_blocks pointer query");
        if (at.type == cudaMemoryTypeUnregistered || !at.devicePointer)
            return fail(PA_ERR_INVALID_ARG, "copy_blocks: a pointer is neither device nor pinned host memory");
        if (i >= 4 && at.type == cudaMemoryTypeHost)
            return fail(PA_ERR_INVALID_ARG, "copy_blocks: block ids must be in device memory");
        dev_ptrs[i] = at.devicePointer;
    }
    const long long block_bytes = (long long)shape->num_kv_heads * shape->block_size * shape->head_dim * 2;
    cudaError_t e = launch_copy_blocks(dev_ptrs[0], dev_ptrs[1], dev_ptrs[2], dev_ptrs[3],
                                       static_cast<const int32_t *>(dev_ptrs[4]),
                                       static_cast<const int32_t *>(dev_ptrs[5]), num_pairs, block_bytes,
                                       src_num_blocks, dst_num_blocks, d->num_sms, d->err, g_validation.load(),
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
    return ok();
}

int pa_decode(const pa_shape_t *shape, const void *q, const void *k_pool, const void *v_pool,
              const int32_t *block_table, int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
              int max_seq_len, void *out, void *workspace, size_t ws_bytes, void *stream) {
    Range range_("pa_decode");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_seqs < 0 || max_seq_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0) return ok();
    if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if ((max_seq_len + shape->block_size - 1) / shape->block_size > max_blocks_per_seq)
        return fail(PA_ERR_INVALID_ARG, "max_seq_len does not fit in max_blocks_per_seq blocks");
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PA_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.block_table = block_table;
        ca.seq_lens = seq_lens;
        ca.num_seqs = num_seqs;
        ca.max_blocks = max_blocks_per_seq;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.max_seq_len = max_seq_len;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    rc = do_decode(shape, q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                   out, workspace, ws_bytes, st, d, val);
    if (rc) return rc;
    return ok();
}

int pa_decode_append(const pa_shape_t *shape, const void *q, const void *k_new, const void *v_new,
                     const int32_t *slot_mapping, void *k_pool, void *v_pool, const int32_t *block_table,
                     int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs, int max_seq_len, void *out,
                     void *workspace, size_t ws_bytes, void *stream) {
    Range range_("pa_decode_append");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_seqs < 0 || max_seq_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0) return ok();
    if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    if (!q || !k_new || !v_new || !slot_mapping || !k_pool || !v_pool || !block_table || !seq_lens || !out)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if ((max_seq_len + shape->block_size - 1) / shape->block_size > max_blocks_per_seq)
        return fail(PA_ERR_INVALID_ARG, "max_seq_len does not fit in max_blocks_per_seq blocks");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(out))
        return fail(PA_ERR_INVALID_ARG, "q, k/v, pools and out must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.slot_mapping = slot_mapping;
        ca.num_tokens = num_seqs;
        ca.block_table = block_table;
        ca.seq_lens = seq_lens;
        ca.num_seqs = num_seqs;
        ca.max_blocks = max_blocks_per_seq;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.max_seq_len = max_seq_len;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    rc = do_decode(shape, q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                   out, workspace, ws_bytes, st, d, val, nullptr, nullptr, 0, k_new, v_new, slot_mapping);
    if (rc) return rc;
    return ok();
}

int pa_kv_append_fp8(const pa_shape_t *shape, const void *k_new, const void *v_new, const int32_t *slot_mapping,
                     int num_tokens, const float *k_scale, const float *v_scale, void *k_pool, void *v_pool,
                     void *stream) {
    Range range_("pa_kv_append_fp8");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return ok();
    if (!k_new || !v_new || !slot_mapping || !k_scale || !v_scale || !k_pool || !v_pool)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return fail(PA_ERR_INVALID_ARG, "k/v and pools must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.slot_mapping = slot_mapping;
        ca.num_tokens = num_tokens;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    cudaError_t e = launch_kv_append_fp8(static_cast<const __nv_bfloat16 *>(k_new),
                                         static_cast<const __nv_bfloat16 *>(v_new), slot_mapping, num_tokens,
                                         shape->num_kv_heads, shape->head_dim, shape->block_size, shape->num_blocks,
                                         k_scale, v_scale, static_cast<uint8_t *>(k_pool),
                                         static_cast<uint8_t *>(v_pool), d->err, val, st);
    if (e != cudaSuccess) return cuda_fail(e, "kv_append_fp8 launch");
    return ok();
}

int pa_decode_fp8(const pa_shape_t *shape, const void *q, const void *k_pool, const void *v_pool,
                  const float *k_scale, const float *v_scale, const int32_t *block_table, int max_blocks_per_seq,
                  const int32_t *seq_lens, int num_seqs, int max_seq_len, void *out, void *workspace,
                  size_t ws_bytes, void *stream) {
    Range range_("pa_decode_fp8");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_seqs < 0 || max_seq_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0) return ok();
    if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    if (!q || !k_pool || !v_pool || !k_scale || !v_scale || !block_table || !seq_lens || !out)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if ((max_seq_len + shape->block_size - 1) / shape->block_size > max_blocks_per_seq)
        return fail(PA_ERR_INVALID_ARG, "max_seq_len does not fit in max_blocks_per_seq blocks");
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PA_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.block_table = block_table;
        ca.seq_lens = seq_lens;
        ca.num_seqs = num_seqs;
        ca.max_blocks = max_blocks_per_seq;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.max_seq_len = max_seq_len;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    rc = do_decode(shape, q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                   out, workspace, ws_bytes, st, d, val, k_scale, v_scale);
    if (rc) return rc;
    return ok();
}

int pa_decode_noalloc(const pa_shape_t *shape, const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                      int max_seq_len, void *out, void *stream) {
    Range range_("pa_decode_noalloc");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_seqs < 0 || max_seq_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0) return ok();
    if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if ((max_seq_len + shape->block_size - 1) / shape->block_size > max_blocks_per_seq)
        return fail(PA_ERR_INVALID_ARG, "max_seq_len does not fit in max_blocks_per_seq blocks");
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PA_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    const int split = decode_split_tokens(num_seqs, shape->num_kv_heads, max_seq_len, shape->block_size,
                                          d->num_sms, g_split_override.load());
    const size_t need = decode_workspace_bytes(num_seqs, shape->num_q_heads, shape->num_kv_heads, shape->head_dim,
                                               decode_max_splits(max_seq_len, split));
    if (need > PA_NOALLOC_SCRATCH_BYTES)
        return fail(PA_ERR_WORKSPACE, "batch needs " + std::to_string(need) +
                                          " bytes of split-K scratch; the built-in buffer holds " +
                                          std::to_string(PA_NOALLOC_SCRATCH_BYTES) +
                                          " (use pa_decode with a caller workspace)");
    void *scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.block_table = block_table;
        ca.seq_lens = seq_lens;
        ca.num_seqs = num_seqs;
        ca.max_blocks = max_blocks_per_seq;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.max_seq_len = max_seq_len;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    rc = do_decode(shape, q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                   out, scratch, PA_NOALLOC_SCRATCH_BYTES, st, d, val, nullptr, nullptr, split);
    if (rc) return rc;
    return ok();
}

int pa_prefill(const pa_shape_t *shape, const void *q, const void *k, const void *v, const int32_t *cu_seqlens_q,
               const int32_t *prefix_lens, const int32_t *block_table, int max_blocks_per_seq, int num_seqs,
               int num_tokens, int max_q_len, void *out, void *stream) {
    Range range_("pa_prefill");
    int rc = check_shape(shape);
    if (rc) return rc;
    if (num_seqs < 0 || num_tokens < 0 || max_q_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (num_seqs == 0 || num_tokens == 0 || max_q_len == 0) return ok();
    if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    if (!q || !k || !v || !cu_seqlens_q || !out) return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (!block_table && prefix_lens)
        return fail(PA_ERR_INVALID_ARG, "prefix_lens needs the paged form (block_table)");
    if (block_table && max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(PA_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.block_table = block_table;
        ca.cu_seqlens = cu_seqlens_q;
        ca.prefix_lens = prefix_lens;
        ca.num_seqs = num_seqs;
        ca.num_tokens = 0;
        ca.max_blocks = max_blocks_per_seq;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.max_q_len = max_q_len;
        ca.max_seq_len = 0x7fffffff;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    rc = do_prefill(shape, q, k, v, cu_seqlens_q, prefix_lens, nullptr, block_table, max_blocks_per_seq,
                    num_seqs, num_tokens, max_q_len, out, st, d, val);
    if (rc) return rc;
    return ok();
}

// Prefill CTA pairs for a mixed step whose halves run side by side: the
// count that gives both the same time under a cost model measured on GB300.
// The prefill pair kernel costs about 2 us per 128-key tile-step of a work
// unit plus 1 us per unit, on one CTA pair; the decode streams about 50 GB/s
// of K/V per SM (a fit to the per-step optimum of a 64-step churn of 512
// sequences and to a 120-decode + 8-prompt step, each timed at 30 pair counts).  With A pair-us of
// prefill work and B SM-us of decode work, A / P = B / (S - 2 P) at
// P = S A / (B + 2 A).  0 (no split) when a half is empty or head_dim is not
// 128 (only the pair kernel takes a pair count).
static int mixed_prefill_pairs(const pa_shape_t *sh, const int32_t *decode_lens, int nd, const int32_t *rows,
                               const int32_t *prefix, int np, int num_sms) {
    if (nd <= 0 || np <= 0 || sh->head_dim != 128 || num_sms < 6) return 0;
    const int group = sh->num_q_heads / sh->num_kv_heads;
    const int per_unit = group % 4 == 0 ? 1 : (group % 2 == 0 ? 2 : 4);   // row tiles of a head in one unit
    const int ny = sh->num_q_heads / (group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1));  // units per level
    double units = 0.0, steps = 0.0;
    for (int i = 0; i < np; ++i) {
        const long long n = rows[i], p0 = prefix ? std::max(0, prefix[i]) : 0;
        if (n <= 0) continue;
        const long long levels = ((n + 127) / 128 + per_unit - 1) / per_unit;
        for (long long px = 0; px < levels; ++px) {
            const long long kv_end = p0 + std::min(n, (px + 1) * per_unit * 128);
            units += ny;
            steps += (double)ny * ((kv_end + 127) / 128);
        }
    }
    double bytes = 0.0;
    for (int i = 0; i < nd; ++i) bytes += (double)std::max(0, decode_lens[i]) * sh->num_kv_heads * sh->head_dim * 4.0;
    const double a = 1.0 * units + 2.0 * steps;  // pair-us
    const double b = bytes / 50e3;               // SM-us at 50 GB/s per SM
    if (a <= 0.0 || b <= 0.0) return 0;
    const int p = (int)std::lround(num_sms * a / (b + 2.0 * a));
    return std::max(1, std::min(p, num_sms / 2 - 1));
}

static int mixed_step(const pa_shape_t *shape, const void *q, const void *k_new, const void *v_new,
                      const int32_t *q_start_loc, const int32_t *seq_lens, const int32_t *slot_mapping,
                      const int32_t *block_table, int max_blocks_per_seq, int num_seqs, int num_decode,
                      int num_tokens, int max_seq_len, int max_q_len, void *k_pool, void *v_pool, void *out,
                      void *workspace, size_t ws_bytes, void *stream, int prefill_pairs) {
    int rc = check_shape(shape);
    if (prefill_pairs < 0) return fail(PA_ERR_INVALID_ARG, "prefill_pairs < 0");
    if (rc) return rc;
    if (num_seqs < 0 || num_decode < 0 || num_decode > num_seqs || num_tokens < 0 || max_seq_len < 0 ||
        max_q_len < 0)
        return fail(PA_ERR_INVALID_ARG, "bad sizes");
    if (num_seqs == 0) return ok();
    if (num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    if (num_tokens < num_decode) return fail(PA_ERR_INVALID_ARG, "num_tokens < num_decode");
    if (!q || !k_new || !v_new || !q_start_loc || !seq_lens || !slot_mapping || !block_table || !k_pool ||
        !v_pool || !out)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if ((max_seq_len + shape->block_size - 1) / shape->block_size > max_blocks_per_seq)
        return fail(PA_ERR_INVALID_ARG, "max_seq_len does not fit in max_blocks_per_seq blocks");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(out))
        return fail(PA_ERR_INVALID_ARG, "q, k/v, pools and out must be 16-byte aligned");
    DevState *d;
    if ((rc = dev_state(&d))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int val = g_validation.load();
    if (val) {
        CheckArgs ca{};
        ca.slot_mapping = slot_mapping;
        ca.num_tokens = num_tokens;
        ca.block_table = block_table;
        ca.seq_lens = seq_lens;
        ca.cu_seqlens = q_start_loc;
        ca.num_seqs = num_seqs;
        ca.max_blocks = max_blocks_per_seq;
        ca.block_size = shape->block_size;
        ca.num_blocks = shape->num_blocks;
        ca.max_seq_len = max_seq_len;
        ca.max_q_len = max_q_len > 1 ? max_q_len : 1;
        ca.decode_rows = num_decode;
        ca.err = d->err;
        if ((rc = run_check(ca, st))) return rc;
    }
    // Decode rows [0, num_decode) are appended by the decode's plan launch,
    // before its attention kernel reads anything; the prompt rows
    // [num_decode, num_tokens) by the append kernel ahead of the prefill.
    const int np = num_seqs - num_decode;
    const bool has_prefill = np > 0 && max_q_len > 0 && num_tokens > 0;
    const size_t row = (size_t)shape->num_kv_heads * shape->head_dim;
    const int prompt_rows = num_tokens - num_decode;
    auto append_prompts = [&](cudaStream_t s) {
        if (prompt_rows <= 0) return (int)PA_OK;
        return do_append(shape, static_cast<const __nv_bfloat16 *>(k_new) + (size_t)num_decode * row,
                         static_cast<const __nv_bfloat16 *>(v_new) + (size_t)num_decode * row,
                         slot_mapping + num_decode, prompt_rows, k_pool, v_pool, s, d, val);
    };
    // prefill_pairs > 0 (and fewer than the SMs hold): the prefill runs on
    // that many CTA pairs and the decode fills the other SMs only, side by side.
    const bool split_sms = has_prefill && num_decode > 0 && prefill_pairs > 0 && shape->head_dim == 128 &&
                           2 * prefill_pairs < d->num_sms;
    auto prefill_on = [&](cudaStream_t s) {
        return do_prefill(shape, q, k_pool, v_pool, q_start_loc + num_decode, nullptr, seq_lens + num_decode,
                          block_table + (size_t)num_decode * max_blocks_per_seq, max_blocks_per_seq, np,
                          num_tokens, max_q_len, out, s, d, val, split_sms ? prefill_pairs : 0);
    };
    auto decode_on = [&](cudaStream_t s) {
        const int dsms = split_sms ? d->num_sms - 2 * prefill_pairs : 0;
        return do_decode(shape, q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens, num_decode,
                         max_seq_len, out, workspace, ws_bytes, s, d, val, nullptr, nullptr, 0, k_new, v_new,
                         slot_mapping, dsms);
    };
    if (num_decode > 0 && has_prefill) {
        std::lock_guard<std::mutex> lk(g_side_mu);
        SideStream *side;
        if ((rc = side_stream(&side))) return rc;
        cudaError_t e = cudaEventRecord(side->fork, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
        if (e != cudaSuccess) return cuda_fail(e, "forking the mixed step");
        // The decode waits for the prompt rows' append too: then the prefill
        // (higher priority) and the decode become ready together, and the
        // prefill's persistent CTA pairs -- one per SM, too large to share one
        // with decode CTAs -- are placed first, on the SMs the decode then
        // leaves to them.  (A decode started earlier would take every SM and
        // the prefill would only start as it drains.)
        rc = append_prompts(side->stream);
        if (e == cudaSuccess) e = cudaEventRecord(side->appended, side->stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, side->appended, 0);
        if (e != cudaSuccess) return cuda_fail(e, "ordering the mixed step");
        if (!rc) rc = prefill_on(side->stream);
        const int rc2 = decode_on(st);
        e = cudaEventRecord(side->join, side->stream);  // join even after a failed launch
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, side->join, 0);
        if (e != cudaSuccess) return cuda_fail(e, "joining the mixed step");
        if (rc) return rc;
        if (rc2) return rc2;
        return ok();
    }
    if (num_decode > 0 && (rc = decode_on(st))) return rc;
    if ((rc = append_prompts(st))) return rc;
    if (has_prefill && (rc = prefill_on(st))) return rc;
    return ok();
}

int pa_mixed_step(const pa_shape_t *shape, const void *q, const void *k_new, const void *v_new,
                  const int32_t *q_start_loc, const int32_t *seq_lens, const int32_t *slot_mapping,
                  const int32_t *block_table, int max_blocks_per_seq, int num_seqs, int num_decode,
                  int num_tokens, int max_seq_len, int max_q_len, void *k_pool, void *v_pool, void *out,
                  void *workspace, size_t ws_bytes, void *stream) {
    Range range_("pa_mixed_step");
    return mixed_step(shape, q, k_new, v_new, q_start_loc, seq_lens, slot_mapping, block_table, max_blocks_per_seq,
                      num_seqs, num_decode, num_tokens, max_seq_len, max_q_len, k_pool, v_pool, out, workspace,
                      ws_bytes, stream, 0);
}

int pa_mixed_step_split(const pa_shape_t *shape, const void *q, const void *k_new, const void *v_new,
                        const int32_t *q_start_loc, const int32_t *seq_lens, const int32_t *slot_mapping,
                        const int32_t *block_table, int max_blocks_per_seq, int num_seqs, int num_decode,
                        int num_tokens, int max_seq_len, int max_q_len, void *k_pool, void *v_pool, void *out,
                        void *workspace, size_t ws_bytes, void *stream, int prefill_pairs) {
    Range range_("pa_mixed_step_split");
    return mixed_step(shape, q, k_new, v_new, q_start_loc, seq_lens, slot_mapping, block_table, max_blocks_per_seq,
                      num_seqs, num_decode, num_tokens, max_seq_len, max_q_len, k_pool, v_pool, out, workspace,
                      ws_bytes, stream, prefill_pairs);
}

int pa_mixed_prefill_pairs(const pa_shape_t *shape, const int32_t *decode_lens, int num_decode,
                           const int32_t *prompt_rows, const int32_t *prefix_lens, int num_prompts, int num_sms,
                           int *pairs) {
    int rc = check_shape(shape);
    if (rc) return rc;
    if (!pairs || num_decode < 0 || num_prompts < 0 || (num_decode > 0 && !decode_lens) ||
        (num_prompts > 0 && !prompt_rows))
        return fail(PA_ERR_INVALID_ARG, "NULL pointer or negative count");
    if (num_sms <= 0) {
        DevState *d;
        if ((rc = dev_state(&d))) return rc;
        num_sms = d->num_sms;
    }
    *pairs = mixed_prefill_pairs(shape, decode_lens, num_decode, prompt_rows, prefix_lens, num_prompts, num_sms);
    return ok();
}

int pa_set_validation(int on) {
    g_validation.store(on ? 1 : 0);
    return ok();
}

int pa_set_decode_split(int tokens) {
    if (tokens < 0) return fail(PA_ERR_INVALID_ARG, "tokens < 0");
    g_split_override.store(tokens);
    return ok();
}

int pa_set_prefill_pairs(int pairs) {
    if (pairs < 0) return fail(PA_ERR_INVALID_ARG, "pairs < 0");
    g_pairs_override.store(pairs);
    return ok();
}

int pa_check_device_error(void *stream) {
    Range range_("pa_check_device_error");
    DevState *d;
    int rc = dev_state(&d);
    if (rc) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    if (word == PA_ERR_BAD_INDEX) return fail(PA_ERR_BAD_INDEX, "device saw an out-of-range index");
    if (word == PA_ERR_TIMEOUT) return fail(PA_ERR_TIMEOUT, "a bounded device wait gave up");
    if (word != 0) return fail(PA_ERR_CUDA, "device error word " + std::to_string(word));
    return ok();
}

const char *pa_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"
