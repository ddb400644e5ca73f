// decode.cu -- paged GQA decode attention, split-K (flash-decoding style).
//
// What it computes (text-generation-inference Router/Webserver deep dive,
// section "Prefill, Decode and past key values": every pass after the prompt
// computes attention only for the new token against the cached past keys and
// values): for each running sequence s and query head h,
//     out[s][h] = sum_j softmax_j(scale * <q[s][h], k_j>) v_j ,  j < seq_lens[s]
// with keys/values read through the block table from the KV head h / G.
//
// Design (GB300, HBM-bound):
//  * Plan (decode_plan_kernel, the first step of the path): its first CTA
//    lists the work items in the workspace -- one per (sequence, KV head,
//    split of `split_tokens` consecutive tokens, i.e. whole KV blocks) that
//    holds tokens: every full split first, then the last splits from longest
//    to shortest.  Nothing is launched for splits a sequence does not have,
//    so a ragged batch of short and long sequences costs what its tokens
//    cost.  With the append fused (pa_decode_append, the mixed step), the
//    launch's other CTAs copy the step's new rows into their slots.
//  * Decode (decode_splitk_kernel, persistent, two CTAs per SM): CTA b
//    takes items b, 2n-1-b, 2n+b, ... of the list (n CTAs; a snake order, so
//    that the sorted sizes even out) and streams all of their KV blocks, one
//    after another, through a ring of shared-memory stages filled by TMA
//    tensor loads (128-byte swizzle): a producer warp whose lane l owns
//    stage l walks the CTA's item sequence on its own and refills its stage
//    as soon as it is free, with the next item's blocks while the current
//    item is still being computed; another lane loads each item's G query
//    rows into a q buffer as soon as the previous item's have been read.  Each block of one KV head is one contiguous B x d chunk of the
//    pool, a stage is 2 (K, V) x d/64 boxes of B rows x 128 bytes.  Block ids
//    are range-checked before use.
//  * Four consumer warps take the blocks round-robin.  Each warp computes the
//    scores of the G query heads of this KV head against 16 keys with
//    m16n8k16 tensor-core MMAs (rows = query heads, padded to 16; the G
//    heads share every K/V byte read), keeps its own online-softmax state
//    with quad shuffles, and accumulates P.V with the same MMA shape.  The
//    tensor-core dot products keep the FP32 pipe free: with G = 8 a CUDA-core
//    dot product would need ~2 G d FMAs per key, as much FP32 issue as the
//    HBM stream leaves room for.
//  * At the end of an item the four states are merged in two steps through a
//    small scratch area (warps 1 and 3 into 0 and 2, then 2 into 0; only the
//    G rows that hold query heads) while the ring keeps filling; a sequence
//    with a single split writes bf16 output directly, otherwise the (max,
//    sum, acc) partials go to the workspace, and the split of a (sequence,
//    KV head) that finishes last -- a per-(sequence, KV head) count taken
//    with an atomic after a fence -- combines them there, its four consumer
//    warps taking the G query heads between them.  No second kernel: the
//    merges of early-finishing sequences overlap the other CTAs' streaming,
//    and a batch whose sequences all fit one split pays nothing for them.
#include <cuda.h>

#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kMergeWarp = kConsumerWarps + 1;  // after the producer warp
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kMergeSlots = 4;  // merge requests queued from the consumers to the merge warp
constexpr int kQLane = 31;  // the producer lane that loads the items' query rows

template <int D, int BS, bool FP8, bool BIG_G>
struct DecodeCfg {
    static constexpr int kEB = FP8 ? 1 : 2;                // bytes per pool element
    // fp8 rows of d = 64 are 64 bytes: two tokens share one 128-byte TMA row
    // (token t in row t / 2, bytes 64 (t % 2) ..), so the boxes keep the
    // 128-byte swizzle; the pool is viewed as rows of 128 bytes.
    static constexpr bool kPacked = FP8 && D == 64;
    static constexpr int kBoxCols = kPacked ? 128 : 128 / kEB;  // elements per 128-byte TMA box row
    static constexpr int kHalves = kPacked ? 1 : D / kBoxCols;  // TMA boxes per row
    static constexpr int kHalfBytes = BS * D * kEB / kHalves;   // one box: BS tokens' share of it
    static constexpr int kKVBytes = kHalves * kHalfBytes;  // K (or V) of one block
    static constexpr int kStageBytes = 2 * kKVBytes;
    // 96 KB of blocks in flight per CTA (64 KB for G > 8, whose larger merge
    // scratch would otherwise leave room for one CTA per SM): more bytes in
    // flight than the DRAM latency needs, with room to spare for the short
    // stalls of the consumers.  A multiple of the consumer warps: stage st is
    // read only by warp st % 4, block after block, so a warp never waits on
    // a stage's barrier more than one phase ahead.
    static constexpr int kRingBudget = BIG_G ? 65536 : 98304;
    static constexpr int kStagesFit = kRingBudget / kStageBytes < 28 ? kRingBudget / kStageBytes : 28;
    static constexpr int kStages = kStagesFit / kConsumerWarps * kConsumerWarps;
    static constexpr int kKSteps = D / 16;                 // QK^T k-steps
    static constexpr int kNTiles = D / 8;                  // PV n-tiles
    static constexpr int kRingBytes = kStages * kStageBytes;
    // merge scratch: two slots of one warp's state (its MMA rows: 8, or 16
    // for G > 8), rows padded by 8 floats
    static constexpr int kRows = BIG_G ? 16 : 8;
    static constexpr int kRow = D + 8;
    static constexpr int kSlotFloats = kRows * kRow + kRows * 2;
    static constexpr int kScratchOff = kRingBytes;
    static constexpr int kQOff = kScratchOff + ((2 * kSlotFloats * 4 + 1023) / 1024) * 1024;
    static constexpr int kQHalves = D / 64;                // q is bf16: 64-column boxes of G rows
    static constexpr int kBarOff = kQOff + kQHalves * 2048;
    // barriers: ring full / empty, q full / empty, merge queue full / empty;
    // then the abort flag (16 bytes) and the merge queue's slots
    static constexpr int kNumBars = 2 * kStages + 2 + 2 * kMergeSlots;
    static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + kMergeSlots * 16 + 1024;
    static_assert((kNumBars * 8) % 16 == 0, "merge slots 16-byte aligned");
    // two: a third would need the registers cut to 128 (spills; measured slower)
    static constexpr int kCtasPerSm = 232448 / (kSmemBytes + 1024) < 2 ? 232448 / (kSmemBytes + 1024) : 2;
    static_assert(kStages >= kConsumerWarps && kStages < kQLane, "one producer lane per stage, and the q lane");
    static_assert(kCtasPerSm == 2, "two CTAs per SM");
};

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ bool len_ok(const DecodeArgs &a, int L, int BS) {
    return L >= 0 && L <= a.max_seq_len && (L + BS - 1) / BS <= a.max_blocks;
}

// Exclusive prefix sum over the 1024 threads of the CTA; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int *tmp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = tmp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        tmp[32 + lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int before = warp ? tmp[32 + warp - 1] : 0;
    *total = tmp[32 + 31];
    __syncthreads();
    return before + x - v;
}

constexpr int kPlanBins = 256;  // last-split sizes (in blocks) sorted by a counting sort

// Splits of a sequence of L > 0 tokens: ceil(L / split), but a last split of
// at most split / 8 tokens joins the one before (so the step's new token
// after a context of whole splits does not make an item, and a merge, of its
// own).  Split c covers tokens [c split, (c + 1) split), the last one up to L.
__device__ __forceinline__ int num_splits(int L, int split) {
    const int ns = (L + split - 1) / split;
    return (ns > 1 && L - (ns - 1) * split <= split / 8) ? ns - 1 : ns;
}

// The plan launch.  CTA 0 (1024 threads, thread t owns a contiguous range of
// sequences): a sequence of L > 0 tokens has ns = ceil(L / split) splits;
// items (s, g, c, L) go first for every sequence's ns - 1 full splits, then
// for the last splits, longest first (counting sort on their length in
// blocks; equal lengths in no fixed order -- an item's result depends on the
// item alone, since its four warps merge by item-local role, so the order
// changes no bit of the output).  Empty sequences get zero
// output here; a bad length sets the error word and gets no item.
// CTAs 1.. (only with the append fused): row s of k_new / v_new, every KV
// head, to slot_mapping[s] of the pools (16-byte pieces, grid-stride).
template <int D, int BS>
__global__ void __launch_bounds__(1024) decode_plan_kernel(const DecodeArgs a) {
    __shared__ int tmp[64];
    __shared__ int bins[kPlanBins];
    // The decode kernel (launched as this one's programmatic dependent) may
    // start now: it waits for this grid's completion before it reads
    // anything this grid writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (a.check_err_first && *(volatile int *)a.err != 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            a.plan_count[0] = 0;
            a.plan_count[1] = a.split_tokens;
        }
        return;
    }
    const int S = a.num_seqs, Hkv = a.num_kv_heads;
    if (blockIdx.x > 0) {
        constexpr int NV = D / 8;  // 16-byte pieces per row
        const long long total = (long long)S * Hkv * NV;
        for (long long x = (long long)(blockIdx.x - 1) * 1024 + threadIdx.x; x < total;
             x += (long long)(gridDim.x - 1) * 1024) {
            const int j = (int)(x % NV);
            const long long sg = x / NV;
            const int g = (int)(sg % Hkv), s = (int)(sg / Hkv);
            const int slot = __ldg(a.slot_mapping + s);
            if (slot < 0) continue;
            if ((long long)slot >= a.num_slots) {
                set_error(a.err, PA_ERR_BAD_INDEX);
                continue;
            }
            const size_t dst = (((size_t)(slot / BS) * Hkv + g) * BS + slot % BS) * D;
            const uint4 kx = __ldg(reinterpret_cast<const uint4 *>(a.k_new + sg * D) + j);
            const uint4 vx = __ldg(reinterpret_cast<const uint4 *>(a.v_new + sg * D) + j);
            reinterpret_cast<uint4 *>(a.k_pool + dst)[j] = kx;
            reinterpret_cast<uint4 *>(a.v_pool + dst)[j] = vx;
        }
        return;
    }
    const int per = (S + 1023) / 1024;
    const int s_beg = min(S, (int)threadIdx.x * per), s_end = min(S, s_beg + per);
    // The tokens per split: the host's choice, or (split_adapt) one of
    // split_tokens * 2^k, k <= kSplitGrowth, from the batch's lengths:
    //  1. no split at all (the smallest such k) when even the longest
    //     sequence is at most 3/5 of a decode CTA's share of the batch's KV
    //     blocks: the snake order then evens the items out, and a split only
    //     adds items and merges;
    //  2. otherwise the largest k that still leaves at least kMinItemsPerCta
    //     items per CTA and no item longer than half of a CTA's share.
    // Each item costs a fixed overhead (its query rows, the four warps'
    // merge, the merge of its splits) besides its blocks, so fewer, longer
    // items are faster as long as the CTAs stay evenly loaded.  (Fit to
    // timings on GB300: 120 contexts U[1, 2048] run 20 % faster unsplit than
    // in 512-token splits; 32 x 32K and a log-uniform [1, 8K] churn want
    // rule 2.)
    int split = a.split_tokens;
    if (a.split_adapt) {
        constexpr int kSplitGrowth = 5, kMinItemsPerCta = 6;
        long long cnt[kSplitGrowth + 1] = {}, tok = 0, blk = 0;
        int lmax = 0;
        for (int s = s_beg; s < s_end; ++s) {
            const int L = a.seq_lens[s];
            if (!len_ok(a, L, BS) || L == 0) continue;
            tok += L;
            blk += (L + BS - 1) / BS;
            lmax = max(lmax, L);
#pragma unroll
            for (int k = 0; k <= kSplitGrowth; ++k) cnt[k] += (L + (split << k) - 1) / (split << k);
        }
        __shared__ long long red[kSplitGrowth + 3][32];
        __shared__ int red_max[32];
        auto block_sum = [&](long long v, int slot) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if ((threadIdx.x & 31) == 0) red[slot][threadIdx.x >> 5] = v;
        };
#pragma unroll
        for (int k = 0; k <= kSplitGrowth; ++k) block_sum(cnt[k], k);
        block_sum(tok, kSplitGrowth + 1);
        block_sum(blk, kSplitGrowth + 2);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
        if ((threadIdx.x & 31) == 0) red_max[threadIdx.x >> 5] = lmax;
        __syncthreads();
        // second level: warp w sums slot w (the next warp takes the maximum)
        __shared__ long long tot[kSplitGrowth + 4];
        {
            const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
            if (w < kSplitGrowth + 3) {
                long long v = red[w][l];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (l == 0) tot[w] = v;
            } else if (w == kSplitGrowth + 3) {
                int v = red_max[l];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
                if (l == 0) tot[w] = v;
            }
        }
        __syncthreads();
        __shared__ int chosen;
        if (threadIdx.x < 32) {  // warp 0, lane k: split_tokens << k
            const int k = threadIdx.x;
            const long long ctas = max(a.num_ctas, 1);
            const long long tok_all = tot[kSplitGrowth + 1] * Hkv, blk_all = tot[kSplitGrowth + 2] * Hkv;
            const long long lm = tot[kSplitGrowth + 3];
            const long long sp = (long long)split << k;
            const bool in_range = k <= kSplitGrowth;
            // rule 1: the smallest k whose split holds the longest sequence
            const bool small_longest = 5 * ((lm + BS - 1) / BS) * ctas <= 3 * blk_all;
            const unsigned whole = __ballot_sync(0xffffffffu, in_range && sp >= lm);
            // rule 2: the largest k such that every k' <= k qualifies
            const bool fits = k >= 1 && in_range && (in_range ? tot[k] : 0) * Hkv >= kMinItemsPerCta * ctas &&
                              sp * 2 * ctas <= tok_all;
            const unsigned bad = __ballot_sync(0xffffffffu, !fits && k >= 1 && in_range);
            const int kmax = bad ? __ffs(bad) - 2 : kSplitGrowth;  // first failing k, minus one
            if (k == 0) chosen = (small_longest && whole) ? split << (__ffs(whole) - 1) : split << kmax;
        }
        __syncthreads();
        split = chosen;
    }
    const int nbins = min(kPlanBins, (split + BS - 1) / BS);
    const int bw = ((split + BS - 1) / BS + nbins - 1) / nbins;  // blocks per bin
    // key 0 = the longest last split
    auto key_of = [&](int L, int ns) { return nbins - min(nbins, ((L - (ns - 1) * split + BS - 1) / BS + bw - 1) / bw); };
    if (threadIdx.x < kPlanBins) bins[threadIdx.x] = 0;
    __syncthreads();
    int nfull = 0;
    for (int s = s_beg; s < s_end; ++s) {
        const int L = a.seq_lens[s];
        if (!len_ok(a, L, BS) || L == 0) continue;
        const int ns = num_splits(L, split);
        nfull += ns - 1;
        atomicAdd(&bins[key_of(L, ns)], 1);
    }
    int total_full, total_last;
    int pf = block_excl_scan(nfull, tmp, &total_full);
    const int start = block_excl_scan(threadIdx.x < kPlanBins ? bins[threadIdx.x] : 0, tmp, &total_last);
    if (threadIdx.x < kPlanBins) bins[threadIdx.x] = start;  // now the next free position of each size
    __syncthreads();
    // Phase 1, a thread per sequence: where its items go (pf: its first full
    // split's row of items, pos: its last split's place among the last
    // splits), into a per-sequence array of the workspace.
    for (int s = s_beg; s < s_end; ++s) {
        const int L = a.seq_lens[s];
        const bool ok = len_ok(a, L, BS);
        int2 at = make_int2(-1, -1);
        if (!ok || L == 0) {
            if (!ok) set_error(a.err, PA_ERR_BAD_INDEX);
            if (ok) {  // an empty context attends to nothing: zeros
                uint4 *o = reinterpret_cast<uint4 *>(a.out + (size_t)s * a.num_q_heads * D);
                for (int i = 0; i < a.num_q_heads * D / 8; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        } else {
            const int ns = num_splits(L, split);
            at = make_int2(pf, total_full + atomicAdd(&bins[key_of(L, ns)], 1));
            pf += ns - 1;
        }
        a.plan_seq[s] = at;
    }
    __syncthreads();
    // Phase 2, a thread per (sequence, KV head), KV heads fastest: the items,
    // so that neighbouring threads write neighbouring descriptors, and the
    // merge count of every (sequence, KV head) set to zero.
    for (int p = threadIdx.x; p < S * Hkv; p += 1024) {
        if (a.merge_cnt) a.merge_cnt[p] = 0;
        const int s = p / Hkv, g = p - s * Hkv;
        const int2 at = a.plan_seq[s];
        if (at.x < 0) continue;
        const int L = a.seq_lens[s];
        const int ns = num_splits(L, split);
        for (int c = 0; c < ns - 1; ++c) a.plan_items[(size_t)(at.x + c) * Hkv + g] = make_int4(s, g, c, L);
        a.plan_items[(size_t)at.y * Hkv + g] = make_int4(s, g, ns - 1, L);
    }
    if (threadIdx.x == 0) {
        a.plan_count[0] = (total_full + total_last) * Hkv;
        a.plan_count[1] = split;
    }
}

// One work item as a warp holds it.
struct Item {
    int s, g, c, L, nsplit, t0, t1, nblk;
    bool valid;
};

template <int BS>
__device__ __forceinline__ Item load_item(const DecodeArgs &a, int k, int num_items, int split) {
    Item it;
    it.valid = k < num_items;
    const int4 v = it.valid ? a.plan_items[k] : make_int4(0, 0, 0, 0);
    it.s = v.x;
    it.g = v.y;
    it.c = v.z;
    it.L = v.w;
    it.nsplit = it.valid ? num_splits(it.L, split) : 1;
    it.t0 = it.c * split;
    it.t1 = it.c == it.nsplit - 1 ? it.L : it.t0 + split;
    it.nblk = it.valid ? (it.t1 - it.t0 + BS - 1) / BS : 0;  // t0 is block aligned
    return it;
}

template <int D, int BS, bool BIG_G, bool FP8>
__global__ void __launch_bounds__(kThreads, DecodeCfg<D, BS, FP8, BIG_G>::kCtasPerSm)
    decode_splitk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using C = DecodeCfg<D, BS, FP8, BIG_G>;
    constexpr int kS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    float *scratch = reinterpret_cast<float *>(smem + C::kScratchOff);
    uint8_t *qbuf = smem + C::kQOff;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *empty = full + kS;
    uint64_t *q_full = empty + kS;
    uint64_t *q_empty = q_full + 1;
    uint64_t *mq_full = q_empty + 1;           // [kMergeSlots] a merge request is in slot i
    uint64_t *mq_empty = mq_full + kMergeSlots;  // [kMergeSlots] the merge warp has taken slot i
    int *s_abort = reinterpret_cast<int *>(mq_empty + kMergeSlots);
    int4 *mq_slot = reinterpret_cast<int4 *>(s_abort + 4);  // (sequence, KV head, splits, -), or s < 0: no more
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, kConsumerWarps);
        for (int i = 0; i < kMergeSlots; ++i) {
            mbar_init(&mq_full[i], 1);
            mbar_init(&mq_empty[i], 1);
        }
        // validation mode: skip everything if an earlier pass found a bad
        // index (read once, so that the whole CTA takes the same branch)
        *s_abort = (a.check_err_first && *(volatile int *)a.err != 0) ? 1 : 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Everything below reads what the plan launch wrote (the items, the
    // appended rows): wait for it to complete.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (*(volatile int *)s_abort) return;

    const int num_items = a.plan_count[0], split = a.plan_count[1];
    const int nctas = gridDim.x;
    auto item_at = [&](int j) {  // the CTA's j-th item (snake order over the list)
        const int k = j * nctas + ((j & 1) ? nctas - 1 - (int)blockIdx.x : (int)blockIdx.x);
        return load_item<BS>(a, k, num_items, split);
    };

    // ---------------------------------------------------------- producer --
    if (warp == kConsumerWarps) {
        if (lane == kQLane) {
            // The items' G query rows, item after item, into the one q buffer,
            // each once the consumers have read the previous item's.
            const uint32_t qbytes = (uint32_t)a.group * 128u * C::kQHalves;
            tma_prefetch_desc(&tm_q);
            int j = 0;
            for (;; ++j) {
                const Item it = item_at(j);
                if (!it.valid) break;
                if (j >= 1 && !mbar_wait(q_empty, (j - 1) & 1, a.err)) {
                    atomicExch(s_abort, 1);
                    break;
                }
                mbar_arrive_expect_tx(q_full, qbytes);
                const int qrow = it.s * a.num_q_heads + it.g * a.group;
#pragma unroll
                for (int hf = 0; hf < C::kQHalves; ++hf) tma_load_2d(qbuf + hf * 2048, &tm_q, q_full, hf * 64, qrow);
            }
            // after a timed-out wait: wait (bounded) for the last load in flight
            if (j >= 1 && *(volatile int *)s_abort) mbar_wait(q_full, (j - 1) & 1, nullptr);
            return;
        }
        if (lane >= kS) return;
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        // Lane l fills stage l with the CTA's blocks l, l + kS, l + 2 kS, ...
        // (numbered across its items), each as soon as the consumer warp of
        // the stage has freed it, independently of the other lanes.
        int j = 0, base = 0;  // the item holding block gi, and its first block
        Item it = item_at(0);
        int last = -1;
        for (int gi = lane;; gi += kS) {
            while (it.valid && gi >= base + it.nblk) {
                base += it.nblk;
                it = item_at(++j);
            }
            if (!it.valid) break;
            const int i = gi - base;
            int32_t blk = a.block_table[(size_t)it.s * a.max_blocks + it.t0 / BS + i];
            if ((unsigned)blk >= (unsigned)a.num_blocks) {
                set_error(a.err, PA_ERR_BAD_INDEX);
                blk = 0;  // never dereference an out-of-range block
            }
            if (gi >= kS && !mbar_wait(&empty[lane], ((gi / kS) - 1) & 1, a.err)) {
                atomicExch(s_abort, 1);
                break;
            }
            mbar_arrive_expect_tx(&full[lane], C::kStageBytes);
            last = gi;
            uint8_t *sk = smem + lane * C::kStageBytes;
            uint8_t *sv = sk + C::kKVBytes;
            const int row = (blk * a.num_kv_heads + it.g) * BS;
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf) {
                tma_load_2d(sk + hf * C::kHalfBytes, &tm_k, &full[lane], hf * C::kBoxCols, C::kPacked ? row / 2 : row);
                tma_load_2d(sv + hf * C::kHalfBytes, &tm_v, &full[lane], hf * C::kBoxCols, C::kPacked ? row / 2 : row);
            }
        }
        // Every block issued is consumed before the consumers leave, unless a
        // wait timed out: then wait (bounded, not giving up on the error word)
        // for this lane's copy in flight before leaving.
        if (last >= 0 && *(volatile int *)s_abort) mbar_wait(&full[lane], (last / kS) & 1, nullptr);
        return;
    }

    // ------------------------------------------------------- merge warp --
    // The split-K merge, in this kernel: for every item of a split sequence
    // the consumers queue (sequence, KV head, splits) once its partials are
    // stored; this warp counts the item in the (sequence, KV head)'s merge
    // count with one acquire-release atomic, and the split that brings the
    // count to the number of splits merges them all.  The consumers' partial
    // stores reach the atomic through the queue's barrier (release / acquire
    // in the CTA) and the atomic's release at GPU scope, which covers what
    // this warp has observed; its acquire makes every other split's partials
    // visible, and they are read from L2 (never L1, which can hold older
    // copies of those lines).  The consumers never wait for any of this.
    if (warp == kMergeWarp) {
        const int G = a.group;
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int slot = n % kMergeSlots;
            if (!mbar_wait(&mq_full[slot], (n / kMergeSlots) & 1, a.err)) {
                atomicExch(s_abort, 1);
                break;
            }
            const int4 req = mq_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&mq_empty[slot]);
            if (req.x < 0) break;
            const int s = req.x, g = req.y, nsplit = req.z;
            uint32_t old = 0;
            if (lane == 0) {
                asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                             : "=r"(old)
                             : "l"(a.merge_cnt + (size_t)s * a.num_kv_heads + g)
                             : "memory");
            }
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old != (uint32_t)(nsplit - 1)) continue;
            // R rows of the group at a time, 32 / R lanes per row, CPL columns
            // per lane: every lane's loads of a split are independent of the
            // others', so a merge takes a few L2 round trips, not one per row.
            const int R = G >= 8 ? 8 : (G >= 4 ? 4 : (G >= 2 ? 2 : 1));
            const int lpr = 32 / R;           // lanes per row
            const int cpl = D / lpr;          // columns per lane: 4 .. 32 (D = 128), 2 .. 16 (D = 64)
            const int rl = lane / lpr, c0 = (lane % lpr) * cpl;
            for (int rb = 0; rb < G; rb += R) {
                const int row = rb + rl;
                const bool live = row < G;
                const size_t p0 = ((size_t)s * a.num_q_heads + g * G + (live ? row : 0)) * a.max_splits;
                const float *ml = a.part_ml + p0 * 2;
                float M = -INFINITY;
#pragma unroll 8
                for (int c = 0; c < nsplit; ++c) M = fmaxf(M, __ldcg(ml + c * 2));
                float accv[32], lsum = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e) accv[e] = 0.f;
#pragma unroll 4
                for (int c = 0; c < nsplit; ++c) {
                    const float2 mlc = __ldcg(reinterpret_cast<const float2 *>(ml + c * 2));
                    const float f = M == -INFINITY ? 0.f : fast_exp2(mlc.x - M);
                    lsum += f * mlc.y;
                    const float *pp = a.part_acc + (p0 + c) * D + c0;
                    if (cpl == 2) {  // D = 64, one row per pass
                        const float2 v = __ldcg(reinterpret_cast<const float2 *>(pp));
                        accv[0] += f * v.x;
                        accv[1] += f * v.y;
                    } else {
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            if (4 * e4 < cpl) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(pp) + e4);
                                accv[4 * e4 + 0] += f * v.x;
                                accv[4 * e4 + 1] += f * v.y;
                                accv[4 * e4 + 2] += f * v.z;
                                accv[4 * e4 + 3] += f * v.w;
                            }
                        }
                    }
                }
                if (live) {
                    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                    __nv_bfloat16 *o = a.out + ((size_t)s * a.num_q_heads + g * G + row) * D + c0;
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        if (e < cpl)
                            *reinterpret_cast<__nv_bfloat162 *>(o + e) =
                                __floats2bfloat162_rn(accv[e] * inv, accv[e + 1] * inv);
                }
            }
        }
        return;
    }

    // --------------------------------------------------------- consumers --
    // Byte offset of 16-byte chunk jj of token t in an fp8 K or V block (the
    // 128-byte swizzle XORs the chunk with the row's low three bits).
    auto kv_off = [](int t, int jj) -> uint32_t {
        if constexpr (C::kPacked) {
            const int pr = t >> 1;
            return pr * 128 + (((jj + 4 * (t & 1)) ^ (pr & 7)) << 4);
        } else {
            return t * 128 + ((jj ^ (t & 7)) << 4);
        }
    };
    const int G = a.group;
    const int r0 = lane >> 2;       // MMA row (query head within the group)
    const int cq = (lane & 3) * 2;  // first of the lane's two columns
    const uint32_t qb = smem_u32(qbuf);
    int base = 0;                   // the CTA-wide index of the item's first block
    int nreq = 0;                   // merge requests queued (warp 0)
    bool ok = true;
    for (int j = 0;; ++j) {
        const Item it = item_at(j);
        if (!it.valid) break;
        const int s = it.s, g = it.g, t0 = it.t0, t1 = it.t1, nblk = it.nblk;
        // ---- the item's query rows (row r of 64-column box hf at 2048 hf + 128 r, 128-byte swizzle)
        if (!mbar_wait(q_full, j & 1, a.err)) ok = false;
        uint32_t qa[C::kKSteps][4];
        auto q2 = [&](int row, int col) {  // bf16 pair (col, col + 1) of a row
            return row < G ? lds_u32(qb + (col >> 6) * 2048 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                                     (col & 7) * 2)
                           : 0u;
        };
        if (FP8) {
            // fp16 A fragments with the k-step's 16 columns permuted to match the
            // byte order ldmatrix gives the fp8 keys: MMA columns 2c, 2c+1 hold
            // d = 4c, 4c+1 and columns 2c+8, 2c+9 hold d = 4c+2, 4c+3 (c = lane % 4).
            const int c4 = (lane & 3) * 4;
            auto cvt = [](uint32_t v) {
                const float2 f = bf16x2_unpack(v);
                return pack_f16x2(f.x, f.y);
            };
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                qa[ks][0] = cvt(q2(r0, ks * 16 + c4));
                qa[ks][2] = cvt(q2(r0, ks * 16 + c4 + 2));
                qa[ks][1] = BIG_G ? cvt(q2(r0 + 8, ks * 16 + c4)) : 0u;
                qa[ks][3] = BIG_G ? cvt(q2(r0 + 8, ks * 16 + c4 + 2)) : 0u;
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                qa[ks][0] = q2(r0, ks * 16 + cq);
                qa[ks][2] = q2(r0, ks * 16 + 8 + cq);
                qa[ks][1] = BIG_G ? q2(r0 + 8, ks * 16 + cq) : 0u;
                qa[ks][3] = BIG_G ? q2(r0 + 8, ks * 16 + 8 + cq) : 0u;
            }
        }
        fence_proxy_async_smem();  // the next item's q load (async proxy) overwrites the buffer
        __syncwarp();
        if (lane == 0) mbar_arrive(q_empty);

        float acc[C::kNTiles][4];
#pragma unroll
        for (int nt = 0; nt < C::kNTiles; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};  // rows r0, r0 + 8 (log2 units)
        float l_run[2] = {0.f, 0.f};              // this lane's share of the row sums
        const float sl = FP8 ? a.scale_log2 * a.k_scale[g] : a.scale_log2;

        // This warp's blocks: CTA-wide index = warp mod 4 (the stage's reader),
        // i.e. the item's blocks i = role, role + 4, ...  The merge below goes
        // by role, not by warp, so an item's result does not depend on where
        // in the CTA's sequence of blocks it starts: the output is the same
        // whatever CTA or list position the plan gives the item.
        const int role = (warp - base % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
        for (int gi = base + role; ok && gi < base + nblk; gi += kConsumerWarps) {
            const int i = gi - base;
            const int st = gi % kS;
            if (!mbar_wait(&full[st], (gi / kS) & 1, a.err)) {
                ok = false;
                break;
            }
            const uint32_t sk = smem_u32(smem + st * C::kStageBytes);
            const uint32_t sv = sk + C::kKVBytes;
            const int tok0 = t0 + i * BS;
            const int valid = t1 - tok0;  // tokens of this block that belong to the sequence
            if (valid < BS) {
                // Rows past the end of the sequence hold stale pool contents; P is
                // zero there, but 0 * NaN would still poison the accumulator.
                uint8_t *vz = smem + st * C::kStageBytes + C::kKVBytes;
                if constexpr (C::kPacked) {
                    // token r: 16-byte chunks c + 4 (r % 2) of row r / 2, swizzled
                    for (int e = lane; valid + (e >> 2) < BS; e += 32) {
                        const int r = valid + (e >> 2), pr = r >> 1;
                        *reinterpret_cast<uint4 *>(vz + pr * 128 + ((((e & 3) + 4 * (r & 1)) ^ (pr & 7)) << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                } else {
                    for (int r = valid + (lane >> 3); r < BS; r += 4) {
#pragma unroll
                        for (int hf = 0; hf < C::kHalves; ++hf)
                            *reinterpret_cast<uint4 *>(vz + hf * C::kHalfBytes + r * 128 + (lane & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                __syncwarp();
            }
#pragma unroll
            for (int sb = 0; sb < BS / 16; ++sb) {
                if (sb * 16 >= valid) break;
                // ---- S = Q K^T over 16 keys (two n-tiles of 8 keys)
                float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                if (FP8) {
                    // one 16-byte chunk of a key row is one k-step; matrices: keys
                    // 0-7 / 8-15 x k-steps 2kp, 2kp+1.  A lane's 4 bytes are d = 4c..4c+3.
                    const int mat = lane >> 3;
                    const int t = sb * 16 + (lane & 7) + ((mat >> 1) << 3);
#pragma unroll
                    for (int kp = 0; kp < C::kKSteps / 2; ++kp) {
                        const int jj = 2 * kp + (mat & 1);
                        const uint32_t addr = sk + kv_off(t, jj);
                        uint32_t b00, b01, b10, b11;  // (keys 0-7, ks), (0-7, ks+1), (8-15, ks), (8-15, ks+1)
                        ldmatrix_x4(addr, b00, b01, b10, b11);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int ks = 2 * kp + u;
                            uint32_t l0, l1, h0, h1;
                            e4m3x4_to_f16x2x2(u ? b01 : b00, l0, l1);
                            e4m3x4_to_f16x2x2(u ? b11 : b10, h0, h1);
                            mma_f16_16816(sacc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], l0, l1);
                            mma_f16_16816(sacc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], h0, h1);
                        }
                    }
                } else {
                    const int mat = lane >> 3;
                    const int t = sb * 16 + (lane & 7) + ((mat >> 1) << 3);
#pragma unroll
                    for (int ks = 0; ks < C::kKSteps; ++ks) {
                        const int jj = 2 * ks + (mat & 1);  // 16-byte chunk over d
                        const uint32_t addr = sk + (jj >> 3) * C::kHalfBytes + t * 128 +
                                              ((((jj & 7) ^ (t & 7))) << 4);
                        uint32_t b00, b01, b10, b11;
                        ldmatrix_x4(addr, b00, b01, b10, b11);
                        mma_bf16_16816(sacc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
                        mma_bf16_16816(sacc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
                    }
                }
                // ---- online softmax (rows r0 and, for G > 8, r0 + 8)
                const int nvalid = valid - sb * 16;  // keys of this sub-block in the sequence
                float p[2][4];
                float alpha[2] = {1.f, 1.f};
#pragma unroll
                for (int rr = 0; rr < (BIG_G ? 2 : 1); ++rr) {
                    float x[4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = nt * 8 + cq + e;
                            x[nt * 2 + e] = key < nvalid ? sacc[nt][rr * 2 + e] * sl : -INFINITY;
                        }
                    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float mn = fmaxf(m_run[rr], mx);
                    alpha[rr] = fast_exp2(m_run[rr] - mn);
                    m_run[rr] = mn;
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[e] = fast_exp2(x[e] - mn);
                    // the running maximum rarely moves after the first blocks
                    if (__any_sync(0xffffffffu, alpha[rr] != 1.f)) {
#pragma unroll
                        for (int nt = 0; nt < C::kNTiles; ++nt) {
                            acc[nt][rr * 2 + 0] *= alpha[rr];
                            acc[nt][rr * 2 + 1] *= alpha[rr];
                        }
                    }
                    p[0][rr * 2 + 0] = x[0];
                    p[0][rr * 2 + 1] = x[1];
                    p[1][rr * 2 + 0] = x[2];
                    p[1][rr * 2 + 1] = x[3];
                }
                if (!BIG_G) {
                    p[0][2] = p[0][3] = p[1][2] = p[1][3] = 0.f;
                }
                auto pk = [&](float lo, float hi) { return FP8 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi); };
                auto psum = [&](uint32_t v) { return FP8 ? f16x2_sum(v) : bf16x2_sum(v); };
                const uint32_t pa0 = pk(p[0][0], p[0][1]);
                const uint32_t pa1 = pk(p[0][2], p[0][3]);
                const uint32_t pa2 = pk(p[1][0], p[1][1]);
                const uint32_t pa3 = pk(p[1][2], p[1][3]);
                // The row sums use the same rounded weights that multiply V, so the
                // output is an exact convex combination of the values.
                l_run[0] = l_run[0] * alpha[0] + (psum(pa0) + psum(pa2));
                if (BIG_G) l_run[1] = l_run[1] * alpha[1] + (psum(pa1) + psum(pa3));
                // ---- acc += P V over the same 16 keys
                if (FP8) {
                    // matrices: keys 0-7 / 8-15 x 16-byte d chunks 2jp, 2jp+1,
                    // transposed: a lane holds, per matrix, keys 2c, 2c+1 x d = 2n, 2n+1
                    // of the chunk (n = lane / 4).  Even d go to one n-tile, odd d
                    // to the next: acc[4 jp + 2 u + par] column 2c + e is
                    // d = 16 (2 jp + u) + 4c + 2e + par.
                    const int mat = lane >> 3;
                    const int t = sb * 16 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
                    for (int jp = 0; jp < D / 32; ++jp) {
                        const int jj = 2 * jp + (mat >> 1);
                        const uint32_t addr = sv + kv_off(t, jj);
                        uint32_t v0, v1, v2, v3;  // (keys 0-7, chunk 2jp), (8-15, 2jp), (0-7, 2jp+1), (8-15, 2jp+1)
                        ldmatrix_x4_trans(addr, v0, v1, v2, v3);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            // bytes (0, 2) -- the even d -- into the low half, (1, 3) into the high half
                            uint32_t le, lo_, he, ho;
                            e4m3x4_to_f16x2x2(__byte_perm(u ? v2 : v0, 0u, 0x3120u), le, lo_);
                            e4m3x4_to_f16x2x2(__byte_perm(u ? v3 : v1, 0u, 0x3120u), he, ho);
                            mma_f16_16816(acc[4 * jp + 2 * u + 0], pa0, pa1, pa2, pa3, le, he);
                            mma_f16_16816(acc[4 * jp + 2 * u + 1], pa0, pa1, pa2, pa3, lo_, ho);
                        }
                    }
                } else {
                    const int mat = lane >> 3;
                    const int t = sb * 16 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
                    for (int np = 0; np < C::kNTiles / 2; ++np) {
                        const int jj = 2 * np + (mat >> 1);
                        const uint32_t addr = sv + (jj >> 3) * C::kHalfBytes + t * 128 +
                                              ((((jj & 7) ^ (t & 7))) << 4);
                        uint32_t v0, v1, v2, v3;
                        ldmatrix_x4_trans(addr, v0, v1, v2, v3);
                        mma_bf16_16816(acc[2 * np], pa0, pa1, pa2, pa3, v0, v1);
                        mma_bf16_16816(acc[2 * np + 1], pa0, pa1, pa2, pa3, v2, v3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        base += nblk;

        // ------------------------------------------- merge the four states --
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
            l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
        }
        // element (row, column) of a lane's accumulator fragment
        auto col_of = [&](int nt, int e) {
            return FP8 ? 16 * (nt >> 1) + 4 * (lane & 3) + (nt & 1) + 2 * e : nt * 8 + cq + e;
        };
        auto put = [&](int slot) {  // this warp's state (its rows < G) into a scratch slot
            float *sa = scratch + slot * C::kSlotFloats;
#pragma unroll
            for (int rr = 0; rr < (BIG_G ? 2 : 1); ++rr) {
                const int row = r0 + rr * 8;
                if (row >= G) continue;
#pragma unroll
                for (int nt = 0; nt < C::kNTiles; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) sa[row * C::kRow + col_of(nt, e)] = acc[nt][rr * 2 + e];
                if ((lane & 3) == 0) {
                    sa[C::kRows * C::kRow + row * 2 + 0] = m_run[rr];
                    sa[C::kRows * C::kRow + row * 2 + 1] = l_run[rr];
                }
            }
        };
        auto take = [&](int slot) {  // combine a scratch slot into this warp's state
            const float *sa = scratch + slot * C::kSlotFloats;
#pragma unroll
            for (int rr = 0; rr < (BIG_G ? 2 : 1); ++rr) {
                const int row = r0 + rr * 8;
                if (row >= G) continue;
                const float mo = sa[C::kRows * C::kRow + row * 2 + 0], lo = sa[C::kRows * C::kRow + row * 2 + 1];
                const float M = fmaxf(m_run[rr], mo);
                const float fa = M == -INFINITY ? 0.f : fast_exp2(m_run[rr] - M);  // 0 for a warp that saw no key
                const float fb = M == -INFINITY ? 0.f : fast_exp2(mo - M);
#pragma unroll
                for (int nt = 0; nt < C::kNTiles; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        acc[nt][rr * 2 + e] = acc[nt][rr * 2 + e] * fa + sa[row * C::kRow + col_of(nt, e)] * fb;
                l_run[rr] = l_run[rr] * fa + lo * fb;
                m_run[rr] = M;
            }
        };
        auto csync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); };
        // The same barrier, true in every consumer thread if p holds in any.
        auto csync_any = [&](bool p) {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
                "bar.red.or.pred po, 1, %2, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
                : "=r"(r)
                : "r"((uint32_t)p), "n"(kConsumerWarps * 32)
                : "memory");
            return r != 0u;
        };
        // two steps: roles 1 and 3 into 0 and 2, then 2 into 0
        csync();  // every warp is done with the item; the previous merge's reads are done
        if (role & 1) put(role >> 1);
        csync();
        if (!(role & 1)) take(role >> 1);
        csync();
        if (role == 2) put(0);
        csync();
        if (role == 0) take(0);
        if (role == 0) {
            const float vs = FP8 ? a.v_scale[g] : 1.f;
#pragma unroll
            for (int rr = 0; rr < (BIG_G ? 2 : 1); ++rr) {
                const int row = r0 + rr * 8;
                if (row >= G) continue;
                const int h = g * G + row;
                if (it.nsplit == 1) {
                    const float inv = l_run[rr] > 0.f ? vs / l_run[rr] : 0.f;
                    __nv_bfloat16 *o = a.out + ((size_t)s * a.num_q_heads + h) * D;
#pragma unroll
                    for (int nt = 0; nt < C::kNTiles; ++nt) {
                        if (FP8) {
                            o[col_of(nt, 0)] = __float2bfloat16_rn(acc[nt][rr * 2 + 0] * inv);
                            o[col_of(nt, 1)] = __float2bfloat16_rn(acc[nt][rr * 2 + 1] * inv);
                        } else {
                            *reinterpret_cast<__nv_bfloat162 *>(o + col_of(nt, 0)) =
                                __floats2bfloat162_rn(acc[nt][rr * 2 + 0] * inv, acc[nt][rr * 2 + 1] * inv);
                        }
                    }
                } else {
                    const size_t pi = ((size_t)s * a.num_q_heads + h) * a.max_splits + it.c;
                    float *pacc = a.part_acc + pi * D;
#pragma unroll
                    for (int nt = 0; nt < C::kNTiles; ++nt) {
                        if (FP8) {
                            pacc[col_of(nt, 0)] = acc[nt][rr * 2 + 0] * vs;
                            pacc[col_of(nt, 1)] = acc[nt][rr * 2 + 1] * vs;
                        } else {
                            *reinterpret_cast<float2 *>(pacc + col_of(nt, 0)) =
                                make_float2(acc[nt][rr * 2 + 0], acc[nt][rr * 2 + 1]);
                        }
                    }
                    if ((lane & 3) == 0) {
                        a.part_ml[pi * 2 + 0] = m_run[rr];
                        a.part_ml[pi * 2 + 1] = l_run[rr];
                    }
                }
            }
        }
        // Every consumer warp takes the same barriers, and all leave together
        // once a wait has failed here or anywhere in the CTA: one barrier
        // reduction decides it for all (a flag read after a plain barrier
        // could change between the warps' reads).
        if (csync_any(!ok || *(volatile int *)s_abort != 0)) {
            if (!ok) atomicExch(s_abort, 1);
            break;
        }
        if (it.nsplit > 1 && warp == 0) {
            // Queue the merge request (always from warp 0, which counts the
            // queue's slots): the partials were stored by the role-0 warp
            // before the barrier above, and the slot's arrival releases them
            // to the merge warp.
            if (lane == 0) {
                const int slot = nreq % kMergeSlots;
                if (nreq < kMergeSlots || mbar_wait(&mq_empty[slot], ((nreq / kMergeSlots) - 1) & 1, a.err)) {
                    mq_slot[slot] = make_int4(s, g, it.nsplit, 0);
                    mbar_arrive(&mq_full[slot]);
                } else {
                    ok = false;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            ++nreq;
        }
    }
    // no more merge requests: the merge warp leaves once it has taken this
    if (warp == 0 && lane == 0) {
        const int slot = nreq % kMergeSlots;
        if (nreq < kMergeSlots || mbar_wait(&mq_empty[slot], ((nreq / kMergeSlots) - 1) & 1, a.err)) {
            mq_slot[slot] = make_int4(-1, 0, 0, 0);
            mbar_arrive(&mq_full[slot]);
        } else {
            atomicExch(s_abort, 1);
        }
    }
}

template <int D, int BS, bool BIG_G, bool FP8>
cudaError_t launch_decode_t(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                            const DecodeArgs &a, int num_sms, cudaStream_t stream) {
    using C = DecodeCfg<D, BS, FP8, BIG_G>;
    static std::atomic<unsigned long long> opted{0};
    cudaError_t e = opt_in_smem(reinterpret_cast<const void *>(decode_splitk_kernel<D, BS, BIG_G, FP8>),
                                C::kSmemBytes, opted);
    if (e != cudaSuccess) return e;
    // Persistent: as many CTAs per SM as fit, fewer when the items (counted
    // on the device; at most every split of every sequence) cannot fill them.
    const long long bound = (long long)a.num_seqs * a.num_kv_heads * a.max_splits;
    const long long ctas =
        std::max(1LL, std::min<long long>((long long)C::kCtasPerSm * std::max(num_sms, 1), bound));
    DecodeArgs b = a;
    b.num_ctas = (int)ctas;
    // the plan's CTA, plus CTAs for the fused append (up to one per SM)
    int plan_ctas = 1;
    if (b.k_new) {
        const long long pieces = (long long)b.num_seqs * b.num_kv_heads * (D / 8);
        plan_ctas += (int)std::min<long long>(std::max(num_sms, 1), (pieces + 1023) / 1024);
    }
    decode_plan_kernel<D, BS><<<plan_ctas, 1024, 0, stream>>>(b);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the decode kernel's CTAs are placed
    // while the plan launch still runs and wait for it in griddepcontrol.wait,
    // so the launch gap between the two overlaps the plan.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_splitk_kernel<D, BS, BIG_G, FP8>, tm_q, tm_k, tm_v, b);
}

}  // namespace

int decode_split_tokens(int num_seqs, int num_kv_heads, int max_seq_len, int block_size,
                        int num_sms, int override_tokens) {
    if (override_tokens > 0)
        return ((override_tokens + block_size - 1) / block_size) * block_size;
    // Splits of 512 tokens keep the tail of a ragged batch short; drop to 256
    // when that still leaves fewer than eight CTAs per SM to schedule.
    int split = 512;
    const long long pairs = (long long)num_seqs * num_kv_heads;
    const long long units = pairs * ((max_seq_len + split - 1) / split);
    if (units < 8LL * num_sms) split = 256;
    return ((split + block_size - 1) / block_size) * block_size;
}

int decode_max_splits(int max_seq_len, int split_tokens) {
    return max_seq_len > 0 ? (max_seq_len + split_tokens - 1) / split_tokens : 1;
}

// Layout: [part_acc S*Hq*max_splits*d floats][part_ml S*Hq*max_splits*2
// floats] (only when max_splits > 1), then the plan, 16-byte aligned:
// [items: S * max_splits * Hkv int4][count: 4 ints][per sequence: int2]
// [merge counts: S * Hkv ints] (the last only when max_splits > 1).
static size_t partials_bytes(int num_seqs, int num_q_heads, int head_dim, int max_splits) {
    if (max_splits <= 1) return 0;
    const size_t n = (size_t)num_seqs * num_q_heads * max_splits;
    return (n * head_dim * sizeof(float) + n * 2 * sizeof(float) + 15) & ~size_t(15);
}

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_splits) {
    return partials_bytes(num_seqs, num_q_heads, head_dim, max_splits) +
           (size_t)num_seqs * std::max(max_splits, 1) * num_kv_heads * sizeof(int4) + 4 * sizeof(int) +
           (size_t)num_seqs * sizeof(int2) + (max_splits > 1 ? (size_t)num_seqs * num_kv_heads * sizeof(int) : 0);
}

void decode_plan_layout(void *ws, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_splits,
                        int4 **items, int **count, int2 **seq, int **merge_cnt) {
    uint8_t *p = static_cast<uint8_t *>(ws) + partials_bytes(num_seqs, num_q_heads, head_dim, max_splits);
    *items = reinterpret_cast<int4 *>(p);
    p += (size_t)num_seqs * std::max(max_splits, 1) * num_kv_heads * sizeof(int4);
    *count = reinterpret_cast<int *>(p);
    *seq = reinterpret_cast<int2 *>(p + 4 * sizeof(int));
    *merge_cnt = max_splits > 1 ? reinterpret_cast<int *>(p + 4 * sizeof(int) + (size_t)num_seqs * sizeof(int2))
                                : nullptr;
}

cudaError_t launch_decode(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          const DecodeArgs &a, int head_dim, int block_size, int num_sms, cudaStream_t stream,
                          bool fp8) {
    const bool big = a.group > 8;
#define PA_DEC(D, BS, F8)                                                                   \
    if (head_dim == D && block_size == BS && fp8 == F8)                                     \
        return big ? launch_decode_t<D, BS, true, F8>(tm_q, tm_k, tm_v, a, num_sms, stream) \
                   : launch_decode_t<D, BS, false, F8>(tm_q, tm_k, tm_v, a, num_sms, stream);
    PA_DEC(128, 16, false)
    PA_DEC(128, 32, false)
    PA_DEC(64, 16, false)
    PA_DEC(64, 32, false)
    PA_DEC(128, 16, true)
    PA_DEC(128, 32, true)
    PA_DEC(64, 16, true)
    PA_DEC(64, 32, true)
#undef PA_DEC
    return cudaErrorInvalidValue;
}

}  // namespace pa
