// prefill_tc2.cu -- causal, ragged (varlen-packed) prefill attention for
// head_dim 128 on CTA pairs: every tcgen05.mma is an M = 256 instruction
// issued once for two SMs (cta_group::2).
//
// What it computes (text-generation-inference Router/Webserver deep dive,
// section "Prefill, Decode and past key values"; ragged index pointers as in
// the Blitzscale docs, section "Model"): row i of sequence s sits at absolute
// position p0 + i and
//     out = softmax(scale * q K^T + causal mask) V   over keys 0 .. p0 + i.
//
// Why pairs: a lone SM reaches the dense tensor peak with 128x128x16 MMAs
// too, but then every MMA also streams all of B (K or V) from its own shared
// memory; shared-memory bandwidth (operand reads + TMA writes) is what bounds
// this kernel.  An M = 256 instruction issued once for two SMs (cta_group::2)
// reads half of B in each CTA, and each CTA loads half of every K/V tile.
//
// Work unit: four 128-row query tiles that read the same KV head -- four
// query heads of one group (group size a multiple of 4), two heads x two row
// tiles (even group size), or four consecutive row tiles of one head.  CTA c
// of a pair holds two of them as sub-tiles k = 0, 1; the pair's sub-tile k is
// one M = 256 MMA operand (CTA 0's rows, then CTA 1's).
//   K tile (128 keys): CTA c loads keys 64c .. 64c+63 (the MMA's B is split
//     along N between the pair), both 64-column halves of d.
//   V tile (128 keys): CTA c loads all keys, d columns 64c .. 64c+63.
//   S_k = Q_k K^T (M=256, N=128, K=128) -> each CTA's TMEM S_k (128 columns).
//   Softmax (two threads per row = TMEM lane, one per 64-key half) writes
//     P_k (bf16 pairs) over S_k columns 0-31 (keys 0-63) and 64-95 (keys
//     64-127), then arrives on the leader.
//   O_k += P_k V (A from TMEM, M=256, N=128: the two d halves, K=128 keys).
//   Per KV tile the leader issues PV_0(t), S_0(t+1), PV_1(t), S_1(t+1): while
//   the tensor core works for one sub-tile the other's softmax runs.  S_k(t+1)
//   overwrites P_k(t) and so waits for PV_k(t) (in-order tensor pipe).
// Persistent: one pair per two SMs walks the work units, dealt longest first
// in rounds of alternating direction, so a pair's prologue and epilogue
// overlap its neighbours' work.  The next unit's Q lands in the other of two Q
// buffers while the current unit runs; the K/V ring and every barrier run on
// across units.
// Warps (four warpgroups; registers moved between them with setmaxnreg):
//   0, 1  issue (leader CTA only) the MMAs of sub-tiles 0 and 1 -- a thread
//         stalls for hundreds of cycles on each mbarrier test, and the other
//         thread's queued MMAs keep the tensor core busy meanwhile; warp 0
//         also allocates TMEM (both CTAs);
//   2     TMA producer;
//   3     tail: zeroes the rows of a unit's last V tile past its last key
//         (stale pool rows could hold NaN, and 0 * NaN = NaN), then tells the
//         leader the tile is ready -- off the producer, which runs on into the
//         next unit's loads meanwhile;
//   4-11  softmax, for both sub-tiles in turn (warp w: rows 32 (w % 4) .. +31,
//         TMEM lane quadrant w % 4; warps 4-7 keys 0-63 of each tile, 8-11
//         keys 64-127).  The two sub-tiles' softmaxes alternate in time anyway
//         (each waits on its own MMAs), so all eight warps take each one: two
//         warps per row on every SM sub-partition roughly halve the softmax's
//         latency, which sets the length of each sub-tile's S -> softmax -> PV
//         chain.  At a sub-tile's last tile they post its row sums and go on
//         to the next unit;
//   12-15 epilogue (warp w: rows of quadrant w % 4): read O_k out of TMEM
//         (releasing it for the next unit's first PV_k), normalise by the row
//         sums, stage the rows in the unit's finished Q buffer and store them
//         with TMA -- while the softmax warps already work on the next unit.
// Loads signal the leader's barriers (cp.async.bulk.tensor .cta_group::2);
// the leader's commits signal both CTAs (multicast).
#include <cuda.h>

#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                       // rows per query sub-tile (per CTA)
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kMmaWarp = 0;        // and kMmaWarp + 1
constexpr int kProducerWarp = 2;
constexpr int kTailWarp = 3;
constexpr int kSoftmaxWarp0 = 4;   // 4 .. 11
constexpr int kEpilogueWarp0 = 12; // 12 .. 15
constexpr int kThreads = 512;
// Registers per thread of each warpgroup after setmaxnreg.  The launch gives
// every thread 65536 / 512 = 128 (the host checks the kernel's count before
// the first launch); the four shares add up to 4 x 128, so every increase is
// covered by the decreases.
constexpr int kRegsControl = 80;   // warps 0-3
constexpr int kRegsSoftmax = 160;  // warps 4-11
constexpr int kRegsEpilogue = 112; // warps 12-15
static_assert(kRegsControl + 2 * kRegsSoftmax + kRegsEpilogue == 4 * (65536 / kThreads), "register split");
static_assert(kRegsControl % 8 == 0 && kRegsSoftmax % 8 == 0 && kRegsEpilogue % 8 == 0, "setmaxnreg granularity");
constexpr uint32_t kTmemCols = 512;            // S_0, S_1, O_0, O_1
constexpr int kBox = 128 * 128;                // one [128 rows][64 bf16] swizzled box set
constexpr int kQBytes = 2 * kBox;              // Q_k: [128][128]
constexpr int kKHalf = 64 * 128;               // [64 keys][64 d]
constexpr int kKBytes = 2 * kKHalf;            // K: 64 keys x 128 d (per CTA)
constexpr int kVBytes = 128 * 128;             // V: 128 keys x 64 d (per CTA)
constexpr int kStageBytes = kKBytes + kVBytes; // one KV tile: K then V
constexpr int kQOff = 0;                       // Q buffers [2 units][2 sub-tiles]
constexpr int kRingOff = 4 * kQBytes;
constexpr int kStages = 3;                     // K/V ring
constexpr int kBarOff = kRingOff + kStages * kStageBytes;
constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 * 4 + 2 + 2 + 2 + 4;
// The schedule: with at most kSeqMax sequences and kMaxLevels row-tile levels
// the units are dealt from a list in shared memory that holds non-empty units
// only; otherwise every (level, head group, sequence) slot is dealt and empty
// ones are skipped.
constexpr int kSeqMax = 256;                             // sequences in the shared-memory schedule
constexpr int kSeqInfoMax = 32;                          // ... with (row0, n, p0) cached there too
constexpr int kMaxLevels = 64;                           // row-tile levels (units per head and sequence)
constexpr int kSeqKeyOff = kBarOff + kNumBars * 8 + 16;  // uint8 [kSeqMax]: a sequence's levels
constexpr int kSeqOrderOff = kSeqKeyOff + kSeqMax;       // uint16 [kSeqMax]: sequences, most levels first
constexpr int kSeqInfoOff = kSeqOrderOff + kSeqMax * 2;  // int [kSeqInfoMax][3]: row0, n, p0
constexpr int kLevelOff = kSeqInfoOff + kSeqInfoMax * 12;   // int [kMaxLevels + 1]: units above a level
constexpr int kCountOff = kLevelOff + (kMaxLevels + 1) * 4; // int [kMaxLevels + 1]: scratch counts
constexpr int kXchgOff = kCountOff + (kMaxLevels + 1) * 4;  // float [kBM]: a row's max / sum between its halves
constexpr int kSmemBytes = kXchgOff + kBM * 4;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kSeqInfoOff % 4 == 0 && kXchgOff % 4 == 0, "alignment");

struct RowTile {
    int h, q0, rows, kv_end;
};

// MODE 0: four heads x one row tile; 1: two heads x two row tiles;
// 2: one head x four row tiles.  y indexes the head group of the unit.
template <int MODE>
__device__ __forceinline__ void row_tile(RowTile &rt, int c, int k, int px, int y, int n, int p0) {
    if (MODE == 0) {
        rt.h = 4 * y + 2 * c + k;
        rt.q0 = px * kBM;
    } else if (MODE == 1) {
        rt.h = 2 * y + c;
        rt.q0 = (2 * px + k) * kBM;
    } else {
        rt.h = y;
        rt.q0 = (4 * px + 2 * k + c) * kBM;
    }
    rt.rows = max(0, min(kBM, n - rt.q0));
    rt.kv_end = p0 + min(n, rt.q0 + kBM);
}

// One work unit, identical in both CTAs and all roles (scalars only, so that
// it lives in registers).
struct Unit {
    int s, px, y, row0, n, p0, g, T, kv_end_max, nkt0, nkt1;
};

// This CTA's sub-tile k of unit u.
template <int MODE>
__device__ __forceinline__ RowTile my_tile(const Unit &u, int c, int k) {
    RowTile rt;
    row_tile<MODE>(rt, c, k, u.px, u.y, u.n, u.p0);
    return rt;
}

constexpr int per_pair(int mode) { return mode == 0 ? 1 : (mode == 1 ? 2 : 4); }   // row tiles per head
constexpr int heads_per_pair(int mode) { return mode == 0 ? 4 : (mode == 1 ? 2 : 1); }

// Unit v (longest causal rows first): false if it has no rows (or its
// sequence's arguments are invalid, which is recorded in the error word).
// A sequence's query rows, prefix and validity (bad arguments are recorded
// in the error word; the sequence then has no work).
template <bool PAGED, int BS>
__device__ __forceinline__ bool seq_rows(const PrefillArgs &a, int s, int &row0, int &n, int &p0) {
    row0 = a.cu_seqlens[s];
    n = a.cu_seqlens[s + 1] - row0;
    p0 = a.prefix_lens ? a.prefix_lens[s] : (a.seq_lens ? a.seq_lens[s] - n : 0);
    const bool bad = n < 0 || p0 < 0 || row0 < 0 || (long long)row0 + n > a.num_tokens || n > a.max_q_len ||
                     (PAGED && (p0 + n + BS - 1) / BS > a.max_blocks) || (!PAGED && p0 != 0);
    if (bad) set_error(a.err, PA_ERR_BAD_INDEX);
    return !bad;
}

// The unit dealt as number v (longest causal rows first): false if it has no
// rows.  In the compact schedule, level lvl (row tile px = npx - 1 - lvl) holds
// ny units for each sequence with more than px levels, in the order of
// seq_order; `lvl` is the caller's cursor (v only grows).  Otherwise v walks
// every (level, sequence, head group) slot.  A sequence's (row0, n, p0) comes
// from shared memory for the first kSeqInfoMax sequences.
template <bool PAGED, int BS, int MODE>
__device__ __forceinline__ bool unit_at(const PrefillArgs &a, const uint8_t *smem, bool compact, int npx, int ny,
                                        int v, int &lvl, Unit &u) {
    const int *lcum = reinterpret_cast<const int *>(smem + kLevelOff);
    const int *seq_info = reinterpret_cast<const int *>(smem + kSeqInfoOff);
    if (compact) {
        while (lvl < npx && v >= lcum[lvl + 1]) ++lvl;
        if (lvl >= npx) return false;
        const int r = v - lcum[lvl];
        u.px = npx - 1 - lvl;
        u.y = r % ny;
        u.s = reinterpret_cast<const uint16_t *>(smem + kSeqOrderOff)[r / ny];
    } else {
        u.px = npx - 1 - v / (ny * a.num_seqs);
        const int rem = v % (ny * a.num_seqs);
        u.y = rem % ny;
        u.s = rem / ny;
    }
    if (u.s < kSeqInfoMax) {
        u.row0 = seq_info[3 * u.s];
        u.n = seq_info[3 * u.s + 1];
        u.p0 = seq_info[3 * u.s + 2];
    } else if (!seq_rows<PAGED, BS>(a, u.s, u.row0, u.n, u.p0)) {
        return false;
    }
    if (u.px * per_pair(MODE) * kBM >= u.n) return false;
    RowTile rt[2][2];  // [cta][sub-tile]
#pragma unroll
    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int k = 0; k < 2; ++k) row_tile<MODE>(rt[cc][k], cc, k, u.px, u.y, u.n, u.p0);
    int e[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        e[k] = 0;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
            if (rt[cc][k].rows > 0) e[k] = max(e[k], rt[cc][k].kv_end);
    }
    u.nkt0 = (e[0] + kBN - 1) / kBN;
    u.nkt1 = (e[1] + kBN - 1) / kBN;
    u.kv_end_max = max(e[0], e[1]);
    u.T = max(u.nkt0, u.nkt1);
    u.g = rt[0][0].h / a.group;
    return u.T > 0;
}

template <int BS, bool PAGED, int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const PrefillArgs a) {
    // Dynamic shared memory starts 1024-byte aligned (checked below: the
    // swizzled TMA/MMA buffers need it).
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *q_full = bar;                     // [2] leader: a unit's Q landed in both CTAs (Q buffer b)
    uint64_t *q_free = q_full + 2;              // [2] local: Q buffer b is free -- both issuers' S MMAs of its
                                                //     unit completed and the 4 epilogue warps' staging in it is read
    uint64_t *tile_full = q_free + 2;           // [kStages] leader: K and V of a tile landed in both CTAs
    uint64_t *tile_free = tile_full + kStages;  // [kStages] both sub-tiles' MMAs on the tile have completed
    uint64_t *s_full = tile_free + kStages;     // [2] S_k(t) is in TMEM (commit, both CTAs)
    uint64_t *p_full = s_full + 2;              // [2] leader: P_k(t) stored by the 16 softmax warps of the pair
    uint64_t *o_done = p_full + 2;              // [2] a unit's last PV_k has completed (commit, both CTAs)
    uint64_t *o_free = o_done + 2;              // [2] leader: the 8 epilogue warps of the pair have read O_k out
    uint64_t *v_last = o_free + 2;              // [2] local (unit parity): this CTA's half of a unit's last V tile landed
    uint64_t *v_tail = v_last + 2;              // [2] leader (unit parity): both halves zeroed past the last key
    uint64_t *mma_fin = v_tail + 2;             // [2] leader: every MMA issued by thread k has completed
    uint64_t *l_ready = mma_fin + 2;            // [2 unit parity][2 sub-tiles] local: the row sums are posted
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar + kNumBars);
    int *s_abort = reinterpret_cast<int *>(s_tmem + 1);
    volatile int *turn_cnt = reinterpret_cast<volatile int *>(s_abort + 1);  // [2] groups queued by thread k
    uint8_t *seq_key = smem + kSeqKeyOff;
    uint16_t *seq_order = reinterpret_cast<uint16_t *>(smem + kSeqOrderOff);
    int *seq_info = reinterpret_cast<int *>(smem + kSeqInfoOff);
    int *lcum = reinterpret_cast<int *>(smem + kLevelOff);
    int *cnt = reinterpret_cast<int *>(smem + kCountOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = (int)cluster_ctarank();
    const int pairs = (int)(gridDim.x >> 1), pair = (int)(blockIdx.x >> 1);
    const int npx = (a.num_q_tiles + per_pair(MODE) - 1) / per_pair(MODE);  // levels
    const int ny = a.num_q_heads / heads_per_pair(MODE);                       // head groups
    const bool compact = a.num_seqs <= kSeqMax && npx <= kMaxLevels;
    // Units are numbered longest first; round rnd deals them to the pairs in
    // alternating directions, which evens out the pairs' total work.
    auto unit_of = [&](int rnd) { return rnd * pairs + ((rnd & 1) ? pairs - 1 - pair : pair); };

    // Under a programmatic dependent launch the CTAs are placed while the
    // previous kernel on the stream finishes (e.g. the append that writes the
    // prompt rows' K/V): nothing is read from global memory before its writes
    // are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // The schedule (identical in both CTAs): each sequence's level count
    // (key), the number of sequences above each level, and the sequences
    // ordered by key, most first (stable, so both CTAs agree).
    if (compact)
        for (int j = threadIdx.x; j <= npx; j += kThreads) cnt[j] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < a.num_seqs && (compact || i < kSeqInfoMax); i += kThreads) {
        int row0, n, p0;
        const bool good = seq_rows<PAGED, BS>(a, i, row0, n, p0);
        if (i < kSeqInfoMax) {
            seq_info[3 * i] = row0;
            seq_info[3 * i + 1] = good ? n : 0;
            seq_info[3 * i + 2] = p0;
        }
        if (compact) {
            const int key = good ? ((n + kBM - 1) / kBM + per_pair(MODE) - 1) / per_pair(MODE) : 0;
            seq_key[i] = (uint8_t)key;
            atomicAdd(&cnt[key], 1);
        }
    }
    __syncthreads();
    if (compact && warp == kSoftmaxWarp0) {
        if (lane == 0) {
            // cnt[j] becomes the number of sequences with more than j levels
            // (= the first slot of key j in the descending order)
            int acc = 0;
            for (int j = npx; j >= 0; --j) {
                const int h = cnt[j];
                cnt[j] = acc;
                acc += h;
            }
            int cum = 0;
            lcum[0] = 0;
            for (int l = 0; l < npx; ++l) {
                cum += ny * cnt[npx - 1 - l];
                lcum[l + 1] = cum;
            }
        }
        __syncwarp();
        for (int b0 = 0; b0 < a.num_seqs; b0 += 32) {
            const int i = b0 + lane;
            const int key = i < a.num_seqs ? (int)seq_key[i] : -1;
            const unsigned grp = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(grp & ((1u << lane) - 1u));
            if (key > 0) seq_order[cnt[key] + rank] = (uint16_t)i;
            __syncwarp();
            if (key > 0 && rank == 0) cnt[key] += __popc(grp);
            __syncwarp();
        }
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&q_full[b], 1);
            mbar_init(&q_free[b], 2 + 4);  // one commit per issuing thread, one arrival per epilogue warp
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 2 * 8);  // one arrival per softmax warp of each CTA
            mbar_init(&o_done[b], 1);
            mbar_init(&o_free[b], 2 * 4);  // one arrival per epilogue warp of each CTA
            mbar_init(&v_last[b], 1);
            mbar_init(&v_tail[b], 2);      // one arrival per CTA's tail warp
            mbar_init(&mma_fin[b], 1);
            mbar_init(&l_ready[2 * b], 4);  // the key-half-0 softmax warps post the rows' sums
            mbar_init(&l_ready[2 * b + 1], 4);
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&tile_full[i], 1);
            mbar_init(&tile_free[i], 2);  // one commit per issuing thread (two if one sub-tile reads the tile)
        }
        turn_cnt[0] = 0;
        turn_cnt[1] = 0;
        // Validation mode: the leader's reading of the error word decides for
        // both CTAs (it may change while the kernel runs).
        *s_abort = (a.check_err_first && *(volatile int *)a.err != 0) ? 1 : 0;
        if (smem_u32(smem) & 1023u) {  // never seen; refuse rather than compute garbage
            set_error(a.err, PA_ERR_UNSUPPORTED);
            *s_abort = 1;
        }
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc_pair(s_tmem, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before anything signals them
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const bool skip = ld_shared_cluster(map_to_cta(smem_u32(s_abort), 0)) != 0;
    const int num_units = compact ? lcum[npx] : npx * ny * a.num_seqs;

    // Each warpgroup takes its share of the registers: every warp of a
    // warpgroup executes the same setmaxnreg at the top of its branch, and the
    // increases wait for the decreases.
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
        if (skip) {
            // nothing to do: fall through to the pair-wide teardown
        } else if (warp == kProducerWarp) {
            // ---------------------------------------------------------- producer --
            constexpr int kBPT = kBN / BS;  // pool blocks per 128-key tile
            constexpr int kTPG = 32 / kBPT;  // tiles per lane group of block ids
            const int oob_row = a.num_blocks * a.num_kv_heads * BS;  // past the pool: TMA fills zeros
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
            }
            int ord = 0, gb = 0, lvl = 0;  // units done, global index of the unit's first tile, schedule cursor
            bool ok = true;
            for (int rnd = 0; rnd * pairs < num_units && ok; ++rnd) {
                const int v = unit_of(rnd);
                if (v >= num_units) continue;
                Unit u;
                if (!unit_at<PAGED, BS, MODE>(a, smem, compact, npx, ny, v, lvl, u)) continue;
                const int qb = ord & 1;
                // Q buffer qb is free once unit ord - 2 is done with it (S MMAs, output staging).
                if (lane == 0 && ord >= 2) ok = mbar_wait(&q_free[qb], ((ord >> 1) - 1) & 1, a.err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok || *(volatile int *)s_abort) break;
                const uint32_t lq = map_to_cta(smem_u32(&q_full[qb]), 0);
                if (lane == 0 && c == 0) mbar_arrive_expect_tx(&q_full[qb], 2 * 2 * kQBytes);
                __syncwarp();
                if (lane < 4) {  // lane = 2 sub-tile + half
                    const RowTile rt = my_tile<MODE>(u, c, lane >> 1);
                    tma_load_3d_pair(smem + kQOff + (2 * qb + (lane >> 1)) * kQBytes + (lane & 1) * kBox, &tm_q, lq,
                                     (lane & 1) * 64, rt.h, u.row0 + rt.q0);
                }
                // Pool rows of the unit's blocks: lane l holds block 32 j + l of
                // lane group j (kTPG tiles); the next group's entries are loaded
                // while the current group is issued.  Each TMA copy of a tile is
                // issued by its own lane.
                const int nb_used = (u.kv_end_max + BS - 1) / BS;
                auto block_row = [&](int bi, const int32_t *btab) {
                    int row = oob_row;
                    if (bi < nb_used) {
                        int blk = btab[bi];
                        if ((unsigned)blk >= (unsigned)a.num_blocks) {
                            set_error(a.err, PA_ERR_BAD_INDEX);
                            blk = 0;  // never dereference an out-of-range block
                        }
                        row = (blk * a.num_kv_heads + u.g) * BS;
                    }
                    return row;
                };
                const int32_t *btab = PAGED ? a.block_table + (size_t)u.s * a.max_blocks : nullptr;
                int row_cur = 0, row_nxt = 0;
                if (PAGED) {
                    row_cur = block_row(lane, btab);
                    row_nxt = block_row(32 + lane, btab);
                }
                for (int t = 0; t < u.T; ++t) {
                    if (PAGED && t > 0 && t % kTPG == 0) {
                        row_cur = row_nxt;
                        row_nxt = block_row((t / kTPG + 1) * 32 + lane, btab);
                    }
                    const int base = (t % kTPG) * kBPT;
                    const int gt = gb + t, st = gt % kStages;
                    uint8_t *dk = smem + kRingOff + st * kStageBytes;
                    uint8_t *dv = dk + kKBytes;
                    if (lane == 0 && gt >= kStages) ok = mbar_wait(&tile_free[st], ((gt / kStages) - 1) & 1, a.err);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok || *(volatile int *)s_abort) break;
                    const bool last = (t == u.T - 1);
                    const uint32_t lb = map_to_cta(smem_u32(&tile_full[st]), 0);
                    if (lane == 0 && c == 0) mbar_arrive_expect_tx(&tile_full[st], last ? 2 * kKBytes : 2 * kStageBytes);
                    // K: this CTA's 64 keys, both halves of d (lane = 2 block + half)
                    const int jb = (lane >> 1) & (64 / BS - 1), hf = lane & 1;
                    const int krow = PAGED ? __shfl_sync(0xffffffffu, row_cur, base + c * (64 / BS) + jb) : 0;
                    if (PAGED) {
                        if (lane < 2 * (64 / BS))
                            tma_load_2d_pair(dk + hf * kKHalf + jb * BS * 128, &tm_k, lb, hf * 64, krow);
                    } else if (lane < 2) {
                        tma_load_3d_pair(dk + hf * kKHalf, &tm_k, lb, hf * 64, u.g, u.row0 + t * kBN + 64 * c);
                    }
                    // V: all 128 keys, this CTA's half of d (lane = block)
                    const int vrow = PAGED ? __shfl_sync(0xffffffffu, row_cur, base + (lane & (kBPT - 1))) : 0;
                    if (!last) {
                        if (PAGED) {
                            if (lane < kBPT) tma_load_2d_pair(dv + lane * BS * 128, &tm_v, lb, c * 64, vrow);
                        } else if (lane == 0) {
                            tma_load_3d_pair(dv, &tm_v, lb, c * 64, u.g, u.row0 + t * kBN);
                        }
                    } else {
                        // The last V tile lands against a local barrier; the tail
                        // warp zeroes its rows past the last key and tells the
                        // leader, while this warp goes on to the next unit.
                        uint64_t *vl = &v_last[ord & 1];
                        if (lane == 0) mbar_arrive_expect_tx(vl, kVBytes);
                        __syncwarp();
                        if (PAGED) {
                            if (lane < kBPT) tma_load_2d(dv + lane * BS * 128, &tm_v, vl, c * 64, vrow);
                        } else if (lane == 0) {
                            tma_load_3d(dv, &tm_v, vl, c * 64, u.g, u.row0 + t * kBN);
                        }
                    }
                    __syncwarp();
                }
                gb += u.T;
                ++ord;
            }
            if (!ok && lane == 0) atomicExch(s_abort, 1);
        } else if (warp == kTailWarp) {
            // -------------------------------------------------------------- tail --
            // A unit's last V tile (this CTA's d half): once it has landed, zero
            // its rows past the unit's last key, then tell the leader.  (Phases of
            // v_last / v_tail cannot alias: the producer loads unit n + 2 only
            // after unit n's epilogue, which follows its last PV.)
            int ord = 0, gb = 0, lvl = 0;  // units done, global index of the unit's first tile, schedule cursor
            bool ok = true;
            for (int rnd = 0; rnd * pairs < num_units && ok; ++rnd) {
                const int v = unit_of(rnd);
                if (v >= num_units) continue;
                Unit u;
                if (!unit_at<PAGED, BS, MODE>(a, smem, compact, npx, ny, v, lvl, u)) continue;
                const int t = u.T - 1;
                uint8_t *dv = smem + kRingOff + ((gb + t) % kStages) * kStageBytes + kKBytes;
                ok = __all_sync(0xffffffffu, mbar_wait(&v_last[ord & 1], (ord >> 1) & 1, a.err));
                if (ok) {
                    const int valid = u.kv_end_max - t * kBN;
                    for (int r = valid + (lane >> 3); r < kBN; r += 4)
                        *reinterpret_cast<uint4 *>(dv + r * 128 + (lane & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive_cluster(map_to_cta(smem_u32(&v_tail[ord & 1]), 0));
                gb += u.T;
                ++ord;
            }
            if (!ok && lane == 0) atomicExch(s_abort, 1);
        } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
            // --------------------------------------------------------- MMA issue --
            // Each issuing warp runs its loop warp-uniformly (descriptors in uniform
            // registers); one elected lane issues every MMA and commit.
            if (c == 0) {
                const int k = warp - kMmaWarp;
                constexpr uint32_t kIdescS = umma_idesc_bf16(2 * kBM, kBN, false, false);
                constexpr uint32_t kIdescO = umma_idesc_bf16(2 * kBM, kD, false, true);
                const uint64_t dk0 = umma_desc_sw128(smem_u32(smem + kRingOff), 16, 1024);
                const uint64_t dv0 = umma_desc_sw128(smem_u32(smem + kRingOff + kKBytes), kBox, 1024);
                const uint32_t tS = tmem + k * kBN, tO = tmem + 2 * kBN + k * kD;
                bool ok = true;
                int ord = 0, gb = 0, lvl = 0;  // units done, first tile of the unit, schedule cursor
                int pc = 0, uo = 0;        // P_k(t) phases seen, units of sub-tile k done
                int gbase[2] = {0, 0};     // groups issued by each thread before this unit
                int mine_q = 0;            // groups this thread has queued
                // Wait until the other thread has queued `target` groups (a
                // monotone count in shared memory).
                auto wait_count = [&](int target) {
                    if (!ok) return;
                    const long long t0 = clock64();
                    bool good = true;  // every lane spins until it sees the count (monotone)
                    for (uint32_t it = 1;; ++it) {
                        if (turn_cnt[1 - k] >= target) break;
                        if ((it & 1023u) == 0 && (clock64() - t0 > kWaitLimitCycles ||
                                                  *(volatile int *)a.err == PA_ERR_TIMEOUT)) {
                            good = false;
                            break;
                        }
                    }
                    good = __all_sync(0xffffffffu, good);
                    if (!good) {
                        if (lane == 0) set_error(a.err, PA_ERR_TIMEOUT);
                        ok = false;
                    }
                };
                for (int rnd = 0; rnd * pairs < num_units && ok; ++rnd) {
                const int v = unit_of(rnd);
                if (v >= num_units) continue;
                    Unit u;
                    if (!unit_at<PAGED, BS, MODE>(a, smem, compact, npx, ny, v, lvl, u)) continue;
                    const int qb = ord & 1;
                    const int nk = k ? u.nkt1 : u.nkt0, nk_other = k ? u.nkt0 : u.nkt1;
                    const int groups[2] = {u.nkt0 > 0 ? u.nkt0 + 1 : 0, u.nkt1 > 0 ? u.nkt1 + 1 : 0};
                    // The two threads take turns, group by group, in the order
                    //   S_0(0), S_1(0), [PV_0(0) S_0(1)], [PV_1(0) S_1(1)], ...
                    // so that the tensor core works for one sub-tile while the
                    // other's softmax runs.  Group j of a unit is S_k(0) for j = 0
                    // and [PV_k(j-1) S_k(j)] after; thread 1 waits for group j of
                    // thread 0, thread 0 for group j - 1 of thread 1 (for j = 0:
                    // for thread 1's previous unit).  Every wait comes before the
                    // turn is taken and every commit after the group's MMAs; the
                    // turn passes four MMAs before a group ends.
                    auto take_turn = [&](int j) {
                        wait_count(k == 1 ? gbase[0] + min(j + 1, groups[0]) : gbase[1] + min(j, groups[1]));
                    };
                    auto pass_turn = [&]() { turn_cnt[k] = ++mine_q; };
                    const uint64_t dq = umma_desc_sw128(smem_u32(smem + kQOff + (2 * qb + k) * kQBytes), 16, 1024);
                    auto wait_tile = [&](int t) {
                        const int gt = gb + t;
                        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_spin(&tile_full[gt % kStages], (gt / kStages) & 1, a.err));
                    };
                    // Every unit's Q is waited for, even by a thread with nothing to
                    // issue in it: its q_free commit below must not reach the
                    // buffer's barrier before the phase of unit ord - 2 is over.
                    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_spin(&q_full[qb], (ord >> 1) & 1, a.err));
                    auto issue_s = [&](int t) {  // S_k(t) = Q_k K(t)^T; the caller waited for tile t
                        const uint64_t bk = dk0 + (uint64_t)((((gb + t) % kStages) * kStageBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            umma_bf16_pair_w(tS, dq + (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                                             bk + (uint64_t)(((kk >> 2) * kKHalf + (kk & 3) * 32) >> 4), kIdescS, kk > 0);
                            if (kk == 3) pass_turn();
                        }
                    };
                    if (nk > 0) {
                        wait_tile(0);
                        take_turn(0);
                        if (ok) {
                            issue_s(0);
                            umma_commit_pair_w(&s_full[k]);
                        }
                    }
                    for (int t = 0; t < nk && ok; ++t) {
                        const bool more = t + 1 < nk;
                        if (more) wait_tile(t + 1);
                        take_turn(t + 1);  // usually passed before P_k(t) is ready
                        if (!ok || !(ok = __all_sync(0xffffffffu, mbar_wait_spin(&p_full[k], pc & 1, a.err)))) break;
                        ++pc;
                        if (t == u.T - 1 && !(ok = __all_sync(0xffffffffu, mbar_wait_spin(&v_tail[ord & 1], (ord >> 1) & 1, a.err)))) break;
                        // O_k is read out by the epilogue warps before this unit's first PV_k overwrites it.
                        if (t == 0 && uo > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait_spin(&o_free[k], (uo - 1) & 1, a.err)))) break;
                        tc_fence_after();
                        // O_k += P_k(t) V(t), P_k from TMEM (written by the softmax warps)
                        const uint64_t bv = dv0 + (uint64_t)((((gb + t) % kStages) * kStageBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            umma_bf16_pair_tmem_a_w(tO, tS + (kk >> 2) * 64 + (kk & 3) * 8, bv + (uint64_t)((kk * 2048) >> 4),
                                                    kIdescO, (t > 0 || kk > 0) ? 1u : 0u);
                            if (kk == 3 && !more) pass_turn();
                        }
                        if (more) issue_s(t + 1);  // overwrites P_k(t): after PV_k(t) in the tensor pipe
                        if (more) {
                            umma_commit_pair_w(&s_full[k]);
                        } else {
                            umma_commit_pair_w(&o_done[k]);
                            umma_commit_pair_w(&q_free[qb]);  // this thread's last S of the unit is done
                        }
                        umma_commit_pair_w(&tile_free[(gb + t) % kStages]);
                        if (t >= nk_other) umma_commit_pair_w(&tile_free[(gb + t) % kStages]);  // the only reader
                    }
                    if (!ok) break;
                    if (nk == 0) umma_commit_pair_w(&q_free[qb]);  // nothing of this thread reads Q buffer qb
                    else ++uo;
                    gbase[0] += groups[0];
                    gbase[1] += groups[1];
                    gb += u.T;
                    ++ord;
                }
                // Do not let the pair tear down TMEM under MMAs still in flight.
                umma_commit_pair_w(&mma_fin[k], 1);
                mbar_wait(&mma_fin[k], 0, a.err);
                if (!ok && lane == 0) atomicExch(s_abort, 1);
            }
            __syncwarp();
        }
    } else if (warp < kEpilogueWarp0) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        if (!skip) {
            // ----------------------------------------------------------- softmax --
            // All eight warps serve both sub-tiles, one tile at a time: warp w owns
            // rows 32q .. 32q+31 (q = w % 4, its TMEM lane quadrant and its SM
            // sub-partition) and key half hf of every tile -- S columns 64 hf ..
            // 64 hf + 63, one thread per row -- so each sub-partition runs two
            // warps on each tile's exponentials.  A thread's weights go to the
            // first 32 of its columns (it only overwrites scores it has read).  The
            // two warps of a quadrant share a row's running maximum and sum
            // through a named barrier of 64 threads and one word per row in shared
            // memory.
            const int hf = (warp - kSoftmaxWarp0) >> 2, q = warp & 3;
            const int r = 32 * q + lane;
            const uint32_t lane_base = (uint32_t)(32 * q) << 16;
            const uint32_t bar_id = 1 + q;
            float *xchg = reinterpret_cast<float *>(smem + kXchgOff) + r;
            const float sl = a.scale_log2;
            bool ok = true;
            int sc0 = 0, sc1 = 0;                  // S_k phases seen
            int lvl = 0, ord = 0;                // schedule cursor, units
            auto wait_warp = [&](uint64_t *bb, uint32_t par) {
                return __all_sync(0xffffffffu, mbar_wait(bb, par, a.err));
            };
            auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory"); };
            // true in both warps of the quadrant if p holds for any of their threads
            auto pair_any = [&](bool p) {
                uint32_t res;
                asm volatile(
                    "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
                    "bar.red.or.pred po, %2, 64, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
                    : "=r"(res)
                    : "r"((uint32_t)p), "r"(bar_id)
                    : "memory");
                return res != 0u;
            };
            // The row's maximum (or sum) over both halves, the same bits in both
            // threads: half 1 posts its value, half 0 combines and posts the
            // result, half 1 reads it.  (A word is written again only after its
            // reader has passed the next barrier.)
            auto pair_combine = [&](float x, bool is_max) {
                if (hf == 1) *xchg = x;
                pair_sync();
                if (hf == 0) {
                    const float y = *xchg;
                    x = is_max ? fmaxf(x, y) : x + y;
                    *xchg = x;
                }
                pair_sync();
                if (hf == 1) x = *xchg;
                return x;
            };
            // One arrival per warp on the leader's barrier, after the warp's
            // tcgen05 work is ordered before it.
            auto arrive_leader = [&](uint64_t *bb) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (c == 0) mbar_arrive(bb);
                    else mbar_arrive_cluster(map_to_cta(smem_u32(bb), 0));
                }
            };
            auto row_max64 = [&](const float *x) {
                float m4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) m4[i] = fmax3(x[i], x[i + 4], x[i + 8]);
#pragma unroll
                for (int j = 12; j < 64; j += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) m4[i] = fmax3(m4[i], x[j + i], j + 4 + i < 64 ? x[j + 4 + i] : -INFINITY);
                return fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
            };
            auto mask64 = [&](float *x, int lim) {
#pragma unroll
                for (int j = 0; j < 64; ++j) x[j] = j < lim ? x[j] : -INFINITY;
            };
            // P = exp2(scale * S - mu) for this half's 64 keys as 32 bf16 pairs at
            // TMEM columns pcol .. pcol + 31 (column j: keys 2j, 2j+1 of the half);
            // returns the row sum of the same rounded weights.  The TMEM stores
            // are left in flight.
            auto exps64_to_tmem = [&](const float *x, float mu, uint32_t pcol) {
                float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int cq = 0; cq < 2; ++cq) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        pk[j] = pack_bf16x2(fast_exp2(fmaf(x[32 * cq + 2 * j], sl, -mu)),
                                            fast_exp2(fmaf(x[32 * cq + 2 * j + 1], sl, -mu)));
                        ls2[j & 1] = add_f32x2(ls2[j & 1], bf16x2_unpack(pk[j]));
                    }
                    tmem_st16_async(pcol + 16 * cq, pk);
                }
                return (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
            };
            auto rescale_o = [&](uint32_t tO, float alpha) {  // this half's 64 columns of O_k
#pragma unroll 1
                for (int cc = 0; cc < 2; ++cc) {
                    float o[32];
                    tmem_ld32(tO + cc * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tO + cc * 32, o);
                }
            };
            for (int rnd = 0; rnd * pairs < num_units && ok; ++rnd) {
                const int v = unit_of(rnd);
                if (v >= num_units) continue;
                Unit u;
                if (!unit_at<PAGED, BS, MODE>(a, smem, compact, npx, ny, v, lvl, u)) continue;
                const int qb = ord & 1;
                ++ord;
                // Per-sub-tile state in scalars: the sub-tile loops below are not
                // unrolled (one copy of the tile body keeps the warps' code small
                // enough to stay in the instruction cache).
                const RowTile my0 = my_tile<MODE>(u, c, 0), my1 = my_tile<MODE>(u, c, 1);
                // keys of this half visible to row r, per sub-tile
                const int lim0 = min(u.p0 + my0.q0 + r + 1, my0.kv_end) - 64 * hf;
                const int lim1 = min(u.p0 + my1.q0 + r + 1, my1.kv_end) - 64 * hf;
                float m0 = 0.f, m1 = 0.f, l0 = 0.f, l1 = 0.f;  // l: this half's share of the row sum
                for (int t = 0; t < u.T && ok; ++t) {
#pragma unroll 1
                    for (int k = 0; k < 2; ++k) {
                        if (t >= (k ? u.nkt1 : u.nkt0)) continue;
                        const uint32_t tS = tmem + lane_base + k * kBN + 64 * hf;
                        const uint32_t tO = tmem + lane_base + 2 * kBN + k * kD + 64 * hf;
                        // S_k(t) completing also means PV_k(t-1) has: O_k is stable
                        // and P_k(t-1) is no longer needed.  Both warps of the
                        // quadrant take every barrier below whatever their waits
                        // returned; a failed wait is acted on together.
                        const bool got = wait_warp(&s_full[k], (k ? sc1 : sc0) & 1);
                        if (k) ++sc1; else ++sc0;
                        tc_fence_after();
                        const int lim = (k ? lim1 : lim0) - t * kBN;  // visible columns of this half
                        // (Read even after a failed wait -- the values are then
                        // unused.)  Warp-uniform branch: only tiles crossing some
                        // row's last key pay for the mask.
                        float v[64];
                        tmem_ld64(tS, v);
                        if (__any_sync(0xffffffffu, lim < 64)) mask64(v, lim);
                        // Key 0 is visible to every row, so the first tile's maximum
                        // is finite; later tiles keep the running maximum unless a
                        // weight would pass 2^63 (or is not finite): then the maximum
                        // moves, O_k (stable) and the sum are rescaled and the
                        // weights are computed again (second pass of the loop).
                        float mr = k ? m1 : m0, lr = k ? l1 : l0, lh = 0.f;
                        bool redo = false;
                        for (;;) {
                            if (t == 0 || redo) {
                                const float mx = pair_combine(got ? row_max64(v) : -INFINITY, true) * sl;
                                if (redo) {
                                    const float m_new = fmaxf(mr, mx);
                                    const float alpha = fast_exp2(mr - m_new);
                                    mr = m_new;
                                    tmem_wait_st();
                                    rescale_o(tO, alpha);
                                    lr *= alpha;
                                } else {
                                    mr = mx;
                                }
                            }
                            lh = got ? exps64_to_tmem(v, mr, tS) : 0.f;
                            if (redo || !pair_any(!got || (t > 0 && !(lh <= 0x1p63f)))) break;
                            if (pair_any(!got)) {
                                ok = false;
                                break;
                            }
                            redo = true;
                        }
                        if (!ok) break;
                        lr = (t == 0) ? lh : lr + lh;
                        if (k) { m1 = mr; l1 = lr; } else { m0 = mr; l0 = lr; }
                        tmem_wait_st();
                        arrive_leader(&p_full[k]);
                        if (t == (k ? u.nkt1 : u.nkt0) - 1) {
                            // The sub-tile's last tile: post the rows' sums for the
                            // epilogue warps, in the first 128 bytes of this
                            // quadrant's part of the unit's Q buffer (S_k(t), its
                            // last reader, has completed).
                            const float l_row = pair_combine(lr, false);
                            if (hf == 0) {
                                reinterpret_cast<float *>(smem + kQOff + (2 * qb + k) * kQBytes + q * 8192)[lane] = l_row;
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&l_ready[2 * qb + k]);
                            }
                        }
                    }
                }
            }
            if (!ok) atomicExch(s_abort, 1);
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
        if (!skip) {
            // ---------------------------------------------------------- epilogue --
            // Warp w (quadrant q = w % 4, rows 32q .. 32q+31 of each sub-tile, all
            // 128 columns): once a unit's last PV_k has completed, read O_k out,
            // release it, normalise by the posted row sums and store -- staged in
            // the unit's Q buffer and written by TMA where all 32 rows belong to
            // the sequence, by plain stores otherwise.  Then release the Q buffer
            // once the stores have read it.
            const int q = warp & 3;
            const int r = 32 * q + lane;
            const uint32_t lane_base = (uint32_t)(32 * q) << 16;
            bool ok = true;
            int uo0 = 0, uo1 = 0, lvl = 0, ord = 0;  // units of sub-tile k done, schedule cursor, units
            uint32_t lph = 0;  // bit 2 b + k: phase of l_ready[2 b + k] (it completes only for units where k has rows)
            for (int rnd = 0; rnd * pairs < num_units && ok; ++rnd) {
                const int v = unit_of(rnd);
                if (v >= num_units) continue;
                Unit u;
                if (!unit_at<PAGED, BS, MODE>(a, smem, compact, npx, ny, v, lvl, u)) continue;
                const int qb = ord & 1;
                ++ord;
#pragma unroll 1
                for (int k = 0; k < 2; ++k) {
                    if ((k ? u.nkt1 : u.nkt0) == 0) continue;
                    const RowTile mk = my_tile<MODE>(u, c, k);
                    const uint32_t tO = tmem + lane_base + 2 * kBN + k * kD;
                    uint8_t *qbuf = smem + kQOff + (2 * qb + k) * kQBytes + q * 8192;
                    const bool od = __all_sync(0xffffffffu, mbar_wait(&o_done[k], (k ? uo1 : uo0) & 1, a.err));
                    if (k) ++uo1; else ++uo0;
                    const bool lok =
                        od && __all_sync(0xffffffffu, mbar_wait(&l_ready[2 * qb + k], (lph >> (2 * qb + k)) & 1u, a.err));
                    lph ^= 1u << (2 * qb + k);
                    if (!lok) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float l_row = reinterpret_cast<const float *>(qbuf)[lane];
                    __syncwarp();  // the posted sums are read before the staging overwrites them
                    const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
                    const bool staged = 32 * q + 32 <= mk.rows;
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {
                        float o[64];
                        tmem_ld64(tO + 64 * hf, o);
                        if (hf == 1) {  // all of this quadrant's O_k is read: release it
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if (c == 0) mbar_arrive(&o_free[k]);
                                else mbar_arrive_cluster(map_to_cta(smem_u32(&o_free[k]), 0));
                            }
                        }
                        // The row's eight 16-byte pieces: into the staging box (one
                        // 64-column box of 32 swizzled 128-byte rows) or, in a
                        // partial warp, straight to the row in memory.
                        uint8_t *dst = staged ? qbuf + hf * 4096 + lane * 128
                                              : reinterpret_cast<uint8_t *>(
                                                    a.out + ((size_t)(u.row0 + mk.q0 + r) * a.num_q_heads + mk.h) * kD + 64 * hf);
                        if (staged || r < mk.rows) {
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) {
                                const uint4 pk = make_uint4(pack_bf16x2(o[8 * jj] * inv, o[8 * jj + 1] * inv),
                                                            pack_bf16x2(o[8 * jj + 2] * inv, o[8 * jj + 3] * inv),
                                                            pack_bf16x2(o[8 * jj + 4] * inv, o[8 * jj + 5] * inv),
                                                            pack_bf16x2(o[8 * jj + 6] * inv, o[8 * jj + 7] * inv));
                                *reinterpret_cast<uint4 *>(dst + ((staged ? (jj ^ (lane & 7)) : jj) << 4)) = pk;
                            }
                        }
                    }
                    if (staged) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tm_o, qbuf, 0, mk.h, u.row0 + mk.q0 + 32 * q);
                            tma_store_3d(&tm_o, qbuf + 4096, 64, mk.h, u.row0 + mk.q0 + 32 * q);
                            bulk_commit_group();
                        }
                    }
                }
                if (!ok) break;
                // The unit's Q buffer is free once the stores have read the staging.
                if (lane == 0) {
                    bulk_wait_read_all();
                    mbar_arrive(&q_free[qb]);
                }
            }
            if (lane == 0) bulk_wait_all();  // the output stores are done before the CTA exits
            if (!ok) atomicExch(s_abort, 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the pair's MMAs may still touch it
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

template <int BS, bool PAGED, int MODE>
cudaError_t launch_pair_t(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          const CUtensorMap &tm_o, const PrefillArgs &a, cudaStream_t stream) {
    static std::atomic<unsigned long long> opted{0};
    const void *kfn = reinterpret_cast<const void *>(prefill_pair_kernel<BS, PAGED, MODE>);
    cudaError_t e0 = opt_in_smem(kfn, kSmemBytes, opted);
    if (e0 != cudaSuccess) return e0;
    // The warpgroups' register shares assume the launch gives each thread
    // exactly 65536 / kThreads registers: with fewer, an increase could never
    // be granted.  Refuse to launch a build where that does not hold.
    static std::atomic<int> regs_checked{0};  // 0 unknown, 1 as assumed, -1 not
    if (regs_checked.load(std::memory_order_acquire) == 0) {
        cudaFuncAttributes fa;
        e0 = cudaFuncGetAttributes(&fa, kfn);
        if (e0 != cudaSuccess) return e0;
        regs_checked.store(fa.numRegs == 65536 / kThreads && fa.maxThreadsPerBlock >= kThreads ? 1 : -1,
                           std::memory_order_release);
    }
    if (regs_checked.load(std::memory_order_acquire) != 1) return cudaErrorInvalidConfiguration;
    const long long units = (long long)((a.num_q_tiles + per_pair(MODE) - 1) / per_pair(MODE)) *
                            (a.num_q_heads / heads_per_pair(MODE)) * a.num_seqs;
    if (units == 0) return cudaSuccess;
    const int pairs = (int)std::min<long long>(units, std::max(1, a.num_sms / 2));
    cudaLaunchAttribute pdl[1];  // a programmatic dependent launch (the kernel waits before reading)
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<BS, PAGED, MODE>, tm_q, tm_k, tm_v, tm_o, a);
}

template <int BS, bool PAGED>
cudaError_t launch_pair_m(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          const CUtensorMap &tm_o, const PrefillArgs &a, cudaStream_t stream) {
    if (a.group % 4 == 0) return launch_pair_t<BS, PAGED, 0>(tm_q, tm_k, tm_v, tm_o, a, stream);
    if (a.group % 2 == 0) return launch_pair_t<BS, PAGED, 1>(tm_q, tm_k, tm_v, tm_o, a, stream);
    return launch_pair_t<BS, PAGED, 2>(tm_q, tm_k, tm_v, tm_o, a, stream);
}

}  // namespace

cudaError_t launch_prefill_pair(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                const CUtensorMap &tm_o, const PrefillArgs &a, int block_size, cudaStream_t stream) {
    if (a.block_table == nullptr) return launch_pair_m<16, false>(tm_q, tm_k, tm_v, tm_o, a, stream);
    if (block_size == 16) return launch_pair_m<16, true>(tm_q, tm_k, tm_v, tm_o, a, stream);
    if (block_size == 32) return launch_pair_m<32, true>(tm_q, tm_k, tm_v, tm_o, a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
