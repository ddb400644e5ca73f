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
// Work unit: a CTA pair owns four 128-row query tiles that read the same KV
// head -- four query heads of one group (group size a multiple of 4), two
// heads x two row tiles (even group size), or four consecutive row tiles of
// one head.  CTA c holds two of them as sub-tiles k = 0, 1; the pair's
// sub-tile k is one M = 256 MMA operand (CTA 0's rows, then CTA 1's).
//   K tile (128 keys): CTA c loads keys 64c .. 64c+63 (the MMA's B is split
//     along N between the pair), both 64-column halves of d.
//   V tile (128 keys): CTA c loads all keys, d columns 64c .. 64c+63.
//   S_k = Q_k K^T (M=256, N=128, K=128) -> each CTA's TMEM S_k (128 columns).
//   Softmax (thread = row = TMEM lane) writes P_k (bf16 pairs) over the first
//     64 columns of S_k, then arrives on the leader.
//   O_k += P_k V (A from TMEM, M=256, N=128: the two d halves, K=128 keys).
//   The leader issues, per KV tile, PV_0(t), S_0(t+1), PV_1(t), S_1(t+1): while
//   the tensor core works for one sub-tile the other's softmax runs.  S_k(t+1)
//   overwrites P_k(t) and so waits for PV_k(t) (in-order tensor pipe).
// Warps: 0 and 1 issue (leader CTA only) the MMAs of sub-tiles 0 and 1 -- a
// thread stalls for hundreds of cycles on each mbarrier test, and the other
// thread's queued MMAs keep the tensor core busy meanwhile; warp 0 also
// allocates TMEM (both CTAs); 2 TMA producer; 3-6 and 7-10 softmax for
// sub-tiles 0 and 1 (warp w: rows 32 (w % 4) .. +31, TMEM lane quadrant
// w % 4, all 128 columns).
// Loads signal the leader's barriers (cp.async.bulk.tensor .cta_group::2);
// the leader's commits signal both CTAs (multicast).  The last V tile is
// loaded against a local barrier in each CTA so its rows past the last key can
// be zeroed (stale pool rows could hold NaN, and 0 * NaN = NaN) before the
// leader is told it is ready.
#include <cuda.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kD = 128;
constexpr int kBM = 128;                       // rows per query sub-tile (per CTA)
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kMmaWarp = 0;       // and kMmaWarp + 1
constexpr int kProducerWarp = 2;
constexpr int kSoftmaxWarp0 = 3;
constexpr int kThreads = 352;
constexpr uint32_t kTmemCols = 512;            // S_0, S_1, O_0, O_1
constexpr int kBox = 128 * 128;                // one [128 rows][64 bf16] swizzled box set
constexpr int kQBytes = 2 * kBox;              // Q_k: [128][128]
constexpr int kKHalf = 64 * 128;               // [64 keys][64 d]
constexpr int kKBytes = 2 * kKHalf;            // K: 64 keys x 128 d (per CTA)
constexpr int kVBytes = 128 * 128;             // V: 128 keys x 64 d (per CTA)
constexpr int kStageBytes = kKBytes + kVBytes; // one KV tile: K then V
constexpr int kQOff = 0;
constexpr int kRingOff = 2 * kQBytes;
constexpr int kStages = 5;                     // K/V ring: five tiles
constexpr int kBarOff = kRingOff + kStages * kStageBytes;
constexpr int kNumBars = 1 + 2 * kStages + 2 * 3 + 4 + 2;
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;

struct RowTile {
    int h, q0, rows, kv_end;
};

// MODE 0: four heads x one row tile; 1: two heads x two row tiles;
// 2: one head x four row tiles.
template <int MODE>
__device__ __forceinline__ void row_tile(RowTile &rt, int c, int k, int px, int n, int p0) {
    if (MODE == 0) {
        rt.h = 4 * blockIdx.y + 2 * c + k;
        rt.q0 = px * kBM;
    } else if (MODE == 1) {
        rt.h = 2 * blockIdx.y + c;
        rt.q0 = (2 * px + k) * kBM;
    } else {
        rt.h = blockIdx.y;
        rt.q0 = (4 * px + 2 * k + c) * kBM;
    }
    rt.rows = max(0, min(kBM, n - rt.q0));
    rt.kv_end = p0 + min(n, rt.q0 + kBM);
}

template <int BS, bool PAGED, int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *q_full = bar;
    uint64_t *tile_full = bar + 1;          // [kStages] leader: K and V of a tile landed in both CTAs
    uint64_t *tile_free = tile_full + kStages;  // [kStages] both sub-tiles' MMAs on the tile have completed
    uint64_t *s_full = tile_free + kStages; // [2] S_k(t) is in TMEM (commit, both CTAs)
    uint64_t *p_full = s_full + 2;          // [2] leader: P_k(t) stored by the 8 softmax warps of the pair
    uint64_t *o_done = p_full + 2;          // [2] the last PV_k has completed (commit, both CTAs)
    uint64_t *v_last = o_done + 2;         // local: this CTA's half of the last V tile landed
    uint64_t *v_tail = v_last + 1;          // leader: both halves zeroed past the last key
    uint64_t *mma_fin = v_tail + 1;         // [2] leader: every MMA issued by thread k has completed
    uint64_t *turn = mma_fin + 2;           // [2] leader: issuing thread k has queued its j-th group
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar + kNumBars);
    int *s_abort = reinterpret_cast<int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = (int)cluster_ctarank();
    const int px = (int)(gridDim.x >> 1) - 1 - (int)(blockIdx.x >> 1);  // longest causal rows first
    const int s = blockIdx.z;

    // ---- geometry (identical in both CTAs, so every early exit is pair-wide)
    const int row0 = a.cu_seqlens[s];
    const int n = a.cu_seqlens[s + 1] - row0;
    const int p0 = a.prefix_lens ? a.prefix_lens[s] : (a.seq_lens ? a.seq_lens[s] - n : 0);
    const bool bad = n < 0 || p0 < 0 || row0 < 0 || (long long)row0 + n > a.num_tokens ||
                     n > a.max_q_len || (PAGED && (p0 + n + BS - 1) / BS > a.max_blocks) ||
                     (!PAGED && p0 != 0);
    if (bad) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_error(a.err, PA_ERR_BAD_INDEX);
        return;
    }
    RowTile rt[2][2];  // [cta][sub-tile]
#pragma unroll
    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int k = 0; k < 2; ++k) row_tile<MODE>(rt[cc][k], cc, k, px, n, p0);
    int nkt[2], kv_end_max = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        int e = 0;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
            if (rt[cc][k].rows > 0) e = max(e, rt[cc][k].kv_end);
        nkt[k] = (e + kBN - 1) / kBN;
        kv_end_max = max(kv_end_max, e);
    }
    const int T = max(nkt[0], nkt[1]);
    if (T == 0) return;
    const int g = rt[0][0].h / a.group;
    RowTile mine[2];  // this CTA's two sub-tiles (no runtime indexing of rt)
#pragma unroll
    for (int k = 0; k < 2; ++k) row_tile<MODE>(mine[k], c, k, px, n, p0);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&tile_full[i], 1);
            mbar_init(&tile_free[i], 2);  // one commit per issuing thread (two if one sub-tile reads the tile)
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], 2 * 4);  // one arrival per softmax warp of each CTA
            mbar_init(&o_done[k], 1);
        }
        mbar_init(v_last, 1);
        mbar_init(v_tail, 2);
        mbar_init(&mma_fin[0], 1);
        mbar_init(&mma_fin[1], 1);
        mbar_init(&turn[0], 1);
        mbar_init(&turn[1], 1);
        // Validation mode: the leader's reading of the error word decides for
        // both CTAs (it may change while the kernel runs).
        *s_abort = (a.check_err_first && *(volatile int *)a.err != 0) ? 1 : 0;
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

    if (skip) {
        // nothing to do: fall through to the pair-wide teardown
    } else if (warp == kProducerWarp) {
        // ---------------------------------------------------------- producer --
        constexpr int kBPT = kBN / BS;  // pool blocks per 128-key tile
        const int nb_used = (kv_end_max + BS - 1) / BS;
        const int oob_row = a.num_blocks * a.num_kv_heads * BS;  // past the pool: TMA fills zeros
        const int32_t *bt = PAGED ? a.block_table + (size_t)s * a.max_blocks : nullptr;
        const uint32_t lq = map_to_cta(smem_u32(q_full), 0);
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (c == 0) mbar_arrive_expect_tx(q_full, 2 * 2 * kQBytes);
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_3d_pair(smem + kQOff + k * kQBytes + hf * kBox, &tm_q, lq, hf * 64, mine[k].h,
                                     row0 + mine[k].q0);
        }
        // Pool rows of the tiles' blocks: lane l holds block 32 j + l of lane
        // group j (kTPG tiles); the next group's entries are loaded while the
        // current group is issued.  Each TMA copy of a tile is issued by its
        // own lane.
        constexpr int kTPG = 32 / kBPT;
        auto block_row = [&](int bi) {
            int row = oob_row;
            if (bi < nb_used) {
                int blk = bt[bi];
                if ((unsigned)blk >= (unsigned)a.num_blocks) {
                    set_error(a.err, PA_ERR_BAD_INDEX);
                    blk = 0;  // never dereference an out-of-range block
                }
                row = (blk * a.num_kv_heads + g) * BS;
            }
            return row;
        };
        int row_cur = 0, row_nxt = 0;
        if (PAGED) {
            row_cur = block_row(lane);
            row_nxt = block_row(32 + lane);
        }
        for (int t = 0; t < T; ++t) {
            if (PAGED && t > 0 && t % kTPG == 0) {
                row_cur = row_nxt;
                row_nxt = block_row((t / kTPG + 1) * 32 + lane);
            }
            const int base = (t % kTPG) * kBPT;
            const int st = t % kStages;
            uint8_t *dk = smem + kRingOff + st * kStageBytes;
            uint8_t *dv = dk + kKBytes;
            bool ok = true;
            if (lane == 0 && t >= kStages) ok = mbar_wait(&tile_free[st], ((t / kStages) - 1) & 1, a.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok || *(volatile int *)s_abort) {
                if (lane == 0) atomicExch(s_abort, 1);
                break;
            }
            const bool last = (t == T - 1);
            const uint32_t lb = map_to_cta(smem_u32(&tile_full[st]), 0);
            if (lane == 0 && c == 0) mbar_arrive_expect_tx(&tile_full[st], last ? 2 * kKBytes : 2 * kStageBytes);
            // K: this CTA's 64 keys, both halves of d (lane = 2 block + half)
            const int jb = (lane >> 1) & (64 / BS - 1), hf = lane & 1;
            const int krow = PAGED ? __shfl_sync(0xffffffffu, row_cur, base + c * (64 / BS) + jb) : 0;
            if (PAGED) {
                if (lane < 2 * (64 / BS)) tma_load_2d_pair(dk + hf * kKHalf + jb * BS * 128, &tm_k, lb, hf * 64, krow);
            } else if (lane < 2) {
                tma_load_3d_pair(dk + hf * kKHalf, &tm_k, lb, hf * 64, g, row0 + t * kBN + 64 * c);
            }
            // V: all 128 keys, this CTA's half of d (lane = block)
            const int vrow = PAGED ? __shfl_sync(0xffffffffu, row_cur, base + (lane & (kBPT - 1))) : 0;
            if (!last) {
                if (PAGED) {
                    if (lane < kBPT) tma_load_2d_pair(dv + lane * BS * 128, &tm_v, lb, c * 64, vrow);
                } else if (lane == 0) {
                    tma_load_3d_pair(dv, &tm_v, lb, c * 64, g, row0 + t * kBN);
                }
            } else {
                // The last V tile: land it against a local barrier, zero its
                // rows past the last key, then tell the leader.
                if (lane == 0) mbar_arrive_expect_tx(v_last, kVBytes);
                __syncwarp();
                if (PAGED) {
                    if (lane < kBPT) tma_load_2d(dv + lane * BS * 128, &tm_v, v_last, c * 64, vrow);
                } else if (lane == 0) {
                    tma_load_3d(dv, &tm_v, v_last, c * 64, g, row0 + t * kBN);
                }
                const bool vok = __all_sync(0xffffffffu, mbar_wait(v_last, 0, a.err));
                if (vok) {
                    const int valid = kv_end_max - t * kBN;
                    for (int r = valid + (lane >> 3); r < kBN; r += 4)
                        *reinterpret_cast<uint4 *>(dv + r * 128 + (lane & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    if (vok) mbar_arrive_cluster(map_to_cta(smem_u32(v_tail), 0));
                    else atomicExch(s_abort, 1);
                }
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // --------------------------------------------------------- MMA issue --
        if (c == 0 && lane == 0) {
            const int k = warp - kMmaWarp;
            const int nk = k == 0 ? nkt[0] : nkt[1];
            const int nk_other = k == 0 ? nkt[1] : nkt[0];
            constexpr uint32_t kIdescS = umma_idesc_bf16(2 * kBM, kBN, false, false);
            constexpr uint32_t kIdescO = umma_idesc_bf16(2 * kBM, kD, false, true);
            const uint64_t dq = umma_desc_sw128(smem_u32(smem + kQOff + k * kQBytes), 16, 1024);
            const uint64_t dk0 = umma_desc_sw128(smem_u32(smem + kRingOff), 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(smem_u32(smem + kRingOff), kBox, 1024);
            const uint32_t tS = tmem + k * kBN, tO = tmem + 2 * kBN + k * kD;
            bool ok = nk == 0 || mbar_wait_spin(q_full, 0, a.err);
            // S_k(t) = Q_k K(t)^T; the caller has waited for tile t.  The turn
            // passes to the other thread four MMAs before the end, so that its
            // wait overlaps MMAs still queued here.
            auto issue_s = [&](int t) {
                const uint64_t bk = dk0 + (uint64_t)(((t % kStages) * kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    umma_bf16_pair(tS, dq + (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                                   bk + (uint64_t)(((kk >> 2) * kKHalf + (kk & 3) * 32) >> 4), kIdescS, kk > 0);
                    if (kk == 3) mbar_arrive(&turn[k]);
                }
            };
            auto wait_tile = [&](int t) {
                if (ok) ok = mbar_wait_spin(&tile_full[t % kStages], (t / kStages) & 1, a.err);
            };
            // The two threads take turns, group by group, in the order
            //   S_0(0), S_1(0), [PV_0(0) S_0(1)], [PV_1(0) S_1(1)], [PV_0(1) S_0(2)], ...
            // so that the tensor core works for one sub-tile while the other's
            // softmax runs.  Group j of thread k is S_k(0) for j = 0 and
            // [PV_k(j-1) S_k(j)] after; thread 1 waits for group j of thread
            // 0, thread 0 for group j - 1 of thread 1 (each thread waits
            // only while the other has MMAs queued).  Every wait comes before
            // the turn is taken and every commit after the group's MMAs, so
            // that a group goes out back to back.
            auto other_group_exists = [&](int j) { return j == 0 ? nk_other > 0 : j - 1 < nk_other; };
            auto take_turn = [&](int j) {  // before this thread's group j
                const int jo = k == 0 ? j - 1 : j;
                if (ok && jo >= 0 && other_group_exists(jo))
                    ok = mbar_wait_spin(&turn[1 - k], jo & 1, a.err);
            };
            if (nk > 0) {
                wait_tile(0);
                take_turn(0);
                if (ok) {
                    issue_s(0);
                    umma_commit_pair(&s_full[k]);
                }
            }
            for (int t = 0; t < nk && ok; ++t) {
                // O_k += P_k(t) V(t), P_k from TMEM (written by the softmax warps)
                const bool more = t + 1 < nk;
                if (more) wait_tile(t + 1);
                take_turn(t + 1);  // usually passed before P_k(t) is ready
                if (!ok || !(ok = mbar_wait_spin(&p_full[k], t & 1, a.err))) break;
                if (t == T - 1 && !(ok = mbar_wait_spin(v_tail, 0, a.err))) break;
                tc_fence_after();
                const uint64_t bv = dv0 + (uint64_t)(((t % kStages) * kStageBytes + kKBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    umma_bf16_pair_tmem_a(tO, tS + kk * 8, bv + (uint64_t)((kk * 2048) >> 4), kIdescO,
                                          (t > 0 || kk > 0) ? 1u : 0u);
                    if (kk == 3 && !more) mbar_arrive(&turn[k]);
                }
                if (more) issue_s(t + 1);  // overwrites P_k(t): after PV_k(t) in the tensor pipe
                if (more) umma_commit_pair(&s_full[k]);
                else umma_commit_pair(&o_done[k]);
                umma_commit_pair(&tile_free[t % kStages]);
                if (t >= nk_other) umma_commit_pair(&tile_free[t % kStages]);  // the only reader of tile t
            }
            // Do not let the pair tear down TMEM under MMAs still in flight.
            umma_commit_pair(&mma_fin[k], 1);
            mbar_wait(&mma_fin[k], 0, a.err);
            if (!ok) atomicExch(s_abort, 1);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- softmax --
        // Warps 2+4k .. 5+4k do sub-tile k; warp w owns rows 32q .. 32q+31 (TMEM
        // lane quadrant q), one row per thread, all 128 columns.
        const int k = (warp - kSoftmaxWarp0) >> 2, q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t tS = tmem + lane_base + k * kBN;
        const uint32_t tO = tmem + lane_base + 2 * kBN + k * kD;
        const RowTile my = k == 0 ? mine[0] : mine[1];
        const int nk = k == 0 ? nkt[0] : nkt[1];
        const uint32_t pf = map_to_cta(smem_u32(&p_full[k]), 0);
        const int lim_abs = min(p0 + my.q0 + r + 1, my.kv_end);
        const float sl = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        auto wait_warp = [&](uint64_t *bb, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bb, par, a.err));
        };
        // One arrival per warp on the leader's barrier, after the warp's
        // tcgen05 work is ordered before it.
        auto arrive_leader = [&](uint64_t *bb, uint32_t remote) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (c == 0) mbar_arrive(bb);
                else mbar_arrive_cluster(remote);
            }
        };
        auto row_max = [&](const float *x) {
            float m4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) m4[i] = fmax3(x[i], x[i + 4], x[i + 8]);
#pragma unroll
            for (int j = 12; j < kBN; j += 8)
#pragma unroll
                for (int i = 0; i < 4; ++i) m4[i] = fmax3(m4[i], x[j + i], j + 4 + i < kBN ? x[j + 4 + i] : -INFINITY);
            return fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
        };
        // P_k(t) = exp2(scale * S - mu) as bf16 pairs over the first 64 columns
        // of S_k (column j: keys 2j, 2j+1); returns the row sum of the same
        // rounded weights.  The TMEM stores are left in flight.
        auto exps_to_tmem = [&](const float *x, float mu) {
            float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int cq = 0; cq < kBN / 32; ++cq) {
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    pk[j] = pack_bf16x2(fast_exp2(fmaf(x[32 * cq + 2 * j], sl, -mu)),
                                        fast_exp2(fmaf(x[32 * cq + 2 * j + 1], sl, -mu)));
                    ls2[j & 1] = add_f32x2(ls2[j & 1], bf16x2_unpack(pk[j]));
                }
                tmem_st16_async(tS + 16 * cq, pk);
            }
            return (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
        };
        for (int t = 0; t < nk; ++t) {
            // S_k(t) completing also means PV_k(t-1) has: O_k is stable and
            // P_k(t-1) is no longer needed.
            if (!wait_warp(&s_full[k], t & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[kBN];
            tmem_ld128(tS, v);
            const int lim = lim_abs - t * kBN;  // visible columns of this row
            // Warp-uniform branch: only tiles crossing some row's last key pay
            // for the mask.
            if (__any_sync(0xffffffffu, lim < kBN)) {
#pragma unroll
                for (int j = 0; j < kBN; ++j) v[j] = j < lim ? v[j] : -INFINITY;
            }
            if (t == 0) {
                // key 0 is visible to every row, so the maximum is finite
                m_run = row_max(v) * sl;
                l_run = exps_to_tmem(v, m_run);
            } else {
                // Exponentials against the running maximum; the row sum shows
                // when the maximum has grown too far (weights above 2^64 or
                // not finite): then move it, rescale O_k (stable: PV_k(t-1)
                // has completed) and redo the tile.
                float l_tile = exps_to_tmem(v, m_run);
                if (__any_sync(0xffffffffu, !(l_tile <= 0x1p64f))) {
                    const float m_new = fmaxf(m_run, row_max(v) * sl);
                    const float alpha = fast_exp2(m_run - m_new);
                    m_run = m_new;
#pragma unroll
                    for (int cc = 0; cc < kD / 32; ++cc) {
                        float o[32];
                        tmem_ld32(tO + cc * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(tO + cc * 32, o);
                    }
                    l_run *= alpha;
                    l_tile = exps_to_tmem(v, m_run);
                }
                l_run += l_tile;
            }
            tmem_wait_st();
            arrive_leader(&p_full[k], pf);
        }
        // --------------------------------------------------------- epilogue --
        if (nk > 0) {
            const bool aborted = !ok || __any_sync(0xffffffffu, *(volatile int *)s_abort != 0);
            if (!aborted && wait_warp(&o_done[k], 0)) {
                tc_fence_after();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                float o[kD];
                tmem_ld128(tO, o);
                if (r < my.rows) {
                    __nv_bfloat16 *orow = a.out + ((size_t)(row0 + my.q0 + r) * a.num_q_heads + my.h) * kD;
#pragma unroll
                    for (int i = 0; i < kD; i += 8) {
                        const uint4 pk = make_uint4(pack_bf16x2(o[i] * inv, o[i + 1] * inv),
                                                    pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv),
                                                    pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv),
                                                    pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv));
                        *reinterpret_cast<uint4 *>(orow + i) = pk;
                    }
                }
            } else {
                atomicExch(s_abort, 1);
            }
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
                          const PrefillArgs &a, cudaStream_t stream) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel<BS, PAGED, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int per_pair = MODE == 0 ? 1 : (MODE == 1 ? 2 : 4);  // row tiles of one head per pair
    const int heads_per_pair = MODE == 0 ? 4 : (MODE == 1 ? 2 : 1);
    dim3 grid(2 * ((a.num_q_tiles + per_pair - 1) / per_pair), a.num_q_heads / heads_per_pair, a.num_seqs);
    prefill_pair_kernel<BS, PAGED, MODE><<<grid, kThreads, kSmemBytes, stream>>>(tm_q, tm_k, tm_v, a);
    return cudaGetLastError();
}

template <int BS, bool PAGED>
cudaError_t launch_pair_m(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          const PrefillArgs &a, cudaStream_t stream) {
    if (a.group % 4 == 0) return launch_pair_t<BS, PAGED, 0>(tm_q, tm_k, tm_v, a, stream);
    if (a.group % 2 == 0) return launch_pair_t<BS, PAGED, 1>(tm_q, tm_k, tm_v, a, stream);
    return launch_pair_t<BS, PAGED, 2>(tm_q, tm_k, tm_v, a, stream);
}

}  // namespace

cudaError_t launch_prefill_pair(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                const PrefillArgs &a, int block_size, cudaStream_t stream) {
    if (a.block_table == nullptr) return launch_pair_m<16, false>(tm_q, tm_k, tm_v, a, stream);
    if (block_size == 16) return launch_pair_m<16, true>(tm_q, tm_k, tm_v, a, stream);
    if (block_size == 32) return launch_pair_m<32, true>(tm_q, tm_k, tm_v, a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
