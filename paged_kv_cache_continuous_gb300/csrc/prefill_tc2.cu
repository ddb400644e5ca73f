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
// Why pairs: on one SM a 128x128x16 tcgen05.mma with both operands in shared
// memory costs ~133 SM cycles however small N is, ~46 % of the per-clock dense
// peak; the same instruction issued for a CTA pair (M = 256, cta_group::2)
// costs ~73 cycles and does twice the work, ~84 % of peak per SM.
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
//   Softmax (thread = row = TMEM lane) writes P_k (bf16) to shared memory in
//     the 128-byte-swizzled K-major layout, then arrives on the leader.
//   O_k += P_k V (M=256, N=128: the two d halves, K=128 keys) -> TMEM O_k.
// Warps: 0-3 and 4-7 softmax for sub-tiles 0 and 1 (warp q: rows 32q ..
// 32q+31, all 128 columns); 8 TMA producer; 9 TMEM allocation (both CTAs)
// and, in the leader CTA only, the MMA issuer.
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
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;            // S_0, S_1, O_0, O_1
constexpr int kBox = 128 * 128;                // one [128 rows][64 bf16] swizzled box set
constexpr int kQBytes = 2 * kBox;              // Q_k: [128][128]
constexpr int kPBytes = 2 * kBox;              // P_k: [128 rows][128 keys]
constexpr int kKHalf = 64 * 128;               // [64 keys][64 d]
constexpr int kSlotBytes = 2 * kKHalf;         // K: 64 keys x 128 d; V: 128 keys x 64 d
constexpr int kQOff = 0;
constexpr int kPOff = 2 * kQBytes;
constexpr int kRingOff = kPOff + 2 * kPBytes;
constexpr int kSlots = 6;
constexpr int kBarOff = kRingOff + kSlots * kSlotBytes;
constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 2 + 2;
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
    uint64_t *slot_full = bar + 1;
    uint64_t *slot_free = slot_full + kSlots;
    uint64_t *s_full = slot_free + kSlots;  // [2]
    uint64_t *p_full = s_full + 2;          // [2] leader: 8 arrivals (the softmax warps of both CTAs)
    uint64_t *o_done = p_full + 2;          // [2]
    uint64_t *v_last = o_done + 2;          // local: this CTA's half of the last V tile landed
    uint64_t *v_tail = v_last + 1;          // leader: both halves zeroed past the last key
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
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&slot_full[i], 1);
            mbar_init(&slot_free[i], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], 2 * 4);  // one arrival per softmax warp of each CTA
            mbar_init(&o_done[k], 1);
        }
        mbar_init(v_last, 1);
        mbar_init(v_tail, 2);
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
        for (int t = 0; t < T; ++t) {
            int rows_of[kBPT];  // pool row of each block of this tile (or past the pool)
            if (PAGED) {
                const int bi = t * kBPT + lane;
                int row = oob_row;
                if (lane < kBPT && bi < nb_used) {
                    int blk = bt[bi];
                    if ((unsigned)blk >= (unsigned)a.num_blocks) {
                        set_error(a.err, PA_ERR_BAD_INDEX);
                        blk = 0;  // never dereference an out-of-range block
                    }
                    row = (blk * a.num_kv_heads + g) * BS;
                }
#pragma unroll
                for (int jb = 0; jb < kBPT; ++jb) rows_of[jb] = __shfl_sync(0xffffffffu, row, jb);
            }
            const bool last_v = (t == T - 1);
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                const int i = 2 * t + kv;
                const int slot = i % kSlots;
                uint8_t *dst = smem + kRingOff + slot * kSlotBytes;
                bool ok = true;
                if (lane == 0 && i >= kSlots) ok = mbar_wait(&slot_free[slot], ((i / kSlots) - 1) & 1, a.err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok || *(volatile int *)s_abort) {
                    if (lane == 0) atomicExch(s_abort, 1);
                    break;
                }
                if (kv == 0) {
                    // K: this CTA's 64 keys, both halves of d
                    if (lane == 0) {
                        const uint32_t lb = map_to_cta(smem_u32(&slot_full[slot]), 0);
                        if (c == 0) mbar_arrive_expect_tx(&slot_full[slot], 2 * kSlotBytes);
                        if (PAGED) {
#pragma unroll
                            for (int jb = 0; jb < 64 / BS; ++jb)
#pragma unroll
                                for (int hf = 0; hf < 2; ++hf)
                                    tma_load_2d_pair(dst + hf * kKHalf + jb * BS * 128, &tm_k, lb, hf * 64,
                                                     c == 0 ? rows_of[jb] : rows_of[64 / BS + jb]);
                        } else {
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf)
                                tma_load_3d_pair(dst + hf * kKHalf, &tm_k, lb, hf * 64, g, row0 + t * kBN + 64 * c);
                        }
                    }
                } else if (!last_v) {
                    // V: all 128 keys, this CTA's half of d
                    if (lane == 0) {
                        const uint32_t lb = map_to_cta(smem_u32(&slot_full[slot]), 0);
                        if (c == 0) mbar_arrive_expect_tx(&slot_full[slot], 2 * kSlotBytes);
                        if (PAGED) {
#pragma unroll
                            for (int jb = 0; jb < kBPT; ++jb)
                                tma_load_2d_pair(dst + jb * BS * 128, &tm_v, lb, c * 64, rows_of[jb]);
                        } else {
                            tma_load_3d_pair(dst, &tm_v, lb, c * 64, g, row0 + t * kBN);
                        }
                    }
                } else {
                    // The last V tile: land it against a local barrier, zero
                    // its rows past the last key, then tell the leader.
                    if (lane == 0) {
                        mbar_arrive_expect_tx(v_last, kSlotBytes);
                        if (PAGED) {
#pragma unroll
                            for (int jb = 0; jb < kBPT; ++jb)
                                tma_load_2d(dst + jb * BS * 128, &tm_v, v_last, c * 64, rows_of[jb]);
                        } else {
                            tma_load_3d(dst, &tm_v, v_last, c * 64, g, row0 + t * kBN);
                        }
                    }
                    const bool vok = __all_sync(0xffffffffu, mbar_wait(v_last, 0, a.err));
                    if (vok) {
                        const int valid = kv_end_max - t * kBN;
                        for (int r = valid + (lane >> 3); r < kBN; r += 4)
                            *reinterpret_cast<uint4 *>(dst + r * 128 + (lane & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) {
                        if (vok) mbar_arrive_cluster(map_to_cta(smem_u32(v_tail), 0));
                        else atomicExch(s_abort, 1);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        // --------------------------------------------------------- MMA issue --
        if (c == 0 && lane == 0) {
            constexpr uint32_t kIdescS = umma_idesc_bf16(2 * kBM, kBN, false, false);
            constexpr uint32_t kIdescO = umma_idesc_bf16(2 * kBM, kD, false, true);
            const uint64_t dq[2] = {umma_desc_sw128(smem_u32(smem + kQOff), 16, 1024),
                                    umma_desc_sw128(smem_u32(smem + kQOff + kQBytes), 16, 1024)};
            const uint64_t dp[2] = {umma_desc_sw128(smem_u32(smem + kPOff), 16, 1024),
                                    umma_desc_sw128(smem_u32(smem + kPOff + kPBytes), 16, 1024)};
            const uint64_t dk0 = umma_desc_sw128(smem_u32(smem + kRingOff), 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(smem_u32(smem + kRingOff), kBox, 1024);
            bool ok = mbar_wait_spin(q_full, 0, a.err);
            auto issue_s = [&](int k, int t) {
                const int i = 2 * t, sl = i % kSlots;
                if (!ok) return;
                const bool first = (k == 0) || nkt[0] <= t;
                const bool last = (k == 1) || nkt[1] <= t;
                if (first) {
                    ok = mbar_wait_spin(&slot_full[sl], (i / kSlots) & 1, a.err);
                    if (ok && t < T - 1)
                        ok = mbar_wait_spin(&slot_full[(i + 1) % kSlots], ((i + 1) / kSlots) & 1, a.err);
                    if (!ok) return;
                }
                tc_fence_after();
                const uint64_t bk = dk0 + (uint64_t)((sl * kSlotBytes) >> 4);
                const uint32_t d = tmem + k * kBN;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_bf16_pair(d, dq[k] + (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                                   bk + (uint64_t)(((kk >> 2) * kKHalf + (kk & 3) * 32) >> 4), kIdescS, kk > 0);
                umma_commit_pair(&s_full[k]);
                if (last) umma_commit_pair(&slot_free[sl]);
            };
            auto issue_pv = [&](int k, int t) {
                const int i = 2 * t + 1, sl = i % kSlots;
                if (!ok || !(ok = mbar_wait_spin(&p_full[k], t & 1, a.err))) return;
                const bool first = (k == 0) || nkt[0] <= t;
                const bool last = (k == 1) || nkt[1] <= t;
                if (t == T - 1 && first && !(ok = mbar_wait_spin(v_tail, 0, a.err))) return;
                tc_fence_after();
                const uint64_t bv = dv0 + (uint64_t)((sl * kSlotBytes) >> 4);
                const uint32_t d = tmem + 2 * kBN + k * kD;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    umma_bf16_pair(d, dp[k] + (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4),
                                   bv + (uint64_t)((kk * 2048) >> 4), kIdescO, (t > 0 || kk > 0) ? 1u : 0u);
                if (t == nkt[k] - 1) umma_commit_pair(&o_done[k]);
                if (last) umma_commit_pair(&slot_free[sl]);
            };
            if (nkt[0] > 0) issue_s(0, 0);
            if (nkt[1] > 0) issue_s(1, 0);
            for (int t = 0; t < T; ++t) {
                if (t < nkt[0]) {
                    issue_pv(0, t);
                    if (t + 1 < nkt[0]) issue_s(0, t + 1);
                }
                if (t < nkt[1]) {
                    issue_pv(1, t);
                    if (t + 1 < nkt[1]) issue_s(1, t + 1);
                }
            }
            if (!ok) atomicExch(s_abort, 1);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- softmax --
        // Warps 4k .. 4k+3 do sub-tile k; warp q owns rows 32q .. 32q+31 (TMEM
        // lane quadrant q), one row per thread, all 128 columns.
        const int k = warp >> 2, q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t tS = tmem + lane_base + k * kBN;
        const uint32_t tO = tmem + lane_base + 2 * kBN + k * kD;
        const RowTile my = k == 0 ? mine[0] : mine[1];
        const int nk = k == 0 ? nkt[0] : nkt[1];
        const uint32_t pf = map_to_cta(smem_u32(&p_full[k]), 0);
        uint8_t *pbuf = smem + kPOff + k * kPBytes;
        const int lim_abs = min(p0 + my.q0 + r + 1, my.kv_end);
        const float sl = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        auto wait_warp = [&](uint64_t *bb, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bb, par, a.err));
        };
        for (int t = 0; t < nk; ++t) {
            if (!wait_warp(&s_full[k], t & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int lim = lim_abs - t * kBN;  // visible columns of this row
            float v[kBN];
            tmem_ld128(tS, v);
            if (lim < kBN) {
#pragma unroll
                for (int j = 0; j < kBN; ++j)
                    if (j >= lim) v[j] = -INFINITY;
            }
            float m4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) m4[i] = fmax3(v[i], v[i + 4], v[i + 8]);
#pragma unroll
            for (int j = 12; j < kBN; j += 8)
#pragma unroll
                for (int i = 0; i < 4; ++i) m4[i] = fmax3(m4[i], v[j + i], j + 4 + i < kBN ? v[j + 4 + i] : -INFINITY);
            const float mx = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
            const float m_new = fmaxf(m_run, mx * sl);
            // Move the running maximum only when it grew by more than 2^8 for
            // some row of the warp; O_k is rescaled after P is written.
            const bool rescale = t > 0 && __any_sync(0xffffffffu, m_new > m_run + 8.f);
            const float alpha = rescale ? fast_exp2(m_run - m_new) : 1.f;
            if (t == 0 || rescale) m_run = m_new;
            const float mu = m_run == -INFINITY ? 0.f : m_run;
            // P_k(t) overwrites P_k(t-1): S_k(t) completing implies PV_k(t-1) read it.
            float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int jj = 0; jj < kBN / 8; ++jj) {
                const uint4 pk = make_uint4(
                    pack_bf16x2(fast_exp2(fmaf(v[jj * 8 + 0], sl, -mu)), fast_exp2(fmaf(v[jj * 8 + 1], sl, -mu))),
                    pack_bf16x2(fast_exp2(fmaf(v[jj * 8 + 2], sl, -mu)), fast_exp2(fmaf(v[jj * 8 + 3], sl, -mu))),
                    pack_bf16x2(fast_exp2(fmaf(v[jj * 8 + 4], sl, -mu)), fast_exp2(fmaf(v[jj * 8 + 5], sl, -mu))),
                    pack_bf16x2(fast_exp2(fmaf(v[jj * 8 + 6], sl, -mu)), fast_exp2(fmaf(v[jj * 8 + 7], sl, -mu))));
                // row sums of the same bf16-rounded weights that multiply V
                ls2[0] = add_f32x2(ls2[0], bf16x2_unpack(pk.x));
                ls2[1] = add_f32x2(ls2[1], bf16x2_unpack(pk.y));
                ls2[0] = add_f32x2(ls2[0], bf16x2_unpack(pk.z));
                ls2[1] = add_f32x2(ls2[1], bf16x2_unpack(pk.w));
                *reinterpret_cast<uint4 *>(pbuf + (jj >> 3) * kBox + r * 128 + (((jj & 7) ^ (r & 7)) << 4)) = pk;
            }
            l_run = l_run * alpha + ((ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y));
            if (rescale) {
                // O_k is stable: S_k(t) completing implies PV_k(t-1) has, and
                // PV_k(t) waits for this warp's arrival below.
#pragma unroll
                for (int cc = 0; cc < kD / 32; ++cc) {
                    float o[32];
                    tmem_ld32(tO + cc * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tO + cc * 32, o);
                }
            }
            // Every thread makes its P row visible to the tensor core, then one
            // arrival per warp on the leader's barrier.
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (c == 0) mbar_arrive(&p_full[k]);
                else mbar_arrive_cluster(pf);
            }
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
