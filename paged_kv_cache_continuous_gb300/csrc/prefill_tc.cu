// prefill_tc.cu -- causal, ragged (varlen-packed) prefill attention on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// What it computes (text-generation-inference Router/Webserver deep dive,
// section "Prefill, Decode and past key values": the first pass over a prompt
// computes the complete attention matrix; the scheduling-loop section adds
// that prompts may be chunked and merged into the running batch): row i of
// sequence s sits at absolute position p0 + i and
//     out = softmax(scale * q K^T + causal mask) V   over keys 0 .. p0 + i.
// Ragged prompts are packed by cu_seqlens (Blitzscale docs, section "Model":
// ragged index-pointer buffers).
//
// One CTA owns two 128-row query sub-tiles that read the same keys: two query
// heads of one KV head (grouped heads) or, with an odd group size, two
// consecutive row tiles of one head.  Every K/V tile is loaded once for both.
// Warp roles (320 threads):
//   warps 0-3, 4-7  softmax warpgroups, one per sub-tile: thread r owns query
//                   row r = TMEM lane r;
//   warp 8          TMA producer: both Q tiles, then K_0, V_0, K_1, V_1, ...
//                   through a ring of 128-key slots (paged form: one box per
//                   KV block and 64-column half; block ids range-checked);
//   warp 9          allocates 512 TMEM columns and issues every MMA from one
//                   thread: S_k = Q_k K^T (M = N = 128, K = d) into TMEM, and
//                   O_k += P_k V (M = 128, N = d, K = 128) with P_k read from
//                   TMEM, where the softmax wrote it over S_k as bf16 pairs.
// Issue order S_A0, S_B0, PV_A0, S_A1, PV_B0, S_B1, PV_A1, ... keeps the
// tensor core busy with one sub-tile while the other's softmax runs.  The
// running maximum is only moved (and O rescaled in TMEM) when it grows by
// more than 2^8.  Row sums use the same bf16-rounded weights that multiply V.
// V rows past the last key of the last tile are zeroed (stale pool rows could
// hold NaN, and 0 * NaN = NaN).
#include <cuda.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kBM = 128;              // rows per query sub-tile
constexpr int kBN = 128;              // keys per KV tile
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;   // S_A, S_B (128 each), O_A, O_B (d each)
constexpr int kTileHalf = 128 * 128;  // bytes of one [128 rows][64 bf16] swizzled box set

template <int D>
struct PrefillCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kQBytes = kHalves * kTileHalf;     // one query sub-tile
    static constexpr int kSlotBytes = kHalves * kTileHalf;  // one 128-key K or V tile
    static constexpr int kRingOff = 2 * kQBytes;
    static constexpr int kSlotsFit = (224 * 1024 - 2 * kQBytes) / kSlotBytes;
    static constexpr int kSlots = kSlotsFit > 8 ? 8 : kSlotsFit;
    static constexpr int kBarOff = kRingOff + kSlots * kSlotBytes;
    static constexpr int kNumBars = 1 + 2 * kSlots + 7;
    static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
};

struct SubTile {
    int h, q0, rows, kv_end, nkt;
};

template <int D, int BS, bool PAGED, bool HEAD_PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *q_full = bar;
    uint64_t *slot_full = bar + 1;
    uint64_t *slot_free = slot_full + C::kSlots;
    uint64_t *s_full = slot_free + C::kSlots;  // [2]
    uint64_t *p_full = s_full + 2;             // [2]
    uint64_t *o_done = p_full + 2;             // [2]
    uint64_t *v_tail = o_done + 2;             // last V tile ready (tail rows zeroed)
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar + C::kNumBars);
    int *s_abort = reinterpret_cast<int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.z;

    if (a.check_err_first && *(volatile int *)a.err != 0) return;
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
    // ---- the two sub-tiles (longest causal rows first)
    SubTile sub[2];
    if (HEAD_PAIR) {
        const int qt = gridDim.x - 1 - blockIdx.x;
        sub[0].h = 2 * blockIdx.y;
        sub[1].h = 2 * blockIdx.y + 1;
        sub[0].q0 = sub[1].q0 = qt * kBM;
    } else {
        const int pair = gridDim.x - 1 - blockIdx.x;
        sub[0].h = sub[1].h = blockIdx.y;
        sub[0].q0 = 2 * pair * kBM;
        sub[1].q0 = (2 * pair + 1) * kBM;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        sub[k].rows = max(0, min(kBM, n - sub[k].q0));
        sub[k].kv_end = sub[k].rows > 0 ? p0 + sub[k].q0 + sub[k].rows : 0;
        sub[k].nkt = sub[k].rows > 0 ? (sub[k].kv_end + kBN - 1) / kBN : 0;
    }
    if (sub[0].rows == 0) return;  // sub-tile 1 starts no earlier than sub-tile 0
    const int g = sub[0].h / a.group;
    const int T = max(sub[0].nkt, sub[1].nkt);  // KV tiles loaded by this CTA
    const int kv_end_max = max(sub[0].kv_end, sub[1].kv_end);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(&slot_full[i], 1);
            mbar_init(&slot_free[i], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], 128);
            mbar_init(&o_done[k], 1);
        }
        mbar_init(v_tail, 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------- producer --
        constexpr int kBPT = kBN / BS;  // pool blocks per KV tile
        const int nb_used = (kv_end_max + BS - 1) / BS;
        const int32_t *bt = PAGED ? a.block_table + (size_t)s * a.max_blocks : nullptr;
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const int nq = sub[1].rows > 0 ? 2 : 1;
            mbar_arrive_expect_tx(q_full, nq * C::kQBytes);
            for (int k = 0; k < nq; ++k)
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf)
                    tma_load_3d(smem + k * C::kQBytes + hf * kTileHalf, &tm_q, q_full, hf * 64, sub[k].h,
                                row0 + sub[k].q0);
        }
        for (int t = 0; t < T; ++t) {
            int ids[kBPT];
            int nload = kBPT;
            if (PAGED) {
                const int bi = t * kBPT + lane;
                int blk = 0;
                if (lane < kBPT && bi < nb_used) {
                    blk = bt[bi];
                    if ((unsigned)blk >= (unsigned)a.num_blocks) {
                        set_error(a.err, PA_ERR_BAD_INDEX);
                        blk = 0;  // never dereference an out-of-range block
                    }
                }
#pragma unroll
                for (int jb = 0; jb < kBPT; ++jb) ids[jb] = __shfl_sync(0xffffffffu, blk, jb);
                nload = min(kBPT, nb_used - t * kBPT);
            }
            if (lane == 0 && !*(volatile int *)s_abort) {
                const uint32_t bytes =
                    PAGED ? (uint32_t)(nload * BS * 128 * C::kHalves) : (uint32_t)C::kSlotBytes;
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    const int i = 2 * t + kv;
                    const int slot = i % C::kSlots;
                    if (i >= C::kSlots && !mbar_wait(&slot_free[slot], ((i / C::kSlots) - 1) & 1, a.err)) {
                        atomicExch(s_abort, 1);
                        break;
                    }
                    const CUtensorMap *tm = kv == 0 ? &tm_k : &tm_v;
                    uint8_t *dst = smem + C::kRingOff + slot * C::kSlotBytes;
                    mbar_arrive_expect_tx(&slot_full[slot], bytes);
                    if (PAGED) {
#pragma unroll
                        for (int jb = 0; jb < kBPT; ++jb)
                            if (jb < nload)
#pragma unroll
                                for (int hf = 0; hf < C::kHalves; ++hf)
                                    tma_load_2d(dst + hf * kTileHalf + jb * BS * 128, tm, &slot_full[slot],
                                                hf * 64, (ids[jb] * a.num_kv_heads + g) * BS);
                    } else {
#pragma unroll
                        for (int hf = 0; hf < C::kHalves; ++hf)
                            tma_load_3d(dst + hf * kTileHalf, tm, &slot_full[slot], hf * 64, g, row0 + t * kBN);
                    }
                }
            }
            __syncwarp();
        }
        // Rows of the last V tile past the last key hold stale pool rows (or
        // nothing); zero them once the tile has landed, then release it to
        // the MMA warp.
        {
            const int t = T - 1;
            const int i = 2 * t + 1;
            const int slot = i % C::kSlots;
            const int valid = kv_end_max - t * kBN;
            bool vok = true;
            if (valid < kBN) {
                vok = __all_sync(0xffffffffu, mbar_wait(&slot_full[slot], (i / C::kSlots) & 1, a.err));
                if (vok) {
                    uint8_t *vt = smem + C::kRingOff + slot * C::kSlotBytes;
                    for (int r = valid + (lane >> 3); r < kBN; r += 4)
#pragma unroll
                        for (int hf = 0; hf < C::kHalves; ++hf)
                            *reinterpret_cast<uint4 *>(vt + hf * kTileHalf + r * 128 + (lane & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                }
                __syncwarp();
            }
            if (lane == 0 && vok) mbar_arrive(v_tail);
        }
    } else if (warp == kMmaWarp) {
        // --------------------------------------------------------- MMA issue --
        // One thread issues everything.  Descriptors are built once; an MMA
        // then costs one add on the start-address field (all shared-memory
        // offsets stay below 2^18, so the 14-bit field never carries).
        if (lane == 0) {
            constexpr uint32_t kIdescS = umma_idesc_bf16(kBM, kBN, false, false);
            constexpr uint32_t kIdescO = umma_idesc_bf16(kBM, D, false, true);
            const uint64_t dq[2] = {umma_desc_sw128(smem_u32(smem), 16, 1024),
                                    umma_desc_sw128(smem_u32(smem + C::kQBytes), 16, 1024)};
            const uint64_t dk0 = umma_desc_sw128(smem_u32(smem + C::kRingOff), 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(smem_u32(smem + C::kRingOff), kTileHalf, 1024);
            bool ok = mbar_wait(q_full, 0, a.err);
            // The first reader of tile t waits for both of its slots (K_t, V_t)
            // once; later groups of the tile only wait for their true inputs.
            auto issue_s = [&](int k, int t) {
                const int i = 2 * t, sl = i % C::kSlots;
                if (!ok) return;
                if (k == 0 || sub[0].nkt <= t) {
                    ok = mbar_wait(&slot_full[sl], (i / C::kSlots) & 1, a.err) &&
                         mbar_wait(&slot_full[(i + 1) % C::kSlots], ((i + 1) / C::kSlots) & 1, a.err);
                    if (!ok) return;
                }
                tc_fence_after();
                const uint64_t bq = dq[k];
                const uint64_t bk = dk0 + (uint64_t)((sl * C::kSlotBytes) >> 4);
                const uint32_t d = tmem + k * kBN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * kTileHalf + (kk & 3) * 32) >> 4);
                    umma_bf16(d, bq + off, bk + off, kIdescS, kk > 0);
                }
                umma_commit(&s_full[k]);
                if (k == 1 || sub[1].nkt <= t) umma_commit(&slot_free[sl]);  // last reader of K_t
            };
            auto issue_pv = [&](int k, int t) {
                const int i = 2 * t + 1, sl = i % C::kSlots;
                if (!ok || !(ok = mbar_wait(&p_full[k], t & 1, a.err))) return;
                const bool first_user = (k == 0) || sub[0].nkt <= t;
                if (t == T - 1 && first_user && !(ok = mbar_wait(v_tail, 0, a.err))) return;
                tc_fence_after();
                const uint64_t bv = dv0 + (uint64_t)((sl * C::kSlotBytes) >> 4);
                const uint32_t tP = tmem + k * kBN;  // P_k: 64 columns of bf16 pairs over S_k
                const uint32_t tO = tmem + 2 * kBN + k * D;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    umma_bf16_tmem_a(tO, tP + kk * 8, bv + (uint64_t)((kk * 2048) >> 4), kIdescO,
                                     (t > 0 || kk > 0) ? 1u : 0u);
                if (t == (k == 0 ? sub[0].nkt : sub[1].nkt) - 1) umma_commit(&o_done[k]);
                if (k == 1 || sub[1].nkt <= t) umma_commit(&slot_free[sl]);  // last reader of V_t
            };
            if (sub[0].nkt > 0) issue_s(0, 0);
            if (sub[1].nkt > 0) issue_s(1, 0);
            for (int t = 0; t < T; ++t) {
                if (t < sub[0].nkt) {
                    issue_pv(0, t);
                    if (t + 1 < sub[0].nkt) issue_s(0, t + 1);
                }
                if (t < sub[1].nkt) {
                    issue_pv(1, t);
                    if (t + 1 < sub[1].nkt) issue_s(1, t + 1);
                }
            }
            if (!ok) atomicExch(s_abort, 1);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- softmax --
        const int k = warp >> 2;              // sub-tile of this warpgroup
        const SubTile st = k == 0 ? sub[0] : sub[1];
        const int r = threadIdx.x & 127;      // query row within the sub-tile, TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + k * kBN;
        const uint32_t tO = tmem + lane_base + 2 * kBN + k * D;
        const int pos = p0 + st.q0 + r;
        const int lim_abs = min(pos + 1, st.kv_end);
        const float sl = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        // Every lane waits; the warp proceeds only if all saw the phase
        // complete, so the warp-collective TMEM accesses stay convergent.
        auto wait_warp = [&](uint64_t *bb, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bb, par, a.err));
        };
        for (int t = 0; t < st.nkt; ++t) {
            if (!wait_warp(&s_full[k], t & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int lim = lim_abs - t * kBN;  // columns < lim are visible to this row
            // The whole row of S in one TMEM load; the causal mask (diagonal
            // tiles only) is applied once, in registers.
            float v[kBN];
            tmem_ld128(tS, v);
            // Warp-uniform branch: only tiles crossing some row's last key pay
            // for the mask.
            if (__any_sync(0xffffffffu, lim < kBN)) {
#pragma unroll
                for (int j = 0; j < kBN; ++j) v[j] = j < lim ? v[j] : -INFINITY;
            }
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = v[i];
#pragma unroll
            for (int j = 8; j < kBN; ++j) m8[j & 7] = fmaxf(m8[j & 7], v[j]);
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            const float m_new = fmaxf(m_run, mx * sl);
            if (t == 0) {
                m_run = m_new;
            } else if (__any_sync(0xffffffffu, m_new > m_run + 8.f)) {
                // O_k is stable here: S_k(t) completing implies PV_k(t-1) has.
                const float alpha = fast_exp2(m_run - m_new);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tO + c * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(tO + c * 32, o);
                }
                l_run *= alpha;
                m_run = m_new;
            }
            const float mu = m_run == -INFINITY ? 0.f : m_run;
            // Weights as bf16 pairs, written over the first 64 columns of S
            // (already read) in one TMEM store.
            uint32_t pk[kBN / 2];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < kBN / 2; ++j) {
                pk[j] = pack_bf16x2(fast_exp2(fmaf(v[2 * j], sl, -mu)), fast_exp2(fmaf(v[2 * j + 1], sl, -mu)));
                ls[j & 3] += bf16x2_sum(pk[j]);
            }
            tmem_st64(tS, pk);
            const float lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
            l_run += lsum;
            tc_fence_before();
            mbar_arrive(&p_full[k]);
        }
        // --------------------------------------------------------- epilogue --
        if (st.nkt > 0) {
            const bool aborted = !ok || __any_sync(0xffffffffu, *(volatile int *)s_abort != 0);
            if (!aborted && wait_warp(&o_done[k], 0)) {
                tc_fence_after();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                __nv_bfloat16 *orow = a.out + ((size_t)(row0 + st.q0 + r) * a.num_q_heads + st.h) * D;
                float o[D];
                if constexpr (D == 128) tmem_ld128(tO, o);
                else tmem_ld64(tO, o);
                if (r < st.rows) {
#pragma unroll
                    for (int i = 0; i < D; i += 8) {
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
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int BS, bool PAGED, bool HEAD_PAIR>
cudaError_t launch_prefill_t(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const PrefillArgs &a, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    static std::atomic<unsigned long long> opted{0};
    cudaError_t e0 = opt_in_smem(reinterpret_cast<const void *>(prefill_tc_kernel<D, BS, PAGED, HEAD_PAIR>),
                                 C::kSmemBytes, opted);
    if (e0 != cudaSuccess) return e0;
    dim3 grid(HEAD_PAIR ? a.num_q_tiles : (a.num_q_tiles + 1) / 2,
              HEAD_PAIR ? a.num_q_heads / 2 : a.num_q_heads, a.num_seqs);
    prefill_tc_kernel<D, BS, PAGED, HEAD_PAIR><<<grid, kThreads, C::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, a);
    return cudaGetLastError();
}

template <int D, int BS, bool PAGED>
cudaError_t launch_prefill_p(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const PrefillArgs &a, cudaStream_t stream) {
    // Two query heads share a KV head when the group size is even.
    if (a.group % 2 == 0) return launch_prefill_t<D, BS, PAGED, true>(tm_q, tm_k, tm_v, a, stream);
    return launch_prefill_t<D, BS, PAGED, false>(tm_q, tm_k, tm_v, a, stream);
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const PrefillArgs &a, int head_dim, int block_size, cudaStream_t stream) {
    const bool paged = a.block_table != nullptr;
#define PA_PRE(D, BS)                                                                         \
    if (head_dim == D && block_size == BS)                                                    \
        return paged ? launch_prefill_p<D, BS, true>(tm_q, tm_k, tm_v, a, stream)             \
                     : launch_prefill_p<D, 16, false>(tm_q, tm_k, tm_v, a, stream);
    PA_PRE(128, 16)
    PA_PRE(128, 32)
    PA_PRE(64, 16)
    PA_PRE(64, 32)
#undef PA_PRE
    return cudaErrorInvalidValue;
}

}  // namespace pa
