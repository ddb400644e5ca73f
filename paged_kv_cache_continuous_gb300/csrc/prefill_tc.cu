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
// One CTA per (128-row query tile, query head, sequence); warp roles:
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r;
//   warp 4     TMA producer: Q once, then K/V tiles of 128 keys into a
//              2-stage ring (paged form: one box per KV block and 64-column
//              half, block ids range-checked);
//   warp 5     allocates 512 TMEM columns and issues the MMAs from one thread:
//              S_t = Q K_t^T (M=N=128, K=d) into one of two S buffers, then
//              O += P_t V_t (M=128, N=d, K=128) into the O buffer; tcgen05.commit
//              signals mbarriers as each group completes.
// Issue order S_0, S_1, PV_0, S_2, PV_1, ... lets S_{t+1} run on the tensor
// core while the softmax warps work on S_t.  P (bf16) goes through shared
// memory in the 128-byte-swizzled K-major layout the MMA reads; the running
// maximum is only moved (and O rescaled in TMEM) when it grows by more than
// 2^8, so most tiles never touch O.  Rows past the sequence's keys in the last
// KV tile are zeroed in V (stale pool rows could hold NaN, and 0 * NaN = NaN).
#include <cuda.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per KV tile
constexpr int kNKV = 2;           // K/V ring stages
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileHalf = 128 * 128;  // bytes of one [128 rows][64 bf16] swizzled box set

template <int D>
struct PrefillCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kQBytes = kHalves * kTileHalf;
    static constexpr int kKVBytes = kHalves * kTileHalf;  // one 128-key K (or V) tile
    static constexpr int kPBytes = 2 * kTileHalf;         // P: [128][128] bf16
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;
    static constexpr int kVOff = kKOff + kNKV * kKVBytes;
    static constexpr int kPOff = kVOff + kNKV * kKVBytes;
    static constexpr int kBarOff = kPOff + 2 * kPBytes;
    static constexpr int kNumBars = 17;
    static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;
};

struct Bars {
    uint64_t *q_full, *k_full, *k_free, *v_full, *v_free, *s_full, *s_free, *p_full, *pv_done;
};

template <int D, int BS, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    Bars B{bar + 0, bar + 1, bar + 3, bar + 5, bar + 7, bar + 9, bar + 11, bar + 13, bar + 15};
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar + C::kNumBars);
    int *s_abort = reinterpret_cast<int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = gridDim.x - 1 - blockIdx.x;  // longest causal rows first
    const int h = blockIdx.y, s = blockIdx.z;
    const int g = h / a.group;

    if (a.check_err_first && *(volatile int *)a.err != 0) return;
    const int row0 = a.cu_seqlens[s];
    const int n = a.cu_seqlens[s + 1] - row0;
    const int p0 = a.prefix_lens ? a.prefix_lens[s] : (a.seq_lens ? a.seq_lens[s] - n : 0);
    const bool bad = n < 0 || p0 < 0 || row0 < 0 || (long long)row0 + n > a.num_tokens ||
                     n > a.max_q_len || (PAGED && (p0 + n + BS - 1) / BS > a.max_blocks) ||
                     (!PAGED && p0 != 0);
    if (bad) {
        if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) set_error(a.err, PA_ERR_BAD_INDEX);
        return;
    }
    const int q0 = qt * kBM;
    if (q0 >= n) return;
    const int rows = min(kBM, n - q0);
    const int kv_end = p0 + q0 + rows;  // keys [0, kv_end) are visible to some row
    const int nkt = (kv_end + kBN - 1) / kBN;

    if (threadIdx.x == 0) {
        mbar_init(B.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.k_full[i], 1);
            mbar_init(&B.k_free[i], 1);
            mbar_init(&B.v_full[i], 1);
            mbar_init(&B.v_free[i], 1);
            mbar_init(&B.s_full[i], 1);
            mbar_init(&B.s_free[i], 128);
            mbar_init(&B.p_full[i], 128);
            mbar_init(&B.pv_done[i], 1);
        }
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tmem_o = tmem + 2 * kBN;

    if (warp == 4) {
        // ---------------------------------------------------------- producer --
        constexpr int kBPT = kBN / BS;  // pool blocks per KV tile
        const int nb_used = (kv_end + BS - 1) / BS;
        const int32_t *bt = PAGED ? a.block_table + (size_t)s * a.max_blocks : nullptr;
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(B.q_full, C::kQBytes);
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_3d(smem + C::kQOff + hf * kTileHalf, &tm_q, B.q_full, hf * 64, h, row0 + q0);
        }
        for (int t = 0; t < nkt; ++t) {
            const int st = t % kNKV;
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
                const uint32_t bytes = PAGED ? (uint32_t)(nload * BS * 128 * C::kHalves) : (uint32_t)C::kKVBytes;
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    uint64_t *fullb = kv == 0 ? &B.k_full[st] : &B.v_full[st];
                    uint64_t *freeb = kv == 0 ? &B.k_free[st] : &B.v_free[st];
                    const CUtensorMap *tm = kv == 0 ? &tm_k : &tm_v;
                    uint8_t *dst = smem + (kv == 0 ? C::kKOff : C::kVOff) + st * C::kKVBytes;
                    if (t >= kNKV && !mbar_wait(freeb, ((t / kNKV) - 1) & 1, a.err)) {
                        atomicExch(s_abort, 1);
                        break;
                    }
                    mbar_arrive_expect_tx(fullb, bytes);
                    if (PAGED) {
#pragma unroll
                        for (int jb = 0; jb < kBPT; ++jb)
                            if (jb < nload)
#pragma unroll
                                for (int hf = 0; hf < C::kHalves; ++hf)
                                    tma_load_2d(dst + hf * kTileHalf + jb * BS * 128, tm, fullb, hf * 64,
                                                (ids[jb] * a.num_kv_heads + g) * BS);
                    } else {
#pragma unroll
                        for (int hf = 0; hf < C::kHalves; ++hf)
                            tma_load_3d(dst + hf * kTileHalf, tm, fullb, hf * 64, g, row0 + t * kBN);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == 5) {
        // --------------------------------------------------------- MMA issue --
        constexpr uint32_t kIdescS = umma_idesc_bf16(kBM, kBN, false, false);
        constexpr uint32_t kIdescO = umma_idesc_bf16(kBM, D, false, true);
        const uint32_t sQ = smem_u32(smem + C::kQOff);
        bool ok = true;
        if (lane == 0) ok = mbar_wait(B.q_full, 0, a.err);
        auto issue_s = [&](int t) {
            const int st = t % kNKV, b = t & 1;
            if (lane == 0 && ok) {
                ok = mbar_wait(&B.k_full[st], (t / kNKV) & 1, a.err);
                if (ok && t >= 2) ok = mbar_wait(&B.s_free[b], ((t - 2) >> 1) & 1, a.err);
                if (ok) {
                    tc_fence_after();
                    const uint32_t sK = smem_u32(smem + C::kKOff + st * C::kKVBytes);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kTileHalf + (kk & 3) * 32;
                        umma_bf16(tmem + b * kBN, umma_desc_sw128(sQ + off, 16, 1024),
                                  umma_desc_sw128(sK + off, 16, 1024), kIdescS, kk > 0);
                    }
                    umma_commit(&B.s_full[b]);
                    umma_commit(&B.k_free[st]);
                }
            }
            __syncwarp();
        };
        auto issue_pv = [&](int u) {
            const int st = u % kNKV, b = u & 1;
            const int valid = kv_end - u * kBN;  // keys of this tile that exist
            const bool zero_tail = valid < kBN;
            if (lane == 0 && ok) ok = mbar_wait(&B.p_full[b], (u >> 1) & 1, a.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok && (zero_tail || lane == 0)) ok = mbar_wait(&B.v_full[st], (u / kNKV) & 1, a.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok && zero_tail) {
                uint8_t *vt = smem + C::kVOff + st * C::kKVBytes;
                for (int r = valid + (lane >> 3); r < kBN; r += 4)
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        *reinterpret_cast<uint4 *>(vt + hf * kTileHalf + r * 128 + (lane & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0 && ok) {
                tc_fence_after();
                const uint32_t sP = smem_u32(smem + C::kPOff + b * C::kPBytes);
                const uint32_t sV = smem_u32(smem + C::kVOff + st * C::kKVBytes);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t ad = umma_desc_sw128(sP + (kk >> 2) * kTileHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(sV + kk * 2048, kTileHalf, 1024);
                    umma_bf16(tmem_o, ad, bd, kIdescO, (u > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&B.pv_done[b]);
                umma_commit(&B.v_free[st]);
            }
            __syncwarp();
        };
        for (int t = 0; t < nkt; ++t) {
            issue_s(t);
            if (t >= 1) issue_pv(t - 1);
        }
        issue_pv(nkt - 1);
        if (!__shfl_sync(0xffffffffu, ok, 0) && lane == 0) atomicExch(s_abort, 1);
    } else {
        // ----------------------------------------------------------- softmax --
        const int r = threadIdx.x;  // query row within the tile, TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int pos = p0 + q0 + r;
        const int lim_abs = min(pos + 1, kv_end);
        const float sl = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        // Every lane waits; the warp proceeds only if all saw the phase
        // complete, so the warp-collective TMEM accesses stay convergent.
        auto wait_warp = [&](uint64_t *bb, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bb, par, a.err));
        };
        for (int t = 0; t < nkt; ++t) {
            const int b = t & 1;
            if (!wait_warp(&B.s_full[b], (t >> 1) & 1)) {
                atomicExch(s_abort, 1);
                break;
            }
            tc_fence_after();
            float x[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) tmem_ld32(tmem + lane_base + b * kBN + c * 32, x + c * 32);
            tc_fence_before();
            mbar_arrive(&B.s_free[b]);

            const int lim = lim_abs - t * kBN;  // columns < lim are visible to this row
            if (lim < kBN) {
#pragma unroll
                for (int j = 0; j < kBN; ++j)
                    if (j >= lim) x[j] = -INFINITY;
            }
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = x[i];
#pragma unroll
            for (int j = 8; j < kBN; ++j) mx8[j & 7] = fmaxf(mx8[j & 7], x[j]);
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float m_tile = mx * sl;
            const float m_new = fmaxf(m_run, m_tile);
            if (t == 0) {
                m_run = m_new;
            } else {
                // Move the running max (and rescale O) only when it grew by
                // more than 8 in log2 units somewhere in the warp; TMEM
                // access is warp-collective.
                const bool want = m_new > m_run + 8.f;
                if (__any_sync(0xffffffffu, want)) {
                    const float alpha = fast_exp2(m_run - m_new);
                    if (!wait_warp(&B.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1)) {
                        atomicExch(s_abort, 1);
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tmem_o + lane_base + c * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(tmem_o + lane_base + c * 32, o);
                    }
                    l_run *= alpha;
                    m_run = m_new;
                }
            }
            const float mu = m_run == -INFINITY ? 0.f : m_run;
            if (t >= 2 && !wait_warp(&B.pv_done[b], ((t - 2) >> 1) & 1)) {
                atomicExch(s_abort, 1);
                break;
            }
            uint8_t *pb = smem + C::kPOff + b * C::kPBytes;
            float lsum = 0.f;
#pragma unroll
            for (int jj = 0; jj < kBN / 8; ++jj) {
                float p8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) p8[e] = fast_exp2(fmaf(x[jj * 8 + e], sl, -mu));
                const uint4 pk = make_uint4(pack_bf16x2(p8[0], p8[1]), pack_bf16x2(p8[2], p8[3]),
                                            pack_bf16x2(p8[4], p8[5]), pack_bf16x2(p8[6], p8[7]));
                // Row sums of the same bf16-rounded weights that multiply V.
                lsum += (bf16x2_sum(pk.x) + bf16x2_sum(pk.y)) + (bf16x2_sum(pk.z) + bf16x2_sum(pk.w));
                const int hf = jj >> 3, c = jj & 7;
                *reinterpret_cast<uint4 *>(pb + hf * kTileHalf + r * 128 + ((c ^ (r & 7)) << 4)) = pk;
            }
            l_run += lsum;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&B.p_full[b]);
        }
        // --------------------------------------------------------- epilogue --
        const bool aborted = __any_sync(0xffffffffu, *(volatile int *)s_abort != 0);
        if (!aborted && wait_warp(&B.pv_done[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1)) {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            __nv_bfloat16 *orow = a.out + ((size_t)(row0 + q0 + r) * a.num_q_heads + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(tmem_o + lane_base + c * 32, o);
                if (r < rows) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        const uint4 pk = make_uint4(pack_bf16x2(o[i] * inv, o[i + 1] * inv),
                                                    pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv),
                                                    pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv),
                                                    pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv));
                        *reinterpret_cast<uint4 *>(orow + c * 32 + i) = pk;
                    }
                }
            }
        } else {
            atomicExch(s_abort, 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int BS, bool PAGED>
cudaError_t launch_prefill_t(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const PrefillArgs &a, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, BS, PAGED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(a.num_q_tiles, a.num_q_heads, a.num_seqs);
    prefill_tc_kernel<D, BS, PAGED><<<grid, kThreads, C::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const PrefillArgs &a, int head_dim, int block_size, cudaStream_t stream) {
    const bool paged = a.block_table != nullptr;
#define PA_PRE(D, BS)                                                                        \
    if (head_dim == D && block_size == BS)                                                   \
        return paged ? launch_prefill_t<D, BS, true>(tm_q, tm_k, tm_v, a, stream)            \
                     : launch_prefill_t<D, 16, false>(tm_q, tm_k, tm_v, a, stream);
    PA_PRE(128, 16)
    PA_PRE(128, 32)
    PA_PRE(64, 16)
    PA_PRE(64, 32)
#undef PA_PRE
    return cudaErrorInvalidValue;
}

}  // namespace pa
