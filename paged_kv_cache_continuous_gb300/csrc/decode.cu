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
//  * One CTA per (split c, KV head g, sequence s).  A split covers
//    `split_tokens` consecutive tokens, i.e. whole KV blocks.
//  * A producer warp streams the split's blocks into an 8 (B=16) or
//    4 (B=32) stage shared-memory ring with TMA tensor loads (128-byte
//    swizzle), one mbarrier pair per stage.  Each block of one KV head is one
//    contiguous B x d bf16 chunk of the pool, so a stage is 2 (K, V) x d/64
//    boxes of B rows x 128 bytes.  Block ids are range-checked before use.
//  * Four consumer warps take the stages round-robin.  Each warp computes the
//    scores of the G query heads of this KV head against 16 keys with
//    m16n8k16 tensor-core MMAs (rows = query heads, padded to 16; the G
//    heads share every K/V byte read), keeps its own online-softmax state
//    with quad shuffles, and accumulates P.V with the same MMA shape.  The
//    tensor-core dot products keep the FP32 pipe free: with G = 8 a CUDA-core
//    dot product would need ~2 G d FMAs per key, as much FP32 issue as the
//    HBM stream leaves room for.
//  * The warps' states are merged through shared memory; a sequence with a
//    single split writes bf16 output directly, otherwise the (max, sum, acc)
//    partials go to the workspace and decode_merge_kernel combines them.
#include <cuda.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

// FP8: the pools hold e4m3 codes (one byte per element) with one scale per KV
// head for K and for V.
template <int D, int BS, bool FP8 = false>
struct DecodeCfg {
    static constexpr int kEB = FP8 ? 1 : 2;                // bytes per pool element
    static constexpr int kBoxCols = 128 / kEB;             // elements per 128-byte TMA box row
    static constexpr int kHalves = D / kBoxCols;           // TMA boxes per row
    static constexpr int kHalfBytes = BS * 128;            // one box: BS rows x 128 B
    static constexpr int kKVBytes = kHalves * kHalfBytes;  // K (or V) of one block
    static constexpr int kStageBytes = 2 * kKVBytes;
    // multiple of kConsumerWarps; fp8 stages are half the bytes, so twice as
    // many keep the same bytes in flight
    static constexpr int kStages = ((BS == 16) ? 8 : 4) * (FP8 ? 2 : 1);
    static constexpr int kKSteps = D / 16;                 // QK^T k-steps
    static constexpr int kNTiles = D / 8;                  // PV n-tiles
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kScratchBytes = kConsumerWarps * 16 * D * 4 + kConsumerWarps * 16 * 8;
    static constexpr int kRegionBytes = kRingBytes > kScratchBytes ? kRingBytes : kScratchBytes;
    static constexpr int kSmemBytes = kRegionBytes + 2 * kStages * 8 + 16 + 1024;
};

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

template <int D, int BS, bool BIG_G, bool FP8>
__global__ void __launch_bounds__(kThreads, 3)
    decode_splitk_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using C = DecodeCfg<D, BS, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kRegionBytes);
    uint64_t *empty = full + C::kStages;
    int *s_abort = reinterpret_cast<int *>(empty + C::kStages);

    const int c = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (a.check_err_first && *(volatile int *)a.err != 0) return;
    const int L = a.seq_lens[s];
    if (L < 0 || L > a.max_seq_len || (L + BS - 1) / BS > a.max_blocks) {
        if (c == 0 && threadIdx.x == 0) set_error(a.err, PA_ERR_BAD_INDEX);
        return;
    }
    const int nsplit = L > 0 ? (L + a.split_tokens - 1) / a.split_tokens : 1;
    if (c >= nsplit) return;
    const int t0 = c * a.split_tokens;
    const int t1 = min(L, t0 + a.split_tokens);
    const int nblk = (t1 - t0 + BS - 1) / BS;  // t0 is block aligned
    const int b0 = t0 / BS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        *s_abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer --
    if (warp == kConsumerWarps) {
        const int32_t *bt = a.block_table + (size_t)s * a.max_blocks + b0;
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        // One lane per stage: lane l fills stage l with blocks l, l + kStages,
        // ..., each as soon as the consumers have freed it, independently of
        // the other lanes, so the TMA issue of a block overlaps its neighbours'.
        constexpr int kLanes = C::kStages;
        static_assert(kLanes <= 32, "one producer lane per stage");
        int last = -1;  // the last block this lane issued (into stage `lane`)
        bool good = true;
        if (lane < kLanes) {
            for (int i = lane; i < nblk; i += kLanes) {
                int32_t blk = bt[i];
                if ((unsigned)blk >= (unsigned)a.num_blocks) {
                    set_error(a.err, PA_ERR_BAD_INDEX);
                    blk = 0;  // never dereference an out-of-range block
                }
                if (i >= C::kStages && !mbar_wait(&empty[lane], ((i / C::kStages) - 1) & 1, a.err)) {
                    good = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[lane], C::kStageBytes);
                last = i;
                uint8_t *sk = smem + lane * C::kStageBytes;
                uint8_t *sv = sk + C::kKVBytes;
                const int row = (blk * a.num_kv_heads + g) * BS;
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    tma_load_2d(sk + hf * C::kHalfBytes, &tm_k, &full[lane], hf * C::kBoxCols, row);
                    tma_load_2d(sv + hf * C::kHalfBytes, &tm_v, &full[lane], hf * C::kBoxCols, row);
                }
            }
        }
        if (!__all_sync(0xffffffffu, good) && lane == 0) atomicExch(s_abort, 1);
        // Drain: every copy this CTA issued has landed before it may exit (a
        // stage's earlier blocks were consumed before it was refilled).
        if (last >= 0) mbar_wait(&full[lane], (last / C::kStages) & 1, a.err);
        return;
    }

    // ----------------------------------------------------------- consumers --
    const int G = a.group;
    const int r0 = lane >> 2;         // MMA row (query head within the group)
    const int cq = (lane & 3) * 2;    // first of the lane's two columns
    const __nv_bfloat16 *qg = a.q + ((size_t)s * a.num_q_heads + (size_t)g * G) * D;

    uint32_t qa[C::kKSteps][4];
    if (FP8) {
        // fp16 A fragments with the k-step's 16 columns permuted to match the
        // byte order ldmatrix gives the fp8 keys: MMA columns 2c, 2c+1 hold
        // d = 4c, 4c+1 and columns 2c+8, 2c+9 hold d = 4c+2, 4c+3 (c = lane % 4).
        const int c4 = (lane & 3) * 4;
        auto qf = [&](int row, int col) {
            return row < G ? pack_f16x2(__bfloat162float(qg[row * D + col]), __bfloat162float(qg[row * D + col + 1]))
                           : 0u;
        };
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
            qa[ks][0] = qf(r0, ks * 16 + c4);
            qa[ks][2] = qf(r0, ks * 16 + c4 + 2);
            qa[ks][1] = BIG_G ? qf(r0 + 8, ks * 16 + c4) : 0u;
            qa[ks][3] = BIG_G ? qf(r0 + 8, ks * 16 + c4 + 2) : 0u;
        }
    } else
#pragma unroll
    for (int ks = 0; ks < C::kKSteps; ++ks) {
        qa[ks][0] = r0 < G ? ld_u32(qg + r0 * D + ks * 16 + cq) : 0u;
        qa[ks][2] = r0 < G ? ld_u32(qg + r0 * D + ks * 16 + 8 + cq) : 0u;
        if (BIG_G) {
            qa[ks][1] = r0 + 8 < G ? ld_u32(qg + (r0 + 8) * D + ks * 16 + cq) : 0u;
            qa[ks][3] = r0 + 8 < G ? ld_u32(qg + (r0 + 8) * D + ks * 16 + 8 + cq) : 0u;
        } else {
            qa[ks][1] = 0u;
            qa[ks][3] = 0u;
        }
    }

    float acc[C::kNTiles][4];
#pragma unroll
    for (int nt = 0; nt < C::kNTiles; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};  // rows r0, r0 + 8 (log2 units)
    float l_run[2] = {0.f, 0.f};              // this lane's share of the row sums
    const float sl = FP8 ? a.scale_log2 * a.k_scale[g] : a.scale_log2;

    for (int i = warp; i < nblk; i += kConsumerWarps) {
        const int st = i % C::kStages;
        if (!mbar_wait(&full[st], (i / C::kStages) & 1, a.err)) {
            atomicExch(s_abort, 1);
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
            for (int r = valid + (lane >> 3); r < BS; r += 4) {
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf)
                    *reinterpret_cast<uint4 *>(vz + hf * C::kHalfBytes + r * 128 + (lane & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
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
                    const uint32_t addr = sk + t * 128 + (((jj ^ (t & 7))) << 4);
                    uint32_t b00, b01, b10, b11;  // (keys 0-7, ks), (0-7, ks+1), (8-15, ks), (8-15, ks+1)
                    ldmatrix_x4(addr, b00, b01, b10, b11);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int ks = 2 * kp + u;
                        const uint32_t lo = u ? b01 : b00, hi = u ? b11 : b10;
                        mma_f16_16816(sacc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], e4m3x2_to_f16x2(lo),
                                      e4m3x2_to_f16x2(lo >> 16));
                        mma_f16_16816(sacc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], e4m3x2_to_f16x2(hi),
                                      e4m3x2_to_f16x2(hi >> 16));
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
#pragma unroll
                for (int nt = 0; nt < C::kNTiles; ++nt) {
                    acc[nt][rr * 2 + 0] *= alpha[rr];
                    acc[nt][rr * 2 + 1] *= alpha[rr];
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
                    const uint32_t addr = sv + t * 128 + (((jj ^ (t & 7))) << 4);
                    uint32_t v0, v1, v2, v3;  // (keys 0-7, chunk 2jp), (8-15, 2jp), (0-7, 2jp+1), (8-15, 2jp+1)
                    ldmatrix_x4_trans(addr, v0, v1, v2, v3);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t lo = u ? v2 : v0, hi = u ? v3 : v1;
#pragma unroll
                        for (int par = 0; par < 2; ++par) {
                            const uint32_t sel = par ? 0x3131u : 0x2020u;  // bytes (1, 3) or (0, 2)
                            mma_f16_16816(acc[4 * jp + 2 * u + par], pa0, pa1, pa2, pa3,
                                          e4m3x2_to_f16x2(__byte_perm(lo, 0u, sel)),
                                          e4m3x2_to_f16x2(__byte_perm(hi, 0u, sel)));
                        }
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

    // ----------------------------------------- merge the four warps' states --
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
        l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
    }
    if (FP8) {
        const float vs = a.v_scale[g];
#pragma unroll
        for (int nt = 0; nt < C::kNTiles; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] *= vs;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    float *red_acc = reinterpret_cast<float *>(smem);                       // [W][16][D]
    float *red_ml = red_acc + kConsumerWarps * 16 * D;                      // [W][16][2]
#pragma unroll
    for (int rr = 0; rr < (BIG_G ? 2 : 1); ++rr) {
        const int row = r0 + rr * 8;
        float *dst = red_acc + (warp * 16 + row) * D;
#pragma unroll
        for (int nt = 0; nt < C::kNTiles; ++nt) {
            if (FP8) {
                const int d0 = 16 * (nt >> 1) + 4 * (lane & 3) + (nt & 1);
                dst[d0] = acc[nt][rr * 2 + 0];
                dst[d0 + 2] = acc[nt][rr * 2 + 1];
            } else {
                *reinterpret_cast<float2 *>(dst + nt * 8 + cq) = make_float2(acc[nt][rr * 2 + 0], acc[nt][rr * 2 + 1]);
            }
        }
        if ((lane & 3) == 0) {
            red_ml[(warp * 16 + row) * 2 + 0] = m_run[rr];
            red_ml[(warp * 16 + row) * 2 + 1] = l_run[rr];
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    if (*(volatile int *)s_abort) return;

    const int tid = threadIdx.x;  // 0 .. 127
    for (int idx = tid; idx < G * D; idx += kConsumerWarps * 32) {
        const int row = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_ml[(w * 16 + row) * 2]);
        float sum_l = 0.f, sum_a = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = red_ml[(w * 16 + row) * 2];
                const float f = fast_exp2(mw - M);  // 0 for a warp that saw no key
                sum_l += f * red_ml[(w * 16 + row) * 2 + 1];
                sum_a += f * red_acc[(w * 16 + row) * D + e];
            }
        }
        const int h = g * G + row;
        if (nsplit == 1) {
            const float o = sum_l > 0.f ? sum_a / sum_l : 0.f;
            a.out[((size_t)s * a.num_q_heads + h) * D + e] = __float2bfloat16_rn(o);
        } else {
            const size_t pi = ((size_t)s * a.num_q_heads + h) * a.max_splits + c;
            a.part_acc[pi * D + e] = sum_a;
            if (e == 0) {
                a.part_ml[pi * 2 + 0] = M;
                a.part_ml[pi * 2 + 1] = sum_l;
            }
        }
    }
}

// Combine the split partials of every (sequence, query head) with more than
// one split: out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * 4 + warp, s = blockIdx.y;
    if (h >= a.num_q_heads) return;
    if (a.check_err_first && *(volatile int *)a.err != 0) return;
    const int L = a.seq_lens[s];
    if (L < 0 || L > a.max_seq_len) return;
    const int nsplit = L > 0 ? (L + a.split_tokens - 1) / a.split_tokens : 1;
    if (nsplit <= 1) return;
    const size_t p0 = ((size_t)s * a.num_q_heads + h) * a.max_splits;
    const float *ml = a.part_ml + p0 * 2;
    float M = -INFINITY;
    for (int c = lane; c < nsplit; c += 32) M = fmaxf(M, ml[c * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    constexpr int E = D / 32;  // elements per lane
    float accv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) accv[e] = 0.f;
    float lsum = 0.f;
    for (int c = 0; c < nsplit; ++c) {
        const float f = fast_exp2(ml[c * 2] - M);
        lsum += f * ml[c * 2 + 1];
        const float *pa = a.part_acc + (p0 + c) * D + lane * E;
        if constexpr (E == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(pa);
            accv[0] += f * v.x;
            accv[1] += f * v.y;
            accv[2] += f * v.z;
            accv[3] += f * v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2 *>(pa);
            accv[0] += f * v.x;
            accv[1] += f * v.y;
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __nv_bfloat16 *o = a.out + ((size_t)s * a.num_q_heads + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<__nv_bfloat162 *>(o + e) = __floats2bfloat162_rn(accv[e] * inv, accv[e + 1] * inv);
}

template <int D, int BS, bool BIG_G, bool FP8>
cudaError_t launch_decode_t(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeArgs &a,
                            cudaStream_t stream) {
    using C = DecodeCfg<D, BS, FP8>;
    static std::atomic<unsigned long long> opted{0};
    cudaError_t e0 = opt_in_smem(reinterpret_cast<const void *>(decode_splitk_kernel<D, BS, BIG_G, FP8>),
                                 C::kSmemBytes, opted);
    if (e0 != cudaSuccess) return e0;
    dim3 grid(a.max_splits, a.num_kv_heads, a.num_seqs);
    decode_splitk_kernel<D, BS, BIG_G, FP8><<<grid, kThreads, C::kSmemBytes, stream>>>(tm_k, tm_v, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.max_splits <= 1) return e;
    dim3 mgrid((a.num_q_heads + 3) / 4, a.num_seqs);
    decode_merge_kernel<D><<<mgrid, 128, 0, stream>>>(a);
    return cudaGetLastError();
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

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_splits) {
    if (max_splits <= 1) return 0;
    const size_t n = (size_t)num_seqs * num_q_heads * max_splits;
    return n * head_dim * sizeof(float) + n * 2 * sizeof(float);
}

cudaError_t launch_decode(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeArgs &a,
                          int head_dim, int block_size, cudaStream_t stream, bool fp8) {
    const bool big = a.group > 8;
#define PA_DEC(D, BS, F8)                                                              \
    if (head_dim == D && block_size == BS && fp8 == F8)                                \
        return big ? launch_decode_t<D, BS, true, F8>(tm_k, tm_v, a, stream)           \
                   : launch_decode_t<D, BS, false, F8>(tm_k, tm_v, a, stream);
    PA_DEC(128, 16, false)
    PA_DEC(128, 32, false)
    PA_DEC(64, 16, false)
    PA_DEC(64, 32, false)
    PA_DEC(128, 16, true)
    PA_DEC(128, 32, true)
#undef PA_DEC
    return cudaErrorInvalidValue;
}

}  // namespace pa
