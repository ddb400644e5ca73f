// rope.cu -- rotary position embedding of a step's new tokens, fused with the
// KV append: one pass over the new tokens rotates their queries (into q_out,
// which the decode / prefill kernels then read) and their keys (written
// straight into the pool slot), and copies their values.
//
// The pages name only the flashinfer build option that compiles its
// position-encoding modes in (Blitzscale docs, section "Build"); the rotation
// is the RoFormer one with the Llama / GPT-NeoX pairing: for a head vector x
// of length d at position p and i < d/2, with f_i = theta^(-2i/d),
//     y[i]       = x[i] cos(p f_i) - x[i + d/2] sin(p f_i)
//     y[i + d/2] = x[i + d/2] cos(p f_i) + x[i] sin(p f_i).
// The host gives each frequency as a 64-bit fixed-point fraction of a turn,
// f_i / (2 pi) (from its double value); p times it modulo 2^64 is the angle's
// part of a turn, exact in integer arithmetic, so cos / sin are taken (in
// float) of an angle in [-pi, pi) whatever the position, with no FP64 work;
// the rotation is float, rounded to bf16.
#include <cuda_bf16.h>

#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kThreads = 256;
constexpr int kTok = 2;    // tokens per CTA pass: their cos / sin first, then all their rows at once
                           // (two rather than four: 20.0 against 20.2 us for a 4096-token step)
constexpr int kItems = 4;  // work items a thread holds in registers at once

// Rotate eight pairs (i .. i+7 with i+d/2 .. i+d/2+7) of one head row: lo / hi
// are 8 bf16 each (16 bytes); cs holds (cos, sin) of the eight pairs.
__device__ __forceinline__ void rotate8(uint4 &lo, uint4 &hi, const float2 *cs) {
    __nv_bfloat162 *l = reinterpret_cast<__nv_bfloat162 *>(&lo);
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&hi);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 a = __bfloat1622float2(l[j]), b = __bfloat1622float2(h[j]);
        const float2 c0 = cs[2 * j], c1 = cs[2 * j + 1];  // (cos, sin) of pairs 2j, 2j+1
        const float y0 = fmaf(a.x, c0.x, -b.x * c0.y), y1 = fmaf(a.y, c1.x, -b.y * c1.y);
        const float z0 = fmaf(b.x, c0.x, a.x * c0.y), z1 = fmaf(b.y, c1.x, a.y * c1.y);
        l[j] = __floats2bfloat162_rn(y0, y1);
        h[j] = __floats2bfloat162_rn(z0, z1);
    }
}

__global__ void __launch_bounds__(kThreads)
    rope_append_kernel(const RopeArgs a, int tpc) {  // tpc <= kTok tokens per pass
    // (cos, sin) per token of the pass and pair i, at i + i / 8: a thread reads
    // the eight pairs of its 16-byte chunk, and the padding puts a warp's eight
    // chunks on distinct banks.
    __shared__ float2 cs[kTok][72];
    __shared__ int s_slot[kTok];     // the token's slot, or -1 if it is not appended (or skipped)
    __shared__ int s_pos_ok[kTok];
    // Under a programmatic dependent launch: the previous kernel's writes (the
    // inputs) are visible past this point.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (a.check_err_first && *(volatile int *)a.err != 0) return;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int d = a.head_dim, half = d / 2;
    const int cpr = half / 8;  // 16-byte chunks per half row
    const long long num_slots = (long long)a.num_blocks * a.block_size;
    for (int t0 = blockIdx.x * tpc; t0 < a.num_tokens; t0 += gridDim.x * tpc) {
        const int nt = min(tpc, a.num_tokens - t0);
        // Work items of the pass: one (token, head, chunk pair) each -- the
        // queries first, then the keys, then the values.
        const int nq = nt * a.num_q_heads * cpr, nk = nt * a.num_kv_heads * cpr;
        const int total = nq + 2 * nk;
        for (int b0 = 0; b0 < total; b0 += kThreads * kItems) {
            // Every load of the batch is issued before anything waits on one
            // (and, in a pass's first batch, before the tables are built).
            uint4 lo[kItems], hi[kItems];
            int meta[kItems];  // kind (0 q, 1 k, 2 v) | token << 2 | chunk << 4 | head << 8
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                const int e = b0 + j * kThreads + (int)threadIdx.x;
                meta[j] = -1;
                if (e < total) {
                    int kind, ee, heads;
                    if (e < nq) {
                        kind = 0, ee = e, heads = a.num_q_heads;
                    } else {
                        kind = e - nq < nk ? 1 : 2;
                        ee = e - nq - (kind == 2 ? nk : 0);
                        heads = a.num_kv_heads;
                    }
                    const int tt = ee / (heads * cpr), r = ee % (heads * cpr);
                    const int h = r / cpr, ch = r % cpr;
                    const __nv_bfloat16 *src = kind == 0 ? a.q : (kind == 1 ? a.k_new : a.v_new);
                    const size_t o = ((size_t)(t0 + tt) * heads + h) * d + ch * 8;
                    lo[j] = *reinterpret_cast<const uint4 *>(src + o);
                    hi[j] = *reinterpret_cast<const uint4 *>(src + o + half);
                    meta[j] = kind | (tt << 2) | (ch << 4) | (h << 8);
                }
            }
            if (b0 == 0) {
                __syncthreads();  // the previous pass's tables are no longer read
                for (int e = threadIdx.x; e < nt * half; e += kThreads) {
                    const int tt = e / half, i = e % half;
                    const int p = __ldg(a.positions + t0 + tt);
                    // p f_i in turns, modulo whole turns: exact integer arithmetic
                    // (no FP64, a slow pipe on this GPU); the top 32 bits read as a
                    // signed fraction of a turn give the angle in [-pi, pi).
                    const unsigned long long tr = (unsigned long long)(unsigned)max(p, 0) * a.turn[i];
                    const float ang = (float)(int)(unsigned)(tr >> 32) * 1.4629180792671596e-09f;  // 2 pi / 2^32
                    float sn, cn;
                    sincosf(ang, &sn, &cn);
                    cs[tt][i + (i >> 3)] = make_float2(cn, sn);
                    if (i == 0) {
                        const int sl = __ldg(a.slot_mapping + t0 + tt);
                        const bool pos_ok = p >= 0, slot_ok = (long long)sl < num_slots;
                        if (!pos_ok || !slot_ok) set_error(a.err, PA_ERR_BAD_INDEX);
                        s_pos_ok[tt] = pos_ok;
                        s_slot[tt] = (pos_ok && slot_ok) ? sl : -1;  // never write outside the pool
                    }
                }
                __syncthreads();
            }
            // Rotate the queries (into q_out) and keys (into their pool slot);
            // copy the values.
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                if (meta[j] < 0) continue;
                const int kind = meta[j] & 3, tt = (meta[j] >> 2) & 3, ch = (meta[j] >> 4) & 15, h = meta[j] >> 8;
                const int i = ch * 8;
                __nv_bfloat16 *dst;
                if (kind == 0) {
                    if (!s_pos_ok[tt]) continue;
                    rotate8(lo[j], hi[j], &cs[tt][i + ch]);
                    dst = a.q_out + ((size_t)(t0 + tt) * a.num_q_heads + h) * d + i;
                } else {
                    const int sl = s_slot[tt];
                    if (sl < 0) continue;
                    if (kind == 1) rotate8(lo[j], hi[j], &cs[tt][i + ch]);
                    const long long blk = sl / a.block_size, off = sl % a.block_size;
                    dst = (kind == 1 ? a.k_pool : a.v_pool) +
                          ((size_t)(blk * a.num_kv_heads + h) * a.block_size + off) * d + i;
                }
                *reinterpret_cast<uint4 *>(dst) = lo[j];
                *reinterpret_cast<uint4 *>(dst + half) = hi[j];
            }
        }
    }
}

}  // namespace

cudaError_t launch_rope_append(const RopeArgs &a, int num_sms, cudaStream_t stream) {
    // Small steps (a decode step's few tokens) take one token per pass, so that
    // they still spread over many SMs; large ones kTok.
    const int tpc = a.num_tokens >= num_sms * 8 ? kTok : 1;
    const int chunks = (a.num_tokens + tpc - 1) / tpc;
    const int blocks = std::max(1, std::min(chunks, num_sms * 8));
    // A programmatic dependent launch: the CTAs may be placed while the
    // previous kernel on the stream finishes; they wait for it before reading.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rope_append_kernel, a, tpc);
}

}  // namespace pa
