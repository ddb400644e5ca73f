// kv_append.cu -- scatter a step's new K/V rows into the paged block pool,
// and the optional index-checking pass of validation mode.
//
// The router's block allocator owns the blocks (TGI architecture wiki,
// data-sketchers.com, section "The Router"); the model server only writes
// each new token's key and value into the slot it was given:
//     k_pool[slot / B][h][slot % B][:] = k_new[i][h][:]   (v alike)
// slot < 0 is padding.  A pure bit copy: 16-byte vector loads and stores,
// consecutive threads on consecutive 16-byte pieces of one (token, head) row,
// so both the read of k_new and the write into the pool are coalesced.
// (Decode steps can instead append their rows in the decode's planning
// launch: pa_decode_append.)
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

// Each thread moves kAppendU 16-byte pieces of K and of V per pass of a
// grid-stride loop; the loads of a pass (the pieces and their slots) are all
// issued before any of them is used, and the pieces of one thread are a CTA
// width apart, so every load and store instruction of a warp covers 512
// contiguous bytes.  32-bit index arithmetic (the host checks that
// T * Hkv * d / 8 fits).
constexpr int kAppendU = 2;

template <int VPR>  // 16-byte pieces per row: d / 8
__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     const int32_t *__restrict__ slot_mapping, int num_vec, int num_kv_heads, int block_size,
                     long long num_slots, uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, int *err,
                     int check_err_first) {
    // A kernel launched after this one as a programmatic dependent (the
    // prefill) may be placed now; it waits for this grid before reading.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (check_err_first && *(volatile int *)err != 0) return;
    const int step = gridDim.x * (256 * kAppendU);
    for (int base = blockIdx.x * (256 * kAppendU) + threadIdx.x; base < num_vec; base += step) {
        uint4 kv[kAppendU], vv[kAppendU];
        int slot[kAppendU], th[kAppendU];
#pragma unroll
        for (int u = 0; u < kAppendU; ++u) {
            const int idx = base + u * 256;
            slot[u] = -1;
            if (idx < num_vec) {
                th[u] = idx / VPR;  // token * Hkv + head
                slot[u] = __ldg(slot_mapping + th[u] / num_kv_heads);
                kv[u] = __ldg(k_new + idx);
                vv[u] = __ldg(v_new + idx);
            }
        }
#pragma unroll
        for (int u = 0; u < kAppendU; ++u) {
            const int sl = slot[u];
            if (sl < 0) continue;
            if ((long long)sl >= num_slots) {
                set_error(err, PA_ERR_BAD_INDEX);
                continue;
            }
            const int idx = base + u * 256;
            const int tok = th[u] / num_kv_heads, h = th[u] - tok * num_kv_heads;
            const int blk = sl / block_size, off = sl - blk * block_size;
            const long long dst = (((long long)blk * num_kv_heads + h) * block_size + off) * VPR + (idx % VPR);
            k_pool[dst] = kv[u];
            v_pool[dst] = vv[u];
        }
    }
}

// fp8 cache: element e of KV head h is stored as the e4m3 code of
// x / scale[h] (IEEE float division, then nearest-even with saturation at
// +-448).  One thread per 16 codes (32 bytes of bf16 in, 16 bytes out).
__global__ void __launch_bounds__(256)
    kv_append_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                         const int32_t *__restrict__ slot_mapping, long long num_vec, int vec_per_row,
                         int num_kv_heads, int block_size, long long num_slots, const float *__restrict__ k_scale,
                         const float *__restrict__ v_scale, uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                         int *err, int check_err_first) {
    if (check_err_first && *(volatile int *)err != 0) return;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < num_vec; idx += stride) {
        const int j = (int)(idx % vec_per_row);  // 16-code piece within the row
        const long long th = idx / vec_per_row;  // token * Hkv + head
        const int h = (int)(th % num_kv_heads);
        const long long tok = th / num_kv_heads;
        const int slot = __ldg(slot_mapping + tok);
        if (slot < 0) continue;
        if ((long long)slot >= num_slots) {
            set_error(err, PA_ERR_BAD_INDEX);
            continue;
        }
        const long long blk = slot / block_size, off = slot % block_size;
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * vec_per_row + j;
        const float ks = __ldg(k_scale + h), vs = __ldg(v_scale + h);
        auto quant = [](const uint4 *src, long long at, float sc) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint4 x = __ldg(src + 2 * at + q);
                const uint32_t in[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int k = 0; k < 4; k += 2) {
                    const float2 a = bf16x2_unpack(in[k]), b = bf16x2_unpack(in[k + 1]);
                    const uint32_t lo = f32x2_to_e4m3x2(a.x / sc, a.y / sc);
                    const uint32_t hi = f32x2_to_e4m3x2(b.x / sc, b.y / sc);
                    w[2 * q + k / 2] = lo | (hi << 16);
                }
            }
            return make_uint4(w[0], w[1], w[2], w[3]);
        };
        k_pool[dst] = quant(k_new, idx, ks);
        v_pool[dst] = quant(v_new, idx, vs);
    }
}

// Validation mode: every index the kernels of one call will read is checked
// here first; a bad one sets the error word (PA_ERR_BAD_INDEX) and the
// call's other kernels, launched with check_err_first, return untouched.
__global__ void __launch_bounds__(256) index_check_kernel(const CheckArgs a) {
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    const int nthr = gridDim.x * blockDim.x;
    const long long num_slots = (long long)a.num_blocks * a.block_size;
    if (a.slot_mapping)
        for (int i = tid; i < a.num_tokens; i += nthr) {
            const int sl = a.slot_mapping[i];
            if (sl >= 0 && (long long)sl >= num_slots) set_error(a.err, PA_ERR_BAD_INDEX);
        }
    for (int s = tid; s < a.num_seqs; s += nthr) {
        int L = -1;
        if (a.seq_lens) {
            L = a.seq_lens[s];
            if (L < 0 || L > a.max_seq_len) {
                set_error(a.err, PA_ERR_BAD_INDEX);
                continue;
            }
        }
        if (a.cu_seqlens) {
            if (s < a.decode_rows && (a.cu_seqlens[s] != s || a.cu_seqlens[s + 1] != s + 1)) {
                set_error(a.err, PA_ERR_BAD_INDEX);
                continue;
            }
            const int n = a.cu_seqlens[s + 1] - a.cu_seqlens[s];
            const int p0 = a.prefix_lens ? a.prefix_lens[s] : (a.seq_lens ? L - n : 0);
            if (n < 0 || n > a.max_q_len || p0 < 0) {
                set_error(a.err, PA_ERR_BAD_INDEX);
                continue;
            }
            if (!a.seq_lens) L = p0 + n;
        }
        if (a.block_table && L >= 0) {
            const int nb = (L + a.block_size - 1) / a.block_size;
            if (nb > a.max_blocks) {
                set_error(a.err, PA_ERR_BAD_INDEX);
                continue;
            }
            for (int b = 0; b < nb; ++b) {
                const int blk = a.block_table[(size_t)s * a.max_blocks + b];
                if (blk < 0 || blk >= a.num_blocks) set_error(a.err, PA_ERR_BAD_INDEX);
            }
        }
    }
}

}  // namespace

cudaError_t launch_kv_append(const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new,
                             const int32_t *slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int num_blocks, __nv_bfloat16 *k_pool,
                             __nv_bfloat16 *v_pool, int *err, int check_err_first, int num_sms,
                             cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const long long nv = (long long)num_tokens * num_kv_heads * (head_dim / 8);
    if (nv > 0x7fffffffLL - 256LL * kAppendU) return cudaErrorInvalidValue;
    const int num_vec = (int)nv;
    // Up to 8 CTAs of 256 threads per SM; larger steps loop (grid stride).
    const unsigned blocks = (unsigned)std::min<long long>((num_vec + 256 * kAppendU - 1) / (256 * kAppendU),
                                                          8LL * std::max(num_sms, 1));
    const long long slots = (long long)num_blocks * block_size;
    auto *kp = reinterpret_cast<uint4 *>(k_pool);
    auto *vp = reinterpret_cast<uint4 *>(v_pool);
    auto *kn = reinterpret_cast<const uint4 *>(k_new);
    auto *vn = reinterpret_cast<const uint4 *>(v_new);
    if (head_dim == 128)
        kv_append_kernel<16><<<blocks, 256, 0, stream>>>(kn, vn, slot_mapping, num_vec, num_kv_heads, block_size,
                                                         slots, kp, vp, err, check_err_first);
    else
        kv_append_kernel<8><<<blocks, 256, 0, stream>>>(kn, vn, slot_mapping, num_vec, num_kv_heads, block_size,
                                                        slots, kp, vp, err, check_err_first);
    return cudaGetLastError();
}

cudaError_t launch_kv_append_fp8(const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new,
                                 const int32_t *slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, const float *k_scale, const float *v_scale,
                                 uint8_t *k_pool, uint8_t *v_pool, int *err, int check_err_first,
                                 cudaStream_t stream) {
    const int vec_per_row = head_dim / 16;  // 16 codes per output vector
    const long long num_vec = (long long)num_tokens * num_kv_heads * vec_per_row;
    if (num_vec == 0) return cudaSuccess;
    const int threads = 256;
    long long blocks = (num_vec + threads - 1) / threads;
    if (blocks > 65535LL * 4) blocks = 65535LL * 4;
    kv_append_fp8_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), slot_mapping, num_vec,
        vec_per_row, num_kv_heads, block_size, (long long)num_blocks * block_size, k_scale, v_scale,
        reinterpret_cast<uint4 *>(k_pool), reinterpret_cast<uint4 *>(v_pool), err, check_err_first);
    return cudaGetLastError();
}

cudaError_t launch_index_check(const CheckArgs &a, cudaStream_t stream) {
    const int work = a.num_tokens > a.num_seqs ? a.num_tokens : a.num_seqs;
    int blocks = (work + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    index_check_kernel<<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
