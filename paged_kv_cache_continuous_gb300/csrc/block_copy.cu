// block_copy.cu -- copy whole KV blocks between pools: inside the GPU for
// copy-on-fork and migration, between the GPU and a pinned host pool for
// swapping.  The pages' server keeps a GPU region and a CPU region for the KV
// cache (Blitzscale docs, section "CacheManager") and moves batches' caches
// between replicas, freeing the source blocks afterwards (section
// "migration_queue"):
//     dst_pool[dst_ids[i]] = src_pool[src_ids[i]]   (K and V, every KV head)
// In the HND pool layout one block is one contiguous Hkv * B * d * 2-byte
// chunk, so a copy is a plain 16-byte-vector stream; a pool in pinned host
// memory is read or written by the GPU at the same address (over NVLink-C2C
// on a Grace host).
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

// blockIdx.y walks the copy pairs, blockIdx.x the 16-byte vectors of a block.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const uint4 *__restrict__ src_k, const uint4 *__restrict__ src_v, uint4 *__restrict__ dst_k,
                       uint4 *__restrict__ dst_v, const int32_t *__restrict__ src_ids,
                       const int32_t *__restrict__ dst_ids, int num_pairs, long long vec_per_block,
                       int src_blocks, int dst_blocks, int *err, int check_err_first) {
    if (check_err_first && *(volatile int *)err != 0) return;
    const long long step = (long long)gridDim.x * blockDim.x;
    for (int i = blockIdx.y; i < num_pairs; i += gridDim.y) {
        const int s = __ldg(src_ids + i), d = __ldg(dst_ids + i);
        if ((unsigned)s >= (unsigned)src_blocks || (unsigned)d >= (unsigned)dst_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, PA_ERR_BAD_INDEX);
            continue;  // never dereference an out-of-range block
        }
        const uint4 *sk = src_k + (long long)s * vec_per_block, *sv = src_v + (long long)s * vec_per_block;
        uint4 *dk = dst_k + (long long)d * vec_per_block, *dv = dst_v + (long long)d * vec_per_block;
        long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
        // two vectors of each pool in flight per thread
        for (; j + step < vec_per_block; j += 2 * step) {
            const uint4 k0 = sk[j], k1 = sk[j + step], v0 = sv[j], v1 = sv[j + step];
            dk[j] = k0;
            dk[j + step] = k1;
            dv[j] = v0;
            dv[j + step] = v1;
        }
        if (j < vec_per_block) {
            const uint4 k0 = sk[j], v0 = sv[j];
            dk[j] = k0;
            dv[j] = v0;
        }
    }
}

}  // namespace

cudaError_t launch_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int32_t *src_ids, const int32_t *dst_ids, int num_pairs,
                               long long block_bytes, int src_blocks, int dst_blocks, int num_sms, int *err,
                               int check_err_first, cudaStream_t stream) {
    const long long vec = block_bytes / 16;
    const int threads = 256;
    const int gx = (int)std::min<long long>((vec + 2LL * threads - 1) / (2LL * threads), 16);
    const int gy = std::min(num_pairs, std::max(1, (num_sms * 8) / gx));
    copy_blocks_kernel<<<dim3(gx, std::min(gy, 65535)), threads, 0, stream>>>(
        static_cast<const uint4 *>(src_k), static_cast<const uint4 *>(src_v), static_cast<uint4 *>(dst_k),
        static_cast<uint4 *>(dst_v), src_ids, dst_ids, num_pairs, vec, src_blocks, dst_blocks, err,
        check_err_first);
    return cudaGetLastError();
}

}  // namespace pa
