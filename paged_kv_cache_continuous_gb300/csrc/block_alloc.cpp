// block_alloc.cpp -- the host block allocator declared in include/pa_alloc.h.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "../../include/pa_alloc.h"

struct pa_block_allocator {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::unordered_map<int64_t, std::vector<int32_t>> tables;
};

extern "C" {

pa_block_allocator *pa_alloc_create(int num_blocks, int block_size, const int32_t *initial_order) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pa_block_allocator *a = new (std::nothrow) pa_block_allocator;
    if (!a) return nullptr;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    std::vector<char> seen(num_blocks, 0);
    a->free_stack.resize(num_blocks);
    for (int i = 0; i < num_blocks; ++i) {
        const int32_t b = initial_order ? initial_order[i] : i;
        if (b < 0 || b >= num_blocks || seen[b]) {
            delete a;
            return nullptr;
        }
        seen[b] = 1;
        a->free_stack[num_blocks - 1 - i] = b;  // order[0] on top
    }
    return a;
}

void pa_alloc_destroy(pa_block_allocator *a) { delete a; }

int pa_alloc_ensure(pa_block_allocator *a, int64_t seq_id, int num_tokens) {
    if (!a || num_tokens < 0) return PA_ERR_INVALID_ARG;
    std::vector<int32_t> &t = a->tables[seq_id];
    const long long want = ((long long)num_tokens + a->block_size - 1) / a->block_size;
    const long long need = want - (long long)t.size();
    if (need <= 0) return PA_OK;
    if (need > (long long)a->free_stack.size()) {
        if (t.empty()) a->tables.erase(seq_id);
        return PA_ERR_NO_BLOCKS;
    }
    for (long long i = 0; i < need; ++i) {
        t.push_back(a->free_stack.back());
        a->free_stack.pop_back();
    }
    return PA_OK;
}

int pa_alloc_release(pa_block_allocator *a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->tables.find(seq_id);
    if (it == a->tables.end()) return PA_ERR_INVALID_ARG;
    for (int32_t b : it->second) a->free_stack.push_back(b);
    a->tables.erase(it);
    return PA_OK;
}

int pa_alloc_num_free(const pa_block_allocator *a) { return a ? (int)a->free_stack.size() : 0; }

int pa_alloc_num_blocks_of(const pa_block_allocator *a, int64_t seq_id) {
    if (!a) return 0;
    auto it = a->tables.find(seq_id);
    return it == a->tables.end() ? 0 : (int)it->second.size();
}

int pa_alloc_block_table(const pa_block_allocator *a, const int64_t *seq_ids, int num_seqs, int width,
                         int32_t fill, int32_t *table_out) {
    if (!a || num_seqs < 0 || width <= 0 || (num_seqs > 0 && (!seq_ids || !table_out)))
        return PA_ERR_INVALID_ARG;
    for (int r = 0; r < num_seqs; ++r) {
        auto it = a->tables.find(seq_ids[r]);
        if (it == a->tables.end() || (int)it->second.size() > width) return PA_ERR_INVALID_ARG;
        int32_t *row = table_out + (size_t)r * width;
        const int n = (int)it->second.size();
        for (int j = 0; j < width; ++j) row[j] = j < n ? it->second[j] : fill;
    }
    return PA_OK;
}

int pa_alloc_slot_mapping(const pa_block_allocator *a, const int64_t *seq_ids, const int32_t *n_new,
                          const int32_t *total_after, int num_seqs, int32_t *slots_out) {
    if (!a || num_seqs < 0 || (num_seqs > 0 && (!seq_ids || !n_new || !total_after || !slots_out)))
        return PA_ERR_INVALID_ARG;
    size_t k = 0;
    for (int r = 0; r < num_seqs; ++r) {
        auto it = a->tables.find(seq_ids[r]);
        if (it == a->tables.end() || n_new[r] < 0 || total_after[r] < n_new[r]) return PA_ERR_INVALID_ARG;
        const std::vector<int32_t> &t = it->second;
        for (int j = 0; j < n_new[r]; ++j) {
            const int p = total_after[r] - n_new[r] + j;
            const size_t bi = (size_t)(p / a->block_size);
            if (bi >= t.size()) return PA_ERR_INVALID_ARG;
            slots_out[k++] = t[bi] * a->block_size + p % a->block_size;
        }
    }
    return PA_OK;
}

}  // extern "C"
