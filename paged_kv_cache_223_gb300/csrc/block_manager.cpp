// block_manager.cpp -- host-side physical block allocator of a paged KV pool: the shared free
// pool, reference counts for blocks named by several block tables, copy-on-write of a shared
// block before it is written, and appending tokens to a sequence (a new block each time the
// sequence crosses a block boundary).
//
// (yangyu.win blog #54, section 5 question 2: a sequence that grows by one block takes one new
// page from the free block pool; parallel samples share the prompt's pages with a reference
// count; on divergence, copy-on-write gives the diverging part its own page. itimpress.au
// "PagedAttention, ...", section 1: requests sharing a prompt point at the same physical blocks.)
#include <mutex>
#include <unordered_map>
#include <vector>

#include "pagedattn.h"

struct pa_block_allocator {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> ref;     // reference count per physical block (0 = free)
    std::vector<int32_t> free_ids;  // the free pool, used as a stack
    std::mutex mu;
};

namespace {

bool valid_live(const pa_block_allocator *a, int32_t id) {
    return id >= 0 && id < a->num_blocks && a->ref[id] > 0;
}

int32_t take(pa_block_allocator *a) {
    const int32_t id = a->free_ids.back();
    a->free_ids.pop_back();
    a->ref[id] = 1;
    return id;
}

}  // namespace

extern "C" {

pa_status pa_allocator_create(int32_t num_blocks, int32_t block_size, pa_block_allocator **out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
    pa_block_allocator *a = new pa_block_allocator();
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    a->free_ids.resize(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) a->free_ids[i] = num_blocks - 1 - i;   // block 0 is taken first
    *out = a;
    return PA_OK;
}

void pa_allocator_destroy(pa_block_allocator *a) { delete a; }

int32_t pa_allocator_num_free(pa_block_allocator *a) {
    if (!a) return -1;
    std::lock_guard<std::mutex> lk(a->mu);
    return (int32_t)a->free_ids.size();
}

int32_t pa_allocator_ref_count(pa_block_allocator *a, int32_t id) {
    if (!a || id < 0 || id >= a->num_blocks) return -1;
    std::lock_guard<std::mutex> lk(a->mu);
    return a->ref[id];
}

pa_status pa_allocator_alloc(pa_block_allocator *a, int32_t n, int32_t *ids) {
    if (!a || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(a->mu);
    if ((size_t)n > a->free_ids.size()) return PA_ERR_OOM;
    for (int32_t i = 0; i < n; ++i) ids[i] = take(a);
    return PA_OK;
}

pa_status pa_allocator_fork(pa_block_allocator *a, const int32_t *ids, int32_t n) {
    if (!a || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(a->mu);
    for (int32_t i = 0; i < n; ++i)
        if (!valid_live(a, ids[i])) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) ++a->ref[ids[i]];
    return PA_OK;
}

pa_status pa_allocator_free(pa_block_allocator *a, const int32_t *ids, int32_t n) {
    if (!a || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(a->mu);
    std::unordered_map<int32_t, int32_t> drops;   // an id may appear more than once
    for (int32_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= a->num_blocks) return PA_ERR_INVALID_ARG;
        if (++drops[ids[i]] > a->ref[ids[i]]) return PA_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i)
        if (--a->ref[ids[i]] == 0) a->free_ids.push_back(ids[i]);
    return PA_OK;
}

pa_status pa_allocator_cow(pa_block_allocator *a, int32_t id, int32_t *out_id, int32_t *copy) {
    if (!a || !out_id || !copy) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(a->mu);
    if (!valid_live(a, id)) return PA_ERR_INVALID_ARG;
    if (a->ref[id] == 1) {
        *out_id = id;
        *copy = 0;
        return PA_OK;
    }
    if (a->free_ids.empty()) return PA_ERR_OOM;
    --a->ref[id];
    *out_id = take(a);
    *copy = 1;
    return PA_OK;
}

pa_status pa_allocator_append(pa_block_allocator *a, int32_t *table_row, int32_t stride, int32_t *len,
                              int32_t n_new, int64_t *slots, int32_t *copy_pair, int32_t *n_copies) {
    if (!a || !table_row || !len || !slots || !copy_pair || !n_copies || n_new < 0 || stride < 1 || *len < 0)
        return PA_ERR_INVALID_ARG;
    const int32_t bs = a->block_size;
    const int64_t L0 = *len, L1 = L0 + n_new;
    if (L1 > (int64_t)stride * bs) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(a->mu);
    *n_copies = 0;
    if (n_new == 0) return PA_OK;
    const int64_t have = (L0 + bs - 1) / bs;              // blocks the table already holds
    const int64_t need = (L1 + bs - 1) / bs;
    for (int64_t j = 0; j < have; ++j)
        if (!valid_live(a, table_row[j])) return PA_ERR_INVALID_ARG;
    // the first new token lands in the partly filled last block, which must be private
    const bool cow = (L0 % bs) != 0 && a->ref[table_row[have - 1]] > 1;
    if ((size_t)(need - have + (cow ? 1 : 0)) > a->free_ids.size()) return PA_ERR_OOM;
    if (cow) {
        const int32_t old = table_row[have - 1];
        --a->ref[old];
        const int32_t fresh = take(a);
        table_row[have - 1] = fresh;
        copy_pair[0] = old;
        copy_pair[1] = fresh;
        *n_copies = 1;
    }
    for (int64_t j = have; j < need; ++j) table_row[j] = take(a);
    for (int64_t t = L0; t < L1; ++t) slots[t - L0] = (int64_t)table_row[t / bs] * bs + t % bs;
    *len = (int32_t)L1;
    return PA_OK;
}

}  // extern "C"
