// Host block allocator for the paged KV pool.
//
// "TensorRT-LLM 深度实战" (chenxutan.com), §3.1 Paged KV Cache: free pages are kept in a
// list that starts as 0..n-1 and is consumed with pop() from its end; a sequence's page
// table lists its pages in the order they were taken; growth adds whole pages once the
// tokens outgrow the capacity; a finished sequence's pages go back to the end of the list
// in table order.  Out-of-memory is checked before anything is taken, so a failing call
// changes nothing (the page's sketch leaks pages popped before it runs dry).
//
// Block reuse (pnsm.cn TensorRT-LLM page, §3.1 KV缓存优化: enable_block_reuse; "TensorRT-LLM
// 推理加速实战" §8: KV Cache Reuse, enable_kv_cache_reuse, like prefix caching): a new sequence
// may share another sequence's full prefix blocks.  Every block carries a reference count; a
// shared prefix that ends inside a block gets a private copy of that block (copy on write), so
// later appends never write a shared block; a block rejoins the free list when its count drops
// to zero.
#include <cstring>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pkv_internal.h"

struct pkv_allocator {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_list;  // back() is handed out next
    std::vector<int32_t> refcnt;     // holders of each block; 0 = on the free list
    std::unordered_map<int64_t, std::vector<int32_t>> tables;
};

namespace pkv {

bool valid_block_size(int bs) { return bs >= 16 && bs <= 256 && (bs & (bs - 1)) == 0; }

pkv_allocator* allocator_new(int num_blocks, int block_size) {
    pkv_allocator* a = new (std::nothrow) pkv_allocator();
    if (!a) return nullptr;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    try {
        a->free_list.resize(num_blocks);
        a->refcnt.assign(num_blocks, 0);
    } catch (...) {
        delete a;
        return nullptr;
    }
    for (int i = 0; i < num_blocks; ++i) a->free_list[i] = i;
    return a;
}

void allocator_delete(pkv_allocator* a) { delete a; }

}  // namespace pkv

extern "C" {

pkv_status pkv_allocator_create(int num_blocks, int block_size, pkv_allocator** out) {
    if (!out || num_blocks < 1 || !pkv::valid_block_size(block_size)) return PKV_ERR_INVALID_ARG;
    pkv_allocator* a = pkv::allocator_new(num_blocks, block_size);
    if (!a) return PKV_ERR_OOM;
    *out = a;
    return PKV_OK;
}

pkv_status pkv_allocator_destroy(pkv_allocator* a) {
    if (!a) return PKV_ERR_INVALID_ARG;
    pkv::allocator_delete(a);
    return PKV_OK;
}

pkv_status pkv_allocator_set_free_order(pkv_allocator* a, const int32_t* order, int n) {
    if (!a || !order || n != a->num_blocks || !a->tables.empty()) return PKV_ERR_INVALID_ARG;
    std::vector<char> seen(n, 0);
    for (int i = 0; i < n; ++i) {
        if (order[i] < 0 || order[i] >= n || seen[order[i]]) return PKV_ERR_INVALID_ARG;
        seen[order[i]] = 1;
    }
    std::memcpy(a->free_list.data(), order, sizeof(int32_t) * (size_t)n);
    return PKV_OK;
}

// Seeded shuffle of the free list: Fisher-Yates in Durstenfeld's form (positions n-1 down to 1,
// each swapped with a uniformly chosen position at or below it), the k-th swap partner drawn
// from the k-th output of splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", 2014: state advanced by the golden-ratio increment, then the mix with
// shifts 30 / 27 / 31 and the two published multipliers).  A partner in [0, i] is the top 53 bits
// of the draw times i + 1, shifted down by 53 (multiply-shift, no modulo bias beyond 2^-53).
pkv_status pkv_allocator_shuffle_free_list(pkv_allocator* a, uint64_t seed) {
    if (!a) return PKV_ERR_INVALID_ARG;
    std::vector<int32_t>& f = a->free_list;
    uint64_t k = 0;
    for (size_t i = f.size(); i-- > 1;) {
        uint64_t z = seed + (k + 1) * 0x9E3779B97F4A7C15ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        ++k;
        const unsigned __int128 prod = (unsigned __int128)(z >> 11) * (unsigned __int128)(i + 1);
        const size_t j = (size_t)(prod >> 53);
        std::swap(f[i], f[j]);
    }
    return PKV_OK;
}

pkv_status pkv_seq_reserve(pkv_allocator* a, int64_t seq_id, int64_t n_tokens) {
    if (!a || n_tokens < 0) return PKV_ERR_INVALID_ARG;
    auto it = a->tables.find(seq_id);
    const int64_t held = it == a->tables.end() ? 0 : (int64_t)it->second.size();
    const int64_t bs = a->block_size;
    const int64_t want = (n_tokens + bs - 1) / bs;
    const int64_t extra = want > held ? want - held : 0;
    if (extra > (int64_t)a->free_list.size()) return PKV_ERR_OOM;
    std::vector<int32_t>& tbl = it == a->tables.end() ? a->tables[seq_id] : it->second;
    tbl.reserve((size_t)(held + extra));
    for (int64_t i = 0; i < extra; ++i) {
        tbl.push_back(a->free_list.back());
        a->refcnt[a->free_list.back()] = 1;
        a->free_list.pop_back();
    }
    return PKV_OK;
}

pkv_status pkv_seq_reserve_many(pkv_allocator* a, const int64_t* seq_ids, const int64_t* n_tokens, int64_t count,
                                int64_t* done) {
    if (!a || count < 0 || (count > 0 && (!seq_ids || !n_tokens))) return PKV_ERR_INVALID_ARG;
    int64_t i = 0;
    pkv_status st = PKV_OK;
    for (; i < count; ++i) {
        st = pkv_seq_reserve(a, seq_ids[i], n_tokens[i]);
        if (st != PKV_OK) break;
    }
    if (done) *done = i;
    return st;
}

pkv_status pkv_seq_release(pkv_allocator* a, int64_t seq_id) {
    if (!a) return PKV_ERR_INVALID_ARG;
    auto it = a->tables.find(seq_id);
    if (it == a->tables.end()) return PKV_ERR_NO_SEQ;
    for (int32_t blk : it->second)
        if (--a->refcnt[blk] == 0) a->free_list.push_back(blk);
    a->tables.erase(it);
    return PKV_OK;
}

pkv_status pkv_seq_share_prefix(pkv_allocator* a, int64_t src_seq, int64_t dst_seq, int64_t n_tokens,
                                int32_t* cow_src_block, int32_t* cow_dst_block) {
    if (!a || n_tokens < 0 || !cow_src_block || !cow_dst_block || src_seq == dst_seq) return PKV_ERR_INVALID_ARG;
    auto src = a->tables.find(src_seq);
    if (src == a->tables.end()) return PKV_ERR_NO_SEQ;
    if (a->tables.count(dst_seq)) return PKV_ERR_INVALID_ARG;
    const int64_t bs = a->block_size;
    if (n_tokens > (int64_t)src->second.size() * bs) return PKV_ERR_BOUNDS;
    const int64_t full = n_tokens / bs;
    const bool partial = n_tokens % bs != 0;
    if (partial && a->free_list.empty()) return PKV_ERR_OOM;
    std::vector<int32_t> tbl(src->second.begin(), src->second.begin() + full);
    for (int32_t blk : tbl) ++a->refcnt[blk];
    *cow_src_block = -1;
    *cow_dst_block = -1;
    if (partial) {
        const int32_t fresh = a->free_list.back();
        a->free_list.pop_back();
        a->refcnt[fresh] = 1;
        *cow_src_block = src->second[(size_t)full];
        *cow_dst_block = fresh;
        tbl.push_back(fresh);
    }
    a->tables.emplace(dst_seq, std::move(tbl));
    return PKV_OK;
}

pkv_status pkv_block_refcount(const pkv_allocator* a, int32_t block, int* out) {
    if (!a || !out || block < 0 || block >= a->num_blocks) return PKV_ERR_INVALID_ARG;
    *out = a->refcnt[block];
    return PKV_OK;
}

pkv_status pkv_seq_num_blocks(const pkv_allocator* a, int64_t seq_id, int* out) {
    if (!a || !out) return PKV_ERR_INVALID_ARG;
    auto it = a->tables.find(seq_id);
    if (it == a->tables.end()) return PKV_ERR_NO_SEQ;
    *out = (int)it->second.size();
    return PKV_OK;
}

pkv_status pkv_num_free_blocks(const pkv_allocator* a, int* out) {
    if (!a || !out) return PKV_ERR_INVALID_ARG;
    *out = (int)a->free_list.size();
    return PKV_OK;
}

pkv_status pkv_free_list(const pkv_allocator* a, int32_t* out, int capacity, int* n) {
    if (!a || !n || (capacity > 0 && !out) || capacity < 0) return PKV_ERR_INVALID_ARG;
    *n = (int)a->free_list.size();
    if (capacity < *n) return PKV_ERR_BOUNDS;
    if (*n) std::memcpy(out, a->free_list.data(), sizeof(int32_t) * (size_t)*n);
    return PKV_OK;
}

pkv_status pkv_get_block_tables(const pkv_allocator* a, const int64_t* seq_ids, int B, int max_blocks,
                                int32_t* out) {
    if (!a || B < 0 || max_blocks < 0 || (B > 0 && (!seq_ids || (max_blocks > 0 && !out)))) return PKV_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b) {  // validate everything before writing anything
        auto it = a->tables.find(seq_ids[b]);
        if (it == a->tables.end()) return PKV_ERR_NO_SEQ;
        if ((int64_t)it->second.size() > max_blocks) return PKV_ERR_BOUNDS;
    }
    for (int b = 0; b < B; ++b) {
        const std::vector<int32_t>& tbl = a->tables.find(seq_ids[b])->second;
        int32_t* row = out + (int64_t)b * max_blocks;
        const int n = (int)tbl.size();
        if (n) std::memcpy(row, tbl.data(), sizeof(int32_t) * (size_t)n);
        for (int k = n; k < max_blocks; ++k) row[k] = -1;
    }
    return PKV_OK;
}

pkv_status pkv_slot_mapping(const pkv_allocator* a, const int64_t* seq_ids, const int64_t* positions, int64_t N,
                            int64_t* out) {
    if (!a || N < 0 || (N > 0 && (!seq_ids || !positions || !out))) return PKV_ERR_INVALID_ARG;
    const int64_t bs = a->block_size;
    // Consecutive tokens usually belong to one sequence: remember the last lookup.
    int64_t last_id = 0;
    const std::vector<int32_t>* last = nullptr;
    for (int64_t i = 0; i < N; ++i) {
        const int64_t pos = positions[i];
        if (pos < 0) {
            out[i] = -1;
            continue;
        }
        if (!last || seq_ids[i] != last_id) {
            auto it = a->tables.find(seq_ids[i]);
            if (it == a->tables.end()) return PKV_ERR_NO_SEQ;
            last = &it->second;
            last_id = seq_ids[i];
        }
        const int64_t k = pos / bs;
        if (k >= (int64_t)last->size()) return PKV_ERR_BOUNDS;
        out[i] = (int64_t)(*last)[(size_t)k] * bs + pos % bs;
    }
    return PKV_OK;
}

pkv_status pkv_stage_prefill(pkv_allocator* a, const int64_t* seq_ids, const int64_t* p0, const int64_t* p1, int n,
                             int max_blocks, int64_t* slots_out, int32_t* cu_out, int32_t* ctx_out,
                             int32_t* tables_out) {
    if (!a || n < 0 || max_blocks < 1 || !cu_out) return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!seq_ids || !p0 || !p1 || !slots_out || !ctx_out || !tables_out)) return PKV_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {  // validate before changing anything
        if (p0[i] < 0 || p1[i] < p0[i] || p1[i] > INT32_MAX) return PKV_ERR_INVALID_ARG;
        total += p1[i] - p0[i];
        if (total > INT32_MAX) return PKV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i) {
        const pkv_status st = pkv_seq_reserve(a, seq_ids[i], p1[i]);
        if (st != PKV_OK) return st;
    }
    const pkv_status st = pkv_get_block_tables(a, seq_ids, n, max_blocks, tables_out);
    if (st != PKV_OK) return st;
    const int64_t bs = a->block_size;
    int64_t r = 0;
    cu_out[0] = 0;
    for (int i = 0; i < n; ++i) {
        const std::vector<int32_t>& tbl = a->tables.find(seq_ids[i])->second;  // reserved above
        for (int64_t pos = p0[i]; pos < p1[i]; ++pos) slots_out[r++] = (int64_t)tbl[(size_t)(pos / bs)] * bs + pos % bs;
        cu_out[i + 1] = (int32_t)r;
        ctx_out[i] = (int32_t)p1[i];
    }
    return PKV_OK;
}

pkv_status pkv_stage_decode(pkv_allocator* a, const int64_t* seq_ids, const int64_t* pos, int n, int n_pad,
                            int max_blocks, int32_t* tables_out, int64_t* slots_out, int32_t* lens_out) {
    if (!a || n < 0 || n_pad < n || max_blocks < 1) return PKV_ERR_INVALID_ARG;
    if (n_pad > 0 && (!tables_out || !slots_out || !lens_out)) return PKV_ERR_INVALID_ARG;
    if (n > 0 && (!seq_ids || !pos)) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)  // validate before changing anything
        if (pos[i] < 0 || pos[i] >= INT32_MAX) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const pkv_status st = pkv_seq_reserve(a, seq_ids[i], pos[i] + 1);
        if (st != PKV_OK) return st;
    }
    const pkv_status st = pkv_get_block_tables(a, seq_ids, n, max_blocks, tables_out);
    if (st != PKV_OK) return st;
    const int64_t bs = a->block_size;
    for (int i = 0; i < n; ++i) {
        const std::vector<int32_t>& tbl = a->tables.find(seq_ids[i])->second;  // reserved above
        slots_out[i] = (int64_t)tbl[(size_t)(pos[i] / bs)] * bs + pos[i] % bs;
        lens_out[i] = (int32_t)(pos[i] + 1);
    }
    for (int i = n; i < n_pad; ++i) {
        slots_out[i] = -1;
        lens_out[i] = 0;
        int32_t* row = tables_out + (int64_t)i * max_blocks;
        for (int k = 0; k < max_blocks; ++k) row[k] = -1;
    }
    return PKV_OK;
}

uint64_t pkv_kv_bytes(int64_t n_layers, int64_t n_kv_heads, int64_t head_dim, int64_t n_tokens, int64_t batch,
                      double bytes_per_elem) {
    // Integer product first (exact), then the element size; 2 * ... keeps half-byte sizes whole.
    const uint64_t elems = 2ull * (uint64_t)n_layers * (uint64_t)n_kv_heads * (uint64_t)head_dim *
                           (uint64_t)n_tokens * (uint64_t)batch;
    return (uint64_t)((long double)elems * (long double)bytes_per_elem);
}

const char* pkv_status_str(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_OOM: return "out of memory (no free blocks or device allocation failed)";
        case PKV_ERR_NO_SEQ: return "unknown sequence id";
        case PKV_ERR_BOUNDS: return "index out of bounds";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_TIMEOUT: return "kernel wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
