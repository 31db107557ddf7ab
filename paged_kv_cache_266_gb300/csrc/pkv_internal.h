// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/pkv.h"

namespace pkv {

// Device error word bits (read and cleared by pkv_check_device_error).
constexpr int kErrBounds = 1;
constexpr int kErrTimeout = 2;

bool valid_block_size(int bs);
pkv_status append_check(const pkv_pool* pool, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                        int64_t N);
pkv_status append_rope_launch(pkv_pool* pool, void* k_new, const void* v_new, const int64_t* slot_mapping,
                              const int64_t* positions, int64_t N, double rope_base, void* q, int n_q_heads,
                              cudaStream_t cs);
pkv_allocator* allocator_new(int num_blocks, int block_size);
void allocator_delete(pkv_allocator* a);

// Launch settings and test hooks taken from the environment when the library loads (and again
// by pkv_debug_reload_env), not on every launch:
//   PKV_TEST_WAIT_LIMIT_MS  > 0: bound of every kernel wait in ms (default 2 s);
//   PKV_TEST_STALL_COPIES   != 0: every pipeline stage expects 16 bytes no copy delivers, so the
//                           bounded waits run out (failure detection tested without a fault);
//   PKV_TEST_STALL_APPENDS  != 0: the decode step's wait for its own append expects one row more
//                           than the kernel quantises, so that bounded wait runs out;
//   PKV_ATTN_CTAS_PER_SM    decode attention CTAs per SM (0: the kernel's default);
//   PKV_ATTN_MAX_STAGES     decode attention pipeline stages at most (0: default).
struct Settings {
    int wait_limit_ms;
    int stall_copies;
    int stall_appends;
    int attn_ctas_per_sm;
    int attn_max_stages;
};
const Settings& settings();

}  // namespace pkv

struct pkv_pool {
    int num_blocks = 0;
    int block_size = 0;
    int n_kv_heads = 0;
    int head_dim = 0;
    pkv_dtype dtype = PKV_KV_BF16;
    int device = 0;
    int sm_count = 0;
    int max_smem_per_sm = 0;    // bytes usable by resident CTAs on one SM
    int max_smem_per_block = 0;  // opt-in dynamic shared memory limit of one CTA

    void* kv = nullptr;  // the block pool, layout documented in pkv.h
    size_t kv_bytes = 0;
    float* scales = nullptr;  // fp8: [num_blocks][n_kv_heads][4]
    size_t scale_bytes = 0;
    uint32_t* amax_scratch = nullptr;  // fp8 append: [num_blocks][n_kv_heads][2] fp32 bits, kept zero between calls
    uint8_t* fresh_scratch = nullptr;  // fp8 append: [num_blocks] "offset 0 written by this call", kept zero
    int* err = nullptr;               // device error word

    // TMA descriptor reading a page part's K and V rows in one copy (see pool.cu).
    CUtensorMap tmap_rows;
    // 16 rows of one 128-byte panel (the tail of a sequence's last page part).
    CUtensorMap tmap_tail;
    // min(bs, 64) rows of one 128-byte panel (prefill: page parts stacked into 128-row panels).
    CUtensorMap tmap_panel;

    pkv_allocator* alloc = nullptr;
};

#define PKV_CUDA_TRY(expr)                       \
    do {                                         \
        cudaError_t e_ = (expr);                 \
        if (e_ != cudaSuccess) return PKV_ERR_CUDA; \
    } while (0)
