// Paged KV block pool: device storage, its TMA descriptor and the device error word.
//
// One pool holds num_blocks blocks of block_size tokens for n_kv_heads heads of K and V
// ("TensorRT-LLM 深度实战", §3.1: fixed-size pages handed out on demand;
// "TensorRT-LLM 推理加速实战", §8: block_size 64 by default, 16 in vLLM; FP8 e4m3 KV).
// Each (block, K|V, head) tile is contiguous, so one page of one head is a single
// bulk/TMA copy.  The layout is documented in include/pkv.h.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <new>

#include "pkv_internal.h"

namespace pkv {

namespace {

int env_int(const char* name) {
    const char* v = std::getenv(name);
    return v && *v ? std::atoi(v) : 0;
}

Settings read_settings() {
    return Settings{env_int("PKV_TEST_WAIT_LIMIT_MS"), env_int("PKV_TEST_STALL_COPIES"),
                    env_int("PKV_TEST_STALL_APPENDS"), env_int("PKV_ATTN_CTAS_PER_SM"),
                    env_int("PKV_ATTN_MAX_STAGES")};
}

Settings g_settings = read_settings();

}  // namespace

const Settings& settings() { return g_settings; }

void attention_configure(pkv_pool* pool);  // decode_attention.cu
void prefill_configure(pkv_pool* pool);    // prefill_attention.cu

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// One descriptor reads a page part's K rows and V rows together.  The pool is viewed as rows
// of head_dim elements (row r = ((blk*2 + kv)*Hkv + h)*bs + t); a K tile's V tile starts Hkv*bs
// rows further, which is the stride of the last dimension.  Box: min(bs, 64) rows of
// 128 bytes (64 bf16 or 128 fp8 elements; 64 bytes for fp8 head_dim 64), for K and V, and for
// bf16 head_dim 128 both 128-byte halves of a row (a panel dimension of stride 128 bytes).
// Shared memory receives [K|V][panel][row][128 bytes], each 128-byte line swizzled so that 8
// rows of one 16-byte column land in 8 different bank groups for ldmatrix.
bool encode_rows_map(pkv_pool* p) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const bool fp8 = p->dtype != PKV_KV_BF16;  // one-byte codes (fp8 or int8)
    const uint64_t esz = fp8 ? 1 : 2;
    const uint64_t row_bytes = (uint64_t)p->head_dim * esz;
    const uint64_t rows = (uint64_t)p->num_blocks * 2 * p->n_kv_heads * p->block_size;
    const uint64_t kv_stride = (uint64_t)p->n_kv_heads * p->block_size * row_bytes;
    const uint32_t inner = fp8 ? (uint32_t)p->head_dim : 64u;  // elements per box row
    const uint32_t box_rows = p->block_size < 64 ? (uint32_t)p->block_size : 64u;
    const CUtensorMapSwizzle swz = inner * esz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r;
    if (!fp8 && p->head_dim == 128) {
        cuuint64_t dims[4] = {64, (cuuint64_t)rows, 2, 2};
        cuuint64_t strides[3] = {(cuuint64_t)row_bytes, 128, (cuuint64_t)kv_stride};
        cuuint32_t box[4] = {64, box_rows, 2, 2};
        r = encode(&p->tmap_rows, dt, 4, p->kv, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, 2};
        cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)kv_stride};
        cuuint32_t box[3] = {inner, box_rows, 2};
        r = encode(&p->tmap_rows, dt, 3, p->kv, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return false;
    // Tail descriptor: 16-row boxes of one 128-byte panel of K or V rows, for the last, partly
    // filled part of a sequence (only its rows holding tokens are copied).
    cuuint64_t dims2[2] = {(cuuint64_t)(fp8 ? p->head_dim : p->head_dim), (cuuint64_t)rows};
    cuuint64_t strides2[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box2[2] = {inner, 16};
    r = encode(&p->tmap_tail, dt, 2, p->kv, dims2, strides2, box2, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    // Panel descriptor (prefill): min(bs, 64) rows of one 128-byte panel of K or V, so that the
    // rows of consecutive page parts land contiguously in one 128-row panel in shared memory.
    cuuint32_t box3[2] = {inner, box_rows};
    r = encode(&p->tmap_panel, dt, 2, p->kv, dims2, strides2, box3, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

void free_pool(pkv_pool* p) {
    if (!p) return;
    if (p->kv) cudaFree(p->kv);
    if (p->scales) cudaFree(p->scales);
    if (p->amax_scratch) cudaFree(p->amax_scratch);
    if (p->fresh_scratch) cudaFree(p->fresh_scratch);
    if (p->err) cudaFree(p->err);
    if (p->alloc) allocator_delete(p->alloc);
    delete p;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_pool_create(int num_blocks, int block_size, int n_kv_heads, int head_dim, pkv_dtype kv_dtype,
                           pkv_pool** out) {
    if (!out || num_blocks < 1 || n_kv_heads < 1 || !pkv::valid_block_size(block_size) ||
        (head_dim != 64 && head_dim != 128) ||
        (kv_dtype != PKV_KV_BF16 && kv_dtype != PKV_KV_FP8_E4M3 && kv_dtype != PKV_KV_INT8))
        return PKV_ERR_INVALID_ARG;
    const uint64_t rows = (uint64_t)num_blocks * 2 * n_kv_heads * block_size;
    if (rows >= (1ull << 31)) return PKV_ERR_INVALID_ARG;  // TMA row coordinates are int32
    pkv_pool* p = new (std::nothrow) pkv_pool();
    if (!p) return PKV_ERR_OOM;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->n_kv_heads = n_kv_heads;
    p->head_dim = head_dim;
    p->dtype = kv_dtype;
    const bool fp8 = kv_dtype != PKV_KV_BF16;  // one-byte codes with scales (fp8 or int8)
    p->alloc = pkv::allocator_new(num_blocks, block_size);
    if (!p->alloc) {
        pkv::free_pool(p);
        return PKV_ERR_OOM;
    }
    pkv_status st = PKV_OK;
    do {
        if (cudaGetDevice(&p->device) != cudaSuccess ||
            cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess ||
            cudaDeviceGetAttribute(&p->max_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p->device) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&p->max_smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device) !=
                cudaSuccess) {
            st = PKV_ERR_CUDA;
            break;
        }
        p->kv_bytes = rows * (uint64_t)head_dim * (fp8 ? 1 : 2);
        if (cudaMalloc(&p->kv, p->kv_bytes) != cudaSuccess) {
            st = PKV_ERR_OOM;
            break;
        }
        if (cudaMalloc(&p->err, sizeof(int)) != cudaSuccess) {
            st = PKV_ERR_OOM;
            break;
        }
        if (fp8) {
            p->scale_bytes = (size_t)num_blocks * n_kv_heads * 4 * sizeof(float);
            if (cudaMalloc(&p->scales, p->scale_bytes) != cudaSuccess ||
                cudaMalloc(&p->amax_scratch, (size_t)num_blocks * n_kv_heads * 2 * sizeof(uint32_t)) != cudaSuccess ||
                cudaMalloc(&p->fresh_scratch, (size_t)num_blocks) != cudaSuccess) {
                st = PKV_ERR_OOM;
                break;
            }
        }
        if (cudaMemset(p->kv, 0, p->kv_bytes) != cudaSuccess || cudaMemset(p->err, 0, sizeof(int)) != cudaSuccess ||
            (fp8 && (cudaMemset(p->scales, 0, p->scale_bytes) != cudaSuccess ||
                     cudaMemset(p->amax_scratch, 0, (size_t)num_blocks * n_kv_heads * 2 * sizeof(uint32_t)) !=
                         cudaSuccess ||
                     cudaMemset(p->fresh_scratch, 0, (size_t)num_blocks) != cudaSuccess)) ||
            cudaDeviceSynchronize() != cudaSuccess) {
            st = PKV_ERR_CUDA;
            break;
        }
        if (!pkv::encode_rows_map(p)) {
            st = PKV_ERR_CUDA;
            break;
        }
        pkv::attention_configure(p);
        pkv::prefill_configure(p);
        if (cudaGetLastError() != cudaSuccess) {
            st = PKV_ERR_CUDA;
            break;
        }
    } while (0);
    if (st != PKV_OK) {
        pkv::free_pool(p);
        return st;
    }
    *out = p;
    return PKV_OK;
}

pkv_status pkv_pool_destroy(pkv_pool* pool) {
    if (!pool) return PKV_ERR_INVALID_ARG;
    pkv::free_pool(pool);
    return PKV_OK;
}

pkv_status pkv_pool_allocator(pkv_pool* pool, pkv_allocator** out) {
    if (!pool || !out) return PKV_ERR_INVALID_ARG;
    *out = pool->alloc;
    return PKV_OK;
}

pkv_status pkv_pool_raw(const pkv_pool* pool, void** kv_dev, size_t* kv_bytes, float** scales_dev,
                        size_t* scale_bytes) {
    if (!pool) return PKV_ERR_INVALID_ARG;
    if (kv_dev) *kv_dev = pool->kv;
    if (kv_bytes) *kv_bytes = pool->kv_bytes;
    if (scales_dev) *scales_dev = pool->scales;
    if (scale_bytes) *scale_bytes = pool->scale_bytes;
    return PKV_OK;
}

pkv_status pkv_check_device_error(pkv_pool* pool) {
    if (!pool) return PKV_ERR_INVALID_ARG;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemcpy(&v, pool->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
    if (v && cudaMemset(pool->err, 0, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    if (v & pkv::kErrTimeout) return PKV_ERR_TIMEOUT;
    if (v & pkv::kErrBounds) return PKV_ERR_BOUNDS;
    return PKV_OK;
}

pkv_status pkv_pool_copy_block(pkv_pool* pool, int32_t src_block, int32_t dst_block, pkv_stream_t stream) {
    if (!pool || src_block < 0 || dst_block < 0 || src_block >= pool->num_blocks || dst_block >= pool->num_blocks)
        return PKV_ERR_INVALID_ARG;
    if (src_block == dst_block) return PKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t block_bytes = pool->kv_bytes / (size_t)pool->num_blocks;  // K and V of every head
    uint8_t* kv = static_cast<uint8_t*>(pool->kv);
    if (cudaMemcpyAsync(kv + (size_t)dst_block * block_bytes, kv + (size_t)src_block * block_bytes, block_bytes,
                        cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (pool->scales) {
        const size_t rec = (size_t)pool->n_kv_heads * 4;  // floats per block
        if (cudaMemcpyAsync(pool->scales + (size_t)dst_block * rec, pool->scales + (size_t)src_block * rec,
                            rec * sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

pkv_status pkv_decode_workspace_init(void* workspace, size_t bytes, pkv_stream_t stream) {
    if (!workspace && bytes) return PKV_ERR_INVALID_ARG;
    if (!bytes) return PKV_OK;
    return cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"

extern "C" pkv_status pkv_debug_reload_env(void) {
    pkv::g_settings = pkv::read_settings();
    return PKV_OK;
}
