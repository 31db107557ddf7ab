// Append / scatter: write each new token's K and V rows into its physical slot.
//
// "TensorRT-LLM 深度实战" (chenxutan.com), §3.1 Paged KV Cache: append_tokens grows a
// sequence by whole pages; the tokens' K/V then live in those pages.  A slot is
// block * block_size + offset (the allocator's slot mapping).
//
// bf16 pools: one 16-byte vector per thread, a (token, K|V, head) row per D/8 threads, so
// both the read of k_new/v_new and the write of the row are coalesced.
//
// fp8 pools ("TensorRT-LLM 深度实战" §4.5 E4M3; "TensorRT-LLM 推理加速实战" §8 fp8_e4m3 KV
// cache): one fp32 scale per (block, K|V, head).  A block's scales are derived by the call
// that writes its offset 0, as amax/448 over that call's tokens in the block (1 when the
// amax is 0); later calls reuse them and saturate.  Three short passes do this without any
// grid-wide synchronisation inside a kernel:
//   1. amax: per row |x| max, atomicMax into a per-(block, K|V, head) scratch word, and a
//      per-block "offset 0 written" flag;
//   2. quantise: derive/lookup the scale, x / scale (IEEE division), RNE-satfinite to E4M3;
//   3. reset: return the scratch words and flags of the touched blocks to zero.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

struct RowIndex {
    int64_t i;  // token
    int kv;     // 0 = K, 1 = V
    int h;      // KV head
};

__device__ __forceinline__ RowIndex row_index(int64_t row, int Hkv) {
    RowIndex r;
    r.i = row / (2 * Hkv);
    const int rem = (int)(row - r.i * 2 * Hkv);
    r.kv = rem / Hkv;
    r.h = rem - r.kv * Hkv;
    return r;
}

__device__ __forceinline__ int64_t tile_elem(int64_t blk, int kv, int h, int Hkv, int bs, int D) {
    return ((blk * 2 + kv) * Hkv + h) * (int64_t)bs * D;
}

// Position of token u (0..15) inside a 16-byte fp8 V panel row (pair order of the MMA).
__device__ __forceinline__ int fp8_v_pos(int u) { return u < 8 ? 4 * (u >> 1) + (u & 1) : 4 * ((u - 8) >> 1) + 2 + (u & 1); }

template <int D>
__global__ void __launch_bounds__(kAppendThreads) append_bf16_kernel(uint16_t* __restrict__ pool,
                                                                      const uint16_t* __restrict__ k_new,
                                                                      const uint16_t* __restrict__ v_new,
                                                                      const int64_t* __restrict__ slots, int64_t N,
                                                                      int Hkv, int bs, int num_blocks, int* err) {
    ptx::grid_launch_dependents();  // a following decode step may begin its set-up
    constexpr int TPR = D / 8;
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gt / TPR;
    const int part = (int)(gt % TPR);
    if (row >= N * 2 * Hkv) return;
    const RowIndex r = row_index(row, Hkv);
    const int64_t slot = __ldg(slots + r.i);
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * bs) {
        if (part == 0 && r.kv == 0 && r.h == 0) atomicOr(err, kErrBounds);
        return;
    }
    const int64_t blk = slot / bs;
    const int t = (int)(slot - blk * bs);
    const uint16_t* src = (r.kv ? v_new : k_new) + (r.i * Hkv + r.h) * D + part * 8;
    uint16_t* dst = pool + tile_elem(blk, r.kv, r.h, Hkv, bs, D) + (int64_t)t * D + part * 8;
    *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads) fp8_amax_kernel(const uint16_t* __restrict__ k_new,
                                                                   const uint16_t* __restrict__ v_new,
                                                                   const int64_t* __restrict__ slots, int64_t N,
                                                                   int Hkv, int bs, int num_blocks,
                                                                   uint32_t* amax, uint8_t* fresh, int* err) {
    ptx::grid_launch_dependents();  // a following decode step may begin its set-up
    constexpr int TPR = D / 8;  // 8 or 16 lanes per row, aligned inside the warp
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gt / TPR;
    const int part = (int)(gt % TPR);
    const bool in_range = row < N * 2 * Hkv;
    uint32_t m = 0;  // max |x| as fp32 bits (non-negative floats order like their bits)
    RowIndex r{0, 0, 0};
    if (in_range) {
        r = row_index(row, Hkv);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>((r.kv ? v_new : k_new) + (r.i * Hkv + r.h) * D + part * 8));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t lo = (w[e] << 16) & 0x7fffffffu, hi = w[e] & 0x7fff0000u;
            m = max(m, max(lo, hi));
        }
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!in_range || part != 0) return;
    const int64_t slot = __ldg(slots + r.i);
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * bs) {
        if (r.kv == 0 && r.h == 0) atomicOr(err, kErrBounds);
        return;
    }
    const int64_t blk = slot / bs;
    atomicMax(amax + (blk * Hkv + r.h) * 2 + r.kv, m);
    if (slot - blk * bs == 0 && r.kv == 0 && r.h == 0) fresh[blk] = 1;
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads) fp8_quant_kernel(uint8_t* __restrict__ pool,
                                                                    float* __restrict__ scales,
                                                                    const uint16_t* __restrict__ k_new,
                                                                    const uint16_t* __restrict__ v_new,
                                                                    const int64_t* __restrict__ slots, int64_t N,
                                                                    int Hkv, int bs, int num_blocks,
                                                                    const uint32_t* __restrict__ amax,
                                                                    const uint8_t* __restrict__ fresh) {
    ptx::grid_launch_dependents();  // a following decode step may begin its set-up
    constexpr int TPR = D / 8;
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gt / TPR;
    const int part = (int)(gt % TPR);
    if (row >= N * 2 * Hkv) return;
    const RowIndex r = row_index(row, Hkv);
    const int64_t slot = __ldg(slots + r.i);
    if (slot < 0 || slot >= (int64_t)num_blocks * bs) return;
    const int64_t blk = slot / bs;
    const int t = (int)(slot - blk * bs);
    float* sp = scales + (blk * Hkv + r.h) * 4 + r.kv;
    float s;
    if (fresh[blk]) {
        const float a = __uint_as_float(amax[(blk * Hkv + r.h) * 2 + r.kv]);
        s = a > 0.0f ? __fdiv_rn(a, 448.0f) : 1.0f;
        if (t == 0 && part == 0) *sp = s;
    } else {
        s = *sp;
    }
    const uint4 v = __ldg(reinterpret_cast<const uint4*>((r.kv ? v_new : k_new) + (r.i * Hkv + r.h) * D + part * 8));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t codes[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float x0 = __fdiv_rn(ptx::bf16lo_to_f32(w[2 * e]), s), x1 = __fdiv_rn(ptx::bf16hi_to_f32(w[2 * e]), s);
        const float x2 = __fdiv_rn(ptx::bf16lo_to_f32(w[2 * e + 1]), s),
                    x3 = __fdiv_rn(ptx::bf16hi_to_f32(w[2 * e + 1]), s);
        codes[e] = ptx::f32x2_to_e4m3x2(x0, x1) | (ptx::f32x2_to_e4m3x2(x2, x3) << 16);
    }
    uint8_t* tile = pool + tile_elem(blk, r.kv, r.h, Hkv, bs, D);
    if (r.kv == 0) {
        *reinterpret_cast<uint2*>(tile + (int64_t)t * D + part * 8) = make_uint2(codes[0], codes[1]);
    } else {
        uint8_t* panel = tile + (int64_t)(t >> 4) * D * 16 + fp8_v_pos(t & 15);
#pragma unroll
        for (int e = 0; e < 8; ++e) panel[(int64_t)(part * 8 + e) * 16] = (uint8_t)(codes[e >> 2] >> (8 * (e & 3)));
    }
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads) fp8_reset_kernel(const int64_t* __restrict__ slots, int64_t N,
                                                                    int Hkv, int bs, int num_blocks,
                                                                    uint32_t* amax, uint8_t* fresh) {
    ptx::grid_launch_dependents();  // a following decode step may begin its set-up
    constexpr int TPR = D / 8;
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gt / TPR;
    if (row >= N * 2 * Hkv || gt % TPR != 0) return;
    const RowIndex r = row_index(row, Hkv);
    const int64_t slot = __ldg(slots + r.i);
    if (slot < 0 || slot >= (int64_t)num_blocks * bs) return;
    const int64_t blk = slot / bs;
    amax[(blk * Hkv + r.h) * 2 + r.kv] = 0u;
    if (r.kv == 0 && r.h == 0) fresh[blk] = 0;
}

template <int D>
pkv_status launch_append(pkv_pool* p, const uint16_t* k, const uint16_t* v, const int64_t* slots, int64_t N,
                         cudaStream_t st) {
    const int64_t threads = N * 2 * p->n_kv_heads * (D / 8);
    const int64_t blocks = (threads + kAppendThreads - 1) / kAppendThreads;
    if (blocks > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    const dim3 grid((unsigned)blocks);
    if (p->dtype == PKV_KV_BF16) {
        append_bf16_kernel<D><<<grid, kAppendThreads, 0, st>>>(static_cast<uint16_t*>(p->kv), k, v, slots, N,
                                                               p->n_kv_heads, p->block_size, p->num_blocks, p->err);
    } else {
        fp8_amax_kernel<D><<<grid, kAppendThreads, 0, st>>>(k, v, slots, N, p->n_kv_heads, p->block_size,
                                                            p->num_blocks, p->amax_scratch, p->fresh_scratch, p->err);
        fp8_quant_kernel<D><<<grid, kAppendThreads, 0, st>>>(static_cast<uint8_t*>(p->kv), p->scales, k, v, slots, N,
                                                             p->n_kv_heads, p->block_size, p->num_blocks,
                                                             p->amax_scratch, p->fresh_scratch);
        fp8_reset_kernel<D><<<grid, kAppendThreads, 0, st>>>(slots, N, p->n_kv_heads, p->block_size, p->num_blocks,
                                                             p->amax_scratch, p->fresh_scratch);
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

namespace pkv {

pkv_status append_check(const pkv_pool* pool, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                        int64_t N) {
    if (!pool || N < 0) return PKV_ERR_INVALID_ARG;
    if (N == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u) return PKV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

}  // namespace pkv

extern "C" pkv_status pkv_append(pkv_pool* pool, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                 int64_t N, pkv_stream_t stream) {
    const pkv_status st = pkv::append_check(pool, k_new, v_new, slot_mapping, N);
    if (st != PKV_OK || N == 0) return st;
    const auto* k = static_cast<const uint16_t*>(k_new);
    const auto* v = static_cast<const uint16_t*>(v_new);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    return pool->head_dim == 128 ? pkv::launch_append<128>(pool, k, v, slot_mapping, N, cs)
                                 : pkv::launch_append<64>(pool, k, v, slot_mapping, N, cs);
}
