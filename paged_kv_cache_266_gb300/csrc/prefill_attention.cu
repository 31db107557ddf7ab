// Chunked-context (prefill) attention over the paged KV pool on the 5th-generation tensor
// cores.  "TensorRT-LLM 深度实战" §7.3: a long input is processed as chunks, each chunk's
// queries attending to everything cached before the chunk and causally within it;
// "TensorRT-LLM 推理加速实战" §7.2: context_fmha is the prefill flash attention, and with
// use_paged_context_fmha it reads K/V from the paged cache.  For sequence b whose chunk holds
// n = cu_q[b+1] - cu_q[b] queries and whose cache holds L = ctx[b] tokens (the chunk's own
// K/V already appended), query i sits at position L - n + i and, for query head j with KV head
// h = j / G,
//     out[cu_q[b] + i][j] = sum_{t <= L-n+i} softmax_t(scale * q . K_b[t]) V_b[t].
//
// Work decomposition: one CTA per (sequence, KV head, tile of 128 query rows).  A row is a
// (token, head-in-group) pair, so a tile covers 128/G consecutive chunk tokens and all G query
// heads of one KV head: every K/V tile brought on chip serves the whole group.  The CTA
// walks the KV tiles of 128 keys that its last token can see:
//   warp 0     TMA producer: one 4-D tensor copy per page part (K and V, both 64-element
//              panels, 128-byte swizzled) into a two-stage ring; parts past the context get a
//              coordinate past the pool, which the copy fills with zeros.
//   warp 1     tensor-memory owner and MMA issuer (one thread):
//                S_j = Q K_j^T   M=128 rows, N=part, K=128 (tcgen05.mma kind::f16, bf16 in,
//                                fp32 accumulator in TMEM, two S buffers)
//                O  += P_j V_j   M=128, N=128, K=16 per instruction, A = P from shared
//                                memory, B = V MN-major straight from the page copy
//              issued one KV tile ahead (S_{j+1} runs while the softmax works on S_j).
//   warps 2-5  one query row per thread (TMEM lane = row): the Q row into shared memory,
//              then per KV tile the S row out of TMEM (tcgen05.ld), causal mask, online
//              softmax in base 2, the O row rescaled in TMEM when the running maximum grows,
//              P as bf16 into shared memory; finally O / l as bf16 to global memory.
// Every mbarrier wait is bounded; on expiry the kernel sets the pool's error word, every role
// stops, and tensor memory is released.
#include <cstdlib>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace prefill {

constexpr int kD = 128;
constexpr int kRows = 128;  // query rows per CTA
constexpr int kKeys = 128;  // keys per KV tile
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kPanelBytes = 128u * 128u;              // 128 rows x 128 bytes
constexpr uint32_t kQBytes = 2 * kPanelBytes;              // Q tile: two 64-element panels
constexpr uint32_t kStageBytes = 4u * kKeys * 128u;        // K and V, two panels each
constexpr uint32_t kPBytes = 2 * kPanelBytes;              // P tile (bf16), two 64-key panels
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffKV + kStages * kStageBytes;
constexpr uint32_t kOffBar = kOffP + kPBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // two S buffers of 128 columns
constexpr uint32_t kColO = 256;  // O: 128 columns
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// mbarrier slots
constexpr int kBarQ = 0;                     // Q rows written (4 softmax warps arrive)
constexpr int kBarFull = 1;                  // [kStages] K/V copies landed (tx bytes)
constexpr int kBarEmpty = kBarFull + kStages;  // [kStages] PV of the stage's tile done (commit)
constexpr int kBarS = kBarEmpty + kStages;   // [2] S_j ready (commit)
constexpr int kBarP = kBarS + 2;             // P_j written (4 softmax warps arrive)
constexpr int kBarO = kBarP + 1;             // PV_j done (commit)
constexpr int kNumBars = kBarO + 1;

struct Params {
    const uint16_t* q;
    uint16_t* out;
    const int32_t* cu_q;
    const int32_t* tables;
    const int32_t* ctx;
    int* err;
    int Hq, Hkv, G, max_blocks, bs, part, num_blocks, tiles;
    int32_t oob_row;  // a row coordinate past the pool: the copy fills the box with zeros
    float scale_log2;
    uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const sm = smem_raw + (base - raw);
    const uint32_t sQ = base + kOffQ, sKV = base + kOffKV, sP = base + kOffP;
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };

    const int b = blockIdx.z, h = blockIdx.y;
    const int tile = p.tiles - 1 - (int)blockIdx.x;  // deepest tiles (most keys) launch first
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    ptx::grid_dependency_wait();  // inputs may come from the preceding append
    const int q0 = p.cu_q[b];
    const int n = p.cu_q[b + 1] - q0;
    const int L = p.ctx[b];
    const int T = kRows / p.G;  // chunk tokens per tile
    const int t0 = tile * T;
    if (t0 >= n) return;
    if (n < 0 || n > L || L > p.max_blocks * p.bs) {
        if (threadIdx.x == 0) atomicOr(p.err, kErrBounds);
        return;
    }
    const int t_last = min(n, t0 + T) - 1;
    const int kv_end = L - n + t_last + 1;  // keys seen by the tile's last token
    const int n_kv = (kv_end + kKeys - 1) / kKeys;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) ptx::mbar_init(bar(i), (i == kBarQ || i == kBarP) ? 4u : 1u);
        abort_s = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_addr(&tmem_base_s), kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const int parts = kKeys / p.part;
    const uint32_t part_bytes = 4u * (uint32_t)p.part * 128u;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        const int32_t* tb = p.tables + (int64_t)b * p.max_blocks;
        for (int j = 0; j < n_kv; ++j) {
            const int s = j % kStages;
            if (j >= kStages) {
                bool ok = true;
                if (lane == 0) ok = ptx::mbar_wait(bar(kBarEmpty + s), ((j / kStages) - 1) & 1, p.wait_ns);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) {
                    if (lane == 0) {
                        atomicOr(p.err, kErrTimeout);
                        abort_s = 1;
                    }
                    break;
                }
            }
            if (__shfl_sync(0xffffffffu, abort_s, 0)) break;  // warp-uniform
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar(kBarFull + s), kStageBytes);
            __syncwarp();
            if (lane < parts) {
                const int tok = j * kKeys + lane * p.part;  // first key of this page part
                int32_t row = p.oob_row;
                if (tok < L) {
                    const int blk = tb[tok / p.bs];
                    if (blk >= 0 && blk < p.num_blocks)
                        row = (int32_t)(((int64_t)2 * blk * p.Hkv + h) * p.bs + (tok % p.bs));
                    else
                        atomicOr(p.err, kErrBounds);
                }
                ptx::tma_load_4d(sKV + (uint32_t)s * kStageBytes + (uint32_t)lane * part_bytes, &tmap, 0, row, 0, 0,
                                 bar(kBarFull + s));
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t tS = tmem + kColS, tO = tmem + kColO;
            const uint32_t idS = ptx::umma_idesc_bf16(128, p.part, 0, 0);
            const uint32_t idO = ptx::umma_idesc_bf16(128, kD, 0, 1);
            bool ok = ptx::mbar_wait(bar(kBarQ), 0, p.wait_ns);
            ptx::tc_fence_after();
            int committed_o = 0;
            for (int j = 0; ok && j <= n_kv; ++j) {
                if (j < n_kv) {
                    const int s = j % kStages;
                    ok = ptx::mbar_wait(bar(kBarFull + s), (j / kStages) & 1, p.wait_ns);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t kst = sKV + (uint32_t)s * kStageBytes;
                    const uint32_t dS = tS + (uint32_t)(j & 1) * kKeys;
                    for (int pi = 0; pi < parts; ++pi) {
                        if (j * kKeys + pi * p.part >= L) break;  // past the context: scores unused
                        const uint32_t kpart = kst + (uint32_t)pi * part_bytes;
#pragma unroll
                        for (int k = 0; k < kD / 16; ++k) {
                            const uint64_t a =
                                ptx::umma_sdesc_sw128(sQ + (uint32_t)(k >> 2) * kPanelBytes + (uint32_t)(k & 3) * 32u,
                                                      16, 1024);
                            const uint64_t bd = ptx::umma_sdesc_sw128(
                                kpart + (uint32_t)(k >> 2) * (uint32_t)p.part * 128u + (uint32_t)(k & 3) * 32u, 16,
                                1024);
                            ptx::umma_bf16(dS + (uint32_t)(pi * p.part), a, bd, idS, k > 0 ? 1u : 0u);
                        }
                    }
                    ptx::umma_commit(bar(kBarS + (j & 1)));
                }
                if (j >= 1) {
                    const int i = j - 1, s = i % kStages;
                    ok = ptx::mbar_wait(bar(kBarP), i & 1, p.wait_ns);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t vst = sKV + (uint32_t)s * kStageBytes;
                    for (int pi = 0; pi < parts; ++pi) {
                        const uint32_t vpart = vst + (uint32_t)pi * part_bytes + 2u * (uint32_t)p.part * 128u;
                        for (int c = 0; c < p.part / 16; ++c) {
                            const int tok = pi * p.part + 16 * c;  // key within the tile
                            if (i * kKeys + tok >= L) break;        // all-zero P columns from here on
                            const uint64_t a = ptx::umma_sdesc_sw128(
                                sP + (uint32_t)(tok >> 6) * kPanelBytes + (uint32_t)((tok & 63) >> 4) * 32u, 16, 1024);
                            const uint64_t bd =
                                ptx::umma_sdesc_sw128(vpart + (uint32_t)c * 2048u, (uint32_t)p.part * 128u, 1024);
                            ptx::umma_bf16(tO, a, bd, idO, (i > 0 || tok > 0) ? 1u : 0u);
                        }
                    }
                    ptx::umma_commit(bar(kBarO));
                    // the producer waits for this stage only if a later tile reuses it; no
                    // arrival is left pending when the CTA exits
                    if (i + kStages < n_kv) ptx::umma_commit(bar(kBarEmpty + s));
                    ++committed_o;
                }
            }
            if (!ok) {
                atomicOr(p.err, kErrTimeout);
                abort_s = 1;
                // let MMAs already issued finish before tensor memory is released
                if (committed_o > 0) ptx::mbar_wait(bar(kBarO), (committed_o - 1) & 1, p.wait_ns);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax / epilogue
        const int qw = warp & 3;  // TMEM lane quarter this warp may access
        const int r = qw * 32 + lane;
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const int tok = t0 + r / p.G, g = r % p.G;
        const bool valid = tok < n;
        const int qlim = min(L - n + tok, L - 1);  // last key this row may see
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)(q0 + tok) * p.Hq + h * p.G + g) * kD);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + kOffQ + (uint32_t)(c >> 3) * kPanelBytes + swz128(r, c & 7)) = v;
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarQ));
        }
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarS + (j & 1)), (j >> 1) & 1, p.wait_ns));
            if (!ok) break;
            ptx::tc_fence_after();
            float x[kKeys];
            {
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    ptx::tmem_ld32(tmem + kColS + (uint32_t)(j & 1) * kKeys + 32u * c + lane_off, v);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(v[e]);
                }
            }
            const int kbase = j * kKeys;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kKeys; ++c) {
                x[c] = (kbase + c <= qlim) ? x[c] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, x[c]);
            }
            const float m_new = fmaxf(m, mx);
            if (j >= 1) {
                ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarO), (j - 1) & 1, p.wait_ns));
                if (!ok) break;
                ptx::tc_fence_after();
                const bool grow = m_new > m && m != -INFINITY;
                if (__any_sync(0xffffffffu, grow)) {
                    const float alpha = grow ? ptx::exp2_approx(m - m_new) : 1.f;
                    l *= alpha;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[32];
                        ptx::tmem_ld32(tmem + kColO + 32u * c + lane_off, v);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        ptx::tmem_st32(tmem + kColO + 32u * c + lane_off, v);
                    }
                    ptx::tmem_wait_st();
                }
            }
            m = m_new;
            const float mu = m == -INFINITY ? 0.f : m;
            uint8_t* prow = sm + kOffP;
#pragma unroll
            for (int c16 = 0; c16 < kKeys / 8; ++c16) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = ptx::exp2_approx(x[8 * c16 + 2 * e] - mu);
                    const float p1 = ptx::exp2_approx(x[8 * c16 + 2 * e + 1] - mu);
                    w[e] = ptx::pack_bf16x2(p0, p1);
                    l += ptx::bf16lo_to_f32(w[e]) + ptx::bf16hi_to_f32(w[e]);
                }
                *reinterpret_cast<uint4*>(prow + (uint32_t)(c16 >> 3) * kPanelBytes + swz128(r, c16 & 7)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarP));
        }
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarO), (n_kv - 1) & 1, p.wait_ns));
        if (ok) {
            ptx::tc_fence_after();
            const float inv = 1.f / l;
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + tok) * p.Hq + h * p.G + g) * kD);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + kColO + 32u * c + lane_off, v);
                ptx::tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 o;
                        o.x = ptx::pack_bf16x2(__uint_as_float(v[8 * e + 0]) * inv, __uint_as_float(v[8 * e + 1]) * inv);
                        o.y = ptx::pack_bf16x2(__uint_as_float(v[8 * e + 2]) * inv, __uint_as_float(v[8 * e + 3]) * inv);
                        o.z = ptx::pack_bf16x2(__uint_as_float(v[8 * e + 4]) * inv, __uint_as_float(v[8 * e + 5]) * inv);
                        o.w = ptx::pack_bf16x2(__uint_as_float(v[8 * e + 6]) * inv, __uint_as_float(v[8 * e + 7]) * inv);
                        dst[4 * c + e] = o;
                    }
                }
            }
        } else if (lane == 0) {
            atomicOr(p.err, kErrTimeout);
            abort_s = 1;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return v && *v ? std::atoi(v) : dflt;
}

}  // namespace prefill

void prefill_configure(pkv_pool* pool) {
    (void)pool;
    cudaFuncSetAttribute(prefill::prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)prefill::kSmemBytes);
}

// Argument checks shared by the prefill entry points; fills the kernel parameters and grid.
pkv_status prefill_prepare(const pkv_pool* pool, const void* q, const int32_t* cu_q, int32_t max_q_len,
                           const int32_t* tables, int32_t max_blocks, const int32_t* ctx, int32_t B, int32_t Hq,
                           float scale, void* out, prefill::Params& p, dim3& grid) {
    using namespace prefill;
    if (!pool || B < 0 || max_q_len < 0 || Hq < 1) return PKV_ERR_INVALID_ARG;
    if (pool->dtype != PKV_KV_BF16 || pool->head_dim != kD) return PKV_ERR_INVALID_ARG;
    if (Hq % pool->n_kv_heads) return PKV_ERR_INVALID_ARG;
    const int G = Hq / pool->n_kv_heads;
    if (G > kRows || (G & (G - 1))) return PKV_ERR_INVALID_ARG;
    if (B > 65535 || pool->n_kv_heads > 65535) return PKV_ERR_INVALID_ARG;
    if (B == 0 || max_q_len == 0) {
        grid = dim3(0);
        return PKV_OK;
    }
    if (!q || !cu_q || !tables || !ctx || !out || max_blocks < 1) return PKV_ERR_INVALID_ARG;
    if (((uintptr_t)q | (uintptr_t)out) & 15u) return PKV_ERR_INVALID_ARG;
    if (((uintptr_t)cu_q | (uintptr_t)tables | (uintptr_t)ctx) & 3u) return PKV_ERR_INVALID_ARG;
    const int T = kRows / G;
    p.q = static_cast<const uint16_t*>(q);
    p.out = static_cast<uint16_t*>(out);
    p.cu_q = cu_q;
    p.tables = tables;
    p.ctx = ctx;
    p.err = pool->err;
    p.Hq = Hq;
    p.Hkv = pool->n_kv_heads;
    p.G = G;
    p.max_blocks = max_blocks;
    p.bs = pool->block_size;
    p.part = pool->block_size < 64 ? pool->block_size : 64;
    p.num_blocks = pool->num_blocks;
    p.tiles = (max_q_len + T - 1) / T;
    p.oob_row = (int32_t)((int64_t)pool->num_blocks * 2 * pool->n_kv_heads * pool->block_size);
    p.scale_log2 = scale * 1.4426950408889634f;
    const int limit_ms = env_int("PKV_TEST_WAIT_LIMIT_MS", 0);
    p.wait_ns = limit_ms > 0 ? (uint64_t)limit_ms * 1000000ull : kWaitLimitNs;
    grid = dim3((unsigned)p.tiles, (unsigned)pool->n_kv_heads, (unsigned)B);
    return PKV_OK;
}

pkv_status prefill_launch(const pkv_pool* pool, const prefill::Params& p, dim3 grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(prefill::kThreads);
    cfg.dynamicSmemBytes = prefill::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill::prefill_kernel, pool->tmap_rows, p) == cudaSuccess ? PKV_OK
                                                                                                  : PKV_ERR_CUDA;
}

}  // namespace pkv

extern "C" {

pkv_status pkv_prefill_attention(pkv_pool* pool, const void* q, const int32_t* cu_q_lens, int32_t max_q_len,
                                 const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                                 int32_t B, int32_t n_q_heads, float scale, void* out, pkv_stream_t stream) {
    pkv::prefill::Params p;
    dim3 grid;
    const pkv_status s = pkv::prefill_prepare(pool, q, cu_q_lens, max_q_len, block_tables, max_blocks, context_lens,
                                              B, n_q_heads, scale, out, p, grid);
    if (s != PKV_OK || grid.x == 0) return s;
    return pkv::prefill_launch(pool, p, grid, (cudaStream_t)stream, false);
}

pkv_status pkv_prefill_step(pkv_pool* pool, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                            int64_t n_new, const void* q, const int32_t* cu_q_lens, int32_t max_q_len,
                            const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens, int32_t B,
                            int32_t n_q_heads, float scale, void* out, pkv_stream_t stream) {
    pkv::prefill::Params p;
    dim3 grid;
    pkv_status s = pkv::append_check(pool, k_new, v_new, slot_mapping, n_new);
    if (s != PKV_OK) return s;
    s = pkv::prefill_prepare(pool, q, cu_q_lens, max_q_len, block_tables, max_blocks, context_lens, B, n_q_heads,
                             scale, out, p, grid);
    if (s != PKV_OK) return s;
    s = pkv_append(pool, k_new, v_new, slot_mapping, n_new, stream);
    if (s != PKV_OK || grid.x == 0) return s;
    return pkv::prefill_launch(pool, p, grid, (cudaStream_t)stream, true);
}

}  // extern "C"
