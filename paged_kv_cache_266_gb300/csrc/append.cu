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
// cache) and int8 pools (the same with amax/127 and symmetric int8 codes): one fp32 scale per
// (block, K|V, head).  A block's scales are derived by the call
// that writes its offset 0, as amax/448 over that call's tokens in the block (1 when the
// amax is 0); later calls reuse them and saturate.  Calls of up to 1024 tokens (a decode step's
// size) do this in one kernel, a CTA per token that finds the call's other tokens in its block by
// scanning the call's slots (quant_append_small_kernel); pkv_decode_step on a one-byte pool does
// the same per row pair inside the attention kernel instead (decode_attention.cu), with the
// element codes of quant.cuh.  Larger calls take three short passes, with no grid-wide
// synchronisation inside a kernel:
//   1. amax: per row |x| max, atomicMax into a per-(block, K|V, head) scratch word, and a
//      per-block "offset 0 written" flag;
//   2. quantise: derive/lookup the scale, x / scale (IEEE division), RNE-satfinite to E4M3;
//   3. reset: return the scratch words and flags of the touched blocks to zero.
#include <cmath>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

using quant::amax_bits;
using quant::fp8_v_pos;
using quant::quant_store;
using quant::tile_elem;

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
        m = amax_bits(__ldg(reinterpret_cast<const uint4*>((r.kv ? v_new : k_new) + (r.i * Hkv + r.h) * D + part * 8)));
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

template <int D, bool I8>
__global__ void __launch_bounds__(kAppendThreads) fp8_quant_kernel(uint8_t* __restrict__ pool,
                                                                    float* __restrict__ scales,
                                                                    const uint16_t* __restrict__ k_new,
                                                                    const uint16_t* __restrict__ v_new,
                                                                    const int64_t* __restrict__ slots, int64_t N,
                                                                    int Hkv, int bs, int num_blocks,
                                                                    const uint32_t* __restrict__ amax,
                                                                    const uint8_t* __restrict__ fresh) {
    ptx::grid_launch_dependents();  // a following decode step may begin its set-up
    ptx::grid_dependency_wait();    // launched behind the amax kernel: its maxima are complete
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
        s = a > 0.0f ? __fdiv_rn(a, I8 ? 127.0f : 448.0f) : 1.0f;
        if (t == 0 && part == 0) *sp = s;
    } else {
        s = *sp;
    }
    const uint4 v = __ldg(reinterpret_cast<const uint4*>((r.kv ? v_new : k_new) + (r.i * Hkv + r.h) * D + part * 8));
    quant_store<D, I8>(pool, v, s, blk, t, r.kv, r.h, part, Hkv, bs);
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads) fp8_reset_kernel(const int64_t* __restrict__ slots, int64_t N,
                                                                    int Hkv, int bs, int num_blocks,
                                                                    uint32_t* amax, uint8_t* fresh) {
    ptx::grid_launch_dependents();  // a following decode step may begin its set-up
    ptx::grid_dependency_wait();    // launched behind the quantising kernel: it has read the scratch
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

// One-pass quantising append for calls of up to kSmallAppendTokens tokens (a decode step appends
// one token per sequence): the same stored bytes and scales as the three passes above, in one
// launch.  One CTA per token, one thread per 8 elements of its K and V rows.  Every warp scans
// the call's slots for the other tokens landing in the token's block: if the call writes the
// block's offset 0 ("fresh"), the scale of each (K|V, head) row is amax/448 (amax/127 for int8)
// over the row and the same rows of those other tokens, which every token of the block computes
// alike; otherwise the stored scale is read (no token of this call writes it).  The usual decode
// step has no such other token, so a fresh block's scale comes from the token's own row.
// No shared memory; the slots are scanned with every thread's loads in flight at once.
constexpr int kSmallAppendTokens = 1024;
constexpr int kSmallThreads = 256;

template <int D, bool I8>
__global__ void __launch_bounds__(kSmallThreads, 4) quant_append_small_kernel(uint8_t* __restrict__ pool,
                                                                                float* __restrict__ scales,
                                                                                const uint16_t* __restrict__ k_new,
                                                                                const uint16_t* __restrict__ v_new,
                                                                                const int64_t* __restrict__ slots,
                                                                                int N, int Hkv, int bs, int num_blocks,
                                                                                int* err) {
    ptx::grid_launch_dependents();  // a following decode step may begin its set-up
    constexpr int TPR = D / 8;                 // threads per row (8 elements each)
    constexpr int RPC = kSmallThreads / TPR;   // rows per CTA pass
    constexpr int kPre = 2;                    // passes whose rows load before the slot scan
    const int i = blockIdx.x;  // this CTA's token
    const int tid = threadIdx.x, part = tid % TPR;
    const int rows = 2 * Hkv;
    auto row_src = [&](int r) {
        const int kv = r / Hkv, h = r - kv * Hkv;
        return reinterpret_cast<const uint4*>((kv ? v_new : k_new) + ((int64_t)i * Hkv + h) * D + part * 8);
    };
    uint4 pre[kPre];
#pragma unroll
    for (int ps = 0; ps < kPre; ++ps) {
        const int r = ps * RPC + tid / TPR;
        pre[ps] = r < rows ? __ldg(row_src(r)) : make_uint4(0u, 0u, 0u, 0u);
    }
    const int64_t cap = (int64_t)num_blocks * bs;
    const int bs_shift = __ffs(bs) - 1;  // block sizes are powers of two
    const int64_t slot = __ldg(slots + i);
    if (slot < 0) return;
    if (slot >= cap) {
        if (tid == 0) atomicOr(err, kErrBounds);
        return;
    }
    const int64_t blk = slot >> bs_shift;
    const int t = (int)(slot & (bs - 1));
    // other tokens of the call in this block, and whether the call writes the block's offset 0:
    // every thread checks slots tid, tid + kSmallThreads, ... (four loads in flight at a time)
    bool same = false, zero = false;
    for (int j0 = tid; j0 < N; j0 += 4 * kSmallThreads) {
        int64_t sj[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * kSmallThreads;
            sj[u] = (j < N && j != i) ? __ldg(slots + j) : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (sj[u] >= 0 && sj[u] < cap && (sj[u] >> bs_shift) == blk) {
                same = true;
                zero |= (sj[u] & (bs - 1)) == 0;
            }
        }
    }
    const bool mates = __syncthreads_or(same) != 0;
    const bool fresh = t == 0 || __syncthreads_or(zero) != 0;
    for (int ps = 0; ps * RPC < rows; ++ps) {  // CTA-uniform trip count
        const int r = ps * RPC + tid / TPR;
        const bool act = r < rows;
        const int kv = act ? r / Hkv : 0, h = act ? r - kv * Hkv : 0;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ps < kPre) {
#pragma unroll
            for (int q = 0; q < kPre; ++q)
                if (q == ps) v = pre[q];
        } else if (act) {
            v = __ldg(row_src(r));
        }
        float s = 1.0f;
        if (fresh) {
            uint32_t m = act ? amax_bits(v) : 0u;
            if (mates && act) {  // rare: several tokens of the call share the block
                const uint16_t* src = kv ? v_new : k_new;
                for (int j = 0; j < N; ++j) {
                    const int64_t sj = __ldg(slots + j);
                    if (j == i || sj < 0 || sj >= cap || (sj >> bs_shift) != blk) continue;
                    m = max(m, amax_bits(__ldg(reinterpret_cast<const uint4*>(src + ((int64_t)j * Hkv + h) * D +
                                                                                 part * 8))));
                }
            }
#pragma unroll
            for (int o = TPR / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float a = __uint_as_float(m);
            s = a > 0.0f ? __fdiv_rn(a, I8 ? 127.0f : 448.0f) : 1.0f;
            if (act && t == 0 && part == 0) scales[(blk * Hkv + h) * 4 + kv] = s;
        } else if (act) {
            s = scales[(blk * Hkv + h) * 4 + kv];
        }
        if (act) quant_store<D, I8>(pool, v, s, blk, t, kv, h, part, Hkv, bs);
    }
}

// ------------------------------------------------------------------ RoPE fused into the append
// Rotary position embedding ("TensorRT-LLM 深度实战" §3.3-3.4: RoPE fused with the attention's
// neighbours, use_fused_rope), in the Llama "rotate half" form: element d < D/2 pairs with
// d + D/2 and at position p the pair turns by p * base^(-2d/D):
//     y[d] = x[d] cos - x[d + D/2] sin,   y[d + D/2] = x[d + D/2] cos + x[d] sin.
// The result is the fp64 rotation (products and sums rounded separately) rounded once to bf16,
// nearest-even; most elements get there through an fp32 computation whose error bound shows
// the rounding cannot differ (see rope_elem).

struct RopeTable {
    double inv_freq[64];  // base^(-2d/D), d < D/2, computed on the host
};

// fp64 -> bf16 bits, round to nearest, ties to even (bf16: 8 significant bits, fp32's exponent
// range, subnormals with unit 2^-133).
__device__ __forceinline__ uint32_t f64_to_bf16_rn(double x) {
    const uint64_t b = (uint64_t)__double_as_longlong(x);
    const uint32_t sign = (uint32_t)(b >> 48) & 0x8000u;
    const int ex = (int)((b >> 52) & 0x7ff);
    const uint64_t man = b & ((1ull << 52) - 1);
    if (ex == 0x7ff) return sign | 0x7f80u | (man ? 0x40u : 0u);  // inf / nan
    if (ex == 0) return sign;                                      // zero or far below bf16's range
    const int e = ex - 1023;                                       // leading bit weight 2^e
    const uint64_t m = (1ull << 52) | man;                         // 53-bit significand
    // number of low significand bits dropped: 45 for normal bf16, more below 2^-126
    const int sh = e >= -126 ? 45 : 45 + (-126 - e);
    if (sh > 54) return sign;  // below half the smallest subnormal
    const uint64_t q = m >> sh, rem = m & ((1ull << sh) - 1), half = 1ull << (sh - 1);
    const uint64_t k = q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0);
    if (e >= -126) {
        // k in [2^7, 2^8]; 2^8 carries into the exponent
        const int be = e + 127 + (k >> 8 ? 1 : 0);
        if (be >= 255) return sign | 0x7f80u;
        return sign | ((uint32_t)be << 7) | (uint32_t)((k >> 8 ? k >> 1 : k) & 0x7f);
    }
    return sign | (uint32_t)k;  // subnormal (k = 2^7 is the smallest normal, 0x0080)
}

// Rotated element, correctly rounded to bf16.  c64/s64 are the fp64 cosine and sine of the
// element's angle and c32/s32 their fp32 roundings (|c32 - c64| <= 2^-25).  Fast path in fp32:
// with the fp32 product and the fused subtraction, the error of y32 against the fp64 rotation
// is below |x| 2^-25 + |xo| 2^-25 + (|xo| + |y|) 2^-24 <= 3 m 2^-24 = E, m = |x| + |xo|.  If y32
// lies farther than E from the bf16 rounding midpoint between its neighbours, the fp64 value
// rounds the same way and the fp32 result is final.  Otherwise (rare: a near tie, heavy
// cancellation, a tiny or non-normal result) the fp64 rotation is computed and rounded.
__device__ __forceinline__ uint32_t rope_elem(float x, float xo, bool first, float c32, float s32, double c64,
                                              double s64) {
    const float p = xo * s32;
    const float y = first ? fmaf(x, c32, -p) : fmaf(x, c32, p);
    const uint32_t yb = __float_as_uint(y);
    const uint32_t ex = (yb >> 23) & 0xffu;
    if (ex > 1u && ex < 254u) {
        // distance to the midpoint in units of y's fp32 ulp (>= |y| 2^-24), against
        // E / ulp <= 3 m / |y| plus slack, compared without dividing
        const float dist = fabsf((float)(int)(yb & 0xffffu) - 32768.0f);
        const float m = fabsf(x) + fabsf(xo), ay = fabsf(y);
        if ((dist - 4.0f) * ay > 3.0f * m && 3.0f * m < 8000.0f * ay)
            return (yb + 0x7fffu + ((yb >> 16) & 1u)) >> 16;  // RNE to bf16, sign kept
    }
    const double xa = (double)x, xb = (double)xo;
    const double v = first ? __dsub_rn(__dmul_rn(xa, c64), __dmul_rn(xb, s64)) : __dadd_rn(__dmul_rn(xa, c64), __dmul_rn(xb, s64));
    return f64_to_bf16_rn(v);
}

// One CTA per token.  Rows of the token: the Hkv K heads (rotated in place in k_new and, when
// the pool is bf16, written into the token's slot), the Hkv V heads (bf16 pool: copied into the
// slot), the Hq query heads (rotated in place).  A row is D/8 threads of 8 elements; the
// partner half of a pair is exchanged by warp shuffle, so rows are rotated in place safely.
template <int D, bool POOL>
__global__ void __launch_bounds__(128) rope_append_kernel(uint16_t* __restrict__ pool, uint16_t* __restrict__ k_new,
                                                          const uint16_t* __restrict__ v_new,
                                                          const int64_t* __restrict__ slots,
                                                          const int64_t* __restrict__ pos, uint16_t* __restrict__ q,
                                                          int Hq, int Hkv, int bs, int num_blocks, int* err,
                                                          const RopeTable tab) {
    ptx::grid_launch_dependents();  // a following attention kernel may begin its set-up
    constexpr int TPR = D / 8;
    constexpr double kTwoPiHi = 6.283185307179586, kTwoPiLo = 2.4492935982947064e-16;  // 2 pi = hi + lo
    __shared__ double c64_s[D / 2], s64_s[D / 2];
    __shared__ float c_s[D / 2], s_s[D / 2];
    const int64_t i = blockIdx.x;
    const double pp = (double)__ldg(pos + i);
    for (int d = threadIdx.x; d < D / 2; d += blockDim.x) {
        const double th = __dmul_rn(pp, tab.inv_freq[d]);
        // reduce to [-pi, pi] first: th - k (2 pi) with 2 pi split in two terms, so the sine and
        // cosine stay on their short path (the reduction error is a few fp64 ulps of the result)
        const double k = rint(th * (1.0 / kTwoPiHi));
        const double r = fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, th));
        double sn, cn;
        sincos(r, &sn, &cn);
        c64_s[d] = cn;
        s64_s[d] = sn;
        c_s[d] = (float)cn;
        s_s[d] = (float)sn;
    }
    __syncthreads();
    int64_t slot = -1;
    if (POOL) {
        slot = __ldg(slots + i);
        if (slot >= (int64_t)num_blocks * bs) {
            if (threadIdx.x == 0) atomicOr(err, kErrBounds);
            slot = -1;
        }
    }
    const int rows = Hkv + (POOL ? Hkv : 0) + (q ? Hq : 0);
    const int part = (int)threadIdx.x % TPR;
    for (int base = 0; base < rows * TPR; base += blockDim.x) {  // same trip count for every thread
        const int task = base + (int)threadIdx.x;
        const bool active = task < rows * TPR;
        const int r = task / TPR;
        // row kind: 0 = K head, 1 = V head, 2 = query head
        const int kind = r < Hkv ? 0 : (POOL && r < 2 * Hkv ? 1 : 2);
        const int head = kind == 0 ? r : (kind == 1 ? r - Hkv : r - (POOL ? 2 * Hkv : Hkv));
        uint16_t* row = kind == 0 ? k_new + (i * Hkv + head) * D : (kind == 2 ? q + (i * Hq + head) * D : nullptr);
        uint4 own = make_uint4(0, 0, 0, 0);
        if (active) own = kind == 1 ? __ldg(reinterpret_cast<const uint4*>(v_new + (i * Hkv + head) * D) + part)
                                    : *(reinterpret_cast<const uint4*>(row) + part);
        uint4 oth;  // the other half of each pair: lane +- TPR/2 within the row
        oth.x = __shfl_xor_sync(0xffffffffu, own.x, TPR / 2);
        oth.y = __shfl_xor_sync(0xffffffffu, own.y, TPR / 2);
        oth.z = __shfl_xor_sync(0xffffffffu, own.z, TPR / 2);
        oth.w = __shfl_xor_sync(0xffffffffu, own.w, TPR / 2);
        if (!active) continue;
        uint4 res = own;
        if (kind != 1) {
            const bool first = part < TPR / 2;
            const uint32_t a[4] = {own.x, own.y, own.z, own.w}, o[4] = {oth.x, oth.y, oth.z, oth.w};
            uint32_t y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int d0 = (part * 8 + 2 * e) % (D / 2);
                const uint32_t lo = rope_elem(ptx::bf16lo_to_f32(a[e]), ptx::bf16lo_to_f32(o[e]), first, c_s[d0],
                                              s_s[d0], c64_s[d0], s64_s[d0]);
                const uint32_t hi = rope_elem(ptx::bf16hi_to_f32(a[e]), ptx::bf16hi_to_f32(o[e]), first, c_s[d0 + 1],
                                              s_s[d0 + 1], c64_s[d0 + 1], s64_s[d0 + 1]);
                y[e] = (lo & 0xffffu) | (hi << 16);
            }
            res = make_uint4(y[0], y[1], y[2], y[3]);
            *(reinterpret_cast<uint4*>(row) + part) = res;
        }
        if (POOL && kind != 2 && slot >= 0) {
            const int64_t blk = slot / bs;
            const int t = (int)(slot - blk * bs);
            *reinterpret_cast<uint4*>(pool + tile_elem(blk, kind, head, Hkv, bs, D) + (int64_t)t * D + part * 8) = res;
        }
    }
}

// Launch `kernel` on `st` as a programmatic dependent of the preceding kernel on the stream: it
// may be scheduled while that one runs and must execute griddepcontrol.wait before reading what
// that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kAppendThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
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
    } else if (N <= kSmallAppendTokens) {
        // one pass: a CTA per token
        const dim3 g1((unsigned)N);
        uint8_t* const kv8 = static_cast<uint8_t*>(p->kv);
        if (p->dtype == PKV_KV_INT8)
            quant_append_small_kernel<D, true><<<g1, kSmallThreads, 0, st>>>(kv8, p->scales, k, v, slots, (int)N,
                                                                           p->n_kv_heads, p->block_size,
                                                                           p->num_blocks, p->err);
        else
            quant_append_small_kernel<D, false><<<g1, kSmallThreads, 0, st>>>(kv8, p->scales, k, v, slots, (int)N,
                                                                            p->n_kv_heads, p->block_size,
                                                                            p->num_blocks, p->err);
    } else {
        // three kernels in a chain of programmatic dependents: the amax kernel waits for the
        // stream as usual; the quantising kernel and the reset are scheduled while their
        // predecessor runs and wait for it before touching the scratch (a decode attention
        // launched behind the reset waits for it in turn, which covers the quantised bytes)
        fp8_amax_kernel<D><<<grid, kAppendThreads, 0, st>>>(k, v, slots, N, p->n_kv_heads, p->block_size,
                                                            p->num_blocks, p->amax_scratch, p->fresh_scratch, p->err);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
        uint8_t* const kv8 = static_cast<uint8_t*>(p->kv);
        const uint32_t* const amax = p->amax_scratch;
        const uint8_t* const fresh = p->fresh_scratch;
        cudaError_t e = p->dtype == PKV_KV_INT8
                            ? launch_dependent(fp8_quant_kernel<D, true>, grid, st, kv8, p->scales, k, v, slots, N,
                                               p->n_kv_heads, p->block_size, p->num_blocks, amax, fresh)
                            : launch_dependent(fp8_quant_kernel<D, false>, grid, st, kv8, p->scales, k, v, slots, N,
                                               p->n_kv_heads, p->block_size, p->num_blocks, amax, fresh);
        if (e != cudaSuccess) return PKV_ERR_CUDA;
        e = launch_dependent(fp8_reset_kernel<D>, grid, st, slots, N, p->n_kv_heads, p->block_size, p->num_blocks,
                             p->amax_scratch, p->fresh_scratch);
        if (e != cudaSuccess) return PKV_ERR_CUDA;
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

namespace pkv {

pkv_status append_rope_launch(pkv_pool* pool, void* k_new, const void* v_new, const int64_t* slot_mapping,
                              const int64_t* positions, int64_t N, double rope_base, void* q, int n_q_heads,
                              cudaStream_t cs) {
    pkv_status st = append_check(pool, k_new, v_new, slot_mapping, N);
    if (st != PKV_OK) return st;
    if (!(rope_base > 1.0) || !std::isfinite(rope_base)) return PKV_ERR_INVALID_ARG;
    if (N == 0) return PKV_OK;
    if (!positions || (reinterpret_cast<uintptr_t>(positions) & 7u)) return PKV_ERR_INVALID_ARG;
    if (q && (n_q_heads < 1 || (reinterpret_cast<uintptr_t>(q) & 15u))) return PKV_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    const int D = pool->head_dim;
    RopeTable tab;
    for (int d = 0; d < 64; ++d) tab.inv_freq[d] = d < D / 2 ? std::pow(rope_base, -2.0 * d / D) : 0.0;
    auto* k = static_cast<uint16_t*>(k_new);
    const auto* v = static_cast<const uint16_t*>(v_new);
    auto* qq = static_cast<uint16_t*>(q);
    const bool bf16 = pool->dtype == PKV_KV_BF16;
    const dim3 grid((unsigned)N);
    auto* kv = static_cast<uint16_t*>(pool->kv);
#define PKV_ROPE(DD, PP)                                                                                           \
    rope_append_kernel<DD, PP><<<grid, 128, 0, cs>>>(kv, k, v, slot_mapping, positions, qq, q ? n_q_heads : 0,      \
                                                     pool->n_kv_heads, pool->block_size, pool->num_blocks, pool->err, \
                                                     tab)
    if (D == 128) {
        if (bf16) PKV_ROPE(128, true); else PKV_ROPE(128, false);
    } else {
        if (bf16) PKV_ROPE(64, true); else PKV_ROPE(64, false);
    }
#undef PKV_ROPE
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    if (bf16) return PKV_OK;
    // low-precision pools: the rotated K rows in k_new go through the regular quantising append
    return D == 128 ? launch_append<128>(pool, k, v, slot_mapping, N, cs) : launch_append<64>(pool, k, v, slot_mapping, N, cs);
}

}  // namespace pkv

extern "C" pkv_status pkv_append_rope(pkv_pool* pool, void* k_new, const void* v_new, const int64_t* slot_mapping,
                                      const int64_t* positions, int64_t N, double rope_base, void* q, int n_q_heads,
                                      pkv_stream_t stream) {
    return pkv::append_rope_launch(pool, k_new, v_new, slot_mapping, positions, N, rope_base, q, n_q_heads,
                                   reinterpret_cast<cudaStream_t>(stream));
}

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
