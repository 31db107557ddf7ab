// Element codes of one-byte pools, shared by the appends and the decode step that quantises its
// new tokens itself.
//
// fp8 pools ("TensorRT-LLM 深度实战" §4.5 E4M3; "TensorRT-LLM 推理加速实战" §8 fp8_e4m3 KV
// cache) and int8 pools (symmetric codes): an element is stored as the code of x / s, with s the
// fp32 scale of its (block, K|V, head) and the quotient an IEEE fp32 division.  The pool layout
// (pkv.h): K rows [bs][D] of codes per (block, head); V in 16-token panels [D][16], the tokens of
// a panel row in the pair order of the attention's MMA.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace pkv {
namespace quant {

__device__ __forceinline__ int64_t tile_elem(int64_t blk, int kv, int h, int Hkv, int bs, int D) {
    return ((blk * 2 + kv) * Hkv + h) * (int64_t)bs * D;
}

// Position of token u (0..15) inside a 16-byte fp8 V panel row (pair order of the MMA).
__device__ __forceinline__ int fp8_v_pos(int u) { return u < 8 ? 4 * (u >> 1) + (u & 1) : 4 * ((u - 8) >> 1) + 2 + (u & 1); }

// max |x| over eight bf16 elements, as fp32 bits (non-negative floats order like their bits)
__device__ __forceinline__ uint32_t amax_bits(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t lo = (w[e] << 16) & 0x7fffffffu, hi = w[e] & 0x7fff0000u;
        m = max(m, max(lo, hi));
    }
    return m;
}

// INT8 code of a quotient x / scale: nearest integer, ties to even (cvt.rni), clamped to
// [-127, 127] (symmetric: -128 is never produced); the byte in the low 8 bits.
__device__ __forceinline__ uint32_t int8_code(float q) {
    const int c = __float2int_rn(q);
    return (uint32_t)(c < -127 ? -127 : (c > 127 ? 127 : c)) & 0xffu;
}

// Quantise eight elements (part `part` of a row: elements 8*part .. 8*part+7) of token slot t of
// block blk, K (kv = 0) or V (kv = 1) of head h, with scale s: x / s as an IEEE fp32 division, then
// E4M3 round-to-nearest-even with saturation (or the int8 code), stored in the pool's layout.
template <int D, bool I8>
__device__ __forceinline__ void quant_store(uint8_t* __restrict__ pool, uint4 v, float s, int64_t blk, int t, int kv,
                                            int h, int part, int Hkv, int bs) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t codes[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float x0 = __fdiv_rn(ptx::bf16lo_to_f32(w[2 * e]), s), x1 = __fdiv_rn(ptx::bf16hi_to_f32(w[2 * e]), s);
        const float x2 = __fdiv_rn(ptx::bf16lo_to_f32(w[2 * e + 1]), s),
                    x3 = __fdiv_rn(ptx::bf16hi_to_f32(w[2 * e + 1]), s);
        if constexpr (I8)
            codes[e] = int8_code(x0) | (int8_code(x1) << 8) | (int8_code(x2) << 16) | (int8_code(x3) << 24);
        else
            codes[e] = ptx::f32x2_to_e4m3x2(x0, x1) | (ptx::f32x2_to_e4m3x2(x2, x3) << 16);
    }
    uint8_t* tile = pool + tile_elem(blk, kv, h, Hkv, bs, D);
    if (kv == 0) {
        *reinterpret_cast<uint2*>(tile + (int64_t)t * D + part * 8) = make_uint2(codes[0], codes[1]);
    } else {
        uint8_t* panel = tile + (int64_t)(t >> 4) * D * 16 + fp8_v_pos(t & 15);
#pragma unroll
        for (int e = 0; e < 8; ++e) panel[(int64_t)(part * 8 + e) * 16] = (uint8_t)(codes[e >> 2] >> (8 * (e & 3)));
    }
}

}  // namespace quant
}  // namespace pkv
