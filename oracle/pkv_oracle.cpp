// Paged-KV decode attention: CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, the package smoke check and the
// benchmark's CPU-baseline / reference leg may load or call this code.  It shares
// no code, header, table or helper with the CUDA library; it is written from the
// pages and the published format definitions, plainly and slowly, in fp64.
//
// Sources (page title, section):
//  * Allocator: "TensorRT-LLM 深度实战" (chenxutan.com), §3.1 Paged KV Cache — a
//    free-page list initialised to 0..n-1, pages taken with pop() from its end,
//    ceil(num_tokens/page_size) pages per request, growth by whole pages when the
//    tokens outgrow capacity, and release appending a finished sequence's pages
//    back in table order.  Out-of-memory leaves the pool unchanged here (the
//    page's sketch leaks already-popped pages; that is a bug, not the method).
//  * Block size choices 16/64: "TensorRT-LLM 推理加速实战" (socake.github.io), §8.
//  * KV memory: same page §8.1 (kv_bytes_per_token = 2 x layers x kv_heads x
//    head_dim x bytes) and the aiqz.cc page, KV缓存管理 (M_kv = 2 n_layers n_heads
//    d_head n_tokens b bytes, with n_heads read as the number of KV heads).
//  * FP8 E4M3 KV cache: "TensorRT-LLM 深度实战" §4.5 (E4M3: 4 exponent, 3 mantissa
//    bits) and "TensorRT-LLM 推理加速实战" §4.1/§8 (fp8_e4m3 KV cache).  Encoding and
//    decoding follow the OCP 8-bit floating point specification (OFP8): bias 7, no
//    infinities, S.1111.111 is NaN, largest finite 448; conversion rounds to
//    nearest-even and saturates to +-448 (satfinite).
//  * Decode attention: "TensorRT-LLM 推理加速实战" §7.2 (masked_mha: one new token
//    attends to the request's cached K/V) — computed here by its definition,
//    out = softmax(scale * q K^T) V over the gathered sequence, per query head,
//    query head j using KV head j / (Hq/Hkv) (GQA sharing, "TensorRT-LLM加速大模型
//    推理实战", csdn page).
//  * Split merge: per-chunk running max m, sum l and weighted sum o merged with
//    M = max m_s, l = sum l_s e^(m_s - M), out = sum e^(m_s - M) o_s / l.
//  * Block reuse: pnsm.cn TensorRT-LLM page §3.1 (enable_block_reuse) and "TensorRT-LLM
//    推理加速实战" §8 (KV cache reuse) — a forked sequence holds its source's whole prefix
//    pages (holder counts), a copy of the partial last one, and pages return to the free
//    list when their last holder releases them.
//  * RoPE fused into the append: "TensorRT-LLM 深度实战" §3.3-3.4 (use_fused_rope), the
//    Llama "rotate half" form (see the function).
//  * Prefill (chunked-context) attention: "TensorRT-LLM 深度实战" §7.3 and "TensorRT-LLM
//    推理加速实战" §7.2 (context_fmha) — every query of a chunk is the decode definition over
//    the tokens up to and including its own position.
//
// Pool byte layout (the storage contract both sides implement independently):
//   tile(blk, kv, h) starts at byte ((blk*2 + kv)*Hkv + h) * bs * D * esz,
//   kv = 0 for K, 1 for V, esz = 2 (bf16) or 1 (fp8, int8).  The `fp8` argument of the pool
//   functions is the element code: 0 bf16, 1 fp8 e4m3, 2 int8 (both 1-byte codes share the layout).
//   bf16 K and V, fp8/int8 K: row-major [bs][D].
//   fp8/int8 V: bs/16 column panels, each [D][16]: (t, d) at (t/16)*D*16 + d*16 + pos(t%16), where
//   a panel row stores its 16 tokens in the order 0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15.
//   fp8 scales: float[num_blocks][Hkv][4]: [.., 0] K scale, [.., 1] V scale.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <unordered_map>
#include <vector>

namespace {

struct Allocator {
    int num_blocks;
    int block_size;
    std::vector<int32_t> free_pages;                          // pop() from the back
    std::unordered_map<int64_t, std::vector<int32_t>> table;  // seq -> pages
    std::vector<int> holders;                                 // sequences holding each page
};

double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

}  // namespace

extern "C" {

// ----------------------------------------------------------------- allocator
void* oracle_alloc_new(int num_blocks, int block_size) {
    Allocator* a = new Allocator();
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    for (int i = 0; i < num_blocks; ++i) a->free_pages.push_back(i);
    a->holders.assign(num_blocks, 0);
    return a;
}

void oracle_alloc_delete(void* p) { delete (Allocator*)p; }

// Replace the free list by `order` (a permutation of 0..n-1); only when nothing is held.
int oracle_alloc_set_free_order(void* p, const int32_t* order, int n) {
    Allocator* a = (Allocator*)p;
    if (!a->table.empty() || n != a->num_blocks) return 1;
    std::vector<int> seen(n, 0);
    for (int i = 0; i < n; ++i) {
        if (order[i] < 0 || order[i] >= n || seen[order[i]]) return 1;
        seen[order[i]] = 1;
    }
    a->free_pages.assign(order, order + n);
    return 0;
}

// Give seq capacity for n_tokens tokens: a new sequence takes ceil(n/bs) pages; a known one
// takes enough extra pages for the tokens beyond its capacity.  0 ok, 2 out of pages.
int oracle_alloc_reserve(void* p, int64_t seq, int64_t n_tokens) {
    Allocator* a = (Allocator*)p;
    if (n_tokens < 0) return 1;
    auto it = a->table.find(seq);
    int64_t have = (it == a->table.end()) ? 0 : (int64_t)it->second.size();
    int64_t capacity = have * a->block_size;
    int64_t need = 0;
    if (n_tokens > capacity) need = (n_tokens - capacity + a->block_size - 1) / a->block_size;
    if (need > (int64_t)a->free_pages.size()) return 2;
    std::vector<int32_t>& pages = a->table[seq];
    for (int64_t i = 0; i < need; ++i) {
        pages.push_back(a->free_pages.back());
        a->holders[a->free_pages.back()] = 1;
        a->free_pages.pop_back();
    }
    return 0;
}

int oracle_alloc_release(void* p, int64_t seq) {
    Allocator* a = (Allocator*)p;
    auto it = a->table.find(seq);
    if (it == a->table.end()) return 3;
    // a page goes back to the free list when its last holder lets go (pages in table order)
    for (int32_t page : it->second) {
        a->holders[page] -= 1;
        if (a->holders[page] == 0) a->free_pages.push_back(page);
    }
    a->table.erase(it);
    return 0;
}

// Block reuse (pnsm.cn page §3.1 enable_block_reuse; "TensorRT-LLM 推理加速实战" §8 KV cache reuse,
// like prefix caching), in this reading: dst starts with src's first n tokens; src's full pages
// among them are shared; a prefix ending inside a page gets a fresh page that the caller fills
// with a copy of src's page.  Returns 0, 3 (no src), 1 (dst exists), 4 (n beyond src), 2 (no page).
int oracle_alloc_share_prefix(void* p, int64_t src, int64_t dst, int64_t n, int32_t* cow_src, int32_t* cow_dst) {
    Allocator* a = (Allocator*)p;
    auto it = a->table.find(src);
    if (it == a->table.end()) return 3;
    if (a->table.count(dst) || src == dst) return 1;
    if (n < 0 || n > (int64_t)it->second.size() * a->block_size) return 4;
    int64_t full = n / a->block_size;
    bool partial = n % a->block_size != 0;
    if (partial && a->free_pages.empty()) return 2;
    std::vector<int32_t> pages;
    for (int64_t k = 0; k < full; ++k) {
        pages.push_back(it->second[k]);
        a->holders[it->second[k]] += 1;
    }
    *cow_src = -1;
    *cow_dst = -1;
    if (partial) {
        int32_t page = a->free_pages.back();
        a->free_pages.pop_back();
        a->holders[page] = 1;
        *cow_src = it->second[full];
        *cow_dst = page;
        pages.push_back(page);
    }
    a->table[dst] = pages;
    return 0;
}

int oracle_alloc_holders(void* p, int32_t page) { return ((Allocator*)p)->holders[page]; }

int oracle_alloc_num_free(void* p) { return (int)((Allocator*)p)->free_pages.size(); }

int oracle_alloc_num_pages(void* p, int64_t seq) {
    Allocator* a = (Allocator*)p;
    auto it = a->table.find(seq);
    return it == a->table.end() ? -1 : (int)it->second.size();
}

// Copy the free list (back = next page handed out) into out[0..num_free).
void oracle_alloc_free_list(void* p, int32_t* out) {
    Allocator* a = (Allocator*)p;
    for (size_t i = 0; i < a->free_pages.size(); ++i) out[i] = a->free_pages[i];
}

// block_tables[B][max_blocks], -1 beyond each sequence's pages.
int oracle_alloc_block_tables(void* p, const int64_t* seqs, int B, int max_blocks, int32_t* out) {
    Allocator* a = (Allocator*)p;
    for (int b = 0; b < B; ++b) {
        auto it = a->table.find(seqs[b]);
        if (it == a->table.end()) return 3;
        if ((int)it->second.size() > max_blocks) return 1;
        for (int k = 0; k < max_blocks; ++k)
            out[(int64_t)b * max_blocks + k] = k < (int)it->second.size() ? it->second[k] : -1;
    }
    return 0;
}

// slot = page[pos / bs] * bs + pos % bs; a negative position maps to slot -1.
int oracle_alloc_slot_mapping(void* p, const int64_t* seqs, const int64_t* pos, int64_t N, int64_t* out) {
    Allocator* a = (Allocator*)p;
    for (int64_t i = 0; i < N; ++i) {
        if (pos[i] < 0) {
            out[i] = -1;
            continue;
        }
        auto it = a->table.find(seqs[i]);
        if (it == a->table.end()) return 3;
        int64_t k = pos[i] / a->block_size;
        if (k >= (int64_t)it->second.size()) return 5;
        out[i] = (int64_t)it->second[k] * a->block_size + pos[i] % a->block_size;
    }
    return 0;
}

// ----------------------------------------------------------------- KV memory
// M_kv = 2 * n_layers * n_kv_heads * d_head * n_tokens * batch * bytes_per_element.
double oracle_m_kv(double n_layers, double n_kv_heads, double d_head, double n_tokens, double batch,
                   double bytes) {
    return 2.0 * n_layers * n_kv_heads * d_head * n_tokens * batch * bytes;
}

// ----------------------------------------------------------------- E4M3 (OCP OFP8)
double oracle_e4m3_decode(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 0xf, m = code & 0x7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? std::ldexp((double)m / 8.0, 1 - 7) : std::ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

// Round-to-nearest-even onto the E4M3 grid with saturation to +-448, by exhaustive search:
// the nearest of the 127 non-negative finite codes, ties to the code with an even mantissa.
uint8_t oracle_e4m3_encode_exhaustive(float x) {
    if (std::isnan(x)) return 0x7f;
    double ax = std::fabs((double)x);
    uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    if (ax >= 448.0) return sign | 0x7e;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        double err = std::fabs(oracle_e4m3_decode((uint8_t)c) - ax);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

// The same rounding, faster: non-negative finite codes increase with their value, so the
// nearest code is one of the two neighbours of |x| on the grid.
uint8_t oracle_e4m3_encode(float x) {
    if (std::isnan(x)) return 0x7f;
    double ax = std::fabs((double)x);
    uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    if (ax >= 448.0) return sign | 0x7e;
    int lo = 0, hi = 0x7e;  // largest code whose value is <= ax
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_decode((uint8_t)mid) <= ax) lo = mid; else hi = mid - 1;
    }
    int c = lo;
    if (c < 0x7e) {
        double below = ax - oracle_e4m3_decode((uint8_t)c);
        double above = oracle_e4m3_decode((uint8_t)(c + 1)) - ax;
        if (above < below || (above == below && ((c + 1) & 1) == 0)) c = c + 1;
    }
    return sign | (uint8_t)c;
}

void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* out, int exhaustive) {
    for (int64_t i = 0; i < n; ++i) out[i] = exhaustive ? oracle_e4m3_encode_exhaustive(x[i]) : oracle_e4m3_encode(x[i]);
}

// ----------------------------------------------------------------- pool layout
static int64_t tile_base(int64_t blk, int kv, int h, int Hkv, int bs, int D, int esz) {
    return (((blk * 2 + kv) * Hkv + h) * (int64_t)bs * D) * esz;
}

// Byte position of token u (0..15) inside a 16-byte fp8 V panel row: tokens are stored in
// the order 0,1,8,9, 2,3,10,11, 4,5,12,13, 6,7,14,15.
static int fp8_v_byte(int u) { return u < 8 ? 4 * (u >> 1) + (u & 1) : 4 * ((u - 8) >> 1) + 2 + (u & 1); }

static int64_t elem_offset(int kv, int t, int d, int bs, int D, int fp8) {
    (void)bs;
    if (fp8 && kv == 1) return (int64_t)(t / 16) * D * 16 + (int64_t)d * 16 + fp8_v_byte(t % 16);
    return (int64_t)t * D + d;
}

// Read K (kv=0) or V (kv=1) element (t in block, d) of block blk, head h, as fp64.
static double pool_value(const uint8_t* pool, const float* scales, int64_t blk, int kv, int h, int t, int d, int Hkv,
                         int bs, int D, int fp8) {
    int esz = fp8 ? 1 : 2;
    int64_t base = tile_base(blk, kv, h, Hkv, bs, D, esz);
    int64_t off = elem_offset(kv, t, d, bs, D, fp8);
    if (!fp8) {
        uint16_t b;
        std::memcpy(&b, pool + base + off * 2, 2);
        return bf16_to_double(b);
    }
    double s = (double)scales[(blk * Hkv + h) * 4 + kv];
    if (fp8 == 2) return (double)(int8_t)pool[base + off] * s;  // INT8 code times its scale
    return oracle_e4m3_decode(pool[base + off]) * s;
}

// ----------------------------------------------------------------- INT8 KV
// INT8 KV cache (a NEXT variant; the pages list INT8 among TensorRT-LLM's quantisation formats,
// pnsm.cn page §1.2, "TensorRT-LLM 深度实战" §4): symmetric codes with the same per-(block,
// K|V, head) scale semantics as the fp8 cache, the scale being amax/127.  A quotient q = x / s
// (fp32) becomes round-to-nearest-even(q) clamped to [-127, 127]; the value read back is
// code * s.
int8_t oracle_int8_encode(float q) {
    if (std::isnan(q)) return 0;
    double r = std::nearbyint((double)q);  // the default rounding mode: ties to even
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int8_t)r;
}

void oracle_int8_encode_array(const float* q, int64_t n, int8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_int8_encode(q[i]);
}

// ----------------------------------------------------------------- append
// Write each token's K and V rows (bf16 bit patterns, [N][Hkv][D]) into its slot.
// bf16 pools store the bits.  fp8 (dtype code 1) and int8 (code 2) pools: for every (block,
// K|V, head) whose offset 0 is written by this call, the scale becomes amax/448 (int8: /127)
// over this call's tokens in that block (1.0 if amax is 0); other blocks keep their stored
// scale; codes are e4m3(x / scale) or int8(x / scale) with an fp32 division.  Slots < 0 are
// skipped.  Returns 0, or 4 for a slot beyond the pool.
int oracle_append(uint8_t* pool, float* scales, int num_blocks, int bs, int Hkv, int D, int fp8,
                  const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots, int64_t N) {
    for (int64_t i = 0; i < N; ++i)
        if (slots[i] >= (int64_t)num_blocks * bs) return 4;
    const uint16_t* src[2] = {k_new, v_new};
    if (!fp8) {
        for (int64_t i = 0; i < N; ++i) {
            if (slots[i] < 0) continue;
            int64_t blk = slots[i] / bs;
            int t = (int)(slots[i] % bs);
            // bf16 tiles are row-major [bs][D]: a token's row for one head is D contiguous elements
            for (int kv = 0; kv < 2; ++kv)
                for (int h = 0; h < Hkv; ++h)
                    std::memcpy(pool + tile_base(blk, kv, h, Hkv, bs, D, 2) + elem_offset(kv, t, 0, bs, D, 0) * 2,
                                src[kv] + (i * Hkv + h) * D, (size_t)D * 2);
        }
        return 0;
    }
    // blocks whose first slot this call writes
    std::vector<char> fresh(num_blocks, 0);
    for (int64_t i = 0; i < N; ++i)
        if (slots[i] >= 0 && slots[i] % bs == 0) fresh[slots[i] / bs] = 1;
    // amax over this call's tokens in each fresh block, per (K|V, head)
    std::vector<float> amax((size_t)num_blocks * Hkv * 2, 0.0f);
    for (int64_t i = 0; i < N; ++i) {
        if (slots[i] < 0 || !fresh[slots[i] / bs]) continue;
        int64_t blk = slots[i] / bs;
        for (int kv = 0; kv < 2; ++kv)
            for (int h = 0; h < Hkv; ++h)
                for (int d = 0; d < D; ++d) {
                    float x = (float)bf16_to_double(src[kv][(i * Hkv + h) * D + d]);
                    float& a = amax[(blk * Hkv + h) * 2 + kv];
                    a = std::max(a, std::fabs(x));
                }
    }
    for (int64_t blk = 0; blk < num_blocks; ++blk) {
        if (!fresh[blk]) continue;
        for (int h = 0; h < Hkv; ++h)
            for (int kv = 0; kv < 2; ++kv) {
                float a = amax[(blk * Hkv + h) * 2 + kv];
                scales[(blk * Hkv + h) * 4 + kv] = a > 0.0f ? a / (fp8 == 2 ? 127.0f : 448.0f) : 1.0f;
            }
    }
    for (int64_t i = 0; i < N; ++i) {
        if (slots[i] < 0) continue;
        int64_t blk = slots[i] / bs;
        int t = (int)(slots[i] % bs);
        for (int kv = 0; kv < 2; ++kv)
            for (int h = 0; h < Hkv; ++h) {
                float s = scales[(blk * Hkv + h) * 4 + kv];
                for (int d = 0; d < D; ++d) {
                    float x = (float)bf16_to_double(src[kv][(i * Hkv + h) * D + d]);
                    pool[tile_base(blk, kv, h, Hkv, bs, D, 1) + elem_offset(kv, t, d, bs, D, 1)] =
                        fp8 == 2 ? (uint8_t)oracle_int8_encode(x / s) : oracle_e4m3_encode(x / s);
                }
            }
    }
    return 0;
}

// ----------------------------------------------------------------- attention
// Dense attention for one KV head's query group, straight from the definition.
// q [G][D], K and V [L][D] (fp64), out [G][D]; L == 0 gives zeros.
void oracle_dense_attention(const double* q, const double* K, const double* V, int64_t L, int D, int G, double scale,
                            double* out) {
    std::vector<double> z((size_t)L);
    for (int j = 0; j < G; ++j) {
        for (int d = 0; d < D; ++d) out[(int64_t)j * D + d] = 0.0;
        if (L == 0) continue;
        double m = -INFINITY;
        for (int64_t t = 0; t < L; ++t) {
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += q[(int64_t)j * D + d] * K[t * D + d];
            z[t] = scale * s;
            m = std::max(m, z[t]);
        }
        double l = 0.0;
        for (int64_t t = 0; t < L; ++t) {
            z[t] = std::exp(z[t] - m);
            l += z[t];
        }
        for (int64_t t = 0; t < L; ++t)
            for (int d = 0; d < D; ++d) out[(int64_t)j * D + d] += z[t] * V[t * D + d];
        for (int d = 0; d < D; ++d) out[(int64_t)j * D + d] /= l;
    }
}

// Gather sequence b's K and V for KV head h into contiguous [L][D] fp64 arrays by walking its
// block table: token t lives in block tables[b][t / bs] at offset t % bs.
static int gather(const uint8_t* pool, const float* scales, int num_blocks, int bs, int Hkv, int D, int fp8,
                  const int32_t* tables, int max_blocks, int b, int h, int64_t L, std::vector<double>& K,
                  std::vector<double>& V) {
    K.assign((size_t)L * D, 0.0);
    V.assign((size_t)L * D, 0.0);
    for (int64_t t = 0; t < L; ++t) {
        int64_t k = t / bs;
        if (k >= max_blocks) return 4;
        int32_t blk = tables[(int64_t)b * max_blocks + k];
        if (blk < 0 || blk >= num_blocks) return 4;
        for (int d = 0; d < D; ++d) {
            K[t * D + d] = pool_value(pool, scales, blk, 0, h, (int)(t % bs), d, Hkv, bs, D, fp8);
            V[t * D + d] = pool_value(pool, scales, blk, 1, h, (int)(t % bs), d, Hkv, bs, D, fp8);
        }
    }
    return 0;
}

// out[B][Hq][D] (fp64) = softmax(scale * q K^T) V per (sequence, query head) over the paged pool.
// q holds bf16 bit patterns [B][Hq][D].  Work is spread over `threads` threads by (b, kv head);
// each output is computed by one thread in the same order regardless of the thread count.
int oracle_decode_attention(const uint8_t* pool, const float* scales, int num_blocks, int bs, int Hkv, int D, int fp8,
                            const uint16_t* q, const int32_t* tables, int max_blocks, const int32_t* lens, int B,
                            int Hq, double scale, double* out, int threads) {
    if (Hq % Hkv != 0) return 1;
    const int G = Hq / Hkv;
    const int64_t units = (int64_t)B * Hkv;
    std::vector<int> status(std::max(threads, 1), 0);
    auto work = [&](int tid, int nt) {
        std::vector<double> K, V, qd((size_t)G * D), o((size_t)G * D);
        for (int64_t u = tid; u < units; u += nt) {
            int b = (int)(u / Hkv), h = (int)(u % Hkv);
            int64_t L = lens[b];
            if (L < 0) {
                status[tid] = 1;
                continue;
            }
            int rc = gather(pool, scales, num_blocks, bs, Hkv, D, fp8, tables, max_blocks, b, h, L, K, V);
            if (rc) {
                status[tid] = rc;
                continue;
            }
            for (int j = 0; j < G; ++j)
                for (int d = 0; d < D; ++d)
                    qd[(size_t)j * D + d] = bf16_to_double(q[((int64_t)b * Hq + h * G + j) * D + d]);
            oracle_dense_attention(qd.data(), K.data(), V.data(), L, D, G, scale, o.data());
            for (int j = 0; j < G; ++j)
                for (int d = 0; d < D; ++d) out[((int64_t)b * Hq + h * G + j) * D + d] = o[(size_t)j * D + d];
        }
    };
    int nt = std::max(1, threads);
    if (nt == 1) {
        work(0, 1);
    } else {
        std::vector<std::thread> pool_threads;
        for (int t = 0; t < nt; ++t) pool_threads.emplace_back(work, t, nt);
        for (auto& th : pool_threads) th.join();
    }
    for (int s : status)
        if (s) return s;
    return 0;
}

// Chunked-context (prefill) attention over the pool: "TensorRT-LLM 深度实战" §7.3 (a long input
// is processed chunk by chunk; each chunk attends to everything cached before it and causally
// within itself) and "TensorRT-LLM 推理加速实战" §7.2 (context_fmha, the prefill attention, with
// use_paged_context_fmha reading the paged cache).  Sequence b's chunk is query rows
// cu_q[b] .. cu_q[b+1]-1 of q ([cu_q[B]][Hq][D] bf16); its K/V are already the last
// q_len = cu_q[b+1]-cu_q[b] of the ctx_lens[b] cached tokens, so query i sits at position
// p = ctx_lens[b] - q_len + i and attends to the tokens at positions 0..p.  Each query is the
// decode-attention definition over a context of p + 1 tokens.  out: [cu_q[B]][Hq][D] fp64.
int oracle_prefill_attention(const uint8_t* pool, const float* scales, int num_blocks, int bs, int Hkv, int D, int fp8,
                             const uint16_t* q, const int32_t* cu_q, const int32_t* tables, int max_blocks,
                             const int32_t* ctx_lens, int B, int Hq, double scale, double* out, int threads) {
    if (Hq % Hkv != 0) return 1;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        const int64_t n = (int64_t)cu_q[b + 1] - cu_q[b];
        if (n < 0 || n > ctx_lens[b]) return 1;
    }
    const int64_t units = (int64_t)B * Hkv;
    std::vector<int> status(std::max(threads, 1), 0);
    auto work = [&](int tid, int nt) {
        std::vector<double> K, V, qd((size_t)G * D), o((size_t)G * D);
        for (int64_t u = tid; u < units; u += nt) {
            const int b = (int)(u / Hkv), h = (int)(u % Hkv);
            const int64_t L = ctx_lens[b], n = (int64_t)cu_q[b + 1] - cu_q[b];
            if (n == 0) continue;
            int rc = gather(pool, scales, num_blocks, bs, Hkv, D, fp8, tables, max_blocks, b, h, L, K, V);
            if (rc) {
                status[tid] = rc;
                continue;
            }
            for (int64_t i = 0; i < n; ++i) {
                const int64_t row = cu_q[b] + i, p = L - n + i;
                for (int j = 0; j < G; ++j)
                    for (int d = 0; d < D; ++d)
                        qd[(size_t)j * D + d] = bf16_to_double(q[(row * Hq + h * G + j) * D + d]);
                oracle_dense_attention(qd.data(), K.data(), V.data(), p + 1, D, G, scale, o.data());
                for (int j = 0; j < G; ++j)
                    for (int d = 0; d < D; ++d) out[(row * Hq + h * G + j) * D + d] = o[(size_t)j * D + d];
            }
        }
    };
    const int nt = std::max(1, threads);
    if (nt == 1) {
        work(0, 1);
    } else {
        std::vector<std::thread> ths;
        for (int t = 0; t < nt; ++t) ths.emplace_back(work, t, nt);
        for (auto& th : ths) th.join();
    }
    for (int s : status)
        if (s) return s;
    return 0;
}

// ---------------------------------------------------------------------------- RoPE
// Rotary position embedding fused into the append ("TensorRT-LLM 深度实战" §3.3: the attention
// kernels also fuse RoPE; the build option use_fused_rope, §3.4).  The pages do not spell RoPE
// out; this is the form the Llama models the workloads follow use ("rotate half"): element d of
// the first half pairs with d + D/2, and at position p the pair turns by the angle
// p * base^(-2d/D):
//     y[d]       = x[d] cos - x[d + D/2] sin
//     y[d + D/2] = x[d + D/2] cos + x[d] sin
// computed in fp64 (products and sums rounded separately), then rounded to bf16 (nearest, ties
// to even).

// fp64 -> bf16 bits, round to nearest even: written from the format's definition (8 significant
// bits, exponent range of fp32, subnormals down to 2^-133).
static uint16_t oracle_f64_to_bf16(double x) {
    if (std::isnan(x)) return 0x7fc0;
    const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
    double a = std::fabs(x);
    if (std::isinf(a)) return sign | 0x7f80;
    if (a == 0.0) return sign;
    int e;
    std::frexp(a, &e);  // a = f * 2^e, f in [0.5, 1): the leading bit has weight 2^(e-1)
    int lead = e - 1;
    if (lead < -126) lead = -126;              // subnormal: fixed unit 2^-133
    const double unit = std::ldexp(1.0, lead - 7);  // one bf16 ulp at this exponent
    double k = std::nearbyint(a / unit);        // exact division by a power of two; ties to even
    double r = k * unit;                        // the rounded magnitude (may carry to 2^(lead+1))
    if (r >= std::ldexp(1.0, 128)) return sign | 0x7f80;
    // r is a bf16 value, so as fp32 its low 16 bits are zero
    const float rf = (float)r;
    uint32_t bits;
    std::memcpy(&bits, &rf, 4);
    return sign | (uint16_t)(bits >> 16);
}

// x, out: [N][H][D] bf16 bits; pos: [N].  out may alias x.
void oracle_rope(const uint16_t* x, const int64_t* pos, int64_t N, int H, int D, double base, uint16_t* out) {
    std::vector<double> row(D);
    for (int64_t i = 0; i < N; ++i)
        for (int h = 0; h < H; ++h) {
            const int64_t off = (i * H + h) * D;
            for (int d = 0; d < D; ++d) row[d] = bf16_to_double(x[off + d]);
            for (int d = 0; d < D / 2; ++d) {
                const double inv_freq = std::pow(base, -2.0 * d / D);
                const double ang = (double)pos[i] * inv_freq;
                const double c = std::cos(ang), s = std::sin(ang);
                const double a = row[d], b = row[d + D / 2];
                const double y0 = a * c - b * s;
                const double y1 = b * c + a * s;
                out[off + d] = oracle_f64_to_bf16(y0);
                out[off + d + D / 2] = oracle_f64_to_bf16(y1);
            }
        }
}

// The same rotation without the final rounding (fp64 out), for the invariants.
void oracle_rope_f64(const double* x, const int64_t* pos, int64_t N, int H, int D, double base, double* out) {
    for (int64_t i = 0; i < N; ++i)
        for (int h = 0; h < H; ++h) {
            const int64_t off = (i * H + h) * D;
            for (int d = 0; d < D / 2; ++d) {
                const double ang = (double)pos[i] * std::pow(base, -2.0 * d / D);
                const double c = std::cos(ang), s = std::sin(ang);
                const double a = x[off + d], b = x[off + d + D / 2];
                out[off + d] = a * c - b * s;
                out[off + d + D / 2] = b * c + a * s;
            }
        }
}

uint16_t oracle_f64_to_bf16_bits(double x) { return oracle_f64_to_bf16(x); }

// Same result computed split-wise: the context is cut into chunks of `chunk` tokens, each chunk
// yields (m, l, o) and the chunks are merged with the log-sum-exp rule.  Single-threaded.
int oracle_decode_attention_split(const uint8_t* pool, const float* scales, int num_blocks, int bs, int Hkv, int D,
                                  int fp8, const uint16_t* q, const int32_t* tables, int max_blocks,
                                  const int32_t* lens, int B, int Hq, double scale, int chunk, double* out) {
    if (Hq % Hkv != 0 || chunk <= 0) return 1;
    const int G = Hq / Hkv;
    std::vector<double> K, V;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hkv; ++h) {
            int64_t L = lens[b];
            int rc = gather(pool, scales, num_blocks, bs, Hkv, D, fp8, tables, max_blocks, b, h, L, K, V);
            if (rc) return rc;
            for (int j = 0; j < G; ++j) {
                int64_t row = ((int64_t)b * Hq + h * G + j) * D;
                std::vector<double> qd(D);
                for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[row + d]);
                std::vector<double> ms, ls;
                std::vector<std::vector<double>> os;
                for (int64_t c0 = 0; c0 < L; c0 += chunk) {
                    int64_t c1 = std::min<int64_t>(L, c0 + chunk);
                    double m = -INFINITY;
                    std::vector<double> z((size_t)(c1 - c0));
                    for (int64_t t = c0; t < c1; ++t) {
                        double s = 0.0;
                        for (int d = 0; d < D; ++d) s += qd[d] * K[t * D + d];
                        z[t - c0] = scale * s;
                        m = std::max(m, z[t - c0]);
                    }
                    double l = 0.0;
                    std::vector<double> o(D, 0.0);
                    for (int64_t t = c0; t < c1; ++t) {
                        double p = std::exp(z[t - c0] - m);
                        l += p;
                        for (int d = 0; d < D; ++d) o[d] += p * V[t * D + d];
                    }
                    ms.push_back(m);
                    ls.push_back(l);
                    os.push_back(o);
                }
                for (int d = 0; d < D; ++d) out[row + d] = 0.0;
                if (ms.empty()) continue;
                double M = *std::max_element(ms.begin(), ms.end());
                double l = 0.0;
                for (size_t s = 0; s < ms.size(); ++s) l += ls[s] * std::exp(ms[s] - M);
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (size_t s = 0; s < ms.size(); ++s) acc += std::exp(ms[s] - M) * os[s][d];
                    out[row + d] = acc / l;
                }
            }
        }
    return 0;
}

// Copy page src's K, V (all heads) and fp8 scales onto page dst of the host pool replica.
void oracle_copy_block(uint8_t* pool, float* scales, int bs, int Hkv, int D, int fp8, int64_t src, int64_t dst) {
    int64_t block_bytes = (int64_t)2 * Hkv * bs * D * (fp8 ? 1 : 2);
    std::memcpy(pool + dst * block_bytes, pool + src * block_bytes, (size_t)block_bytes);
    if (fp8) std::memcpy(scales + dst * Hkv * 4, scales + src * Hkv * 4, sizeof(float) * Hkv * 4);
}

// Pool geometry helpers for callers that size host replicas.
int64_t oracle_pool_bytes(int num_blocks, int bs, int Hkv, int D, int fp8) {
    return (int64_t)num_blocks * 2 * Hkv * bs * D * (fp8 ? 1 : 2);
}

int64_t oracle_scale_floats(int num_blocks, int Hkv) { return (int64_t)num_blocks * Hkv * 4; }

// Byte offset of element (t in block, d) of block blk, head h, K (kv=0) or V (kv=1).
int64_t oracle_elem_byte(int64_t blk, int kv, int h, int t, int d, int bs, int Hkv, int D, int fp8) {
    int esz = fp8 ? 1 : 2;
    return tile_base(blk, kv, h, Hkv, bs, D, esz) + elem_offset(kv, t, d, bs, D, fp8) * esz;
}

}  // extern "C"
