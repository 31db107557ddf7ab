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
// Work decomposition: one CTA per (sequence, KV head, pair of 128-row query tiles); CTAs of
// the sequences with the most causal work are dispatched first.  A row is
// a (token, head-in-group) pair, so a tile covers 128/G consecutive chunk tokens and all G
// query heads of one KV head, and every K/V tile brought on chip serves both query tiles and
// the whole group.  The CTA walks the KV tiles of 128 keys its last token can see:
//   warps 0, 2 TMA producers of a K ring (3 tiles) and a V ring (2 tiles): a tile is two
//              128-row panels (the 64-element halves, 128-byte swizzled), one 2-D tensor copy
//              per (page part, half) stacking the parts' rows; parts past the context get a
//              coordinate past the pool, which the copy fills with zeros.  K and V are released
//              separately (after the last S, after the last PV), so K runs further ahead.
//   warp 1     tensor-memory owner and MMA issuer (one thread), per KV tile j and query tile t:
//                O_t += P_t(j) V_j      M=128, N=128, K=16 per instruction, A = P straight
//                                       from tensor memory, B = V MN-major from the page copy
//                S_t(j+1) = Q_t K_{j+1}^T  M=128, N=128, K=16 per instruction, written over
//                                       P_t(j): the tensor pipe runs one thread's MMAs in
//                                       issue order
//              with descriptors built once and advanced by constant offsets (issuing must
//              stay faster than the ~65 cycles an M=128 N=128 K=16 MMA takes), so one
//              tile's MMAs run while the other tile's softmax works.
//   warp 3     idle (it completes the control warpgroup, which gives registers away)
//   warps 4-7, 8-11  one softmax warpgroup per query tile, one row per thread (TMEM lane =
//              row): the Q row into shared memory, then per KV tile the S row out of TMEM,
//              causal mask on the tiles that cross the row's position, online softmax in base
//              2 with the scale folded into one FMA, the O row rescaled in TMEM only when the
//              running maximum grows by more than 2^8 (the stale maximum keeps P <= 256), and
//              P back into TMEM as bf16.  On the first KV tile P is carried as a bf16 pair
//              (hi + lo, two MMAs): short contexts have all their weight there, and a single
//              bf16 P would add its rounding to the output's.  Finally O / l as bf16.
// TMEM: S_0 | S_1 | O_0 | O_1, 128 fp32 columns each; P_t (bf16 pairs) lives in S_t's columns.
//
// FP8-E4M3 and INT8 pools (KV != 0): the tensor cores take one 16-bit type for both operands,
// so the codes are widened on chip to f16 -- K' = the codes themselves (exact), whose scale, one
// per page part, multiplies the score in the softmax; V' = code x f16(scale x 2^-eV), with a
// power of two per (sequence, KV head) that keeps the values in f16's range; q goes to f16
// exactly with a power of two per row; P is f16; the powers of two return in the score scale
// and the epilogue.  512 threads: warp 0 issues the code copies (two tiles deep: at head_dim 128
// a K tile's codes land in the upper half of its own ring slot and are widened in place), warp 1
// the MMAs, warps 2-7 widen (K rows into the K ring; V, kept by the pool as 16-token panels
// [d][16 codes], into V^T, which the P.V MMA reads K-major), warps 8-15 run the softmax.
//
// Every mbarrier wait is bounded; on expiry the kernel sets the pool's error word, every role
// stops, and tensor memory is released.
#include <cmath>
#include <cstdlib>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace prefill {

constexpr int kRows = 128;   // query rows per tile
constexpr int kTiles = 2;    // query tiles per CTA
constexpr int kKeys = 128;   // keys per KV tile
constexpr int kKStages = 3;  // K ring slots (barriers); a K tile is free once both tiles' S MMAs have read it
constexpr int kVStages = 2;  // V ring: a V tile is free once both tiles' PV MMAs have read it
constexpr int kThreads = 128 + kTiles * 128;  // bf16 pools: control warpgroup + one softmax warpgroup per tile
constexpr int kThreadsOne = kThreads + 128;    // one-byte pools: + a widening warpgroup
constexpr int kConverters = 6;                 // one-byte pools: widening warps 2, 3 (control) and 4-7
// register splits (setmaxnreg).  bf16: launched at 168 per thread (65536 / 384, rounded down to
// 8), i.e. 64512 for the block; control 128 x 56 + softmax 256 x 224 = 64512 fits exactly.
// One-byte: launched at 128 (65536 / 512); control and widening 256 x 40 + softmax 256 x 216 =
// 65536 fits exactly.
constexpr uint32_t kRegsControl = 56, kRegsSoftmax = 224;
constexpr uint32_t kRegsControlOne = 40, kRegsSoftmaxOne = 216;
static_assert(128 * kRegsControl + kTiles * 128 * kRegsSoftmax <= kThreads * 168, "register split");
static_assert(256 * kRegsControlOne + kTiles * 128 * kRegsSoftmaxOne <= kThreadsOne * 128, "register split");
constexpr uint32_t kPanelBytes = 128u * 128u;      // 128 rows x 128 bytes (64 bf16 of a row)
constexpr uint32_t kOffQ = 0;
// Shared-memory layout for head_dim D (64 or 128): a row of Q, K or V is D / 64 panels of 16-bit
// elements.  One-byte pools (ONE) keep two K stages and stage the codes (D bytes a row) for the
// widening warps, two tiles deep: with D = 128 a K tile's codes land in the upper half of its
// own ring slot and are widened in place (a code row is overwritten only by the panel-1 row of
// the same key, written after the whole row was read), V's in two stages of their own; with
// D = 64 both K and V have two code stages.
template <int D, bool ONE>
struct Layout {
    static constexpr int kPanels = D / 64;
    static constexpr int kKSt = ONE ? 2 : kKStages;                // K ring stages in use
    static constexpr uint32_t kQBytes = kPanels * kPanelBytes;     // one Q tile
    static constexpr uint32_t kHalfBytes = kPanels * kPanelBytes;  // K (or V) of one KV tile
    static constexpr uint32_t kCodeRow = D;                        // bytes of one row of codes
    static constexpr uint32_t kCodeBytes = ONE ? kKeys * kCodeRow : 0u;  // codes of one K (or V) tile
    static constexpr bool kInPlaceK = ONE && D == 128;
    static constexpr uint32_t kOffK = kOffQ + kTiles * kQBytes;
    static constexpr uint32_t kOffV = kOffK + kKSt * kHalfBytes;
    static constexpr uint32_t kOffCodeK = kOffV + kVStages * kHalfBytes;  // [2] K code stages (D = 64)
    static constexpr uint32_t kOffCodeV = kOffCodeK + (ONE && !kInPlaceK ? 2 * kCodeBytes : 0u);  // [2] V
    static constexpr uint32_t kOffBar = kOffCodeV + (ONE ? 2 * kCodeBytes : 0u);
    static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(kOffCodeK % 1024 == 0 && kOffCodeV % 1024 == 0, "code stages on a swizzle-pattern boundary");
    static_assert(!kInPlaceK || kCodeBytes * 2 == kHalfBytes, "K codes fill the upper half of their slot");
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (P stays <= 2^8)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kEndBar = 1;      // named barrier: every role done before TMEM is released
constexpr int kMaxRankedSeqs = 512;  // above this the sequences are dispatched in index order
constexpr int kSmallRankedSeqs = 64;  // up to this the ranking reads the inputs directly
static_assert(kMaxRankedSeqs * sizeof(int64_t) <= kTiles * Layout<64, false>::kQBytes, "dispatch ranking fits the Q tiles' space");

// mbarrier slots
constexpr int kBarQ = 0;                          // Q rows of both tiles written (8 warps arrive)
constexpr int kBarKFull = 1;                      // [kKStages] K copies landed (tx bytes)
constexpr int kBarKEmpty = kBarKFull + kKStages;  // [kKStages] last S MMA reading the K tile done
constexpr int kBarVFull = kBarKEmpty + kKStages;  // [kVStages] V copies landed (tx bytes)
constexpr int kBarVEmpty = kBarVFull + kVStages;  // [kVStages] last PV MMA reading the V tile done
constexpr int kBarS = kBarVEmpty + kVStages;      // [kTiles] S_t(j) ready (commit)
constexpr int kBarP = kBarS + kTiles;             // [kTiles] P_t(j) in TMEM (4 warps arrive)
constexpr int kBarO = kBarP + kTiles;             // [kTiles] last PV_t done (commit)
constexpr int kBarCode = kBarO + kTiles;          // [2 K, 2 V] code stages landed (one-byte pools; tx bytes)
constexpr int kBarDrain = kBarCode + 4;           // MMAs in flight done (error path)
constexpr int kNumBars = kBarDrain + 1;
static_assert(kNumBars * 8 <= 256, "barrier area");

struct Params {
    const uint16_t* q;
    uint16_t* out;
    const int32_t* cu_q;
    const int32_t* tables;
    const int32_t* ctx;
    const float* scales;  // one-byte pools: [num_blocks][Hkv][4] (K scale, V scale, unused, unused)
    int* err;
    int B, Hq, Hkv, G, max_blocks, bs, part, num_blocks, tiles;
    int32_t oob_row;  // a row coordinate past the pool: the copy fills the box with zeros
    float scale_log2;
    uint64_t wait_ns;
    uint32_t stall_tx;  // test hook: extra bytes every K/V stage expects and no copy delivers
};

// S = Q K^T over K = 64 (head_dim 64): four K=16 MMAs within one 128-byte panel of A and of B
// (descriptor start addresses advance by 32 bytes a step), the first one overwriting D.
__device__ __forceinline__ void umma_ss_k64_x4(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                               uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b32 al, bl;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 pf, %1, %1;\n\tsetp.eq.b32 pt, %1, %1;\n\t"
        "mov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, pf;\n\t"
        "add.u32 al, %1, 2;\n\tadd.u32 bl, %2, 2;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, pt;\n\t"
        "add.u32 al, %1, 4;\n\tadd.u32 bl, %2, 4;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, pt;\n\t"
        "add.u32 al, %1, 6;\n\tadd.u32 bl, %2, 6;\n\tmov.b64 a, {al, %3};\n\tmov.b64 b, {bl, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, pt;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc));
}

// 2^e as two normal fp32 factors (x * a * b scales x exactly while the result stays normal);
// e is clamped to [-252, 252], beyond which no finite product of such factors is normal anyway.
__device__ __forceinline__ void pow2_pair(int e, float& a, float& b) {
    e = max(-252, min(252, e));
    const int ea = e / 2, eb = e - ea;
    a = __int_as_float((127 + ea) << 23);
    b = __int_as_float((127 + eb) << 23);
}

// Exponent of the leading bit of a positive finite fp32 given by its bits (subnormals included).
__device__ __forceinline__ int lead_exp(uint32_t bits) {
    const int E = (int)(bits >> 23);
    return E ? E - 127 : (31 - __clz((int)bits)) - 149;
}

// Four one-byte codes (byte 0 first) -> two f16x2 holding the codes' values exactly: E4M3 by
// the hardware conversion (every E4M3 value is an f16); INT8 in [-127, 127] by writing code + 128
// into the low mantissa bits of 1024.0 (f16 0x6400) and subtracting 1152, both exact.
template <int KV>
__device__ __forceinline__ void widen4(uint32_t four, uint32_t& lo, uint32_t& hi) {
    if constexpr (KV == 2) {
        const uint32_t x = four ^ 0x80808080u;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(__byte_perm(x, 0x64u, 0x4140)), "r"(0x64806480u));
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(__byte_perm(x, 0x64u, 0x4342)), "r"(0x64806480u));
    } else {
        lo = ptx::e4m3x2_to_f16x2(four);
        hi = ptx::e4m3x2_to_f16x2(four >> 16);
    }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// a pair of widened codes times the part's scale (an f16 pair), rounded to f16
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B both f16 (F16) or both bf16.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, int a_mn, int b_mn, bool f16) {
    return f16 ? (ptx::umma_idesc_bf16(M, N, a_mn, b_mn) & ~((7u << 7) | (7u << 10)))
               : ptx::umma_idesc_bf16(M, N, a_mn, b_mn);
}

// Eight steps of D += A B with A (P) in tensor memory, 8 columns (16 keys) per step, and B = V^T
// K-major (one 128-byte swizzled line of 64 keys per d): a step advances B by 32 bytes (+2 in
// the start field), keys 64-127 sit one panel of D lines further (+PANEL).  Step kk runs only if
// kk < nk; step 0 accumulates only if acc0 != 0.
template <uint32_t PANEL>
__device__ __forceinline__ void umma_ts_kmajor_x8(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                                  uint32_t idesc, uint32_t acc0, int nk) {
    asm volatile(
        "{\n\t.reg .pred pa, pt, g1, g2, g3, g4, g5, g6, g7;\n\t.reg .b32 ta, bl;\n\t.reg .b64 b;\n\t"
        "setp.ne.b32 pa, %5, 0;\n\tsetp.eq.b32 pt, %5, %5;\n\t"
        "setp.gt.s32 g1, %6, 1;\n\tsetp.gt.s32 g2, %6, 2;\n\tsetp.gt.s32 g3, %6, 3;\n\t"
        "setp.gt.s32 g4, %6, 4;\n\tsetp.gt.s32 g5, %6, 5;\n\tsetp.gt.s32 g6, %6, 6;\n\t"
        "setp.gt.s32 g7, %6, 7;\n\t"
        "mov.b64 b, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, pa;\n\t"
        "add.u32 ta, %1, 8;\n\tadd.u32 bl, %2, 2;\n\tmov.b64 b, {bl, %3};\n\t"
        "@g1 tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t"
        "add.u32 ta, %1, 16;\n\tadd.u32 bl, %2, 4;\n\tmov.b64 b, {bl, %3};\n\t"
        "@g2 tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t"
        "add.u32 ta, %1, 24;\n\tadd.u32 bl, %2, 6;\n\tmov.b64 b, {bl, %3};\n\t"
        "@g3 tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t"
        "add.u32 ta, %1, 32;\n\tadd.u32 bl, %2, %7;\n\tmov.b64 b, {bl, %3};\n\t"
        "@g4 tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t"
        "add.u32 ta, %1, 40;\n\tadd.u32 bl, %2, %8;\n\tmov.b64 b, {bl, %3};\n\t"
        "@g5 tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t"
        "add.u32 ta, %1, 48;\n\tadd.u32 bl, %2, %9;\n\tmov.b64 b, {bl, %3};\n\t"
        "@g6 tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t"
        "add.u32 ta, %1, 56;\n\tadd.u32 bl, %2, %10;\n\tmov.b64 b, {bl, %3};\n\t"
        "@g7 tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %4, pt;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc0), "r"(nk), "n"(PANEL), "n"(PANEL + 2), "n"(PANEL + 4),
        "n"(PANEL + 6));
}

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

// KV: 0 bf16 pool, 1 FP8-E4M3 pool, 2 INT8 pool.
template <int PART, int D, int KV>
__global__ void __launch_bounds__(KV != 0 ? kThreadsOne : kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap, const Params p) {
    static_assert(PART == 16 || PART == 32 || PART == 64, "page part of 16, 32 or 64 rows");
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    constexpr bool ONE = KV != 0;  // one-byte codes with per-(block, head) scales
    using LY = Layout<D, ONE>;
    constexpr int KS = LY::kKSt;
    constexpr int kThr = ONE ? kThreadsOne : kThreads;
    constexpr int kSmWarp0 = ONE ? 8 : 4;  // first softmax warp
    // one-byte pools with page parts of 32 or more keys take V's scale in the softmax exponent
    // (V widened exactly); with parts of 16 (eight scales a tile) the widening applies it
    constexpr bool VS = ONE && PART >= 32;
    constexpr uint32_t kQBytes = LY::kQBytes, kHalfBytes = LY::kHalfBytes;
    constexpr uint32_t kOffK = LY::kOffK, kOffV = LY::kOffV, kOffBar = LY::kOffBar;
    constexpr int kPanels = LY::kPanels;
    constexpr int kParts = kKeys / PART;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const sm = smem_raw + (base - raw);
    const uint32_t sK = base + kOffK, sV = base + kOffV;
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    ptx::grid_dependency_wait();  // inputs may come from the preceding append
    // Dispatch order (1-D grid, CTAs start roughly in index order): sequences by decreasing
    // causal work n (2L - n), then the pairs of a sequence deepest first, heads fastest -- the
    // longest jobs start first, so the last wave holds the short ones.
    const int per_seq = p.Hkv * p.tiles;
    const int rank = (int)(blockIdx.x / (unsigned)per_seq);
    const int rem = (int)(blockIdx.x % (unsigned)per_seq);
    const int h = rem % p.Hkv;
    const int pair = p.tiles - 1 - rem / p.Hkv;
    int b = rank;
    if (p.B <= kSmallRankedSeqs) {
        // few sequences: rank straight from the (cached) global inputs
        __shared__ int seq_of_rank_small;
        if (threadIdx.x == 0) seq_of_rank_small = -1;
        __syncthreads();
        auto work = [&](int i) -> int64_t {
            const int64_t nn = p.cu_q[i + 1] - p.cu_q[i], ll = p.ctx[i];
            return nn * (2 * ll - nn);
        };
        for (int i = threadIdx.x; i < p.B; i += kThr) {
            const int64_t wi = work(i);
            int r = 0;
            for (int k = 0; k < p.B; ++k) {
                const int64_t wk = work(k);
                r += (wk > wi || (wk == wi && k < i)) ? 1 : 0;
            }
            if (r == rank) seq_of_rank_small = i;
        }
        __syncthreads();
        b = seq_of_rank_small;
    } else if (p.B <= kMaxRankedSeqs) {
        // each sequence's work, loaded once into the Q tiles' space (free until the softmax
        // warps stage Q, after the block barrier below); then every thread ranks its sequences
        // against all of them from shared memory (B^2 comparisons per CTA)
        __shared__ int seq_of_rank;
        int64_t* work_s = reinterpret_cast<int64_t*>(sm + kOffQ);
        for (int i = threadIdx.x; i < p.B; i += kThr) {
            const int64_t nn = p.cu_q[i + 1] - p.cu_q[i], ll = p.ctx[i];
            work_s[i] = nn * (2 * ll - nn);
        }
        if (threadIdx.x == 0) seq_of_rank = -1;
        __syncthreads();
        for (int i = threadIdx.x; i < p.B; i += kThr) {
            const int64_t wi = work_s[i];
            int r = 0;
            for (int k = 0; k < p.B; ++k) {
                const int64_t wk = work_s[k];
                r += (wk > wi || (wk == wi && k < i)) ? 1 : 0;
            }
            if (r == rank) seq_of_rank = i;
        }
        __syncthreads();
        b = seq_of_rank;
    }
    const int q0 = p.cu_q[b];
    const int n = p.cu_q[b + 1] - q0;
    const int L = p.ctx[b];
    const int T = kRows / p.G;  // chunk tokens per query tile
    const int t0 = pair * kTiles * T;
    if (t0 >= n) return;
    if (n < 0 || n > L || L > p.max_blocks * p.bs) {
        if (threadIdx.x == 0) atomicOr(p.err, kErrBounds);
        return;
    }
    // KV tiles each query tile needs (0: the tile lies past the chunk)
    int nkv[kTiles];
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        const int first = t0 + t * T;
        const int last = min(n, first + T) - 1;
        nkv[t] = first < n ? (L - n + last + 1 + kKeys - 1) / kKeys : 0;
    }
    const int last_tile = nkv[1] > 0 ? 1 : 0;
    const int n_kv = nkv[last_tile];  // the last active tile sees the most keys

    // One-byte pools: the largest V scale over this sequence's blocks for head h (per warp here,
    // combined after the barrier below).  It fixes the power of two 2^-eV that brings
    // code x scale into f16 range (largest |value| below 2^16) for the widened V tiles.
    __shared__ uint32_t scale_max_s[kThreadsOne / 32];
    if constexpr (ONE) {
        const int32_t* tb = p.tables + (int64_t)b * p.max_blocks;
        const int nb = (L + p.bs - 1) / p.bs;
        uint32_t mv = 0;  // fp32 bits: non-negative scales order like their bits
        for (int i = threadIdx.x; i < nb; i += kThr) {
            const int blk = tb[i];
            if (blk >= 0 && blk < p.num_blocks) mv = max(mv, __float_as_uint(p.scales[((int64_t)blk * p.Hkv + h) * 4 + 1]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mv = max(mv, __shfl_xor_sync(0xffffffffu, mv, o));
        if (lane == 0) scale_max_s[warp] = mv;
    }
    // eV such that the largest V scale times 2^-eV lies in [64, 128): codes up to 448 (E4M3) or
    // 127 (INT8) then give |value| < 2^16 in f16.  0 for a sequence whose scales are all zero.
    auto scale_exp_v = [&]() -> int {
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < kThr / 32; ++w) m = max(m, scale_max_s[w]);
        return m ? lead_exp(m) - 6 : 0;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool wg_arrive = i == kBarQ || (i >= kBarP && i < kBarP + kTiles);
            // one-byte pools: a K / V ring slot is full once every widening warp has written its share
            const bool widened = ONE && ((i >= kBarKFull && i < kBarKFull + kKStages) ||
                                         (i >= kBarVFull && i < kBarVFull + kVStages));
            ptx::mbar_init(bar(i), i == kBarQ ? 8u : (wg_arrive ? 4u : (widened ? (uint32_t)kConverters : 1u)));
        }
        abort_s = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_addr(&tmem_base_s), kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp < kSmWarp0) {
      ptx::regs_dec<ONE ? kRegsControlOne : kRegsControl>();  // whole warpgroups, one instruction each
      if (ONE && warp == 0) {
        // ---------------------------------------------------------------- one-byte code copies
        // Two code stages per stream: tile j's copies go out once its stage is free -- a K slot
        // holding its own codes once the S MMAs of tile j-2 have read it, a separate stage once
        // the widening warps are done with tile j-2.  One 2-D copy of PART code rows per page
        // part (rows past the context read zeros).
        const int32_t* tb = p.tables + (int64_t)b * p.max_blocks;
        auto issue = [&](int kv, int j) {
            const uint32_t cbar = bar(kBarCode + 2 * kv + (j & 1));
            const uint32_t dst = kv ? base + LY::kOffCodeV + (uint32_t)(j & 1) * LY::kCodeBytes
                                 : LY::kInPlaceK ? sK + (uint32_t)(j & 1) * kHalfBytes + LY::kCodeBytes
                                                 : base + LY::kOffCodeK + (uint32_t)(j & 1) * LY::kCodeBytes;
            if (lane == 0) ptx::mbar_arrive_expect_tx(cbar, LY::kCodeBytes + p.stall_tx);
            __syncwarp();
            if (lane < kParts) {
                const int tok = j * kKeys + lane * PART;
                int32_t row = p.oob_row;
                if (tok < L) {
                    const int blk = tb[tok / p.bs];
                    if (blk >= 0 && blk < p.num_blocks)
                        row = (int32_t)((((int64_t)2 * blk + kv) * p.Hkv + h) * p.bs + (tok % p.bs));
                    else if (kv == 0)
                        atomicOr(p.err, kErrBounds);
                }
                ptx::tma_load_2d(dst + (uint32_t)(lane * PART) * LY::kCodeRow, &tmap, 0, row, cbar);
            }
        };
        bool ok = true;
        for (int j = 0; j < n_kv && ok; ++j) {
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                if (j >= 2) {
                    // the stage of tile j-2: the K slot read by its S MMAs (in place), else widened
                    const int free_bar = kv ? kBarVFull : LY::kInPlaceK ? kBarKEmpty : kBarKFull;
                    if (lane == 0) ok = ptx::mbar_wait(bar(free_bar + (j & 1)), ((j >> 1) - 1) & 1, p.wait_ns);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok || __shfl_sync(0xffffffffu, abort_s, 0)) {
                        ok = false;
                        break;
                    }
                }
                issue(kv, j);
            }
        }
        if (lane == 0 && !ok) {
            if (!abort_s) atomicOr(p.err, kErrTimeout);
            abort_s = 1;
        }
        __syncwarp();
        ptx::named_barrier_sync(kEndBar, kThr);
      } else if (ONE && warp >= 2) {
        // ---------------------------------------------------------------- one-byte widening
        // Six warps (2, 3, 4-7) widen each tile.  K rows go to the K ring as the 128-byte swizzled
        // panels the S MMA reads, the codes' values exactly (their scale joins the score in the
        // softmax); V becomes code x (scale x 2^-eV), the scale that of the code's (block, head),
        // rounded once to f16.  V, which the pool keeps as 16-token panels [d][16
        // codes] in the pair order 0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15 (one 16-byte chunk = the
        // 16 tokens of one d), goes to the V ring as V^T, K-major for the P.V MMA: [64-key
        // panel][d line][128 bytes: 64 keys] -- no transpose, four byte permutes restore the
        // token order.  The passes of a tile (4 K rows or 32 d of one 16-key group each with
        // D = 128; 8 rows or 32 d with D = 64) are dealt round-robin to the warps.
        const int cw = warp - 2;  // 0..5
        const int32_t* tb = p.tables + (int64_t)b * p.max_blocks;
        float fav = 1.f, fbv = 1.f;  // 2^-eV (parts of 16: the widening applies V's scale)
        if constexpr (!VS) pow2_pair(-scale_exp_v(), fav, fbv);
        constexpr int kPassK = D == 128 ? 32 : 16;  // passes per tile: K
        constexpr int kPassV = D / 4;               // passes per tile: V (8 groups x D / 32)
        constexpr uint32_t kVtPanel = (uint32_t)D * 128u;

        // lane pi < kParts: part pi's V scale of tile j (0 past the context; K codes are widened
        // exactly and their scale joins the score in the softmax)
        auto load_scales = [&](int j, float& sv) {
            sv = 0.f;
            if (lane < kParts) {
                const int tok = j * kKeys + lane * PART;
                if (tok < L) {
                    const int blk = tb[tok / p.bs];
                    if (blk >= 0 && blk < p.num_blocks) sv = p.scales[((int64_t)blk * p.Hkv + h) * 4 + 1];
                }
            }
        };
        // Every lane waits (bounded) for the codes of tile j (stage j & 1) itself, as the decode
        // kernel's consumers do: a copy's bytes are visible to the threads that observe its phase
        // complete, and every lane reads them (one spinning lane followed by a single poll of the
        // others failed the one-byte parity tests).  Unless the codes sit in the slot itself,
        // lane 0 then waits for the ring slot (the MMAs of tile j-2 done with it) and the warp
        // follows.
        auto wait2 = [&](int kv, int j, bool slot_wait) -> bool {
            bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarCode + 2 * kv + (j & 1)), (j >> 1) & 1, p.wait_ns));
            if (ok && slot_wait && j >= 2) {
                const int emptyb = kv ? kBarVEmpty : kBarKEmpty;
                if (lane == 0) ok = ptx::mbar_wait(bar(emptyb + (j & 1)), ((j >> 1) - 1) & 1, p.wait_ns);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
            return ok;
        };
        float svn = 0.f;
        if constexpr (!VS) load_scales(0, svn);
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const float svc = svn;
            if constexpr (!VS) {
                if (j + 1 < n_kv) load_scales(j + 1, svn);  // in flight while this tile is widened
            }
            // ---- K
            ok = wait2(0, j, !LY::kInPlaceK);
            if (!ok || __shfl_sync(0xffffffffu, abort_s, 0)) break;
            {
                const uint32_t dst0 = sK + (uint32_t)(j % KS) * kHalfBytes;
                // in place: the codes fill the slot's upper half (panel 1), code row r under the
                // panel-1 row of key r, which this pass writes only after reading the whole row
                const uint32_t codeK = LY::kInPlaceK ? dst0 + LY::kCodeBytes
                                                     : base + LY::kOffCodeK + (uint32_t)(j & 1) * LY::kCodeBytes;
#pragma unroll 1
                for (int i = cw; i < kPassK; i += kConverters) {
                    if constexpr (D == 128) {
                        const int rs = lane >> 3, c = lane & 7, r = 4 * i + rs;
                        const uint4 w = lds128(codeK + (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4));
                        uint32_t o[8];
                        widen4<KV>(w.x, o[0], o[1]);
                        widen4<KV>(w.y, o[2], o[3]);
                        widen4<KV>(w.z, o[4], o[5]);
                        widen4<KV>(w.w, o[6], o[7]);
                        const uint32_t dst = dst0 + (uint32_t)(c >> 2) * kPanelBytes;
                        const int cc = (c & 3) * 2;
                        sts128(dst + swz128(r, cc), o[0], o[1], o[2], o[3]);
                        sts128(dst + swz128(r, cc + 1), o[4], o[5], o[6], o[7]);
                    } else {
                        // 64-byte code rows, 64-byte swizzle: chunk c of row r at c ^ ((r >> 1) & 3)
                        const int rs = lane >> 2, c = lane & 3, r = 8 * i + rs;
                        const uint4 w = lds128(codeK + (uint32_t)r * 64u + ((uint32_t)(c ^ ((r >> 1) & 3)) << 4));
                        uint32_t o[8];
                        widen4<KV>(w.x, o[0], o[1]);
                        widen4<KV>(w.y, o[2], o[3]);
                        widen4<KV>(w.z, o[4], o[5]);
                        widen4<KV>(w.w, o[6], o[7]);
                        sts128(dst0 + swz128(r, 2 * c), o[0], o[1], o[2], o[3]);
                        sts128(dst0 + swz128(r, 2 * c + 1), o[4], o[5], o[6], o[7]);
                    }
                }
            }
            ptx::fence_proxy_async_smem();  // the S MMAs (async proxy) read what was written
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarKFull + j % KS));
            // ---- V
            ok = wait2(1, j, true);
            if (!ok || __shfl_sync(0xffffffffu, abort_s, 0)) break;
            {
                const uint32_t dst0 = sV + (uint32_t)(j % kVStages) * kHalfBytes;
                const uint32_t codeV = base + LY::kOffCodeV + (uint32_t)(j & 1) * LY::kCodeBytes;
#pragma unroll 1
                for (int i = cw; i < kPassV; i += kConverters) {
                    const int G = i / (D / 32), d = 32 * (i % (D / 32)) + lane;
                    uint32_t s2 = 0u;
                    if constexpr (!VS) {
                        const float v = __shfl_sync(0xffffffffu, svc, (16 * G) / PART) * fav * fbv;
                        s2 = ptx::pack_f16x2(v, v);
                    }
                    uint32_t src;
                    if constexpr (D == 128)
                        src = codeV + (uint32_t)(16 * G + (d >> 3)) * 128u + ((uint32_t)((d & 7) ^ ((d >> 3) & 7)) << 4);
                    else
                        src = codeV + (uint32_t)(16 * G + (d >> 2)) * 64u + ((uint32_t)((d & 3) ^ ((d >> 3) & 3)) << 4);
                    const uint4 w = lds128(src);
                    uint32_t o[8];
                    widen4<KV>(__byte_perm(w.x, w.y, 0x5410), o[0], o[1]);  // tokens 0-3
                    widen4<KV>(__byte_perm(w.z, w.w, 0x5410), o[2], o[3]);  // tokens 4-7
                    widen4<KV>(__byte_perm(w.x, w.y, 0x7632), o[4], o[5]);  // tokens 8-11
                    widen4<KV>(__byte_perm(w.z, w.w, 0x7632), o[6], o[7]);  // tokens 12-15
                    if constexpr (!VS) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = mul_f16x2(o[e], s2);
                    }
                    const uint32_t dst = dst0 + (uint32_t)(G >> 2) * kVtPanel + (uint32_t)d * 128u;
                    const int cc = (G & 3) * 2;
                    sts128(dst + ((uint32_t)(cc ^ (d & 7)) << 4), o[0], o[1], o[2], o[3]);
                    sts128(dst + ((uint32_t)((cc + 1) ^ (d & 7)) << 4), o[4], o[5], o[6], o[7]);
                }
            }
            ptx::fence_proxy_async_smem();  // the P.V MMAs read what was written
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarVFull + j % kVStages));
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, kErrTimeout);
            abort_s = 1;
        }
        __syncwarp();
        ptx::named_barrier_sync(kEndBar, kThr);
      } else if (!ONE && (warp == 0 || warp == 2)) {
        // ---------------------------------------------------------------- producers (bf16 pools)
        // warp 0 fills the K ring, warp 2 the V ring; each KV tile is two 128-row panels (the
        // 64-element halves), one 2-D copy of PART rows per (page part, half)
        const int kv = warp == 0 ? 0 : 1;
        const int stages = kv ? kVStages : KS;
        const uint32_t ring = kv ? sV : sK;
        const int full = kv ? kBarVFull : kBarKFull, empty = kv ? kBarVEmpty : kBarKEmpty;
        const int32_t* tb = p.tables + (int64_t)b * p.max_blocks;
        for (int j = 0; j < n_kv; ++j) {
            const int s = j % stages;
            if (j >= stages) {
                bool ok = true;
                if (lane == 0) ok = ptx::mbar_wait(bar(empty + s), ((j / stages) - 1) & 1, p.wait_ns);
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
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar(full + s), kHalfBytes + p.stall_tx);
            __syncwarp();
            if (lane < kPanels * kParts) {
                const int pi = lane / kPanels, q = lane % kPanels;
                const int tok = j * kKeys + pi * PART;  // first key of this page part
                int32_t row = p.oob_row;
                if (tok < L) {
                    const int blk = tb[tok / p.bs];
                    if (blk >= 0 && blk < p.num_blocks)
                        row = (int32_t)((((int64_t)2 * blk + kv) * p.Hkv + h) * p.bs + (tok % p.bs));
                    else if (kv == 0 && q == 0)
                        atomicOr(p.err, kErrBounds);
                }
                ptx::tma_load_2d(ring + (uint32_t)s * kHalfBytes + (uint32_t)q * kPanelBytes + (uint32_t)(pi * PART) * 128u,
                                 &tmap, q * 64, row, bar(full + s));
            }
        }
        ptx::named_barrier_sync(kEndBar, kThr);
      } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // descriptors are built once; the start-address field counts 16-byte units, so moving
            // an operand by X bytes adds X >> 4 (addresses stay below 256 KB: no carry out)
            // operands f16 for one-byte pools (widened K/V, rescaled Q, P), bf16 otherwise
            constexpr uint32_t idS = idesc_f16kind(128, kKeys, 0, 0, ONE);
            constexpr uint32_t idO = idesc_f16kind(128, D, 0, ONE ? 0 : 1, ONE);  // one-byte: V^T K-major
            // a descriptor's high half (stride, version, swizzle) is the same for Q and K; V's
            // differs only in the low half (its panel stride)
            const uint64_t dQ0 = ptx::umma_sdesc_sw128(base + kOffQ, 16, 1024);
            const uint64_t dK0 = ptx::umma_sdesc_sw128(sK, 16, 1024);
            const uint64_t dV0 = ONE ? ptx::umma_sdesc_sw128(sV, 16, 1024) : ptx::umma_sdesc_sw128(sV, kPanelBytes, 1024);
            const uint32_t hi = (uint32_t)(dQ0 >> 32);
            const uint32_t q_lo = (uint32_t)dQ0, k_lo = (uint32_t)dK0, v_lo = (uint32_t)dV0;
            int k_ready = 0, v_ready = 0;  // K / V tiles whose copies this thread has waited for
            bool ok = ptx::mbar_wait(bar(kBarQ), 0, p.wait_ns);
            ptx::tc_fence_after();
            auto wait_k = [&](int j) -> bool {
                if (j < k_ready) return true;
                if (!ptx::mbar_wait(bar(kBarKFull + j % KS), (j / KS) & 1, p.wait_ns)) return false;
                ptx::tc_fence_after();
                k_ready = j + 1;
                return true;
            };
            auto wait_v = [&](int j) -> bool {
                if (j < v_ready) return true;
                if (!ptx::mbar_wait(bar(kBarVFull + j % kVStages), (j / kVStages) & 1, p.wait_ns)) return false;
                ptx::tc_fence_after();
                v_ready = j + 1;
                return true;
            };
            // S_t(j) = Q_t K_j^T: 8 MMAs of N = 128 (keys past the context give unused scores),
            // issued as one asm block: the issuing thread cannot run ahead of the tensor pipe, so
            // any arithmetic between two MMAs would be exposed.
            auto issue_s = [&](int t, int j) {
                if constexpr (D == 128)
                    ptx::umma_ss_k128_x8(tmem + (uint32_t)(t * kKeys), q_lo + (uint32_t)t * (kQBytes >> 4),
                                         k_lo + (uint32_t)(j % KS) * (kHalfBytes >> 4), hi, idS);
                else
                    umma_ss_k64_x4(tmem + (uint32_t)(t * kKeys), q_lo + (uint32_t)t * (kQBytes >> 4),
                                        k_lo + (uint32_t)(j % KS) * (kHalfBytes >> 4), hi, idS);
                ptx::umma_commit(bar(kBarS + t));
                // the last tile's S releases the K tile, if a later tile reuses its slot
                if (t == last_tile && j + KS < n_kv) ptx::umma_commit(bar(kBarKEmpty + j % KS));
            };
            // O_t += P_t(j) V_j: 16 keys per MMA, A from TMEM; on the first KV tile also the lo part
            auto issue_pv = [&](int t, int j) {
                const uint32_t dv = v_lo + (uint32_t)(j % kVStages) * (kHalfBytes >> 4);
                const uint32_t tP = tmem + (uint32_t)(t * kKeys), tO = tmem + kColO + (uint32_t)(t * D);
                const int left = L - j * kKeys;  // keys of this tile inside the context (> 0)
                const int nk = left >= kKeys ? kKeys / 16 : (left + 15) / 16;
                if constexpr (ONE) {  // B = V^T, K-major lines of 64 keys, panels of D lines
                    umma_ts_kmajor_x8<(uint32_t)D * 8u>(tO, tP, dv, hi, idO, j > 0 ? 1u : 0u, nk);
                    if (j == 0) umma_ts_kmajor_x8<(uint32_t)D * 8u>(tO, tP + 64u, dv, hi, idO, 1u, nk);
                } else {
                    ptx::umma_ts_x8(tO, tP, dv, hi, idO, j > 0 ? 1u : 0u, nk);
                    if (j == 0) ptx::umma_ts_x8(tO, tP + 64u, dv, hi, idO, 1u, nk);
                }
            };
            if (ok) ok = wait_k(0);
            if (ok)
                for (int t = 0; t < kTiles; ++t)
                    if (nkv[t] > 0) issue_s(t, 0);
            for (int j = 0; ok && j < n_kv; ++j) {
                for (int t = 0; t < kTiles && ok; ++t) {
                    if (j >= nkv[t]) continue;
                    const bool more = j + 1 < nkv[t];
                    // everything PV_t(j) and S_t(j+1) need, before either is issued: the two
                    // batches then go out back to back and the tensor pipe's short queue stays full
                    ok = wait_v(j) && (!more || wait_k(j + 1));
                    if (!ok) break;
                    ok = ptx::mbar_wait(bar(kBarP + t), j & 1, p.wait_ns);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    issue_pv(t, j);
                    if (more) issue_s(t, j + 1);  // commits S_t and, for the last tile, K_{j+1}'s slot
                    else ptx::umma_commit(bar(kBarO + t));
                    if (t == last_tile && j + kVStages < n_kv) ptx::umma_commit(bar(kBarVEmpty + j % kVStages));
                }
            }
            if (!ok) {
                atomicOr(p.err, kErrTimeout);
                abort_s = 1;
                // let MMAs already issued finish before tensor memory is released
                ptx::umma_commit(bar(kBarDrain));
                ptx::mbar_wait(bar(kBarDrain), 0, p.wait_ns);
            }
        }
        __syncwarp();
        // every role has finished with tensor memory: release it
        ptx::named_barrier_sync(kEndBar, kThr);
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
      } else {
        ptx::named_barrier_sync(kEndBar, kThr);  // warp 3: idle member of the control warpgroup
      }
    } else {
        ptx::regs_inc<ONE ? kRegsSoftmaxOne : kRegsSoftmax>();
        // ---------------------------------------------------------------- softmax / epilogue
        const int t = (warp - kSmWarp0) >> 2;  // query tile of this warpgroup
        const int qw = warp & 3;        // TMEM lane quarter this warp may access
        const int r = qw * 32 + lane;
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const uint32_t tS = tmem + (uint32_t)(t * kKeys) + lane_off;
        const uint32_t tO = tmem + kColO + (uint32_t)(t * D) + lane_off;
        const int tok = t0 + t * T + r / p.G, g = r % p.G;
        const bool valid = tok < n;
        const int qlim = min(L - n + tok, L - 1);  // last key this row may see
        int eq = 0;  // one-byte pools: the row is staged as q x 2^eq in f16
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)(q0 + tok) * p.Hq + h * p.G + g) * D);
            uint8_t* qt = sm + kOffQ + (uint32_t)t * kQBytes;
            if constexpr (ONE) {
                // the MMA takes f16 with the widened K/V: scale the row by the power of two that
                // puts its largest |q| in [2^15, 2^16), then convert -- exact for every element
                // down to 2^-24 below that maximum (2^-31 of the row's largest term), so the
                // products are those of the bf16 q; the power of two leaves with the score scale
                uint4 v[D / 8];
                uint32_t mx = 0;  // largest bf16 magnitude bits of the row (they order like the values)
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    v[c] = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                    mx = max(mx, max(max(v[c].x & 0x7fffu, (v[c].x >> 16) & 0x7fffu),
                                     max(v[c].y & 0x7fffu, (v[c].y >> 16) & 0x7fffu)));
                    mx = max(mx, max(max(v[c].z & 0x7fffu, (v[c].z >> 16) & 0x7fffu),
                                     max(v[c].w & 0x7fffu, (v[c].w >> 16) & 0x7fffu)));
                }
                if (mx) eq = 15 - lead_exp(mx << 16);
                float fa, fb;
                pow2_pair(eq, fa, fb);
                auto cv = [&](uint32_t x) {
                    return ptx::pack_f16x2(ptx::bf16lo_to_f32(x) * fa * fb, ptx::bf16hi_to_f32(x) * fa * fb);
                };
#pragma unroll
                for (int c = 0; c < D / 8; ++c)
                    *reinterpret_cast<uint4*>(qt + (uint32_t)(c >> 3) * kPanelBytes + swz128(r, c & 7)) =
                        make_uint4(cv(v[c].x), cv(v[c].y), cv(v[c].z), cv(v[c].w));
            } else {
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(qt + (uint32_t)(c >> 3) * kPanelBytes + swz128(r, c & 7)) = v;
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarQ));
        }
        const int my_nkv = nkv[t];
        // scores in base 2: S x scale x log2(e).  One-byte pools compute S' = (q 2^eq).code: the
        // key's scale (that of its page part) multiplies the score here, per part of PART keys
        float c2 = p.scale_log2;
        // One-byte pools: per page part q of the tile, kmul[q] = c2 x 2^-eq x the part's K scale
        // multiplies the scores; with parts of 32 or more keys lgv[q] = log2(the part's V scale x
        // 2^-eV) also joins the exponent, so P' = p x V scale x 2^-eV comes out of the same ex2
        // and V is widened exactly, the row sum taking P' x 2^-lgv[q] (the p the definition sums).
        float kmul[kParts], lgv[kParts];
        float2 snext = make_float2(1.f, 1.f);  // lane q < kParts: part q's (K, V) scales of the next tile
        const int32_t* tbs = p.tables + (int64_t)b * p.max_blocks;
        // part `lane`'s scales of tile j (1 past the context: a multiplier > 0 keeps masked -inf
        // scores -inf)
        auto load_scales2 = [&](int j) -> float2 {
            float2 v = make_float2(1.f, 1.f);
            if (lane < kParts) {
                const int tok = j * kKeys + lane * PART;
                if (tok < L) {
                    const int blk = tbs[tok / p.bs];
                    if (blk >= 0 && blk < p.num_blocks)
                        v = *reinterpret_cast<const float2*>(p.scales + ((int64_t)blk * p.Hkv + h) * 4);
                }
            }
            return v;
        };
        float vfa = 1.f, vfb = 1.f;  // 2^-eV
        if constexpr (ONE) {
            float fa, fb;
            pow2_pair(-eq, fa, fb);
            c2 = c2 * fa * fb;
            pow2_pair(-scale_exp_v(), vfa, vfb);
            snext = load_scales2(0);
        }
        // P into tensor memory: f16 beside f16 V (one-byte pools), bf16 otherwise
        auto packP = [](float lo, float hi) { return ONE ? ptx::pack_f16x2(lo, hi) : ptx::pack_bf16x2(lo, hi); };
        float m = -INFINITY, l = 0.f;  // running maximum (scaled, base 2) and sum
        bool ok = true;
        for (int j = 0; j < my_nkv; ++j) {
            if constexpr (ONE) {
#pragma unroll
                for (int q = 0; q < kParts; ++q) {
                    kmul[q] = c2 * __shfl_sync(0xffffffffu, snext.x, q);
                    if constexpr (VS) lgv[q] = __log2f(__shfl_sync(0xffffffffu, snext.y, q) * vfa * vfb);
                }
                if (j + 1 < my_nkv) snext = load_scales2(j + 1);  // in flight while this tile waits
            }
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarS + t), j & 1, p.wait_ns));
            if (!ok) break;
            ptx::tc_fence_after();
            uint32_t sraw[kKeys];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(sraw + 32 * c));
            ptx::tmem_wait_ld();
            const int kbase = j * kKeys;
            if (kbase + kKeys - 1 > qlim) {  // the tile crosses this row's position: mask
#pragma unroll
                for (int c = 0; c < kKeys; ++c)
                    if (kbase + c > qlim) sraw[c] = __float_as_uint(-INFINITY);
            }
            // row maximum: three-input max into 4 independent accumulators (64 instructions,
            // no serial chain of 128 dependent ones)
            float mt;  // this tile's maximum, scaled (finite: key kbase <= qlim)
            if constexpr (ONE) {
                // per page part: its maximum times its multiplier (both > 0 scales), then across parts
                mt = -INFINITY;
#pragma unroll
                for (int q = 0; q < kParts; ++q) {
                    float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
                    for (int c = q * PART; c < (q + 1) * PART; c += 4) {
                        a0 = ptx::max3(a0, __uint_as_float(sraw[c]), __uint_as_float(sraw[c + 1]));
                        a1 = ptx::max3(a1, __uint_as_float(sraw[c + 2]), __uint_as_float(sraw[c + 3]));
                    }
                    mt = fmaxf(mt, fmaxf(a0, a1) * kmul[q]);
                }
            } else {
                float mx4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) mx4[e] = -INFINITY;
#pragma unroll
                for (int c = 0; c < kKeys; c += 2)
                    mx4[(c >> 1) & 3] = ptx::max3(mx4[(c >> 1) & 3], __uint_as_float(sraw[c]), __uint_as_float(sraw[c + 1]));
                mt = ptx::max3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]) * c2;
            }
            // lazy rescale: keep the running maximum unless this tile exceeds it by 2^8
            const bool grow = mt > m + kRescaleLog2;
            if (__any_sync(0xffffffffu, grow && j > 0)) {
                const float alpha = (grow && j > 0) ? ptx::exp2_approx(m - mt) : 1.f;
                l *= alpha;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tO + 32u * c, v);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    ptx::tmem_st32(tO + 32u * c, v);
                }
            }
            if (grow) m = mt;
            // p = 2^(s * c2 - m) for a pair of columns per instruction; l accumulates in 4
            // packed pairs (8 independent sums, columns 2e, 2e + 1 into pair e mod 4)
            const uint64_t c2x2 = ptx::f32x2(c2, c2), nmx2 = ptx::f32x2(-m, -m);
            uint64_t l4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) l4[e] = 0ull;  // +0.0f in both halves
            if (j == 0) {  // P as hi + lo bf16 pair: columns 0-63 and 64-127; l from p itself
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t hi[32], lo[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int q = (64 * c + 2 * e) / PART;  // page part of this pair (unrolled)
                        const float mul = ONE ? kmul[q] : c2, nm = VS ? lgv[q] - m : -m;
                        const float2 x = ptx::f32x2_split(ptx::fma_f32x2(
                            ptx::f32x2(__uint_as_float(sraw[64 * c + 2 * e]), __uint_as_float(sraw[64 * c + 2 * e + 1])),
                            ONE ? ptx::f32x2(mul, mul) : c2x2, VS ? ptx::f32x2(nm, nm) : nmx2));
                        const float p0 = ptx::exp2_approx(x.x), p1 = ptx::exp2_approx(x.y);
                        hi[e] = packP(p0, p1);
                        if constexpr (ONE) {
                            const float2 hv = ptx::f16x2_to_f32x2(hi[e]);
                            lo[e] = packP(p0 - hv.x, p1 - hv.y);
                        } else {
                            lo[e] = packP(p0 - ptx::bf16lo_to_f32(hi[e]), p1 - ptx::bf16hi_to_f32(hi[e]));
                        }
                        if constexpr (VS) {
                            const float iv = ptx::exp2_approx(-lgv[q]);
                            l4[e & 3] = ptx::fma_f32x2(ptx::f32x2(p0, p1), ptx::f32x2(iv, iv), l4[e & 3]);
                        } else {
                            l4[e & 3] = ptx::add_f32x2(l4[e & 3], ptx::f32x2(p0, p1));
                        }
                    }
                    ptx::tmem_st32(tS + 32u * c, hi);
                    ptx::tmem_st32(tS + 64u + 32u * c, lo);
                }
            } else {  // l from the unrounded p: the rounding of P averages out over the context
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t hi[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int q = (64 * c + 2 * e) / PART;  // page part of this pair (unrolled)
                        const float mul = ONE ? kmul[q] : c2, nm = VS ? lgv[q] - m : -m;
                        const float2 x = ptx::f32x2_split(ptx::fma_f32x2(
                            ptx::f32x2(__uint_as_float(sraw[64 * c + 2 * e]), __uint_as_float(sraw[64 * c + 2 * e + 1])),
                            ONE ? ptx::f32x2(mul, mul) : c2x2, VS ? ptx::f32x2(nm, nm) : nmx2));
                        const float p0 = ptx::exp2_approx(x.x), p1 = ptx::exp2_approx(x.y);
                        hi[e] = packP(p0, p1);
                        if constexpr (VS) {
                            const float iv = ptx::exp2_approx(-lgv[q]);
                            l4[e & 3] = ptx::fma_f32x2(ptx::f32x2(p0, p1), ptx::f32x2(iv, iv), l4[e & 3]);
                        } else {
                            l4[e & 3] = ptx::add_f32x2(l4[e & 3], ptx::f32x2(p0, p1));
                        }
                    }
                    ptx::tmem_st32(tS + 32u * c, hi);
                }
            }
            {
                const float2 a = ptx::f32x2_split(l4[0]), b = ptx::f32x2_split(l4[1]);
                const float2 cc = ptx::f32x2_split(l4[2]), d = ptx::f32x2_split(l4[3]);
                l += ((a.x + a.y) + (b.x + b.y)) + ((cc.x + cc.y) + (d.x + d.y));
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarP + t));
        }
        if (ok && my_nkv > 0) {
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarO + t), 0, p.wait_ns));
            if (ok) {
                ptx::tc_fence_after();
                float inv = 1.f / l;
                if constexpr (ONE) {  // O was accumulated over V x 2^-eV
                    float fa, fb;
                    pow2_pair(scale_exp_v(), fa, fb);
                    inv = inv * fa * fb;
                }
                uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + tok) * p.Hq + h * p.G + g) * D);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(tO + 32u * c, v);
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
            }
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, kErrTimeout);
            abort_s = 1;
        }
        ptx::tc_fence_before();
        ptx::named_barrier_sync(kEndBar, kThr);
    }
}

}  // namespace prefill

namespace {

template <int KV>
void configure_kv() {
    using namespace prefill;
    constexpr int s128 = (int)Layout<128, KV != 0>::kSmemBytes, s64 = (int)Layout<64, KV != 0>::kSmemBytes;
    cudaFuncSetAttribute(prefill_kernel<16, 128, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, s128);
    cudaFuncSetAttribute(prefill_kernel<32, 128, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, s128);
    cudaFuncSetAttribute(prefill_kernel<64, 128, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, s128);
    cudaFuncSetAttribute(prefill_kernel<16, 64, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, s64);
    cudaFuncSetAttribute(prefill_kernel<32, 64, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, s64);
    cudaFuncSetAttribute(prefill_kernel<64, 64, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, s64);
}

// the instance for (page part, head_dim, KV type)
template <int KV>
const void* kernel_for(int part, bool d64) {
    using prefill::prefill_kernel;
    if (d64) {
        switch (part) {
            case 16: return (const void*)prefill_kernel<16, 64, KV>;
            case 32: return (const void*)prefill_kernel<32, 64, KV>;
            default: return (const void*)prefill_kernel<64, 64, KV>;
        }
    }
    switch (part) {
        case 16: return (const void*)prefill_kernel<16, 128, KV>;
        case 32: return (const void*)prefill_kernel<32, 128, KV>;
        default: return (const void*)prefill_kernel<64, 128, KV>;
    }
}

}  // namespace

void prefill_configure(pkv_pool* pool) {
    (void)pool;
    configure_kv<0>();
    configure_kv<1>();
    configure_kv<2>();
}

// Argument checks shared by the prefill entry points; fills the kernel parameters and grid.
pkv_status prefill_prepare(const pkv_pool* pool, const void* q, const int32_t* cu_q, int32_t max_q_len,
                           const int32_t* tables, int32_t max_blocks, const int32_t* ctx, int32_t B, int32_t Hq,
                           float scale, void* out, prefill::Params& p, dim3& grid) {
    using namespace prefill;
    if (!pool || B < 0 || max_q_len < 0 || Hq < 1) return PKV_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;  // masking relies on scale > 0
    if (pool->head_dim != 64 && pool->head_dim != 128) return PKV_ERR_INVALID_ARG;
    if (Hq % pool->n_kv_heads) return PKV_ERR_INVALID_ARG;
    const int G = Hq / pool->n_kv_heads;
    if (G > kRows || (G & (G - 1))) return PKV_ERR_INVALID_ARG;
    if (pool->n_kv_heads > 65535) return PKV_ERR_INVALID_ARG;
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
    p.scales = pool->scales;
    p.err = pool->err;
    p.Hq = Hq;
    p.Hkv = pool->n_kv_heads;
    p.G = G;
    p.max_blocks = max_blocks;
    p.bs = pool->block_size;
    p.part = pool->block_size < 64 ? pool->block_size : 64;
    p.num_blocks = pool->num_blocks;
    p.tiles = (max_q_len + kTiles * T - 1) / (kTiles * T);  // pairs of query tiles
    p.oob_row = (int32_t)((int64_t)pool->num_blocks * 2 * pool->n_kv_heads * pool->block_size);
    p.scale_log2 = scale * 1.4426950408889634f;
    // Test hooks for the bounded waits (failure detection is tested without a GPU fault): a
    // shorter wait limit, and K/V stages that expect 16 bytes no copy delivers, so the waits run
    // out and the call reports PKV_ERR_TIMEOUT (both off unless set, see Settings).
    const Settings& hooks = settings();
    p.wait_ns = hooks.wait_limit_ms > 0 ? (uint64_t)hooks.wait_limit_ms * 1000000ull : kWaitLimitNs;
    p.stall_tx = hooks.stall_copies ? 16u : 0u;
    p.B = B;
    const int64_t ctas = (int64_t)B * pool->n_kv_heads * p.tiles;
    if (ctas > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    grid = dim3((unsigned)ctas);
    return PKV_OK;
}

pkv_status prefill_launch(const pkv_pool* pool, const prefill::Params& p, dim3 grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(pool->dtype != PKV_KV_BF16 ? prefill::kThreadsOne : prefill::kThreads);
    const bool d64 = pool->head_dim == 64;
    const bool one = pool->dtype != PKV_KV_BF16;
    cfg.dynamicSmemBytes = d64 ? (one ? prefill::Layout<64, true>::kSmemBytes : prefill::Layout<64, false>::kSmemBytes)
                               : (one ? prefill::Layout<128, true>::kSmemBytes : prefill::Layout<128, false>::kSmemBytes);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const void* fn = pool->dtype == PKV_KV_FP8_E4M3 ? kernel_for<1>(p.part, d64)
                     : pool->dtype == PKV_KV_INT8   ? kernel_for<2>(p.part, d64)
                                                    : kernel_for<0>(p.part, d64);
    void* args[] = {const_cast<CUtensorMap*>(&pool->tmap_panel), const_cast<prefill::Params*>(&p)};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
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
