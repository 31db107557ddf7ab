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
//              stay faster than the ~65 cycles an M=128 N=128 K=16 MMA takes).
//              so one tile's MMAs run while the other tile's softmax works.
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
constexpr int kKStages = 3;  // K ring: a K tile is free once both tiles' S MMAs have read it
constexpr int kVStages = 2;  // V ring: a V tile is free once both tiles' PV MMAs have read it
constexpr int kThreads = 128 + kTiles * 128;  // control warpgroup + one softmax warpgroup per tile
// register split (setmaxnreg): launched at 168 per thread (65536 / 384, rounded down to 8),
// i.e. 64512 for the block; control 128 x 48 + softmax 256 x 224 = 63488 fits.
constexpr uint32_t kRegsControl = 48, kRegsSoftmax = 224;
static_assert(128 * kRegsControl + kTiles * 128 * kRegsSoftmax <= kThreads * 168, "register split");
constexpr uint32_t kPanelBytes = 128u * 128u;      // 128 rows x 128 bytes (64 bf16 of a row)
constexpr uint32_t kOffQ = 0;
// Shared-memory layout for head_dim D (64 or 128): a row of Q, K or V is D / 64 panels.
template <int D>
struct Layout {
    static constexpr int kPanels = D / 64;
    static constexpr uint32_t kQBytes = kPanels * kPanelBytes;     // one Q tile
    static constexpr uint32_t kHalfBytes = kPanels * kPanelBytes;  // K (or V) of one KV tile
    static constexpr uint32_t kOffK = kOffQ + kTiles * kQBytes;
    static constexpr uint32_t kOffV = kOffK + kKStages * kHalfBytes;
    static constexpr uint32_t kOffBar = kOffV + kVStages * kHalfBytes;
    static constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (P stays <= 2^8)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kEndBar = 1;      // named barrier: every role done before TMEM is released
constexpr int kMaxRankedSeqs = 512;  // above this the sequences are dispatched in index order
constexpr int kSmallRankedSeqs = 64;  // up to this the ranking reads the inputs directly
static_assert(kMaxRankedSeqs * sizeof(int64_t) <= kTiles * Layout<64>::kQBytes, "dispatch ranking fits the Q tiles' space");

// mbarrier slots
constexpr int kBarQ = 0;                          // Q rows of both tiles written (8 warps arrive)
constexpr int kBarKFull = 1;                      // [kKStages] K copies landed (tx bytes)
constexpr int kBarKEmpty = kBarKFull + kKStages;  // [kKStages] last S MMA reading the K tile done
constexpr int kBarVFull = kBarKEmpty + kKStages;  // [kVStages] V copies landed (tx bytes)
constexpr int kBarVEmpty = kBarVFull + kVStages;  // [kVStages] last PV MMA reading the V tile done
constexpr int kBarS = kBarVEmpty + kVStages;      // [kTiles] S_t(j) ready (commit)
constexpr int kBarP = kBarS + kTiles;             // [kTiles] P_t(j) in TMEM (4 warps arrive)
constexpr int kBarO = kBarP + kTiles;             // [kTiles] last PV_t done (commit)
constexpr int kBarDrain = kBarO + kTiles;         // MMAs in flight done (error path)
constexpr int kNumBars = kBarDrain + 1;
static_assert(kNumBars * 8 <= 256, "barrier area");

struct Params {
    const uint16_t* q;
    uint16_t* out;
    const int32_t* cu_q;
    const int32_t* tables;
    const int32_t* ctx;
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

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

template <int PART, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap, const Params p) {
    static_assert(PART == 16 || PART == 32 || PART == 64, "page part of 16, 32 or 64 rows");
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    using LY = Layout<D>;
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
        for (int i = threadIdx.x; i < p.B; i += kThreads) {
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
        for (int i = threadIdx.x; i < p.B; i += kThreads) {
            const int64_t nn = p.cu_q[i + 1] - p.cu_q[i], ll = p.ctx[i];
            work_s[i] = nn * (2 * ll - nn);
        }
        if (threadIdx.x == 0) seq_of_rank = -1;
        __syncthreads();
        for (int i = threadIdx.x; i < p.B; i += kThreads) {
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

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool wg_arrive = i == kBarQ || (i >= kBarP && i < kBarP + kTiles);
            ptx::mbar_init(bar(i), i == kBarQ ? 8u : (wg_arrive ? 4u : 1u));
        }
        abort_s = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_addr(&tmem_base_s), kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp < 4) {
      ptx::regs_dec<kRegsControl>();  // the whole control warpgroup, one instruction
      if (warp == 0 || warp == 2) {
        // ---------------------------------------------------------------- producers
        // warp 0 fills the K ring, warp 2 the V ring; each KV tile is two 128-row panels (the
        // 64-element halves), one 2-D copy of PART rows per (page part, half)
        const int kv = warp == 0 ? 0 : 1;
        const int stages = kv ? kVStages : kKStages;
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
        ptx::named_barrier_sync(kEndBar, kThreads);
      } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // descriptors are built once; the start-address field counts 16-byte units, so moving
            // an operand by X bytes adds X >> 4 (addresses stay below 256 KB: no carry out)
            constexpr uint32_t idS = ptx::umma_idesc_bf16(128, kKeys, 0, 0);
            constexpr uint32_t idO = ptx::umma_idesc_bf16(128, D, 0, 1);
            // a descriptor's high half (stride, version, swizzle) is the same for Q and K; V's
            // differs only in the low half (its panel stride)
            const uint64_t dQ0 = ptx::umma_sdesc_sw128(base + kOffQ, 16, 1024);
            const uint64_t dK0 = ptx::umma_sdesc_sw128(sK, 16, 1024);
            const uint64_t dV0 = ptx::umma_sdesc_sw128(sV, kPanelBytes, 1024);
            const uint32_t hi = (uint32_t)(dQ0 >> 32);
            const uint32_t q_lo = (uint32_t)dQ0, k_lo = (uint32_t)dK0, v_lo = (uint32_t)dV0;
            int k_ready = 0, v_ready = 0;  // K / V tiles whose copies this thread has waited for
            bool ok = ptx::mbar_wait(bar(kBarQ), 0, p.wait_ns);
            ptx::tc_fence_after();
            auto wait_k = [&](int j) -> bool {
                if (j < k_ready) return true;
                if (!ptx::mbar_wait(bar(kBarKFull + j % kKStages), (j / kKStages) & 1, p.wait_ns)) return false;
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
                                         k_lo + (uint32_t)(j % kKStages) * (kHalfBytes >> 4), hi, idS);
                else
                    umma_ss_k64_x4(tmem + (uint32_t)(t * kKeys), q_lo + (uint32_t)t * (kQBytes >> 4),
                                        k_lo + (uint32_t)(j % kKStages) * (kHalfBytes >> 4), hi, idS);
                ptx::umma_commit(bar(kBarS + t));
                // the last tile's S releases the K tile, if a later tile reuses its slot
                if (t == last_tile && j + kKStages < n_kv) ptx::umma_commit(bar(kBarKEmpty + j % kKStages));
            };
            // O_t += P_t(j) V_j: 16 keys per MMA, A from TMEM; on the first KV tile also the lo part
            auto issue_pv = [&](int t, int j) {
                const uint32_t dv = v_lo + (uint32_t)(j % kVStages) * (kHalfBytes >> 4);
                const uint32_t tP = tmem + (uint32_t)(t * kKeys), tO = tmem + kColO + (uint32_t)(t * D);
                const int left = L - j * kKeys;  // keys of this tile inside the context (> 0)
                const int nk = left >= kKeys ? kKeys / 16 : (left + 15) / 16;
                ptx::umma_ts_x8(tO, tP, dv, hi, idO, j > 0 ? 1u : 0u, nk);
                if (j == 0) ptx::umma_ts_x8(tO, tP + 64u, dv, hi, idO, 1u, nk);
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
        ptx::named_barrier_sync(kEndBar, kThreads);
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
      } else {
        ptx::named_barrier_sync(kEndBar, kThreads);  // warp 3: idle member of the control warpgroup
      }
    } else {
        ptx::regs_inc<kRegsSoftmax>();
        // ---------------------------------------------------------------- softmax / epilogue
        const int t = (warp - 4) >> 2;  // query tile of this warpgroup
        const int qw = warp & 3;        // TMEM lane quarter this warp may access
        const int r = qw * 32 + lane;
        const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
        const uint32_t tS = tmem + (uint32_t)(t * kKeys) + lane_off;
        const uint32_t tO = tmem + kColO + (uint32_t)(t * D) + lane_off;
        const int tok = t0 + t * T + r / p.G, g = r % p.G;
        const bool valid = tok < n;
        const int qlim = min(L - n + tok, L - 1);  // last key this row may see
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)(q0 + tok) * p.Hq + h * p.G + g) * D);
            uint8_t* qt = sm + kOffQ + (uint32_t)t * kQBytes;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(qt + (uint32_t)(c >> 3) * kPanelBytes + swz128(r, c & 7)) = v;
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarQ));
        }
        const int my_nkv = nkv[t];
        const float c2 = p.scale_log2;
        float m = -INFINITY, l = 0.f;  // running maximum (scaled, base 2) and sum
        bool ok = true;
        for (int j = 0; j < my_nkv; ++j) {
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
            float mx4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) mx4[e] = -INFINITY;
#pragma unroll
            for (int c = 0; c < kKeys; c += 2)
                mx4[(c >> 1) & 3] = ptx::max3(mx4[(c >> 1) & 3], __uint_as_float(sraw[c]), __uint_as_float(sraw[c + 1]));
            const float smax = ptx::max3(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
            const float mt = smax * c2;  // this tile's maximum, scaled (finite: key kbase <= qlim)
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
                        const float2 x = ptx::f32x2_split(ptx::fma_f32x2(
                            ptx::f32x2(__uint_as_float(sraw[64 * c + 2 * e]), __uint_as_float(sraw[64 * c + 2 * e + 1])),
                            c2x2, nmx2));
                        const float p0 = ptx::exp2_approx(x.x), p1 = ptx::exp2_approx(x.y);
                        hi[e] = ptx::pack_bf16x2(p0, p1);
                        lo[e] = ptx::pack_bf16x2(p0 - ptx::bf16lo_to_f32(hi[e]), p1 - ptx::bf16hi_to_f32(hi[e]));
                        l4[e & 3] = ptx::add_f32x2(l4[e & 3], ptx::f32x2(p0, p1));
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
                        const float2 x = ptx::f32x2_split(ptx::fma_f32x2(
                            ptx::f32x2(__uint_as_float(sraw[64 * c + 2 * e]), __uint_as_float(sraw[64 * c + 2 * e + 1])),
                            c2x2, nmx2));
                        const float p0 = ptx::exp2_approx(x.x), p1 = ptx::exp2_approx(x.y);
                        hi[e] = ptx::pack_bf16x2(p0, p1);
                        l4[e & 3] = ptx::add_f32x2(l4[e & 3], ptx::f32x2(p0, p1));
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
                const float inv = 1.f / l;
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
        ptx::named_barrier_sync(kEndBar, kThreads);
    }
}

}  // namespace prefill

void prefill_configure(pkv_pool* pool) {
    (void)pool;
    using namespace prefill;
    cudaFuncSetAttribute(prefill_kernel<16, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<128>::kSmemBytes);
    cudaFuncSetAttribute(prefill_kernel<32, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<128>::kSmemBytes);
    cudaFuncSetAttribute(prefill_kernel<64, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<128>::kSmemBytes);
    cudaFuncSetAttribute(prefill_kernel<16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<64>::kSmemBytes);
    cudaFuncSetAttribute(prefill_kernel<32, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<64>::kSmemBytes);
    cudaFuncSetAttribute(prefill_kernel<64, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Layout<64>::kSmemBytes);
}

// Argument checks shared by the prefill entry points; fills the kernel parameters and grid.
pkv_status prefill_prepare(const pkv_pool* pool, const void* q, const int32_t* cu_q, int32_t max_q_len,
                           const int32_t* tables, int32_t max_blocks, const int32_t* ctx, int32_t B, int32_t Hq,
                           float scale, void* out, prefill::Params& p, dim3& grid) {
    using namespace prefill;
    if (!pool || B < 0 || max_q_len < 0 || Hq < 1) return PKV_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;  // masking relies on scale > 0
    if (pool->dtype != PKV_KV_BF16 || (pool->head_dim != 64 && pool->head_dim != 128)) return PKV_ERR_INVALID_ARG;
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
    cfg.blockDim = dim3(prefill::kThreads);
    const bool d64 = pool->head_dim == 64;
    cfg.dynamicSmemBytes = d64 ? prefill::Layout<64>::kSmemBytes : prefill::Layout<128>::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    using prefill::prefill_kernel;
    cudaError_t e;
    if (d64) {
        switch (p.part) {
            case 16: e = cudaLaunchKernelEx(&cfg, prefill_kernel<16, 64>, pool->tmap_panel, p); break;
            case 32: e = cudaLaunchKernelEx(&cfg, prefill_kernel<32, 64>, pool->tmap_panel, p); break;
            default: e = cudaLaunchKernelEx(&cfg, prefill_kernel<64, 64>, pool->tmap_panel, p); break;
        }
    } else {
        switch (p.part) {
            case 16: e = cudaLaunchKernelEx(&cfg, prefill_kernel<16, 128>, pool->tmap_panel, p); break;
            case 32: e = cudaLaunchKernelEx(&cfg, prefill_kernel<32, 128>, pool->tmap_panel, p); break;
            default: e = cudaLaunchKernelEx(&cfg, prefill_kernel<64, 128>, pool->tmap_panel, p); break;
        }
    }
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
