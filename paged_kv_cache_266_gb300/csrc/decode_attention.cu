// Decode attention over the paged KV pool ("TensorRT-LLM 推理加速实战", §7.2 masked_mha: the
// decode phase attends one new query token per request to that request's cached K/V; §8:
// paged blocks of 16/64 tokens, FP8 e4m3 KV).  For sequence b and query head j, with KV head
// h = j / G (GQA sharing, "TensorRT-LLM加速大模型推理实战"):
//     out[b][j] = sum_t softmax_t(scale * q[b][j] . K_b[t]) V_b[t].
//
// Work decomposition (GB300: 152 SMs, HBM-bound):
//  * Every (sequence, KV head) pair's context is cut into 64-token groups; the groups of all
//    pairs, laid end to end (pairs in (b, h) order), are split into gridDim.x contiguous,
//    equal ranges, one per CTA.  The grid is sized to the resident CTA count, so one wave
//    streams the whole pool at an even rate whatever the context-length mix.
//  * A CTA is one producer warp and four consumer warps.  The producer walks its range and,
//    per group, issues TMA tensor copies (cp.async.bulk.tensor, 128-byte swizzled rows) of the
//    K and V rows of that group's pages into a ring of shared-memory stages, completion
//    tracked by mbarriers; plus the query rows at each new pair and, for fp8, the 16-byte
//    scale records of the pages.  Block ids come from the block table, fetched 32 groups
//    ahead by the producer's lanes.
//  * Consumer warp w owns tokens [16w, 16w+16) of every group.  The whole query group of
//    the KV head (G <= 8 heads) is one MMA N-tile, so each K/V byte is read from HBM once:
//        S^T[16 tok][8 heads] = K[16 tok][D] . Q^T    (mma.sync m16n8k16, fp32 accumulate)
//        online softmax on S^T in registers (base-2 exponent, scale*log2 e folded in)
//        P^T -> B fragment via movmatrix (register transpose, no shared-memory round trip)
//        O^T[D][8 heads] += V^T[D][16 tok] . P^T       (ldmatrix.trans for bf16 V)
//    fp8 codes are widened to f16 in registers (exact); the K scale multiplies the scores,
//    the V scale is folded into the running rescale factor.  The query rows are scaled per
//    head by a power of two into f16's range before their conversion, which keeps it exact
//    for any bf16 query; the inverse power of two joins the head's score scale.
//  * When a pair ends inside the CTA the four warps' (max, sum, O) states are merged through
//    shared memory and the result is written as bf16.  A pair cut between CTAs leaves one
//    partial state per CTA in the workspace; the last CTA to finish (atomic ticket, no
//    waiting) merges them with the log-sum-exp rule in slot order, so results do not depend
//    on timing.
//  * pkv_decode_step on a one-byte pool appends inside this kernel: while the producers look up
//    their first block ids, the consumer warps of all CTAs quantise the step's new K/V rows into
//    the pool, one warp per row pair, and count them in the workspace; every producer waits for
//    the count before it reads a page or a scale.  The launch is cooperative (every CTA resident
//    at once), as CTAs wait on rows other CTAs write.  A separate append kernel would take the
//    registers the third one-byte CTA of each SM needs, so that CTA could start only after it.
//
// Every mbarrier wait is bounded (2 s of wall time); on expiry the kernel sets the pool's
// error word and finishes without touching memory outside its buffers.
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace pkv {
namespace attn {

constexpr int kConsumerWarps = 4;
constexpr int kGroup = 16 * kConsumerWarps;  // tokens per pipeline stage
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxG = 8;
constexpr int kMaxStages = 8;
constexpr int kMaxBatch = 4096;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kFusedAppendMax = 1024;  // pkv_decode_step quantises up to this many tokens in-kernel
// The step's own append counts its items in kAppCounters words kAppStride ints apart (separate
// 128-byte lines, so the items' atomics and the producers' polls spread over the L2), followed by
// the word that counts CTAs done with the pool.
constexpr int kAppCounters = 32;
constexpr int kAppStride = 32;
constexpr int kAppWords = kAppCounters * kAppStride + 1;
constexpr uint32_t kCombineBar = 1;  // named barrier of the consumer warps

struct Params {
    const uint16_t* q;
    const int32_t* tables;
    const int32_t* lens;
    uint16_t* out;
    const uint8_t* pool;
    const float* scales;
    int* counters;
    float* partials;  // O of the partial states [slots][G][D]
    float* part_ml;   // their (max, sum) [slots][G][2]
    int* err;
    int B, Hq, Hkv, G, max_blocks, bs, num_blocks;
    int box_rows;  // rows per TMA box: min(bs, kGroup)
    int ppg;       // page parts per group: kGroup / box_rows
    int stages;
    uint32_t stage_bytes, off_q, off_s;  // within a stage: page parts, query rows, fp8 scale pairs
    uint32_t off_bar, off_misc, off_cmb, off_lens;  // within the shared-memory block
    float scale_log2;
    uint64_t wait_ns;   // bound of every mbarrier wait
    uint32_t stall_tx;  // test hook: bytes each stage expects beyond its copies (0 in normal use)
    // pkv_decode_step on a one-byte pool: its n_new tokens' K and V rows ([n_new][Hkv][D] bf16)
    // and slots, quantised into the pool by this kernel (n_new = 0: nothing to append); app:
    // kAppWords workspace words (item counters, CTAs done), zero between calls.
    const uint16_t* k_new;
    const uint16_t* v_new;
    const int64_t* slots;
    int* app;
    int n_new;
    int app_extra;  // test hook: row pairs the wait expects beyond those quantised (0 in normal use)
};

// misc words in shared memory
constexpr int kMiscAbort = 0;
constexpr int kMiscMergeParts = 1;
constexpr int kQuickMergeParts = 4;  // merges of up to this many parts load everything at once
                                     // (bf16 only: the one-byte kernels are capped at 128 registers)
constexpr int kMiscMergeFirst = 2;
constexpr uint32_t kMiscQinvBytes = 32;  // after the misc words: [kConsumerWarps][kMaxG] floats

__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity, volatile int* misc, uint64_t limit_ns) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (misc[kMiscAbort]) return false;
            if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

__device__ __forceinline__ void flag_abort(const Params& p, volatile int* misc) {
    misc[kMiscAbort] = 1;
    atomicOr(p.err, kErrTimeout);
}

// Largest b with Hkv * cumg[b] <= e (pairs of empty sequences have no groups and are skipped).
__device__ __forceinline__ int find_seq(const int32_t* cumg, int B, int Hkv, int64_t e) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)Hkv * cumg[mid] <= e) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// ------------------------------------------------------------------ the step's own append
// Items: the RPP rows of one token that one warp covers (D/8 lanes of 8 elements per row), items
// of token i numbered i * nrp ... i * nrp + nrp - 1.
template <int D>
__device__ __forceinline__ int append_items(const Params& p) {
    constexpr int RPP = 32 / (D / 8);
    return p.n_new * ((2 * p.Hkv + RPP - 1) / RPP);
}

// Consumer warp `warp` quantises items warp * gridDim.x + blockIdx.x, ... into the pool, with the
// codes and scales of the appends (quant.cuh): a token opening its block (offset 0, or another
// token of the call at offset 0 of the same block) sets the scale of each (K|V, head) row to the
// row's amax over the call's tokens in that block / 448 (int8: / 127); any other token uses the
// stored scale, which no token of the call writes.  Each item is counted in one of the
// kAppCounters words once its stores are visible at GPU scope and to TMA reads.
struct AppendPre {
    int64_t slot;
    uint4 v;
};

// The first item's slot and row, loaded before the kernel's set-up so that they arrive meanwhile.
template <int D>
__device__ __forceinline__ AppendPre append_preload(const Params& p, int warp) {
    constexpr int TPR = D / 8, RPP = 32 / TPR;
    const int lane = threadIdx.x & 31, part = lane % TPR, rsub = lane / TPR;
    const int rows = 2 * p.Hkv, nrp = (rows + RPP - 1) / RPP;
    const int it = warp * (int)gridDim.x + (int)blockIdx.x;
    AppendPre pre{-1, make_uint4(0u, 0u, 0u, 0u)};
    if (it < append_items<D>(p)) {
        const int i = it / nrp, r = (it - i * nrp) * RPP + rsub;
        pre.slot = __ldg(p.slots + i);
        if (r < rows) {
            const int kv = r / p.Hkv, h = r - kv * p.Hkv;
            pre.v = __ldg(reinterpret_cast<const uint4*>((kv ? p.v_new : p.k_new) + ((int64_t)i * p.Hkv + h) * D + part * 8));
        }
    }
    return pre;
}

template <int D, bool I8>
__device__ void append_rows(const Params& p, int warp, const AppendPre& pre) {
    constexpr int TPR = D / 8, RPP = 32 / TPR;
    const int lane = threadIdx.x & 31, part = lane % TPR, rsub = lane / TPR;
    const int rows = 2 * p.Hkv, nrp = (rows + RPP - 1) / RPP, items = append_items<D>(p);
    const int64_t cap = (int64_t)p.num_blocks * p.bs;
    const int bs_shift = __ffs(p.bs) - 1;  // block sizes are powers of two
    uint8_t* pool = const_cast<uint8_t*>(p.pool);
    float* scales = const_cast<float*>(p.scales);
    for (int it = warp * (int)gridDim.x + (int)blockIdx.x; it < items; it += kConsumerWarps * (int)gridDim.x) {
        const int i = it / nrp, r = (it - i * nrp) * RPP + rsub;
        const bool act = r < rows;
        const int kv = act ? r / p.Hkv : 0, h = act ? r - kv * p.Hkv : 0;
        const bool first = it == warp * (int)gridDim.x + (int)blockIdx.x;
        const int64_t slot = first ? pre.slot : __ldg(p.slots + i);
        const uint4 v = first ? pre.v
                        : act ? __ldg(reinterpret_cast<const uint4*>((kv ? p.v_new : p.k_new) +
                                                                     ((int64_t)i * p.Hkv + h) * D + part * 8))
                              : make_uint4(0u, 0u, 0u, 0u);
        if (slot >= cap && lane == 0 && it == i * nrp) atomicOr(p.err, kErrBounds);
        if (slot >= 0 && slot < cap) {  // one token per item: the same branch for the whole warp
            const int64_t blk = slot >> bs_shift;
            const int t = (int)(slot & (p.bs - 1));
            float* sp = scales + (blk * p.Hkv + h) * 4 + kv;
            const float stored = act ? __ldcg(sp) : 1.0f;  // used only if the block is not fresh
            // the call's other tokens in this block, and whether one of them writes offset 0
            bool same = false, zero = false;
            for (int j0 = lane; j0 < p.n_new; j0 += 4 * 32) {
                int64_t sj[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = j0 + 32 * u;
                    sj[u] = (j < p.n_new && j != i) ? __ldg(p.slots + j) : -1;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (sj[u] >= 0 && sj[u] < cap && (sj[u] >> bs_shift) == blk) {
                        same = true;
                        zero |= (sj[u] & (p.bs - 1)) == 0;
                    }
                }
            }
            const bool mates = __any_sync(0xffffffffu, same);
            const bool fresh = t == 0 || __any_sync(0xffffffffu, zero);
            float sc = stored;
            if (fresh) {
                uint32_t m = act ? quant::amax_bits(v) : 0u;
                if (mates && act) {  // rare: several tokens of the call share the block
                    const uint16_t* src = kv ? p.v_new : p.k_new;
                    for (int j = 0; j < p.n_new; ++j) {
                        const int64_t sj = __ldg(p.slots + j);
                        if (j == i || sj < 0 || sj >= cap || (sj >> bs_shift) != blk) continue;
                        m = max(m, quant::amax_bits(__ldg(
                                       reinterpret_cast<const uint4*>(src + ((int64_t)j * p.Hkv + h) * D + part * 8))));
                    }
                }
#pragma unroll
                for (int o = TPR / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
                const float a = __uint_as_float(m);
                sc = a > 0.0f ? __fdiv_rn(a, I8 ? 127.0f : 448.0f) : 1.0f;
                if (act && t == 0 && part == 0) *sp = sc;
            }
            if (act) quant::quant_store<D, I8>(pool, v, sc, blk, t, kv, h, part, p.Hkv, p.bs);
        }
        ptx::fence_proxy_async_global();
        __syncwarp();  // orders every lane's stores before lane 0's release, which covers them all
        if (lane == 0) ptx::red_add_release_gpu(p.app + (it % kAppCounters) * kAppStride, 1);
    }
}

// Producer warp: wait (bounded) until every item of the step's append is counted (lane k reads
// counter k with acquire ordering, the warp sums them); then the pool's pages (TMA) and scales
// read by this warp include the new rows.  Returns false if the wait ran out.
template <int D>
__device__ bool wait_appends(const Params& p) {
    static_assert(kAppCounters == 32, "one counter per lane");
    const int lane = threadIdx.x & 31;
    const int need = append_items<D>(p) + p.app_extra;
    const int* ctr = p.app + lane * kAppStride;
    bool ok = true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {  // every exit is taken by the whole warp at once
        if (__reduce_add_sync(0xffffffffu, (unsigned)ptx::ld_acquire_gpu(ctr)) >= (unsigned)need) break;
        if ((i & 63u) == 0 && __any_sync(0xffffffffu, ptx::globaltimer_ns() - t0 > p.wait_ns)) {
            ok = false;
            break;
        }
    }
    ptx::fence_proxy_async_global();
    return ok;
}

// Producer warp, once this CTA reads nothing more of the pool: count the CTA done; the last CTA
// returns every counter to zero for the next call.  Only after a wait that succeeded (otherwise
// the words are left as they are and the workspace must be initialised again).
__device__ void appends_done(const Params& p) {
    const int lane = threadIdx.x & 31;
    int last = 0;
    if (lane == 0) last = ptx::atomic_add_acq_rel_gpu(p.app + kAppCounters * kAppStride, 1) == (int)gridDim.x - 1;
    if (__shfl_sync(0xffffffffu, last, 0)) {
        atomicExch(p.app + lane * kAppStride, 0);
        if (lane == 0) atomicExch(p.app + kAppCounters * kAppStride, 0);
    }
}

// ------------------------------------------------------------------ producer warp
struct GroupDesc {
    int b, h, g;
    int32_t id[4];
    float sk[4], sv[4];  // fp8 scales of the group's pages (loaded one batch after the ids)
};

// Returns false if the wait for the step's own append ran out.
template <bool FP8, int D>
__device__ bool producer(const CUtensorMap* tmap, const CUtensorMap* tmap_tail, const Params& p, const int32_t* cumg, const int32_t* lens_s,
                         int64_t R0, int64_t R1, uint32_t sbase, uint32_t bar_full, uint32_t bar_empty,
                         volatile int* misc) {
    constexpr int kEsz = FP8 ? 1 : 2;
    const int lane = threadIdx.x & 31;

    auto describe = [&](int64_t e, GroupDesc& d) {
        d.b = -1;
        if (e >= R1) return;
        const int b = find_seq(cumg, p.B, p.Hkv, e);
        const int ng = cumg[b + 1] - cumg[b];
        const int r = (int)(e - (int64_t)p.Hkv * cumg[b]);  // < Hkv * ng
        d.b = b;
        d.h = r / ng;
        d.g = r - d.h * ng;
        const int npages = (lens_s[b] + p.bs - 1) / p.bs;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = p.ppg > 1 ? d.g * p.ppg + i : (d.g * kGroup) / p.bs;
            d.id[i] = (i < p.ppg && k < npages) ? __ldg(p.tables + (int64_t)b * p.max_blocks + k) : -1;
        }
    };
    // fp8: the pages' scale pairs, once their block ids have arrived (out-of-range ids read 0);
    // coherent loads, as this kernel's own append may have written them
    auto fetch_scales = [&](GroupDesc& d) {
        if constexpr (FP8) {
            if (d.b < 0) return;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int blk = (d.id[i] >= 0 && d.id[i] < p.num_blocks) ? d.id[i] : 0;
                const float2 v = __ldcg(reinterpret_cast<const float2*>(p.scales + ((int64_t)blk * p.Hkv + d.h) * 4));
                d.sk[i] = v.x;
                d.sv[i] = v.y;
            }
        }
    };

    // Three batches of 32 group descriptors in flight: ids of batch +2 and scales of batch +1
    // load while batch 0 is issued.
    GroupDesc cur, nxt, nxt2;
    describe(R0 + lane, cur);
    describe(R0 + 32 + lane, nxt);
    int s = 0;
    uint32_t round = 0;
    int64_t issued = 0;
    bool ok = true;
    const uint32_t part_bytes = 2u * (uint32_t)p.box_rows * D * kEsz;  // K rows + V rows of one page part
    // When launched behind this step's append (programmatic dependent launch), the pool and its
    // block scales (which the append sets on a block's first write) are read only after that
    // kernel has finished; otherwise this returns at once.  When this kernel appends the step's
    // tokens itself, they are read only after every row is in.  Block tables and lengths are
    // inputs the append does not write, so their look-ups above overlap it.
    ptx::grid_dependency_wait();
    const bool appended = !(FP8 && p.n_new > 0) || wait_appends<D>(p);
    if (!appended) {
        if (lane == 0) flag_abort(p, misc);
        ok = false;
    }
    fetch_scales(cur);
    for (int64_t e0 = R0; e0 < R1 && ok; e0 += 32) {
        describe(e0 + 64 + lane, nxt2);
        fetch_scales(nxt);
        const int n = (int)(R1 - e0 < 32 ? R1 - e0 : 32);
        for (int j = 0; j < n; ++j) {
            const int b = __shfl_sync(0xffffffffu, cur.b, j);
            const int h = __shfl_sync(0xffffffffu, cur.h, j);
            const int g = __shfl_sync(0xffffffffu, cur.g, j);
            const int id0 = __shfl_sync(0xffffffffu, cur.id[0], j);
            const int id1 = __shfl_sync(0xffffffffu, cur.id[1], j);
            const int id2 = __shfl_sync(0xffffffffu, cur.id[2], j);
            const int id3 = __shfl_sync(0xffffffffu, cur.id[3], j);
            const int64_t e = e0 + j;
            const bool first = (e == R0) || (g == 0);
            int nparts = 1;
            if (p.ppg > 1) nparts = min(p.ppg, (lens_s[b] + p.bs - 1) / p.bs - g * p.ppg);
            // rows of the last part that hold tokens; a partly filled last part is copied in
            // 16-row boxes up to its last token
            const int tail_rows = min(p.box_rows, lens_s[b] - g * kGroup - (nparts - 1) * p.box_rows);
            const int tail16 = (tail_rows + 15) >> 4;
            const bool tail_short = p.box_rows > 16 && tail_rows <= p.box_rows - 16;  // saves a 16-row box
            const uint32_t st = sbase + (uint32_t)s * p.stage_bytes;
            const uint32_t fb = bar_full + 8 * s;
            if (lane == 0) {
                ok = !misc[kMiscAbort] && ptx::mbar_wait(bar_empty + 8 * s, (round & 1) ^ 1, p.wait_ns);
                if (!ok) flag_abort(p, misc);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const int part = lane & 3;
            int blk = part == 0 ? id0 : part == 1 ? id1 : part == 2 ? id2 : id3;
            if (FP8) {  // scale pairs into the (now free) stage before it is published
                const float sk0 = __shfl_sync(0xffffffffu, cur.sk[0], j), sv0 = __shfl_sync(0xffffffffu, cur.sv[0], j);
                const float sk1 = __shfl_sync(0xffffffffu, cur.sk[1], j), sv1 = __shfl_sync(0xffffffffu, cur.sv[1], j);
                const float sk2 = __shfl_sync(0xffffffffu, cur.sk[2], j), sv2 = __shfl_sync(0xffffffffu, cur.sv[2], j);
                const float sk3 = __shfl_sync(0xffffffffu, cur.sk[3], j), sv3 = __shfl_sync(0xffffffffu, cur.sv[3], j);
                if (lane < nparts) {
                    const float sk = part == 0 ? sk0 : part == 1 ? sk1 : part == 2 ? sk2 : sk3;
                    const float sv = part == 0 ? sv0 : part == 1 ? sv1 : part == 2 ? sv2 : sv3;
                    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(st + p.off_s + 8 * lane), "f"(sk), "f"(sv)
                                 : "memory");
                }
                __syncwarp();
            }
            if (lane == 0)
                ptx::mbar_arrive_expect_tx(fb, (uint32_t)(nparts - (tail_short ? 1 : 0)) * part_bytes +
                                                   (tail_short ? (uint32_t)tail16 * 32u * D * kEsz : 0u) +
                                                   (first ? (uint32_t)(p.G * D * 2) : 0u) + p.stall_tx);
            __syncwarp();  // the expect-tx precedes every lane's copies
            // Lanes 0..nparts-1 issue one page part each (K and V rows in one tensor copy) and
            // lane 4 the query rows, so a stage's copies go out in parallel.
            if (lane < nparts) {
                if (blk < 0 || blk >= p.num_blocks) {  // keep the byte count exact, read block 0
                    atomicOr(p.err, kErrBounds);
                    blk = 0;
                }
                const int row_off = p.ppg > 1 ? 0 : (g * kGroup) & (p.bs - 1);
                const int32_t rowK = (int32_t)(((int64_t)(2 * blk) * p.Hkv + h) * p.bs + row_off);
                const uint32_t dst = st + (uint32_t)lane * part_bytes;
                if (tail_short && lane == nparts - 1) {
                    constexpr int kPanels = FP8 ? 1 : D / 64;
                    constexpr uint32_t kPanelRowBytes = FP8 ? D : 128;
                    const int32_t rowV = rowK + p.Hkv * p.bs;
                    for (int t = 0; t < tail16; ++t)
#pragma unroll
                        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
                            for (int q = 0; q < kPanels; ++q)
                                ptx::tma_load_2d(dst + (uint32_t)((kv * kPanels + q) * p.box_rows + 16 * t) * kPanelRowBytes,
                                                 tmap_tail, q * 64, (kv ? rowV : rowK) + 16 * t, fb);
                } else if (!FP8 && D == 128) {
                    ptx::tma_load_4d(dst, tmap, 0, rowK, 0, 0, fb);
                } else {
                    ptx::tma_load_3d(dst, tmap, 0, rowK, 0, fb);
                }
            } else if (lane == 4 && first) {
                ptx::bulk_load(st + p.off_q, p.q + ((int64_t)b * p.Hq + (int64_t)h * p.G) * D, (uint32_t)(p.G * D * 2),
                               fb);
            }
            ++issued;
            if (++s == p.stages) {
                s = 0;
                ++round;
            }
        }
        cur = nxt;
        nxt = nxt2;
    }
    // Do not leave while copies into this CTA's shared memory may still be landing.
    if (lane == 0) {
        const int64_t lo = issued > p.stages ? issued - p.stages : 0;
        for (int64_t qq = issued - 1; qq >= lo; --qq)
            if (!ptx::mbar_wait(bar_full + 8 * (int)(qq % p.stages), (uint32_t)((qq / p.stages) & 1), p.wait_ns)) {
                flag_abort(p, misc);
                break;
            }
    }
    __syncwarp();
    return appended;
}

// ------------------------------------------------------------------ consumer math
struct SoftmaxState {
    float m[2];  // running max (base-2 units) of heads 2c, 2c+1
    float l[2];  // per-lane partial sums of exp2(z - m)
};

// Online-softmax step on one 16-token S^T tile.  acc: (t=g, j=2c), (g, 2c+1), (g+8, 2c),
// (g+8, 2c+1); sl0 / sl1 scale the scores of heads 2c / 2c+1.  Returns the rescale factors of
// the two heads and the probabilities.
__device__ __forceinline__ void softmax_step(const float (&acc)[4], float sl0, float sl1, int nvalid, int g8,
                                             SoftmaxState& st, float (&pr)[4], float& a0, float& a1) {
    float z0 = acc[0] * sl0, z1 = acc[1] * sl1, z2 = acc[2] * sl0, z3 = acc[3] * sl1;
    if (nvalid < 16) {
        if (g8 >= nvalid) z0 = z1 = -INFINITY;
        if (g8 + 8 >= nvalid) z2 = z3 = -INFINITY;
    }
    float t0 = fmaxf(z0, z2), t1 = fmaxf(z1, z3);
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
        t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o));
        t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, o));
    }
    const float m0 = fmaxf(st.m[0], t0), m1 = fmaxf(st.m[1], t1);
    a0 = ptx::exp2_approx(st.m[0] - m0);
    a1 = ptx::exp2_approx(st.m[1] - m1);
    st.m[0] = m0;
    st.m[1] = m1;
    pr[0] = ptx::exp2_approx(z0 - m0);
    pr[1] = ptx::exp2_approx(z1 - m1);
    pr[2] = ptx::exp2_approx(z2 - m0);
    pr[3] = ptx::exp2_approx(z3 - m1);
}

// kst / vst: the K and V halves of the warp's page part; row0: the warp's first row in it;
// pstride: bytes between the two 128-byte panels of a row (bf16 head_dim 128).
template <int D>
__device__ __forceinline__ void tile_bf16(uint32_t kst, uint32_t vst, int row0, uint32_t pstride, int nvalid,
                                          const uint32_t (&qf)[D / 16][2], float (&o)[D / 16][4], SoftmaxState& st,
                                          float sl, int lane) {
    constexpr int KS = D / 16;
    const int rr = lane & 7, mat = lane >> 3, g8 = lane >> 2, c4 = lane & 3;
    // two independent accumulation chains over the k-steps halve the dependent MMA latency
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    const int krow = row0 + rr + ((mat & 1) << 3);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int chunk = 2 * ks + (mat >> 1);
        const uint32_t addr = kst + (chunk >> 3) * pstride + krow * 128 + (((chunk & 7) ^ rr) << 4);
        uint32_t a0, a1, a2, a3;
        ptx::ldsm_x4(addr, a0, a1, a2, a3);
        ptx::mma_bf16((ks & 1) ? acc2 : acc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
    float pr[4], f0, f1;
    softmax_step(acc, sl, sl, nvalid, g8, st, pr, f0, f1);
    const uint32_t p01 = ptx::pack_bf16x2(pr[0], pr[1]), p23 = ptx::pack_bf16x2(pr[2], pr[3]);
    // the sums use the rounded probabilities the MMA multiplies with
    st.l[0] = st.l[0] * f0 + ptx::bf16lo_to_f32(p01) + ptx::bf16lo_to_f32(p23);
    st.l[1] = st.l[1] * f1 + ptx::bf16hi_to_f32(p01) + ptx::bf16hi_to_f32(p23);
    const uint32_t pb0 = ptx::movmatrix_trans(p01), pb1 = ptx::movmatrix_trans(p23);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= f0;
        o[mt][1] *= f1;
        o[mt][2] *= f0;
        o[mt][3] *= f1;
    }
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (nvalid < 16) {  // V rows past the context may hold stale bits: zero them
        mlo = (2 * c4 < nvalid ? 0x0000ffffu : 0u) | (2 * c4 + 1 < nvalid ? 0xffff0000u : 0u);
        mhi = (2 * c4 + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * c4 + 9 < nvalid ? 0xffff0000u : 0u);
    }
    const int vrow = row0 + rr + ((mat >> 1) << 3);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        const int chunk = 2 * mt + (mat & 1);
        const uint32_t addr = vst + (chunk >> 3) * pstride + vrow * 128 + (((chunk & 7) ^ rr) << 4);
        uint32_t v0, v1, v2, v3;
        ptx::ldsm_x4_trans(addr, v0, v1, v2, v3);
        ptx::mma_bf16(o[mt], v0 & mlo, v1 & mlo, v2 & mhi, v3 & mhi, pb0, pb1);
    }
}

template <int D>
__device__ __forceinline__ uint32_t fp8_k_addr(uint32_t kst, int row, int chunk) {
    if (D == 128) return kst + row * 128 + ((chunk ^ (row & 7)) << 4);
    return kst + row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// Row d of the warp's [D][16] V panel: the panel's bytes arrive as 16 swizzled lines of D bytes
// starting at line row0 of the V half.
template <int D>
__device__ __forceinline__ uint32_t fp8_v_addr(uint32_t vst, int row0, int d) {
    if (D == 128) {
        const int line = row0 + (d >> 3);
        return vst + line * 128 + (((d & 7) ^ (line & 7)) << 4);
    }
    const int line = row0 + (d >> 2);
    return vst + line * 64 + (((d & 3) ^ ((line >> 1) & 3)) << 4);
}

// Four 1-byte codes (byte 0 first) -> two f16x2 (codes 0,1 and 2,3), exactly: E4M3 codes by the
// hardware conversion; int8 codes in [-127, 127] by placing code + 128 (the sign bit flipped)
// into the mantissa of 1024.0 (f16 bits 0x6400 | byte) and subtracting 1152 (both steps exact
// in this range): one flip for four codes, one byte permute and one f16x2 subtraction per pair.
template <bool I8>
__device__ __forceinline__ void widen4(uint32_t four, uint32_t& lo, uint32_t& hi) {
    if constexpr (I8) {
        const uint32_t x = four ^ 0x80808080u;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(__byte_perm(x, 0x64u, 0x4140)), "r"(0x64806480u));
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(__byte_perm(x, 0x64u, 0x4342)), "r"(0x64806480u));
    } else {
        lo = ptx::e4m3x2_to_f16x2(four);
        hi = ptx::e4m3x2_to_f16x2(four >> 16);
    }
}

// qinv: the warp's per-head 2^-e (load_q_f16), undoing the power-of-two scaling of the query rows.
template <int D, bool I8>
__device__ __forceinline__ void tile_fp8(uint32_t kst, uint32_t vst, int row0, int nvalid,
                                         const uint32_t (&qf)[D / 16][2], float (&o)[D / 16][4], SoftmaxState& st,
                                         float sl, float sk, float sv, float& sv_prev, const float* qinv, int lane) {
    constexpr int KS = D / 16;
    const int rr = lane & 7, mat = lane >> 3, g8 = lane >> 2, c4 = lane & 3;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    const int krow = row0 + rr + ((mat & 1) << 3);
#pragma unroll
    for (int kk = 0; kk < KS / 2; ++kk) {
        uint32_t r0, r1, r2, r3;
        ptx::ldsm_x4(fp8_k_addr<D>(kst, krow, 2 * kk + (mat >> 1)), r0, r1, r2, r3);
        uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
        widen4<I8>(r0, l0, h0);
        widen4<I8>(r1, l1, h1);
        widen4<I8>(r2, l2, h2);
        widen4<I8>(r3, l3, h3);
        ptx::mma_f16(acc, l0, l1, h0, h1, qf[2 * kk][0], qf[2 * kk][1]);
        ptx::mma_f16(acc2, l2, l3, h2, h3, qf[2 * kk + 1][0], qf[2 * kk + 1][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
    float pr[4], f0, f1;
    const float slk = sl * sk;  // then an exact power-of-two factor per head
    const float2 qi = *reinterpret_cast<const float2*>(qinv + 2 * c4);
    softmax_step(acc, slk * qi.x, slk * qi.y, nvalid, g8, st, pr, f0, f1);
    const uint32_t p01 = ptx::pack_f16x2(pr[0], pr[1]), p23 = ptx::pack_f16x2(pr[2], pr[3]);
    const float2 q01 = ptx::f16x2_to_f32x2(p01), q23 = ptx::f16x2_to_f32x2(p23);
    st.l[0] = st.l[0] * f0 + q01.x + q23.x;
    st.l[1] = st.l[1] * f1 + q01.y + q23.y;
    const uint32_t pb0 = ptx::movmatrix_trans(p01), pb1 = ptx::movmatrix_trans(p23);
    // O is kept in units of the current tile's V scale: rescale by alpha * s_prev / s_cur
    const float ratio = __fdividef(sv_prev, sv);
    sv_prev = sv;
    f0 *= ratio;
    f1 *= ratio;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= f0;
        o[mt][1] *= f1;
        o[mt][2] *= f0;
        o[mt][3] *= f1;
    }
    // V panel row d holds tokens 2c,2c+1,2c+8,2c+9 in this lane's 4 bytes
    uint32_t bm = 0xffffffffu;
    if (nvalid < 16)
        bm = (2 * c4 < nvalid ? 0x000000ffu : 0u) | (2 * c4 + 1 < nvalid ? 0x0000ff00u : 0u) |
             (2 * c4 + 8 < nvalid ? 0x00ff0000u : 0u) | (2 * c4 + 9 < nvalid ? 0xff000000u : 0u);
#pragma unroll
    for (int mm = 0; mm < KS / 2; ++mm) {
        uint32_t r0, r1, r2, r3;
        ptx::ldsm_x4(fp8_v_addr<D>(vst, row0, 32 * mm + lane), r0, r1, r2, r3);
        r0 &= bm;
        r1 &= bm;
        r2 &= bm;
        r3 &= bm;
        uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
        widen4<I8>(r0, l0, h0);
        widen4<I8>(r1, l1, h1);
        widen4<I8>(r2, l2, h2);
        widen4<I8>(r3, l3, h3);
        ptx::mma_f16(o[2 * mm], l0, l1, h0, h1, pb0, pb1);
        ptx::mma_f16(o[2 * mm + 1], l2, l3, h2, h3, pb0, pb1);
    }
}

// 2^k as fp32 for k in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// Query B-fragments of the group's G heads (rows >= G are zero), bf16 KV: the bf16 bits as they
// are.
template <int D>
__device__ __forceinline__ void load_q_bf16(uint32_t (&qf)[D / 16][2], const uint8_t* qs, int G, int lane) {
    const int g8 = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        if (g8 >= G) {
            qf[ks][0] = qf[ks][1] = 0u;
        } else {
            const uint32_t* row = reinterpret_cast<const uint32_t*>(qs + (size_t)g8 * D * 2);
            qf[ks][0] = row[(16 * ks + 2 * c4) >> 1];
            qf[ks][1] = row[(16 * ks + 8 + 2 * c4) >> 1];
        }
    }
}

// One-byte KV: the codes widen exactly to f16 and the MMA runs on f16, so the query rows are
// converted to f16 too.  To keep that conversion exact for any bf16 row, each head's row is first
// multiplied by 2^e, e chosen so that the row's largest magnitude lands in [2^15, 2^16) (bf16's
// 8-bit significand then fits f16 exactly up to 65280 < 65504); qinv[j] receives 2^-e of head j,
// which the score scale of head j takes on (a power of two: the scores equal the unscaled ones,
// roundings included).  Elements more than 2^29 below the row's maximum fall under f16's normal
// range and are rounded to its subnormal grid: an error below 2^-39 of the row maximum per
// element, under the fp32 accumulation's own rounding.  A zero row keeps e = 0.  qinv is this
// warp's slot of kMaxG floats in shared memory (registers are the one-byte kernels' limit).
template <int D>
__device__ __forceinline__ void load_q_f16(uint32_t (&qf)[D / 16][2], const uint8_t* qs, int G, int lane,
                                           float* qinv) {
    constexpr int KS = D / 16;
    const int g8 = lane >> 2, c4 = lane & 3;
    // logical k 2c,2c+1 | 2c+8,2c+9 <-> physical d 4c..4c+3 (matches the one-byte K fragment)
    const uint2* row = reinterpret_cast<const uint2*>(qs + ((size_t)g8 * D + 4 * c4) * 2);
    uint32_t mx = 0;  // largest |q| of the row, as bf16 magnitude bits (they order like the values)
    if (g8 < G) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const uint2 v = row[4 * ks];
            mx = max(mx, max(max(v.x & 0x7fffu, (v.x >> 16) & 0x7fffu), max(v.y & 0x7fffu, (v.y >> 16) & 0x7fffu)));
        }
    }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int e = 0;
    if (mx) {
        const int E = (int)(mx >> 7);  // biased exponent; 0 for a subnormal maximum
        const int lead = E ? E - 127 : (31 - __clz((int)mx)) - 133;  // exponent of its leading bit
        e = 15 - lead;  // in [-112, 148] for finite values
    }
    // 2^e as two factors, each a normal fp32 power of two
    const int ea = e >> 1;
    const float fa = pow2f(ea), fb = pow2f(e - ea);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        if (g8 >= G) {
            qf[ks][0] = qf[ks][1] = 0u;
        } else {
            const uint2 v = row[4 * ks];
            qf[ks][0] = ptx::pack_f16x2(ptx::bf16lo_to_f32(v.x) * fa * fb, ptx::bf16hi_to_f32(v.x) * fa * fb);
            qf[ks][1] = ptx::pack_f16x2(ptx::bf16lo_to_f32(v.y) * fa * fb, ptx::bf16hi_to_f32(v.y) * fa * fb);
        }
    }
    if (c4 == 0) qinv[g8] = pow2f(-e);  // heads >= G: 1 (unused)
    __syncwarp();
}

// Merge the four warps' states of pair (b, h) and write the output (pair complete in this CTA)
// or a partial state plus a ticket (pair cut between CTAs; the last one merges all parts).
//
// Shared-memory combine area: O [4 warps][G][D+4], m and l [4][G], merge weights [4][G], and the
// pair's max and sum [G] each.  Partial states in the workspace: O [slot][G][D] and (m, l)
// [slot][G][2]; slot = pair + CTA index.
template <int D, int QUICK>
__device__ void finish_pair(const Params& p, const float (&o)[D / 16][4], const SoftmaxState& st, float osc, int b,
                            int h, bool complete, int64_t Ng, int64_t C, const int32_t* cumg, uint8_t* smem,
                            volatile int* misc) {
    constexpr int kCT = kConsumerWarps * 32;
    constexpr int kStride = D + 4;  // keeps rows 16-byte aligned and spreads the fragment stores over banks
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, c4 = lane & 3;
    const int G = p.G;
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float* cO = reinterpret_cast<float*>(smem + p.off_cmb);
    float* cM = cO + kConsumerWarps * G * kStride;
    float* cL = cM + kConsumerWarps * G;
    float* cW = cL + kConsumerWarps * G;
    float* cMp = cW + kConsumerWarps * G;  // pair max per head
    float* cLp = cMp + G;                   // pair sum per head
    const int j0 = 2 * c4, j1 = 2 * c4 + 1;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int d = 16 * mt + g8;
        if (j0 < G) {
            cO[(warp * G + j0) * kStride + d] = o[mt][0] * osc;
            cO[(warp * G + j0) * kStride + d + 8] = o[mt][2] * osc;
        }
        if (j1 < G) {
            cO[(warp * G + j1) * kStride + d] = o[mt][1] * osc;
            cO[(warp * G + j1) * kStride + d + 8] = o[mt][3] * osc;
        }
    }
    if (g8 == 0) {
        if (j0 < G) {
            cM[warp * G + j0] = st.m[0];
            cL[warp * G + j0] = l0;
        }
        if (j1 < G) {
            cM[warp * G + j1] = st.m[1];
            cL[warp * G + j1] = l1;
        }
    }
    ptx::named_barrier_sync(kCombineBar, kCT);
    if (tid < G) {  // per head: the pair's max, the four warps' weights and the pair's sum
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cM[w * G + tid]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float f = ptx::exp2_approx(cM[w * G + tid] - M);
            cW[w * G + tid] = f;
            L += f * cL[w * G + tid];
        }
        cMp[tid] = M;
        cLp[tid] = L;
    }
    ptx::named_barrier_sync(kCombineBar, kCT);
    const int pair = b * p.Hkv + h;
    uint16_t* out = p.out + ((int64_t)b * p.Hq + (int64_t)h * G) * D;
    const int64_t slot = (int64_t)pair + blockIdx.x;
    float* part_o = p.partials + slot * G * D;
    for (int e = tid; e < G * (D / 4); e += kCT) {
        const int j = e / (D / 4), d = (e % (D / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float f = cW[w * G + j];
            const float4 v = *reinterpret_cast<const float4*>(cO + (w * G + j) * kStride + d);
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
        }
        if (complete) {
            const float inv = 1.f / cLp[j];
            *reinterpret_cast<uint2*>(out + j * D + d) =
                make_uint2(ptx::pack_bf16x2(acc.x * inv, acc.y * inv), ptx::pack_bf16x2(acc.z * inv, acc.w * inv));
        } else {
            *reinterpret_cast<float4*>(part_o + j * D + d) = acc;
        }
    }
    if (!complete) {
        if (tid < G) *reinterpret_cast<float2*>(p.part_ml + (slot * G + tid) * 2) = make_float2(cMp[tid], cLp[tid]);
        // One thread takes the pair's ticket with an acquire-release atomic: the release publishes
        // the CTA's partial state (every thread's stores precede it through the barrier), the
        // acquire lets the last of the parts read all the others' after the next barrier.
        ptx::named_barrier_sync(kCombineBar, kCT);
        if (tid == 0) {
            const int ng = cumg[b + 1] - cumg[b];
            const int64_t e_first = (int64_t)p.Hkv * cumg[b] + (int64_t)h * ng;
            const int64_t e_last = e_first + ng - 1;
            const int c1 = (int)(((e_first + 1) * C - 1) / Ng);
            const int c2 = (int)(((e_last + 1) * C - 1) / Ng);
            const int ticket = ptx::atomic_add_acq_rel_gpu(p.counters + pair, 1);
            const bool last_part = ticket == c2 - c1;
            misc[kMiscMergeParts] = last_part ? c2 - c1 + 1 : 0;
            misc[kMiscMergeFirst] = c1;
        }
        ptx::named_barrier_sync(kCombineBar, kCT);
        const int nparts = misc[kMiscMergeParts];
        if (nparts && nparts <= QUICK) {
            if constexpr (QUICK > 0) {
                // A pair cut into a few parts (the usual case: a CTA boundary falls inside it, and the
                // CTA reaching the pair last merges as its final work): every thread loads the parts'
                // (m, l) and its slice of their O at once -- one round trip -- and forms the maximum,
                // the sum and the weighted O itself, in part order.
                const int64_t s0 = (int64_t)pair + misc[kMiscMergeFirst];
                for (int e = tid; e < G * (D / 4); e += kCT) {
                    const int j = e / (D / 4), d = (e % (D / 4)) * 4;
                    float2 ml[QUICK];
                    float4 v[QUICK];
#pragma unroll
                    for (int u = 0; u < QUICK; ++u) {
                        if (u < nparts) {
                            ml[u] = __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((s0 + u) * G + j) * 2));
                            v[u] = __ldcg(reinterpret_cast<const float4*>(p.partials + ((s0 + u) * G + j) * D + d));
                        }
                    }
                    float M = -INFINITY;
#pragma unroll
                    for (int u = 0; u < QUICK; ++u)
                        if (u < nparts) M = fmaxf(M, ml[u].x);
                    float L = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < QUICK; ++u) {
                        if (u < nparts) {
                            const float w = ptx::exp2_approx(ml[u].x - M);
                            L += w * ml[u].y;
                            acc.x += w * v[u].x;
                            acc.y += w * v[u].y;
                            acc.z += w * v[u].z;
                            acc.w += w * v[u].w;
                        }
                    }
                    const float inv = 1.f / L;
                    *reinterpret_cast<uint2*>(out + j * D + d) =
                        make_uint2(ptx::pack_bf16x2(acc.x * inv, acc.y * inv), ptx::pack_bf16x2(acc.z * inv, acc.w * inv));
                }
                if (tid == 0) p.counters[pair] = 0;
            }
        } else if (nparts) {
            const int64_t s0 = (int64_t)pair + misc[kMiscMergeFirst];
            // per head: max and sum over the parts, 16 threads per head
            {
                const int j = tid >> 4, sl = tid & 15;
                float M = -INFINITY, L = 0.f;
                if (j < G) {
                    for (int s = sl; s < nparts; s += 16) M = fmaxf(M, __ldcg(p.part_ml + ((s0 + s) * G + j) * 2));
                }
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                if (j < G) {
                    for (int s = sl; s < nparts; s += 16) {
                        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((s0 + s) * G + j) * 2));
                        L += ptx::exp2_approx(ml.x - M) * ml.y;
                    }
                }
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
                if (j < G && sl == 0) {
                    cMp[j] = M;
                    cLp[j] = L;
                }
            }
            ptx::named_barrier_sync(kCombineBar, kCT);
            for (int e = tid; e < G * (D / 4); e += kCT) {
                const int j = e / (D / 4), d = (e % (D / 4)) * 4;
                const float M = cMp[j];
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                int s = 0;
                for (; s + 4 <= nparts; s += 4) {  // four independent loads in flight
                    float f[4];
                    float4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        f[u] = __ldcg(p.part_ml + ((s0 + s + u) * G + j) * 2);
                        v[u] = __ldcg(reinterpret_cast<const float4*>(p.partials + ((s0 + s + u) * G + j) * D + d));
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float w = ptx::exp2_approx(f[u] - M);
                        acc.x += w * v[u].x;
                        acc.y += w * v[u].y;
                        acc.z += w * v[u].z;
                        acc.w += w * v[u].w;
                    }
                }
                for (; s < nparts; ++s) {
                    const float w = ptx::exp2_approx(__ldcg(p.part_ml + ((s0 + s) * G + j) * 2) - M);
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(p.partials + ((s0 + s) * G + j) * D + d));
                    acc.x += w * v.x;
                    acc.y += w * v.y;
                    acc.z += w * v.z;
                    acc.w += w * v.w;
                }
                const float inv = 1.f / cLp[j];
                *reinterpret_cast<uint2*>(out + j * D + d) =
                    make_uint2(ptx::pack_bf16x2(acc.x * inv, acc.y * inv), ptx::pack_bf16x2(acc.z * inv, acc.w * inv));
            }
            if (tid == 0) p.counters[pair] = 0;
        }
    }
    ptx::named_barrier_sync(kCombineBar, kCT);
}

template <bool FP8, int D, bool I8>
__device__ void consumer(const Params& p, const int32_t* cumg, const int32_t* lens_s, int64_t R0, int64_t R1,
                         int64_t Ng, int64_t C, uint8_t* smem, uint32_t sbase, uint32_t bar_full, uint32_t bar_empty,
                         volatile int* misc) {
    constexpr int KS = D / 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t qf[KS][2];
    float o[KS][4];
    SoftmaxState st;
    float sv_prev = 1.f;
    // one-byte KV: this warp's per-head undo of the query scaling (kMaxG floats)
    float* qinv = reinterpret_cast<float*>(smem + p.off_misc + kMiscQinvBytes) + warp * kMaxG;
    int b = find_seq(cumg, p.B, p.Hkv, R0);
    int ng = cumg[b + 1] - cumg[b];
    const int r = (int)(R0 - (int64_t)p.Hkv * cumg[b]);
    int h = r / ng;
    int g = r - h * ng;
    int g_first = g;
    int s = 0;
    uint32_t round = 0;
    bool alive = true;
    const int pidx = (16 * warp) / p.box_rows;  // page part holding this warp's tokens
    const int prow = (16 * warp) % p.box_rows;  // the warp's first row inside that part
    const uint32_t part_bytes = 2u * (uint32_t)p.box_rows * D * (FP8 ? 1 : 2);
    for (int64_t e = R0; e < R1; ++e) {
        const bool first = (e == R0) || (g == 0);
        const bool last = (e == R1 - 1) || (g == ng - 1);
        const uint32_t st_addr = sbase + (uint32_t)s * p.stage_bytes;
        if (alive && !wait_full(bar_full + 8 * s, round & 1, misc, p.wait_ns)) {
            alive = false;
            flag_abort(p, misc);
        }
        if (first) {
            if constexpr (FP8)
                load_q_f16<D>(qf, smem + (st_addr - sbase) + p.off_q, p.G, lane, qinv);
            else
                load_q_bf16<D>(qf, smem + (st_addr - sbase) + p.off_q, p.G, lane);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            st.m[0] = st.m[1] = -INFINITY;
            st.l[0] = st.l[1] = 0.f;
            sv_prev = 1.f;
            g_first = g;
        }
        const int nvalid = min(16, lens_s[b] - g * kGroup - 16 * warp);
        if (alive && nvalid > 0) {
            const uint32_t kst = st_addr + (uint32_t)pidx * part_bytes;  // the warp's page part: K rows, then V rows
            const uint32_t vst = kst + part_bytes / 2;
            if (FP8) {
                const float2 sc = *reinterpret_cast<const float2*>(smem + (st_addr - sbase) + p.off_s + 8 * pidx);
                tile_fp8<D, I8>(kst, vst, prow, nvalid, qf, o, st, p.scale_log2, sc.x, sc.y, sv_prev, qinv, lane);
            } else {
                tile_bf16<D>(kst, vst, prow, (uint32_t)p.box_rows * 128, nvalid, qf, o, st, p.scale_log2, lane);
            }
        }
        __syncwarp();
        // A warp that gave up waiting no longer releases stages: the stage's phase is unknown, so
        // the producer must not reuse it (its own bounded wait then runs out).
        if (lane == 0 && alive) ptx::mbar_arrive(bar_empty + 8 * s);
        if (last) finish_pair<D, FP8 ? 0 : kQuickMergeParts>(p, o, st, FP8 ? sv_prev : 1.f, b, h, g_first == 0 && g == ng - 1, Ng, C, cumg, smem,
                                 misc);
        if (++s == p.stages) {
            s = 0;
            ++round;
        }
        if (++g == ng) {
            g = 0;
            if (++h == p.Hkv) {
                h = 0;
                do {
                    ++b;
                } while (b < p.B && cumg[b + 1] == cumg[b]);
                if (b < p.B) ng = cumg[b + 1] - cumg[b];
            }
        }
    }
}

template <bool FP8, int D, bool I8 = false>
__global__ void __launch_bounds__(kThreads, FP8 ? 3 : 2) decode_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                          const __grid_constant__ CUtensorMap tmap_tail,
                                                                          const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    AppendPre pre{-1, make_uint4(0u, 0u, 0u, 0u)};
    if constexpr (FP8) {
        if (p.n_new > 0 && warp < kConsumerWarps) pre = append_preload<D>(p, warp);
    }
    int32_t* cumg = reinterpret_cast<int32_t*>(smem + p.off_lens);
    int32_t* lens_s = cumg + p.B + 1;
    volatile int* misc = reinterpret_cast<volatile int*>(smem + p.off_misc);
    const uint32_t bar_full = sbase + p.off_bar, bar_empty = bar_full + 8 * p.stages;

    // Context lengths (clamped to the table's capacity) and per-sequence group prefix sums.
    if (warp == 0) {
        const int cap = p.max_blocks * p.bs;
        const int per = (p.B + 31) >> 5;
        const int b0 = min(p.B, lane * per), b1 = min(p.B, b0 + per);
        int sum = 0;
        bool bad = false;
        for (int bb = b0; bb < b1; ++bb) {
            int L = __ldg(p.lens + bb);
            if (L < 0 || L > cap) {
                bad = true;
                L = min(max(L, 0), cap);
            }
            lens_s[bb] = L;
            sum += (L + kGroup - 1) / kGroup;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - sum;
        for (int bb = b0; bb < b1; ++bb) {
            cumg[bb] = run;
            run += (lens_s[bb] + kGroup - 1) / kGroup;
        }
        if (lane == 31) cumg[p.B] = incl;
        if (bad && blockIdx.x == 0) atomicOr(p.err, kErrBounds);
        if (lane == 0) {
            misc[kMiscAbort] = 0;
            misc[kMiscMergeParts] = 0;
        }
    }
    if (tid == 32) {
        for (int s = 0; s < p.stages; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, kConsumerWarps);
        }
        ptx::fence_barrier_init();
    }
    if (tid == 64) {
        ptx::prefetch_tensormap(&tmap);
        ptx::prefetch_tensormap(&tmap_tail);
    }
    __syncthreads();

    // Groups are split over C = min(grid, groups) CTAs, so every participating CTA owns at
    // least one group and a pair cut between CTAs has exactly one part per CTA in between.
    const int64_t Ng = (int64_t)p.Hkv * cumg[p.B];
    const int64_t C = Ng < (int64_t)gridDim.x ? Ng : (int64_t)gridDim.x;
    int64_t R0 = 0, R1 = 0;
    if ((int64_t)blockIdx.x < C) {
        R0 = (int64_t)blockIdx.x * Ng / C;
        R1 = ((int64_t)blockIdx.x + 1) * Ng / C;
    }

    if (warp == kConsumerWarps) {
        bool appended = true;
        if (R0 < R1) {
            appended = producer<FP8, D>(&tmap, &tmap_tail, p, cumg, lens_s, R0, R1, sbase, bar_full, bar_empty, misc);
        } else if (FP8 && p.n_new > 0) {  // no groups here, but every CTA takes part in the count
            appended = wait_appends<D>(p);
            if (!appended && lane == 0) atomicOr(p.err, kErrTimeout);
        }
        if (FP8 && p.n_new > 0 && appended) appends_done(p);
        return;
    }
    if constexpr (FP8) {
        if (p.n_new > 0) append_rows<D, I8>(p, warp, pre);
    }
    // Sequences with an empty context get zeros (no group covers them).
    for (int bb = blockIdx.x; bb < p.B; bb += gridDim.x) {
        if (lens_s[bb] != 0) continue;
        uint4* row = reinterpret_cast<uint4*>(p.out + (int64_t)bb * p.Hq * D);
        for (int i = tid; i < p.Hq * D / 8; i += kConsumerWarps * 32) row[i] = make_uint4(0, 0, 0, 0);
    }
    if (R0 < R1) consumer<FP8, D, I8>(p, cumg, lens_s, R0, R1, Ng, C, smem, sbase, bar_full, bar_empty, misc);
}

// ------------------------------------------------------------------ host side
struct Plan {
    int stages = 0, ctas_per_sm = 0, grid = 0;
    uint32_t stage_bytes = 0, off_q = 0, off_s = 0;
    uint32_t off_bar = 0, off_misc = 0, off_cmb = 0, off_lens = 0, smem_bytes = 0;
    size_t counters_bytes = 0, slots = 0, ws_bytes = 0;
};

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

const void* kernel_for(const pkv_pool* pool) {
    const bool i8 = pool->dtype == PKV_KV_INT8;
    const bool fp8 = pool->dtype != PKV_KV_BF16;  // one-byte codes (fp8 or int8)
    if (pool->head_dim == 128)
        return i8 ? (const void*)decode_kernel<true, 128, true>
                  : fp8 ? (const void*)decode_kernel<true, 128> : (const void*)decode_kernel<false, 128>;
    return i8 ? (const void*)decode_kernel<true, 64, true>
              : fp8 ? (const void*)decode_kernel<true, 64> : (const void*)decode_kernel<false, 64>;
}

bool compute_plan(const pkv_pool* pool, int B, int G, int pref_ctas, int max_stages_env, Plan& pl);

// The launch plan depends only on these values (not on the pool's address or contents), so the
// plans of recent shapes are kept per host thread: a decode loop pays the shared-memory layout
// and the occupancy query once per batch shape instead of once per step.
struct PlanKey {
    int B, G, Hkv, dtype, D, bs, sm_count, smem_block, smem_sm, device, pref, max_stages;
    bool operator==(const PlanKey& o) const {
        return B == o.B && G == o.G && Hkv == o.Hkv && dtype == o.dtype && D == o.D && bs == o.bs &&
               sm_count == o.sm_count && smem_block == o.smem_block && smem_sm == o.smem_sm && device == o.device &&
               pref == o.pref && max_stages == o.max_stages;
    }
};

bool make_plan(const pkv_pool* pool, int B, int G, Plan& pl) {
    const bool q8 = pool->dtype != PKV_KV_BF16;
    const Settings& cfg = settings();
    const int pref = cfg.attn_ctas_per_sm > 0 ? cfg.attn_ctas_per_sm : (q8 ? 3 : 2);
    const int max_stages = cfg.attn_max_stages > 0 ? cfg.attn_max_stages : kMaxStages;
    const PlanKey key{B, G, pool->n_kv_heads, (int)pool->dtype, pool->head_dim, pool->block_size, pool->sm_count,
                      pool->max_smem_per_block, pool->max_smem_per_sm, pool->device, pref, max_stages};
    constexpr int kSlots = 8;
    thread_local PlanKey keys[kSlots];
    thread_local Plan plans[kSlots];
    thread_local int used = 0, next = 0;
    for (int i = 0; i < used; ++i)
        if (keys[i] == key) {
            pl = plans[i];
            return true;
        }
    if (!compute_plan(pool, B, G, pref, max_stages, pl)) return false;
    keys[next] = key;
    plans[next] = pl;
    next = (next + 1) % kSlots;
    if (used < kSlots) ++used;
    return true;
}

bool compute_plan(const pkv_pool* pool, int B, int G, int pref_ctas, int max_stages_env, Plan& pl) {
    const bool fp8 = pool->dtype != PKV_KV_BF16;  // one-byte codes (fp8 or int8)
    const uint32_t D = (uint32_t)pool->head_dim, esz = fp8 ? 1 : 2;
    const uint32_t region = kGroup * D * esz;
    pl.off_q = 2 * region;  // kGroup rows of K and of V, as ppg page parts
    pl.off_s = pl.off_q + align_up((uint32_t)G * D * 2, 128);
    pl.stage_bytes = align_up(pl.off_s + (fp8 ? 8u * 4 : 0u), 1024);
    const uint32_t cmb = align_up((kConsumerWarps * G * (D + 4) + 3 * kConsumerWarps * G + 2 * G) * 4, 16);
    const uint32_t lens = align_up((2u * B + 1) * 4, 16);
    const uint32_t misc = kMiscQinvBytes + kConsumerWarps * kMaxG * 4;  // misc words, query factors
    const uint32_t fixed = 1024 + misc + cmb + lens;
    // fp8 tiles carry half the bytes of bf16 ones, so fp8 runs three CTAs per SM (its kernel is
    // compiled for that register budget) to keep enough tiles in flight
    const int pref = pref_ctas;
    const int max_stages = std::max(2, std::min(kMaxStages, max_stages_env));
    pl.stages = 0;
    for (int ctas = std::max(1, pref); ctas >= 1; --ctas) {
        const int budget = std::min(pool->max_smem_per_block, pool->max_smem_per_sm / ctas - 1024);
        if (budget <= (int)fixed) continue;
        int S = (int)((budget - fixed) / (pl.stage_bytes + 16));
        S = std::min(S, max_stages);
        if (S >= 2) {
            pl.stages = S;
            pl.ctas_per_sm = ctas;
            break;
        }
    }
    if (!pl.stages) return false;
    pl.off_bar = (uint32_t)pl.stages * pl.stage_bytes;
    pl.off_misc = pl.off_bar + 16u * pl.stages;
    pl.off_cmb = align_up(pl.off_misc + misc, 16);
    pl.off_lens = pl.off_cmb + cmb;
    pl.smem_bytes = pl.off_lens + lens + 1024;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel_for(pool), kThreads, pl.smem_bytes) != cudaSuccess ||
        occ < 1)
        return false;
    pl.ctas_per_sm = std::min(pl.ctas_per_sm, occ);
    pl.grid = pl.ctas_per_sm * pool->sm_count;
    const size_t pairs = (size_t)B * pool->n_kv_heads;
    // merge tickets [pairs], then (from a 128-byte boundary) the words of the step's own append
    pl.counters_bytes = ((pairs + kAppStride - 1) / kAppStride * kAppStride + kAppWords) * sizeof(int);
    pl.counters_bytes = (pl.counters_bytes + 255) / 256 * 256;
    pl.slots = pairs + (size_t)pl.grid;
    pl.ws_bytes = pl.counters_bytes + pl.slots * G * (D + 2) * sizeof(float);
    return true;
}

// Argument checks, launch plan and kernel parameters for one decode-attention call.
pkv_status prepare(const pkv_pool* pool, const void* q, const int32_t* block_tables, int max_blocks,
                   const int32_t* context_lens, int B, int n_q_heads, float scale, void* out, void* workspace,
                   size_t workspace_bytes, Plan& pl, Params& p) {
    if (!pool || B < 0 || B > kMaxBatch || n_q_heads < 1 || n_q_heads % pool->n_kv_heads) return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    const int G = n_q_heads / pool->n_kv_heads;
    if (G > kMaxG || max_blocks < 1 || (int64_t)max_blocks * pool->block_size >= (1ll << 31))
        return PKV_ERR_INVALID_ARG;
    if (!q || !block_tables || !context_lens || !out || !workspace) return PKV_ERR_INVALID_ARG;
    if (((uintptr_t)q | (uintptr_t)out) & 15u || (uintptr_t)workspace & 255u ||
        ((uintptr_t)block_tables | (uintptr_t)context_lens) & 3u)
        return PKV_ERR_INVALID_ARG;
    if (!make_plan(pool, B, G, pl)) return PKV_ERR_CUDA;
    if (workspace_bytes < pl.ws_bytes) return PKV_ERR_INVALID_ARG;
    p.q = static_cast<const uint16_t*>(q);
    p.tables = block_tables;
    p.lens = context_lens;
    p.out = static_cast<uint16_t*>(out);
    p.pool = static_cast<const uint8_t*>(pool->kv);
    p.scales = pool->scales;
    p.counters = static_cast<int*>(workspace);
    p.app = p.counters + ((size_t)B * pool->n_kv_heads + kAppStride - 1) / kAppStride * kAppStride;
    p.k_new = p.v_new = nullptr;
    p.slots = nullptr;
    p.n_new = 0;
    p.app_extra = 0;
    p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.counters_bytes);
    p.part_ml = p.partials + pl.slots * G * pool->head_dim;
    p.err = pool->err;
    p.B = B;
    p.Hq = n_q_heads;
    p.Hkv = pool->n_kv_heads;
    p.G = G;
    p.max_blocks = max_blocks;
    p.bs = pool->block_size;
    p.num_blocks = pool->num_blocks;
    p.box_rows = std::min(pool->block_size, kGroup);
    p.ppg = kGroup / p.box_rows;
    p.stages = pl.stages;
    p.stage_bytes = pl.stage_bytes;
    p.off_q = pl.off_q;
    p.off_s = pl.off_s;
    p.off_bar = pl.off_bar;
    p.off_misc = pl.off_misc;
    p.off_cmb = pl.off_cmb;
    p.off_lens = pl.off_lens;
    p.scale_log2 = scale * 1.4426950408889634f;
    // Test hooks for the bounded waits (failure detection is tested without a GPU fault): a
    // shorter wait limit, and stages that expect 16 bytes no copy delivers, so the waits run out
    // and the call reports PKV_ERR_TIMEOUT (both off unless set, see Settings).
    const Settings& hooks = settings();
    p.wait_ns = hooks.wait_limit_ms > 0 ? (uint64_t)hooks.wait_limit_ms * 1000000ull : kWaitLimitNs;
    p.stall_tx = hooks.stall_copies ? 16u : 0u;
    return PKV_OK;
}

// Launch on `st`.  With `pdl` the kernel may start while the preceding kernel on the stream
// (an append of this step) is still running: it prepares everything that does not read the
// pool and waits (griddepcontrol.wait) before its first page copy.  A kernel that appends the
// step's tokens itself (p.n_new > 0) is launched cooperatively: its CTAs wait on rows other CTAs
// write, so all of them must be resident at once (the grid is the SMs' resident capacity).
pkv_status launch(const pkv_pool* pool, const Plan& pl, const Params& p, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (p.n_new > 0) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (pdl || p.n_new > 0) ? 1 : 0;
    const bool i8 = pool->dtype == PKV_KV_INT8;
    const bool fp8 = pool->dtype != PKV_KV_BF16;  // one-byte codes (fp8 or int8)
    cudaError_t e;
    if (pool->head_dim == 128)
        e = i8    ? cudaLaunchKernelEx(&cfg, decode_kernel<true, 128, true>, pool->tmap_rows, pool->tmap_tail, p)
            : fp8 ? cudaLaunchKernelEx(&cfg, decode_kernel<true, 128>, pool->tmap_rows, pool->tmap_tail, p)
                  : cudaLaunchKernelEx(&cfg, decode_kernel<false, 128>, pool->tmap_rows, pool->tmap_tail, p);
    else
        e = i8    ? cudaLaunchKernelEx(&cfg, decode_kernel<true, 64, true>, pool->tmap_rows, pool->tmap_tail, p)
            : fp8 ? cudaLaunchKernelEx(&cfg, decode_kernel<true, 64>, pool->tmap_rows, pool->tmap_tail, p)
                  : cudaLaunchKernelEx(&cfg, decode_kernel<false, 64>, pool->tmap_rows, pool->tmap_tail, p);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace attn

void attention_configure(pkv_pool* pool) {
    cudaFuncSetAttribute(attn::kernel_for(pool), cudaFuncAttributeMaxDynamicSharedMemorySize,
                         pool->max_smem_per_block);
}

}  // namespace pkv

extern "C" {

pkv_status pkv_decode_workspace_bytes(const pkv_pool* pool, int B, int n_q_heads, int max_blocks, size_t* out) {
    (void)max_blocks;
    if (!pool || !out || B < 0 || B > pkv::attn::kMaxBatch || n_q_heads < 1 || n_q_heads % pool->n_kv_heads)
        return PKV_ERR_INVALID_ARG;
    const int G = n_q_heads / pool->n_kv_heads;
    if (G > pkv::attn::kMaxG) return PKV_ERR_INVALID_ARG;
    pkv::attn::Plan pl;
    if (!pkv::attn::make_plan(pool, B, G, pl)) return PKV_ERR_CUDA;
    *out = pl.ws_bytes;
    return PKV_OK;
}

pkv_status pkv_decode_attention(const pkv_pool* pool, const void* q, const int32_t* block_tables, int max_blocks,
                                const int32_t* context_lens, int B, int n_q_heads, float scale, void* out,
                                void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
    pkv::attn::Plan pl;
    pkv::attn::Params p;
    const pkv_status st = pkv::attn::prepare(pool, q, block_tables, max_blocks, context_lens, B, n_q_heads, scale, out,
                                             workspace, workspace_bytes, pl, p);
    if (st != PKV_OK || B == 0) return st;
    return pkv::attn::launch(pool, pl, p, reinterpret_cast<cudaStream_t>(stream), false);
}

pkv_status pkv_decode_step(pkv_pool* pool, const void* k_new, const void* v_new, const int64_t* slot_mapping, int64_t N,
                           const void* q, const int32_t* block_tables, int max_blocks, const int32_t* context_lens, int B,
                           int n_q_heads, float scale, void* out, void* workspace, size_t workspace_bytes,
                           pkv_stream_t stream) {
    pkv::attn::Plan pl;
    pkv::attn::Params p;
    pkv_status st = pkv::append_check(pool, k_new, v_new, slot_mapping, N);
    if (st != PKV_OK) return st;
    st = pkv::attn::prepare(pool, q, block_tables, max_blocks, context_lens, B, n_q_heads, scale, out, workspace,
                            workspace_bytes, pl, p);
    if (st != PKV_OK) return st;
    if (pool->dtype != PKV_KV_BF16 && B > 0 && N > 0 && N <= pkv::attn::kFusedAppendMax) {
        // one-byte pool: the attention kernel quantises the new tokens itself
        p.k_new = static_cast<const uint16_t*>(k_new);
        p.v_new = static_cast<const uint16_t*>(v_new);
        p.slots = slot_mapping;
        p.n_new = (int)N;
        p.app_extra = pkv::settings().stall_appends ? 1 : 0;
        return pkv::attn::launch(pool, pl, p, reinterpret_cast<cudaStream_t>(stream), false);
    }
    st = pkv_append(pool, k_new, v_new, slot_mapping, N, stream);
    if (st != PKV_OK || B == 0) return st;
    return pkv::attn::launch(pool, pl, p, reinterpret_cast<cudaStream_t>(stream), N > 0);
}

pkv_status pkv_decode_step_rope(pkv_pool* pool, void* k_new, const void* v_new, const int64_t* slot_mapping,
                                const int64_t* positions, int64_t N, double rope_base, void* q,
                                const int32_t* block_tables, int max_blocks, const int32_t* context_lens, int B,
                                int n_q_heads, float scale, void* out, void* workspace, size_t workspace_bytes,
                                pkv_stream_t stream) {
    pkv::attn::Plan pl;
    pkv::attn::Params p;
    pkv_status st = pkv::append_check(pool, k_new, v_new, slot_mapping, N);
    if (st != PKV_OK) return st;
    if (N != B) return PKV_ERR_INVALID_ARG;  // one new token (and one query row) per sequence
    st = pkv::attn::prepare(pool, q, block_tables, max_blocks, context_lens, B, n_q_heads, scale, out, workspace,
                            workspace_bytes, pl, p);
    if (st != PKV_OK) return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // rotates k_new and q in place and appends; the attention reads q only after waiting on it
    st = pkv::append_rope_launch(pool, k_new, v_new, slot_mapping, positions, N, rope_base, q, n_q_heads, cs);
    if (st != PKV_OK || B == 0) return st;
    return pkv::attn::launch(pool, pl, p, cs, true);
}

}  // extern "C"

// ------------------------------------------------------------------ allocation-free variant
// For callers that cannot allocate a workspace (see pkv_decode_attention_static in pkv.h): the
// scratch is this fixed array in the library's device image.  Host code must not use the
// symbol itself as a pointer (on the host it is only a stand-in); the device address comes from
// cudaGetSymbolAddress, looked up once per device.

namespace pkv {
namespace attn {

static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_ws_mutex;
void* g_static_ws_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on `device`, which must be the current device.
pkv_status static_workspace(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_static_ws_mutex);
    if (!g_static_ws_ptr[device]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return PKV_ERR_CUDA;
        g_static_ws_ptr[device] = ptr;
    }
    *out = g_static_ws_ptr[device];
    return PKV_OK;
}

}  // namespace attn
}  // namespace pkv

extern "C" pkv_status pkv_decode_attention_static(const pkv_pool* pool, const void* q, const int32_t* block_tables,
                                                  int max_blocks, const int32_t* context_lens, int B, int n_q_heads,
                                                  float scale, void* out, pkv_stream_t stream) {
    if (!pool) return PKV_ERR_INVALID_ARG;
    size_t need = 0;
    const pkv_status st = pkv_decode_workspace_bytes(pool, B, n_q_heads, max_blocks, &need);
    if (st != PKV_OK) return st;
    if (need > PKV_STATIC_WORKSPACE_BYTES) return PKV_ERR_INVALID_ARG;  // beyond the fixed scratch
    if (B == 0) return PKV_OK;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return PKV_ERR_CUDA;
    if (cur != pool->device) return PKV_ERR_INVALID_ARG;
    void* ws = nullptr;
    const pkv_status ws_st = pkv::attn::static_workspace(cur, &ws);
    if (ws_st != PKV_OK) return ws_st;
    // the merge tickets at the front of the workspace must start at zero
    if (cudaMemsetAsync(ws, 0, (size_t)B * pool->n_kv_heads * sizeof(int), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_decode_attention(pool, q, block_tables, max_blocks, context_lens, B, n_q_heads, scale, out, ws,
                                PKV_STATIC_WORKSPACE_BYTES, stream);
}
