// decode_kernels.cuh - split-KV MLA decode over a paged 576-wide latent cache.
//
// Method ("DeepSeek-V2" explainer, Steps 6-8): every head scores the absorbed
// query against the shared latent rows, s_j = scale * q_abs . [c_j | k^R_j]
// (content and RoPE channels add inside the softmax, Step 7), and the output
// stays in latent space, o = sum_j softmax(s)_j c_j (W^UV is applied later).
//
// B300 design: one cluster of two CTAs (two SMs) per work item.
//   CTA rank 0, the "score" CTA: streams the 64-token pages with one 3-D TMA box per page
//     into three page stages (the partner re-reads each page from L2 shortly after); the
//     item's absorbed query (128 x 576) first passes through two stage
//     positions and is copied into tensor memory, where it is the MMA A operand.  It
//     computes S = Q K^T (M = 128 heads, N = 64 tokens, K = 576) with tcgen05: one thread
//     cannot issue N = 64 MMAs fast enough to keep the tensor pipe busy, so two issuers
//     take alternate pages, each into its own S buffer in TMEM; the next page's MMAs run
//     while the softmax warps read this one's.  Eight softmax warps
//     run the online softmax with lazy rescaling and write P (bf16, 128 x 64) plus
//     per-head factors straight from registers into a ring of messages in global memory
//     (it stays in L2).
//   CTA rank 1, the "accumulate" CTA: holds O = 128 heads x 512 latent fp32, i.e.
//     all 512 TMEM columns, streams the same pages' 512 latent columns (L2 hits:
//     the score CTA has just pulled them from HBM), bulk-copies each P message
//     into shared memory, and runs O += P V (M = 128, N = 256 x 2, K = 64); its
//     eight epilogue warps rescale O when asked and write the normalised output.
// The split keeps both 256 KB accumulators on chip without recomputing S: O alone
// fills a whole SM's tensor memory, and the query alone would fill most of its
// shared memory.  P travels through L2 rather than distributed shared memory,
// whose bandwidth between the two SMs of a pair is far below what one 16 KB
// message per page needs; only the small ready/free signals are remote arrives.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mla {

constexpr int kHeads = 128;
constexpr int kDc = 512;
constexpr int kDr = 64;
constexpr int kD = kDc + kDr;        // 576
constexpr int kPage = 64;            // tokens per page == tokens per tile
constexpr int kBoxBytes = kPage * 128;  // one 64-row x 64-column bf16 block (128-byte rows)
constexpr int kBoxesS = kD / 64;     // 9 blocks per page for scoring (c and k^R)
constexpr int kBoxesV = kDc / 64;    // 8 blocks per page for the value side (c only)
constexpr uint32_t kStageS = kBoxesS * kBoxBytes;  // 73728: one whole page (score CTA stage)
constexpr int kStagesS = 3;          // score CTA page stages
constexpr uint32_t kQRopeOff = 4 * kHeads * 128;  // in a query stage: 4 content blocks, then 64 heads' RoPE block
constexpr uint32_t kStageV = kBoxesV * kBoxBytes;  // 65536: a page's 512 latent columns (accumulate CTA stage)
constexpr int kStagesV = 2;          // accumulate CTA page stages
constexpr int kPBufs = 4;            // accumulate CTA: P messages held in shared memory
constexpr int kRing = 16;            // P messages in flight through global memory, per CTA pair
constexpr int kMaxBatch = 4;         // most messages published behind one cluster-scope fence
constexpr int kPBytes = kHeads * kPage * 2;  // 16 KB of bf16 probabilities
constexpr int kMetaBytes = 1024;     // alpha[128] f32, inv_l[128] f32
constexpr uint32_t kMsgBytes = kPBytes + kMetaBytes;  // one message: P, then its factors
// Lazy rescale threshold, log2 units: the running reference m moves only when a page maximum
// exceeds it by more than this.  Probabilities are then at most 2^40 relative to m: bf16 P and
// fp32 row sums and O keep their relative precision at any scale, and with at most 2^17 tokens
// and |values| far below 2^60 nothing overflows fp32 (2^127).  A small threshold (8) made
// peaked rows rescale O on about a quarter of the pages of a 128K context.
constexpr float kTau = 40.0f;
constexpr int kMaxClusters = 80;     // CTA pairs the workspace is sized for (B300: 74)

// TMEM columns
constexpr uint32_t kTmemS = 0;       // score CTA: S tile of buffer b at 64 b
constexpr uint32_t kTmemQR = 128;    // score CTA: Q RoPE part (block 8, bf16 pairs) at 128 .. 159
constexpr uint32_t kTmemQ = 256;     // score CTA: Q content part (blocks 0-7, bf16 pairs) at 256 .. 511
constexpr uint32_t kTmemCols = 512;

// Shared memory (offsets from a 1024-aligned base).  Score CTA: three page stages at 0 (an
// item's query passes through the first two of its positions).  Accumulate CTA: two page
// stages at 0, the P buffers (each a whole message: P, then its factors), the event buffer.
// Barriers sit at the same offset in both CTAs (the partner arrives on them).
constexpr uint32_t kOffPBuf = kStagesV * kStageV;                   // accumulate: kPBufs x 17 KB
constexpr uint32_t kOffEvt = kOffPBuf + kPBufs * kMsgBytes;         // accumulate: alpha / inv_l, type, P buffer
constexpr uint32_t kAccumEnd = kOffEvt + 1040;
constexpr uint32_t kScoreEnd = kStagesS * kStageS;
constexpr uint32_t kOffBar = kScoreEnd > kAccumEnd ? kScoreEnd : kAccumEnd;
constexpr int kStagesMax = kStagesS > kStagesV ? kStagesS : kStagesV;
constexpr int kBarFull = 0;                          // page stages
constexpr int kBarEmpty = kBarFull + kStagesMax;
constexpr int kBarSFull = kBarEmpty + kStagesMax;    // score: S tile [buffer] complete
constexpr int kBarSEmpty = kBarSFull + 2;            // score: S tile [buffer] read by the softmax warps
constexpr int kBarQReady = kBarSEmpty + 2;           // score: the item's Q is in TMEM
constexpr int kBarQAck = kBarQReady + 1;             // score: both issuers have seen the item's QReady
constexpr int kBarDrain = kBarQAck + 1;              // MMA warps: all of a warp's MMAs done [warp], at exit
constexpr int kBarPFree = kBarDrain + 2;             // score: ring slot consumed (partner arrives)
constexpr int kBarPReady = kBarPFree + kRing;        // accumulate: a ring slot written (partner arrives)
constexpr int kBarPStaged = kBarPReady + kRing;      // score: all rows of a ring slot written
constexpr int kBarPFull = kBarPStaged + kRing;       // accumulate: P buffer landed
constexpr int kBarPBufFree = kBarPFull + kPBufs;     // accumulate: P buffer used by the MMAs and the releaser
constexpr int kBarMmaEvt = kBarPBufFree + kPBufs;    // accumulate: event for the epilogue warps
constexpr int kBarCorrEvt = kBarMmaEvt + 1;          // accumulate: event served
constexpr int kBarXSum = kBarCorrEvt + 1;            // score: row-sum swap, [quadrant]
constexpr int kNumBars = kBarXSum + 4;
constexpr uint32_t kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kOffXSum = (kOffAbort + 4 + 15u) & ~15u;  // score: row-sum exchange [2 sums][2][128] f32
constexpr uint32_t kDecodeSmem = kOffXSum + 2 * 2 * kHeads * 4 + 1024;  // + slack to align the base
// warps: 0-7 softmax (score) / epilogue (accumulate), 8 page producer, 9-10 the two score MMA
// issuers (score) / 9-11 PV MMA, P loader, releaser (accumulate), 12 shipper (score)
constexpr int kDecodeThreads = 13 * 32;
constexpr int kWarpProducer = 8, kWarpMma = 9, kWarpShipper = 12;
static_assert(kDecodeSmem <= 227u * 1024u, "decode kernel shared memory exceeds the per-CTA limit");
static_assert(kTmemQ + 32u * (kBoxesS - 1) <= kTmemCols && kTmemS + 64u * 2 <= kTmemQR && kTmemQR + 32u <= kTmemQ,
              "score CTA tensor memory overflow");
static_assert(kMsgBytes % 1024 == 0, "P buffers must stay 1024-byte aligned (128-byte swizzle atoms)");
static_assert(2 * kStageS == 8 * kHeads * 128 + kHeads * 128, "an item's query fills the two score stages");
// the epilogue stages its output through the P buffer of the item's last page: 2 KB per warp
static_assert(8 * 2048 <= kPBytes, "epilogue staging does not fit a P buffer");

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, 0, 0);    // A = Q (TMEM), B = K tile, K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);  // A = P K-major, B = V MN-major

constexpr uint32_t kEvtRescale = 1u, kEvtEpilogue = 2u;

// One unit of work: tiles [tb, te) of query (b, t) where bt = b * Tq + t, whose visible
// prefix is n_vis tokens.  slot < 0: the item covers the whole query and writes the final
// output; slot >= 0: it writes a partial (o / l in fp32, lse) into workspace slot `slot`.
// 32 bytes, read as two 16-byte loads.
struct __align__(16) Item {
    int bt, tb, te, slot, b, n_vis, pad0, pad1;
};
struct PlanHeader {
    int n_items;
    int n_bt;
    int max_items;
    int max_slots;
    int n_split;  // queries split into more than one item (0: the combine kernel has nothing to do)
    int pad[59];
};
// per query (b, t): number of splits, first partial slot, tiles, first item
struct BtInfo {
    int splits, slot_base, tiles, item_off;
};

struct DecodeParams {
    const __nv_bfloat16 *q_abs;   // [B, Tq, 128, 576]
    const int32_t *block_table;   // [B, max_pages]
    const int32_t *seq_lens;      // [B]
    __nv_bfloat16 *o_lat;         // [B, Tq, 128, 512]
    float *lse;                   // [B, Tq, 128]
    const PlanHeader *hdr;
    const Item *items;            // max_items entries
    float *part_o;                // [slots, 128, 512]
    float *part_lse;              // [slots, 128]
    uint8_t *ring;                // [clusters, kRing, kMsgBytes] P messages
    int B, Tq, causal, num_pages, max_pages, max_items;
    float sl2;                    // scale * log2(e)
};

struct ItemInfo {
    int b, bt, tb, te, slot, n_vis;
};

__device__ __forceinline__ int visible_tokens(int L, int Tq, int t, int causal) {
    if (!causal) return L;
    int n = L - (Tq - 1 - t);
    return n < 0 ? 0 : n;
}

__device__ __forceinline__ ItemInfo load_item(const DecodeParams &p, int i) {
    const int4 *src = reinterpret_cast<const int4 *>(p.items + i);
    const int4 a = src[0], c = src[1];
    ItemInfo x;
    x.bt = a.x;
    x.tb = a.y;
    x.te = a.z;
    x.slot = a.w;
    x.b = c.x;
    x.n_vis = c.y;
    return x;
}

// Static "snake" schedule over the plan's items (sorted longest first):
// round r gives item r*C + k to cluster k on even rounds and r*C + C-1-k on odd ones.
__device__ __forceinline__ int schedule(int r, int cid, int ncl) {
    return r * ncl + ((r & 1) ? (ncl - 1 - cid) : cid);
}

// A cluster's walk over its items.  The first item (round 0 is item `cid`) is read together
// with the plan header, before the item count is known, so the two reads overlap.
struct Sched {
    int cid, ncl, n_items;
    ItemInfo first;
    __device__ __forceinline__ bool get(const DecodeParams &p, int r, ItemInfo &it) const {
        const int i = schedule(r, cid, ncl);
        if (i >= n_items) return false;
        it = r == 0 ? first : load_item(p, i);
        return true;
    }
};

// ---------------------------------------------------------------------------
// Plan: split counts, items (longest first), partial slots.  One CTA.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;
constexpr int kMinChunkTiles = 4;

__device__ __forceinline__ int block_excl_scan(int v, int *tmp /*[32]*/, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        tmp[lane] = w;  // inclusive per-warp prefix
    }
    __syncthreads();
    int warp_off = warp > 0 ? tmp[warp - 1] : 0;
    *total = tmp[(blockDim.x >> 5) - 1];
    __syncthreads();
    return warp_off + x - v;
}

constexpr int kPlanSmemBt = 2048;  // queries planned in shared memory; larger batches use workspace scratch

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, int B, int Tq, int causal, int max_pages,
            int n_clusters, int num_splits, PlanHeader *hdr, Item *items, BtInfo *info,
            int *scratch /* 4 * B * Tq ints, used when B * Tq > kPlanSmemBt */, int max_items, int max_slots) {
    // launched as a programmatic dependent of its predecessor (often the previous call's
    // combine kernel, which lets it get resident early): nothing is read or written before that
    // predecessor has completed -- it may have written seq_lens, or still read this workspace
    grid_dependency_wait();
    grid_launch_dependents();  // the decode kernel may start its prologue while the plan is made
    __shared__ int s_tmp[32];
    __shared__ int s_key[kPlanThreads];
    __shared__ int s_ord[kPlanThreads];
    __shared__ int s_arr[4 * kPlanSmemBt];
    const int tid = threadIdx.x;
    const int n_bt = B * Tq;
    const int nthr = (int)blockDim.x;  // up to kPlanThreads; the host launches as few as the batch needs
    const int per = (n_bt + nthr - 1) / nthr;
    int *const base = n_bt <= kPlanSmemBt ? s_arr : scratch;
    const int stride = n_bt <= kPlanSmemBt ? kPlanSmemBt : n_bt;
    int *const tiles = base, *const splits = base + stride, *const slot_base = base + 2 * stride,
              *const item_off = base + 3 * stride;

    // 1. tiles per query, total work
    int w_local = 0;
    for (int bt = tid * per; bt < min(n_bt, (tid + 1) * per); ++bt) {
        int b = bt / Tq, t = bt - b * Tq;
        int L = seq_lens[b];
        if (L < 0 || L > max_pages * kPage) {
            if (t == 0) raise_status(0x2u);
            L = L < 0 ? 0 : max_pages * kPage;
        }
        int n = visible_tokens(L, Tq, t, causal);
        int T = (n + kPage - 1) / kPage;
        tiles[bt] = T;
        w_local += T;
    }
    int W_total;
    block_excl_scan(w_local, s_tmp, &W_total);
    const long long W = W_total;

    // 2. split counts
    for (int bt = tid * per; bt < min(n_bt, (tid + 1) * per); ++bt) {
        int T = tiles[bt];
        int s = 1;
        int cap = T / kMinChunkTiles > 1 ? T / kMinChunkTiles : 1;
        if (num_splits > 0) {
            s = num_splits < (T > 0 ? T : 1) ? num_splits : (T > 0 ? T : 1);
        } else if (W > 0 && T > 0) {
            if (n_bt <= n_clusters) {
                s = (int)(((long long)n_clusters * T) / W);
            } else {
                long long c = (W + n_clusters - 1) / n_clusters;
                s = (int)((T + c - 1) / c);
            }
            s = s < 1 ? 1 : (s > cap ? cap : s);
        }
        splits[bt] = s;
    }
    __syncthreads();

    // 3. order: longest chunk first (rank sort when it fits one element per thread)
    const bool sorted = n_bt <= nthr;
    if (sorted) {
        int key = -1;
        if (tid < n_bt) {
            int T = tiles[tid], s = splits[tid];
            key = (T + s - 1) / s;
        }
        s_key[tid] = key;
        __syncthreads();
        if (tid < n_bt) {
            int rank = 0;
            for (int j = 0; j < n_bt; ++j) {
                int kj = s_key[j];
                rank += (kj > key) || (kj == key && j < tid);
            }
            s_ord[rank] = tid;
        }
        __syncthreads();
    }

    // 4. item offsets in that order, partial slots in natural order
    int items_local = 0, slots_local = 0;
    for (int k = tid * per; k < min(n_bt, (tid + 1) * per); ++k) {
        int bt = sorted ? s_ord[k] : k;
        items_local += splits[bt];
        slots_local += splits[k] > 1 ? splits[k] : 0;
    }
    int n_items, n_slots, n_split;
    int ioff = block_excl_scan(items_local, s_tmp, &n_items);
    int soff = block_excl_scan(slots_local, s_tmp, &n_slots);
    int split_local = 0;
    for (int k = tid * per; k < min(n_bt, (tid + 1) * per); ++k) split_local += splits[k] > 1 ? 1 : 0;
    block_excl_scan(split_local, s_tmp, &n_split);
    const bool overflow = n_items > max_items || n_slots > max_slots;
    for (int k = tid * per; k < min(n_bt, (tid + 1) * per); ++k) {
        int bt = sorted ? s_ord[k] : k;
        item_off[bt] = ioff;
        ioff += splits[bt];
        int s2 = splits[k];
        slot_base[k] = s2 > 1 ? soff : -1;
        soff += s2 > 1 ? s2 : 0;
    }
    __syncthreads();

    // 5. items and the per-query info the combine kernel reads (on overflow nothing is
    //    scheduled and nothing is combined)
    for (int bt = tid * per; bt < min(n_bt, (tid + 1) * per); ++bt) {
        BtInfo in;
        in.splits = overflow ? 0 : splits[bt];
        in.slot_base = slot_base[bt];
        in.tiles = tiles[bt];
        in.item_off = item_off[bt];
        info[bt] = in;
        const int b = bt / Tq;
        int L = seq_lens[b];
        L = L < 0 ? 0 : (L > max_pages * kPage ? max_pages * kPage : L);
        const int n_vis = visible_tokens(L, Tq, bt - b * Tq, causal);
        for (int j = 0; j < in.splits; ++j) {
            Item it;
            it.bt = bt;
            it.b = b;
            it.n_vis = n_vis;
            it.pad0 = it.pad1 = 0;
            it.tb = (int)(((long long)in.tiles * j) / in.splits);
            it.te = (int)(((long long)in.tiles * (j + 1)) / in.splits);
            it.slot = in.splits > 1 ? in.slot_base + j : -1;
            items[in.item_off + j] = it;
        }
    }
    if (tid == 0) {
        if (overflow) raise_status(0x8u);
        hdr->n_items = overflow ? 0 : n_items;
        hdr->n_split = overflow ? 0 : n_split;
        hdr->n_bt = n_bt;
        hdr->max_items = max_items;
        hdr->max_slots = max_slots;
    }
}

// ---------------------------------------------------------------------------
// Decode kernel (cluster of 2: rank 0 scores, rank 1 accumulates)
// ---------------------------------------------------------------------------
struct Smem {
    uint32_t base;  // shared::cta address of the aligned base
    __device__ __forceinline__ uint32_t bar(int i) const { return base + kOffBar + 8u * i; }
    __device__ __forceinline__ uint32_t stage(uint32_t s, uint32_t bytes) const { return base + s * bytes; }
    __device__ __forceinline__ uint32_t pbuf(uint32_t j) const { return base + kOffPBuf + j * kMsgBytes; }
    __device__ __forceinline__ uint32_t meta(uint32_t j) const { return pbuf(j) + kPBytes; }
    __device__ __forceinline__ uint32_t evt() const { return base + kOffEvt; }
};

// L2 eviction policies.  Every page is read twice, by the score CTA and microseconds later by
// its partner: the first read uses the normal priority, the second lets the lines go
// (evict_first) -- measured faster than asking L2 to keep them on the first read (evict_last),
// which crowds the working set.  The P ring is rewritten in place and should never leave L2
// (evict_last).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_3d(uint32_t smem_dst, const void *tmap, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(pol)
        : "memory");
}
// global -> shared::cta bulk copy, completion counted on a local barrier
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void st_global_v8_hint(void *dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                                                  uint32_t f, uint32_t g, uint32_t h, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(dst), "r"(a),
                 "r"(b), "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_global_f32_hint(void *dst, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// arrive on a barrier of another CTA with no ordering of this thread's memory operations
// (a pure "slot consumed" signal; nothing written by this thread is published by it)
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Waits whose lanes must stay converged (warp-collective instructions follow): lane 0 waits,
// the outcome is broadcast, and on a failed wait the whole warp leaves together.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait<kCluster>(bar, parity, abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
// Waits of warps that run warp-collective instructions: every lane waits (keeping the warp
// converged, which measured much faster here than one lane waiting and broadcasting), and if
// any lane gave up, the whole warp gives up together.
#define MLA_WAIT_WARP(bar_, par_, ab_) \
    if (__any_sync(0xffffffffu, !mbar_wait(bar_, par_, ab_))) return
// The same all-lane wait, returning the outcome.  The single-thread roles below (shipper, P
// loader, releaser) run as whole warps for it: a lone waiting thread measured a much slower
// wake-up than a converged warp waiting together (about 6% of a batch-64 decode call when the
// page producers and the PV warp waited on one lane).
template <bool kCluster = false>
__device__ __forceinline__ bool all_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    return !__any_sync(0xffffffffu, !mbar_wait<kCluster>(bar, parity, abort));
}

// Page ids of an item, read from the block table 32 tiles at a time (one per lane), one chunk
// ahead of use.  The entries are loaded raw and checked when a page is taken, so start() only
// issues the loads: a caller can start them before other work without waiting for them.
struct PageIds {
    int cur, nxt, chunk;
    __device__ __forceinline__ static int raw(const DecodeParams &p, int b, int tile) {
        return p.block_table[(size_t)b * p.max_pages + tile];
    }
    __device__ __forceinline__ void start(const DecodeParams &p, const ItemInfo &it, int lane) {
        chunk = it.tb;
        cur = it.tb + lane < it.te ? raw(p, it.b, it.tb + lane) : 0;
        nxt = it.tb + 32 + lane < it.te ? raw(p, it.b, it.tb + 32 + lane) : 0;
    }
    // page of `tile` (tiles visited in order); warp-collective.  An entry outside [0, num_pages)
    // sets MLA_DEV_BAD_BLOCK_TABLE and reads page 0 instead.
    __device__ __forceinline__ int get(const DecodeParams &p, const ItemInfo &it, int tile, int lane) {
        if (tile - chunk == 32) {
            chunk += 32;
            cur = nxt;
            nxt = chunk + 32 + lane < it.te ? raw(p, it.b, chunk + 32 + lane) : 0;
        }
        int pg = __shfl_sync(0xffffffffu, cur, tile - chunk);
        if (pg < 0 || pg >= p.num_pages) {
            if (lane == 0) raise_status(0x1u);
            pg = 0;
        }
        return pg;
    }
    // raw entry of a tile at most 32 ahead of the last one taken (no check); warp-collective
    __device__ __forceinline__ int peek(int tile) {
        const int d = tile - chunk;
        const int a = __shfl_sync(0xffffffffu, cur, d & 31);
        const int b = __shfl_sync(0xffffffffu, nxt, d & 31);
        return d < 32 ? a : b;
    }
};

// Accumulate CTA, page producer (a whole warp; lane 0 issues): one box per page, its 512 latent
// columns (blocks 0-7), into a 2-stage ring.  One large box rather than several small ones:
// the TMA engine has a fixed cost per box of the order of the transfer of 40 KB.  The tensor
// map views the pool as (64 columns, rows, 9 column blocks) with strides (2 B, 1152 B, 128 B),
// so a box lands as consecutive 64-row x 128-byte swizzled blocks -- the MMAs' operand layout.
// These reads are a page's second: L2 may drop the lines afterwards (evict_first).
// The loops below return the number of stage positions whose loads they issued; the role then
// drains the last of them (normal exit or abort), so no copy lands after the CTA has moved on.
__device__ __forceinline__ void drain_stages(const Smem &sm, uint32_t issued, uint32_t stages) {
    if ((threadIdx.x & 31) == 0)
        for (uint32_t k = (issued > stages ? issued - stages : 0); k < issued; ++k)
            if (!mbar_wait_drain(sm.bar(kBarFull + k % stages), (k / stages) & 1u)) break;
    __syncwarp();
}

__device__ __forceinline__ void value_producer_loop(const DecodeParams &p, const CUtensorMap *tmap, const Smem &sm,
                                                    const Sched &sc, volatile int *abort, uint32_t &u, Tracer &tr) {
    const int lane = threadIdx.x & 31;
    const uint64_t pol = l2_policy_evict_first();
    ItemInfo it;
    PageIds ids;
    for (int r = 0; sc.get(p, r, it); ++r) {
        ids.start(p, it, lane);
        for (int tile = it.tb; tile < it.te; ++tile, ++u) {
            const int pg = ids.get(p, it, tile, lane);
            const uint32_t s = u % kStagesV;
            tr.at(0x50);
            MLA_WAIT_WARP(sm.bar(kBarEmpty + s), ((u / kStagesV) & 1u) ^ 1u, abort);
            if (lane == 0) {
                mbar_arrive_expect_tx(sm.bar(kBarFull + s), kStageV);
                tma_load_3d(sm.stage(s, kStageV), tmap, 0, pg * kPage, 0, sm.bar(kBarFull + s), pol);
            }
            tr.at(0x51);
            __syncwarp();
        }
    }
}
__device__ __forceinline__ void role_value_producer(const DecodeParams &p, const CUtensorMap *tmap, const Smem &sm,
                                                    const Sched &sc, volatile int *abort, Tracer &tr) {
    uint32_t u = 0;
    value_producer_loop(p, tmap, sm, sc, abort, u, tr);
    drain_stages(sm, u, kStagesV);
}

// Score CTA, page producer (a whole warp; lane 0 issues).  Its stage sequence holds, per item,
// first the absorbed query -- position 0: column blocks 0-3 of all heads and the RoPE block of
// heads 0-63; position 1: blocks 4-7 and the RoPE block of heads 64-127, which exactly fills the
// two stages of its positions -- and then one whole page per position.  Every transfer is one
// large box (the TMA engine's cost per box is high).  Pages are read first here, at the normal
// L2 priority (the partner's second read lets them go); the query is read once (evict_first).
__device__ __forceinline__ void score_producer_loop(const DecodeParams &p, const CUtensorMap *pages,
                                                    const CUtensorMap *qc, const CUtensorMap *qr, const Smem &sm,
                                                    const Sched &sc, volatile int *abort, uint32_t &u, Tracer &tr) {
    const int lane = threadIdx.x & 31;
    const uint64_t keep = l2_policy_evict_normal(), once = l2_policy_evict_first();
    ItemInfo it;
    PageIds ids;
    for (int r = 0; sc.get(p, r, it); ++r) {
        if (it.te <= it.tb) continue;
        const int row0 = it.bt * kHeads;
        ids.start(p, it, lane);  // only issues the block-table loads; they land during the query's
        for (int hq = 0; hq < 2; ++hq, ++u) {
            const uint32_t s = u % kStagesS;
            tr.at(0x12);
            MLA_WAIT_WARP(sm.bar(kBarEmpty + s), ((u / kStagesS) & 1u) ^ 1u, abort);
            tr.at(0x13);
            if (lane == 0) {
                mbar_arrive_expect_tx(sm.bar(kBarFull + s), kStageS);
                tma_load_3d(sm.stage(s, kStageS), qc, 0, row0, 4 * hq, sm.bar(kBarFull + s), once);
                tma_load_3d(sm.stage(s, kStageS) + kQRopeOff, qr, 0, row0 + 64 * hq, kBoxesS - 1, sm.bar(kBarFull + s),
                            once);
            }
            __syncwarp();
        }
        for (int tile = it.tb; tile < it.te; ++tile, ++u) {
            const int pg = ids.get(p, it, tile, lane);
            const uint32_t s = u % kStagesS;
            tr.at(0x10);
            MLA_WAIT_WARP(sm.bar(kBarEmpty + s), ((u / kStagesS) & 1u) ^ 1u, abort);
            tr.at(0x11);
            if (lane == 0) {
                mbar_arrive_expect_tx(sm.bar(kBarFull + s), kStageS);
                tma_load_3d(sm.stage(s, kStageS), pages, 0, pg * kPage, 0, sm.bar(kBarFull + s), keep);
            }
            {
                // the next page, when it does not follow this one in the pool, is prefetched into
                // L2 now: on a randomly paged pool that measured about 5% faster; for pages in
                // pool order the prefetch cost more than it saved, so none is issued
                const int t2 = tile + 1;
                const int pg2 = ids.peek(t2);
                if (lane == 0 && t2 < it.te && pg2 >= 0 && pg2 < p.num_pages && pg2 != pg + 1)
                    tma_prefetch_l2_3d(pages, 0, pg2 * kPage, 0);
            }
            __syncwarp();
        }
    }
}
__device__ __forceinline__ void role_score_producer(const DecodeParams &p, const CUtensorMap *pages,
                                                    const CUtensorMap *qc, const CUtensorMap *qr, const Smem &sm,
                                                    const Sched &sc, volatile int *abort, Tracer &tr) {
    uint32_t u = 0;
    score_producer_loop(p, pages, qc, qr, sm, sc, abort, u, tr);
    drain_stages(sm, u, kStagesS);
}

// Score CTA, MMA issuer warp kMe.  One thread cannot issue N = 64 MMAs fast enough to keep the
// tensor pipe busy; two can.  The issuers take alternate pages -- page g goes to issuer g & 1 and
// into S buffer g & 1 -- and each computes the whole S = Q . K_tile^T of its pages (column blocks
// 0-7 and the RoPE block 8, A from TMEM), so the pipe sees two independent streams.  Both
// issuers still walk every stage position in order: the page's issuer commits its MMAs to the
// stage's empty barrier and the other one adds a plain arrival once the page has landed, so a
// stage is refilled only after both have passed it -- a parity wait can then never see its
// barrier a phase behind or two phases ahead.  Both hand the two query stages back (one plain
// arrival each) once the softmax warps report the query in TMEM.  The whole warp runs the loop,
// so the descriptors stay warp-uniform values; one lane issues the MMAs and commits.
template <int kMe>
__device__ __forceinline__ void score_mma_loop(const DecodeParams &p, const Smem &sm, uint32_t tmem, const Sched &sc,
                                               volatile int *abort, Tracer &tr) {
    const bool leader = (threadIdx.x & 31) == 0;
    uint32_t g = 0, ic = 0, u = 0;
    ItemInfo it;
    for (int r = 0; sc.get(p, r, it); ++r) {
        if (it.te <= it.tb) continue;
        tr.at(0x20);
        MLA_WAIT_WARP(sm.bar(kBarQReady), ic & 1u, abort);
        tr.at(0x21);
        tc_fence_after();
        ++ic;
        // acknowledge: the softmax warps complete the next item's QReady only after both issuers
        // have seen this one, so an issuer with no page in an item cannot fall two phases behind
        if (leader) {
            mbar_arrive(sm.bar(kBarQAck));
            mbar_arrive(sm.bar(kBarEmpty + u % kStagesS));
            mbar_arrive(sm.bar(kBarEmpty + (u + 1) % kStagesS));
        }
        __syncwarp();
        u += 2;
        for (int tile = it.tb; tile < it.te; ++tile, ++g, ++u) {
            const uint32_t s = u % kStagesS, buf = (uint32_t)kMe;
            // every position is waited for in order, so no parity wait can run ahead of its
            // barrier; a position of the other issuer's page only gets this warp's release
            tr.at(0x22);
            MLA_WAIT_WARP(sm.bar(kBarFull + s), (u / kStagesS) & 1u, abort);
            if ((g & 1u) != (uint32_t)kMe) {
                tr.at(0x24);
                if (leader) mbar_arrive(sm.bar(kBarEmpty + s));
                __syncwarp();
                continue;
            }
            tr.at(0x23);
            MLA_WAIT_WARP(sm.bar(kBarSEmpty + (int)buf), ((g >> 1) & 1u) ^ 1u, abort);
            tr.at(0x25);
            tc_fence_after();
            const uint32_t d = tmem + kTmemS + buf * 64u;
            const uint32_t st = sm.stage(s, kStageS);
            const uint64_t b0 = sdesc_sw128(st, 16u, 1024u);
            if (leader) {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const uint32_t bx = (uint32_t)k >> 2, kk = (uint32_t)k & 3u;
                    mma_ts(d, tmem + kTmemQ + bx * 32u + kk * 8u, b0 + (uint64_t)((bx * kBoxBytes + kk * 32u) >> 4),
                           kIdescS, k != 0);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // the RoPE block
                    mma_ts(d, tmem + kTmemQR + kk * 8u, b0 + (uint64_t)((8u * kBoxBytes + 32u * kk) >> 4), kIdescS, 1u);
                mma_commit(sm.bar(kBarEmpty + s));
                mma_commit(sm.bar(kBarSFull + (int)buf));
            }
            tr.at(0x26);
            __syncwarp();
        }
    }
}
// On any exit, normal or after an abort, every MMA this warp issued has completed before the
// CTA can free its tensor memory: a final commit, waited for with the abort-ignoring bound.
template <int kMe>
__device__ __forceinline__ void role_score_mma(const DecodeParams &p, const Smem &sm, uint32_t tmem, const Sched &sc,
                                               volatile int *abort, Tracer &tr) {
    score_mma_loop<kMe>(p, sm, tmem, sc, abort, tr);
    if ((threadIdx.x & 31) == 0) {
        mma_commit(sm.bar(kBarDrain + kMe));
        mbar_wait_drain(sm.bar(kBarDrain + kMe), 0);
    }
    __syncwarp();
}

// Score CTA, softmax warps.  Eight warps, two per sub-partition: warp w owns heads
// 32(w%4) .. 32(w%4)+31 (its TMEM lane quadrant) and columns [32 hf, 32 hf + 32) of each page,
// hf = w / 4.  Both threads of a head read the whole S row to take its maximum, so they make
// identical rescale decisions without exchanging anything; they swap their row sums through
// shared memory on an item's last page.  Per page: online softmax with lazy rescaling, write the
// half-row of the P message (bf16 in the UMMA K-major 128-byte-swizzle image, the rescale factor,
// and 1/l on the item's last page) into the ring, then signal the shipper.
__device__ __forceinline__ void role_softmax(const DecodeParams &p, const Smem &sm, uint32_t tmem, const Sched &scd,
                                             volatile int *abort, Tracer &tr) {
    const int w = threadIdx.x >> 5, q4 = w & 3, hf = w >> 2, lane = threadIdx.x & 31;
    const int h = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = p.sl2;
    const uint32_t row_off = (uint32_t)(h >> 3) * 1024u + (uint32_t)(h & 7) * 128u;
    uint8_t *const ring = p.ring + (size_t)scd.cid * kRing * kMsgBytes;
    const uint32_t xsum = sm.base + kOffXSum;
    const uint64_t keep = l2_policy_evict_last();
    uint32_t sc = 0, nsum = 0, us = 0;
    int staged_pending = -1;  // ring slot whose message is written but not yet released to the shipper
    ItemInfo it;
    for (int r = 0; scd.get(p, r, it); ++r) {
        if (it.te <= it.tb) {
            if (hf == 0) p.lse[(size_t)it.bt * kHeads + h] = -INFINITY;
            continue;
        }
        // both issuers have seen the previous item's QReady before this item's can complete
        // (nsum counts the items finished so far)
        tr.at(0x30);
        if (nsum > 0) MLA_WAIT_WARP(sm.bar(kBarQAck), (nsum - 1u) & 1u, abort);
        // this head's absorbed query, from the item's two query stages (the previous item's MMAs
        // are done: its last S tile has been read): content blocks 4 hf .. 4 hf + 3 -> TMEM lane h
        // (bf16 pairs), and for hf = 1 the RoPE block -> TMEM lane h too.  Both stages hold
        // 128-byte swizzled rows whose swizzle phase is h & 7.  The issuers free the stages.
        {
            const uint32_t pc = us + (uint32_t)hf;
            MLA_WAIT_WARP(sm.bar(kBarFull + pc % kStagesS), (pc / kStagesS) & 1u, abort);
            const uint32_t stc = sm.stage(pc % kStagesS, kStageS) + (uint32_t)h * 128u;
#pragma unroll 1
            for (int bq = 0; bq < 4; ++bq) {
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[4 * c]), "=r"(v[4 * c + 1]), "=r"(v[4 * c + 2]), "=r"(v[4 * c + 3])
                                 : "r"(stc + (uint32_t)bq * (kHeads * 128u) + (uint32_t)((c ^ (lane & 7)) * 16))
                                 : "memory");
                tmem_st32(tmem + lane_off + kTmemQ + (4u * hf + bq) * 32u, v);
            }
            if (hf) {
                const uint32_t pr = us + (uint32_t)(q4 >> 1);  // heads 0-63: first stage, 64-127: second
                if (pr != pc) MLA_WAIT_WARP(sm.bar(kBarFull + pr % kStagesS), (pr / kStagesS) & 1u, abort);
                const uint32_t src = sm.stage(pr % kStagesS, kStageS) + kQRopeOff + (uint32_t)(h & 63) * 128u;
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v[4 * c]), "=r"(v[4 * c + 1]), "=r"(v[4 * c + 2]), "=r"(v[4 * c + 3])
                                 : "r"(src + (uint32_t)((c ^ (lane & 7)) * 16))
                                 : "memory");
                tmem_st32(tmem + lane_off + kTmemQR, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(sm.bar(kBarQReady));
            tr.at(0x31);
            us += 2u + (uint32_t)(it.te - it.tb);
        }
        // l: the row sum of the unrounded probabilities (for the lse); lr: the sum of the bf16
        // probabilities the PV product actually uses, which normalises O -- numerator and
        // denominator then carry the same rounding, which matters when a few tokens dominate
        float m = 0.f, l = 0.f, lr = 0.f, lt = 0.f, lrt = 0.f;
        for (int tile = it.tb; tile < it.te; ++tile, ++sc) {
            const uint32_t buf = sc & 1u;
            tr.at(0x32);
            MLA_WAIT_WARP(sm.bar(kBarSFull + (int)buf), (sc >> 1) & 1u, abort);
            tr.at(0x33);
            tc_fence_after();
            // this thread's half of the row, and the other half for the row maximum only: both
            // threads of a head then take the same maximum (fmaxf is exact and order-free)
            // without exchanging anything
            const int vrow = min(kPage, it.n_vis - tile * kPage);  // valid columns of the page
            float s[32], omx;
            {
                uint32_t a[32], b[32];
                tmem_ld32(tmem + lane_off + kTmemS + buf * 64u + 32u * hf, a);
                tmem_ld32(tmem + lane_off + kTmemS + buf * 64u + 32u * (1 - hf), b);
                tmem_ld_wait_dep(a);
                tmem_ld_wait_dep(b);
                const int vo = vrow - 32 * (1 - hf);
                if (vo >= 32) {
                    omx = fmax3(fmax3(__uint_as_float(b[0]), __uint_as_float(b[1]), __uint_as_float(b[2])),
                                fmax3(__uint_as_float(b[3]), __uint_as_float(b[4]), __uint_as_float(b[5])),
                                __uint_as_float(b[6]));
#pragma unroll
                    for (int c = 7; c < 31; c += 2)
                        omx = fmax3(omx, __uint_as_float(b[c]), __uint_as_float(b[c + 1]));
                    omx = fmaxf(omx, __uint_as_float(b[31]));
                } else {  // the page's ragged tail
                    omx = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 32; ++c) omx = c < vo ? fmaxf(omx, __uint_as_float(b[c])) : omx;
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(a[c]);
            }
            tc_fence_before();
            mbar_arrive(sm.bar(kBarSEmpty + (int)buf));
            tr.at(0x34);
            // the previous page's message, whose stores have had a page's time to complete, is
            // released to the shipper now rather than right after them (the release would wait
            // for them)
            if (staged_pending >= 0) {
                mbar_arrive(sm.bar(kBarPStaged + staged_pending));
                staged_pending = -1;
            }

            const int valid = vrow - 32 * hf;  // columns of this half
            if (valid < 32) {
#pragma unroll
                for (int c = 0; c < 32; ++c) s[c] = c < valid ? s[c] : -INFINITY;
            }
            float lmx = fmax3(fmax3(s[0], s[1], s[2]), fmax3(s[3], s[4], s[5]), s[6]);
#pragma unroll
            for (int c = 7; c < 31; c += 2) lmx = fmax3(lmx, s[c], s[c + 1]);
            lmx = fmaxf(lmx, s[31]);
            const float mx = fmaxf(lmx, omx) * sl2;
            const bool first = tile == it.tb;
            const bool last = tile == it.te - 1;
            float alpha = 1.f;
            if (first) {
                m = mx;
            } else if (mx > m + kTau) {
                alpha = ex2_approx(m - mx);
                l *= alpha;
                lr *= alpha;
                m = mx;
            }
            // p = 2^(s sl2 - m) on pairs: one paired FMA, two exponentials, one bf16 pair; the two
            // row sums on pairs too
            uint32_t pk[16];
            uint64_t ls2[2] = {0ull, 0ull}, lr2[2] = {0ull, 0ull};
            const uint64_t sl2x2 = f32x2(sl2, sl2), nmx2 = f32x2(-m, -m);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                float y0, y1;
                f32x2_split(fma_f32x2(f32x2(s[2 * c], s[2 * c + 1]), sl2x2, nmx2), y0, y1);
                const float a = ex2_approx(y0), b = ex2_approx(y1);
                pk[c] = pack_bf16x2(a, b);
                ls2[c & 1] = add_f32x2(ls2[c & 1], f32x2(a, b));
                lr2[c & 1] = add_f32x2(lr2[c & 1], f32x2(bf16lo_to_f32(pk[c]), bf16hi_to_f32(pk[c])));
            }
            {
                float a0, a1, b0, b1;
                f32x2_split(add_f32x2(ls2[0], ls2[1]), a0, a1);
                f32x2_split(add_f32x2(lr2[0], lr2[1]), b0, b1);
                l += a0 + a1;
                lr += b0 + b1;
            }
            if (last) {  // the whole row's sums, for 1/l and the lse
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(xsum + (uint32_t)(hf * kHeads + h) * 4u), "f"(l) : "memory");
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(xsum + (uint32_t)((2 + hf) * kHeads + h) * 4u), "f"(lr)
                             : "memory");
                const uint32_t sbar = sm.bar(kBarXSum + q4);
                mbar_arrive(sbar);
                MLA_WAIT_WARP(sbar, nsum & 1u, abort);
                ++nsum;
                float ol, olr;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(ol) : "r"(xsum + (uint32_t)((1 - hf) * kHeads + h) * 4u) : "memory");
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(olr) : "r"(xsum + (uint32_t)((3 - hf) * kHeads + h) * 4u)
                             : "memory");
                lt = hf == 0 ? l + ol : ol + l;  // the same sums, in the same order, in both halves
                lrt = hf == 0 ? lr + olr : olr + lr;
            }

            // the message, straight into its ring slot once the partner has taken the slot's
            // previous content (a plain signal: that copy completed before the partner
            // arrived): this half-row of P in the UMMA K-major 128-byte-swizzle image, the
            // rescale factor, and 1/l on the item's last page
            const uint32_t rs = sc % kRing;
            tr.at(0x35);
            MLA_WAIT_WARP(sm.bar(kBarPFree + rs), ((sc / kRing) & 1u) ^ 1u, abort);
            tr.at(0x36);
            uint8_t *msg = ring + (size_t)rs * kMsgBytes;
            // chunks 2v and 2v + 1 of this half-row land in one aligned 32-byte sector (the swizzle
            // flips the low bit of the chunk index, or not): one 32-byte store per pair
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const uint32_t p0 = (uint32_t)((4 * hf + 2 * v) ^ (h & 7));
                const bool swap = (p0 & 1u) != 0;
                uint32_t w8[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w8[i] = swap ? pk[8 * v + 4 + i] : pk[8 * v + i];
                    w8[4 + i] = swap ? pk[8 * v + i] : pk[8 * v + 4 + i];
                }
                st_global_v8_hint(msg + row_off + (p0 & ~1u) * 16u, w8[0], w8[1], w8[2], w8[3], w8[4], w8[5], w8[6],
                                  w8[7], keep);
            }
            if (hf == 0) {
                st_global_f32_hint(msg + kPBytes + 4u * h, alpha, keep);
                if (last) st_global_f32_hint(msg + kPBytes + 4u * (kHeads + h), 1.0f / lrt, keep);
            }
            // local release; the shipper publishes the slot to the partner.  An item's last message
            // goes at once (the partner's epilogue waits for it); the others are released after the
            // next page's scores have been read, by when their stores are done
            if (last)
                mbar_arrive(sm.bar(kBarPStaged + rs));
            else
                staged_pending = (int)rs;
            tr.at(0x37);
        }
        if (hf == 0) {
            const float lse = (m + __log2f(lt)) * 0.69314718055994531f;
            if (it.slot < 0)
                p.lse[(size_t)it.bt * kHeads + h] = lse;
            else
                p.part_lse[(size_t)it.slot * kHeads + h] = lse;
        }
    }
}

// Score CTA, shipper (a warp that waits together; lane 0 acts): publishes the messages the softmax warps have written to
// the partner.  It waits for the oldest unpublished message, takes the later ones of the same
// item that are already complete (up to kMaxBatch), and publishes them together: one
// cluster-scope release fence, then a relaxed remote arrival per message.  The fence waits
// for the rows' stores to complete and costs about a microsecond here, so messages that pile
// up meanwhile share the next one, while a message that comes alone (an item's first and
// last pages) goes out at once.  The shipper acquired the rows through the local barriers
// and the fence is cumulative, so the partner's acquire sees every row.
__device__ __forceinline__ void role_shipper(const DecodeParams &p, const Smem &sm, const Sched &sc,
                                             volatile int *abort, Tracer &tr) {
    const bool lead = (threadIdx.x & 31) == 0;
    uint32_t g = 0;
    ItemInfo it;
    for (int r = 0; sc.get(p, r, it); ++r) {
        const uint32_t end = g + (uint32_t)(it.te > it.tb ? it.te - it.tb : 0);
        while (g < end) {
            tr.at(0x40);
            if (!all_wait(sm.bar(kBarPStaged + g % kRing), (g / kRing) & 1u, abort)) return;
            tr.at(0x41);
            uint32_t n = 1;
            if (lead) {
                while (g + n < end && n < (uint32_t)kMaxBatch &&
                       mbar_test(sm.bar(kBarPStaged + (g + n) % kRing), ((g + n) / kRing) & 1u))
                    ++n;
                fence_acq_rel_cluster();
                for (uint32_t k = 0; k < n; ++k)
                    mbar_arrive_cluster_relaxed(mapa_shared(sm.bar(kBarPReady + (g + k) % kRing), 1));
            }
            n = __shfl_sync(0xffffffffu, n, 0);
            tr.at(0x4200 + n);
            g += n;
        }
    }
}

// Accumulate CTA, releaser (a warp that waits together; lane 0 acts): hands each ring slot back to the partner as soon as
// its message has landed in shared memory, off the MMA warp's path.  Its local arrival is
// the second one each P buffer needs before the loader refills it, so this thread can never
// fall a whole buffer cycle behind the barrier it watches.
__device__ __forceinline__ void role_releaser(const DecodeParams &p, const Smem &sm, const Sched &sc,
                                              volatile int *abort) {
    const bool lead = (threadIdx.x & 31) == 0;
    uint32_t g = 0;
    ItemInfo it;
    for (int r = 0; sc.get(p, r, it); ++r) {
        for (int tile = it.tb; tile < it.te; ++tile, ++g) {
            if (!all_wait(sm.bar(kBarPFull + g % kPBufs), (g / kPBufs) & 1u, abort)) return;
            if (lead) {
                mbar_arrive_cluster_relaxed(mapa_shared(sm.bar(kBarPFree + g % kRing), 0));
                mbar_arrive(sm.bar(kBarPBufFree + g % kPBufs));
            }
            __syncwarp();
        }
    }
}

// Accumulate CTA, P loader (a warp that waits together; lane 0 copies): ring slot -> shared P buffer, as soon as the
// partner has published it and the buffer's previous message has been used.
__device__ __forceinline__ void p_loader_loop(const DecodeParams &p, const Smem &sm, const Sched &sc,
                                              volatile int *abort, uint32_t &g, Tracer &tr) {
    const uint8_t *ring = p.ring + (size_t)sc.cid * kRing * kMsgBytes;
    const uint64_t keep = l2_policy_evict_last();
    ItemInfo it;
    for (int r = 0; sc.get(p, r, it); ++r) {
        for (int tile = it.tb; tile < it.te; ++tile, ++g) {
            const uint32_t rs = g % kRing, jp = g % kPBufs;
            tr.at(0x60);
            if (!all_wait<true>(sm.bar(kBarPReady + rs), (g / kRing) & 1u, abort)) return;
            tr.at(0x61);
            fence_proxy_async_global();  // the partner's writes, before our async-proxy reads
            if (!all_wait(sm.bar(kBarPBufFree + jp), ((g / kPBufs) & 1u) ^ 1u, abort)) return;
            tr.at(0x62);
            if ((threadIdx.x & 31) == 0) {
                mbar_arrive_expect_tx(sm.bar(kBarPFull + jp), kMsgBytes);
                // P and its factors are contiguous in both places: one copy (the copy engine's
                // cost per transfer is high)
                bulk_load_g2s(sm.pbuf(jp), ring + (size_t)rs * kMsgBytes, kMsgBytes, sm.bar(kBarPFull + jp), keep);
            }
            __syncwarp();
        }
    }
}
// the copies issued last may still be in flight after an abort: wait for them (bounded)
__device__ __forceinline__ void role_p_loader(const DecodeParams &p, const Smem &sm, const Sched &sc,
                                              volatile int *abort, Tracer &tr) {
    uint32_t g = 0;
    p_loader_loop(p, sm, sc, abort, g, tr);
    if ((threadIdx.x & 31) == 0)
        for (uint32_t k = (g > (uint32_t)kPBufs ? g - kPBufs : 0); k < g; ++k)
            if (!mbar_wait_drain(sm.bar(kBarPFull + k % kPBufs), (k / kPBufs) & 1u)) break;
    __syncwarp();
}

// Accumulate CTA, MMA warp: O += P V, two N = 256 halves, K = 64 in 4 steps.  It also
// hands rescale and epilogue events to the epilogue warps through the local event buffer:
// the event data is written, then the event barrier gets two arrivals -- this warp's
// (release: the data is visible) and the MMA commit (all earlier MMAs have completed).
__device__ __forceinline__ void accum_mma_loop(const DecodeParams &p, const Smem &sm, uint32_t tmem, const Sched &sc,
                                               volatile int *abort, Tracer &tr) {
    const int lane = threadIdx.x & 31;
    uint32_t g = 0, cv = 0;
    bool pending_epilogue = false;
    uint32_t staging_buf = 0;  // P buffer the epilogue warps are writing the output through
    const uint32_t evt = sm.evt();
    ItemInfo it;
    for (int r = 0; sc.get(p, r, it); ++r) {
        for (int tile = it.tb; tile < it.te; ++tile, ++g) {
            const uint32_t jp = g % kPBufs;
            const bool first = tile == it.tb, last = tile == it.te - 1;
            const uint32_t valid = (uint32_t)min(kPage, it.n_vis - tile * kPage);
            tr.at(0x70);
            MLA_WAIT_WARP(sm.bar(kBarPFull + jp), (g / kPBufs) & 1u, abort);
            tr.at(0x71);
            const uint32_t mt = sm.meta(jp);
            if (first) {
                if (pending_epilogue) {  // the previous item's O must have been read out
                    if (!warp_wait(sm.bar(kBarCorrEvt), cv & 1u, abort)) return;
                    ++cv;
                    pending_epilogue = false;
                    if (lane == 0) mbar_arrive(sm.bar(kBarPBufFree + staging_buf));  // staging done
                }
            } else {
                float4 a4;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(a4.x), "=f"(a4.y), "=f"(a4.z), "=f"(a4.w)
                             : "r"(mt + 16u * lane)
                             : "memory");
                const bool any = __any_sync(0xffffffffu, a4.x != 1.f || a4.y != 1.f || a4.z != 1.f || a4.w != 1.f);
                if (any) {
                    // rescale event: per-head factors to the event buffer, then wait for the rows
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(evt + 16u * lane), "f"(a4.x),
                                 "f"(a4.y), "f"(a4.z), "f"(a4.w)
                                 : "memory");
                    __syncwarp();
                    if (lane == 0) {
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(evt + 1024u), "r"(kEvtRescale) : "memory");
                        mbar_arrive(sm.bar(kBarMmaEvt));
                        mma_commit(sm.bar(kBarMmaEvt));
                    }
                    __syncwarp();
                    tr.at(0x72);
                    if (!warp_wait(sm.bar(kBarCorrEvt), cv & 1u, abort)) return;
                    tr.at(0x73);
                    ++cv;
                }
            }
            const uint64_t a0 = sdesc_sw128(sm.pbuf(jp), 16u, 1024u);
            const uint32_t s = g % kStagesV;
            MLA_WAIT_WARP(sm.bar(kBarFull + s), (g / kStagesV) & 1u, abort);
            tr.at(0x74);
            const uint32_t vb = sm.stage(s, kStageV);
            if (last && valid < (uint32_t)kPage) {
                // rows past the end of the sequence may hold anything (even NaN): zero them,
                // since 0 * NaN would poison O even though their probabilities are 0
                const uint32_t nrow = kPage - valid;
                for (uint32_t e = lane; e < nrow * 8u * kBoxesV; e += 32) {
                    const uint32_t bx = e / (nrow * 8u), rem = e % (nrow * 8u);
                    const uint32_t row = valid + rem / 8u, ch = rem % 8u;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vb + bx * kBoxBytes + row * 128u +
                                                                                   ch * 16u),
                                 "r"(0u)
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const uint64_t v0 = sdesc_sw128(vb + (uint32_t)n * 4u * kBoxBytes, (uint32_t)kBoxBytes, 1024u);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss(tmem + 256u * n, a0 + (uint64_t)((32u * k) >> 4), v0 + (uint64_t)((2048u * k) >> 4),
                               kIdescPV, !(first && k == 0));
                }
                mma_commit(sm.bar(kBarEmpty + s));
                // an item's last P buffer is released after the epilogue has used it
                if (!last) mma_commit(sm.bar(kBarPBufFree + jp));
            }
            tr.at(0x75);
            __syncwarp();
            if (last) {
                // epilogue event: 1/l per head to the event buffer
                asm volatile("{\n\t.reg .b32 x, y, z, w;\n\t"
                             "ld.shared.v4.b32 {x, y, z, w}, [%0];\n\t"
                             "st.shared.v4.b32 [%1], {x, y, z, w};\n\t}" ::"r"(mt + 512u + 16u * lane),
                             "r"(evt + 512u + 16u * lane)
                             : "memory");
                __syncwarp();
                if (lane == 0) {
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(evt + 1024u), "r"(kEvtEpilogue) : "memory");
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(evt + 1028u), "r"(jp) : "memory");
                    mbar_arrive(sm.bar(kBarMmaEvt));
                    mma_commit(sm.bar(kBarMmaEvt));
                }
                pending_epilogue = true;
                staging_buf = jp;
            }
            __syncwarp();
        }
    }
    if (pending_epilogue) warp_wait(sm.bar(kBarCorrEvt), cv & 1u, abort);
}
// every MMA this warp issued has completed before the CTA can free its tensor memory
__device__ __forceinline__ void role_accum_mma(const DecodeParams &p, const Smem &sm, uint32_t tmem, const Sched &sc,
                                               volatile int *abort, Tracer &tr) {
    accum_mma_loop(p, sm, tmem, sc, abort, tr);
    if ((threadIdx.x & 31) == 0) {
        mma_commit(sm.bar(kBarDrain));
        mbar_wait_drain(sm.bar(kBarDrain), 0);
    }
    __syncwarp();
}

// Accumulate CTA, epilogue warps.  Eight warps: warp w owns heads 32(w%4) .. +31 (its TMEM
// lane quadrant) and latent columns [256 hf, 256 hf + 256), hf = w / 4.  They serve events --
// rescale their part of the O rows, or write the normalised output of the finished item.
// A thread holds one row of O, so the output goes through shared memory (2 KB per warp, in
// the item's last P buffer, whose MMAs have completed): each thread stages 64 bytes of its row,
// then each store instruction writes 64 contiguous bytes of 8 rows instead of 16 bytes of 32.
// The staged 16-byte chunks are rotated by row so that neither side has bank conflicts.
__device__ __forceinline__ void stage_and_store(uint32_t stg, int lane, const uint32_t (&v)[16], uint8_t *row0,
                                                size_t row_bytes) {
    const uint32_t rot = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + (uint32_t)lane * 64u +
                                                                     (((uint32_t)k ^ rot) * 16u)),
                     "r"(v[4 * k]), "r"(v[4 * k + 1]), "r"(v[4 * k + 2]), "r"(v[4 * k + 3])
                     : "memory");
    __syncwarp();
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
        const uint32_t rr = 8u * s4 + ((uint32_t)lane >> 2), j = (uint32_t)lane & 3u;
        uint4 x;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                     : "r"(stg + rr * 64u + ((j ^ ((rr >> 1) & 3u)) * 16u))
                     : "memory");
        *reinterpret_cast<uint4 *>(row0 + rr * row_bytes + j * 16u) = x;
    }
    __syncwarp();
}

__device__ __forceinline__ void role_accum_epilogue(const DecodeParams &p, const Smem &sm, uint32_t tmem,
                                                    const Sched &sc, volatile int *abort, Tracer &tr) {
    const int w = threadIdx.x >> 5, q4 = w & 3, hf = w >> 2, lane = threadIdx.x & 31;
    const int h = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t col0 = 256u * hf;
    const uint32_t evt = sm.evt();
    uint32_t ev = 0;
    ItemInfo it;
    for (int r = 0; sc.get(p, r, it); ++r) {
        if (it.te <= it.tb) {
            uint4 *o = reinterpret_cast<uint4 *>(p.o_lat + ((size_t)it.bt * kHeads + h) * kDc + col0);
            for (int c = 0; c < 256 * 2 / 16; ++c) o[c] = make_uint4(0, 0, 0, 0);
            continue;
        }
        for (;;) {
            tr.at(0x80);
            MLA_WAIT_WARP(sm.bar(kBarMmaEvt), ev & 1u, abort);
            tr.at(0x81);
            ++ev;
            tc_fence_after();
            uint32_t type;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(type) : "r"(evt + 1024u) : "memory");
            if (type == kEvtRescale) {
                float alpha;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(alpha) : "r"(evt + 4u * h) : "memory");
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_off + col0 + c * 32u, v);
                        tmem_ld_wait_dep(v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(tmem + lane_off + col0 + c * 32u, v);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(sm.bar(kBarCorrEvt));
                tr.at(0x82);
                continue;
            }
            float inv_l;
            uint32_t jp;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(inv_l) : "r"(evt + 512u + 4u * h) : "memory");
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(jp) : "r"(evt + 1028u) : "memory");
            const uint32_t stg = sm.pbuf(jp) + (uint32_t)w * 2048u;
            // each chunk's TMEM load is issued before the previous chunk is stored
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + col0, v);
            if (it.slot < 0) {
                uint8_t *row0 = reinterpret_cast<uint8_t *>(p.o_lat + ((size_t)it.bt * kHeads + q4 * 32) * kDc + col0);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    tmem_ld_wait_dep(v);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv_l, __uint_as_float(v[2 * e + 1]) * inv_l);
                    if (c + 1 < 8) tmem_ld32(tmem + lane_off + col0 + (c + 1) * 32u, v);
                    stage_and_store(stg, lane, pk, row0 + c * 64, (size_t)kDc * 2);
                }
            } else {
                uint8_t *row0 = reinterpret_cast<uint8_t *>(p.part_o + ((size_t)it.slot * kHeads + q4 * 32) * kDc + col0);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    tmem_ld_wait_dep(v);
                    uint32_t lo[16], hi[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        lo[e] = __float_as_uint(__uint_as_float(v[e]) * inv_l);
                        hi[e] = __float_as_uint(__uint_as_float(v[16 + e]) * inv_l);
                    }
                    if (c + 1 < 8) tmem_ld32(tmem + lane_off + col0 + (c + 1) * 32u, v);
                    stage_and_store(stg, lane, lo, row0 + c * 128, (size_t)kDc * 4);
                    stage_and_store(stg, lane, hi, row0 + c * 128 + 64, (size_t)kDc * 4);
                }
            }
            // the staging writes (generic proxy) before the loader's next bulk copy into the buffer
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(sm.bar(kBarCorrEvt));
            tr.at(0x84);
            break;
        }
    }
}

// Launched with a cluster dimension of 2 (rank 0 scores, rank 1 accumulates), 13 warps:
// 0-7 softmax (rank 0) / epilogue (rank 1), 8 page producer, 9-10 the two score MMA
// issuers (rank 0) / 9-11 the PV MMA warp, the P loader and the ring-slot releaser (rank 1),
// 12 the message shipper (rank 0).
__global__ void __launch_bounds__(kDecodeThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_v,
              const __grid_constant__ CUtensorMap tmap_qc, const __grid_constant__ CUtensorMap tmap_qr,
              const DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Tracer tr;
    tr.at(0x8001);
    tr.at(0x01);
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();
    uint8_t *const gbase = smem_raw + (sm.base - raw);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + kOffAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffTmemPtr);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesMax; ++s) {
            mbar_init(sm.bar(kBarFull + s), 1);
            // score: the page's issuer commits and the other issuer arrives (both arrive for a
            // query stage); accumulate: the PV MMA commit
            mbar_init(sm.bar(kBarEmpty + s), rank == 0 ? 2 : 1);
        }
        for (int j = 0; j < 2; ++j) mbar_init(sm.bar(kBarSFull + j), 1);  // the page's issuer commits
        for (int j = 0; j < 2; ++j) mbar_init(sm.bar(kBarSEmpty + j), 256);  // every softmax thread
        mbar_init(sm.bar(kBarQReady), 256);
        mbar_init(sm.bar(kBarQAck), 2);             // each score issuer, once per item
        for (int j = 0; j < 2; ++j) mbar_init(sm.bar(kBarDrain + j), 1);
        for (int j = 0; j < kRing; ++j) {
            mbar_init(sm.bar(kBarPFree + j), 1);     // score CTA: the partner's releaser
            mbar_init(sm.bar(kBarPReady + j), 1);    // accumulate CTA: the partner's shipper
            mbar_init(sm.bar(kBarPStaged + j), 256); // score CTA: softmax threads
        }
        for (int j = 0; j < kPBufs; ++j) {
            mbar_init(sm.bar(kBarPFull + j), 1);     // accumulate CTA: armed by the P loader
            mbar_init(sm.bar(kBarPBufFree + j), 2);  // accumulate CTA: MMA commit (or epilogue done) + releaser
        }
        mbar_init(sm.bar(kBarMmaEvt), 2);            // MMA warp arrive + MMA commit
        mbar_init(sm.bar(kBarCorrEvt), 256);  // every epilogue thread
        for (int j = 0; j < 4; ++j) mbar_init(sm.bar(kBarXSum + j), 64);  // the two warps of a quadrant
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(sm.base + kOffTmemPtr, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpProducer && (threadIdx.x & 31) == 0) {
        if (rank == 0) {
            tma_prefetch_desc(&tmap_s);
            tma_prefetch_desc(&tmap_qc);
            tma_prefetch_desc(&tmap_qr);
        } else {
            tma_prefetch_desc(&tmap_v);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the partner's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched as a programmatic dependent of the plan kernel: everything above overlapped it;
    // the plan's results are read only after it has completed
    grid_dependency_wait();
    tr.at(0x02);
    grid_launch_dependents();  // let the combine kernel's blocks get resident early
    Sched sc;
    sc.cid = (int)cluster_id_x();
    sc.ncl = (int)nclusters_x();
    sc.n_items = p.hdr->n_items;
    sc.first = load_item(p, sc.cid < p.max_items ? sc.cid : 0);  // needed only if cid < n_items

    if (warp < 8) {
        if (rank == 0)
            role_softmax(p, sm, tmem, sc, abort, tr);
        else
            role_accum_epilogue(p, sm, tmem, sc, abort, tr);
    } else if (warp == kWarpProducer) {
        if (rank == 0)
            role_score_producer(p, &tmap_s, &tmap_qc, &tmap_qr, sm, sc, abort, tr);
        else
            role_value_producer(p, &tmap_v, sm, sc, abort, tr);
    } else if (warp < kWarpMma + 3) {
        if (rank == 0) {
            if (warp == kWarpMma) role_score_mma<0>(p, sm, tmem, sc, abort, tr);
            if (warp == kWarpMma + 1) role_score_mma<1>(p, sm, tmem, sc, abort, tr);
        } else if (warp == kWarpMma) {
            role_accum_mma(p, sm, tmem, sc, abort, tr);
        } else if (warp == kWarpMma + 1) {
            role_p_loader(p, sm, sc, abort, tr);
        } else {
            role_releaser(p, sm, sc, abort);
        }
    } else if (warp == kWarpShipper) {
        if (rank == 0) role_shipper(p, sm, sc, abort, tr);
    }
    tr.at(0x03);

    // every thread's own tensor-memory loads and stores have completed (they may be in flight
    // when a role left early after an abort)
    tmem_ld_wait();
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA retires while its partner may still arrive on it
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    tr.at(0x04);
    tr.at(0x8004);
}

// ---------------------------------------------------------------------------
// LSE combine: merge the partials of queries that were split.
// ---------------------------------------------------------------------------
// The LSE merge of one (query, head) row's partial results, by 64 threads taking 8 columns each.
constexpr int kCombineThreads = 256;
constexpr int kCombineHeads = kCombineThreads / 64;  // rows per block
__device__ __forceinline__ void combine_row(const float *o_base, size_t o_stride, const float *lse_base,
                                            size_t lse_stride, int n_parts, int col0, __nv_bfloat16 *o_out,
                                            float *lse_out, bool write_lse) {
    // lse = log sum_r exp(lse_r), taken about the largest; the 64 threads of a row read the
    // same lse values (one line, from L1)
    float mx = -INFINITY;
    for (int r = 0; r < n_parts; ++r) mx = fmaxf(mx, lse_base[r * lse_stride]);
    float L = -INFINITY;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    if (mx != -INFINITY) {
        float tot = 0.f;
        for (int r = 0; r < n_parts; ++r) tot += expf(lse_base[r * lse_stride] - mx);
        L = mx + logf(tot);
        // eight parts at a time, all their loads in flight before any is used; a part whose
        // weight is 0 (lse = -inf) is left out, whatever its output holds
        for (int r0 = 0; r0 < n_parts; r0 += 8) {
            float w[8];
            float4 x0[8], x1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r0 + j < n_parts) {
                    w[j] = expf(lse_base[(r0 + j) * lse_stride] - L);
                    const float4 *src = reinterpret_cast<const float4 *>(o_base + (r0 + j) * o_stride + col0);
                    x0[j] = src[0];
                    x1[j] = src[1];
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r0 + j < n_parts && w[j] != 0.f) {
                    a0.x = fmaf(w[j], x0[j].x, a0.x);
                    a0.y = fmaf(w[j], x0[j].y, a0.y);
                    a0.z = fmaf(w[j], x0[j].z, a0.z);
                    a0.w = fmaf(w[j], x0[j].w, a0.w);
                    a1.x = fmaf(w[j], x1[j].x, a1.x);
                    a1.y = fmaf(w[j], x1[j].y, a1.y);
                    a1.z = fmaf(w[j], x1[j].z, a1.z);
                    a1.w = fmaf(w[j], x1[j].w, a1.w);
                }
            }
        }
    }
    *reinterpret_cast<uint4 *>(o_out + col0) = make_uint4(pack_bf16x2(a0.x, a0.y), pack_bf16x2(a0.z, a0.w),
                                                          pack_bf16x2(a1.x, a1.y), pack_bf16x2(a1.z, a1.w));
    if (write_lse) *lse_out = L;
}

// block kCombineThreads, one wave of blocks: each takes (query, 4-head group) units in turn and
// merges the queries that were split into more than one item (64 threads per head row, 8
// columns each).  When the plan split nothing, every block returns after one read of the plan
// header.
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const PlanHeader *__restrict__ hdr, const BtInfo *__restrict__ info, const float *__restrict__ part_o,
               const float *__restrict__ part_lse, __nv_bfloat16 *__restrict__ o_lat, float *__restrict__ lse) {
    grid_launch_dependents();  // a following call's plan kernel may get resident; it waits for us
    grid_dependency_wait();    // launched as a programmatic dependent of the decode kernel
    if (hdr->n_split == 0) return;
    const int n_units = hdr->n_bt * (kHeads / kCombineHeads);
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int bt = u / (kHeads / kCombineHeads);
        const BtInfo in = info[bt];
        if (in.splits <= 1) continue;
        const int h = (u % (kHeads / kCombineHeads)) * kCombineHeads + (threadIdx.x >> 6);
        const int col0 = (threadIdx.x & 63) * 8;
        combine_row(part_o + ((size_t)in.slot_base * kHeads + h) * kDc, (size_t)kHeads * kDc,
                    part_lse + (size_t)in.slot_base * kHeads + h, kHeads, in.splits, col0,
                    o_lat + ((size_t)bt * kHeads + h) * kDc, lse + (size_t)bt * kHeads + h, (threadIdx.x & 63) == 0);
    }
}

// grid ceil(rows / kCombineHeads), block kCombineThreads: dense parts [n_parts, rows, 512]
__global__ void __launch_bounds__(kCombineThreads)
combine_rows_kernel(const float *__restrict__ o_parts, const float *__restrict__ lse_parts, int n_parts, int rows,
                    __nv_bfloat16 *__restrict__ o_out, float *__restrict__ lse_out) {
    const int row = blockIdx.x * kCombineHeads + (threadIdx.x >> 6);
    if (row >= rows) return;
    const int col0 = (threadIdx.x & 63) * 8;
    combine_row(o_parts + (size_t)row * kDc, (size_t)rows * kDc, lse_parts + row, (size_t)rows, n_parts, col0,
                o_out + (size_t)row * kDc, lse_out + row, (threadIdx.x & 63) == 0);
}

}  // namespace mla
