// decode_kernels.cuh - split-KV MLA decode over a paged 576-wide latent cache.
//
// Method ("DeepSeek-V2" explainer, Steps 6-8): every head scores the absorbed
// query against the shared latent rows, s_j = scale * q_abs . [c_j | k^R_j]
// (content and RoPE channels add inside the softmax, Step 7), and the output
// stays in latent space, o = sum_j softmax(s)_j c_j (W^UV is applied later).
//
// B300 design: one cluster of two CTAs (two SMs) per work item.
//   CTA rank 0, the "score" CTA: holds the 128x576 absorbed query of the item in
//     tensor memory (A operand, 288 columns), streams the 64-token pages with TMA
//     (9 boxes of 64 tokens x 64 columns, 128-byte swizzle), computes
//     S = Q K^T (M = 128 heads, N = 64 tokens, K = 576) with tcgen05 into a
//     double-buffered TMEM tile, runs the online softmax (one thread per head,
//     lazy rescaling), and ships P (bf16, 128 x 64) plus per-head rescale factors
//     to its partner with a shared->cluster bulk copy.
//   CTA rank 1, the "accumulate" CTA: holds O = 128 heads x 512 latent fp32, i.e.
//     all 512 TMEM columns, streams the same pages' 512 latent columns, and runs
//     O += P V (M = 128, N = 256 x 2, K = 64) with tcgen05; its four epilogue
//     warps rescale O when the partner asks, and write the normalised output.
// The split keeps both 256 KB accumulators on chip without recomputing S: O alone
// fills a whole SM's tensor memory, and the query alone would fill most of its
// shared memory.
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
constexpr uint32_t kStageS = kBoxesS * kBoxBytes;  // 73728: one whole page
constexpr uint32_t kStageV = kBoxesV * kBoxBytes;  // 65536: a page's latent columns
constexpr int kStages = 2;           // page stages per CTA
constexpr int kPBufs = 4;            // P messages in flight between the two CTAs
constexpr int kPBytes = kHeads * kPage * 2;  // 16 KB of bf16 probabilities
constexpr int kMetaBytes = 1040;     // alpha[128] f32, inv_l[128] f32, flags, valid, pad
constexpr int kMetaStride = 1088;
constexpr float kTau = 8.0f;         // lazy rescale threshold, log2 units (factor 256)

// TMEM columns
constexpr uint32_t kTmemS = 0;       // score CTA: S buffers at 0 and 64
constexpr uint32_t kTmemQ = 128;     // score CTA: Q (bf16 pairs) at 128 .. 415
constexpr uint32_t kTmemCols = 512;

// Shared memory (offsets from a 1024-aligned base).  The message area and the barriers sit
// at the same offsets in both CTAs (the partner addresses them remotely); the page stages
// follow, 72 KB each in the score CTA and 64 KB each in the accumulate CTA.
constexpr uint32_t kOffP = 0;                                       // kPBufs x 16 KB
constexpr uint32_t kOffMeta = kOffP + kPBufs * kPBytes;             // kPBufs x 1088
constexpr uint32_t kOffEvt = kOffMeta + kPBufs * kMetaStride;       // alpha[128], inv_l[128], type
constexpr uint32_t kOffBar = kOffEvt + 1040;
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kBarFull + kStages;
constexpr int kBarSFull = kBarEmpty + kStages;
constexpr int kBarSEmpty = kBarSFull + 2;
constexpr int kBarQReady = kBarSEmpty + 2;
constexpr int kBarPFree = kBarQReady + 1;
constexpr int kBarPFull = kBarPFree + kPBufs;
constexpr int kBarPStaged = kBarPFull + kPBufs;
constexpr int kBarMmaEvt = kBarPStaged + kPBufs;
constexpr int kBarCorrEvt = kBarMmaEvt + 1;
constexpr int kNumBars = kBarCorrEvt + 1;
constexpr uint32_t kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kOffAny = kOffAbort + 4;  // kPBufs words: OR of the rescale requests per message
constexpr uint32_t kOffStages = (kOffAny + 4 * kPBufs + 1023u) & ~1023u;
constexpr uint32_t kDecodeSmem = kOffStages + kStages * kStageS + 1024;  // + slack to align the base

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, 0, 0);    // A = Q (TMEM), B = K tile, K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);  // A = P K-major, B = V MN-major

constexpr uint32_t kFlagFirst = 1u, kFlagRescale = 2u, kFlagLast = 4u;
constexpr uint32_t kEvtRescale = 1u, kEvtEpilogue = 2u;

// One unit of work: tiles [tb, te) of query (b, t) where bt = b * Tq + t.
// slot < 0: the item covers the whole query and writes the final output;
// slot >= 0: it writes a partial (o / l in fp32, lse) into workspace slot `slot`.
struct Item {
    int bt, tb, te, slot;
};
struct PlanHeader {
    int n_items;
    int n_bt;
    int max_items;
    int max_slots;
    int pad[60];
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
    const Item *items;
    float *part_o;                // [slots, 128, 512]
    float *part_lse;              // [slots, 128]
    int B, Tq, causal, num_pages, max_pages;
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
    Item it = p.items[i];
    ItemInfo x;
    x.bt = it.bt;
    x.b = it.bt / p.Tq;
    int t = it.bt - x.b * p.Tq;
    x.tb = it.tb;
    x.te = it.te;
    x.slot = it.slot;
    int L = p.seq_lens[x.b];
    L = L < 0 ? 0 : (L > p.max_pages * kPage ? p.max_pages * kPage : L);
    x.n_vis = visible_tokens(L, p.Tq, t, p.causal);
    return x;
}

// Static "snake" schedule over the plan's items (sorted longest first):
// round r gives item r*C + k to cluster k on even rounds and r*C + C-1-k on odd ones.
__device__ __forceinline__ int schedule(int r, int cid, int ncl) {
    return r * ncl + ((r & 1) ? (ncl - 1 - cid) : cid);
}

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

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, int B, int Tq, int causal, int max_pages,
            int n_clusters, int num_splits, PlanHeader *hdr, Item *items, BtInfo *info,
            int max_items, int max_slots) {
    __shared__ int s_tmp[32];
    __shared__ int s_key[kPlanThreads];
    __shared__ int s_ord[kPlanThreads];
    const int tid = threadIdx.x;
    const int n_bt = B * Tq;
    const int per = (n_bt + kPlanThreads - 1) / kPlanThreads;

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
        info[bt].tiles = T;
        w_local += T;
    }
    int W_total;
    block_excl_scan(w_local, s_tmp, &W_total);
    const long long W = W_total;

    // 2. split counts
    for (int bt = tid * per; bt < min(n_bt, (tid + 1) * per); ++bt) {
        int T = info[bt].tiles;
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
        info[bt].splits = s;
    }
    __syncthreads();

    // 3. order: longest chunk first (rank sort when it fits one element per thread)
    const bool sorted = n_bt <= kPlanThreads;
    if (sorted) {
        int key = -1;
        if (tid < n_bt) {
            int T = info[tid].tiles, s = info[tid].splits;
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
        items_local += info[bt].splits;
        slots_local += info[k].splits > 1 ? info[k].splits : 0;
    }
    int n_items, n_slots;
    int item_off = block_excl_scan(items_local, s_tmp, &n_items);
    int slot_off = block_excl_scan(slots_local, s_tmp, &n_slots);
    const bool overflow = n_items > max_items || n_slots > max_slots;
    for (int k = tid * per; k < min(n_bt, (tid + 1) * per); ++k) {
        int bt = sorted ? s_ord[k] : k;
        info[bt].item_off = item_off;
        item_off += info[bt].splits;
        int s2 = info[k].splits;
        info[k].slot_base = s2 > 1 ? slot_off : -1;
        slot_off += s2 > 1 ? s2 : 0;
    }
    __syncthreads();

    // 5. items (on overflow nothing is scheduled and nothing is combined)
    if (overflow) {
        for (int bt = tid * per; bt < min(n_bt, (tid + 1) * per); ++bt) info[bt].splits = 0;
    } else {
        for (int bt = tid * per; bt < min(n_bt, (tid + 1) * per); ++bt) {
            BtInfo in = info[bt];
            for (int j = 0; j < in.splits; ++j) {
                Item it;
                it.bt = bt;
                it.tb = (int)(((long long)in.tiles * j) / in.splits);
                it.te = (int)(((long long)in.tiles * (j + 1)) / in.splits);
                it.slot = in.splits > 1 ? in.slot_base + j : -1;
                items[in.item_off + j] = it;
            }
        }
    }
    if (tid == 0) {
        if (overflow) raise_status(0x8u);
        hdr->n_items = overflow ? 0 : n_items;
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
    __device__ __forceinline__ uint32_t stage(uint32_t s, uint32_t bytes) const { return base + kOffStages + s * bytes; }
    __device__ __forceinline__ uint32_t pbuf(uint32_t j) const { return base + kOffP + j * kPBytes; }
    __device__ __forceinline__ uint32_t meta(uint32_t j) const { return base + kOffMeta + j * kMetaStride; }
    __device__ __forceinline__ uint32_t evt() const { return base + kOffEvt; }
};

__device__ __forceinline__ void tma_load_3d(uint32_t smem_dst, const void *tmap, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Producer: one TMA per page.  The tensor map views the pool as (64 columns, rows, column
// blocks) with strides (2 B, 1152 B, 128 B), so a single box lands in shared memory as
// `blocks` consecutive 64-row x 128-byte swizzled blocks -- the operand layout of the MMAs.
__device__ __forceinline__ void role_producer(const DecodeParams &p, const CUtensorMap *tmap, const Smem &sm,
                                              uint32_t stage_bytes, int cid, int ncl, int n_items,
                                              volatile int *abort) {
    uint32_t g = 0;
    for (int r = 0;; ++r) {
        int i = schedule(r, cid, ncl);
        if (i >= n_items) break;
        ItemInfo it = load_item(p, i);
        for (int tile = it.tb; tile < it.te; ++tile, ++g) {
            int pg = p.block_table[(size_t)it.b * p.max_pages + tile];
            if (pg < 0 || pg >= p.num_pages) {
                raise_status(0x1u);
                pg = 0;
            }
            const uint32_t s = g % kStages;
            if (!mbar_wait(sm.bar(kBarEmpty + s), ((g / kStages) & 1u) ^ 1u, abort)) return;
            mbar_arrive_expect_tx(sm.bar(kBarFull + s), stage_bytes);
            tma_load_3d(sm.stage(s, stage_bytes), tmap, 0, pg * kPage, 0, sm.bar(kBarFull + s));
        }
    }
    // let every load issued land before the CTA can retire (bounded)
    for (uint32_t k = (g > kStages ? g - kStages : 0); k < g; ++k)
        if (!mbar_wait(sm.bar(kBarFull + k % kStages), (k / kStages) & 1u, abort)) return;
}

// Score CTA, MMA issuer (one thread): S_j = Q . K_tile^T, K = 576 in 36 steps.
__device__ __forceinline__ void role_score_mma(const DecodeParams &p, const Smem &sm, uint32_t tmem, int cid,
                                               int ncl, int n_items, volatile int *abort) {
    uint32_t g = 0, ic = 0;
    for (int r = 0;; ++r) {
        int i = schedule(r, cid, ncl);
        if (i >= n_items) break;
        ItemInfo it = load_item(p, i);
        if (it.te <= it.tb) continue;
        if (!mbar_wait(sm.bar(kBarQReady), ic & 1u, abort)) return;
        tc_fence_after();
        ++ic;
        for (int tile = it.tb; tile < it.te; ++tile, ++g) {
            const uint32_t j = g & 1u, s = g % kStages;
            if (!mbar_wait(sm.bar(kBarSEmpty + j), ((g >> 1) & 1u) ^ 1u, abort)) return;
            if (!mbar_wait(sm.bar(kBarFull + s), (g / kStages) & 1u, abort)) return;
            tc_fence_after();
            const uint32_t d = tmem + kTmemS + j * 64u;
            const uint32_t kb = sm.stage(s, kStageS);
#pragma unroll 1
            for (int bx = 0; bx < kBoxesS; ++bx) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint64_t bdesc = sdesc_sw128(kb + bx * kBoxBytes + 32u * k, 16u, 1024u);
                    mma_ts(d, tmem + kTmemQ + bx * 32u + k * 8u, bdesc, kIdescS, (bx | k) != 0);
                }
            }
            mma_commit(sm.bar(kBarEmpty + s));
            mma_commit(sm.bar(kBarSFull + j));
        }
    }
}

// Score CTA, softmax warps (thread = head).
__device__ __forceinline__ void role_softmax(const DecodeParams &p, const Smem &sm, uint32_t tmem, int cid,
                                             int ncl, int n_items, volatile int *abort,
                                             volatile uint32_t *any_words) {
    const int h = threadIdx.x;  // 0..127
    const uint32_t lane_off = (uint32_t)((threadIdx.x >> 5) * 32) << 16;
    const float sl2 = p.sl2;
    uint32_t sc = 0;
    for (int r = 0;; ++r) {
        int i = schedule(r, cid, ncl);
        if (i >= n_items) break;
        ItemInfo it = load_item(p, i);
        if (it.te <= it.tb) {
            p.lse[(size_t)it.bt * kHeads + h] = -INFINITY;
            continue;
        }
        // absorbed query of this head -> TMEM lane h (bf16 pairs, 288 columns)
        {
            const uint4 *q = reinterpret_cast<const uint4 *>(p.q_abs + ((size_t)it.bt * kHeads + h) * kD);
#pragma unroll 1
            for (int c = 0; c < kBoxesS; ++c) {
                uint32_t v[32];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    uint4 x = __ldg(q + c * 8 + u);
                    v[4 * u + 0] = x.x;
                    v[4 * u + 1] = x.y;
                    v[4 * u + 2] = x.z;
                    v[4 * u + 3] = x.w;
                }
                tmem_st32(tmem + lane_off + kTmemQ + c * 32u, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(sm.bar(kBarQReady));
        }
        float m = 0.f, l = 0.f;
        for (int tile = it.tb; tile < it.te; ++tile, ++sc) {
            const uint32_t j = sc & 1u;
            if (!mbar_wait(sm.bar(kBarSFull + j), (sc >> 1) & 1u, abort)) return;
            tc_fence_after();
            uint32_t sr[64];
            {
                uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
                uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
                tmem_ld32(tmem + lane_off + kTmemS + j * 64u, a);
                tmem_ld32(tmem + lane_off + kTmemS + j * 64u + 32u, b);
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(sm.bar(kBarSEmpty + j));

            const int valid = min(kPage, it.n_vis - tile * kPage);
            float s[64];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float v = c < valid ? __uint_as_float(sr[c]) : -INFINITY;
                s[c] = v;
                mx = fmaxf(mx, v);
            }
            mx *= sl2;
            const bool first = tile == it.tb;
            const bool last = tile == it.te - 1;
            bool resc = false;
            float alpha = 1.f;
            if (first) {
                m = mx;
            } else if (mx > m + kTau) {
                alpha = ex2_approx(m - mx);
                l *= alpha;
                m = mx;
                resc = true;
            }
            uint32_t pk[32];
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float a = ex2_approx(fmaf(s[2 * c], sl2, -m));
                float b = ex2_approx(fmaf(s[2 * c + 1], sl2, -m));
                pk[c] = pack_bf16x2(a, b);
                lsum += a + b;  // the row sum uses the unrounded probabilities (exact lse)
            }
            l += lsum;

            // ship P, alpha (and 1/l on the last tile) to the accumulate CTA
            const uint32_t jp = sc % kPBufs, use = sc / kPBufs;
            if (!mbar_wait<true>(sm.bar(kBarPFree + jp), (use & 1u) ^ 1u, abort)) return;
            {
                const uint32_t row = sm.pbuf(jp) + (uint32_t)(h >> 3) * 1024u + (uint32_t)(h & 7) * 128u;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t addr = row + (uint32_t)((c ^ (h & 7)) * 16);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c]),
                                 "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                                 : "memory");
                }
                const uint32_t mt = sm.meta(jp);
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(mt + 4u * h), "f"(alpha) : "memory");
                if (last)
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(mt + 512u + 4u * h), "f"(1.0f / l) : "memory");
            }
            if (resc) atomicOr(const_cast<unsigned int *>(any_words + jp), 1u);
            fence_proxy_async_smem();
            mbar_arrive(sm.bar(kBarPStaged + jp));
            if (h == 0) {
                // all 128 rows staged: send the message (bounded wait, no hardware barrier)
                if (!mbar_wait(sm.bar(kBarPStaged + jp), use & 1u, abort)) return;
                const uint32_t any = any_words[jp];
                any_words[jp] = 0u;
                const uint32_t flags = (first ? kFlagFirst : 0u) | (any ? kFlagRescale : 0u) | (last ? kFlagLast : 0u);
                const uint32_t mt = sm.meta(jp);
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(mt + 1024u), "r"(flags), "r"((uint32_t)valid)
                             : "memory");
                fence_proxy_async_smem();
                const uint32_t peer_full = mapa_shared(sm.bar(kBarPFull + jp), 1);
                bulk_copy_s2c(mapa_shared(sm.pbuf(jp), 1), sm.pbuf(jp), kPBytes, peer_full);
                bulk_copy_s2c(mapa_shared(mt, 1), mt, kMetaBytes, peer_full);
            }
        }
        const float lse = (m + __log2f(l)) * 0.69314718055994531f;
        if (it.slot < 0)
            p.lse[(size_t)it.bt * kHeads + h] = lse;
        else
            p.part_lse[(size_t)it.slot * kHeads + h] = lse;
    }
}

// Accumulate CTA, MMA warp: O += P V, two N = 256 halves, K = 64 in 4 steps.  It also
// hands rescale and epilogue events to the epilogue warps through the local event buffer:
// the event data is written, then the event barrier gets two arrivals -- this warp's
// (release: the data is visible) and the MMA commit (all earlier MMAs have completed).
__device__ __forceinline__ void role_accum_mma(const DecodeParams &p, const Smem &sm, uint32_t tmem, int cid,
                                               int ncl, int n_items, volatile int *abort) {
    const int lane = threadIdx.x & 31;
    uint32_t g = 0, cv = 0;
    bool pending_epilogue = false;
    const uint32_t evt = sm.evt();
    for (int r = 0;; ++r) {
        int i = schedule(r, cid, ncl);
        if (i >= n_items) break;
        ItemInfo it = load_item(p, i);
        for (int tile = it.tb; tile < it.te; ++tile, ++g) {
            const uint32_t jp = g % kPBufs, use = g / kPBufs, s = g % kStages;
            if (lane == 0) mbar_arrive_expect_tx(sm.bar(kBarPFull + jp), kPBytes + kMetaBytes);
            __syncwarp();
            if (!mbar_wait<true>(sm.bar(kBarPFull + jp), use & 1u, abort)) return;
            const uint32_t mt = sm.meta(jp);
            uint32_t flags, valid;
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(flags), "=r"(valid) : "r"(mt + 1024u) : "memory");
            const bool first = flags & kFlagFirst, last = flags & kFlagLast;
            if (first) {
                if (pending_epilogue) {  // the previous item's O must have been read out
                    if (!mbar_wait(sm.bar(kBarCorrEvt), cv & 1u, abort)) return;
                    ++cv;
                    pending_epilogue = false;
                }
            } else if (flags & kFlagRescale) {
                // rescale event: per-head factors to the event buffer, then wait for the rows
                asm volatile("{\n\t.reg .b32 x, y, z, w;\n\t"
                             "ld.shared.v4.b32 {x, y, z, w}, [%0];\n\t"
                             "st.shared.v4.b32 [%1], {x, y, z, w};\n\t}" ::"r"(mt + 16u * lane),
                             "r"(evt + 16u * lane)
                             : "memory");
                __syncwarp();
                if (lane == 0) {
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(evt + 1024u), "r"(kEvtRescale) : "memory");
                    mbar_arrive(sm.bar(kBarMmaEvt));
                    mma_commit(sm.bar(kBarMmaEvt));
                }
                __syncwarp();
                if (!mbar_wait(sm.bar(kBarCorrEvt), cv & 1u, abort)) return;
                ++cv;
            }
            if (!mbar_wait(sm.bar(kBarFull + s), (g / kStages) & 1u, abort)) return;
            const uint32_t vb = sm.stage(s, kStageV);
            if (last && valid < (uint32_t)kPage) {
                // rows past the end of the sequence may hold anything (even NaN): zero them,
                // since 0 * NaN would poison O even though their probabilities are 0
                const uint32_t nrow = kPage - valid;
                for (uint32_t e = lane; e < nrow * 8u * kBoxesV; e += 32) {
                    uint32_t bx = e / (nrow * 8u), rem = e % (nrow * 8u);
                    uint32_t row = valid + rem / 8u, ch = rem % 8u;
                    uint32_t addr = vb + bx * kBoxBytes + row * 128u + ch * 16u;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int n = 0; n < 2; ++n) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint64_t adesc = sdesc_sw128(sm.pbuf(jp) + 32u * k, 16u, 1024u);
                        uint64_t bdesc = sdesc_sw128(vb + 4u * n * kBoxBytes + 2048u * k, (uint32_t)kBoxBytes, 1024u);
                        mma_ss(tmem + 256u * n, adesc, bdesc, kIdescPV, !(first && k == 0));
                    }
                }
                mma_commit(sm.bar(kBarEmpty + s));
            }
            if (last) {
                // epilogue event: 1/l per head to the event buffer
                asm volatile("{\n\t.reg .b32 x, y, z, w;\n\t"
                             "ld.shared.v4.b32 {x, y, z, w}, [%0];\n\t"
                             "st.shared.v4.b32 [%1], {x, y, z, w};\n\t}" ::"r"(mt + 512u + 16u * lane),
                             "r"(evt + 512u + 16u * lane)
                             : "memory");
            }
            __syncwarp();
            if (lane == 0) {
                mma_commit_mc(sm.bar(kBarPFree + jp), (uint16_t)0x1);  // message consumed (meta read above)
                if (last) {
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(evt + 1024u), "r"(kEvtEpilogue) : "memory");
                    mbar_arrive(sm.bar(kBarMmaEvt));
                    mma_commit(sm.bar(kBarMmaEvt));
                }
            }
            __syncwarp();
            if (last) pending_epilogue = true;
        }
    }
    if (pending_epilogue) mbar_wait(sm.bar(kBarCorrEvt), cv & 1u, abort);
}

// Accumulate CTA, epilogue warps (thread = head): serve events -- rescale O rows, or
// write the normalised output of the finished item.
__device__ __forceinline__ void role_accum_epilogue(const DecodeParams &p, const Smem &sm, uint32_t tmem,
                                                    int cid, int ncl, int n_items, volatile int *abort) {
    const int h = threadIdx.x;  // 0..127
    const uint32_t lane_off = (uint32_t)((threadIdx.x >> 5) * 32) << 16;
    const uint32_t evt = sm.evt();
    uint32_t ev = 0;
    for (int r = 0;; ++r) {
        int i = schedule(r, cid, ncl);
        if (i >= n_items) break;
        ItemInfo it = load_item(p, i);
        if (it.te <= it.tb) {
            uint4 *o = reinterpret_cast<uint4 *>(p.o_lat + ((size_t)it.bt * kHeads + h) * kDc);
            for (int c = 0; c < kDc * 2 / 16; ++c) o[c] = make_uint4(0, 0, 0, 0);
            continue;
        }
        for (;;) {
            if (!mbar_wait(sm.bar(kBarMmaEvt), ev & 1u, abort)) return;
            ++ev;
            tc_fence_after();
            uint32_t type;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(type) : "r"(evt + 1024u) : "memory");
            if (type == kEvtRescale) {
                float alpha;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(alpha) : "r"(evt + 4u * h) : "memory");
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < kDc / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_off + c * 32u, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(tmem + lane_off + c * 32u, v);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(sm.bar(kBarCorrEvt));
                continue;
            }
            float inv_l;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(inv_l) : "r"(evt + 512u + 4u * h) : "memory");
#pragma unroll 1
            for (int c = 0; c < kDc / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + c * 32u, v);
                tmem_ld_wait();
                if (it.slot < 0) {
                    uint4 *o = reinterpret_cast<uint4 *>(p.o_lat + ((size_t)it.bt * kHeads + h) * kDc + c * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]) * inv_l, __uint_as_float(v[8 * u + 1]) * inv_l);
                        w.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]) * inv_l, __uint_as_float(v[8 * u + 3]) * inv_l);
                        w.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]) * inv_l, __uint_as_float(v[8 * u + 5]) * inv_l);
                        w.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]) * inv_l, __uint_as_float(v[8 * u + 7]) * inv_l);
                        o[u] = w;
                    }
                } else {
                    float4 *o = reinterpret_cast<float4 *>(p.part_o + ((size_t)it.slot * kHeads + h) * kDc + c * 32);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        o[u] = make_float4(__uint_as_float(v[4 * u + 0]) * inv_l, __uint_as_float(v[4 * u + 1]) * inv_l,
                                           __uint_as_float(v[4 * u + 2]) * inv_l, __uint_as_float(v[4 * u + 3]) * inv_l);
                }
            }
            tc_fence_before();
            mbar_arrive(sm.bar(kBarCorrEvt));
            break;
        }
    }
}

// Launched with a cluster dimension of 2 (rank 0 scores, rank 1 accumulates).
__global__ void __launch_bounds__(192, 1)
decode_kernel(const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_v,
              const DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x(), ncl = (int)nclusters_x();
    uint8_t *const gbase = smem_raw + (sm.base - raw);
    volatile int *abort = reinterpret_cast<volatile int *>(gbase + kOffAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffTmemPtr);
    volatile uint32_t *any_words = reinterpret_cast<volatile uint32_t *>(gbase + kOffAny);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(sm.bar(kBarFull + s), 1);
            mbar_init(sm.bar(kBarEmpty + s), 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(sm.bar(kBarSFull + j), 1);
            mbar_init(sm.bar(kBarSEmpty + j), 128);
        }
        for (int j = 0; j < kPBufs; ++j) {
            mbar_init(sm.bar(kBarPFree + j), 1);     // score CTA: the partner's MMA commit
            mbar_init(sm.bar(kBarPFull + j), 1);     // accumulate CTA: armed by its MMA warp
            mbar_init(sm.bar(kBarPStaged + j), 128); // score CTA: all rows written
            any_words[j] = 0u;
        }
        mbar_init(sm.bar(kBarQReady), 128);
        mbar_init(sm.bar(kBarMmaEvt), 2);            // MMA warp arrive + MMA commit
        mbar_init(sm.bar(kBarCorrEvt), 128);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(sm.base + kOffTmemPtr, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && (threadIdx.x & 31) == 0) tma_prefetch_desc(rank == 0 ? &tmap_s : &tmap_v);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the partner's barriers exist before any remote arrive or copy
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_items = p.hdr->n_items;

    if (warp == 4) {
        if ((threadIdx.x & 31) == 0) {
            if (rank == 0)
                role_producer(p, &tmap_s, sm, kStageS, cid, ncl, n_items, abort);
            else
                role_producer(p, &tmap_v, sm, kStageV, cid, ncl, n_items, abort);
        }
    } else if (warp == 5) {
        if (rank == 0) {
            if ((threadIdx.x & 31) == 0) role_score_mma(p, sm, tmem, cid, ncl, n_items, abort);
        } else {
            role_accum_mma(p, sm, tmem, cid, ncl, n_items, abort);
        }
    } else {
        if (rank == 0)
            role_softmax(p, sm, tmem, cid, ncl, n_items, abort, any_words);
        else
            role_accum_epilogue(p, sm, tmem, cid, ncl, n_items, abort);
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA retires while its partner may still write into it
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// LSE combine: merge the partials of queries that were split.
// ---------------------------------------------------------------------------
// thread block = 8 heads x 16 threads, each thread 32 latent columns
__device__ __forceinline__ void combine_row(const float *o_base, size_t o_stride, const float *lse_base,
                                            size_t lse_stride, int n_parts, int col0, __nv_bfloat16 *o_out,
                                            float *lse_out, bool write_lse) {
    float mx = -INFINITY;
    for (int r = 0; r < n_parts; ++r) mx = fmaxf(mx, lse_base[r * lse_stride]);
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    float L = -INFINITY;
    if (mx != -INFINITY) {
        float tot = 0.f;
        for (int r = 0; r < n_parts; ++r) tot += expf(lse_base[r * lse_stride] - mx);
        L = mx + logf(tot);
        for (int r = 0; r < n_parts; ++r) {
            const float w = expf(lse_base[r * lse_stride] - L);
            if (w == 0.f) continue;
            const float4 *src = reinterpret_cast<const float4 *>(o_base + r * o_stride + col0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float4 x = src[u];
                acc[4 * u + 0] = fmaf(w, x.x, acc[4 * u + 0]);
                acc[4 * u + 1] = fmaf(w, x.y, acc[4 * u + 1]);
                acc[4 * u + 2] = fmaf(w, x.z, acc[4 * u + 2]);
                acc[4 * u + 3] = fmaf(w, x.w, acc[4 * u + 3]);
            }
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(o_out + col0);
#pragma unroll
    for (int u = 0; u < 4; ++u)
        dst[u] = make_uint4(pack_bf16x2(acc[8 * u + 0], acc[8 * u + 1]), pack_bf16x2(acc[8 * u + 2], acc[8 * u + 3]),
                            pack_bf16x2(acc[8 * u + 4], acc[8 * u + 5]), pack_bf16x2(acc[8 * u + 6], acc[8 * u + 7]));
    if (write_lse) *lse_out = L;
}

// grid (n_bt, 16), block 128: queries that were split into more than one item
__global__ void __launch_bounds__(128)
combine_kernel(const BtInfo *__restrict__ info, const float *__restrict__ part_o,
               const float *__restrict__ part_lse, __nv_bfloat16 *__restrict__ o_lat, float *__restrict__ lse) {
    const int bt = blockIdx.x;
    const BtInfo in = info[bt];
    if (in.splits <= 1) return;
    const int h = blockIdx.y * 8 + (threadIdx.x >> 4);
    const int col0 = (threadIdx.x & 15) * 32;
    combine_row(part_o + ((size_t)in.slot_base * kHeads + h) * kDc, (size_t)kHeads * kDc,
                part_lse + (size_t)in.slot_base * kHeads + h, kHeads, in.splits, col0,
                o_lat + ((size_t)bt * kHeads + h) * kDc, lse + (size_t)bt * kHeads + h, (threadIdx.x & 15) == 0);
}

// grid ceil(rows / 8), block 128: dense parts [n_parts, rows, 512]
__global__ void __launch_bounds__(128)
combine_rows_kernel(const float *__restrict__ o_parts, const float *__restrict__ lse_parts, int n_parts, int rows,
                    __nv_bfloat16 *__restrict__ o_out, float *__restrict__ lse_out) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 4);
    if (row >= rows) return;
    const int col0 = (threadIdx.x & 15) * 32;
    combine_row(o_parts + (size_t)row * kDc, (size_t)rows * kDc, lse_parts + row, (size_t)rows, n_parts, col0,
                o_out + (size_t)row * kDc, lse_out + row, (threadIdx.x & 15) == 0);
}

}  // namespace mla
