// sparse_kernels.cuh - the indexer's decode path (the DeepSeek page, "KV cache data movement
// minimization"): every cached token also keeps a small index vector; a decoding token scores
// all of them with one dot product each, keeps the k best, and attends over those tokens only.
//
//   index_score_kernel   s[b, t] = q_idx[b] . k_idx(b, t) for every cached token t < L_b: a
//                        stream over the paged index cache (d_idx bf16 per token, or d_idx E4M3
//                        codes and one fp32 scale per token), fp32 sums.  It moves d_idx * 2 (or
//                        d_idx + 4) bytes per token and does d_idx multiply-adds, so it runs at
//                        HBM speed: consecutive lanes read consecutive 16-byte pieces of the same
//                        page, eight loads in flight per lane.
//   topk_gather_kernel   the k largest scores of each sequence (ties: the lower index; NaN
//                        below every number), by a radix select over the scores' order-keeping
//                        32-bit keys, one byte per pass, on a cluster of CTAs that each own a
//                        contiguous slice of the sequence and add their 256-bin histograms
//                        through distributed shared memory; after the second pass each warp
//                        keeps the few positions that can still be picked in an ordered list, and
//                        the later passes and the compaction read only those.  The same kernel
//                        writes the selected
//                        positions in ascending order and copies the selected cache rows into a
//                        compact page pool, which the dense decode then walks (its lengths and an
//                        identity block table included): the gather costs k rows of traffic,
//                        against L_b rows of index vectors read to find them.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cstdint>

#include "decode_kernels.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kSparsePage = 64;          // tokens per page (index cache and latent cache alike)
constexpr int kSparseRow = 576;          // latent cache row: c (512) | k^R (64)
constexpr int kScoreThreads = 256;
constexpr int kScoreUnroll = 8;          // 16-byte loads in flight per lane
constexpr int kTopkCluster = 8;          // CTAs per sequence (portable cluster size)
constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkBins = 256;           // one byte of the key per pass
constexpr int kTopkPickCap = 512;    // picks per CTA whose positions are kept in shared memory
constexpr int kTopkCandCap = 64;     // keys per CTA offered to the cluster after the second pass
constexpr int kTopkListCap = 128;    // positions per warp list (keys at or above the first pass's bin)

// Order-keeping key of an fp32 score: larger score, larger key.  -0 is +0 (they tie), every NaN
// maps to 0, below -inf's key (0x007FFFFF).
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// A 32-bit word of another CTA's shared memory (a shared::cluster address from mapa_shared).
__device__ __forceinline__ uint32_t topk_ld_cluster(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Sequence length check shared by both kernels: a length outside [0, cap] is recorded and clamped.
__device__ __forceinline__ int sparse_len(const int32_t *seq_lens, int b, int cap, bool report) {
    int L = seq_lens[b];
    if (L < 0 || L > cap) {
        if (report) raise_status(0x2u);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// ---------------------------------------------------------------------------------------------
// Index scores.  LPT = lanes per token = d_idx / 8 (bf16) or d_idx / 16 (E4M3): each lane holds
// the 8 or 16 query coordinates of its 16-byte piece of a token and reads those coordinates of
// 32 / LPT tokens per 512-byte warp load.  A CTA of 8 warps takes pages j = c * 8 + w (and every
// ctas_per_seq * 8 pages after) of sequence b = blockIdx.x / ctas_per_seq.
// ---------------------------------------------------------------------------------------------
struct ScoreParams {
    const __nv_bfloat16 *q_idx;     // [B, d_idx]
    const void *idx_pool;           // [num_pages, 64, d_idx] bf16, or E4M3 codes
    const float *idx_scale;         // [num_pages, 64]: per-token scales of E4M3 codes
    const int32_t *block_table;     // [B, max_pages]
    const int32_t *seq_lens;        // [B]
    float *scores;                  // [B, max_pages * 64]
    int num_pages, max_pages, ctas_per_seq;
};

// Two E4M3 codes (low byte first) as two floats; the conversion is exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(pair & 0xFFFFu), __NV_E4M3);
    return __half22float2(__half2(h));
}

// E4M3 = false: bf16 index vectors, 8 per 16-byte piece.  E4M3 = true: 16 codes per piece, and the
// token's dot product is multiplied by its scale.
template <int LPT, bool E4M3>
__global__ void __launch_bounds__(kScoreThreads) index_score_kernel(ScoreParams p) {
    constexpr int kPer = E4M3 ? 16 : 8;                // index coordinates per lane piece
    constexpr int kTokPerLoad = 32 / LPT;
    constexpr int kLoadsPerPage = kSparsePage / kTokPerLoad;
    constexpr int kU = kLoadsPerPage < kScoreUnroll ? kLoadsPerPage : kScoreUnroll;
    constexpr int kDIdx = LPT * kPer;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = blockIdx.x / p.ctas_per_seq, c = blockIdx.x % p.ctas_per_seq;
    const long long row_len = (long long)p.max_pages * kSparsePage;
    const int L = sparse_len(p.seq_lens, b, (int)row_len, c == 0 && threadIdx.x == 0);
    const int n_pages = (L + kSparsePage - 1) / kSparsePage;
    const int sub = lane % LPT, tok = lane / LPT;

    float q[kPer];
#pragma unroll
    for (int h = 0; h < kPer / 8; ++h) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p.q_idx + (size_t)b * kDIdx + sub * kPer + h * 8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[h * 8 + 2 * i] = bf16lo_to_f32(w[i]);
            q[h * 8 + 2 * i + 1] = bf16hi_to_f32(w[i]);
        }
    }
    float *out = p.scores + (size_t)b * row_len;
    const int stride = p.ctas_per_seq * (kScoreThreads / 32);
    for (int j = c * (kScoreThreads / 32) + warp; j < n_pages; j += stride) {
        const int pg = p.block_table[(size_t)b * p.max_pages + j];
        const int base = j * kSparsePage;
        if (pg < 0 || pg >= p.num_pages) {
            if (lane == 0) raise_status(0x1u);
            for (int i = lane; i < kSparsePage && base + i < L; i += 32) out[base + i] = __int_as_float(0x7FC00000);
            continue;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.idx_pool) +
                                                           (size_t)pg * kSparsePage * kDIdx * (E4M3 ? 1 : 2)) +
                           lane;
        // the page's 64 token scales, two per lane, loaded beside the codes
        float sc_lo = 1.f, sc_hi = 1.f;
        if constexpr (E4M3) {
            sc_lo = __ldg(p.idx_scale + (size_t)pg * kSparsePage + lane);
            sc_hi = __ldg(p.idx_scale + (size_t)pg * kSparsePage + 32 + lane);
        }
#pragma unroll
        for (int g = 0; g < kLoadsPerPage; g += kU) {
            uint4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) v[u] = __ldcs(src + (g + u) * 32);
            float s[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                float a = 0.f;
                if constexpr (E4M3) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f0 = e4m3x2_to_float2(w[i]), f1 = e4m3x2_to_float2(w[i] >> 16);
                        a = fmaf(q[4 * i], f0.x, a);
                        a = fmaf(q[4 * i + 1], f0.y, a);
                        a = fmaf(q[4 * i + 2], f1.x, a);
                        a = fmaf(q[4 * i + 3], f1.y, a);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a = fmaf(q[2 * i], bf16lo_to_f32(w[i]), a);
                        a = fmaf(q[2 * i + 1], bf16hi_to_f32(w[i]), a);
                    }
                }
                s[u] = a;
            }
#pragma unroll
            for (int off = LPT / 2; off > 0; off >>= 1) {
#pragma unroll
                for (int u = 0; u < kU; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
            }
            if constexpr (E4M3) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = (g + u) * kTokPerLoad + tok;  // token within the page
                    const float a = __shfl_sync(0xffffffffu, sc_lo, i & 31), b2 = __shfl_sync(0xffffffffu, sc_hi, i & 31);
                    s[u] *= i < 32 ? a : b2;
                }
            }
            if (sub == 0) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = (g + u) * kTokPerLoad + tok;  // token within the page
                    if (base + i < L) out[base + i] = s[u];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Top-k and gather.  Grid: batch * kTopkCluster CTAs in clusters of kTopkCluster, cluster b for
// sequence b; CTA r owns positions [r * chunk, min(L, (r + 1) * chunk)), chunk a multiple of 4.
// ---------------------------------------------------------------------------------------------
struct TopkParams {
    const float *scores;            // [B, max_pages * 64]
    const int32_t *seq_lens;        // [B]
    const __nv_bfloat16 *kv_pool;   // [num_pages, 64, 576]
    const int32_t *block_table;     // [B, max_pages]
    int32_t *sel_index;             // [B, k]: selected positions ascending, then -1
    __nv_bfloat16 *sel_pool;        // [B * npk, 64, 576]: sequence b's rows on pages b*npk ..
    int32_t *sel_block_table;       // [B, npk]: b * npk + j
    int32_t *sel_lens;              // [B]: min(k, L_b)
    int num_pages, max_pages, k, npk;
    int staged;                     // 1: each CTA first copies its slice's keys into shared memory
    // optional: the decode plan of the output (one whole item per sequence), in the decode
    // workspace, so the decode that follows needs no plan launch
    PlanHeader *plan_hdr;
    Item *plan_items;
    BtInfo *plan_info;
    int plan_max_items, plan_max_slots;
};

// Slice positions that fit the staged key copy (dynamic shared memory next to TopkSmem).
constexpr int kTopkStageKeys = 48 * 1024;
constexpr int kTopkSlicePages = kTopkStageKeys / kSparsePage + 2;  // block-table entries of a slice

struct TopkSmem {
    uint32_t hist[4][kTopkBins];    // this CTA's histogram of each pass (read by the whole cluster)
    uint32_t tot[kTopkBins];        // the cluster's sum, this pass
    uint32_t warp_sum[kTopkWarps];
    uint32_t warp_sum2[kTopkWarps];
    uint32_t rank_gt[kTopkCluster]; // every CTA's keys above the threshold key, and equal to it,
    uint32_t rank_eq[kTopkCluster]; //   from the histograms read during the passes
    uint32_t pick[2];               // the chosen bin, and the keys in bins above it
    int32_t slice_bt[kTopkSlicePages];  // block-table entries of the slice's pages
    int32_t wlist[kTopkWarps][kTopkListCap];  // each warp's positions whose key's top byte is at
                                              // least the first pass's chosen byte, in order
    uint32_t wlist_n[kTopkWarps];
    uint32_t list_overflow;
    uint32_t cand[kTopkCandCap];    // this CTA's keys that carry the second pass's 16-bit prefix
    uint32_t cand_n;
    uint32_t xoff[kTopkCluster + 1];  // every rank's candidate count, as offsets
    uint32_t all_key[kTopkCluster * kTopkCandCap];  // the cluster's candidates, rank by rank
    uint8_t all_rank[kTopkCluster * kTopkCandCap];
    int32_t pick_pos[kTopkPickCap]; // this CTA's first picks (positions), in output order
    int32_t src_row[kTopkPickCap];  // their pool rows (page * 64 + slot), -1 for a bad page
};

// The keys of positions e .. e+3 (e a multiple of 4, e < hi): from the staged copy, or straight
// from the scores.
__device__ __forceinline__ void topk_keys4(const uint32_t *staged_keys, const float *row, bool staged, int lo, int e,
                                           uint32_t (&k)[4]) {
    if (staged) {
        const uint4 v = *reinterpret_cast<const uint4 *>(staged_keys + (e - lo));
        k[0] = v.x, k[1] = v.y, k[2] = v.z, k[3] = v.w;
    } else {
        const float4 v = *reinterpret_cast<const float4 *>(row + e);
        k[0] = score_key(v.x), k[1] = score_key(v.y), k[2] = score_key(v.z), k[3] = score_key(v.w);
    }
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }

__global__ void __launch_bounds__(kTopkThreads) topk_gather_kernel(TopkParams p) {
    __shared__ TopkSmem sm;
    extern __shared__ __align__(16) uint32_t staged_keys[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t r = cluster_ctarank();
    const int b = blockIdx.x / kTopkCluster;
    const long long row_len = (long long)p.max_pages * kSparsePage;
    const int L = sparse_len(p.seq_lens, b, (int)row_len, r == 0 && tid == 0);
    const int sel_len = L < p.k ? L : p.k;
    const int chunk = (((L + kTopkCluster - 1) / kTopkCluster) + 3) & ~3;
    const int lo = min(L, (int)r * chunk), hi = min(L, lo + chunk);
    const float *row = p.scores + (size_t)b * row_len;
    const bool take_all = p.k >= L;
    const bool fits = p.staged != 0;                 // the slice fits the shared-memory copies
    const bool staged = fits && !take_all;
    const int page0 = lo / kSparsePage;
    // warp w's sub-slice [wlo, whi): a multiple of 128 positions, 4 consecutive ones per lane per step
    const int wspan = (((hi - lo) + kTopkWarps - 1) / kTopkWarps + 127) & ~127;
    const int wlo = min(hi, lo + warp * wspan), whi = min(hi, wlo + wspan);
    const uint32_t lt = (1u << lane) - 1u;
    Tracer tr;
    tr.at(0x8200);

    for (int i = tid; i < 4 * kTopkBins; i += kTopkThreads) (&sm.hist[0][0])[i] = 0u;
    if (tid < kTopkCluster) sm.rank_gt[tid] = sm.rank_eq[tid] = 0u;
    if (tid == 0) sm.list_overflow = 0u;
    if (fits && hi > lo)
        for (int j = tid; j <= (hi - 1) / kSparsePage - page0; j += kTopkThreads)
            sm.slice_bt[j] = p.block_table[(size_t)b * p.max_pages + page0 + j];
    __syncthreads();
    // Copy the slice's keys into shared memory once (every pass reads them again), eight 16-byte
    // loads in flight per thread, and count the first pass's histogram (the top byte) on the way.
    if (staged) {
        constexpr int kU = 8;
        for (int e0 = lo + 4 * tid; e0 < hi; e0 += 4 * kTopkThreads * kU) {
            float4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = e0 + 4 * kTopkThreads * u;
                if (e < hi) v[u] = *reinterpret_cast<const float4 *>(row + e);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = e0 + 4 * kTopkThreads * u;
                if (e < hi) {
                    const uint4 k4 = make_uint4(score_key(v[u].x), score_key(v[u].y), score_key(v[u].z),
                                                score_key(v[u].w));
                    *reinterpret_cast<uint4 *>(staged_keys + (e - lo)) = k4;
                    atomicAdd(&sm.hist[0][k4.x >> 24], 1u);
                    if (e + 1 < hi) atomicAdd(&sm.hist[0][k4.y >> 24], 1u);
                    if (e + 2 < hi) atomicAdd(&sm.hist[0][k4.z >> 24], 1u);
                    if (e + 3 < hi) atomicAdd(&sm.hist[0][k4.w >> 24], 1u);
                }
            }
        }
    }
    __syncthreads();
    tr.at(0x8201);

    // Radix select of the need-th largest key, one byte per pass from the top.  After pass p every
    // CTA also knows, for every rank q, how many of q's keys lie above the chosen prefix (bins
    // above the chosen one) and, after the last pass, equal to the threshold key: the histograms
    // it read carry them, so the output offsets need no exchange of their own.
    uint32_t prefix = 0, mask = 0, need = (uint32_t)p.k;  // need: keys still to take at the prefix
    if (!take_all) {
        // rank q's keys in the chosen bins' upper neighbours so far (this thread's bin only); added
        // over the block once, after the last pass
        uint32_t acc_gt[kTopkCluster], acc_eq[kTopkCluster];
#pragma unroll
        for (int q = 0; q < kTopkCluster; ++q) acc_gt[q] = acc_eq[q] = 0u;
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            if (pass == 1 && staged) {
                // Scan the keys once more and keep, per warp and in position order, every position
                // whose top byte is at least the first pass's chosen one: the keys that can still
                // be picked (typically a few percent).  The later passes and the compaction read
                // only these lists, unless one overflowed.
                const uint32_t v0 = prefix >> 24;
                uint32_t n = 0;
                for (int e0 = wlo; e0 < whi; e0 += 128) {
                    const int e = e0 + 4 * lane;
                    uint32_t k4[4] = {0u, 0u, 0u, 0u};
                    if (e < whi) topk_keys4(staged_keys, row, true, lo, e, k4);
                    uint32_t in_bits = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t top = k4[i] >> 24;
                        if (e + i < whi && top >= v0) {
                            in_bits |= 1u << i;
                            if (top == v0) atomicAdd(&sm.hist[1][(k4[i] >> 16) & 0xFFu], 1u);
                        }
                    }
                    uint32_t slot = n, step = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t bal = __ballot_sync(0xffffffffu, (in_bits >> i) & 1u);
                        slot += __popc(bal & lt);
                        step += __popc(bal);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if ((in_bits >> i) & 1u) {
                            if (slot < (uint32_t)kTopkListCap) sm.wlist[warp][slot] = e + i;
                            ++slot;
                        }
                    n += step;
                }
                if (lane == 0) {
                    sm.wlist_n[warp] = n;
                    if (n > (uint32_t)kTopkListCap) sm.list_overflow = 1u;
                }
            } else if (pass >= 2 && staged && !sm.list_overflow) {
                const uint32_t n = sm.wlist_n[warp];
                for (uint32_t j = lane; j < n; j += 32) {
                    const uint32_t key = staged_keys[sm.wlist[warp][j] - lo];
                    if ((key & mask) == prefix) atomicAdd(&sm.hist[pass][(key >> shift) & 0xFFu], 1u);
                }
            } else if (pass > 0 || !staged) {
                for (int e = lo + 4 * tid; e < hi; e += 4 * kTopkThreads) {
                    uint32_t k4[4];
                    topk_keys4(staged_keys, row, staged, lo, e, k4);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (e + i < hi && (k4[i] & mask) == prefix) atomicAdd(&sm.hist[pass][(k4[i] >> shift) & 0xFFu], 1u);
                }
            }
            tr.at(0x8210 + pass);
            cluster_sync_all();  // every CTA's histogram of this pass is complete
            tr.at(0x8240 + pass);
            uint32_t h[kTopkCluster];
            if (tid < kTopkBins) {
                const uint32_t a = smem_u32(&sm.hist[pass][tid]);
#pragma unroll
                for (int q = 0; q < kTopkCluster; ++q) h[q] = topk_ld_cluster(mapa_shared(a, (uint32_t)q));
                uint32_t s = 0;
#pragma unroll
                for (int q = 0; q < kTopkCluster; ++q) s += h[q];
                sm.tot[tid] = s;
            }
            if (pass == 3) cluster_arrive_relaxed();  // this CTA has read the others' shared memory
            __syncthreads();
            tr.at(0x8250 + pass);
            // suffix sums from the top bin down: bin v holds the need-th largest key when the
            // keys in the bins above it number fewer than `need` and those with it at least `need`
            if (tid < kTopkBins) {
                const int rev = kTopkBins - 1 - tid;  // thread tid scans bin 255 - tid
                const uint32_t cnt = sm.tot[rev];
                uint32_t x = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                if (lane == 31) sm.warp_sum[warp] = x;
                __syncwarp();
                asm volatile("bar.sync 1, 256;" ::: "memory");
                uint32_t before = 0;
                for (int w = 0; w < warp; ++w) before += sm.warp_sum[w];
                const uint32_t incl = before + x, above = incl - cnt;
                if (above < need && incl >= need) {
                    sm.pick[0] = (uint32_t)rev;
                    sm.pick[1] = above;
                }
            }
            __syncthreads();
            tr.at(0x8260 + pass);
            const uint32_t v = sm.pick[0];
            need -= sm.pick[1];
            prefix |= v << shift;
            mask |= 0xFFu << shift;
            // every rank's keys in the bins above v (and, last pass, in bin v itself)
            if (tid < kTopkBins) {
#pragma unroll
                for (int q = 0; q < kTopkCluster; ++q) {
                    acc_gt[q] += (uint32_t)tid > v ? h[q] : 0u;
                    acc_eq[q] += (pass == 3 && (uint32_t)tid == v) ? h[q] : 0u;
                }
            }
            __syncthreads();  // pick[] and warp_sum[] are rewritten by the next pass
            tr.at(0x8220 + pass);
            if (pass == 1 && staged) {
                // After two bytes only a few keys still carry the prefix (about 30 per sequence of
                // normally spread scores).  Each CTA offers its own; after one cluster barrier every
                // CTA reads them all and finds the threshold key among them directly, instead of two
                // more histogram passes.  If any CTA has more than kTopkCandCap of them (tie-heavy
                // scores), every CTA sees it and the passes go on.
                if (tid == 0) sm.cand_n = 0u;
                __syncthreads();
                auto offer = [&](uint32_t key, bool in) {  // whole warps call this
                    const uint32_t bal = __ballot_sync(0xffffffffu, in);
                    if (bal == 0u) return;
                    uint32_t base = 0;
                    if (lane == 0) base = atomicAdd(&sm.cand_n, (uint32_t)__popc(bal));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    if (in) {
                        const uint32_t slot = base + __popc(bal & lt);
                        if (slot < (uint32_t)kTopkCandCap) sm.cand[slot] = key;
                    }
                };
                if (!sm.list_overflow) {
                    const uint32_t n = sm.wlist_n[warp];
                    for (uint32_t j0 = 0; j0 < n; j0 += 32) {
                        const uint32_t j = j0 + lane;
                        const uint32_t key = j < n ? staged_keys[sm.wlist[warp][j] - lo] : 0u;
                        offer(key, j < n && (key & mask) == prefix);
                    }
                } else {
                    for (int e0 = wlo; e0 < whi; e0 += 128) {
                        const int e = e0 + 4 * lane;
                        uint32_t k4[4] = {0u, 0u, 0u, 0u};
                        if (e < whi) topk_keys4(staged_keys, row, true, lo, e, k4);
#pragma unroll
                        for (int i = 0; i < 4; ++i) offer(k4[i], e + i < whi && (k4[i] & mask) == prefix);
                    }
                }
                __syncthreads();
                cluster_sync_all();  // every CTA's candidates are published
                if (tid < 32) {  // one warp: lane q reads rank q's count, a scan makes the offsets
                    uint32_t n = lane < kTopkCluster ? topk_ld_cluster(mapa_shared(smem_u32(&sm.cand_n), (uint32_t)lane))
                                                     : 0u;
                    if (n > (uint32_t)kTopkCandCap) n = 1u << 20;  // an overflow poisons the total
                    uint32_t x = n;
#pragma unroll
                    for (int o = 1; o < kTopkCluster; o <<= 1) {
                        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += y;
                    }
                    if (lane < kTopkCluster) sm.xoff[lane + 1] = x;
                    if (lane == 0) sm.xoff[0] = 0u;
                }
                __syncthreads();
                const uint32_t total = sm.xoff[kTopkCluster];
                if (total <= (uint32_t)(kTopkCluster * kTopkCandCap)) {
                    if (tid < (int)total) {
                        int q = 0;
                        while (sm.xoff[q + 1] <= (uint32_t)tid) ++q;
                        const uint32_t a = smem_u32(&sm.cand[tid - (int)sm.xoff[q]]);
                        sm.all_key[tid] = topk_ld_cluster(mapa_shared(a, (uint32_t)q));
                        sm.all_rank[tid] = (uint8_t)q;
                    }
                    cluster_arrive_relaxed();  // this CTA has read the others' shared memory
                    __syncthreads();
                    // the need-th largest candidate: fewer than `need` candidates above it, at least
                    // `need` at or above it
                    if (tid < (int)total) {
                        const uint32_t mine = sm.all_key[tid];
                        uint32_t gt = 0, ge = 0;
                        for (uint32_t j = 0; j < total; ++j) {
                            const uint32_t o = sm.all_key[j];
                            gt += o > mine ? 1u : 0u;
                            ge += o >= mine ? 1u : 0u;
                        }
                        if (gt < need && ge >= need) {
                            sm.pick[0] = mine;
                            sm.pick[1] = gt;
                        }
                    }
                    __syncthreads();
                    const uint32_t T = sm.pick[0];
                    if (tid < (int)total) {
                        const uint32_t key = sm.all_key[tid];
                        if (key > T) atomicAdd(&sm.rank_gt[sm.all_rank[tid]], 1u);
                        else if (key == T) atomicAdd(&sm.rank_eq[sm.all_rank[tid]], 1u);
                    }
                    need -= sm.pick[1];
                    prefix = T;
                    mask = 0xFFFFFFFFu;
                    tr.at(0x8270);
                    break;
                }
            }
        }
        if (tid < kTopkBins) {
#pragma unroll
            for (int q = 0; q < kTopkCluster; ++q) {
                if (acc_gt[q]) atomicAdd(&sm.rank_gt[q], acc_gt[q]);
                if (acc_eq[q]) atomicAdd(&sm.rank_eq[q], acc_eq[q]);
            }
        }
    } else if (tid < kTopkCluster) {
        // every position is taken: rank q's picks are its whole slice
        const int qlo = min(L, tid * chunk);
        sm.rank_gt[tid] = (uint32_t)(min(L, qlo + chunk) - qlo);
    }
    __syncthreads();
    // where this CTA's picks go: after the lower ranks' picks; equal keys go to the lowest ranks
    // (lowest positions) first, `need` of them in all
    uint32_t out_off = 0, eq_before = 0;
    for (uint32_t q = 0; q < r; ++q) {
        const uint32_t eq = sm.rank_eq[q];
        out_off += sm.rank_gt[q] + (eq_before >= need ? 0u : min(eq, need - eq_before));
        eq_before += eq;
    }
    const uint32_t cta_picks = sm.rank_gt[r] + (eq_before >= need ? 0u : min(sm.rank_eq[r], need - eq_before));
    tr.at(0x8231);

    // Compaction.  Warp w owns positions [wlo, whi) of the CTA's slice (a multiple of 128 long, 4
    // consecutive positions per lane per step): it counts its keys above the threshold key
    // `prefix` and equal to it, then writes its picks in position order after those of the lower
    // ranks and lower warps.
    int32_t *sel_out = p.sel_index + (size_t)b * p.k;
    const bool use_lists = staged && !take_all && !sm.list_overflow;
    if (take_all) {
        for (int e = lo + tid; e < hi; e += kTopkThreads) sel_out[e] = e;
    } else if (use_lists) {
        // the same compaction over the warps' lists (every key above or equal to the threshold is
        // in them, in position order)
        const uint32_t n = sm.wlist_n[warp];
        {
            uint32_t gt = 0, eq = 0;
            for (uint32_t j = lane; j < n; j += 32) {
                const uint32_t key = staged_keys[sm.wlist[warp][j] - lo];
                gt += key > prefix ? 1u : 0u;
                eq += key == prefix ? 1u : 0u;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                gt += __shfl_xor_sync(0xffffffffu, gt, off);
                eq += __shfl_xor_sync(0xffffffffu, eq, off);
            }
            if (lane == 0) {
                sm.warp_sum[warp] = gt;
                sm.warp_sum2[warp] = eq;
            }
        }
        __syncthreads();
        uint32_t n_out = out_off, n_eq = eq_before;
        for (int w = 0; w < warp; ++w) {
            const uint32_t eqw = sm.warp_sum2[w];
            n_out += sm.warp_sum[w] + (n_eq >= need ? 0u : min(eqw, need - n_eq));
            n_eq += eqw;
        }
        for (uint32_t j0 = 0; j0 < n; j0 += 32) {
            const uint32_t j = j0 + lane;
            int32_t e = 0;
            uint32_t key = 0;
            if (j < n) {
                e = sm.wlist[warp][j];
                key = staged_keys[e - lo];
            }
            const bool is_gt = j < n && key > prefix, is_eq = j < n && key == prefix;
            const uint32_t bal_eq = __ballot_sync(0xffffffffu, is_eq);
            const uint32_t eq_rank = n_eq + __popc(bal_eq & lt);
            const bool pick = is_gt || (is_eq && eq_rank < need);
            const uint32_t bal_pick = __ballot_sync(0xffffffffu, pick);
            if (pick) {
                const uint32_t pos = n_out + __popc(bal_pick & lt);
                if (pos < (uint32_t)p.k) {
                    sel_out[pos] = e;
                    if (pos - out_off < (uint32_t)kTopkPickCap) sm.pick_pos[pos - out_off] = e;
                } else {
                    raise_status(0x10u);
                }
            }
            n_out += __popc(bal_pick);
            n_eq += __popc(bal_eq);
        }
    } else {
        {
            uint32_t gt = 0, eq = 0;
            for (int e = wlo + 4 * lane; e < whi; e += 128) {
                uint32_t k4[4];
                topk_keys4(staged_keys, row, staged, lo, e, k4);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (e + i < whi) {
                        gt += k4[i] > prefix ? 1u : 0u;
                        eq += k4[i] == prefix ? 1u : 0u;
                    }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                gt += __shfl_xor_sync(0xffffffffu, gt, off);
                eq += __shfl_xor_sync(0xffffffffu, eq, off);
            }
            if (lane == 0) {
                sm.warp_sum[warp] = gt;
                sm.warp_sum2[warp] = eq;
            }
        }
        __syncthreads();
        uint32_t n_out = out_off, n_eq = eq_before;
        for (int w = 0; w < warp; ++w) {
            const uint32_t eqw = sm.warp_sum2[w];
            n_out += sm.warp_sum[w] + (n_eq >= need ? 0u : min(eqw, need - n_eq));
            n_eq += eqw;
        }
        for (int e0 = wlo; e0 < whi; e0 += 128) {
            const int e = e0 + 4 * lane;
            uint32_t gt_bits = 0, eq_bits = 0;
            if (e < whi) {
                uint32_t k4[4];
                topk_keys4(staged_keys, row, staged, lo, e, k4);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (e + i < whi) {
                        gt_bits |= (k4[i] > prefix ? 1u : 0u) << i;
                        eq_bits |= (k4[i] == prefix ? 1u : 0u) << i;
                    }
            }
            if (!__any_sync(0xffffffffu, (gt_bits | eq_bits) != 0u)) continue;
            // ranks among the warp's equal keys and picks: the lower lanes' flags come first
            uint32_t eq_rank = n_eq, eq_step = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t bal = __ballot_sync(0xffffffffu, (eq_bits >> i) & 1u);
                eq_rank += __popc(bal & lt);
                eq_step += __popc(bal);
            }
            uint32_t pick_bits = gt_bits;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if ((eq_bits >> i) & 1u) {
                    if (eq_rank < need) pick_bits |= 1u << i;
                    ++eq_rank;
                }
            uint32_t pos = n_out, pick_step = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t bal = __ballot_sync(0xffffffffu, (pick_bits >> i) & 1u);
                pos += __popc(bal & lt);
                pick_step += __popc(bal);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if ((pick_bits >> i) & 1u) {
                    // the counts guarantee pos < k; a violation is recorded, never written
                    if (pos < (uint32_t)p.k) {
                        sel_out[pos] = e + i;
                        if (pos - out_off < (uint32_t)kTopkPickCap) sm.pick_pos[pos - out_off] = e + i;
                    } else {
                        raise_status(0x10u);
                    }
                    ++pos;
                }
            n_out += pick_step;
            n_eq += eq_step;
        }
    }
    __syncthreads();  // this CTA's positions are written (and visible to the block)
    tr.at(0x8232);

    // Gather this CTA's rows [out_off, out_off + cta_picks) into the compact pool: first every
    // row's pool row (from the slice's block-table entries), then all copies, 16 bytes per thread
    // per unit, six units in flight per thread.
    const size_t seq_row0 = (size_t)b * p.npk * kSparsePage;
    const uint32_t n_rows = min(cta_picks, (uint32_t)p.k - min(out_off, (uint32_t)p.k));
    auto resolve = [&](uint32_t i) -> int {  // pool row of this CTA's i-th pick, or -1
        int t;
        if (take_all) t = (int)(out_off + i);
        else t = i < (uint32_t)kTopkPickCap ? sm.pick_pos[i] : sel_out[out_off + i];
        const int j = t / kSparsePage;
        const int pg = fits ? sm.slice_bt[j - page0] : p.block_table[(size_t)b * p.max_pages + j];
        if (pg < 0 || pg >= p.num_pages) return -1;
        return pg * kSparsePage + t % kSparsePage;
    };
    for (uint32_t i = tid; i < n_rows && i < (uint32_t)kTopkPickCap; i += kTopkThreads) sm.src_row[i] = resolve(i);
    __syncthreads();
    tr.at(0x8233);
    constexpr int kUnits = kSparseRow / 8;  // 16-byte pieces of a row
    constexpr int kGatherU = 6;
    const uint4 *pool4 = reinterpret_cast<const uint4 *>(p.kv_pool);
    uint4 *out4 = reinterpret_cast<uint4 *>(p.sel_pool) + (seq_row0 + out_off) * kUnits;
    const uint32_t n_units = n_rows * kUnits;
    for (uint32_t base = 0; base < n_units; base += kTopkThreads * kGatherU) {
        uint4 v[kGatherU];
#pragma unroll
        for (int u = 0; u < kGatherU; ++u) {
            const uint32_t unit = base + tid + u * kTopkThreads;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (unit < n_units) {
                const uint32_t i = unit / kUnits;
                const int src = i < (uint32_t)kTopkPickCap ? sm.src_row[i] : resolve(i);
                if (src >= 0) v[u] = __ldcs(pool4 + (size_t)src * kUnits + unit % kUnits);
                else if (unit % kUnits == 0) raise_status(0x1u);
            }
        }
#pragma unroll
        for (int u = 0; u < kGatherU; ++u) {
            const uint32_t unit = base + tid + u * kTopkThreads;
            if (unit < n_units) out4[unit] = v[u];
        }
    }
    tr.at(0x8234);
    // the last CTA fills the tail: zero rows past sel_len on the sequence's compact pages, -1
    // positions past sel_len; the first writes the identity block table and the length
    if (r == kTopkCluster - 1) {
        const size_t first = seq_row0 + (size_t)sel_len, end = seq_row0 + (size_t)p.npk * kSparsePage;
        uint4 *z = reinterpret_cast<uint4 *>(p.sel_pool);
        for (size_t j = first * (kSparseRow / 8) + tid; j < end * (kSparseRow / 8); j += kTopkThreads)
            z[j] = make_uint4(0u, 0u, 0u, 0u);
        for (int j = sel_len + tid; j < p.k; j += kTopkThreads) sel_out[j] = -1;
    }
    if (r == 0) {
        for (int j = tid; j < p.npk; j += kTopkThreads) p.sel_block_table[(size_t)b * p.npk + j] = b * p.npk + j;
        if (tid == 0) {
            p.sel_lens[b] = sel_len;
            if (p.plan_items != nullptr) {
                // the plan the decode's planner makes for one unsplit query per sequence (the
                // item order only changes which CTA pair takes which item)
                const int tiles = (sel_len + kSparsePage - 1) / kSparsePage;
                Item it;
                it.bt = b, it.tb = 0, it.te = tiles, it.slot = -1, it.b = b, it.n_vis = sel_len;
                it.pad0 = it.pad1 = 0;
                p.plan_items[b] = it;
                BtInfo in;
                in.splits = 1, in.slot_base = -1, in.tiles = tiles, in.item_off = b;
                p.plan_info[b] = in;
                if (b == 0) {
                    p.plan_hdr->n_items = (int)(gridDim.x / kTopkCluster);
                    p.plan_hdr->n_bt = (int)(gridDim.x / kTopkCluster);
                    p.plan_hdr->n_split = 0;
                    p.plan_hdr->max_items = p.plan_max_items;
                    p.plan_hdr->max_slots = p.plan_max_slots;
                }
            }
        }
    }
    // no CTA leaves while another may still read its histograms
    if (!take_all) cluster_wait();
}

}  // namespace mla
