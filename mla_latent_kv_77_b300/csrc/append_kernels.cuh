// append_kernels.cuh - the cache write for new tokens, the step before the decode
// ("DeepSeek-V2" explainer, Step 5, the paper's equation 9, and Step 7):
//   row[n] = [ W^DKV h_n (512) | RoPE_pos(W^KR h_n) (64) ]
// written into the paged pool at row block_table[b, pos / 64] * 64 + pos % 64, where token t of
// sequence b has position pos = seq_lens[b] - Tq + t (the lengths already count the new tokens,
// as in the causal decode).
//
// One tcgen05 GEMM, D[token, column] = sum_k h[token, k] W[column, k], in one kernel: tokens fill
// the 128-row M side, the 576 output columns are split into tiles of BN (W^DKV supplies columns
// 0-511, W^KR 512-575), and the rows are finished (RoPE, bf16, scatter) in the same kernel.  Two
// shapes:
//   BN = 64, K split over a thread-block cluster of S <= 8 CTAs: for a decode step's few new
//     tokens.  With one token tile, 9 column tiles x 8 splits = 72 CTAs (9 clusters, which all fit
//     at once) each stream 10 of the 80 K blocks of a 5120-wide model.  Each CTA stages its fp32
//     partial tile in shared memory, and CTA r of the cluster adds its share of the rows of all S
//     partials, in rank order, through distributed shared memory: no partial sums go to global
//     memory and there is no second kernel.  With at most 64 tokens only the first 64 rows of h
//     are loaded: the MMA's other 64 rows read whatever follows in shared memory and give
//     accumulator rows that are never used.
//   BN = 144, no split: for a prompt's thousands of tokens, where the token tiles alone fill the
//     GPU; four column tiles keep the shared-memory operand traffic per MMA low.  The last one
//     spans W^DKV's rows 432-511 and all of W^KR: it is two segments of 80 and 64 weight rows,
//     each with its own MMAs into its own accumulator columns.
// Loads are few and large: each TMA copy brings C consecutive 64-wide K blocks of h (or of one
// weight segment) at once, as C stacked 128-byte-swizzled blocks (a 3-D view of the row-major
// matrix), so a CTA of the decode shape issues four copies in all; issuing one small box per K
// block and weight slice cost more time than moving the bytes.
//
// RoPE angles never use FP64 (which B300 runs at a small fraction of its FP32 rate): pair i's
// rate theta_i / (2 pi) is passed as a 64-bit binary fraction of a turn, so pos * rate modulo one
// turn is an exact 64-bit integer product; its top 24 bits give the angle to 2^-24 of a turn for
// any position, and sincospif does the rest.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mla {

constexpr int kAppendCols = 576;    // d_c + d_R: one cache row
constexpr int kAppendLatent = 512;  // d_c: columns from W^DKV
constexpr int kAppendPairs = (kAppendCols - kAppendLatent) / 2;
constexpr int kAppendTileM = 128;   // tokens per CTA
constexpr int kAppendThreads = 192;  // warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 epilogue
constexpr int kAppendMaxSplits = 8;  // portable cluster size
constexpr uint32_t kAppendSmemCap = 227u * 1024u;

// BN output columns per CTA; AROWS rows of h loaded per K block (64 when the call has at most 64
// tokens, else the full 128-row tile)
template <int BN, int AROWS>
struct AppendShape {
    static constexpr int kColTiles = kAppendCols / BN;
    static constexpr uint32_t kBlockBytes = (AROWS + BN) * 128u;  // one K block of h and weights
    static constexpr bool kReduce = BN == 64;                     // K split over the cluster
    static constexpr int kMaxStages = 8;
    static constexpr uint32_t kRegionCap = kAppendSmemCap - 256u - 1024u;
    static constexpr uint32_t kSmem = kAppendSmemCap;
    static constexpr uint32_t kTmemCols = BN <= 32 ? 32u : (BN <= 64 ? 64u : (BN <= 128 ? 128u : 256u));
    // fp32 partial tile staged for the cluster reduction: AROWS rows of BN floats
    static constexpr uint32_t kStageRowBytes = BN * 4u;
    // K blocks per copy that leave room for two stages
    static constexpr int kMaxChunk = (int)(kRegionCap / (2u * kBlockBytes));
    static_assert(kAppendCols % BN == 0 && BN % 16 == 0 && kMaxChunk >= 1, "bad append tile");
    static_assert(!kReduce || (uint32_t)AROWS * kStageRowBytes <= 2u * kBlockBytes, "staging exceeds a stage");
};

struct AppendParams {
    const int32_t *block_table;  // [batch, max_pages]
    const int32_t *seq_lens;     // [batch], counting the new tokens
    __nv_bfloat16 *pool;         // [num_pages, 64, 576]
    int n_tokens, q_len, num_pages, max_pages;  // q_len: new rows per sequence (tokens, or merged blocks)
    int nkb;     // 64-wide K blocks of d_model
    int splits;  // K splits = cluster size (BN = 64 only; 1, 2, 4 or 8)
    int m;       // compressed write: tokens merged into each row (1 for the plain write)
    int chunk;   // K blocks per copy (the tensor maps' box depth), at most the shape's kMaxChunk
    uint64_t turns[kAppendPairs];  // pair i: theta_i / (2 pi) as a fraction of 2^64
};

// Pool row of new token n (and its position), or nullptr when the token has no valid slot: a
// negative position or one past the block table (MLA_DEV_BAD_SEQ_LEN), or a page outside the pool
// (MLA_DEV_BAD_BLOCK_TABLE).  Nothing is written for such a token; its sequence's other tokens
// are written where their own slots are valid.
__device__ __forceinline__ __nv_bfloat16 *append_row(const AppendParams &p, int n, int &pos) {
    const int b = n / p.q_len, t = n - b * p.q_len;
    pos = p.seq_lens[b] - p.q_len + t;
    if (pos < 0 || (pos >> 6) >= p.max_pages) {
        raise_status(0x2u);
        return nullptr;
    }
    const int pg = p.block_table[(size_t)b * p.max_pages + (pos >> 6)];
    if (pg < 0 || pg >= p.num_pages) {
        raise_status(0x1u);
        return nullptr;
    }
    return p.pool + ((size_t)pg * 64 + (pos & 63)) * kAppendCols;
}

// Turn the pair (x0, x1) counter-clockwise by pos * theta_i, theta_i / (2 pi) = turns / 2^64.
__device__ __forceinline__ void rope_pair(float &x0, float &x1, int pos, uint64_t turns) {
    const uint64_t frac = (uint64_t)(uint32_t)pos * turns;  // modulo 2^64: whole turns drop out
    const float u = (float)(uint32_t)(frac >> 40) * 0x1p-23f;  // twice the fraction of a turn
    float s, c;
    sincospif(u, &s, &c);
    const float y0 = x0 * c - x1 * s;
    const float y1 = x0 * s + x1 * c;
    x0 = y0;
    x1 = y1;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_dep16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    // volatile keeps it after the cluster barrier; no memory clobber, so several can be in flight
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Four finished numbers of token n's row (columns col..col+3): RoPE where they are k^R, bf16.
__device__ __forceinline__ void append_store4(const AppendParams &p, __nv_bfloat16 *dst, int pos, int col,
                                              float4 v) {
    if (col >= kAppendLatent) {
        const int i = (col - kAppendLatent) / 2;
        rope_pair(v.x, v.y, pos, p.turns[i]);
        rope_pair(v.z, v.w, pos, p.turns[i + 1]);
    }
    *reinterpret_cast<uint2 *>(dst + col) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// The weight rows of column tile ct as at most two segments, each one TMA copy per chunk and its
// own MMAs: rows [row, row + rows) of W^DKV (map a: BN-row boxes, map b: (512 % BN)-row boxes) or of
// W^KR (map r: 64-row boxes), landing in accumulator columns [col, col + rows) of the tile.
struct AppendSeg {
    const CUtensorMap *map;
    int row, rows, col;
};
// The compressed write's column tile ct instead holds 32 row components and their 32 z
// components: rows [32 ct, 32 ct + 32) of W^DKV or W^KR (maps a, r: 32-row boxes) in columns 0-31
// and the same rows of W^Z (map b) in columns 32-63.
template <int BN, bool COMP>
__device__ __forceinline__ int append_segments(int ct, const CUtensorMap *wa, const CUtensorMap *wb,
                                               const CUtensorMap *wr, AppendSeg (&seg)[2]) {
    if constexpr (COMP) {
        const int c0 = ct * 32;
        seg[0] = {c0 < kAppendLatent ? wa : wr, c0 < kAppendLatent ? c0 : c0 - kAppendLatent, 32, 0};
        seg[1] = {wb, c0, 32, 32};
        return 2;
    }
    const int r0 = ct * BN, r1 = r0 + BN;
    if (r1 <= kAppendLatent) {
        seg[0] = {wa, r0, BN, 0};
        return 1;
    }
    if (r0 >= kAppendLatent) {
        seg[0] = {wr, r0 - kAppendLatent, BN, 0};
        return 1;
    }
    seg[0] = {wb, r0, kAppendLatent - r0, 0};
    seg[1] = {wr, 0, r1 - kAppendLatent, kAppendLatent - r0};
    return 2;
}

// The compressed write's part of the cluster reduction.  The CTAs of the cluster share the
// tile's 32 components (8 four-component groups, 8 / splits each), all rows: per block of m
// tokens and per four components, a thread adds the partners' partial sums of each token's row
// values (staged columns 0-31) and z values (32-63), turns the k^R pairs at the token's own
// position, and merges the m tokens with a softmax over them taken per component (running
// maximum, as the decode's softmax does), then writes the block's four merged numbers (bf16) to
// the pool row of its compressed position.
// One token's contribution to a block's merge, for four components: the partners' partial sums
// of its row values and z values, its k^R pairs turned at its position, then the running
// softmax update (max, denominator, numerator) per component.
__device__ __forceinline__ void append_merge_token(const AppendParams &p, uint32_t base, int r_in, int quad, int comp,
                                                   int pos, int splits, float (&mx)[4], float (&den)[4],
                                                   float (&num)[4]) {
    const uint32_t off_v = base + (uint32_t)r_in * 256u + (uint32_t)((quad ^ (r_in & 7)) * 16);
    const uint32_t off_z = off_v + 128u;
    float4 xv[kAppendMaxSplits], xz[kAppendMaxSplits];
#pragma unroll
    for (int r = 0; r < kAppendMaxSplits; ++r)
        if (r < splits) {
            xv[r] = ld_dsmem_f4(mapa_shared(off_v, (uint32_t)r));
            xz[r] = ld_dsmem_f4(mapa_shared(off_z, (uint32_t)r));
        }
    float4 v = xv[0], z = xz[0];
#pragma unroll
    for (int r = 1; r < kAppendMaxSplits; ++r)
        if (r < splits) {
            v.x += xv[r].x; v.y += xv[r].y; v.z += xv[r].z; v.w += xv[r].w;
            z.x += xz[r].x; z.y += xz[r].y; z.z += xz[r].z; z.w += xz[r].w;
        }
    if (comp >= kAppendLatent) {
        const int pair = (comp - kAppendLatent) / 2;
        rope_pair(v.x, v.y, pos, p.turns[pair]);
        rope_pair(v.z, v.w, pos, p.turns[pair + 1]);
    }
    const float vv[4] = {v.x, v.y, v.z, v.w}, zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float nm = fmaxf(mx[e], zz[e]);
        const float keep = expf(mx[e] - nm), w = expf(zz[e] - nm);
        den[e] = fmaf(den[e], keep, w);
        num[e] = fmaf(num[e], keep, w * vv[e]);
        mx[e] = nm;
    }
}

// The compressed write's part of the cluster reduction.  The CTAs of the cluster share the
// tile's 32 components (8 four-component groups, 8 / splits each), all rows: per block of m
// tokens and per four components the partners' partial sums of each token's row values (staged
// columns 0-31) and z values (32-63) are added, the k^R pairs turned at the token's own position,
// and the m tokens merged with a softmax over them taken per component (running maximum, as the
// decode's softmax does); the block's four merged numbers go (bf16) to the pool row of its
// compressed position.  Blocks of fewer than 32 tokens take one thread each; larger ones a warp,
// whose lanes take every 32nd token and then combine their running sums.
template <int AROWS>
__device__ __forceinline__ void append_merge(const AppendParams &p, uint32_t base, int et, int sp, int mt, int ct,
                                             int splits, bool any_abort) {
    const int m = p.m;
    const int blocks = AROWS / m, quads = 8 / splits;
    const bool by_warp = m >= 32;
    const int lane = et & 31, workers = by_warp ? 4 : 128, me = by_warp ? et >> 5 : et;
    for (int idx = me; idx < blocks * quads && !any_abort; idx += workers) {
        const int gl = idx / quads, quad = sp * quads + idx % quads;
        const int r_first = gl * m;
        const int n_first = mt * kAppendTileM + r_first;
        if (n_first >= p.n_tokens) continue;
        int P = 0;
        __nv_bfloat16 *dst = append_row(p, n_first / m, P);
        const int comp = ct * 32 + quad * 4;
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float den[4] = {0.f, 0.f, 0.f, 0.f}, num[4] = {0.f, 0.f, 0.f, 0.f};
        if (by_warp) {
            for (int i = lane; i < m; i += 32) append_merge_token(p, base, r_first + i, quad, comp, P * m + i, splits, mx, den, num);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, mx[e], o);
                    const float d2 = __shfl_xor_sync(0xffffffffu, den[e], o);
                    const float n2 = __shfl_xor_sync(0xffffffffu, num[e], o);
                    const float nm = fmaxf(mx[e], m2);
                    const float a = expf(mx[e] - nm), b = expf(m2 - nm);
                    den[e] = den[e] * a + d2 * b;
                    num[e] = num[e] * a + n2 * b;
                    mx[e] = nm;
                }
            }
            if (lane != 0) continue;
        } else {
            for (int i = 0; i < m; ++i) append_merge_token(p, base, r_first + i, quad, comp, P * m + i, splits, mx, den, num);
        }
        if (dst != nullptr)
            *reinterpret_cast<uint2 *>(dst + comp) = make_uint2(pack_bf16x2(num[0] / den[0], num[1] / den[1]),
                                                                pack_bf16x2(num[2] / den[2], num[3] / den[3]));
    }
}

// grid (splits, column tiles, token tiles), kAppendThreads threads, clusters of (splits, 1, 1).
// Tensor maps are 3-D views (64 K, rows, K blocks) with boxes (64, rows, p.chunk):
//   tmap_h:  h [n_tokens, d_model], AROWS-row boxes
//   tmap_wa: W^DKV [512, d_model], BN-row boxes;  tmap_wb: W^DKV, (512 % BN)-row boxes (BN = 144)
//   tmap_wr: W^KR [64, d_model], 64-row boxes
// COMP (the compressed write, BN = 64 only): tmap_wa, tmap_wr with 32-row boxes, and tmap_wb is
// W^Z [576, d_model] with 32-row boxes.
template <int BN, int AROWS, bool COMP>
__global__ void __launch_bounds__(kAppendThreads, 1)
append_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_wa,
              const __grid_constant__ CUtensorMap tmap_wb, const __grid_constant__ CUtensorMap tmap_wr,
              const __grid_constant__ AppendParams p) {
    using S = AppendShape<BN, AROWS>;
    static_assert(!COMP || S::kReduce, "the compressed write merges rows in the cluster reduction");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sp = blockIdx.x, ct = blockIdx.y, mt = blockIdx.z;
    const int kb0 = (int)((long long)sp * p.nkb / p.splits);
    const int nk = (int)((long long)(sp + 1) * p.nkb / p.splits) - kb0;  // >= 1 since splits <= nkb
    const int C = p.chunk;
    const int n_chunks = (nk + C - 1) / C;
    const uint32_t a_bytes = (uint32_t)C * AROWS * 128u;     // a chunk of h: C blocks of AROWS rows
    const uint32_t stage_bytes = (uint32_t)C * S::kBlockBytes;
    const int n_stages = min(S::kMaxStages, (int)(S::kRegionCap / stage_bytes));  // >= 2
    // after the stage region: barriers full[s], empty[kMaxStages + s], accumulator done, drain;
    // then the TMEM address (+240) and the abort flag (+248)
    constexpr int kBarAcc = 2 * S::kMaxStages, kBarDrain = kBarAcc + 1;
    auto bar = [&](int i) { return base + S::kRegionCap + 8u * i; };
    const uint32_t abort_addr = base + S::kRegionCap + 248;
    volatile int *abort = reinterpret_cast<volatile int *>(smem_raw + (base - raw) + S::kRegionCap + 248);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + S::kRegionCap + 240);
    AppendSeg seg[2];
    const int n_seg = append_segments<BN, COMP>(ct, &tmap_wa, &tmap_wb, &tmap_wr, seg);
    Tracer tr;
    tr.at(0x8101);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2 * S::kMaxStages + 2; ++s) mbar_init(bar(s), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(base + S::kRegionCap + 240, S::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_h);
        for (int g = 0; g < n_seg; ++g) tma_prefetch_desc(seg[g].map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    tr.at(0x102);
    // reduce shape: the pool slot of this thread's first row of the reduction, looked up while
    // the weights stream in
    constexpr int kChunks4 = BN / 4;  // four-column chunks per row
    const int rows_per = AROWS / p.splits;
    const int et = threadIdx.x - 64;
    int pre_pos = 0;
    __nv_bfloat16 *pre_dst = nullptr;

    // the producer and MMA roles run as whole warps that wait together (a lone waiting thread
    // wakes up late); lane 0 issues the copies and the MMAs
    if (warp == 0) {
        int issued = 0;
        for (int i = 0; i < n_chunks; ++i, ++issued) {
            const int s = i % n_stages;
            if (__any_sync(0xffffffffu, !mbar_wait(bar(S::kMaxStages + s), ((i / n_stages) & 1) ^ 1, abort))) break;
            if (lane == 0) {
                const uint32_t sb = base + s * stage_bytes;
                const int kbx = kb0 + i * C;
                // a box reaching past n_tokens, past d_model or past this split's K range still
                // lands (zero-filled, or blocks the MMAs skip) and counts its full bytes
                mbar_arrive_expect_tx(bar(s), stage_bytes);
                tma_load_3d_nohint(sb, &tmap_h, 0, mt * kAppendTileM, kbx, bar(s));
                uint32_t b = sb + a_bytes;
                for (int g = 0; g < n_seg; ++g) {
                    tma_load_3d_nohint(b, seg[g].map, 0, seg[g].row, kbx, bar(s));
                    b += (uint32_t)C * seg[g].rows * 128u;
                }
            }
            __syncwarp();
        }
        tr.at(0x111);
        // wait for the last loads (normal exit or abort) before the CTA may move on
        if (lane == 0)
            for (int k = issued > n_stages ? issued - n_stages : 0; k < issued; ++k)
                if (!mbar_wait_drain(bar(k % n_stages), (k / n_stages) & 1)) break;
        __syncwarp();
        tr.at(0x112);
    } else if (warp == 1) {
        uint32_t idesc[2];
        for (int g = 0; g < n_seg; ++g) idesc[g] = idesc_bf16_f32(128, (uint32_t)seg[g].rows, 0, 0);
        for (int i = 0; i < n_chunks; ++i) {
            const int s = i % n_stages;
            if (__any_sync(0xffffffffu, !mbar_wait(bar(s), (i / n_stages) & 1, abort))) break;
            if (i == 0) tr.at(0x120);
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sb = base + s * stage_bytes;
                const int nb = min(C, nk - i * C);
                // descriptors of the chunk's first block; a block further on adds its byte offset
                // / 16 to the start-address field, a 16-wide K step adds 2
                const uint64_t a0 = sdesc_sw128(sb, 16u, 1024u);
                uint64_t b0[2];
                uint32_t off = a_bytes;
                for (int g = 0; g < n_seg; ++g) {
                    b0[g] = sdesc_sw128(sb + off, 16u, 1024u);
                    off += (uint32_t)C * seg[g].rows * 128u;
                }
                for (int j = 0; j < nb; ++j) {
                    // A: 128 rows from block j of the chunk (with AROWS = 64 the last 64 rows are
                    // whatever follows, giving accumulator rows nothing reads)
                    const uint64_t ad = a0 + (uint64_t)(j * AROWS * 8);
                    for (int g = 0; g < n_seg; ++g) {
                        const uint64_t bd = b0[g] + (uint64_t)(j * seg[g].rows * 8);
#pragma unroll
                        for (int k = 0; k < 4; ++k)  // both operands K-major, 16 K per MMA
                            mma_ss(tmem + (uint32_t)seg[g].col, ad + 2u * k, bd + 2u * k, idesc[g], (i | j | k) != 0);
                    }
                }
                mma_commit(bar(S::kMaxStages + s));
            }
            __syncwarp();
        }
        tr.at(0x121);
        if (lane == 0) {
            mma_commit(bar(kBarAcc));
            // every MMA issued has completed before the CTA may free its tensor memory
            mma_commit(bar(kBarDrain));
            mbar_wait_drain(bar(kBarDrain), 0);
        }
        __syncwarp();
    } else {
        // epilogue: warps 2..5 -> TMEM lane quadrants 2, 3, 0, 1; lane = token row of the tile
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        if constexpr (S::kReduce && !COMP) {
            if (et < rows_per * kChunks4) {
                const int n = mt * kAppendTileM + sp * rows_per + et / kChunks4;
                if (n < p.n_tokens) pre_dst = append_row(p, n, pre_pos);
            }
        }
        // tcgen05.ld is warp-collective: the whole warp takes the same branch around it
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarAcc), 0, abort));
        tr.at(0x130);
        if (ok) {
            tc_fence_after();
            if constexpr (S::kReduce) {
                // the fp32 partial tile -> shared memory (the drained stage region), row-major
                // [AROWS][BN]; within each 128-byte half of a row the 16-byte chunks are rotated by
                // the row, so a warp's stores spread over the banks.  Warps whose rows are all
                // beyond AROWS have nothing to stage.
                if (q * 32 < AROWS) {
                    const uint32_t rb = base + (uint32_t)row * S::kStageRowBytes;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_off + 32u * c, v);
                        tmem_ld_wait_dep(v);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             rb + (uint32_t)(c * 128 + ((e ^ (row & 7)) * 16))),
                                         "r"(v[4 * e]), "r"(v[4 * e + 1]), "r"(v[4 * e + 2]), "r"(v[4 * e + 3])
                                         : "memory");
                    }
                }
            } else {
                const int n = mt * kAppendTileM + row;
                int pos = 0;
                __nv_bfloat16 *dst = n < p.n_tokens ? append_row(p, n, pos) : nullptr;
                // every lane loads (the loads are warp-collective); only rows with a slot store
#pragma unroll 1
                for (int c = 0; c < BN / 16; ++c) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_off + 16u * c, v);
                    tmem_ld_wait_dep16(v);
                    if (dst == nullptr) continue;
                    const int col = ct * BN + 16 * c;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        append_store4(p, dst, pos, col + 4 * e,
                                      make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                  __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3])));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, S::kTmemCols);
    }
    tr.at(0x131);
    if constexpr (S::kReduce) {
        // every CTA of the cluster has staged its partial tile (or aborted)
        cluster_sync_all();
        tr.at(0x140);
        if (warp >= 2) {
            const int splits = p.splits;
            bool any_abort = false;
            for (int r = 0; r < splits; ++r) any_abort |= ld_dsmem_u32(mapa_shared(abort_addr, (uint32_t)r)) != 0u;
            if constexpr (COMP) {
                append_merge<AROWS>(p, base, et, sp, mt, ct, splits, any_abort);
            } else
            // this CTA's rows of the tile: rows_per = AROWS / splits rows of BN / 4 four-column chunks
            for (int idx = et; idx < rows_per * kChunks4 && !any_abort; idx += 128) {
                const int r_in = sp * rows_per + idx / kChunks4, chunk = idx % kChunks4;
                const int n = mt * kAppendTileM + r_in;
                if (n >= p.n_tokens) continue;
                const uint32_t off = base + (uint32_t)r_in * S::kStageRowBytes + (uint32_t)((chunk & ~7) * 16) +
                                     (uint32_t)(((chunk & 7) ^ (r_in & 7)) * 16);
                int pos = pre_pos;
                __nv_bfloat16 *dst = pre_dst;
                if (idx != et) dst = append_row(p, n, pos);  // its loads overlap the ones below
                // every partner's partial first (all in flight), then the sum in rank order
                float4 x[kAppendMaxSplits];
#pragma unroll
                for (int r = 0; r < kAppendMaxSplits; ++r)
                    if (r < splits) x[r] = ld_dsmem_f4(mapa_shared(off, (uint32_t)r));
                float4 acc = x[0];
#pragma unroll
                for (int r = 1; r < kAppendMaxSplits; ++r)
                    if (r < splits) {
                        acc.x += x[r].x;
                        acc.y += x[r].y;
                        acc.z += x[r].z;
                        acc.w += x[r].w;
                    }
                if (dst != nullptr) append_store4(p, dst, pos, ct * BN + chunk * 4, acc);
            }
        }
        tr.at(0x141);
        // no CTA leaves while its partners still read its shared memory
        cluster_sync_relaxed();
    }
    tr.at(0x8142);
}

}  // namespace mla
