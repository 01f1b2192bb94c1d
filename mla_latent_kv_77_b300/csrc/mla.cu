// mla.cu - C ABI of the MLA decode library (declared in include/mla.h).
// Host side only: argument checks, TMA descriptors, launch configuration.
// Every numeric step runs in the kernels of decode_kernels.cuh, gemm_kernels.cuh,
// append_kernels.cuh and sparse_kernels.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mla.h"
#include "../../include/mla_testing.h"
#include "append_kernels.cuh"
#include "decode_kernels.cuh"
#include "gemm_kernels.cuh"
#include "sparse_kernels.cuh"

namespace mla {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxRows = 65536;       // batch * q_len limit of the planner
constexpr int kMaxQLen = 64;
constexpr int kMaxAppendTokens = 1 << 20;  // new tokens per cache write (a long prefill)
constexpr int kMaxDModel = 1 << 16;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sms = 0;
    int clusters = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Per-device setup, once: capability check, kernel attributes, co-resident CTA pairs.
mla_status_t device_setup(int *dev_out, DeviceInfo **info_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MLA_ERR_CUDA;
        d.supported = (prop.major == 10 && prop.minor == 3);
        d.sms = prop.multiProcessorCount;
        if (d.supported) {
            // every kernel of a decode call asks for the maximum shared-memory carveout, so the
            // SMs need not switch their L1 / shared split between the plan, decode and combine
            for (const void *fn : {(const void *)plan_kernel, (const void *)combine_kernel,
                                   (const void *)combine_rows_kernel, (const void *)decode_kernel,
                                   (const void *)head_gemm_kernel, (const void *)append_kernel<64, 64, false>,
                                   (const void *)append_kernel<64, 128, false>, (const void *)append_kernel<144, 128, false>,
                                   (const void *)append_kernel<64, 64, true>, (const void *)append_kernel<64, 128, true>})
                cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
            cudaGetLastError();
            if (cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecodeSmem) !=
                    cudaSuccess ||
                cudaFuncSetAttribute(head_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmemMax) !=
                    cudaSuccess ||
                cudaFuncSetAttribute(append_kernel<64, 64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AppendShape<64, 64>::kSmem) != cudaSuccess ||
                cudaFuncSetAttribute(append_kernel<64, 128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AppendShape<64, 128>::kSmem) != cudaSuccess ||
                cudaFuncSetAttribute(append_kernel<144, 128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AppendShape<144, 128>::kSmem) != cudaSuccess ||
                cudaFuncSetAttribute(append_kernel<64, 64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AppendShape<64, 64>::kSmem) != cudaSuccess ||
                cudaFuncSetAttribute(append_kernel<64, 128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AppendShape<64, 128>::kSmem) != cudaSuccess ||
                cudaFuncSetAttribute(topk_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kTopkStageKeys * sizeof(uint32_t))) != cudaSuccess)
                return MLA_ERR_CUDA;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * (d.sms / 2), 1, 1);
            cfg.blockDim = dim3(kDecodeThreads, 1, 1);
            cfg.dynamicSmemBytes = kDecodeSmem;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int nc = 0;
            if (cudaOccupancyMaxActiveClusters(&nc, (const void *)decode_kernel, &cfg) != cudaSuccess || nc <= 0) {
                cudaGetLastError();
                nc = d.sms / 2;
            }
            d.clusters = nc < kMaxClusters ? nc : kMaxClusters;
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return MLA_ERR_CUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    if (!d.supported) return MLA_ERR_UNSUPPORTED;
    *dev_out = dev;
    *info_out = &d;
    return MLA_OK;
}

// 2-D bf16 tensor map: `rows` rows of `cols` elements, `row_bytes` apart; boxes of
// box_cols x box_rows with 128-byte swizzle (box_cols * 2 must be 128).
bool tmap_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
             uint32_t box_rows) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D view of a [rows, 576] bf16 array (the latent page pool, or the absorbed queries) for TMA:
// (64 columns, rows, 9 column blocks) with strides (2 B, 1152 B, 128 B).  A box of
// (64, box_rows, blocks) lands as `blocks` consecutive box_rows x 128-byte swizzled blocks.
bool tmap_row_blocks(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows, uint32_t blocks) {
    cuuint64_t dims[3] = {64, rows, (cuuint64_t)kBoxesS};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, 128};
    cuuint32_t box[3] = {64, box_rows, blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D view (64 columns, rows, blocks) of a [rows, 64 * blocks] bf16 array with strides (2 B,
// row bytes, 128 B): a box of (64, box_rows, box_blocks) lands as `box_blocks` consecutive
// box_rows x 128-byte swizzled blocks (the row-block view of mla_decode's pages, for any width)
bool tmap_col_blocks(CUtensorMap *m, const void *base, uint64_t rows, uint32_t blocks, uint32_t box_rows,
                     uint32_t box_blocks) {
    cuuint64_t dims[3] = {64, rows, blocks};
    cuuint64_t strides[2] = {(cuuint64_t)blocks * 128, 128};
    cuuint32_t box[3] = {64, box_rows, box_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor maps are encoded once per (device, array, rows, box) and reused: a decode step of a
// serving loop sees the same pool every call, and often the same query buffer.
struct MapEntry {
    int dev;
    const void *base;
    uint64_t rows;
    uint32_t box_rows, blocks;
    CUtensorMap map;
};
constexpr int kMapCache = 32;
MapEntry g_maps[kMapCache];
int g_maps_n = 0, g_maps_next = 0;
std::mutex g_map_mu;

bool map_cached(CUtensorMap *m, int dev, const void *base, uint64_t rows, uint32_t box_rows, uint32_t blocks) {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < g_maps_n; ++i) {
        const MapEntry &e = g_maps[i];
        if (e.dev == dev && e.base == base && e.rows == rows && e.box_rows == box_rows && e.blocks == blocks) {
            *m = e.map;
            return true;
        }
    }
    if (!tmap_row_blocks(m, base, rows, box_rows, blocks)) return false;
    MapEntry &e = g_maps[g_maps_next];
    e.dev = dev;
    e.base = base;
    e.rows = rows;
    e.box_rows = box_rows;
    e.blocks = blocks;
    e.map = *m;
    g_maps_next = (g_maps_next + 1) % kMapCache;
    if (g_maps_n < kMapCache) ++g_maps_n;
    return true;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
    size_t hdr, items, info, scratch, ring, part_lse, part_o, total;
    int max_items, max_slots;
};

bool ws_layout(int batch, int q_len, int num_splits, WsLayout *w) {
    if (batch < 1 || q_len < 1 || q_len > kMaxQLen || num_splits < 0 || num_splits > 4096) return false;
    const long long n_bt = (long long)batch * q_len;
    if (n_bt > kMaxRows) return false;
    long long mi = num_splits > 0 ? n_bt * num_splits : n_bt + kMaxClusters;
    if (mi > (1ll << 24)) return false;
    w->max_items = (int)mi;
    w->max_slots = (int)mi;
    size_t off = 0;
    w->hdr = off;
    off = align_up(off + sizeof(PlanHeader), 256);
    w->items = off;
    off = align_up(off + sizeof(Item) * (size_t)mi, 256);
    w->info = off;
    off = align_up(off + sizeof(BtInfo) * (size_t)n_bt, 256);
    w->scratch = off;  // the planner's per-query arrays, for batches too large for its shared memory
    off = align_up(off + (n_bt > kPlanSmemBt ? sizeof(int) * 4 * (size_t)n_bt : 0), 256);
    w->ring = off;  // P messages between the two CTAs of each pair
    off = align_up(off + (size_t)kMaxClusters * kRing * kMsgBytes, 256);
    w->part_lse = off;
    off = align_up(off + sizeof(float) * kHeads * (size_t)mi, 256);
    w->part_o = off;
    off = align_up(off + sizeof(float) * kHeads * kDc * (size_t)mi, 256);
    w->total = off;
    return true;
}

// Shape of the cache write for n_tokens new tokens: a few token tiles take 64-column tiles with K
// split over a cluster of up to 8 CTAs (72 CTAs for one tile), loading only 64 rows of h when
// there are at most 64 tokens; twelve or more token tiles fill the GPU by themselves and take
// 144-column tiles without a split.  chunk = K blocks per TMA copy: about a fifth of a split's K
// range, so the MMAs start on the first copy while the others land (all of them in flight when
// the stages hold them); two for the prompt shape, whose long K loop runs on three stages.
struct AppendConfig {
    int bn, arows, splits, chunk;
};
AppendConfig append_config(int n_tokens, int d_model) {
    const int tiles = (n_tokens + kAppendTileM - 1) / kAppendTileM;
    const int nkb = d_model / 64;
    if (tiles >= 12) return {144, 128, 1, nkb < 2 ? 1 : 2};
    int s = 1;
    while (2 * s <= kAppendMaxSplits && 2 * s * tiles <= kAppendMaxSplits && 2 * s <= nkb) s *= 2;
    const int arows = n_tokens <= 64 ? 64 : 128;
    const int nk_max = (nkb + s - 1) / s;
    const int cap = arows == 64 ? AppendShape<64, 64>::kMaxChunk : AppendShape<64, 128>::kMaxChunk;
    int c = (nk_max + 4) / 5;
    if (c > cap) c = cap;
    return {64, arows, s, c < 1 ? 1 : c};
}

// RoPE pair i turns by theta_i = base^(-2i/64) per position; as a fraction of a turn, theta_i / (2 pi)
// < 1, held as an unsigned 64-bit binary fraction (exact in double: the value is below 2^62)
uint64_t rope_turns(double base, int i) {
    const double rate = std::pow(base, -2.0 * i / 64.0) / (2.0 * 3.14159265358979323846);
    return (uint64_t)std::ldexp(rate, 64);
}

// One thread waits on a barrier that nothing completes; the bounded wait gives up.
__global__ void bounded_wait_probe_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        mbar_wait(smem_u32(&bar), 0u, &abort_flag, limit_ns);
    }
}

// kernels enqueued so far (see mla_test_launch_count)
std::atomic<uint64_t> g_launches{0};

mla_status_t launch_error(uint64_t kernels = 1) {
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    g_launches += kernels;
    return MLA_OK;
}

constexpr int kMaxTopK = 1 << 18;
constexpr int kSparseWholePages = 16;  // selections up to this many pages per sequence are not split

// Workspace of the indexer decode: scores, selection, compact pool and its table, then the
// decode's own workspace.
struct SparseWs {
    size_t scores, sel_index, sel_pool, sel_bt, sel_lens, dec, dec_bytes, total;
    int npk;
};
bool sparse_ws_layout(int batch, int max_pages, int k, SparseWs *w) {
    if (batch < 1 || batch > kMaxRows || max_pages < 1 || k < 1 || k > kMaxTopK) return false;
    if ((long long)max_pages * kPage > 0x7fffffffll) return false;
    w->npk = (k + kPage - 1) / kPage;
    const size_t dec0 = mla_decode_workspace_size(batch, 1, 0), dec1 = mla_decode_workspace_size(batch, 1, 1);
    const size_t dec = dec0 > dec1 ? dec0 : dec1;
    if (dec == 0) return false;
    size_t off = 0;
    w->scores = off;
    off = align_up(off + sizeof(float) * (size_t)batch * max_pages * kPage, 256);
    w->sel_index = off;
    off = align_up(off + sizeof(int32_t) * (size_t)batch * k, 256);
    w->sel_pool = off;
    off = align_up(off + (size_t)batch * w->npk * kPage * kSparseRow * 2, 256);
    w->sel_bt = off;
    off = align_up(off + sizeof(int32_t) * (size_t)batch * w->npk, 256);
    w->sel_lens = off;
    off = align_up(off + sizeof(int32_t) * (size_t)batch, 256);
    w->dec = off;
    w->dec_bytes = dec;
    w->total = off + dec;
    return true;
}

// The index-score launch for a bf16 index cache, or E4M3 codes with per-token scales.
mla_status_t index_scores_impl(const void *q_idx, const void *idx_pool, const float *idx_scale, bool e4m3,
                               const int32_t *block_table, const int32_t *seq_lens, int batch, int d_idx,
                               int num_pages, int max_pages, float *scores, mla_stream_t stream) {
    if (!q_idx || !idx_pool || !block_table || !seq_lens || !scores) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || num_pages < 1 || max_pages < 1) return MLA_ERR_INVALID_ARG;
    if (d_idx != 32 && d_idx != 64 && d_idx != 128 && d_idx != 256) return MLA_ERR_SHAPE;
    if (batch > kMaxRows || (long long)max_pages * kPage > 0x7fffffffll ||
        (long long)num_pages * kPage * d_idx > (1ll << 40))
        return MLA_ERR_SHAPE;
    if (!aligned16(q_idx) || !aligned16(idx_pool) || !aligned4(scores) || !aligned4(block_table) ||
        !aligned4(seq_lens) || (e4m3 && !aligned4(idx_scale)))
        return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    // about 32 warps per SM over the whole batch, each taking a few pages of one sequence
    const long long warps = (long long)info->sms * 32;
    const long long pages = (long long)batch * max_pages;
    const long long per_warp = pages <= warps ? 1 : (pages + warps - 1) / warps;
    const int wpc = kScoreThreads / 32;
    const int cps = (int)((max_pages + wpc * per_warp - 1) / (wpc * per_warp));
    ScoreParams p;
    p.q_idx = static_cast<const __nv_bfloat16 *>(q_idx);
    p.idx_pool = idx_pool;
    p.idx_scale = idx_scale;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.scores = scores;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.ctas_per_seq = cps;
    const dim3 grid((unsigned)((long long)batch * cps));
    cudaStream_t s = (cudaStream_t)stream;
    if (e4m3) {
        switch (d_idx) {
            case 32: index_score_kernel<2, true><<<grid, kScoreThreads, 0, s>>>(p); break;
            case 64: index_score_kernel<4, true><<<grid, kScoreThreads, 0, s>>>(p); break;
            case 128: index_score_kernel<8, true><<<grid, kScoreThreads, 0, s>>>(p); break;
            default: index_score_kernel<16, true><<<grid, kScoreThreads, 0, s>>>(p); break;
        }
    } else {
        switch (d_idx) {
            case 32: index_score_kernel<4, false><<<grid, kScoreThreads, 0, s>>>(p); break;
            case 64: index_score_kernel<8, false><<<grid, kScoreThreads, 0, s>>>(p); break;
            case 128: index_score_kernel<16, false><<<grid, kScoreThreads, 0, s>>>(p); break;
            default: index_score_kernel<32, false><<<grid, kScoreThreads, 0, s>>>(p); break;
        }
    }
    return launch_error();
}

// The decode launch: the split plan (unless the caller's kernel already wrote it into the
// workspace: one item per query), the decode, the LSE combine.  Arguments already checked.
mla_status_t decode_enqueue(const void *q_abs, const void *kv_pool, const int32_t *block_table,
                            const int32_t *seq_lens, int batch, int q_len, int num_pages, int max_pages, float scale,
                            int causal, int num_splits, void *o_lat, float *lse, uint8_t *ws, const WsLayout &w,
                            int dev, const DeviceInfo *info, bool run_plan, cudaStream_t s) {
    // pages: all 9 column blocks (score stage) or the 8 latent blocks (value stage) of one page;
    // queries: 4 content blocks of all 128 heads, or the RoPE block of 64 heads
    const uint64_t pool_rows = (uint64_t)num_pages * kPage, q_rows = (uint64_t)batch * q_len * kHeads;
    CUtensorMap tmap_s, tmap_v, tmap_qc, tmap_qr;
    if (!map_cached(&tmap_s, dev, kv_pool, pool_rows, kPage, kBoxesS) ||
        !map_cached(&tmap_v, dev, kv_pool, pool_rows, kPage, kBoxesV) ||
        !map_cached(&tmap_qc, dev, q_abs, q_rows, kHeads, 4) || !map_cached(&tmap_qr, dev, q_abs, q_rows, 64, 1))
        return MLA_ERR_CUDA;

    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(ws + w.hdr);
    Item *items = reinterpret_cast<Item *>(ws + w.items);
    BtInfo *bt_info = reinterpret_cast<BtInfo *>(ws + w.info);
    const int n_bt = batch * q_len;

    if (run_plan) {
        // one thread per query up to kPlanThreads (the rank sort wants that), in whole warps, at
        // least four: a small batch plans with few threads and few warps to synchronise
        const int plan_threads = n_bt >= kPlanThreads ? kPlanThreads : (n_bt <= 128 ? 128 : (n_bt + 31) / 32 * 32);
        // a programmatic dependent of whatever precedes it (it waits for that to complete before
        // reading anything): its launch overlaps the previous call's combine kernel
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3(1, 1, 1);
        pcfg.blockDim = dim3((unsigned)plan_threads, 1, 1);
        pcfg.stream = s;
        cudaLaunchAttribute pat[1];
        pat[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pat[0].val.programmaticStreamSerializationAllowed = 1;
        pcfg.attrs = pat;
        pcfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&pcfg, plan_kernel, seq_lens, batch, q_len, causal ? 1 : 0, max_pages, info->clusters,
                               num_splits, hdr, items, bt_info, reinterpret_cast<int *>(ws + w.scratch),
                               w.max_items, w.max_slots) != cudaSuccess) {
            cudaGetLastError();
            return MLA_ERR_CUDA;
        }
    }

    DecodeParams p;
    p.q_abs = static_cast<const __nv_bfloat16 *>(q_abs);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.o_lat = static_cast<__nv_bfloat16 *>(o_lat);
    p.lse = lse;
    p.hdr = hdr;
    p.items = items;
    p.part_o = reinterpret_cast<float *>(ws + w.part_o);
    p.part_lse = reinterpret_cast<float *>(ws + w.part_lse);
    p.ring = ws + w.ring;
    p.B = batch;
    p.Tq = q_len;
    p.causal = causal ? 1 : 0;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.max_items = w.max_items;
    p.sl2 = scale * 1.4426950408889634f;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * info->clusters, 1, 1);
    cfg.blockDim = dim3(kDecodeThreads, 1, 1);
    cfg.dynamicSmemBytes = kDecodeSmem;
    cfg.stream = s;
    // the decode and combine kernels are programmatic dependents of their predecessors: their
    // launch and prologue overlap the predecessor, and they wait for its results on the device
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, decode_kernel, tmap_s, tmap_v, tmap_qc, tmap_qr, p) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    cudaLaunchConfig_t ccfg = {};
    const int units = n_bt * (kHeads / kCombineHeads);
    ccfg.gridDim = dim3(units < 2 * info->sms ? units : 2 * info->sms, 1, 1);
    ccfg.blockDim = dim3(kCombineThreads, 1, 1);
    ccfg.stream = s;
    ccfg.attrs = &at[1];
    ccfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&ccfg, combine_kernel, (const PlanHeader *)hdr, (const BtInfo *)bt_info, (const float *)p.part_o,
                           (const float *)p.part_lse, p.o_lat, lse) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    g_launches += run_plan ? 3 : 2;  // plan, decode, combine
    return MLA_OK;
}
// (end of the decode launch code)

// The top-k launch (arguments already checked).  plan_ws != null: the kernel also writes the
// decode plan of its output into that decode workspace (layout w): one whole item per sequence.
mla_status_t topk_enqueue(const float *scores, const int32_t *seq_lens, const void *kv_pool,
                          const int32_t *block_table, int batch, int num_pages, int max_pages, int k,
                          int32_t *sel_index, void *sel_pool, int32_t *sel_block_table, int32_t *sel_lens,
                          uint8_t *plan_ws, int plan_max_items, int plan_max_slots, cudaStream_t s,
                          const WsLayout *w = nullptr) {
    TopkParams p;
    p.scores = scores;
    p.seq_lens = seq_lens;
    p.kv_pool = static_cast<const __nv_bfloat16 *>(kv_pool);
    p.block_table = block_table;
    p.sel_index = sel_index;
    p.sel_pool = static_cast<__nv_bfloat16 *>(sel_pool);
    p.sel_block_table = sel_block_table;
    p.sel_lens = sel_lens;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.k = k;
    p.npk = (k + kPage - 1) / kPage;
    p.plan_hdr = plan_ws && w ? reinterpret_cast<PlanHeader *>(plan_ws + w->hdr) : nullptr;
    p.plan_items = plan_ws && w ? reinterpret_cast<Item *>(plan_ws + w->items) : nullptr;
    p.plan_info = plan_ws && w ? reinterpret_cast<BtInfo *>(plan_ws + w->info) : nullptr;
    p.plan_max_items = plan_max_items;
    p.plan_max_slots = plan_max_slots;
    // the largest slice any CTA can own (a sequence of max_pages * 64 tokens): staged in shared
    // memory when it fits
    const long long max_chunk = (((long long)max_pages * kPage + kTopkCluster - 1) / kTopkCluster + 3) & ~3ll;
    p.staged = max_chunk <= kTopkStageKeys ? 1 : 0;
    const size_t dyn = p.staged ? (size_t)max_chunk * sizeof(uint32_t) : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(batch * kTopkCluster), 1, 1);
    cfg.blockDim = dim3(kTopkThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kTopkCluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, topk_gather_kernel, p) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    g_launches += 1;
    return MLA_OK;
}

// Device address of the library-owned decode scratch on each device, looked up once.
void *g_scratch_addr[kMaxDevices] = {};

}  // namespace

// Scratch for mla_decode_static_scratch: lives in the library's own device memory, so
// that entry point never allocates.  Every device that loads the library holds it until
// the process exits.  Host code must not pass this name to a kernel: on the host it is
// only a stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_decode_scratch[MLA_STATIC_SCRATCH_BYTES];

}  // namespace mla

using namespace mla;

extern "C" {

int mla_version(void) { return 100; }

const char *mla_status_string(mla_status_t s) {
    switch (s) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
        case MLA_ERR_SHAPE: return "MLA_ERR_SHAPE";
        case MLA_ERR_ALIGNMENT: return "MLA_ERR_ALIGNMENT";
        case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
        case MLA_ERR_DEVICE_FAULT: return "MLA_ERR_DEVICE_FAULT";
    }
    return "MLA_ERR_UNKNOWN";
}

uint64_t mla_cache_bytes(int64_t tokens, int layers, int d_c, int d_r, int bytes_per_elem) {
    if (tokens < 0 || layers < 0 || d_c < 0 || d_r < 0 || bytes_per_elem < 0) return 0;
    return (uint64_t)tokens * (uint64_t)layers * (uint64_t)(d_c + d_r) * (uint64_t)bytes_per_elem;
}

size_t mla_decode_workspace_size(int batch, int q_len, int num_splits) {
    WsLayout w;
    if (!ws_layout(batch, q_len, num_splits, &w)) return 0;
    return w.total;
}

mla_status_t mla_cache_append(const void *h, const void *w_dkv, const void *w_kr, const int32_t *block_table,
                              const int32_t *seq_lens, int batch, int q_len, int d_model, int num_pages,
                              int max_pages, float rope_base, void *kv_pool, mla_stream_t stream) {
    if (!h || !w_dkv || !w_kr || !block_table || !seq_lens || !kv_pool) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || q_len < 1 || num_pages < 1 || max_pages < 1) return MLA_ERR_INVALID_ARG;
    if (!(rope_base > 1.f) || !std::isfinite(rope_base)) return MLA_ERR_INVALID_ARG;
    const long long n_tokens = (long long)batch * q_len;
    if (n_tokens > kMaxAppendTokens || d_model < 64 || d_model % 64 != 0 || d_model > kMaxDModel) return MLA_ERR_SHAPE;
    if ((long long)num_pages * kPage > 0x7fffffffll || (long long)max_pages * kPage > 0x7fffffffll) return MLA_ERR_SHAPE;
    if (!aligned16(h) || !aligned16(w_dkv) || !aligned16(w_kr) || !aligned16(kv_pool) || !aligned4(block_table) ||
        !aligned4(seq_lens))
        return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    const AppendConfig cf = append_config((int)n_tokens, d_model);
    const uint32_t nkb = (uint32_t)(d_model / 64);
    CUtensorMap th, twa, twb, twr;
    if (!tmap_col_blocks(&th, h, (uint64_t)n_tokens, nkb, (uint32_t)cf.arows, (uint32_t)cf.chunk) ||
        !tmap_col_blocks(&twa, w_dkv, kAppendLatent, nkb, (uint32_t)cf.bn, (uint32_t)cf.chunk) ||
        !tmap_col_blocks(&twr, w_kr, kAppendCols - kAppendLatent, nkb, kAppendCols - kAppendLatent,
                         (uint32_t)cf.chunk))
        return MLA_ERR_CUDA;
    if (kAppendLatent % cf.bn == 0)
        twb = twa;  // no column tile straddles the two matrices
    else if (!tmap_col_blocks(&twb, w_dkv, kAppendLatent, nkb, (uint32_t)(kAppendLatent % cf.bn), (uint32_t)cf.chunk))
        return MLA_ERR_CUDA;
    AppendParams p;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.pool = static_cast<__nv_bfloat16 *>(kv_pool);
    p.n_tokens = (int)n_tokens;
    p.q_len = q_len;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.nkb = d_model / 64;
    p.splits = cf.splits;
    p.chunk = cf.chunk;
    p.m = 1;
    for (int i = 0; i < kAppendPairs; ++i) p.turns[i] = rope_turns((double)rope_base, i);
    const unsigned token_tiles = (unsigned)((n_tokens + kAppendTileM - 1) / kAppendTileM);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kAppendThreads, 1, 1);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cf.splits;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (cf.bn == 64 && cf.arows == 64) {
        cfg.gridDim = dim3((unsigned)cf.splits, AppendShape<64, 64>::kColTiles, token_tiles);
        cfg.dynamicSmemBytes = AppendShape<64, 64>::kSmem;
        e = cudaLaunchKernelEx(&cfg, append_kernel<64, 64, false>, th, twa, twb, twr, p);
    } else if (cf.bn == 64) {
        cfg.gridDim = dim3((unsigned)cf.splits, AppendShape<64, 128>::kColTiles, token_tiles);
        cfg.dynamicSmemBytes = AppendShape<64, 128>::kSmem;
        e = cudaLaunchKernelEx(&cfg, append_kernel<64, 128, false>, th, twa, twb, twr, p);
    } else {
        cfg.gridDim = dim3(1, AppendShape<144, 128>::kColTiles, token_tiles);
        cfg.dynamicSmemBytes = AppendShape<144, 128>::kSmem;
        e = cudaLaunchKernelEx(&cfg, append_kernel<144, 128, false>, th, twa, twb, twr, p);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    return launch_error(1);
}

mla_status_t mla_cache_append_compressed(const void *h, const void *w_dkv, const void *w_kr, const void *w_z,
                                         const int32_t *block_table, const int32_t *seq_lens, int batch, int n_blocks,
                                         int m, int d_model, int num_pages, int max_pages, float rope_base,
                                         void *kv_pool, mla_stream_t stream) {
    if (!h || !w_dkv || !w_kr || !w_z || !block_table || !seq_lens || !kv_pool) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || n_blocks < 1 || num_pages < 1 || max_pages < 1) return MLA_ERR_INVALID_ARG;
    if (m < 1 || m > kAppendTileM || (m & (m - 1)) != 0) return MLA_ERR_INVALID_ARG;
    if (!(rope_base > 1.f) || !std::isfinite(rope_base)) return MLA_ERR_INVALID_ARG;
    const long long n_tokens = (long long)batch * n_blocks * m;
    if (n_tokens > kMaxAppendTokens || d_model < 64 || d_model % 64 != 0 || d_model > kMaxDModel) return MLA_ERR_SHAPE;
    if ((long long)num_pages * kPage > 0x7fffffffll || (long long)max_pages * kPage > 0x7fffffffll) return MLA_ERR_SHAPE;
    if (!aligned16(h) || !aligned16(w_dkv) || !aligned16(w_kr) || !aligned16(w_z) || !aligned16(kv_pool) ||
        !aligned4(block_table) || !aligned4(seq_lens))
        return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    // 64-column tiles of 32 row components and their 32 z components; K split over a cluster of
    // at most 4 CTAs (so the 18 column tiles' clusters all fit at once), which share the merge by
    // components
    const int tiles = (int)((n_tokens + kAppendTileM - 1) / kAppendTileM);
    const int nkb = d_model / 64;
    const int arows = n_tokens <= 64 ? 64 : 128;
    int sp = 1;
    while (2 * sp <= 4 && 2 * sp * tiles <= kAppendMaxSplits && 2 * sp <= nkb) sp *= 2;
    const int nk_max = (nkb + sp - 1) / sp;
    const int cap = arows == 64 ? AppendShape<64, 64>::kMaxChunk : AppendShape<64, 128>::kMaxChunk;
    int chunk = (nk_max + 4) / 5;
    if (chunk > cap) chunk = cap;
    if (chunk < 1) chunk = 1;
    CUtensorMap th, twa, twz, twr;
    if (!tmap_col_blocks(&th, h, (uint64_t)n_tokens, (uint32_t)nkb, (uint32_t)arows, (uint32_t)chunk) ||
        !tmap_col_blocks(&twa, w_dkv, kAppendLatent, (uint32_t)nkb, 32, (uint32_t)chunk) ||
        !tmap_col_blocks(&twr, w_kr, kAppendCols - kAppendLatent, (uint32_t)nkb, 32, (uint32_t)chunk) ||
        !tmap_col_blocks(&twz, w_z, kAppendCols, (uint32_t)nkb, 32, (uint32_t)chunk))
        return MLA_ERR_CUDA;
    AppendParams p;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.pool = static_cast<__nv_bfloat16 *>(kv_pool);
    p.n_tokens = (int)n_tokens;
    p.q_len = n_blocks;
    p.num_pages = num_pages;
    p.max_pages = max_pages;
    p.nkb = nkb;
    p.splits = sp;
    p.chunk = chunk;
    p.m = m;
    for (int i = 0; i < kAppendPairs; ++i) p.turns[i] = rope_turns((double)rope_base, i);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kAppendThreads, 1, 1);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)sp;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)sp, kAppendCols / 32, (unsigned)tiles);
    cfg.dynamicSmemBytes = AppendShape<64, 64>::kSmem;
    cudaError_t e = arows == 64 ? cudaLaunchKernelEx(&cfg, append_kernel<64, 64, true>, th, twa, twz, twr, p)
                                : cudaLaunchKernelEx(&cfg, append_kernel<64, 128, true>, th, twa, twz, twr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    return launch_error(1);
}

// 3-D bf16 view (cols, heads, tokens) of a [tokens, 128, cols] output for the GEMMs' TMA stores:
// boxes of 128 columns x 1 head x 128 tokens, no swizzle (the staged tile is plain row-major)
bool tmap_out(CUtensorMap *m, const void *base, uint64_t cols, uint64_t n_tokens) {
    cuuint64_t dims[3] = {cols, (cuuint64_t)kHeads, n_tokens};
    cuuint64_t strides[2] = {cols * 2, cols * 2 * kHeads};
    cuuint32_t box[3] = {128, 1, (cuuint32_t)kGemmTileN};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

mla_status_t mla_absorb_q(const void *q_nope, const void *q_rope, const void *w_uk, void *q_abs, int n_tokens,
                          int n_heads, mla_stream_t stream) {
    if (!q_nope || !q_rope || !w_uk || !q_abs) return MLA_ERR_INVALID_ARG;
    if (n_tokens < 1) return MLA_ERR_INVALID_ARG;
    if (n_heads != kHeads) return MLA_ERR_UNSUPPORTED;
    if (n_tokens > kMaxRows) return MLA_ERR_SHAPE;
    if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_abs)) return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    CUtensorMap tw, tx, to;
    if (!tmap_col_blocks(&tw, w_uk, (uint64_t)kHeads * 128, kDc / 64, 64, kDc / 64)) return MLA_ERR_CUDA;
    if (!tmap_2d(&tx, q_nope, (uint64_t)kHeads * 128, (uint64_t)n_tokens, (uint64_t)kHeads * 128 * 2, 64, 128))
        return MLA_ERR_CUDA;
    if (!tmap_out(&to, q_abs, kD, (uint64_t)n_tokens)) return MLA_ERR_CUDA;
    GemmParams p;
    p.mode = kModeAbsorb;
    p.n_tokens = n_tokens;
    p.q_rope = static_cast<const __nv_bfloat16 *>(q_rope);
    p.q_abs = static_cast<__nv_bfloat16 *>(q_abs);
    dim3 grid(kHeads, (n_tokens + kGemmTileN - 1) / kGemmTileN);
    head_gemm_kernel<<<grid, kGemmThreads, gemm_smem(kAbsorbRegion), (cudaStream_t)stream>>>(tw, tx, to, p);
    return launch_error();
}

mla_status_t mla_up_proj(const void *o_lat, const void *w_uv, void *out, int n_tokens, int n_heads,
                         mla_stream_t stream) {
    if (!o_lat || !w_uv || !out) return MLA_ERR_INVALID_ARG;
    if (n_tokens < 1) return MLA_ERR_INVALID_ARG;
    if (n_heads != kHeads) return MLA_ERR_UNSUPPORTED;
    if (n_tokens > kMaxRows) return MLA_ERR_SHAPE;
    if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    CUtensorMap tw, tx, to;
    if (!tmap_2d(&tw, w_uv, kDc, (uint64_t)kHeads * 128, kDc * 2, 64, 128)) return MLA_ERR_CUDA;
    if (!tmap_2d(&tx, o_lat, (uint64_t)kHeads * kDc, (uint64_t)n_tokens, (uint64_t)kHeads * kDc * 2, 64, 128))
        return MLA_ERR_CUDA;
    if (!tmap_out(&to, out, 128, (uint64_t)n_tokens)) return MLA_ERR_CUDA;
    GemmParams p;
    p.mode = kModeUpProj;
    p.n_tokens = n_tokens;
    p.q_rope = nullptr;
    p.q_abs = nullptr;
    dim3 grid(kHeads, (n_tokens + kGemmTileN - 1) / kGemmTileN);
    head_gemm_kernel<<<grid, kGemmThreads, gemm_smem(kUpRegion), (cudaStream_t)stream>>>(tw, tx, to, p);
    return launch_error();
}

mla_status_t mla_decode(const void *q_abs, const void *kv_pool, const int32_t *block_table, const int32_t *seq_lens,
                        int batch, int q_len, int n_heads, int num_pages, int max_pages, float scale, int causal,
                        int num_splits, void *o_lat, float *lse, void *workspace, size_t workspace_bytes,
                        mla_stream_t stream) {
    if (!q_abs || !kv_pool || !block_table || !seq_lens || !o_lat || !lse) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || q_len < 1 || num_pages < 1 || max_pages < 1 || num_splits < 0) return MLA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return MLA_ERR_INVALID_ARG;
    if (n_heads != kHeads) return MLA_ERR_UNSUPPORTED;
    if (q_len > kMaxQLen || (long long)batch * q_len > kMaxRows) return MLA_ERR_SHAPE;
    if ((long long)num_pages * kPage > 0x7fffffffll || (long long)max_pages * kPage > 0x7fffffffll) return MLA_ERR_SHAPE;
    if (!aligned16(q_abs) || !aligned16(kv_pool) || !aligned16(o_lat) || !aligned4(lse) || !aligned4(block_table) ||
        !aligned4(seq_lens))
        return MLA_ERR_ALIGNMENT;
    WsLayout w;
    if (!ws_layout(batch, q_len, num_splits, &w)) return MLA_ERR_SHAPE;
    if (!workspace || workspace_bytes < w.total) return MLA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;

    return decode_enqueue(q_abs, kv_pool, block_table, seq_lens, batch, q_len, num_pages, max_pages, scale, causal,
                          num_splits, o_lat, lse, static_cast<uint8_t *>(workspace), w, dev, info, true,
                          (cudaStream_t)stream);
}

mla_status_t mla_decode_static_scratch(const void *q_abs, const void *kv_pool, const int32_t *block_table,
                                       const int32_t *seq_lens, int batch, int q_len, int n_heads, int num_pages,
                                       int max_pages, float scale, int causal, int num_splits, void *o_lat,
                                       float *lse, mla_stream_t stream) {
    const size_t need = mla_decode_workspace_size(batch, q_len, num_splits);
    if (need == 0)  // sizes mla_decode itself rejects: let it report the reason
        return mla_decode(q_abs, kv_pool, block_table, seq_lens, batch, q_len, n_heads, num_pages, max_pages,
                          scale, causal, num_splits, o_lat, lse, nullptr, 0, stream);
    if (need > (size_t)MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_scratch_addr[dev] == nullptr) {
            // first call on this device (which is current): find where the array lives
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_decode_scratch) != cudaSuccess || addr == nullptr) {
                cudaGetLastError();
                return MLA_ERR_CUDA;
            }
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    return mla_decode(q_abs, kv_pool, block_table, seq_lens, batch, q_len, n_heads, num_pages, max_pages, scale,
                      causal, num_splits, o_lat, lse, scratch, (size_t)MLA_STATIC_SCRATCH_BYTES, stream);
}

mla_status_t mla_combine(const float *o_parts, const float *lse_parts, int n_parts, int rows, void *o_out,
                         float *lse_out, mla_stream_t stream) {
    if (!o_parts || !lse_parts || !o_out || !lse_out) return MLA_ERR_INVALID_ARG;
    if (n_parts < 1 || rows < 1) return MLA_ERR_INVALID_ARG;
    if (!aligned16(o_parts) || !aligned4(lse_parts) || !aligned16(o_out) || !aligned4(lse_out))
        return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    combine_rows_kernel<<<(rows + kCombineHeads - 1) / kCombineHeads, kCombineThreads, 0, (cudaStream_t)stream>>>(
        o_parts, lse_parts, n_parts, rows, static_cast<__nv_bfloat16 *>(o_out), lse_out);
    return launch_error();
}

mla_status_t mla_index_scores(const void *q_idx, const void *idx_pool, const int32_t *block_table,
                              const int32_t *seq_lens, int batch, int d_idx, int num_pages, int max_pages,
                              float *scores, mla_stream_t stream) {
    return index_scores_impl(q_idx, idx_pool, nullptr, false, block_table, seq_lens, batch, d_idx, num_pages,
                             max_pages, scores, stream);
}

mla_status_t mla_index_scores_e4m3(const void *q_idx, const void *idx_codes, const float *idx_scale,
                                   const int32_t *block_table, const int32_t *seq_lens, int batch, int d_idx,
                                   int num_pages, int max_pages, float *scores, mla_stream_t stream) {
    if (!idx_scale) return MLA_ERR_INVALID_ARG;
    return index_scores_impl(q_idx, idx_codes, idx_scale, true, block_table, seq_lens, batch, d_idx, num_pages,
                             max_pages, scores, stream);
}

mla_status_t mla_topk_gather(const float *scores, const int32_t *seq_lens, const void *kv_pool,
                             const int32_t *block_table, int batch, int num_pages, int max_pages, int k,
                             int32_t *sel_index, void *sel_pool, int32_t *sel_block_table, int32_t *sel_lens,
                             mla_stream_t stream) {
    if (!scores || !seq_lens || !kv_pool || !block_table || !sel_index || !sel_pool || !sel_block_table || !sel_lens)
        return MLA_ERR_INVALID_ARG;
    if (batch < 1 || num_pages < 1 || max_pages < 1 || k < 1) return MLA_ERR_INVALID_ARG;
    if (k > kMaxTopK || batch > kMaxRows || (long long)max_pages * kPage > 0x7fffffffll) return MLA_ERR_SHAPE;
    if (!aligned16(scores) || !aligned16(kv_pool) || !aligned16(sel_pool) || !aligned4(seq_lens) ||
        !aligned4(block_table) || !aligned4(sel_index) || !aligned4(sel_block_table) || !aligned4(sel_lens))
        return MLA_ERR_ALIGNMENT;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    return topk_enqueue(scores, seq_lens, kv_pool, block_table, batch, num_pages, max_pages, k, sel_index, sel_pool,
                        sel_block_table, sel_lens, nullptr, 0, 0, (cudaStream_t)stream);
}

size_t mla_decode_sparse_workspace_size(int batch, int max_pages, int k) {
    SparseWs w;
    if (!sparse_ws_layout(batch, max_pages, k, &w)) return 0;
    return w.total;
}

mla_status_t mla_decode_sparse(const void *q_abs, const void *q_idx, const void *kv_pool, const void *idx_pool,
                               const float *idx_scale, const int32_t *block_table, const int32_t *seq_lens,
                               int batch, int n_heads, int d_idx, int num_pages, int max_pages, int k, float scale,
                               void *o_lat, float *lse, int32_t *sel_index, void *workspace,
                               size_t workspace_bytes, mla_stream_t stream) {
    if (!q_abs || !q_idx || !kv_pool || !idx_pool || !block_table || !seq_lens || !o_lat || !lse)
        return MLA_ERR_INVALID_ARG;
    if (batch < 1 || num_pages < 1 || max_pages < 1 || k < 1) return MLA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return MLA_ERR_INVALID_ARG;
    if (n_heads != kHeads) return MLA_ERR_UNSUPPORTED;
    if (d_idx != 32 && d_idx != 64 && d_idx != 128 && d_idx != 256) return MLA_ERR_SHAPE;
    SparseWs w;
    if (!sparse_ws_layout(batch, max_pages, k, &w)) return MLA_ERR_SHAPE;
    if ((long long)batch * w.npk > 0x7fffffffll / kPage) return MLA_ERR_SHAPE;
    if (!workspace || workspace_bytes < w.total) return MLA_ERR_WORKSPACE;
    if (!aligned16(workspace) || !aligned16(q_abs) || !aligned16(o_lat) || !aligned4(lse) ||
        (sel_index && !aligned4(sel_index)))
        return MLA_ERR_ALIGNMENT;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *scores = reinterpret_cast<float *>(ws + w.scores);
    int32_t *sel = sel_index ? sel_index : reinterpret_cast<int32_t *>(ws + w.sel_index);
    void *sel_pool = ws + w.sel_pool;
    int32_t *sel_bt = reinterpret_cast<int32_t *>(ws + w.sel_bt);
    int32_t *sel_lens = reinterpret_cast<int32_t *>(ws + w.sel_lens);
    mla_status_t st = index_scores_impl(q_idx, idx_pool, idx_scale, idx_scale != nullptr, block_table, seq_lens,
                                        batch, d_idx, num_pages, max_pages, scores, stream);
    if (st != MLA_OK) return st;
    // A selection of at most 16 pages per sequence is decoded whole, one item per sequence (split
    // into pieces, each piece's fp32 partial epilogue and the merge cost more than its pages).
    // That plan is written by the top-k kernel itself, so the decode needs no plan launch.
    const bool whole = w.npk <= kSparseWholePages;
    if (!whole) {
        st = mla_topk_gather(scores, seq_lens, kv_pool, block_table, batch, num_pages, max_pages, k, sel, sel_pool,
                             sel_bt, sel_lens, stream);
        if (st != MLA_OK) return st;
        return mla_decode(q_abs, sel_pool, sel_bt, sel_lens, batch, 1, n_heads, batch * w.npk, w.npk, scale, 0, 0,
                          o_lat, lse, ws + w.dec, w.dec_bytes, stream);
    }
    int dev;
    DeviceInfo *info;
    st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    WsLayout dl;
    if (!ws_layout(batch, 1, 1, &dl) || dl.total > w.dec_bytes) return MLA_ERR_SHAPE;
    cudaStream_t s = (cudaStream_t)stream;
    st = topk_enqueue(scores, seq_lens, kv_pool, block_table, batch, num_pages, max_pages, k, sel, sel_pool, sel_bt,
                      sel_lens, ws + w.dec, dl.max_items, dl.max_slots, s, &dl);
    if (st != MLA_OK) return st;
    return decode_enqueue(q_abs, sel_pool, sel_bt, sel_lens, batch, 1, batch * w.npk, w.npk, scale, 0, 1, o_lat, lse,
                          ws + w.dec, dl, dev, info, false, s);
}

mla_status_t mla_test_bounded_wait(int limit_ms, mla_stream_t stream) {
    if (limit_ms < 1 || limit_ms > 10000) return MLA_ERR_INVALID_ARG;
    int dev;
    DeviceInfo *info;
    mla_status_t st = device_setup(&dev, &info);
    if (st != MLA_OK) return st;
    bounded_wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ms * 1000000ull);
    return launch_error();
}

#ifdef MLA_TRACE
// Timeline build only: where the kernels write their per-warp event records (see Tracer).
int mla_trace_set(void *buf) { return cudaMemcpyToSymbol(g_trace, &buf, sizeof(buf)) == cudaSuccess ? 0 : 6; }
#endif

uint64_t mla_test_launch_count(void) { return g_launches.load(); }

mla_status_t mla_get_device_status(mla_stream_t stream, uint32_t *err_word) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MLA_ERR_CUDA;
    uint32_t v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_status, &z, sizeof(z)) != cudaSuccess) return MLA_ERR_CUDA;
    if (err_word) *err_word = v;
    return v ? MLA_ERR_DEVICE_FAULT : MLA_OK;
}

}  // extern "C"
