// gemm_kernels.cuh - per-head tcgen05 GEMMs around the decode:
//   absorb:  q_abs[n,h,0:512] = W_UK[h]^T q_nope[n,h,:]      ("DeepSeek-V2" explainer, Step 6)
//            q_abs[n,h,512:576] = q_rope[n,h,:]              (Step 7: RoPE query passes through)
//   up-proj: out[n,h,:] = W_UV[h] o_lat[n,h,:]                (Step 5 values, applied after attention)
//
// Both are computed transposed so that the 128-row tensor-core M dimension is filled by weight
// rows even for a handful of tokens: D^T[m, n] with m over the weight dimension (a 128-wide
// latent chunk, or the 128 head dims) and n over a 128-token tile.  One CTA per (head, token
// tile) streams that head's whole weight matrix once:
//   absorb:  K = d_h = 128 in two 64-wide chunks; each stage holds W_UK[h]^T for all 512 latent
//            columns (four MN-major 128 x 64 tiles) and the token tile; the four 128-column
//            accumulators fill the 512 TMEM columns;
//   up-proj: K = d_c = 512 in eight 64-wide chunks through a ring of stages; one accumulator.
// The epilogue converts each 128 x 128 accumulator to bf16 in shared memory, laid out as the
// output's rows (token-major), and writes it with one TMA tensor store: the weight index m is
// the output's contiguous dimension, so a thread that owns one m (one TMEM lane) cannot write
// contiguous bytes by itself.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mla {

constexpr int kGemmTileN = 128;                        // tokens per CTA
constexpr uint32_t kGemmTileBytes = 128u * 64u * 2u;   // one 128 x 64 bf16 operand tile (16 KB)
constexpr int kAbsorbAcc = 4;                          // absorb: 128-wide latent chunks per CTA (all 512 latent)
constexpr uint32_t kAbsorbStage = (kAbsorbAcc + 1) * kGemmTileBytes;  // the W_UK^T tiles + the token tile
constexpr int kAbsorbStages = 2;                       // = the two K chunks: everything in flight
constexpr uint32_t kUpStage = 2u * kGemmTileBytes;     // W_UV tile + the token tile
constexpr int kUpStages = 5;
constexpr uint32_t kOutTileBytes = 128u * 128u * 2u;   // one bf16 output tile: 128 tokens x 128 columns
constexpr uint32_t kAbsorbRegion = kAbsorbStages * kAbsorbStage;  // 160 KB
constexpr uint32_t kUpRegion = kUpStages * kUpStage;              // 160 KB
static_assert(kAbsorbAcc * kOutTileBytes <= kAbsorbRegion && kOutTileBytes <= kUpRegion,
              "output staging exceeds the stage region");
// shared memory: the mode's stage region, then the barriers (+ slack to align the base)
constexpr uint32_t gemm_smem(uint32_t region) { return region + 256 + 1024; }
constexpr uint32_t kGemmSmemMax = gemm_smem(kUpRegion);
constexpr int kModeAbsorb = 0, kModeUpProj = 1;
constexpr int kGemmThreads = 192;  // warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 epilogue

struct GemmParams {
    int mode;
    int n_tokens;
    const __nv_bfloat16 *q_rope;  // absorb only: [N, 128, 64], copied into q_abs[..., 512:576]
    __nv_bfloat16 *q_abs;         // absorb only: [N, 128, 576]
};

__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t smem_src, int32_t x, int32_t y, int32_t z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(smem_src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// grid (128 heads, token tiles), kGemmThreads threads.
//   tmap_w: absorb: W_UK as (64 latent, (h, d) rows, 8 latent blocks) (64 x 64 x 8 boxes); up-proj: W_UV as
//           [(h, d) rows, 512 latent] (64 latent x 128 rows boxes)
//   tmap_x: absorb: q_nope as [tokens, (h, d)]; up-proj: o_lat as [tokens, (h, latent)] (64 x 128 boxes)
//   tmap_o: the output as (columns, heads, tokens): absorb q_abs (576, 128, N), up-proj out
//           (128, 128, N); boxes of 128 columns x 1 head x 128 tokens
__global__ void __launch_bounds__(kGemmThreads, 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                 const __grid_constant__ CUtensorMap tmap_o, const GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool absorb = p.mode == kModeAbsorb;
    const int h = blockIdx.x, nt = blockIdx.y;
    const int nk = absorb ? 2 : 8;                       // 64-wide K chunks
    const int stages = absorb ? kAbsorbStages : kUpStages;
    const uint32_t stage_bytes = absorb ? kAbsorbStage : kUpStage;
    const int n_acc = absorb ? kAbsorbAcc : 1;           // 128-column accumulators
    const uint32_t kGemmOffBar = absorb ? kAbsorbRegion : kUpRegion;
    const uint32_t tmem_cols = absorb ? 512u : 128u;
    // barriers: full[0..4], empty[5..9], acc (all MMAs done) 10, staged (epilogue tile written) 11,
    // rope 12, drain 13
    auto bar = [&](int i) { return base + kGemmOffBar + 8u * i; };
    volatile int *abort = reinterpret_cast<volatile int *>(smem_raw + (base - raw) + kGemmOffBar + 128);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + kGemmOffBar + 120);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 5; ++s) {
            mbar_init(bar(s), 1);
            mbar_init(bar(5 + s), 1);
        }
        mbar_init(bar(10), 1);
        mbar_init(bar(11), 128);
        mbar_init(bar(12), 1);
        mbar_init(bar(13), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(base + kGemmOffBar + 120, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_o);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the producer and MMA roles run as whole warps that wait together (a lone waiting thread
    // wakes up late); lane 0 issues the copies and the MMAs
    if (warp == 0) {
        uint32_t issued = 0;
        for (int kc = 0; kc < nk; ++kc, ++issued) {
            const int s = kc % stages;
            if (__any_sync(0xffffffffu, !mbar_wait(bar(5 + s), ((kc / stages) & 1) ^ 1, abort))) break;
            if (lane == 0) {
                const uint32_t a = base + s * stage_bytes;
                mbar_arrive_expect_tx(bar(s), stage_bytes);
                if (absorb) {
                    // W_UK viewed as (64 latent columns, (h, d) rows, 8 latent blocks): one box of 64 d
                    // rows x all 512 latent columns lands as eight 64 x 64 blocks, i.e. four MN-major
                    // 128 (latent) x 64 (d) tiles
                    tma_load_3d_nohint(a, &tmap_w, 0, h * 128 + kc * 64, 0, bar(s));
                    // q_nope viewed as [tokens, (h, d)]: 128 tokens x 64 d
                    tma_load_2d(a + kAbsorbAcc * kGemmTileBytes, &tmap_x, h * 128 + kc * 64, nt * kGemmTileN, bar(s));
                } else {
                    // W_UV viewed as [(h, d) rows, 512 latent columns]: 128 d x 64 latent
                    tma_load_2d(a, &tmap_w, kc * 64, h * 128, bar(s));
                    // o_lat viewed as [tokens, (h, latent)]: 128 tokens x 64 latent
                    tma_load_2d(a + kGemmTileBytes, &tmap_x, h * 512 + kc * 64, nt * kGemmTileN, bar(s));
                }
            }
            __syncwarp();
        }
        // wait for the last loads (normal exit or abort) before the CTA may move on
        if (lane == 0)
            for (uint32_t k = issued > (uint32_t)stages ? issued - stages : 0; k < issued; ++k)
                if (!mbar_wait_drain(bar(k % stages), (k / stages) & 1)) break;
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t idesc = absorb ? idesc_bf16_f32(128, 128, 1, 0) : idesc_bf16_f32(128, 128, 0, 0);
        for (int kc = 0; kc < nk; ++kc) {
            const int s = kc % stages;
            if (__any_sync(0xffffffffu, !mbar_wait(bar(s), (kc / stages) & 1, abort))) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t a = base + s * stage_bytes;
                const uint32_t b = a + (absorb ? (uint32_t)kAbsorbAcc : 1u) * kGemmTileBytes;
                for (int mc = 0; mc < n_acc; ++mc) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // absorb: A = W_UK^T chunk, MN-major (latent contiguous), K = 16 d rows per step
                        // up-proj: A = W_UV chunk, K-major (latent contiguous along K)
                        const uint64_t adesc = absorb ? sdesc_sw128(a + mc * kGemmTileBytes + 2048u * k, 8192u, 1024u)
                                                      : sdesc_sw128(a + 32u * k, 16u, 1024u);
                        const uint64_t bdesc = sdesc_sw128(b + 32u * k, 16u, 1024u);
                        mma_ss(tmem + 128u * mc, adesc, bdesc, idesc, (kc | k) != 0);
                    }
                }
                mma_commit(bar(5 + s));
            }
            __syncwarp();
        }
        if (lane == 0) {
            mma_commit(bar(10));
            // every MMA issued has completed before the CTA may free its tensor memory
            mma_commit(bar(13));
            mbar_wait_drain(bar(13), 0);
        }
        __syncwarp();
    } else {
        // epilogue: warps 2..5 -> TMEM lane quadrants 2, 3, 0, 1; lane = weight-side index m
        const int q = warp & 3;
        const int m = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int et = threadIdx.x - 64;  // 0..127
        if (absorb) {
            // the RoPE query, unchanged, into q_abs[..., 512:576] while the MMAs run: one token row
            // (128 bytes) per thread
            const int n = nt * kGemmTileN + et;
            if (n < p.n_tokens) {
                const uint4 *src = reinterpret_cast<const uint4 *>(p.q_rope + ((size_t)n * 128 + h) * 64);
                uint4 *dst = reinterpret_cast<uint4 *>(p.q_abs + ((size_t)n * 128 + h) * 576 + 512);
#pragma unroll
                for (int u = 0; u < 8; ++u) dst[u] = src[u];
            }
        }
        // tcgen05.ld is warp-collective: the whole warp takes the same branch around it
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(10), 0, abort));
        if (ok) {
            tc_fence_after();
            // each accumulator -> bf16 -> shared tile [token][128 columns] (256-byte rows); a store
            // instruction writes 32 consecutive columns of one token row (conflict-free)
            for (int mc = 0; mc < n_acc; ++mc) {
                const uint32_t tile = base + mc * kOutTileBytes;
#pragma unroll 1
                for (int c = 0; c < kGemmTileN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + 128u * mc + c * 32u, v);
                    tmem_ld_wait_dep(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const __nv_bfloat16 x = __float2bfloat16_rn(__uint_as_float(v[e]));
                        asm volatile("st.shared.b16 [%0], %1;" ::"r"(tile + (uint32_t)(c * 32 + e) * 256u + (uint32_t)m * 2u),
                                     "h"(*reinterpret_cast<const unsigned short *>(&x))
                                     : "memory");
                    }
                }
            }
            fence_proxy_async_smem();  // the tiles (generic proxy writes) before the TMA store reads them
        }
        mbar_arrive(bar(11));
        if (et == 0 && mbar_wait(bar(11), 0, abort) && ok) {
            // tokens past n_tokens fall outside the output tensor and are not written
            for (int mc = 0; mc < n_acc; ++mc)
                tma_store_3d(&tmap_o, base + mc * kOutTileBytes, mc * 128, h, nt * kGemmTileN);
            bulk_commit_group();
            bulk_wait_group_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

}  // namespace mla
