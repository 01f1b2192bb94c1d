// gemm_kernels.cuh - per-head tcgen05 GEMMs around the decode:
//   absorb:  q_abs[n,h,0:512] = W_UK[h]^T q_nope[n,h,:]      ("DeepSeek-V2" explainer, Step 6)
//            q_abs[n,h,512:576] = q_rope[n,h,:]              (Step 7: RoPE query passes through)
//   up-proj: out[n,h,:] = W_UV[h] o_lat[n,h,:]                (Step 5 values, applied after attention)
//
// Both are computed transposed so that the 128-row tensor-core M dimension is
// filled by weight rows even for a handful of tokens: D^T[m, n] with m over the
// weight dimension (a 128-wide latent chunk, or the 128 head dims) and n over a
// 128-token tile.  Weights and activations are staged by TMA in 64-column boxes
// with 128-byte swizzle; the fp32 accumulator lives in 128 TMEM columns; the
// epilogue writes bf16 with one thread per output feature, so each warp store
// covers 32 consecutive features of one token.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace mla {

constexpr int kGemmStages = 4;
constexpr int kGemmTileN = 128;                      // tokens per CTA
constexpr uint32_t kGemmStageBytes = 32768;          // A 16 KB + B 16 KB
constexpr uint32_t kGemmOffBar = kGemmStages * kGemmStageBytes;
constexpr uint32_t kGemmSmem = kGemmOffBar + 256 + 1024;
constexpr int kModeAbsorb = 0, kModeUpProj = 1;

struct GemmParams {
    int mode;
    int n_tokens;
    const __nv_bfloat16 *q_rope;  // absorb only: [N, 128, 64]
    __nv_bfloat16 *out;           // absorb: q_abs [N, 128, 576]; up-proj: [N, 128, 128]
};

// grid: absorb (128 heads, 4 latent chunks, token tiles); up-proj (128 heads, 1, token tiles)
__global__ void __launch_bounds__(192, 1)
head_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                 const GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, mc = blockIdx.y, nt = blockIdx.z;
    const bool absorb = p.mode == kModeAbsorb;
    const int nk = absorb ? 2 : 8;  // 64-wide K chunks: d_h = 128 or d_c = 512
    auto bar = [&](int i) { return base + kGemmOffBar + 8u * i; };  // full[0..3], empty[4..7], done[8]
    volatile int *abort = reinterpret_cast<volatile int *>(smem_raw + (base - raw) + kGemmOffBar + 80);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + kGemmOffBar + 72);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(bar(s), 1);
            mbar_init(bar(kGemmStages + s), 1);
        }
        mbar_init(bar(2 * kGemmStages), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(base + kGemmOffBar + 72, 128);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kGemmStages;
                if (!mbar_wait(bar(kGemmStages + s), ((kc / kGemmStages) & 1) ^ 1, abort)) break;
                const uint32_t a = base + s * kGemmStageBytes, b = a + 16384u;
                mbar_arrive_expect_tx(bar(s), kGemmStageBytes);
                if (absorb) {
                    // W_UK viewed as [(h, d) rows, 512 latent columns]: two 64x64 boxes -> M = 128 latent
                    tma_load_2d(a, &tmap_w, mc * 128, h * 128 + kc * 64, bar(s));
                    tma_load_2d(a + 8192u, &tmap_w, mc * 128 + 64, h * 128 + kc * 64, bar(s));
                    // q_nope viewed as [tokens, (h, d)]: 128 tokens x 64 d
                    tma_load_2d(b, &tmap_x, h * 128 + kc * 64, nt * kGemmTileN, bar(s));
                } else {
                    // W_UV viewed as [(h, d) rows, 512 latent columns]: 128 d x 64 latent
                    tma_load_2d(a, &tmap_w, kc * 64, h * 128, bar(s));
                    // o_lat viewed as [tokens, (h, latent)]: 128 tokens x 64 latent
                    tma_load_2d(b, &tmap_x, h * 512 + kc * 64, nt * kGemmTileN, bar(s));
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = absorb ? idesc_bf16_f32(128, 128, 1, 0) : idesc_bf16_f32(128, 128, 0, 0);
            bool ok = true;
            for (int kc = 0; kc < nk && ok; ++kc) {
                const int s = kc % kGemmStages;
                if (!mbar_wait(bar(s), (kc / kGemmStages) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = base + s * kGemmStageBytes, b = a + 16384u;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // absorb: A = W_UK^T chunk, MN-major (latent contiguous), K = 16 d rows per step
                    // up-proj: A = W_UV chunk, K-major (latent contiguous along K)
                    const uint64_t adesc = absorb ? sdesc_sw128(a + 2048u * k, 8192u, 1024u)
                                                  : sdesc_sw128(a + 32u * k, 16u, 1024u);
                    const uint64_t bdesc = sdesc_sw128(b + 32u * k, 16u, 1024u);
                    mma_ss(tmem, adesc, bdesc, idesc, (kc | k) != 0);
                }
                mma_commit(bar(kGemmStages + s));
            }
            mma_commit(bar(2 * kGemmStages));
        }
    } else {
        // epilogue: warps 2..5 -> TMEM lane quadrants 2, 3, 0, 1
        const int q = warp & 3;
        const int row = q * 32 + lane;  // weight-side index of this thread
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        if (mbar_wait(bar(2 * kGemmStages), 0, abort)) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kGemmTileN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + c * 32u, v);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int n = nt * kGemmTileN + c * 32 + e;
                    if (n < p.n_tokens) {
                        const __nv_bfloat16 x = __float2bfloat16_rn(__uint_as_float(v[e]));
                        if (absorb)
                            p.out[((size_t)n * 128 + h) * 576 + mc * 128 + row] = x;
                        else
                            p.out[((size_t)n * 128 + h) * 128 + row] = x;
                    }
                }
            }
        }
        if (absorb && mc == 0) {
            // RoPE query: copied unchanged into the last 64 columns
            const int t = threadIdx.x - 64;  // 0..127
            const int n = nt * kGemmTileN + t;
            if (n < p.n_tokens) {
                const uint4 *src = reinterpret_cast<const uint4 *>(p.q_rope + ((size_t)n * 128 + h) * 64);
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)n * 128 + h) * 576 + 512);
#pragma unroll
                for (int u = 0; u < 8; ++u) dst[u] = src[u];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

}  // namespace mla
