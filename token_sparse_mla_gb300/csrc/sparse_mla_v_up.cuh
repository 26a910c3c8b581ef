// The v_up projection of the attention output on tcgen05 tensor cores (sm_103a).
//
// The latent output O [T, h, 512] of the sparse attention "is consumed by the v_up
// projection" (vLLM PR #60220, Details): per head, 512 -> v_head_dim, with v_head_dim 128
// (DeepSeek-V3.2) or 256 (GLM-5) at kv_lora_rank 512 (PR #55738 report, the
// `_is_masked_mha_available` geometry table):
//
//   Y[t, h, n] = sum_{k < 512} O[t, h, k] * W[h, n, k]       W [h, v, 512] bf16, Y [T, h, v] bf16
//
// A dense contraction (2 * 512 * v flops per (token, head), O read once), so it runs as a
// GEMM per head on the tensor cores: M = 128 tokens, N = 128 outputs, K = 512 in eight
// 64-wide SW128 panels.  Each CTA owns one (head, 128-output slice) and a contiguous run of
// 128-token tiles: its W slice (128 KB) is loaded once and stays in shared memory, the O
// panels stream through a six-stage TMA ring, and the fp32 accumulator lives in TMEM, double
// buffered so the epilogue of one tile overlaps the MMAs of the next.
//
// Roles (192 threads):
//   warp 0      TMA producer (one thread): the W slice, then O panels into the ring.
//   warp 1      MMA issuer (one thread) and TMEM owner: 4 x tcgen05.mma (M128 N128 K16) per
//               panel, a commit per panel (frees the stage) and per tile (accumulator ready).
//   warps 2-5   epilogue: each warp reads its TMEM lane quadrant (32 tokens) with
//               32x32b loads, rounds to bf16 and stores 256 contiguous bytes per token.
// Every wait is bounded; a CTA that gives up drains its copies and MMAs before it leaves.
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kVupRows = 128;                      // tokens per tile (MMA M)
constexpr int kVupN = 128;                         // outputs per CTA (MMA N)
constexpr int kVupPanels = kDV / 64;               // K = 512 in 64-wide panels
constexpr int kVupStages = 6;                      // 96 KB of O in flight (four stages: 60.3 us, six: 55.5 us)
constexpr int kVupPanelBytes = 128 * 128;          // 128 rows x 64 bf16, SW128
constexpr int kVupThreads = 192;
constexpr int kVupTmemCols = 2 * kVupN;            // two accumulators

struct VupLayout {
    static constexpr int kOffW = 0;                                          // [8 panels][128 n][64 k]
    static constexpr int kOffA = kOffW + kVupPanels * kVupPanelBytes;        // [6 stages][128 t][64 k]
    static constexpr int kOffBar = kOffA + kVupStages * kVupPanelBytes;
    static constexpr int kNumBars = 1 + 2 * kVupStages + 4 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;                  // tmem base, abort flag
    static constexpr int kBytes = kOffMisc + 16;
    static_assert(kOffA % 1024 == 0, "swizzled operands need 1 KB alignment");
    static_assert(kBytes <= 232448, "shared memory budget (227 KB)");
};

enum : int {
    kVbW = 0,
    kVbFull = 1,                            // +stage
    kVbEmpty = 1 + kVupStages,              // +stage
    kVbAccFull = 1 + 2 * kVupStages,        // +buffer
    kVbAccEmpty = 3 + 2 * kVupStages,       // +buffer
    kVbDrain = 5 + 2 * kVupStages
};

struct VupParams {
    __nv_bfloat16* y;   // [T, h, v]
    int32_t T, h, v;
    int32_t cpg;        // CTAs per (head, output slice)
    int32_t mtiles;     // ceil(T / 128)
};

__global__ void __launch_bounds__(kVupThreads, 1)
    sparse_mla_v_up_kernel(const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_w,
                           const VupParams p) {
    using L = VupLayout;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    if (sbase & 1023u) {  // uniform across the grid: every CTA leaves before any barrier
        if (threadIdx.x == 0) atomicOr(&g_smla_error, kErrLayout);
        return;
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* sAbort = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * i; };
    auto wait = [&](int i, uint32_t parity) -> bool {
        return ptx::mbar_wait(bar(i), parity, sAbort, &g_smla_error, kErrTimeout, kWaitLimitNs);
    };

    // this CTA: output slice g = (head hh, 128-output block nh) and tiles [j0, j1) of it
    const int halves = p.v / kVupN;
    const int g = static_cast<int>(blockIdx.x) / p.cpg;
    const int kc = static_cast<int>(blockIdx.x) % p.cpg;
    const int hh = g / halves, nh = g % halves;
    const int j0 = static_cast<int>(static_cast<int64_t>(kc) * p.mtiles / p.cpg);
    const int j1 = static_cast<int>(static_cast<int64_t>(kc + 1) * p.mtiles / p.cpg);
    const int nt = j1 - j0;

    if (threadIdx.x == 0) {
        *sAbort = 0;
        ptx::mbar_init(bar(kVbW), 1);
        for (int s = 0; s < kVupStages; ++s) {
            ptx::mbar_init(bar(kVbFull + s), 1);
            ptx::mbar_init(bar(kVbEmpty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(kVbAccFull + b), 1);
            ptx::mbar_init(bar(kVbAccEmpty + b), 4);
        }
        ptx::mbar_init(bar(kVbDrain), 1);
        ptx::fence_mbarrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(sbase + L::kOffMisc, kVupTmemCols);
        ptx::tmem_relinquish();
    }
    // launched as a programmatic dependent: O may be the previous launch's output
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kOffMisc);

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0 && nt > 0) {
            ptx::prefetch_tmap(&tm_o);
            ptx::prefetch_tmap(&tm_w);
            ptx::mbar_arrive_expect_tx(bar(kVbW), static_cast<uint32_t>(kVupPanels * kVupPanelBytes));
            for (int pn = 0; pn < kVupPanels; ++pn)
                ptx::tma_load_3d(sbase + L::kOffW + pn * kVupPanelBytes, &tm_w, 64 * pn, kVupN * nh, hh, bar(kVbW));
            int it = 0;
            bool ok = true;
            for (int j = j0; j < j1 && ok; ++j) {
                for (int pn = 0; pn < kVupPanels; ++pn) {
                    const int s = it % kVupStages;
                    if (it >= kVupStages && !(ok = wait(kVbEmpty + s, ((it / kVupStages) - 1) & 1))) break;
                    ptx::mbar_arrive_expect_tx(bar(kVbFull + s), static_cast<uint32_t>(kVupPanelBytes));
                    ptx::tma_load_3d(sbase + L::kOffA + s * kVupPanelBytes, &tm_o, 64 * pn, hh, kVupRows * j,
                                     bar(kVbFull + s));
                    ++it;
                }
            }
            // no copy may still be landing when the CTA leaves: W and the ring's last loads
            ptx::mbar_wait(bar(kVbW), 0, nullptr, &g_smla_error, 0u, kDrainLimitNs);
            for (int i = it - (it < kVupStages ? it : kVupStages); i < it; ++i)
                ptx::mbar_wait(bar(kVbFull + i % kVupStages), (i / kVupStages) & 1, nullptr, &g_smla_error, 0u,
                               kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0 && nt > 0) {
            constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kVupRows, kVupN, 0, 0);
            const uint64_t dw = ptx::smem_desc_sw128(sbase + L::kOffW, 16, 1024);
            const uint64_t da = ptx::smem_desc_sw128(sbase + L::kOffA, 16, 1024);
            bool ok = wait(kVbW, 0);
            int it = 0;
            for (int jj = 0; jj < nt && ok; ++jj) {
                const int buf = jj & 1;
                if (jj >= 2 && !(ok = wait(kVbAccEmpty + buf, ((jj >> 1) - 1) & 1))) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(buf * kVupN);
                for (int pn = 0; pn < kVupPanels; ++pn, ++it) {
                    const int s = it % kVupStages;
                    if (!(ok = wait(kVbFull + s, (it / kVupStages) & 1))) break;
                    ptx::tc_fence_after();
                    const uint64_t a0 = da + static_cast<uint64_t>((s * kVupPanelBytes) >> 4);
                    const uint64_t b0 = dw + static_cast<uint64_t>((pn * kVupPanelBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16_ss(d, a0 + ((kk * 32) >> 4), b0 + ((kk * 32) >> 4), kIdesc, (pn | kk) != 0);
                    ptx::mma_commit(bar(kVbEmpty + s));
                }
                if (!ok) break;
                ptx::mma_commit(bar(kVbAccFull + buf));
            }
            ptx::mma_commit(bar(kVbDrain));
            ptx::mbar_wait(bar(kVbDrain), 0, nullptr, &g_smla_error, 0u, kDrainLimitNs);
        }
        __syncwarp();
    } else {
        // ================================================================ epilogue
        const int quad = warp & 3;  // the TMEM lane quadrant this warp may read
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        for (int jj = 0; jj < nt; ++jj) {
            const int buf = jj & 1;
            bool ok = true;
            if (lane == 0) ok = wait(kVbAccFull + buf, (jj >> 1) & 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (!ok) break;
            ptx::tc_fence_after();
            const int64_t t = static_cast<int64_t>(j0 + jj) * kVupRows + quad * 32 + lane;
            uint4* yrow = reinterpret_cast<uint4*>(p.y + (t * p.h + hh) * p.v + nh * kVupN);
#pragma unroll 1
            for (int c = 0; c < kVupN / 16; ++c) {
                uint32_t r[16];
                SMLA_TMEM_LD16(tmem + lane_base + static_cast<uint32_t>(buf * kVupN + c * 16), r);
                ptx::tmem_wait_ld();
                if (t < p.T) {
                    uint4 v0, v1;
                    v0.x = pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1]));
                    v0.y = pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3]));
                    v0.z = pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5]));
                    v0.w = pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7]));
                    v1.x = pack_bf16x2(__uint_as_float(r[8]), __uint_as_float(r[9]));
                    v1.y = pack_bf16x2(__uint_as_float(r[10]), __uint_as_float(r[11]));
                    v1.z = pack_bf16x2(__uint_as_float(r[12]), __uint_as_float(r[13]));
                    v1.w = pack_bf16x2(__uint_as_float(r[14]), __uint_as_float(r[15]));
                    yrow[2 * c] = v0;
                    yrow[2 * c + 1] = v1;
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kVbAccEmpty + buf));
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kVupTmemCols);
    }
}

}  // namespace smla
