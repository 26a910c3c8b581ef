// Token-sparse MLA forward for 8 or 16 heads per token (the native small-head path).
//
// With 8 or 16 heads the contractions per 64 KV rows are tiny (64 x 16 x 576 for the logits):
// a tcgen05.mma costs about 46 cycles whatever its N up to 64, so the 52 instructions a 64-row
// block needs at N = 16 would take longer than the block's HBM time.  Here both contractions run
// as warp-level m16n8k16 bf16 MMAs (fp32 accumulate) with the heads as the 8-wide N dimension,
// so h = 8 carries no padding at all, and the accumulators live in registers:
//
//   S^T[32 rows, h]  = K_blk[32 x 576] . Q^T   - the 576-dim reduction is split over the four
//                                                compute warps (9 k-steps of 16 dims each, Q^T
//                                                fragments held in registers for the whole CTA),
//                                                partial sums reduced through shared memory;
//   O^T[512, h]     += V_blk^T[512 x 32] . P^T - split over the warps by output dims (128 each);
//                                                V^T comes from the SAME shared-memory tile as K
//                                                through ldmatrix.trans.
//
// Rows arrive in 32-row stages (36,864 bytes; five in flight) gathered by seven producer warps
// (gather_rows, shared with the tcgen05 kernel).  Each compute warp takes eight of the block's
// rows for the softmax: masking, a running max per head in log2 units with conditional
// rescaling (only when the max grows by more than 2^8), fp32 partial sums, P^T (bf16) to shared
// memory.  Splits over a thread-block cluster merge through distributed shared memory exactly as
// in the tcgen05 kernel.
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kSmRows = 32;                                          // KV rows per stage
constexpr int kSmStages = 5;
constexpr int kSmComputeWarps = 4;
constexpr int kSmThreads = 32 * (kProducerWarps + kSmComputeWarps);  // 352
constexpr int kSmCompute0 = 32 * kProducerWarps;                     // first compute thread
constexpr int kSmKSteps = kDQK / 16 / kSmComputeWarps;               // 9 k-steps per warp

template <int H>
struct SmallLayout {
    static_assert(H == 8 || H == 16, "the small-head kernel runs 8 or 16 heads");
    static constexpr int kNT = H / 8;                                // n-tiles of 8 heads
    static constexpr int kPanelBytes = kSmRows * 128;                // 4096
    static constexpr int kStageBytes = kPanels * kPanelBytes;        // 36864
    static constexpr int kOffKV = 0;
    static constexpr int kOffRed = kSmStages * kStageBytes;          // S partials, float4 per lane
    static constexpr int kRedBytes = kSmComputeWarps * 2 * kNT * 32 * 16;
    static constexpr int kPStride = 80;                              // bytes per head row of P^T
    static constexpr int kOffP = kOffRed + kRedBytes;
    static constexpr int kOffHr = kOffP + H * kPStride;              // [8][H]: per-warp reductions,
                                                                     // per-source merge weights
    static constexpr int kOffM = kOffHr + kMaxSplits * H * 4;        // running max (log2 units)
    static constexpr int kOffAlpha = kOffM + H * 4;                  // rescale factor / 1/L / weight
    static constexpr int kOffML = kOffAlpha + H * 4;                 // final m[H], L[H]
    static constexpr int kOffRecvML = kOffML + 2 * H * 4;            // [kMaxSplits][2H] (m, L) of peers
    static constexpr int kOffRecv = kOffRecvML + kMaxSplits * 2 * H * 4;  // [splits][H][512/splits] fp32
    static constexpr int kOffBar = kOffRecv + H * kDV * 4;           // full[5], empty[5]
    static constexpr int kOffMisc = kOffBar + 2 * kSmStages * 8;     // abort flag
    static constexpr int kBytes = kOffMisc + 16;
    static_assert(kOffP % 16 == 0, "ldmatrix rows need 16-byte alignment");
    static_assert(kBytes <= 232448, "shared memory budget (227 KB)");
    static_assert(kOffRecv % 16 == 0 && kOffBar % 8 == 0, "alignment of the merge buffers");
    static_assert(H * kDV * 2 <= kSmStages * kStageBytes, "output staging fits the stages");
};

namespace mma16816 {
// D (16x8 fp32) += A (16x16 bf16, row) . B (16x8 bf16, col)
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr)
                 : "memory");
}
}  // namespace mma16816

template <int H, int KVF>
__global__ void __launch_bounds__(kSmThreads, 1) sparse_mla_fwd_small_kernel(const FwdParams p) {
    using L = SmallLayout<H>;
    constexpr int NT = L::kNT;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    if (sbase & 1023u) {  // uniform across the grid: every CTA leaves before any barrier
        if (threadIdx.x == 0) atomicOr(&g_smla_error, kErrLayout);
        return;
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t sKV = sbase + L::kOffKV;
    const uint32_t sP = sbase + L::kOffP;
    float4* sRedS = reinterpret_cast<float4*>(smem + L::kOffRed);
    float* sHr = reinterpret_cast<float*>(smem + L::kOffHr);
    float* sM = reinterpret_cast<float*>(smem + L::kOffM);
    float* sAlpha = reinterpret_cast<float*>(smem + L::kOffAlpha);
    float* sML = reinterpret_cast<float*>(smem + L::kOffML);
    volatile int* sAbort = reinterpret_cast<volatile int*>(smem + L::kOffMisc);
    const uint32_t bar_full0 = sbase + L::kOffBar;
    const uint32_t bar_empty0 = sbase + L::kOffBar + 8 * kSmStages;

    // ---- work of this CTA
    const int splits = p.splits;
    const int t = blockIdx.x / splits;
    const int rank = blockIdx.x % splits;  // == %cluster_ctarank when splits > 1
    const int nblk_total = (p.topk + kSmRows - 1) / kSmRows;
    const int per_split = (nblk_total + splits - 1) / splits;
    const int b_begin = min(nblk_total, rank * per_split);
    const int b_end = min(nblk_total, b_begin + per_split);
    const int nb = b_end - b_begin;
    const int j0 = b_begin * kSmRows;
    const int j1 = min(p.topk, b_end * kSmRows);
    const int32_t* idx_row = p.indices + static_cast<int64_t>(t) * p.topk;

    if (threadIdx.x == 0) {
        *sAbort = 0;
        for (int s = 0; s < kSmStages; ++s) {
            ptx::mbar_init(bar_full0 + 8 * s, 32 * kProducerWarps);
            ptx::mbar_init(bar_empty0 + 8 * s, kSmComputeWarps);
        }
        ptx::fence_mbarrier_init();
    }
    if (threadIdx.x >= kSmCompute0 && threadIdx.x - kSmCompute0 < H) sM[threadIdx.x - kSmCompute0] = -CUDART_INF_F;
    __syncthreads();
    // peers push into this CTA's receive buffers at the end; the matching wait below makes sure
    // every CTA of the cluster has started before any of them writes to another
    if (splits > 1) ptx::cluster_arrive_relaxed();

    // O^T accumulators of the compute warps (fragment layout: dims 128*cw + 16*mt + g (+8),
    // heads 8*nt + 2*tq (+1)); declared here because the cluster merge below reads them
    float o[8][SmallLayout<H>::kNT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;

    if (warp < kProducerWarps) {
        // ================================================================ producers
        gather_rows<kSmRows, kSmStages, KVF>(p, idx_row, j0, j1, nb, warp, lane, sKV, bar_full0, bar_empty0,
                                             sAbort);
    } else {
        // ================================================================ compute warps
        const int cw = warp - kProducerWarps;   // 0..3
        const int wtid = threadIdx.x - kSmCompute0;
        const int g = lane >> 2;                // MMA fragment row group
        const int tq = lane & 3;                // MMA fragment column pair
        const int li = lane & 7, lj = lane >> 3;  // ldmatrix: row within matrix, matrix index
        const float c = p.sm_scale_log2;
        bool failed = false;

        // Q^T fragments (B operand of S^T) for this warp's nine 16-dim k-steps, all heads
        uint32_t bq[kSmKSteps][NT][2];
        {
            const __nv_bfloat16* qt = p.q + static_cast<int64_t>(t) * p.h * kDQK;
#pragma unroll
            for (int kk = 0; kk < kSmKSteps; ++kk) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const unsigned int* qr = reinterpret_cast<const unsigned int*>(
                        qt + (nt * 8 + g) * kDQK + 16 * (kSmKSteps * cw + kk) + 2 * tq);
                    bq[kk][nt][0] = __ldg(qr);
                    bq[kk][nt][1] = __ldg(qr + 4);
                }
            }
        }
        // this warp's softmax rows: 8 of the block's 32 (m-tile cw/2, half cw%2), one per lane group
        const int mt_s = cw >> 1, half = cw & 1;
        const int rr = mt_s * 16 + half * 8 + g;
        // slot validity of this lane's row, loaded kAhead blocks ahead
        constexpr int kAhead = 8;
        int slot_q[kAhead];
#pragma unroll
        for (int i = 0; i < kAhead; ++i)
            slot_q[i] = i < nb ? entry_slot(idx_row, j0 + i * kSmRows + rr, j1, p.num_slots) : -1;

        float lsum[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) lsum[nt][0] = lsum[nt][1] = 0.f;

        for (int b = 0; b < nb; ++b) {
            const int s = b % kSmStages;
            const uint32_t stb = sKV + s * L::kStageBytes;
            const bool valid = slot_q[0] >= 0;
#pragma unroll
            for (int i = 0; i + 1 < kAhead; ++i) slot_q[i] = slot_q[i + 1];
            slot_q[kAhead - 1] =
                (b + kAhead < nb) ? entry_slot(idx_row, j0 + (b + kAhead) * kSmRows + rr, j1, p.num_slots) : -1;
            bool ok = true;
            if (lane == 0)
                ok = ptx::mbar_wait(bar_full0 + 8 * s, (b / kSmStages) & 1, sAbort, &g_smla_error, kErrTimeout,
                                    kWaitLimitNs);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (!ok) failed = true;

            // ---- partial S^T over this warp's 144 dims, all 32 rows
            float cs[2][NT][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) cs[mt][nt][e] = 0.f;
            if (ok) {
#pragma unroll
                for (int kk = 0; kk < kSmKSteps; ++kk) {
                    const int K = kSmKSteps * cw + kk;
                    const uint32_t pan = stb + (K >> 2) * L::kPanelBytes;
                    const int chunk = (K & 3) * 2 + (lj >> 1);
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        const int row = mt * 16 + (lj & 1) * 8 + li;  // row & 7 == li
                        uint32_t a[4];
                        mma16816::ldsm_x4(a, pan + row * 128 + ((chunk ^ li) << 4));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma16816::mma(cs[mt][nt], a, bq[kk][nt][0], bq[kk][nt][1]);
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    sRedS[((cw * 2 + mt) * NT + nt) * 32 + lane] =
                        make_float4(cs[mt][nt][0], cs[mt][nt][1], cs[mt][nt][2], cs[mt][nt][3]);
            ptx::named_bar_sync(1, 128);

            // ---- logits of this warp's rows: sum of the four partials, scaled and masked
            float x[NT][2];
            bool need = false;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float4 acc = sRedS[((0 * 2 + mt_s) * NT + nt) * 32 + lane];
#pragma unroll
                for (int w = 1; w < kSmComputeWarps; ++w) {
                    const float4 v = sRedS[((w * 2 + mt_s) * NT + nt) * 32 + lane];
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
                const float s0 = half ? acc.z : acc.x;
                const float s1 = half ? acc.w : acc.y;
                x[nt][0] = valid ? s0 * c : -CUDART_INF_F;
                x[nt][1] = valid ? s1 * c : -CUDART_INF_F;
                need |= x[nt][0] > sM[nt * 8 + 2 * tq] + kRescaleLog2;
                need |= x[nt][1] > sM[nt * 8 + 2 * tq + 1] + kRescaleLog2;
            }
            // one warp-set barrier per block in the common case (no new max, no abort)
            if (ptx::named_bar_red_or(1, 128, need || failed || *sAbort)) {
                if (ptx::named_bar_red_or(1, 128, failed || *sAbort)) {
                    failed = true;
                    break;
                }
                // the running max of some head grew: new max per head, rescale O and the sums
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float mx = x[nt][e];
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        if (lane < 4) sHr[cw * H + nt * 8 + 2 * lane + e] = mx;
                    }
                }
                ptx::named_bar_sync(1, 128);
                if (wtid < H) {
                    const float mo = sM[wtid];
                    float mb = sHr[wtid];
#pragma unroll
                    for (int w = 1; w < kSmComputeWarps; ++w) mb = fmaxf(mb, sHr[w * H + wtid]);
                    const float mn = fmaxf(mo, mb);
                    sAlpha[wtid] = (mo == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(mo - mn);
                    sM[wtid] = mn;
                }
                ptx::named_bar_sync(1, 128);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float a = sAlpha[nt * 8 + 2 * tq + e];
                        lsum[nt][e] *= a;
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            o[mt][nt][e] *= a;
                            o[mt][nt][2 + e] *= a;
                        }
                    }
                }
            }
            // ---- P = 2^(x - m): fp32 partial sums, bf16 P^T[h][row] for the PV product
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = nt * 8 + 2 * tq + e;
                    const float pr = (x[nt][e] == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(x[nt][e] - sM[h]);
                    lsum[nt][e] += pr;
                    ptx::st_shared_u16(sP + h * L::kPStride + rr * 2, bf16_bits(pr));
                }
            }
            ptx::named_bar_sync(1, 128);

            // ---- O^T[this warp's 128 dims, h] += V^T . P^T over the block's 32 rows
            if (ok) {
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    uint32_t bp[NT][2];
                    if constexpr (NT == 1) {
                        mma16816::ldsm_x2(bp[0][0], bp[0][1],
                                          sP + li * L::kPStride + (16 * kk + 8 * (lj & 1)) * 2);
                    } else {
                        uint32_t r4[4];
                        mma16816::ldsm_x4(r4, sP + ((lj >> 1) * 8 + li) * L::kPStride + (16 * kk + 8 * (lj & 1)) * 2);
                        bp[0][0] = r4[0]; bp[0][1] = r4[1];
                        bp[NT - 1][0] = r4[2]; bp[NT - 1][1] = r4[3];
                    }
                    const int krow = 16 * kk + (lj >> 1) * 8 + li;  // krow & 7 == li
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const int d0 = 128 * cw + 16 * mt;
                        const int chunk = ((d0 & 63) >> 3) + (lj & 1);
                        uint32_t a[4];
                        mma16816::ldsm_x4_trans(a, stb + (d0 >> 6) * L::kPanelBytes + krow * 128 + ((chunk ^ li) << 4));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma16816::mma(o[mt][nt], a, bp[nt][0], bp[nt][1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_empty0 + 8 * s);  // this warp is done with the stage
        }

        // ---- per-head totals L over the block rows of all four warps
        const bool aborted = ptx::named_bar_red_or(1, 128, failed || *sAbort);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = lsum[nt][e];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                if (lane < 4) sHr[cw * H + nt * 8 + 2 * lane + e] = v;
            }
        }
        ptx::named_bar_sync(1, 128);
        if (wtid < H) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kSmComputeWarps; ++w) tot += sHr[w * H + wtid];
            if (aborted || nb == 0) tot = 0.f;
            sML[wtid] = sM[wtid];
            sML[H + wtid] = tot;
            sAlpha[wtid] = tot > 0.f ? 1.0f / tot : 0.f;
        }
        ptx::named_bar_sync(1, 128);

        if (splits == 1 && !aborted) {
            // O = O^T / L as bf16, staged as out[t] ([h][512], contiguous) in the free stage
            // memory, then written with 16-byte stores
            uint16_t* so = reinterpret_cast<uint16_t*>(smem + L::kOffKV);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int d = 128 * cw + 16 * mt + g;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int h = nt * 8 + 2 * tq;
                    so[h * kDV + d] = bf16_bits(o[mt][nt][0] * sAlpha[h]);
                    so[(h + 1) * kDV + d] = bf16_bits(o[mt][nt][1] * sAlpha[h + 1]);
                    so[h * kDV + d + 8] = bf16_bits(o[mt][nt][2] * sAlpha[h]);
                    so[(h + 1) * kDV + d + 8] = bf16_bits(o[mt][nt][3] * sAlpha[h + 1]);
                }
            }
            ptx::named_bar_sync(1, 128);
            const uint4* src = reinterpret_cast<const uint4*>(so);
            uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(t) * p.h * kDV);
            for (int v = wtid; v < p.h * (kDV / 8); v += 128) dst[v] = src[v];
            if (wtid < p.h) {
                const float tot = sML[H + wtid];
                p.lse[static_cast<int64_t>(t) * p.h + wtid] =
                    tot > 0.f ? (sML[wtid] + log2f(tot)) * 0.69314718055994531f : -CUDART_INF_F;
            }
        }
        if (splits > 1 && (failed || aborted)) sAbort[0] = 1;
    }

    __syncthreads();

    if (splits > 1) {
        // ================================================================ cluster merge
        // CTA k of the cluster owns output dims [k*ds, (k+1)*ds).  Every CTA pushes its per-head
        // (m, L) and its unnormalised partial O for each owner's dims into that owner's receive
        // buffers; after one cluster barrier each owner weights the partials by 2^(m_j - M) / sum_j
        // L_j 2^(m_j - M) and stores its dims.  No CTA reads another's memory after the barrier.
        const int ds = kDV / splits;
        ptx::cluster_wait();  // every CTA has started (pairs with the arrive at the top)
        if (warp >= kProducerWarps) {
            const int cw = warp - kProducerWarps;
            const int wtid = threadIdx.x - kSmCompute0;
            const int g = lane >> 2, tq = lane & 3;
            const bool have = nb > 0 && *sAbort == 0;
            const uint32_t recv = sbase + L::kOffRecv;
            const uint32_t recv_ml = sbase + L::kOffRecvML;
            if (wtid < H) {
                const float m = have ? sML[wtid] : -CUDART_INF_F;
                const float l = have ? sML[H + wtid] : 0.f;
                for (int k = 0; k < splits; ++k) {
                    ptx::st_shared_cluster_f32(ptx::map_shared_rank(recv_ml + (rank * 2 * H + wtid) * 4, k), m);
                    ptx::st_shared_cluster_f32(ptx::map_shared_rank(recv_ml + (rank * 2 * H + H + wtid) * 4, k), l);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    const int d = 128 * cw + 16 * mt + g + 8 * hi;
                    const int k = d / ds;
                    const int dd = d - k * ds;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int h = nt * 8 + 2 * tq + e;
                            const uint32_t la = recv + static_cast<uint32_t>(((rank * H + h) * ds + dd) * 4);
                            ptx::st_shared_cluster_f32(ptx::map_shared_rank(la, k), have ? o[mt][nt][2 * hi + e] : 0.f);
                        }
                    }
                }
            }
        }
        ptx::cluster_sync();  // all pushes are visible to their owners
        if (warp >= kProducerWarps) {
            const int wtid = threadIdx.x - kSmCompute0;
            const float* rml = reinterpret_cast<const float*>(smem + L::kOffRecvML);
            const float* rcv = reinterpret_cast<const float*>(smem + L::kOffRecv);
            if (wtid < H) {
                float M = -CUDART_INF_F;
                for (int j = 0; j < splits; ++j) M = fmaxf(M, rml[j * 2 * H + wtid]);
                float Lt = 0.f;
                for (int j = 0; j < splits; ++j) {
                    const float mj = rml[j * 2 * H + wtid], lj = rml[j * 2 * H + H + wtid];
                    if (mj != -CUDART_INF_F && lj > 0.f) Lt += lj * ptx::ex2_approx(mj - M);
                }
                for (int j = 0; j < splits; ++j) {
                    const float mj = rml[j * 2 * H + wtid], lj = rml[j * 2 * H + H + wtid];
                    sHr[j * H + wtid] = (Lt > 0.f && mj != -CUDART_INF_F && lj > 0.f) ? ptx::ex2_approx(mj - M) / Lt : 0.f;
                }
                if (rank == 0 && wtid < p.h)
                    p.lse[static_cast<int64_t>(t) * p.h + wtid] =
                        Lt > 0.f ? (M + log2f(Lt)) * 0.69314718055994531f : -CUDART_INF_F;
            }
            ptx::named_bar_sync(1, 128);
            // eight dims of one head per item, stored as one 16-byte vector
            const int per_head = ds / 8;
            for (int it = wtid; it < p.h * per_head; it += 128) {
                const int hh = it / per_head;
                const int dd = (it % per_head) * 8;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int j = 0; j < splits; ++j) {
                    const float w = sHr[j * H + hh];
                    const float4 lo = *reinterpret_cast<const float4*>(rcv + (j * H + hh) * ds + dd);
                    const float4 hv = *reinterpret_cast<const float4*>(rcv + (j * H + hh) * ds + dd + 4);
                    acc[0] += w * lo.x; acc[1] += w * lo.y; acc[2] += w * lo.z; acc[3] += w * lo.w;
                    acc[4] += w * hv.x; acc[5] += w * hv.y; acc[6] += w * hv.z; acc[7] += w * hv.w;
                }
                uint4 packed;
                packed.x = pack_bf16x2(acc[0], acc[1]);
                packed.y = pack_bf16x2(acc[2], acc[3]);
                packed.z = pack_bf16x2(acc[4], acc[5]);
                packed.w = pack_bf16x2(acc[6], acc[7]);
                *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * p.h + hh) * kDV + rank * ds + dd) = packed;
            }
        }
    }
}

}  // namespace smla
