// Token-sparse MLA forward, bf16 latent cache, tcgen05/TMEM tensor cores (sm_103a).
//
// One CTA handles one (query token, split) pair: the token's top-k list is cut
// into `splits` contiguous ranges of 64-row blocks, one per CTA of a thread-block
// cluster, and the partial results are merged on chip through distributed shared
// memory (no global workspace; vLLM PR #60220, Details/Limitations, describes the
// per-call o_accum split-KV buffer this avoids).
//
// The pass is bound by the KV row gather (PR #55738 report, 功能与动机: the
// per-token top-k MQA kernel is HBM-bound by its KV gather).  bf16 rows are fetched
// with 16-byte cp.async by the producer warps, one warp per row at a time (each
// warp instruction moves 512 contiguous bytes of a row), written straight into
// the 128-byte-swizzled K-major operand layout; invalid entries are zero-filled
// without a memory read.  fp8 rows are loaded into registers, dequantised and
// stored into the same layout.
//
// Roles (384 threads for bf16 rows, 448 for fp8 rows):
//   warp 0      S^T issuer (one thread) and TMEM owner.  Swap-AB form, so the head
//               count only has to fill the MMA's N dimension (no padding to 64):
//                 S^T[64 rows, HP]        = K_blk[64 x 576] . Q^T          (M=64)
//   warps 1-NP  producers: gather of 64 rows per stage, 2 stages.  NP = 6 for bf16 rows
//               (cp.async copies); NP = 8 for fp8 rows, whose producers dequantise in
//               registers and hold a row's loads per lane (8 rows a warp instead of 11).
//   warp NP+1   PV issuer (one thread):
//                 O^T[512 dims, HP]      += V_blk^T[512 x 64] . P^T        (4 x M=128)
//               V^T is read from the SAME shared-memory tile as K, as an MN-major
//               operand.
//   last 4      softmax warpgroup (warp w reads TMEM lane quadrant w % 4): reads S^T from TMEM (16x256b loads: two KV rows and
//               a quarter of the heads per thread, all 32 lanes busy), masks invalid
//               entries, keeps a running max per head in log2 units and only rescales
//               O when that max grows by more than 2^8, keeps fp32 partial softmax sums
//               in registers, writes P^T (bf16) to shared memory, runs the epilogue.
//   A thread that issues an MMA waits while the tensor cores take it, so the two products
//   have an issuer each: PV(b) goes out as soon as P^T(b) is ready, even while S^T(b+1)'s
//   36 MMAs are still being issued, and the softmax of one block overlaps the MMAs of its
//   neighbours.
//
// HP is the MMA N size: the head count rounded up to 16 (h = 8 runs N = 16 with
// the upper 8 query rows zero in shared memory; nothing is padded in HBM).
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kRows = 64;                           // KV rows per pipeline stage
constexpr int kPanelBytes = kRows * 128;            // one panel of a 64-row stage
constexpr int kStageBytes = kPanels * kPanelBytes;  // 73728 bytes = 64 rows x 1152
constexpr int kStages = 2;
template <int KVF>
struct TcRoles {
    static constexpr int kProducers = KVF == 1 ? 8 : 6;    // producer warps 1 .. kProducers
    static constexpr int kPvWarp = 1 + kProducers;          // the PV issuer's warp
    static constexpr int kThreads = 32 * (kPvWarp + 1 + 4); // 384 (bf16) / 448 (fp8)
    static constexpr int kSoftmaxThread0 = 32 * (kPvWarp + 1);
};

template <int HP>
struct Layout {
    static_assert(HP == 16 || HP == 32 || HP == 64, "MMA N must be 16, 32 or 64");
    static constexpr int kQBytes = kPanels * HP * 128;
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQBytes;
    // P^T of block b (HP rows x 64 bf16) lives in the rope panel of block b's own stage
    static constexpr int kOffRed = kOffKV + kStages * kStageBytes;  // [4 warps][HP]
    static constexpr int kOffM = kOffRed + 4 * HP * 4;             // running max (log2 units)
    static constexpr int kOffAlpha = kOffM + HP * 4;               // rescale factor / 1/L / merge weight
    static constexpr int kOffML = kOffAlpha + HP * 4;              // final m[HP], L[HP]
    static constexpr int kOffBar = kOffML + 2 * HP * 4;
    static constexpr int kNumBars = 13;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
    static constexpr int kBytes = kOffMisc + 16;
    // TMEM columns: O^T [0,4HP) | S^T x2 [4HP,6HP)
    static constexpr int kColS = 4 * HP;
    static constexpr int kTmemCols = (6 * HP <= 128) ? 128 : ((6 * HP <= 256) ? 256 : 512);
    static_assert(6 * HP <= kTmemCols, "TMEM budget");
    static_assert(kOffKV % 1024 == 0 && kStageBytes % 1024 == 0, "swizzled operands need 1 KB alignment");
    static_assert(HP * 128 <= kPanelBytes, "P^T fits a stage's rope panel");
    static_assert(kBytes <= 232448, "shared memory budget (227 KB)");
    static_assert(HP * kDV * 4 <= kStages * kStageBytes, "merge buffer fits the stages");
};

// barrier slots
enum : int {
    kBarQ = 0,
    kBarKvFull = 1,   // +stage
    kBarKvEmpty = 3,  // +stage
    kBarSFull = 5,    // +buffer
    kBarSEmpty = 7,   // +buffer
    kBarPFull = 9,
    kBarPvDone = 10,  // +stage: PV of the blocks of that stage (so a wait never falls two phases behind)
    kBarDrain = 12
};

// KVF: 0 = bf16 rows of 576 values (1152 bytes); 1 = fp8 rows of 656 bytes
// ([512 e4m3 | 4 fp32 scales, one per 128 latent values | 64 bf16 rope]), dequantised by the
// producers into the same bf16 operand tile.
template <int HP, int KVF>
__global__ void __launch_bounds__(TcRoles<KVF>::kThreads, 1)
    sparse_mla_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const FwdParams p) {
    using L = Layout<HP>;
    constexpr int kTcProducers = TcRoles<KVF>::kProducers;
    constexpr int kTcPvWarp = TcRoles<KVF>::kPvWarp;
    constexpr int kSoftmaxThread0 = TcRoles<KVF>::kSoftmaxThread0;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    if (sbase & 1023u) {  // uniform across the grid: every CTA leaves before any barrier
        if (threadIdx.x == 0) atomicOr(&g_smla_error, kErrLayout);
        return;
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t sQ = sbase + L::kOffQ;
    const uint32_t sKV = sbase + L::kOffKV;
    const uint32_t sRope = sKV + (kPanels - 1) * kPanelBytes;  // stage 0's rope panel
    float* sRed = reinterpret_cast<float*>(smem + L::kOffRed);
    float* sM = reinterpret_cast<float*>(smem + L::kOffM);
    float* sAlpha = reinterpret_cast<float*>(smem + L::kOffAlpha);
    float* sML = reinterpret_cast<float*>(smem + L::kOffML);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
    volatile int* sAbort = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * static_cast<uint32_t>(i); };
    auto wait = [&](int i, uint32_t parity) -> bool {
        return ptx::mbar_wait(bar(i), parity, sAbort, &g_smla_error, kErrTimeout, kWaitLimitNs);
    };

    // ---- work of this CTA
    const int splits = p.splits;
    const int t = blockIdx.x / splits;
    const int rank = blockIdx.x % splits;  // == %cluster_ctarank when splits > 1
    const int nblk_total = (p.topk + kRows - 1) / kRows;
    const int per_split = (nblk_total + splits - 1) / splits;
    const int b_begin = min(nblk_total, rank * per_split);
    const int b_end = min(nblk_total, b_begin + per_split);
    const int nb = b_end - b_begin;
    const int j0 = b_begin * kRows;             // first list entry of this CTA
    const int j1 = min(p.topk, b_end * kRows);  // one past the last
    const int32_t* idx_row = p.indices + static_cast<int64_t>(t) * p.topk;

    // ---- set-up
    if (threadIdx.x == 0) {
        *sAbort = 0;
        ptx::mbar_init(bar(kBarQ), 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(kBarKvFull + s), 32 * kTcProducers);
            ptx::mbar_init(bar(kBarKvEmpty + s), 1);
            ptx::mbar_init(bar(kBarSFull + s), 1);
            ptx::mbar_init(bar(kBarSEmpty + s), 4);
        }
        ptx::mbar_init(bar(kBarPFull), 4);
        ptx::mbar_init(bar(kBarPvDone), 1);
        ptx::mbar_init(bar(kBarPvDone + 1), 1);
        ptx::mbar_init(bar(kBarDrain), 2);  // one commit from each issuer
        ptx::fence_mbarrier_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(sbase + L::kOffMisc, L::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp >= 1 && warp <= kTcProducers && p.h < HP) {
        // zero the query rows h..HP-1 of every panel (the MMA N padding of h = 8)
        const int pad_rows = HP - p.h;
        const int n16 = kPanels * pad_rows * 8;
        for (int i = threadIdx.x - 32; i < n16; i += 32 * kTcProducers) {
            const int pn = i / (pad_rows * 8);
            const int rem = i % (pad_rows * 8);
            *reinterpret_cast<uint4*>(smem + L::kOffQ + pn * HP * 128 + (p.h + rem / 8) * 128 +
                                      (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
    }
    if (warp > kTcPvWarp) {
        const int wtid = threadIdx.x - kSoftmaxThread0;
        if (wtid < HP) sM[wtid] = -CUDART_INF_F;
    }
    // launched as a programmatic dependent: nothing above touched global memory
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *sTmem;

    if (warp == 0) {
        // ================================================================ S^T issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(64, HP, 0, 0);
            ptx::prefetch_tmap(&tm_q);
            ptx::mbar_arrive_expect_tx(bar(kBarQ), static_cast<uint32_t>(kPanels * p.h * 128));
            for (int pn = 0; pn < kPanels; ++pn)
                ptx::tma_load_3d(sQ + pn * HP * 128, &tm_q, pn * 64, 0, t, bar(kBarQ));
            // Descriptors differ from a base only in the start-address field (address >> 4,
            // low 14 bits), so each operand is its base descriptor plus a constant.
            const uint64_t dq = ptx::smem_desc_sw128(sQ, 16, 1024);
            const uint64_t dkv = ptx::smem_desc_sw128(sKV, 16, 1024);
            bool ok = wait(kBarQ, 0);
            for (int b = 0; ok && b < nb; ++b) {
                // rows of block b landed; S^T buffer b % 2 read out by the softmax of block b - 2
                const int s = b & 1;
                ok = wait(kBarKvFull + s, (b >> 1) & 1);
                if (ok && b >= 2) ok = wait(kBarSEmpty + s, ((b >> 1) - 1) & 1);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint64_t a0 = dkv + static_cast<uint64_t>((s * kStageBytes) >> 4);
                const uint32_t d = tmem + L::kColS + s * HP;
#pragma unroll
                for (int pn = 0; pn < kPanels; ++pn) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        ptx::mma_bf16_ss(d, a0 + ((pn * kPanelBytes + k * 32) >> 4),
                                         dq + ((pn * HP * 128 + k * 32) >> 4), kIdescS, (pn | k) != 0);
                    }
                }
                ptx::mma_commit(bar(kBarSFull + s));
            }
            // every MMA of both issuers done before TMEM is read out or released; an aborted
            // CTA also waits for its Q copy so that nothing is in flight when it leaves
            ptx::mma_commit(bar(kBarDrain));
            ptx::mbar_wait(bar(kBarDrain), 0, nullptr, &g_smla_error, 0u, kDrainLimitNs);
            if (*sAbort) ptx::mbar_wait(bar(kBarQ), 0, nullptr, &g_smla_error, 0u, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp <= kTcProducers) {
        // ================================================================ producers
        gather_rows<kRows, kStages, KVF, kTcProducers>(p, idx_row, j0, j1, nb, warp - 1, lane, sKV,
                                                       bar(kBarKvFull), bar(kBarKvEmpty), sAbort);
    } else if (warp == kTcPvWarp) {
        // ================================================================ PV issuer
        if (lane == 0) {
            constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, HP, 1, 0);
            const uint64_t dv = ptx::smem_desc_sw128(sKV, kPanelBytes, 1024);
            const uint64_t dp = ptx::smem_desc_sw128(sRope, 16, 1024);  // P^T, stage 0
            for (int b = 0; b < nb; ++b) {
                if (!wait(kBarPFull, b & 1)) break;  // P^T of block b from the softmax
                ptx::tc_fence_after();
                const int s = b & 1;
                const uint64_t v0 = dv + static_cast<uint64_t>((s * kStageBytes) >> 4);
                const uint64_t p0 = dp + static_cast<uint64_t>((s * kStageBytes) >> 4);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t acc = (b > 0 || k > 0) ? 1u : 0u;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        ptx::mma_bf16_ss(tmem + i * HP, v0 + ((2 * i * kPanelBytes + k * 2048) >> 4),
                                         p0 + ((k * 32) >> 4), kIdescPV, acc);
                }
                ptx::mma_commit(bar(kBarKvEmpty + s));
                ptx::mma_commit(bar(kBarPvDone + s));
            }
            ptx::mma_commit(bar(kBarDrain));
        }
        __syncwarp();
    } else {
        // ================================================================ softmax warpgroup
        // Warp `quad` owns block rows quad*16 .. quad*16+15 (M=64 accumulator: TMEM lanes
        // 32*quad + 0..15).  The 16x256b TMEM load hands thread (g = lane/4, tq = lane%4) rows
        // g and g+8 of them and, in each 8-column group i, heads 8i + 2tq and 8i + 2tq + 1 (the
        // mma accumulator layout), so all 32 lanes work.
        const int wtid = threadIdx.x - kSoftmaxThread0;
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const int g = lane >> 2, tq = lane & 3;
        const int r0 = quad * 16 + g, r1 = r0 + 8;
        constexpr int NG = HP / 8;
        const float c = p.sm_scale_log2;
        bool failed = false;
        // raw list entries of this thread's two rows for the next block (checked when used)
        int raw0 = fetch_entry(idx_row, j0 + r0, j1, nb > 0);
        int raw1 = fetch_entry(idx_row, j0 + r1, j1, nb > 0);
        // P^T[h][r] of a block in stage s (128B-swizzled K-major rows of 64 bf16, eight heads
        // per 1 KB atom), over the stage's rope panel: the logits are done with it, and the
        // stage is refilled only after this block's PV
        auto p_addr = [&](int s, int h, int r) -> uint32_t {
            return sRope + static_cast<uint32_t>(s * kStageBytes) + (h >> 3) * 1024 + (h & 7) * 128 +
                   ((((r >> 3) ^ (h & 7)) << 4) | ((r & 7) << 1));
        };
        // fp32 partial softmax sums of this thread's heads 8i + 2tq + e over its two rows
        float lsum[NG][2];
#pragma unroll
        for (int i = 0; i < NG; ++i) lsum[i][0] = lsum[i][1] = 0.f;

        for (int b = 0; b < nb; ++b) {
            const int s = b & 1;
            const bool v0 = valid_slot(raw0, p.num_slots) >= 0;
            const bool v1 = valid_slot(raw1, p.num_slots) >= 0;
            raw0 = fetch_entry(idx_row, j0 + (b + 1) * kRows + r0, j1, b + 1 < nb);
            raw1 = fetch_entry(idx_row, j0 + (b + 1) * kRows + r1, j1, b + 1 < nb);
            bool ok = true;
            if (lane == 0) ok = wait(kBarSFull + s, (b >> 1) & 1);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            // sv[i] = {row g: head 8i+2tq, 8i+2tq+1 | row g+8: same heads}, as scaled logits
            uint32_t sv[NG][4];
            bool need = false;
            if (ok) {
                ptx::tc_fence_after();
#pragma unroll
                for (int i = 0; i < NG; ++i) ptx::tmem_ld_16x256b(tmem + lane_base + L::kColS + s * HP + 8 * i, sv[i]);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(kBarSEmpty + s));
#pragma unroll
                for (int i = 0; i < NG; ++i) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float mo = sM[8 * i + 2 * tq + e] + kRescaleLog2;
                        const float x0 = v0 ? __uint_as_float(sv[i][e]) * c : -CUDART_INF_F;
                        const float x1 = v1 ? __uint_as_float(sv[i][2 + e]) * c : -CUDART_INF_F;
                        sv[i][e] = __float_as_uint(x0);
                        sv[i][2 + e] = __float_as_uint(x1);
                        need |= (x0 > mo) || (x1 > mo);
                    }
                }
            } else {
                failed = true;
#pragma unroll
                for (int i = 0; i < NG; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sv[i][e] = __float_as_uint(-CUDART_INF_F);
            }
            // one warpgroup barrier per block in the common case (no new max, no abort)
            if (ptx::named_bar_red_or(1, 128, need || failed || *sAbort)) {
                if (ptx::named_bar_red_or(1, 128, failed || *sAbort)) {
                    failed = true;
                    break;
                }
                // the running max of some head grew: new max, rescale O and the partial sums
#pragma unroll
                for (int i = 0; i < NG; ++i) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float mx = fmaxf(__uint_as_float(sv[i][e]), __uint_as_float(sv[i][2 + e]));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        if (g == 0) sRed[quad * HP + 8 * i + 2 * tq + e] = mx;
                    }
                }
                ptx::named_bar_sync(1, 128);
                if (wtid < HP) {
                    const float mo = sM[wtid];
                    const float mb = fmaxf(fmaxf(sRed[wtid], sRed[HP + wtid]),
                                           fmaxf(sRed[2 * HP + wtid], sRed[3 * HP + wtid]));
                    const float mn = fmaxf(mo, mb);
                    sAlpha[wtid] = (mo == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(mo - mn);
                    sM[wtid] = mn;
                }
                ptx::named_bar_sync(1, 128);
#pragma unroll
                for (int i = 0; i < NG; ++i) {
                    lsum[i][0] *= sAlpha[8 * i + 2 * tq];
                    lsum[i][1] *= sAlpha[8 * i + 2 * tq + 1];
                }
                if (b > 0) {  // O^T complete: PV(b - 1) done
                    bool okw = true;
                    if (lane == 0) okw = wait(kBarPvDone + ((b - 1) & 1), ((b - 1) >> 1) & 1);
                    okw = __shfl_sync(0xffffffffu, okw, 0);
                    __syncwarp();
                    if (okw) {
                        ptx::tc_fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < HP / 16; ++cc) {
                            float a[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) a[e] = sAlpha[cc * 16 + e];
#pragma unroll 1
                            for (int blk = 0; blk < 4; ++blk) {  // the four O^T column blocks
                                uint32_t o[16];
                                const uint32_t ta = tmem + lane_base + blk * HP + cc * 16;
                                SMLA_TMEM_LD16(ta, o);
                                ptx::tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    o[e] = __float_as_uint(__uint_as_float(o[e]) * a[e]);
                                SMLA_TMEM_ST16(ta, o);
                            }
                        }
                        ptx::tmem_wait_st();
                    } else {
                        failed = true;
                    }
                }
            }
            // P = 2^(x - m) for this thread's 2 rows x 2*NG heads
            uint16_t pb[NG][4];
#pragma unroll
            for (int i = 0; i < NG; ++i) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float m = sM[8 * i + 2 * tq + e];
                    const float x0 = __uint_as_float(sv[i][e]), x1 = __uint_as_float(sv[i][2 + e]);
                    const float p0 = (x0 == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(x0 - m);
                    const float p1 = (x1 == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(x1 - m);
                    lsum[i][e] += p0 + p1;
                    pb[i][e] = bf16_bits(p0);
                    pb[i][2 + e] = bf16_bits(p1);
                }
            }
#pragma unroll
            for (int i = 0; i < NG; ++i) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = 8 * i + 2 * tq + e;
                    ptx::st_shared_u16(p_addr(s, h, r0), pb[i][e]);
                    ptx::st_shared_u16(p_addr(s, h, r1), pb[i][2 + e]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kBarPFull));
        }

        // ---- the last PV, then per-head totals L = sum of the threads' partial sums
        const bool aborted = ptx::named_bar_red_or(1, 128, failed || *sAbort);
        failed = aborted;
        if (nb > 0 && !aborted) {
            bool okw = true;
            if (lane == 0) okw = wait(kBarPvDone + ((nb - 1) & 1), ((nb - 1) >> 1) & 1);
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            if (okw) ptx::tc_fence_after();
            failed = !okw;
        }
        const bool have_o = nb > 0 && !failed;
#pragma unroll
        for (int i = 0; i < NG; ++i) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = lsum[i][e];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                if (g == 0) sRed[quad * HP + 8 * i + 2 * tq + e] = v;
            }
        }
        ptx::named_bar_sync(1, 128);
        if (wtid < HP) {
            const float tot =
                have_o ? sRed[wtid] + sRed[HP + wtid] + sRed[2 * HP + wtid] + sRed[3 * HP + wtid] : 0.f;
            sML[wtid] = sM[wtid];
            sML[HP + wtid] = tot;
            sAlpha[wtid] = tot > 0.f ? 1.0f / tot : 0.f;
        }
        ptx::named_bar_sync(1, 128);

        if (splits == 1 && !aborted) {
            // O = O^T / L as bf16, staged as out[t] ([h][512], contiguous) in the free stage memory,
            // then written with 16-byte stores
            uint16_t* so = reinterpret_cast<uint16_t*>(smem + L::kOffKV);
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const int d = i * 128 + quad * 32 + lane;
#pragma unroll 1
                for (int cc = 0; cc < HP / 16; ++cc) {
                    uint32_t ov[16];
                    if (have_o) {
                        SMLA_TMEM_LD16(tmem + lane_base + i * HP + cc * 16, ov);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) ov[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int h = cc * 16 + e;
                        if (h < p.h) so[h * kDV + d] = bf16_bits(__uint_as_float(ov[e]) * sAlpha[h]);
                    }
                }
            }
            ptx::named_bar_sync(1, 128);
            const uint4* src = reinterpret_cast<const uint4*>(so);
            uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(t) * p.h * kDV);
            for (int v = wtid; v < p.h * (kDV / 8); v += 128) dst[v] = src[v];
            if (wtid < p.h) {
                const float tot = sML[HP + wtid];
                p.lse[static_cast<int64_t>(t) * p.h + wtid] =
                    tot > 0.f ? (sML[wtid] + log2f(tot)) * 0.69314718055994531f : -CUDART_INF_F;
            }
        }
        ptx::tc_fence_before();
        if (splits > 1 && failed) sAbort[0] = 1;
    }

    __syncthreads();

    if (splits > 1) {
        // ================================================================ cluster merge
        ptx::cluster_sync();  // every CTA's (m, L) is in its shared memory
        float* obuf = reinterpret_cast<float*>(smem + L::kOffKV);  // [HP][512] fp32
        if (warp > kTcPvWarp) {
            const int wtid = threadIdx.x - kSoftmaxThread0;
            const int quad = warp & 3;
            const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
            const bool have_o = nb > 0 && *sAbort == 0;
            if (wtid < HP) {
                const uint32_t a_m = ptx::smem_u32(sML + wtid);
                const uint32_t a_l = ptx::smem_u32(sML + HP + wtid);
                float mk[kMaxSplits], lk[kMaxSplits];
#pragma unroll
                for (int k = 0; k < kMaxSplits; ++k) {
                    mk[k] = k < splits ? ptx::ld_shared_cluster_f32(ptx::map_shared_rank(a_m, k)) : -CUDART_INF_F;
                    lk[k] = k < splits ? ptx::ld_shared_cluster_f32(ptx::map_shared_rank(a_l, k)) : 0.f;
                }
                float M = -CUDART_INF_F;
#pragma unroll
                for (int k = 0; k < kMaxSplits; ++k) M = fmaxf(M, mk[k]);
                float Lt = 0.f;
#pragma unroll
                for (int k = 0; k < kMaxSplits; ++k)
                    if (mk[k] != -CUDART_INF_F && lk[k] > 0.f) Lt += lk[k] * ptx::ex2_approx(mk[k] - M);
                const float mine = sML[wtid];
                sAlpha[wtid] = (Lt > 0.f && mine != -CUDART_INF_F && sML[HP + wtid] > 0.f)
                                   ? ptx::ex2_approx(mine - M) / Lt
                                   : 0.f;
                if (rank == 0 && wtid < p.h)
                    p.lse[static_cast<int64_t>(t) * p.h + wtid] =
                        Lt > 0.f ? (M + log2f(Lt)) * 0.69314718055994531f : -CUDART_INF_F;
            }
            ptx::named_bar_sync(1, 128);
            if (have_o) ptx::tc_fence_after();
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const int d = i * 128 + quad * 32 + lane;
#pragma unroll 1
                for (int cc = 0; cc < HP / 16; ++cc) {
                    uint32_t ov[16];
                    if (have_o) {
                        SMLA_TMEM_LD16(tmem + lane_base + i * HP + cc * 16, ov);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) ov[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        obuf[(cc * 16 + e) * kDV + d] = __uint_as_float(ov[e]) * sAlpha[cc * 16 + e];
                }
            }
            ptx::tc_fence_before();
        }
        ptx::cluster_sync();  // every CTA's weighted partial O is in its shared memory
        if (warp > kTcPvWarp) {
            // this CTA sums dims [rank*ds, (rank+1)*ds) of every head over the cluster,
            // eight dims per item, and stores them as one 16-byte vector
            const int wtid = threadIdx.x - kSoftmaxThread0;
            const int ds = kDV / splits;
            const int per_head = ds / 8;
            const uint32_t ob = ptx::smem_u32(obuf);
            for (int it = wtid; it < p.h * per_head; it += 128) {
                const int hh = it / per_head;
                const int d0 = rank * ds + (it % per_head) * 8;
                const uint32_t a = ob + static_cast<uint32_t>((hh * kDV + d0) * 4);
                float4 lo[kMaxSplits], hi[kMaxSplits];
#pragma unroll
                for (int k = 0; k < kMaxSplits; ++k) {
                    if (k < splits) {
                        const uint32_t ra = ptx::map_shared_rank(a, k);
                        lo[k] = ptx::ld_shared_cluster_v4(ra);
                        hi[k] = ptx::ld_shared_cluster_v4(ra + 16);
                    } else {
                        lo[k] = hi[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < kMaxSplits; ++k) {
                    acc[0] += lo[k].x; acc[1] += lo[k].y; acc[2] += lo[k].z; acc[3] += lo[k].w;
                    acc[4] += hi[k].x; acc[5] += hi[k].y; acc[6] += hi[k].z; acc[7] += hi[k].w;
                }
                uint4 packed;
                packed.x = pack_bf16x2(acc[0], acc[1]);
                packed.y = pack_bf16x2(acc[2], acc[3]);
                packed.z = pack_bf16x2(acc[4], acc[5]);
                packed.w = pack_bf16x2(acc[6], acc[7]);
                *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * p.h + hh) * kDV + d0) = packed;
            }
        }
        ptx::cluster_sync();  // no CTA leaves while a peer still reads its shared memory
    }

    // ---- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace smla
