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
// Rows arrive in 32-row stages (six in flight at 8 heads, five at 16; fp8 rows through a raw
// ring, see small_gather) gathered by seven producer warps (eight for fp8).  Each compute warp takes eight of the
// block's rows for the softmax: masking, a running max per head in log2 units with conditional
// rescaling (only when the max grows by more than 2^8), fp32 partial sums, P^T (bf16) to shared
// memory.
//
// Work partition: the T * nblk row blocks (nblk = ceil(topk / 32) per token, token-major) are
// cut into `grid` equal contiguous ranges, one per CTA.  A CTA walks its range as consecutive
// token segments; its producers stream straight across token boundaries.  A token whose whole
// list lies in one CTA is normalised and stored directly.  When every list falls into 2, 4 or 8
// whole parts (the default below one CTA per SM) the parts of a token form a thread-block
// cluster and merge through distributed shared memory; otherwise (cuts anywhere, explicit split
// counts only) each part leaves (m, L, unnormalised O) in a global scratch slot and, after a
// grid-wide barrier, every participant merges one slice of the output dims.  Both merges weigh
// the parts by 2^(m_j - M) / sum_j L_j 2^(m_j - M) in a fixed order, so results repeat bit for
// bit.
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kSmRows = 32;                                          // KV rows per stage
constexpr int kSmStagesBf16 = 5;                                     // bf16 cache: operand stages
constexpr int kSmStagesBf16H8 = 6;                                   // (six fit at 8 heads)
constexpr int kSmStagesFp8 = 3;                                      // fp8 cache: operand stages ...
constexpr int kSmRawStages = 4;                                      // ... fed by a raw-row ring
constexpr int kSmRawStageBytes = kSmRows * kFp8RowBytes;             // 20992
constexpr int kSmComputeWarps = 4;
// Warp roles: producer warps first, then the four compute warps.  The fp8 cache takes eight
// producers (each dequantises four rows of a block; 384 threads), bf16 seven (352 threads).
// Measured on the four-sequence fp8 batch: 4.48 -> 4.40 ms with the eighth warp; rows
// assigned so each SM sub-partition (warp % 4) dequantises eight rows, with one warp taking
// eight, ran at 6.15 ms: the warp with the most rows sets the pace.
template <int KVF>
struct SmRoles {
    static constexpr int kProducers = KVF == 1 ? 8 : kProducerWarps;
    static constexpr int kThreads = 32 * (kProducers + kSmComputeWarps);
    static constexpr int kCompute0 = 32 * kProducers;  // first compute thread
};
constexpr int kSmKSteps = kDQK / 16 / kSmComputeWarps;               // 9 k-steps per warp
// Stage layout: row r at r * 1168 bytes (1152 + 16).  Consecutive rows then start four banks
// apart, so the eight row addresses of every ldmatrix hit disjoint banks without a swizzle, and
// a whole row can be copied as one contiguous block.
constexpr int kSmRowStride = 1168;
constexpr int kSmStageBytes = kSmRows * kSmRowStride;                 // 37376
// bf16 rows [0, kSmBulkRows) of each stage are copied by one producer warp with one bulk copy
// (TMA) per row, the other rows by six warps with 16-byte cp.async.  Measured on the decode
// batch, 0 to 20 bulk rows per stage run within 2 % of each other (the SM streams about
// 44 GB/s either way) and 24 or more are slower; 14 keeps both engines in use.
constexpr int kSmBulkRows = 14;
// Cluster merge: a CTA's unnormalised O^T as [h][516] fp32 in its own stage memory.  516 = 512 + 4
// puts the fragment stores of a warp (heads 2*tq (+1), dims g) on 32 distinct banks and keeps
// every head row 16-byte aligned for the vector loads of the other CTAs.
constexpr int kSmLocStride = kDV + 4;

template <int H, int KVF>
struct SmallLayout {
    static_assert(H == 8 || H == 16, "the small-head kernel runs 8 or 16 heads");
    static constexpr int kNT = H / 8;                                // n-tiles of 8 heads
    static constexpr int kStages = KVF == 1 ? kSmStagesFp8 : (H == 8 ? kSmStagesBf16H8 : kSmStagesBf16);
    static constexpr int kStageBytes = kSmStageBytes;
    static constexpr int kOffKV = 0;
    static constexpr int kOffRaw = kStages * kStageBytes;            // fp8: raw 656-byte rows
    static constexpr int kRawBytes = KVF == 0 ? 0 : kSmRawStages * kSmRawStageBytes;
    static constexpr int kOffRed = kOffRaw + kRawBytes;              // S partials, float4 per lane
    static constexpr int kRedBytes = kSmComputeWarps * 2 * kNT * 32 * 16;
    static constexpr int kPStride = 80;                              // bytes per head row of P^T
    static constexpr int kOffP = kOffRed + kRedBytes;
    static constexpr int kOffHr = kOffP + H * kPStride;              // [4][H] per-warp reductions
    static constexpr int kOffM = kOffHr + kSmComputeWarps * H * 4;   // running max (log2 units)
    static constexpr int kOffAlpha = kOffM + H * 4;                  // rescale factor / 1/L
    static constexpr int kOffML = kOffAlpha + H * 4;                 // segment m[H], L[H]
    static constexpr int kOffBar = kOffML + 2 * H * 4;               // full[stages], empty[stages]
    static constexpr int kOffMisc = kOffBar + 2 * kStages * 8;       // abort flag
    static constexpr int kOffMask = kOffMisc + 16;                   // valid-row mask per stage
    static constexpr int kOffMrg = kOffMask + 32;                    // merge: m, L, weight [16][H] each
    static constexpr int kBytes = kOffMrg + 3 * kMaxParts * H * 4;
    // scratch slot of one partial segment: m[H], L[H], then O^T unnormalised as [H][512] fp32
    static constexpr int kSlotFloats = 2 * H + H * kDV;
    static_assert(kOffP % 16 == 0 && kOffRaw % 16 == 0, "16-byte aligned shared buffers");
    static_assert(H * kDV * 2 <= kStages * kStageBytes, "output staging fits the stages");
    static_assert(kStages * 4 <= 32, "stage masks fit their slot");
    static_assert(H * kSmLocStride * 4 + 2 * H * 4 <= kStages * kStageBytes, "cluster merge buffers fit the stages");
    static_assert(kBytes <= 232448, "shared memory budget (227 KB)");
    static_assert(kOffBar % 8 == 0, "mbarrier alignment");
};

// Balanced partition of W row blocks over G CTAs: CTA i takes q + (i < r) blocks (q = W / G,
// r = W % G), starting at flat_begin(i).  G <= W, so q >= 1 and no range is empty.
__device__ __forceinline__ int64_t flat_begin(int64_t i, int64_t q, int64_t r) { return i * q + (i < r ? i : r); }

// The CTA whose range holds block x.
__device__ __forceinline__ int64_t flat_owner(int64_t x, int64_t q, int64_t r) {
    const int64_t big = r * (q + 1);
    return x < big ? x / (q + 1) : r + (x - big) / q;
}

// Grid-wide barrier of a cooperative launch (sense reversal): bar[0] counts arrivals, bar[32]
// is the generation.  Each CTA reads the generation, then arrives; the last arrival resets the
// count and advances the generation, which releases the others.  The count is back at zero after
// every completed barrier, so launches of any grid size (and CUDA graph replays) can share the
// words.  Bounded: gives up after kWaitLimitNs and reports a timeout.
__device__ __forceinline__ bool grid_barrier(unsigned int* bar, unsigned int grid) {
    unsigned int* count = bar;
    unsigned int* gen = bar + 32;  // its own 128-byte line
    const unsigned int g = ptx::ld_acquire_gpu_u32(gen);
    if (atomicAdd(count, 1u) == grid - 1u) {
        *reinterpret_cast<volatile unsigned int*>(count) = 0u;
        ptx::st_release_gpu_u32(gen, g + 1u);
        return true;
    }
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::ld_acquire_gpu_u32(gen) == g) {
        if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_smla_error, kErrTimeout);
            return false;
        }
        __nanosleep(100);
    }
    return true;
}

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

// Full-barrier arrivals per stage: bf16 -> six cp.async warps (one per thread) + the bulk warp's
// lane 0 (with the expected bytes); fp8 -> all seven warps (one per thread).
template <int KVF>
__host__ __device__ constexpr int small_full_count() {
    return KVF == 0 ? 32 * (kProducerWarps - 1) + 1 : 32 * SmRoles<1>::kProducers;
}

// KV row gather of the small-head kernel (producer warp pw), into NST stages of kSmRows
// rows in the padded row-major layout.  Invalid entries become zero rows.  Lane i of every
// producer warp holds the list entry of row i; the last warp also publishes the stage's mask of
// valid rows (bit i = row i) in sMask[stage] before its arrival on the full barrier, so the
// compute warps read validity from shared memory after their wait.
//   bf16: warp 6 takes rows [0, kSmBulkRows), one row per lane, one cp.async.bulk of 1152 bytes
//         each; warps 0-5 take rows kSmBulkRows + pw + 6 i with 16-byte cp.async.
//   fp8:  warps 0-7 take rows pw + 8 i.  Raw 656-byte rows are copied with cp.async into a ring
//         of kSmRawStages blocks, kSmRawStages - 1 blocks ahead of use (about 63 KB in flight);
//         then each lane dequantises 16 latent bytes of a row with its tile scale (e4m3 -> f16
//         exactly, x scale in fp32, -> bf16 round to nearest even) into the bf16 operand stage,
//         and lanes 0-7 copy the 128 bf16 rope bytes.
template <int KVF, int NST>
__device__ __forceinline__ void small_gather(const FwdParams& p, int64_t x0, int nb, int pw, int lane, uint32_t sKV,
                                             uint32_t sRaw, uint32_t bar_full0, uint32_t bar_empty0,
                                             uint32_t sMask, volatile int* sAbort) {
    // List entries are loaded kAhead blocks (256 entries) ahead into a ring indexed by
    // b % kAhead; the block loop is unrolled kAhead times so each ring index is static and an
    // entry is first read kAhead blocks after its load was issued.
    constexpr int kAhead = 8;
    constexpr int kRow0 = KVF == 0 ? kSmBulkRows : 0;
    constexpr int kWarps = KVF == 0 ? kProducerWarps - 1 : SmRoles<1>::kProducers;
    constexpr int kPerWarp = (kSmRows - kRow0 + kWarps - 1) / kWarps;
    constexpr uint32_t kBulkMask = kSmBulkRows >= 32 ? 0xffffffffu : ((1u << kSmBulkRows) - 1u);
    const bool mask_warp = pw == SmRoles<KVF>::kProducers - 1;
    // fetch cursor: token ft, first list entry fj of the next block to fetch (blocks x0, x0+1, ...)
    const int kpad = p.nblk * kSmRows;
    int ft = static_cast<int>(x0 / p.nblk);
    int fj = static_cast<int>(x0 - static_cast<int64_t>(ft) * p.nblk) * kSmRows;
    auto fetch = [&](bool pred) -> int {
        const int v = fetch_entry(p.indices + static_cast<int64_t>(ft) * p.topk, fj + lane, p.topk, pred);
        fj += kSmRows;
        if (fj >= kpad) {
            fj = 0;
            ++ft;
        }
        return v;
    };
    int ring[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) ring[u] = fetch(u < nb);
    // fp8: this warp's rows pw + 7 i of block bb, raw (656 bytes each) into raw stage
    // bb % kSmRawStages: lanes copy the 32 latent chunks, lanes 0-8 the scales and rope.
    // Invalid entries copy nothing and leave zeros (src-size 0), which dequantise to zeros.
    auto issue_raw = [&](int bb, int slot_lane) {
        const uint32_t rs = sRaw + (bb % kSmRawStages) * kSmRawStageBytes;
        const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) {
            const int r = pw + kWarps * i;
            if (r < kSmRows) {
                const int slot = __shfl_sync(0xffffffffu, slot_lane, r);
                const uint8_t* src = kv8 + static_cast<int64_t>(slot < 0 ? 0 : slot) * kFp8RowBytes;
                const uint32_t nbytes = slot < 0 ? 0u : 16u;
                const uint32_t rd = rs + r * kFp8RowBytes;
                ptx::cp_async_16(rd + lane * 16, src + lane * 16, nbytes);
                if (lane < 9) ptx::cp_async_16(rd + 512 + lane * 16, src + 512 + lane * 16, nbytes);
            }
        }
    };
    if constexpr (KVF == 1) {
#pragma unroll
        for (int k = 0; k + 1 < kSmRawStages; ++k) {
            if (k < nb) issue_raw(k, valid_slot(ring[k], p.num_slots));
            ptx::cp_async_commit();
        }
    }
    bool aborted = false;
    for (int b0 = 0; b0 < nb && !aborted; b0 += kAhead) {
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const int b = b0 + u;
            if (b >= nb) break;
            const int s = b % NST;
            const uint32_t full = bar_full0 + 8u * s;
            const int my_slot = valid_slot(ring[u], p.num_slots);  // slot of row `lane`
            if (p.checked && mask_warp) flag_out_of_range(ring[u], my_slot);
            if constexpr (KVF == 1) {
                // raw rows of block b + kSmRawStages - 1 (their entries sit in the ring already)
                const int ahead = valid_slot(ring[(u + kSmRawStages - 1) % kAhead], p.num_slots);
                if (b + kSmRawStages - 1 < nb) issue_raw(b + kSmRawStages - 1, ahead);
                ptx::cp_async_commit();  // one group per block, empty past the end
            }
            ring[u] = fetch(b + kAhead < nb);
            const uint32_t vmask = __ballot_sync(0xffffffffu, my_slot >= 0);
            if (b >= NST) {
                bool ok = true;
                if (lane == 0)
                    ok = ptx::mbar_wait(bar_empty0 + 8u * s, ((b / NST) - 1) & 1, sAbort, &g_smla_error,
                                        kErrTimeout, kWaitLimitNs);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                __syncwarp();
                if (!ok) {
                    aborted = true;
                    break;
                }
            }
            const uint32_t st = sKV + s * kSmStageBytes;
            if constexpr (KVF == 0) {
                if (mask_warp) {
                    const bool bulk_row = lane < kSmBulkRows;
                    if (bulk_row && my_slot < 0)  // zero row; written before this warp's arrive below
                        for (int c = 0; c < 72; ++c)
                            ptx::st_shared_v4(st + lane * kSmRowStride + c * 16, make_uint4(0u, 0u, 0u, 0u));
                    __syncwarp();
                    if (lane == 0) {
                        ptx::st_shared_u32(sMask + 4u * s, vmask);
                        ptx::mbar_arrive_expect_tx(full, __popc(vmask & kBulkMask) * (kDQK * 2));
                    }
                    __syncwarp();
                    if (bulk_row && my_slot >= 0)
                        ptx::bulk_load(st + lane * kSmRowStride,
                                       reinterpret_cast<const char*>(p.kv) + static_cast<int64_t>(my_slot) * (kDQK * 2),
                                       kDQK * 2, full);
                } else {
#pragma unroll 1
                    for (int i = 0; i < kPerWarp; ++i) {
                        const int r = kRow0 + pw + kWarps * i;
                        if (r >= kSmRows) break;
                        const int slot = __shfl_sync(0xffffffffu, my_slot, r);
                        const char* src =
                            reinterpret_cast<const char*>(p.kv) + static_cast<int64_t>(slot < 0 ? 0 : slot) * (kDQK * 2);
                        const uint32_t nbytes = slot < 0 ? 0u : 16u;
#pragma unroll
                        for (int cc = 0; cc < 3; ++cc) {
                            const int c = lane + 32 * cc;  // 16-byte chunk of the 1152-byte row
                            if (c < 72) ptx::cp_async_16(st + r * kSmRowStride + c * 16, src + c * 16, nbytes);
                        }
                    }
                    ptx::cp_async_arrive_noinc(full);
                }
            } else {
                // block b's raw rows are complete for this thread's own copies once at most
                // kSmRawStages - 1 younger groups are pending; the warp barrier shares them
                ptx::cp_async_wait_group<kSmRawStages - 1>();
                __syncwarp();
                const uint32_t rs = sRaw + (b % kSmRawStages) * kSmRawStageBytes;
#pragma unroll
                for (int i = 0; i < kPerWarp; ++i) {
                    const int r = pw + kWarps * i;
                    if (r < kSmRows) {
                        // lane l converts dims [8l, 8l + 8) and [256 + 8l, 256 + 8l + 8): each of the
                        // two stores below then writes 512 contiguous bytes, without bank conflicts
                        // (16 consecutive dims per lane made every store two-way conflicted: 256 of
                        // ~1600 shared-memory wavefronts per block, measured with ncu)
                        const uint32_t rr = rs + r * kFp8RowBytes;
                        const uint2 la = ptx::ld_shared_v2(rr + 8 * lane);
                        const uint2 lb = ptx::ld_shared_v2(rr + 256 + 8 * lane);
                        const float sa = ptx::ld_shared_f32(rr + 512 + 4 * (lane >> 4));
                        const float sb = ptx::ld_shared_f32(rr + 512 + 4 * (2 + (lane >> 4)));
                        uint4 v0, v1;
                        v0.x = ptx::e4m3x2_scaled_bf16x2(la.x & 0xFFFFu, sa);
                        v0.y = ptx::e4m3x2_scaled_bf16x2(la.x >> 16, sa);
                        v0.z = ptx::e4m3x2_scaled_bf16x2(la.y & 0xFFFFu, sa);
                        v0.w = ptx::e4m3x2_scaled_bf16x2(la.y >> 16, sa);
                        v1.x = ptx::e4m3x2_scaled_bf16x2(lb.x & 0xFFFFu, sb);
                        v1.y = ptx::e4m3x2_scaled_bf16x2(lb.x >> 16, sb);
                        v1.z = ptx::e4m3x2_scaled_bf16x2(lb.y & 0xFFFFu, sb);
                        v1.w = ptx::e4m3x2_scaled_bf16x2(lb.y >> 16, sb);
                        const uint32_t rd = st + r * kSmRowStride;
                        ptx::st_shared_v4(rd + lane * 16, v0);         // dims 8 lane .. +7
                        ptx::st_shared_v4(rd + (32 + lane) * 16, v1);  // dims 256 + 8 lane .. +7
                        if (lane < 8) ptx::st_shared_v4(rd + (64 + lane) * 16, ptx::ld_shared_v4(rr + 528 + 16 * lane));
                    }
                }
                if (mask_warp && lane == 0) ptx::st_shared_u32(sMask + 4u * s, vmask);
                ptx::mbar_arrive(full);
            }
        }
    }
    ptx::cp_async_wait_all();  // no cp.async may still be in flight when the CTA leaves
    if (KVF == 0 && mask_warp && (aborted || *sAbort)) {
        // bulk copies have no per-thread wait: give any still in flight time to land (bounded)
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 2000000ull) {
        }
    }
}

// Q^T fragments (B operand of S^T) of token t for compute warp cw's nine 16-dim k-steps.
template <int H>
__device__ __forceinline__ void load_q_frags(const FwdParams& p, int t, int cw, int lane,
                                             uint32_t (&bq)[kSmKSteps][H / 8][2]) {
    const int g = lane >> 2, tq = lane & 3;
    const __nv_bfloat16* qt = p.q + static_cast<int64_t>(t) * H * kDQK;
#pragma unroll
    for (int kk = 0; kk < kSmKSteps; ++kk) {
#pragma unroll
        for (int nt = 0; nt < H / 8; ++nt) {
            const unsigned int* qr = reinterpret_cast<const unsigned int*>(
                qt + (nt * 8 + g) * kDQK + 16 * (kSmKSteps * cw + kk) + 2 * tq);
            bq[kk][nt][0] = __ldg(qr);
            bq[kk][nt][1] = __ldg(qr + 4);
        }
    }
}

// Cluster merge of token t's list, cut into ns aligned parts, one per CTA of the cluster
// (rank = part).  Every CTA has left its unnormalised O^T as [H][kSmLocStride] fp32 at `loc`
// in its own shared memory, followed by (m, L) per head as [H][2]; the caller has passed a
// cluster barrier since.  Each thread of CTA `rank` takes items (head, 8 output dims) of the
// dims [rank*ds, (rank+1)*ds), ds = 512/ns: it loads that piece of every part and the parts'
// (m, L) with vector loads from the other CTAs' shared memory (all in flight at once), weights
// part j by 2^(m_j - M) / sum_i L_i 2^(m_i - M) (M the largest m_i), sums in part order and
// stores eight bf16.  Rank 0 also stores the LSE.
template <int H>
__device__ __forceinline__ void cluster_pull_merge(const FwdParams& p, int t, uint32_t loc, int ns, int rank) {
    const int ds = kDV / ns;
    const int per_head = ds / 8;
    for (int it = threadIdx.x; it < H * per_head; it += blockDim.x) {
        const int hh = it / per_head;
        const int dd = rank * ds + (it % per_head) * 8;
        // (m, L) of every part, and the first four parts' pieces, in flight together
        float2 ml[kMaxSplits];
        float4 lo[4], hi[4];
#pragma unroll
        for (int j = 0; j < kMaxSplits; ++j)
            if (j < ns)
                ml[j] = ptx::ld_shared_cluster_v2(ptx::map_shared_rank(loc, j) +
                                                  static_cast<uint32_t>((H * kSmLocStride + 2 * hh) * 4));
        auto load4 = [&](int j0) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (j0 + u < ns) {
                    const uint32_t base = ptx::map_shared_rank(loc, j0 + u);
                    lo[u] = ptx::ld_shared_cluster_v4(base + static_cast<uint32_t>((hh * kSmLocStride + dd) * 4));
                    hi[u] = ptx::ld_shared_cluster_v4(base + static_cast<uint32_t>((hh * kSmLocStride + dd + 4) * 4));
                }
            }
        };
        load4(0);
        float M = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < kMaxSplits; ++j)
            if (j < ns) M = fmaxf(M, ml[j].x);
        float Lt = 0.f;
        float w[kMaxSplits];
#pragma unroll
        for (int j = 0; j < kMaxSplits; ++j) {
            w[j] = 0.f;
            if (j < ns && ml[j].x != -CUDART_INF_F && ml[j].y > 0.f) {
                w[j] = ptx::ex2_approx(ml[j].x - M);
                Lt += ml[j].y * w[j];
            }
        }
        const float inv = Lt > 0.f ? 1.0f / Lt : 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j0 = 0; j0 < kMaxSplits; j0 += 4) {
            if (j0 >= ns) break;
            if (j0 > 0) load4(j0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (j0 + u < ns) {
                    const float wj = w[j0 + u] * inv;
                    acc[0] += wj * lo[u].x; acc[1] += wj * lo[u].y; acc[2] += wj * lo[u].z; acc[3] += wj * lo[u].w;
                    acc[4] += wj * hi[u].x; acc[5] += wj * hi[u].y; acc[6] += wj * hi[u].z; acc[7] += wj * hi[u].w;
                }
            }
        }
        uint4 packed;
        packed.x = pack_bf16x2(acc[0], acc[1]);
        packed.y = pack_bf16x2(acc[2], acc[3]);
        packed.z = pack_bf16x2(acc[4], acc[5]);
        packed.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t) * H + hh) * kDV + dd) = packed;
        if (rank == 0 && dd == 0)
            p.lse[static_cast<int64_t>(t) * H + hh] = Lt > 0.f ? (M + log2f(Lt)) * 0.69314718055994531f : -CUDART_INF_F;
    }
}

// CL: the launch is a cluster launch (p.splits > 1, aligned parts merged in the cluster).  The
// merge is compiled only into those kernels: at 16 heads the compute warps sit at the register
// limit of 11 warps per SM (168), and the merge code alone moved their allocation into spills
// (an 80 -> 83 us loss on a 16-head launch that never merges).
template <int H, int KVF, bool CL>
__global__ void __launch_bounds__(SmRoles<KVF>::kThreads, 1) sparse_mla_fwd_small_kernel(const FwdParams p) {
    constexpr int kSmCompute0 = SmRoles<KVF>::kCompute0;
    constexpr int kSmProducers = SmRoles<KVF>::kProducers;
    using L = SmallLayout<H, KVF>;
    constexpr int NT = L::kNT;
    constexpr int NST = L::kStages;
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
    const uint32_t bar_empty0 = sbase + L::kOffBar + 8 * NST;

    // ---- this CTA's blocks [x0, x0 + nb) of the token-major block sequence
    const int64_t W = static_cast<int64_t>(p.T) * p.nblk;
    const int64_t fq = W / p.grid, fr = W % p.grid;
    const int64_t x0 = flat_begin(blockIdx.x, fq, fr);
    const int nb = static_cast<int>(fq + (static_cast<int64_t>(blockIdx.x) < fr ? 1 : 0));

    if (threadIdx.x == 0) {
        *sAbort = 0;
        for (int s = 0; s < NST; ++s) {
            ptx::mbar_init(bar_full0 + 8 * s, small_full_count<KVF>());
            ptx::mbar_init(bar_empty0 + 8 * s, kSmComputeWarps);
        }
        ptx::fence_mbarrier_init();
    }
    if (threadIdx.x >= kSmCompute0 && threadIdx.x - kSmCompute0 < H) sM[threadIdx.x - kSmCompute0] = -CUDART_INF_F;
    // Launched as a programmatic dependent: nothing above reads global memory.  Warp 0 moves the
    // list entries of the CTA's first eight blocks and its first token's q into L2 first: a
    // prefetch returns no data and fills no L1, and L2 is where the previous launch's stores
    // land, so the loads after the wait still see that launch's results.
    if (warp == 0) {
        const int64_t tp = x0 / p.nblk;
        const int jp = static_cast<int>(x0 - tp * p.nblk) * kSmRows;
        const int32_t* ib = p.indices + tp * p.topk + jp;
        if (lane < 8 && jp + lane * 32 < p.topk) ptx::prefetch_l2(ib + lane * 32);
        const char* qb = reinterpret_cast<const char*>(p.q + tp * H * kDQK);
        for (int l = lane; l < H * kDQK * 2 / 128; l += 32) ptx::prefetch_l2(qb + l * 128);
    }
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    __syncthreads();

    if (warp < kSmProducers) {
        // ================================================================ producers
        small_gather<KVF, NST>(p, x0, nb, warp, lane, sKV, sbase + L::kOffRaw, bar_full0, bar_empty0,
                               sbase + L::kOffMask, sAbort);
        if constexpr (CL) {  // the cluster merge: every thread takes part
            ptx::cluster_sync();
            cluster_pull_merge<H>(p, static_cast<int>(x0 / p.nblk), sKV, p.splits,
                                  static_cast<int>(blockIdx.x) % p.splits);
            __syncwarp();
            ptx::cluster_sync();
        }
        return;
    }
    // ==================================================================== compute warps
    const int cw = warp - kSmProducers;   // 0..3
    const int wtid = threadIdx.x - kSmCompute0;
    const int g = lane >> 2;                // MMA fragment row group
    const int tq = lane & 3;                // MMA fragment column pair
    const int li = lane & 7, lj = lane >> 3;  // ldmatrix: row within matrix, matrix index
    const float c = p.sm_scale_log2;
    bool failed = false;

    // O^T accumulators (fragment layout: dims 128*cw + 16*mt + g (+8), heads 8*nt + 2*tq (+1))
    float o[8][NT][4];
    float lsum[NT][2];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) lsum[nt][0] = lsum[nt][1] = 0.f;

    // this warp's softmax rows: 8 of the block's 32 (m-tile cw/2, half cw%2), one per lane group
    const int mt_s = cw >> 1, half = cw & 1;
    const int rr = mt_s * 16 + half * 8 + g;

    // segment cursor: token t, first list entry jb of the current block
    const int kpad = p.nblk * kSmRows;
    const int t_first = static_cast<int>(x0 / p.nblk);
    int t = t_first;
    int jb = static_cast<int>(x0 - static_cast<int64_t>(t) * p.nblk) * kSmRows;
    bool seg_from_start = jb == 0;
    uint32_t bq[kSmKSteps][NT][2];
    load_q_frags<H>(p, t, cw, lane, bq);

    for (int b = 0; b < nb; ++b) {
        const int s = b % NST;
        const uint32_t stb = sKV + s * L::kStageBytes;
        bool ok = true;
        if (lane == 0)
            ok = ptx::mbar_wait(bar_full0 + 8 * s, (b / NST) & 1, sAbort, &g_smla_error, kErrTimeout,
                                kWaitLimitNs);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        if (!ok) failed = true;
        // valid rows of this block, published by the producers before their arrival
        const bool valid = (ptx::ld_shared_u32(sbase + L::kOffMask + 4u * s) >> rr) & 1u;

        // ---- partial S^T over this warp's 144 dims, all 32 rows
        // at 16 heads two accumulator sets (even and odd k-steps) halve the dependent MMA chains
        // (measured: 94 -> 80 us on the h=16 sweep; at 8 heads it costs ~1 %, so one set)
        constexpr bool kTwoSets = NT > 1;
        float cs[2][NT][4], cs2[2][NT][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) cs[mt][nt][e] = cs2[mt][nt][e] = 0.f;
        if (ok) {
#pragma unroll
            for (int kk = 0; kk < kSmKSteps; ++kk) {
                const int K = kSmKSteps * cw + kk;
                const uint32_t kchunk = static_cast<uint32_t>((2 * K + (lj >> 1)) * 16);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int row = mt * 16 + (lj & 1) * 8 + li;
                    uint32_t a[4];
                    mma16816::ldsm_x4(a, stb + row * kSmRowStride + kchunk);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (kTwoSets && (kk & 1))
                            mma16816::mma(cs2[mt][nt], a, bq[kk][nt][0], bq[kk][nt][1]);
                        else
                            mma16816::mma(cs[mt][nt], a, bq[kk][nt][0], bq[kk][nt][1]);
                    }
                }
            }
            if constexpr (kTwoSets) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) cs[mt][nt][e] += cs2[mt][nt][e];
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
                    mma16816::ldsm_x2(bp[0][0], bp[0][1], sP + li * L::kPStride + (16 * kk + 8 * (lj & 1)) * 2);
                } else {
                    uint32_t r4[4];
                    mma16816::ldsm_x4(r4, sP + ((lj >> 1) * 8 + li) * L::kPStride + (16 * kk + 8 * (lj & 1)) * 2);
                    bp[0][0] = r4[0]; bp[0][1] = r4[1];
                    bp[NT - 1][0] = r4[2]; bp[NT - 1][1] = r4[3];
                }
                const int krow = 16 * kk + (lj >> 1) * 8 + li;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int d0 = 128 * cw + 16 * mt;
                    uint32_t a[4];
                    mma16816::ldsm_x4_trans(a, stb + krow * kSmRowStride + (d0 / 8 + (lj & 1)) * 16);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816::mma(o[mt][nt], a, bp[nt][0], bp[nt][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty0 + 8 * s);  // this warp is done with the stage

        const bool token_end = jb + kSmRows >= kpad;
        if (!token_end && b + 1 < nb) {
            jb += kSmRows;
            continue;
        }
        // ================================================================ end of a token segment
        // ---- per-head totals L over the block rows of all four warps
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
            sML[wtid] = sM[wtid];
            sML[H + wtid] = tot;
            sAlpha[wtid] = tot > 0.f ? 1.0f / tot : 0.f;
        }
        ptx::named_bar_sync(1, 128);

        if (seg_from_start && token_end) {
            // ---- the whole list was here: O = O^T / L as bf16.  After the CTA's last block the
            // stage memory is free: out[t] ([h][512]) is staged there and written with 16-byte
            // stores; a list that ends earlier in the range is written straight from registers.
            const bool last = b + 1 == nb;
            uint16_t* so = last ? reinterpret_cast<uint16_t*>(smem + L::kOffKV)
                                : reinterpret_cast<uint16_t*>(p.out + static_cast<int64_t>(t) * H * kDV);
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
            if (last) {
                ptx::named_bar_sync(1, 128);
                const uint4* src = reinterpret_cast<const uint4*>(so);
                uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(t) * H * kDV);
                for (int v = wtid; v < H * (kDV / 8); v += 128) dst[v] = src[v];
            }
            if (wtid < H) {
                const float tot = sML[H + wtid];
                p.lse[static_cast<int64_t>(t) * H + wtid] =
                    tot > 0.f ? (sML[wtid] + log2f(tot)) * 0.69314718055994531f : -CUDART_INF_F;
            }
        } else if (CL) {
            // ---- an aligned part of a list (one per CTA of the cluster): (m, L) stay in sML and
            // O^T in registers for the cluster merge after the loop
        } else {
            // ---- part of a list cut between CTAs: leave (m, L, O^T) in this CTA's slot; the
            // parts are merged after the grid barrier below
            float* slot = p.part + (static_cast<int64_t>(blockIdx.x) * 2 + (t == t_first ? 0 : 1)) * L::kSlotFloats;
            if (wtid < H) {
                slot[wtid] = sML[wtid];
                slot[H + wtid] = sML[H + wtid];
            }
            float* so = slot + 2 * H;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int d = 128 * cw + 16 * mt + g;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int h = nt * 8 + 2 * tq;
                    so[h * kDV + d] = o[mt][nt][0];
                    so[(h + 1) * kDV + d] = o[mt][nt][1];
                    so[h * kDV + d + 8] = o[mt][nt][2];
                    so[(h + 1) * kDV + d + 8] = o[mt][nt][3];
                }
            }
        }
        if (b + 1 == nb) break;
        // ---- next token: fresh running state and its Q^T fragments
        ptx::named_bar_sync(1, 128);  // every warp is done with sM / sML / sAlpha / the staging
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) lsum[nt][0] = lsum[nt][1] = 0.f;
        if (wtid < H) sM[wtid] = -CUDART_INF_F;
        ++t;
        jb = 0;
        seg_from_start = true;
        load_q_frags<H>(p, t, cw, lane, bq);
    }
    if (failed) *sAbort = 1;  // producers still waiting for a free stage give up
    if constexpr (CL) {
        // ================================================================ cluster merge
        // The list of token t is cut into p.splits aligned parts, one per CTA of a thread-block
        // cluster (rank = part).  Every warp is past the end-of-segment barriers, so no warp
        // reads the stages any more: O^T and (m, L) go to this CTA's own stage memory, and after
        // a cluster barrier every thread of the CTA pulls and merges its share of the output
        // (cluster_pull_merge).  The second barrier keeps each CTA's memory alive until the
        // other CTAs have read it.
        const bool have = nb > 0 && !failed;
        float* loc = reinterpret_cast<float*>(smem + L::kOffKV);  // [H][kSmLocStride], then [H][2]
        if (wtid < H) {
            loc[H * kSmLocStride + 2 * wtid] = have ? sML[wtid] : -CUDART_INF_F;
            loc[H * kSmLocStride + 2 * wtid + 1] = have ? sML[H + wtid] : 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d = 128 * cw + 16 * mt + g;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int h = nt * 8 + 2 * tq;
                loc[h * kSmLocStride + d] = have ? o[mt][nt][0] : 0.f;
                loc[(h + 1) * kSmLocStride + d] = have ? o[mt][nt][1] : 0.f;
                loc[h * kSmLocStride + d + 8] = have ? o[mt][nt][2] : 0.f;
                loc[(h + 1) * kSmLocStride + d + 8] = have ? o[mt][nt][3] : 0.f;
            }
        }
        ptx::cluster_sync();
        cluster_pull_merge<H>(p, t, sKV, p.splits, static_cast<int>(blockIdx.x) % p.splits);
        __syncwarp();
        ptx::cluster_sync();
        return;
    }
    if (p.part == nullptr) return;  // every list lay within one CTA

    // ==================================================================== merge of cut lists
    // Every CTA arrives once (also after an abort, so no CTA waits for ever); the launch is
    // cooperative, so all CTAs are resident and the barrier cannot wait on an unscheduled CTA.
    __threadfence();
    ptx::named_bar_sync(1, 128);
    if (wtid == 0) {
        const bool ok = grid_barrier(p.gbar, static_cast<unsigned int>(p.grid));
        if (!ok) *sAbort = 1;
    }
    ptx::named_bar_sync(1, 128);
    if (*sAbort) return;
    __threadfence();
    // This CTA takes, for each cut list it holds a part of (its first and its last token), one
    // slice of the 512 output dims: participant k of n takes dims [8 floor(64k/n), 8 floor(64(k+1)/n)).
    const int t_last = static_cast<int>((x0 + nb - 1) / p.nblk);
    float* mM = reinterpret_cast<float*>(smem + L::kOffMrg);
    float* mL = mM + kMaxParts * H;
    float* mW = mL + kMaxParts * H;
    for (int tt = t_first; tt <= t_last; tt += (t_last > t_first ? t_last - t_first : 1)) {
        const int64_t tok0 = static_cast<int64_t>(tt) * p.nblk;
        const int64_t i_first = flat_owner(tok0, fq, fr);
        const int64_t i_last = flat_owner(tok0 + p.nblk - 1, fq, fr);
        if (i_first == i_last) continue;  // a whole list: already stored
        const int n = static_cast<int>(i_last - i_first + 1);  // <= kMaxParts (host plan)
        const int k = static_cast<int>(blockIdx.x - i_first);
        auto slot_of = [&](int64_t j) -> const float* {
            const int64_t tj = flat_begin(j, fq, fr) / p.nblk;  // first token of CTA j
            return p.part + (j * 2 + (tt == tj ? 0 : 1)) * L::kSlotFloats;
        };
        // items of this CTA's slice: (head, 8 dims); the parts are summed in CTA order, four at
        // a time.  The loads of the first four parts of this thread's first item are issued
        // before the weights are known, so a cut list held by at most four CTAs costs one
        // round trip to L2.
        const int c0 = (64 * k) / n, c1 = (64 * (k + 1)) / n;
        const int items = H * (c1 - c0);
        auto load_group = [&](int it, int j0, float4 (&v)[4][2]) {
            const int hh = it / (c1 - c0);
            const int dd = (c0 + it % (c1 - c0)) * 8;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool in = j0 + u < n;
                const float* oj = slot_of(i_first + (in ? j0 + u : 0)) + 2 * H + hh * kDV + dd;
                v[u][0] = in ? __ldcg(reinterpret_cast<const float4*>(oj)) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[u][1] = in ? __ldcg(reinterpret_cast<const float4*>(oj + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        float4 pre[4][2];
        if (wtid < items) load_group(wtid, 0, pre);
        ptx::named_bar_sync(1, 128);  // the previous list's weights are no longer read
        for (int e = wtid; e < n * H; e += 128) {
            const float* sj = slot_of(i_first + e / H);
            mM[e] = __ldcg(sj + e % H);
            mL[e] = __ldcg(sj + H + e % H);
        }
        ptx::named_bar_sync(1, 128);
        if (wtid < H) {
            float M = -CUDART_INF_F;
            for (int j = 0; j < n; ++j) M = fmaxf(M, mM[j * H + wtid]);
            float Lt = 0.f;
            for (int j = 0; j < n; ++j) {
                const float mj = mM[j * H + wtid], lj = mL[j * H + wtid];
                if (mj != -CUDART_INF_F && lj > 0.f) Lt += lj * ptx::ex2_approx(mj - M);
            }
            const float inv = Lt > 0.f ? 1.0f / Lt : 0.f;
            for (int j = 0; j < n; ++j) {
                const float mj = mM[j * H + wtid], lj = mL[j * H + wtid];
                mW[j * H + wtid] = (mj != -CUDART_INF_F && lj > 0.f) ? ptx::ex2_approx(mj - M) * inv : 0.f;
            }
            if (k == 0)
                p.lse[static_cast<int64_t>(tt) * H + wtid] =
                    Lt > 0.f ? (M + log2f(Lt)) * 0.69314718055994531f : -CUDART_INF_F;
        }
        ptx::named_bar_sync(1, 128);
        for (int it = wtid; it < items; it += 128) {
            const int hh = it / (c1 - c0);
            const int dd = (c0 + it % (c1 - c0)) * 8;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j0 = 0; j0 < n; j0 += 4) {
                float4 v[4][2];
                if (it == wtid && j0 == 0) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        v[u][0] = pre[u][0];
                        v[u][1] = pre[u][1];
                    }
                } else {
                    load_group(it, j0, v);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float w = j0 + u < n ? mW[(j0 + u) * H + hh] : 0.f;
                    acc[0] += w * v[u][0].x; acc[1] += w * v[u][0].y;
                    acc[2] += w * v[u][0].z; acc[3] += w * v[u][0].w;
                    acc[4] += w * v[u][1].x; acc[5] += w * v[u][1].y;
                    acc[6] += w * v[u][1].z; acc[7] += w * v[u][1].w;
                }
            }
            uint4 packed;
            packed.x = pack_bf16x2(acc[0], acc[1]);
            packed.y = pack_bf16x2(acc[2], acc[3]);
            packed.z = pack_bf16x2(acc[4], acc[5]);
            packed.w = pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(tt) * H + hh) * kDV + dd) = packed;
        }
        if (t_last == t_first) break;
    }
}

}  // namespace smla
