// The masked dense route for short prefills (sm_103a): the per-token top-k lists scattered
// into a bit mask, then dense multi-head attention over the request's per-head K and V in
// which the mask alone decides which positions attend.
//
// PR #55738 report, 实现拆解 (implementation breakdown) items 2 and 5: prefills whose top-k
// covers most of the history go through a scatter of the top-k lists (_scatter_topk_single_req)
// and an FA4 attention with a mask_mod instead of the per-token top-k MQA kernel; the
// `_is_masked_mha_available` geometry table gives (heads, qk_nope, qk_rope, v_head) =
// (128, 128, 64, 128) for DeepSeek-V3.2, (64, 192, 64, 256) for GLM-5 and (64, 256, 0, 256) for
// the NoPE layout.  The pages give neither the mask layout nor the arithmetic; read here as:
//   mask row t: ceil(S / 32) uint32 words, bit s % 32 of word s / 32 set iff position s is in
//   token t's list (entries outside [0, S) set nothing, a repeated position sets one bit);
//   per token and head: softmax over the set positions of scale * q.k, O = P.V, natural-log
//   LSE; a row with no bit set gives O = 0 and LSE = -inf.
//
// sparse_mla_scatter_mask_kernel: one CTA per row (grid-stride), the row's words built in shared
// memory with atomic ORs and written with 16-byte stores.  HBM-bound: the lists in, the mask out.
//
// sparse_mla_masked_mha_kernel<DQK, DV>: one CTA per (128-query tile, head).  Unlike the gather,
// every K/V tile is shared by the tile's 128 queries, so this is a dense contraction on the
// tensor cores:
//   S[128 q, 64 keys]  = Q[128 x DQK] . K_tile^T        (M=128, N=64; Q from TMEM, K from smem)
//   O[128 q, DV]      += P[128 x 64] . V_tile[64 x DV]  (M=128, N=DV; P from TMEM, V MN-major)
// TMEM holds S, P (two buffers, bf16 pairs), Q (bf16 pairs, written once) and O; shared memory
// is a K/V ring of as many stages as fit (3 or 4).  Roles (352 threads):
//   warp 0      TMA producer (one thread): Q once into the ring (stage 1 on, before the key-tile
//               pre-pass), then K and V tiles, one copy per tile (a 4-D map whose outer dimension
//               is the 64-wide panel); V runs one tile behind K (K(j) waits for S(j - stages),
//               V(j - 1) for PV(j - 1 - stages), the order in which the tensor cores finish them);
//   warp 1      S issuer (one thread) and TMEM owner: S(j) once its tile has landed and the
//               softmax warps hold S(j - 1) in registers;
//   last warp   PV issuer (one thread): PV(j) once P(j) is in TMEM and V(j) has landed (two
//               issuing threads, because a thread that issued MMAs stalls while the tensor cores
//               run them, and its next wait would leave them idle);
//   warps 2-9   Q from shared memory into TMEM, then softmax and epilogue, kMmParts (two) warps
//               per TMEM lane quadrant, one query row per thread, each on 64 / kMmParts keys of
//               a tile and DV / kMmParts columns of O.  The row's mask bits, a running max in
//               log2 units with O rescaled only when the max grows by more than 2^8 (a barrier
//               reduction per tile over the quadrant's warps says whether any row grew; only then
//               do they swap maxima through shared memory), fp32 row sums per warp, P as bf16
//               pairs into TMEM buffer j % 2.  O / l leaves through shared memory and one TMA
//               store.  (Four warps per quadrant measured 0.679 ms against 0.614 on the 4096-token
//               GLM-5 chunk: the extra barrier arrivals cost more than the shorter passes save.)
// Before the loop the CTA marks the 64-key tiles in which any of its rows has a bit set; only
// those tiles are loaded and multiplied (lists over causal histories never reach past the
// tile's last query, sparse lists skip whole tiles).  Every wait is bounded; a CTA that gives
// up drains its copies and MMAs before it frees TMEM.
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kMmBM = 128;                     // queries per tile (MMA M)
constexpr int kMmBN = 64;                      // keys per tile
constexpr int kMmMaxStages = 4;               // K/V ring depth: as many as shared memory holds, up to 4
constexpr int kMmNumBars = 26;
constexpr int kMmParts = 2;                    // softmax warps per TMEM lane quadrant
constexpr int kMmSoftmaxWarps = 4 * kMmParts;
constexpr int kMmThreads = 96 + 32 * kMmSoftmaxWarps;  // producer, S issuer, softmax warps, PV issuer
constexpr int kMmMaxS = 65536;                 // positions per request
constexpr int kMmMaxTiles = kMmMaxS / kMmBN;   // 1024 key tiles
constexpr int kScatterThreads = 256;
constexpr int kScatterMaxS = 1 << 20;          // the row's words live in shared memory (128 KB)

template <int DQK, int DV>
struct MmLayout {
    static_assert(DQK == 192 || DQK == 256, "q/k head dim 192 or 256");
    static_assert(DV == 128 || DV == 256, "v head dim 128 or 256");
    static constexpr int kQP = DQK / 64;                       // 64-wide panels of k
    static constexpr int kVP = DV / 64;                        // 64-wide panels of v
    static constexpr int kKPanel = kMmBN * 128;                // 64 rows x 128 bytes
    static constexpr int kStageBytes = (kQP + kVP) * kKPanel;  // K tile then V tile
    static constexpr int kFixedBytes = kMmMaxTiles / 8 + kMmMaxTiles * 2 + kMmNumBars * 8 + 16 + kMmParts * kMmBM * 4;
    static constexpr int kStages = (232448 - kFixedBytes) / kStageBytes < kMmMaxStages
                                       ? (232448 - kFixedBytes) / kStageBytes
                                       : kMmMaxStages;
    static constexpr int kOffKV = 0;
    // Q lands (TMA, SW128 panels of 128 rows) in the ring from stage 1 on, until the softmax warps
    // have copied it into TMEM; stage 0 holds the pre-pass's word flags until the first K load
    static constexpr int kQPanel = kMmBM * 128;
    static constexpr int kOffQ = kOffKV + kStageBytes;
    static constexpr int kOffTiles = kOffKV + kStages * kStageBytes;  // active key tiles: bitmap, then list
    static constexpr int kOffList = kOffTiles + kMmMaxTiles / 8;
    static constexpr int kOffBar = kOffList + kMmMaxTiles * 2;
    static constexpr int kOffMisc = kOffBar + kMmNumBars * 8;  // tmem base, abort flag, tile count
    static constexpr int kOffX = kOffMisc + 16;                // row maxima / sums swapped by a warp group
    static constexpr int kBytes = kOffX + kMmParts * kMmBM * 4;
    // TMEM columns: S [0, 64) | P x2 (bf16 pairs) [64, 128) | Q (bf16 pairs) [128, 128 + DQK/2)
    // | O [256, 256 + DV)
    static constexpr int kColS = 0;
    static constexpr int kColP = 64;
    static constexpr int kColQ = 128;
    static constexpr int kColO = 256;
    static constexpr int kTmemCols = 512;
    static_assert(kColQ + DQK / 2 <= kColO && kColO + DV <= kTmemCols, "TMEM columns");
    static_assert(kStages >= 2, "at least two K/V stages");
    static_assert(kOffQ + kQP * kQPanel <= kOffKV + kStages * kStageBytes, "Q fits the ring after stage 0");
    static_assert(kMmMaxS / 32 * 4 + 32 * 4 <= kStageBytes, "word flags and prefix sums fit stage 0");
    static_assert(kVP * kQPanel <= kStages * kStageBytes, "the O tile fits the ring");
    static_assert(kStageBytes % 1024 == 0, "SW128 alignment");
    static_assert(kBytes <= 232448, "shared memory budget (227 KB)");
};

enum : int {
    kMbKFull = 0,    // +stage: the K tile landed
    kMbKEmpty = 4,   // +stage: S of the tile is done, its K panels may be refilled
    kMbVFull = 8,    // +stage: the V tile landed
    kMbVEmpty = 12,  // +stage: PV of the tile is done, its V panels may be refilled
    kMbSFull = 16,
    kMbSEmpty = 17,  // the softmax warps hold S in registers: the next S may be written
    kMbPFull = 18,   // +buffer
    kMbPEmpty = 20,  // +buffer
    kMbPvDone = 22,
    kMbDrain = 23,
    kMbQFull = 24,   // the softmax warps have written Q into TMEM
    kMbQLoad = 25    // Q landed in shared memory
};

struct ScatterParams {
    const int32_t* idx;   // [T, topk] positions
    uint32_t* mask;       // [T, W]
    int64_t S;
    int32_t T, topk, W;
};

__global__ void __launch_bounds__(kScatterThreads)
    sparse_mla_scatter_mask_kernel(const ScatterParams p) {
    extern __shared__ __align__(16) uint32_t words[];
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int W = p.W;
    const bool vec = (W & 3) == 0;  // rows start on 16-byte boundaries
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
        for (int i = threadIdx.x; i < W; i += kScatterThreads) words[i] = 0u;
        __syncthreads();
        const int32_t* row = p.idx + t * p.topk;
        for (int j = threadIdx.x; j < p.topk; j += kScatterThreads) {
            const int v = __ldg(row + j);
            if (v >= 0 && static_cast<int64_t>(v) < p.S) atomicOr(&words[v >> 5], 1u << (v & 31));
        }
        __syncthreads();
        uint32_t* out = p.mask + t * W;
        if (vec) {
            for (int i = threadIdx.x; i < W / 4; i += kScatterThreads)
                reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(words)[i];
        } else {
            for (int i = threadIdx.x; i < W; i += kScatterThreads) out[i] = words[i];
        }
        __syncthreads();
    }
}

struct MmParams {
    __nv_bfloat16* out;      // [T, h, DV]
    float* lse;              // [T, h]
    const uint32_t* mask;    // [T, W]
    int64_t S;
    int32_t T, h, W;
    int32_t nq;              // ceil(T / 128)
    float sm_scale_log2;     // scale * log2(e)
};

template <int DQK, int DV>
__global__ void __launch_bounds__(kMmThreads, 1)
    sparse_mla_masked_mha_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                                 const MmParams p) {
    using L = MmLayout<DQK, DV>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = ptx::smem_u32(smem);
    if (sbase & 1023u) {  // uniform across the grid: every CTA leaves before any barrier
        if (threadIdx.x == 0) atomicOr(&g_smla_error, kErrLayout);
        return;
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* sAbort = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
    volatile int* sNact = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 8);
    uint32_t* sBits = reinterpret_cast<uint32_t*>(smem + L::kOffTiles);
    uint16_t* sList = reinterpret_cast<uint16_t*>(smem + L::kOffList);
    auto bar = [&](int i) -> uint32_t { return sbase + L::kOffBar + 8u * static_cast<uint32_t>(i); };
    auto wait = [&](int i, uint32_t parity) -> bool {
        return ptx::mbar_wait(bar(i), parity, sAbort, &g_smla_error, kErrTimeout, kWaitLimitNs);
    };

    // the query tiles of one head next to each other, so the CTAs in flight share a few heads'
    // K and V in L2 (all heads' K/V of a long request exceed it); heaviest tiles first within a
    // head (later queries reach more key tiles)
    const int qt = p.nq - 1 - static_cast<int>(blockIdx.x) % p.nq;
    const int hh = static_cast<int>(blockIdx.x) / p.nq;
    const int t0 = qt * kMmBM;
    const int n_tiles = static_cast<int>((p.S + kMmBN - 1) / kMmBN);

    if (threadIdx.x == 0) {
        *sAbort = 0;
        for (int s = 0; s < L::kStages; ++s) {
            ptx::mbar_init(bar(kMbKFull + s), 1);
            ptx::mbar_init(bar(kMbKEmpty + s), 1);
            ptx::mbar_init(bar(kMbVFull + s), 1);
            ptx::mbar_init(bar(kMbVEmpty + s), 1);
        }
        ptx::mbar_init(bar(kMbSFull), 1);
        ptx::mbar_init(bar(kMbSEmpty), kMmSoftmaxWarps);
        ptx::mbar_init(bar(kMbQFull), 8);  // the quadrants' first two warps copy Q
        ptx::mbar_init(bar(kMbQLoad), 1);
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(kMbPFull + b), kMmSoftmaxWarps);
            ptx::mbar_init(bar(kMbPEmpty + b), 1);
        }
        ptx::mbar_init(bar(kMbPvDone), 1);
        ptx::mbar_init(bar(kMbDrain), 2);  // one commit from each issuing thread
        ptx::fence_mbarrier_init();
    }
    for (int i = threadIdx.x; i < kMmMaxTiles / 32; i += kMmThreads) sBits[i] = 0u;
    if (warp == 1) {
        ptx::tmem_alloc(sbase + L::kOffMisc, L::kTmemCols);
        ptx::tmem_relinquish();
    }
    // launched as a programmatic dependent: the mask may be the previous launch's output
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    __syncthreads();
    if (threadIdx.x == 0) {  // Q's copy runs under the pre-pass
        ptx::prefetch_tmap(&tm_q);
        ptx::mbar_arrive_expect_tx(bar(kMbQLoad), static_cast<uint32_t>(L::kQP * L::kQPanel));
        ptx::tma_load_4d(sbase + L::kOffQ, &tm_q, 0, t0, hh, 0, bar(kMbQLoad));
    }

    // ---- the key tiles any row of this query tile attends to (tile k covers words 2k and 2k + 1).
    // Each warp takes rows, its lanes the row's words (coalesced, independent loads); a nonzero
    // word raises its flag in the first K/V stage (free until the first load) with a plain store,
    // since every writer stores the same value; then each tile ORs its two flags into the bitmap.  (An
    // atomic on the bitmap per nonzero word put every row of the query tile on the same one or
    // two words: 18.7 M shared-memory bank conflicts per launch on the 4096-token chunk.)
    volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(smem + L::kOffKV);
    static_assert(L::kStageBytes >= kMmMaxS / 32 * 4, "word flags fit a K/V stage");
    for (int w = threadIdx.x; w < p.W; w += kMmThreads) sFlag[w] = 0u;
    __syncthreads();
    {
        // each warp ORs its rows' words in registers, all of its rows' loads in flight at once,
        // then raises the flags of the nonzero words
        const int nrows = p.T - t0 < kMmBM ? p.T - t0 : kMmBM;
        constexpr int kWarps = kMmThreads / 32;
        constexpr int kRows = (kMmBM + kWarps - 1) / kWarps;  // rows per warp
        if ((p.W & 3) == 0 && (reinterpret_cast<uintptr_t>(p.mask) & 15u) == 0) {
            const int W4 = p.W >> 2;
            for (int cw = lane; cw < W4; cw += 32) {
                uint4 v[kRows];
#pragma unroll
                for (int i = 0; i < kRows; ++i) {
                    const int r = warp + i * kWarps;
                    v[i] = r < nrows ? __ldg(reinterpret_cast<const uint4*>(p.mask + static_cast<int64_t>(t0 + r) * p.W) + cw)
                                     : make_uint4(0u, 0u, 0u, 0u);
                }
                uint4 acc = v[0];
#pragma unroll
                for (int i = 1; i < kRows; ++i) {
                    acc.x |= v[i].x;
                    acc.y |= v[i].y;
                    acc.z |= v[i].z;
                    acc.w |= v[i].w;
                }
                if (acc.x) sFlag[4 * cw] = 1u;
                if (acc.y) sFlag[4 * cw + 1] = 1u;
                if (acc.z) sFlag[4 * cw + 2] = 1u;
                if (acc.w) sFlag[4 * cw + 3] = 1u;
            }
        } else {
            for (int w = lane; w < p.W; w += 32) {
                uint32_t v[kRows];
#pragma unroll
                for (int i = 0; i < kRows; ++i) {
                    const int r = warp + i * kWarps;
                    v[i] = r < nrows ? __ldg(p.mask + static_cast<int64_t>(t0 + r) * p.W + w) : 0u;
                }
                uint32_t acc = 0u;
#pragma unroll
                for (int i = 0; i < kRows; ++i) acc |= v[i];
                if (acc) sFlag[w] = 1u;
            }
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < n_tiles; k += kMmThreads) {
        const bool any = sFlag[2 * k] != 0u || (2 * k + 1 < p.W && sFlag[2 * k + 1] != 0u);
        if (any) atomicOr(&sBits[k >> 5], 1u << (k & 31));
    }
    __syncthreads();
    // compact list of the active tiles in ascending order: warp 0 scans the bitmap words' counts
    // (one word per lane), then every thread places its tiles
    int* sPre = reinterpret_cast<int*>(smem + L::kOffKV + kMmMaxS / 32 * 4);
    if (warp == 0) {
        const uint32_t bits = lane < (n_tiles + 31) / 32 ? sBits[lane] : 0u;
        const int cnt = __popc(bits);
        int pre = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, pre, o);
            if (lane >= o) pre += v;
        }
        sPre[lane] = pre - cnt;
        if (lane == 31) *sNact = pre;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < n_tiles; k += kMmThreads) {
        const uint32_t word = sBits[k >> 5];
        if ((word >> (k & 31)) & 1u)
            sList[sPre[k >> 5] + __popc(word & ((1u << (k & 31)) - 1u))] = static_cast<uint16_t>(k);
    }
    ptx::fence_proxy_async_smem();  // the flags' and prefix sums' memory is next written by TMA
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kOffMisc);
    const int nact = *sNact;

    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0 && nact > 0) {
            ptx::prefetch_tmap(&tm_k);
            ptx::prefetch_tmap(&tm_v);
            // one copy per tile: the maps' outermost dimension is the 64-wide panel, so a box lands
            // as the panels of the SW128 operand one after another.  K and V of a tile refill
            // separately, V one tile behind K: K(j) waits for S(j - stages), V(j - 1) for
            // PV(j - 1 - stages), the order in which the tensor cores finish them, so no K load
            // waits behind a V slot
            int jk = 0, jv = 0;  // K and V tiles issued
            for (int j = 0; j <= nact; ++j) {
                if (j == 1 && !wait(kMbQFull, 0)) break;  // stages 1 on hold Q until it is in TMEM
                if (j < nact) {
                    const int s = j % L::kStages;
                    if (j >= L::kStages && !wait(kMbKEmpty + s, ((j / L::kStages) - 1) & 1)) break;
                    ptx::mbar_arrive_expect_tx(bar(kMbKFull + s), static_cast<uint32_t>(L::kQP * L::kKPanel));
                    ptx::tma_load_4d(sbase + L::kOffKV + s * L::kStageBytes, &tm_k, 0,
                                     static_cast<int>(sList[j]) * kMmBN, hh, 0, bar(kMbKFull + s));
                    ++jk;
                }
                if (j >= 1) {
                    const int jj = j - 1, s = jj % L::kStages;
                    if (jj >= L::kStages && !wait(kMbVEmpty + s, ((jj / L::kStages) - 1) & 1)) break;
                    ptx::mbar_arrive_expect_tx(bar(kMbVFull + s), static_cast<uint32_t>(L::kVP * L::kKPanel));
                    ptx::tma_load_4d(sbase + L::kOffKV + s * L::kStageBytes + L::kQP * L::kKPanel, &tm_v, 0,
                                     static_cast<int>(sList[jj]) * kMmBN, hh, 0, bar(kMbVFull + s));
                    ++jv;
                }
            }
            // no copy may still be landing when the CTA leaves
            for (int i = jk - (jk < L::kStages ? jk : L::kStages); i < jk; ++i)
                ptx::mbar_wait(bar(kMbKFull + i % L::kStages), (i / L::kStages) & 1, nullptr, &g_smla_error, 0u,
                               kDrainLimitNs);
            for (int i = jv - (jv < L::kStages ? jv : L::kStages); i < jv; ++i)
                ptx::mbar_wait(bar(kMbVFull + i % L::kStages), (i / L::kStages) & 1, nullptr, &g_smla_error, 0u,
                               kDrainLimitNs);
        }
        if (lane == 0) ptx::mbar_wait(bar(kMbQLoad), 0, nullptr, &g_smla_error, 0u, kDrainLimitNs);
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ S issuer (TMEM owner)
        // S(j) = Q K_j^T with Q from TMEM (16 dims: 8 columns) and K from the ring; S is one
        // buffer, rewritten once the softmax warps hold S(j - 1) in registers
        if (lane == 0 && nact > 0) {
            constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kMmBM, kMmBN, 0, 0);
            const uint64_t dk = ptx::smem_desc_sw128(sbase + L::kOffKV, 16, 1024);
            bool ok = wait(kMbQFull, 0);
            for (int j = 0; ok && j < nact; ++j) {
                const int s = j % L::kStages;
                if (!(ok = wait(kMbKFull + s, (j / L::kStages) & 1))) break;
                if (j >= 1 && !(ok = wait(kMbSEmpty, (j - 1) & 1))) break;
                ptx::tc_fence_after();
                const uint64_t k0 = dk + static_cast<uint64_t>((s * L::kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk)
                    ptx::mma_bf16_ts(tmem + L::kColS, tmem + L::kColQ + 8 * kk,
                                     k0 + (((kk >> 2) * L::kKPanel + (kk & 3) * 32) >> 4), kIdescS,
                                     kk != 0 ? 1u : 0u);
                ptx::mma_commit(bar(kMbSFull));
                ptx::mma_commit(bar(kMbKEmpty + s));
            }
        }
        if (lane == 0) {  // this thread's MMAs are done before TMEM is freed
            ptx::mma_commit(bar(kMbDrain));
            ptx::mbar_wait(bar(kMbDrain), 0, nullptr, &g_smla_error, 0u, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == kMmThreads / 32 - 1) {
        // ================================================================ PV issuer
        // O += P(j) V_j with P from TMEM buffer j % 2 (16 keys: 8 columns) and V MN-major from the
        // ring.  A thread of its own, so that a PV waiting for its P or V never holds back an S
        // (an issuing thread stalls while the tensor cores run what it issued).
        if (lane == 0 && nact > 0) {
            constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kMmBM, DV, 0, 1);
            const uint64_t dv = ptx::smem_desc_sw128(sbase + L::kOffKV + L::kQP * L::kKPanel, L::kKPanel, 1024);
            for (int j = 0; j < nact; ++j) {
                const int s = j % L::kStages;
                if (!wait(kMbPFull + (j & 1), (j >> 1) & 1)) break;
                if (!wait(kMbVFull + s, (j / L::kStages) & 1)) break;
                ptx::tc_fence_after();
                const uint64_t v0 = dv + static_cast<uint64_t>((s * L::kStageBytes) >> 4);
                const uint32_t p0 = tmem + static_cast<uint32_t>(L::kColP + (j & 1) * (kMmBN / 2));
#pragma unroll
                for (int k = 0; k < kMmBN / 16; ++k)
                    ptx::mma_bf16_ts(tmem + L::kColO, p0 + 8 * k, v0 + ((k * 2048) >> 4), kIdescPV,
                                     (j > 0 || k > 0) ? 1u : 0u);
                ptx::mma_commit(bar(kMbVEmpty + s));
                ptx::mma_commit(bar(kMbPEmpty + (j & 1)));
                ptx::mma_commit(bar(kMbPvDone));
            }
        }
        if (lane == 0) {
            ptx::mma_commit(bar(kMbDrain));
            ptx::mbar_wait(bar(kMbDrain), 0, nullptr, &g_smla_error, 0u, kDrainLimitNs);
        }
        __syncwarp();
    } else {
        // ================================================================ softmax / epilogue
        // kMmParts warps per TMEM lane quadrant: `part` takes keys [kKeys * part, kKeys * part +
        // kKeys) of each tile and O columns [kOCols * part, kOCols * part + kOCols).  The
        // quadrant's warps share one named barrier per tile, a reduction that says whether any of
        // their rows' maxima grew by more than 2^8 (or one of them gave up on a wait); only then do
        // they swap their tile maxima through shared memory.  Every thread of the group takes the
        // same barriers in the same order, so a warp that gives up keeps going to the next
        // reduction, and the whole group leaves the loop there.
        constexpr int kKeys = kMmBN / kMmParts;   // keys of a tile per warp
        constexpr int kOCols = DV / kMmParts;     // O columns per warp
        constexpr uint32_t kGroup = 32u * kMmParts;
        const int quad = warp & 3;
        const int part = (warp - 2) >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const int r = quad * 32 + lane;          // query row of this thread (its TMEM lane)
        const int64_t t = t0 + r;
        const bool live = t < p.T;
        const uint32_t* mrow = p.mask + (live ? t : 0) * p.W;
        const float c = p.sm_scale_log2;
        const uint32_t grp_bar = 1u + static_cast<uint32_t>(quad);
        volatile float* sX = reinterpret_cast<volatile float*>(smem + L::kOffX);  // [kMmParts][128]
        const int ocol0 = part * kOCols;
        float m = -CUDART_INF_F, l = 0.f;
        bool failed = false;
        auto warp_wait = [&](int i, uint32_t parity) -> bool {
            bool okw = true;
            if (lane == 0) okw = wait(i, parity);
            okw = __shfl_sync(0xffffffffu, okw, 0);
            __syncwarp();
            return okw;
        };
        // this warp's kKeys mask bits of tile j (word 2k + kKeys * part / 32 of tile k)
        auto mask_word = [&](int j) -> uint32_t {
            uint32_t w = 0u;
            if (live && j < nact) {
                const int wi = 2 * static_cast<int>(sList[j]) + (kKeys * part) / 32;
                if (wi < p.W) w = __ldg(mrow + wi) >> ((kKeys * part) % 32);
            }
            return w;
        };
        // the group's values of row r meet in shared memory: each posts its own, all read all
        auto group_max = [&](float mine) -> float {
            sX[part * kMmBM + r] = mine;
            ptx::named_bar_sync(grp_bar, kGroup);
            float v = sX[r];
#pragma unroll
            for (int q = 1; q < kMmParts; ++q) {
                const float o = sX[q * kMmBM + r];
                v = (v != v || o != o) ? CUDART_NAN_F : fmaxf(v, o);
            }
            return v;
        };
        if (nact > 0 && part < 2 && !(failed = !warp_wait(kMbQLoad, 0))) {
            // Q (its TMA copy issued before the pre-pass; rows past the last token are zero) into
            // TMEM, the A operand of every S, by the quadrant's first two warps: row r in lane r,
            // dims 2c and 2c + 1 in column c (warp `part`: dims DQK/2 * part .. DQK/2 * part +
            // DQK/2 - 1).  The row's 16-byte chunk q of a 64-dim SW128 panel sits at
            // ((q ^ (r & 7)) << 4).
#pragma unroll
            for (int cc = 0; cc < DQK / 64; ++cc) {
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int d0 = part * (DQK / 2) + 8 * (4 * cc + e);  // first dim of the chunk
                    const uint32_t q = static_cast<uint32_t>((d0 & 63) >> 3);
                    const uint4 v = ptx::ld_shared_v4(sbase + L::kOffQ + (d0 >> 6) * L::kQPanel + r * 128 +
                                                      ((q ^ static_cast<uint32_t>(r & 7)) << 4));
                    w[4 * e] = v.x;
                    w[4 * e + 1] = v.y;
                    w[4 * e + 2] = v.z;
                    w[4 * e + 3] = v.w;
                }
                SMLA_TMEM_ST16(tmem + lane_base + L::kColQ + part * (DQK / 4) + 16 * cc, w);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kMbQFull));
        }
        uint32_t mw = mask_word(0);
        for (int j = 0; j < nact; ++j) {
            const uint32_t cur = mw;
            mw = mask_word(j + 1);
            if (!failed && !warp_wait(kMbSFull, j & 1)) failed = true;
            uint32_t sv[kKeys];
            float mx = -CUDART_INF_F;
            if (!failed) {
                ptx::tc_fence_after();
#pragma unroll
                for (int q = 0; q < kKeys / 16; ++q) SMLA_TMEM_LD16(tmem + lane_base + L::kColS + kKeys * part + 16 * q, sv + 16 * q);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(kMbSEmpty));
                // scaled logits of the set positions (log2 units) and their max (eight partial
                // maxima: no long dependency chain)
                float mxa[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mxa[i] = -CUDART_INF_F;
#pragma unroll
                for (int i = 0; i < kKeys / 2; ++i) {
                    const float2 y = ptx::mul2(make_float2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                                               make_float2(c, c));
                    const float x0 = (cur & (1u << (2 * i))) ? y.x : -CUDART_INF_F;
                    const float x1 = (cur & (1u << (2 * i + 1))) ? y.y : -CUDART_INF_F;
                    sv[2 * i] = __float_as_uint(x0);
                    sv[2 * i + 1] = __float_as_uint(x1);
                    mxa[(2 * i) & 7] = fmaxf(mxa[(2 * i) & 7], x0);
                    mxa[(2 * i + 1) & 7] = fmaxf(mxa[(2 * i + 1) & 7], x1);
                }
                mx = fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])),
                           fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])));
            }
            bool pv_waited = false;
            if (ptx::named_bar_red_or(grp_bar, kGroup, failed || mx > m + kRescaleLog2)) {
                // the row's max over the group's keys (NaN: a warp of the group gave up)
                const float v = group_max(failed ? CUDART_NAN_F : mx);
                if (v != v) {
                    failed = true;
                    break;
                }
                mx = v;
                const bool grow = mx > m + kRescaleLog2;
                if (__any_sync(0xffffffffu, grow)) {
                    // the running max of some row grew by more than 2^8: that row's O columns and
                    // sum are rescaled (the other rows of the warp multiply by 1); O must be
                    // complete
                    float alpha = 1.f;
                    if (grow) {
                        const float mn = fmaxf(m, mx);
                        alpha = (m == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(m - mn);
                        m = mn;
                        l *= alpha;
                    }
                    if (j > 0) {
                        if (!warp_wait(kMbPvDone, (j - 1) & 1)) {
                            failed = true;
                            continue;  // the next reduction takes the whole group out
                        }
                        pv_waited = true;
                        ptx::tc_fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < kOCols / 16; ++cc) {
                            uint32_t o[16];
                            SMLA_TMEM_LD16(tmem + lane_base + L::kColO + ocol0 + cc * 16, o);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            SMLA_TMEM_ST16(tmem + lane_base + L::kColO + ocol0 + cc * 16, o);
                        }
                        ptx::tmem_wait_st();
                    }
                }
            }
            // P = 2^(x - m) as bf16, row sums in fp32 (a masked position holds -inf and gives 0;
            // m is -inf only while every position seen so far is masked, and then any finite
            // offset serves); P buffer j % 2 is rewritten only after PV(j - 2) has read it
            const float nm = m == -CUDART_INF_F ? 0.f : -m;
            uint32_t pk[kKeys / 2];
            float2 la[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) la[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kKeys / 2; ++i) {
                const float2 d = ptx::add2(make_float2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                                           make_float2(nm, nm));
                const float2 pp = make_float2(ptx::ex2_approx(d.x), ptx::ex2_approx(d.y));
                la[i & 3] = ptx::add2(la[i & 3], pp);
                pk[i] = pack_bf16x2(pp.x, pp.y);
            }
            l += ((la[0].x + la[0].y) + (la[1].x + la[1].y)) + ((la[2].x + la[2].y) + (la[3].x + la[3].y));
            if (j >= 2 && !pv_waited) {
                if (!warp_wait(kMbPEmpty + (j & 1), ((j >> 1) - 1) & 1)) {
                    failed = true;
                    continue;
                }
            }
            // P(j) into its TMEM buffer, the operand A of PV(j): row r in lane r, keys 2c and
            // 2c + 1 in column c (this warp: keys kKeys * part .. kKeys * part + kKeys - 1)
            ptx::tc_fence_after();
            if constexpr (kKeys == 32) {
                SMLA_TMEM_ST16(tmem + lane_base + L::kColP + (j & 1) * (kMmBN / 2) + (kKeys / 2) * part, pk);
            } else {
                SMLA_TMEM_ST8(tmem + lane_base + L::kColP + (j & 1) * (kMmBN / 2) + (kKeys / 2) * part, pk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kMbPFull + (j & 1)));
        }
        // ---- epilogue: O / l as bf16 and the natural-log LSE.  The group's row sums meet in
        // shared memory (two barriers, taken by every warp of the group whatever happened in the
        // loop).
        bool have_o = nact > 0 && !failed;
        if (have_o) {
            have_o = warp_wait(kMbPvDone, (nact - 1) & 1);
            if (have_o) ptx::tc_fence_after();
        }
        ptx::named_bar_sync(grp_bar, kGroup);  // every read of sX in the loop is done
        sX[part * kMmBM + r] = l;
        ptx::named_bar_sync(grp_bar, kGroup);
        float lt = 0.f;
#pragma unroll
        for (int q = 0; q < kMmParts; ++q) lt += sX[q * kMmBM + r];
        // O goes out through shared memory (the K/V ring, idle once the last PV is done) as
        // DV/64 SW128 panels of 128 rows, then one TMA store: the rows' own global addresses are
        // h * DV * 2 bytes apart, so direct stores would touch a line per lane
        if (!failed) {
            const float inv = (have_o && lt > 0.f) ? 1.0f / lt : 0.f;
            // this warp's kOCols columns, up to four 16-column TMEM loads per wait
            constexpr int kChunks = kOCols / 16;
            constexpr int kBatch = kChunks < 4 ? kChunks : 4;
#pragma unroll 1
            for (int cg = 0; cg < kChunks / kBatch; ++cg) {
                uint32_t o[kBatch][16];
                if (have_o) {
#pragma unroll
                    for (int g = 0; g < kBatch; ++g)
                        SMLA_TMEM_LD16(tmem + lane_base + L::kColO + ocol0 + (kBatch * cg + g) * 16, o[g]);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int g = 0; g < kBatch; ++g)
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[g][e] = 0u;
                }
#pragma unroll
                for (int g = 0; g < kBatch; ++g) {
                    uint4 v0, v1;
                    v0.x = pack_bf16x2(__uint_as_float(o[g][0]) * inv, __uint_as_float(o[g][1]) * inv);
                    v0.y = pack_bf16x2(__uint_as_float(o[g][2]) * inv, __uint_as_float(o[g][3]) * inv);
                    v0.z = pack_bf16x2(__uint_as_float(o[g][4]) * inv, __uint_as_float(o[g][5]) * inv);
                    v0.w = pack_bf16x2(__uint_as_float(o[g][6]) * inv, __uint_as_float(o[g][7]) * inv);
                    v1.x = pack_bf16x2(__uint_as_float(o[g][8]) * inv, __uint_as_float(o[g][9]) * inv);
                    v1.y = pack_bf16x2(__uint_as_float(o[g][10]) * inv, __uint_as_float(o[g][11]) * inv);
                    v1.z = pack_bf16x2(__uint_as_float(o[g][12]) * inv, __uint_as_float(o[g][13]) * inv);
                    v1.w = pack_bf16x2(__uint_as_float(o[g][14]) * inv, __uint_as_float(o[g][15]) * inv);
                    const int d0 = ocol0 + 16 * (kBatch * cg + g);  // first dim of chunk pair (2 x 8 dims)
                    const uint32_t prow = sbase + L::kOffKV + (d0 >> 6) * L::kQPanel + r * 128;
                    const uint32_t q0 = static_cast<uint32_t>((d0 & 63) >> 3);
                    ptx::st_shared_v4(prow + ((q0 ^ static_cast<uint32_t>(r & 7)) << 4), v0);
                    ptx::st_shared_v4(prow + (((q0 + 1) ^ static_cast<uint32_t>(r & 7)) << 4), v1);
                }
            }
            ptx::fence_proxy_async_smem();
            if (live && part == 0)
                p.lse[t * p.h + hh] = (have_o && lt > 0.f) ? (m + log2f(lt)) * 0.69314718055994531f : -CUDART_INF_F;
        }
        if (failed) *sAbort = 1;
        // all the softmax warps' rows are in shared memory (none gave up): one thread stores the
        // tile; rows past the last token fall outside the map and are not written
        if (!ptx::named_bar_red_or(5u, 32u * kMmSoftmaxWarps, failed) && warp == 2 && lane == 0) {
            ptx::tma_store_4d(&tm_o, sbase + L::kOffKV, 0, t0, hh, 0);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read_0();  // shared memory may not be released before it is read
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace smla
