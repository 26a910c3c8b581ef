// Top-k selection of the index lists from per-position scores: the step before the sparse
// attention.  The indexer scores every position of a token's causal history and keeps the top
// k as a fixed-width int32 list whose order does not matter (vLLM PR #54951, Summary and
// Additional checks).  The pages do not give the indexer's scoring, so the scores are the
// input here.  Row t keeps the topk positions with the largest scores among [0, len[t]), ties
// to the lower position, written in ascending position order, mapped through a block table of
// 64-slot blocks to cache slots (or left as positions), -1 padded when the history is shorter.
//
// One CTA per row.  Radix select on an order-preserving 32-bit key, one byte per pass: a
// shared-memory histogram of the candidates that match the prefix found so far, then one warp
// scans the 256 bins from the top for the bin where the count reaches the number still to take.
// Each pass scans the row, four scores per 16-byte load when the row is 16-byte aligned.
// After four passes the threshold key is exact; a last scan in position order writes every
// key above it and the first ties at it, with a block-wide scan giving each selected position
// its output slot.  The first scan reads the row from HBM; the later ones find it in L1 or L2.
// (Copying the candidates left after the first byte into shared memory for the last two
// passes, through one shared counter, measured slower: 2.73 vs 2.39 ms on the prefill rows.)
// 256 threads a CTA: at 48 registers five rows share an SM, so one row's barrier-separated
// phases overlap another's scans (1.74 ms on the prefill rows, 2.25 ms at 512 threads).
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkPerThread = 4;                          // consecutive scores per thread
constexpr int kTopkChunk = kTopkThreads * kTopkPerThread;  // scores per compaction step

struct TopkParams {
    const float* scores;         // [T, S]
    const int32_t* len;          // [T]: row t's causal history [0, len[t])
    const int32_t* block_table;  // [ceil(S / 64)] or null
    int32_t* out;                // [T, topk]
    int64_t S;
    int32_t T, topk;
};

// Order-preserving key: a larger score gives a larger unsigned key.
__device__ __forceinline__ uint32_t score_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sums of two per-thread counts, and their block totals.
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb, uint32_t& ta,
                                            uint32_t& tb, uint32_t* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t xa = __shfl_up_sync(0xffffffffu, ia, o);
        const uint32_t xb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += xa;
            ib += xb;
        }
    }
    if (lane == 31) {
        s_warp[warp] = ia;
        s_warp[kTopkWarps + warp] = ib;
    }
    __syncthreads();
    uint32_t wa = 0, wb = 0, sa = 0, sb = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
        const uint32_t va = s_warp[w], vb = s_warp[kTopkWarps + w];
        if (w < warp) {
            wa += va;
            wb += vb;
        }
        sa += va;
        sb += vb;
    }
    ea = wa + ia - a;
    eb = wb + ib - b;
    ta = sa;
    tb = sb;
    __syncthreads();  // s_warp is reused by the next call
}

__global__ void __launch_bounds__(kTopkThreads) sparse_mla_topk_kernel(const TopkParams p) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_warp[2 * kTopkWarps];
    __shared__ uint32_t s_sel[2];
    // launched as a programmatic dependent: the scores may be the previous launch's output
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int64_t t = blockIdx.x;
    const float* row = p.scores + t * p.S;
    int32_t* orow = p.out + t * p.topk;
    int64_t n64 = p.len[t];
    n64 = n64 < 0 ? 0 : (n64 > p.S ? p.S : n64);  // a length outside [0, S] is clamped
    const int n = static_cast<int>(n64);
    const int k = n < p.topk ? n : p.topk;
    const bool take_all = k == n;  // the history is no longer than topk: every position

    // ---- radix select of the threshold key: the k-th largest, one byte per pass
    uint32_t prefix = 0, pmask = 0, krem = static_cast<uint32_t>(k);
    if (threadIdx.x == 0) s_sel[0] = s_sel[1] = 0u;  // read only after a barrier
    // 16-byte loads when the row starts on a 16-byte boundary (S a multiple of 4)
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    const int n4 = vec ? n / 4 : 0;
    if (!take_all) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
            __syncthreads();
            auto count = [&](float x) {
                const uint32_t key = score_key(x);
                if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            };
            const float4* row4 = reinterpret_cast<const float4*>(row);
            for (int i = threadIdx.x; i < n4; i += kTopkThreads) {
                const float4 v = __ldg(row4 + i);
                count(v.x);
                count(v.y);
                count(v.z);
                count(v.w);
            }
            for (int i = 4 * n4 + threadIdx.x; i < n; i += kTopkThreads) count(__ldg(row + i));
            __syncthreads();
            if (threadIdx.x < 32) {
                // lane l holds bins 255 - 8l - j (j = 0..7), highest first
                const int lane = threadIdx.x;
                uint32_t c[8], tot = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = hist[255 - 8 * lane - j];
                    tot += c[j];
                }
                uint32_t incl = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += x;
                }
                const uint32_t above = incl - tot;  // candidates in higher bins
                const bool mine = above < krem && krem <= above + tot;
                const unsigned m = __ballot_sync(0xffffffffu, mine);
                if (lane == __ffs(m) - 1) {
                    uint32_t a = above;
                    int bin = -1;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (bin < 0) {
                            if (a + c[j] >= krem)
                                bin = 255 - 8 * lane - j;
                            else
                                a += c[j];
                        }
                    }
                    s_sel[0] = static_cast<uint32_t>(bin);
                    s_sel[1] = a;
                }
            }
            __syncthreads();
            krem -= s_sel[1];
            prefix |= s_sel[0] << shift;
            pmask |= 0xFFu << shift;
            __syncthreads();  // hist and s_sel are rewritten by the next pass
        }
    }

    // ---- every key above the threshold and the first krem ties at it, in position order
    uint32_t base_gt = 0, base_eq = 0;
    for (int c0 = 0; c0 < n; c0 += kTopkChunk) {
        const int i0 = c0 + static_cast<int>(threadIdx.x) * kTopkPerThread;
        uint32_t flags = 0, ngt = 0, neq = 0;  // 2 bits per score: above, tie
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            const int i = i0 + e;
            if (i < n) {
                const uint32_t key = take_all ? 0u : score_key(__ldg(row + i));
                if (take_all || key > prefix) {
                    flags |= 1u << (2 * e);
                    ++ngt;
                } else if (key == prefix) {
                    flags |= 2u << (2 * e);
                    ++neq;
                }
            }
        }
        uint32_t egt, eeq, tgt, teq;
        block_scan2(ngt, neq, egt, eeq, tgt, teq, s_warp);
        uint32_t rgt = base_gt + egt, req = base_eq + eeq;
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            const int i = i0 + e;
            const uint32_t f = (flags >> (2 * e)) & 3u;
            int slot_out = -1;
            if (f == 1u) {
                slot_out = static_cast<int>(rgt + (req < krem ? req : krem));
                ++rgt;
            } else if (f == 2u) {
                if (req < krem) slot_out = static_cast<int>(rgt + req);
                ++req;
            }
            if (slot_out >= 0 && slot_out < k)  // always below k; the check keeps every store in the row
                orow[slot_out] = p.block_table ? __ldg(p.block_table + (i >> 6)) * 64 + (i & 63) : i;
        }
        base_gt += tgt;
        base_eq += teq;
    }
    for (int i = k + static_cast<int>(threadIdx.x); i < p.topk; i += kTopkThreads) orow[i] = -1;
}

}  // namespace smla
