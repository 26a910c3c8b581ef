// Top-k selection of the index lists from per-position scores: the step before the sparse
// attention.  The indexer scores every position of a token's causal history and keeps the top
// k as a fixed-width int32 list whose order does not matter (vLLM PR #54951, Summary and
// Additional checks).  The pages do not give the indexer's scoring, so the scores are the
// input here.  Row t keeps the topk positions with the largest scores among [0, len[t]), ties
// to the lower position, written in ascending position order, mapped through a block table of
// 64-slot blocks to cache slots (or left as positions), -1 padded when the history is shorter.
//
// One CTA per row.  Radix select on an order-preserving 32-bit key: a 4096-bin shared-memory
// histogram of the keys' top 12 bits over the row, a block-wide scan of the bins from the top
// for the bin where the count reaches k, then one more scan of the row that copies the keys of
// that bin into shared memory, each warp into its own region through its own counter (a few
// hundred keys on score distributions like a normal one; one counter for the CTA serialised
// them).  The remaining 20 bits are found in passes of 8, 8 and 4 bits over those candidates
// alone; when a warp's share overflows its region (many equal scores), those passes scan the
// row instead.
// The threshold key is then exact; a last scan in position order writes every key above it and
// the first ties at it, with a block-wide scan giving each selected position its output slot.
// Each scan of the row takes four scores per 16-byte load when the row is 16-byte aligned; the
// first reads it from HBM, the later ones find it in L1 or L2.  So three scans of the row
// instead of five (one histogram per byte).  256 threads a CTA: several rows share an SM and
// one row's barrier-separated phases overlap another's scans.
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkPerThread = 16;                         // consecutive scores per thread
constexpr int kTopkChunk = kTopkThreads * kTopkPerThread;  // scores per compaction step
constexpr int kTopkBins0 = 4096;                           // first pass: the top 12 key bits
constexpr int kTopkCand = 2048;                            // candidate keys held in shared memory
constexpr int kTopkCandW = kTopkCand / kTopkWarps;         // per warp

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

// The bin of hist[0, nb) (nb = 16, 256 or 4096) where the count of keys, taken from the top bin
// down, reaches krem (1 <= krem <= the total): thread i covers nb / 256 bins (one when nb <=
// 256) from the top, a block-wide scan of the threads' totals finds the one thread whose bins
// hold the krem-th key, and that thread writes the bin and the count above it to s_sel[0..1].
// Every thread reads them after the closing barrier.
__device__ __forceinline__ void topk_find_bin(const uint32_t* hist, int nb, uint32_t krem, uint32_t* s_warp,
                                              uint32_t* s_sel) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nb > kTopkThreads ? nb / kTopkThreads : 1;
    const int top = nb - 1 - per * tid;  // this thread's highest bin
    uint32_t tot = 0;
    if (top >= 0)
        for (int j = 0; j < per; ++j) tot += hist[top - j];
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t above = incl - tot;
    for (int w = 0; w < warp; ++w) above += s_warp[w];
    if (above < krem && krem <= above + tot) {
        uint32_t a = above;
        for (int j = 0; j < per; ++j) {
            const uint32_t c = hist[top - j];
            if (a + c >= krem) {
                s_sel[0] = static_cast<uint32_t>(top - j);
                s_sel[1] = a;
                break;
            }
            a += c;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads, 5) sparse_mla_topk_kernel(const TopkParams p) {
    __shared__ uint32_t hist[kTopkBins0];
    __shared__ uint32_t cand[kTopkCand];
    __shared__ uint32_t s_warp[2 * kTopkWarps];
    __shared__ uint32_t s_sel[2];
    __shared__ uint32_t s_cnt[kTopkWarps];  // candidates per warp (each warp fills its own region)
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

    // ---- radix select of the threshold key: the k-th largest
    uint32_t prefix = 0, pmask = 0, krem = static_cast<uint32_t>(k);
    // 16-byte loads when the row starts on a 16-byte boundary (S a multiple of 4)
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    const int n4 = vec ? n / 4 : 0;
    auto scan_row = [&](auto&& visit) {
        const float4* row4 = reinterpret_cast<const float4*>(row);
        for (int i = threadIdx.x; i < n4; i += kTopkThreads) {
            const float4 v = __ldg(row4 + i);
            visit(score_key(v.x));
            visit(score_key(v.y));
            visit(score_key(v.z));
            visit(score_key(v.w));
        }
        for (int i = 4 * n4 + threadIdx.x; i < n; i += kTopkThreads) visit(score_key(__ldg(row + i)));
    };
    if (!take_all) {
        // pass 1: the top 12 bits of every key
        for (int i = threadIdx.x; i < kTopkBins0; i += kTopkThreads) hist[i] = 0;
        if (threadIdx.x < kTopkWarps) s_cnt[threadIdx.x] = 0;
        __syncthreads();
        scan_row([&](uint32_t key) { atomicAdd(&hist[key >> 20], 1u); });
        __syncthreads();
        topk_find_bin(hist, kTopkBins0, krem, s_warp, s_sel);
        krem -= s_sel[1];
        prefix = s_sel[0] << 20;
        pmask = 0xFFF00000u;
        // pass 2: the keys of that bin into shared memory, each warp into its own region of the
        // buffer through its own counter (one counter for the CTA serialised a few hundred
        // atomics); the counts go on past the regions
        {
            const int w = threadIdx.x >> 5;
            scan_row([&](uint32_t key) {
                if ((key & pmask) == prefix) {
                    const uint32_t c = atomicAdd(&s_cnt[w], 1u);
                    if (c < kTopkCandW) cand[w * kTopkCandW + c] = key;
                }
            });
        }
        __syncthreads();
        bool in_smem = true;
#pragma unroll
        for (int w = 0; w < kTopkWarps; ++w) in_smem = in_smem && s_cnt[w] <= static_cast<uint32_t>(kTopkCandW);
        // passes 3-5: key bits 19-12, 11-4 and 3-0, over the candidates (over the row when
        // they did not fit)
#pragma unroll 1
        for (int step = 0; step < 3; ++step) {
            const int shift = step == 0 ? 12 : (step == 1 ? 4 : 0);
            const int nb = step == 2 ? 16 : 256;
            for (int i = threadIdx.x; i < nb; i += kTopkThreads) hist[i] = 0;
            __syncthreads();
            auto count = [&](uint32_t key) {
                if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
            };
            if (in_smem) {
                for (int c = threadIdx.x; c < kTopkCand; c += kTopkThreads)
                    if (static_cast<uint32_t>(c % kTopkCandW) < s_cnt[c / kTopkCandW]) count(cand[c]);
            } else {
                scan_row(count);
            }
            __syncthreads();
            topk_find_bin(hist, nb, krem, s_warp, s_sel);
            krem -= s_sel[1];
            prefix |= s_sel[0] << shift;
            pmask |= static_cast<uint32_t>(nb - 1) << shift;
            __syncthreads();  // hist and s_sel are rewritten by the next pass
        }
    }

    // ---- every key above the threshold and the first krem ties at it, in position order
    uint32_t base_gt = 0, base_eq = 0;
    for (int c0 = 0; c0 < n; c0 += kTopkChunk) {
        const int i0 = c0 + static_cast<int>(threadIdx.x) * kTopkPerThread;
        float xs[kTopkPerThread];
        if (!take_all) {
            if (vec && i0 + kTopkPerThread <= n) {  // i0 is a multiple of 16: aligned
#pragma unroll
                for (int e = 0; e < kTopkPerThread / 4; ++e) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(row + i0) + e);
                    xs[4 * e] = v.x;
                    xs[4 * e + 1] = v.y;
                    xs[4 * e + 2] = v.z;
                    xs[4 * e + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < kTopkPerThread; ++e) xs[e] = i0 + e < n ? __ldg(row + i0 + e) : 0.f;
            }
        }
        // bit e of gt / eq: score i0 + e is above the threshold / equal to it
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            if (i0 + e < n) {
                const uint32_t key = take_all ? 0u : score_key(xs[e]);
                gt |= static_cast<uint32_t>(take_all || key > prefix) << e;
                eq |= static_cast<uint32_t>(!take_all && key == prefix) << e;
            }
        }
        uint32_t egt, eeq, tgt, teq;
        block_scan2(__popc(gt), __popc(eq), egt, eeq, tgt, teq, s_warp);
        uint32_t rgt = base_gt + egt, req = base_eq + eeq;
        // only the marked scores, in position order
        for (uint32_t m = gt | eq; m != 0u; m &= m - 1u) {
            const int e = __ffs(m) - 1;
            const int i = i0 + e;
            int slot_out = -1;
            if ((gt >> e) & 1u) {
                slot_out = static_cast<int>(rgt + (req < krem ? req : krem));
                ++rgt;
            } else {
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
