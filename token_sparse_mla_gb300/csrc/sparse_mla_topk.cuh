// Top-k selection of the index lists from per-position scores: the step before the sparse
// attention.  The indexer scores every position of a token's causal history and keeps the top
// k as a fixed-width int32 list whose order does not matter (vLLM PR #54951, Summary and
// Additional checks).  The pages do not give the indexer's scoring, so the scores are the
// input here.  Row t keeps the topk positions with the largest scores among [0, len[t]), ties
// to the lower position (-0 and +0 are equal scores), written in ascending position order,
// mapped through a block table of 64-slot blocks to cache slots (or left as positions), -1
// padded when the history is shorter.
//
// One CTA per row, radix select on an order-preserving 32-bit key.  Pass 1 reads the row from
// HBM (four 16-byte loads a thread per 4096 scores) into a 4096-bin shared-memory histogram of
// the keys' top 12 bits; a block-wide scan of the bins from the top finds the bin B where the
// count reaches k.  Every key in a bin above B is selected, so when those keys and B's own
// number at most 4096 (a few hundred more than k on score distributions like a normal one),
// pass 2 reads the row once more (mostly from L2), 32 consecutive positions per warp load: one
// warp ballot of "score >= the lowest score of bin B" per load is one word of a candidate
// bitmap in position order.  A block-wide scan of the words' popcounts then places every
// candidate's position in shared memory, in order.  The remaining 20 key bits are found in two
// 10-bit passes over the candidates in B (their scores gathered once into registers, 16 a
// thread), and the lists come out of ballots over the candidates, 32 consecutive ones per warp
// row: two reads of the row in all.  When bin B holds too many keys (many equal scores), pass 2
// keeps B's keys alone (each warp in its own region while they fit), 8-, 8- and 4-bit passes
// find the rest of the threshold, over those keys or over the row, and a last scan of the row
// writes the lists.
#pragma once

#include <type_traits>

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkGroups = 4;                               // 16-byte loads a thread per scan step
constexpr int kTopkChunk = kTopkThreads * 4 * kTopkGroups;   // scores per scan step
constexpr int kTopkBins0 = 4096;                             // pass 1: the top 12 key bits
constexpr int kTopkBins1 = 1024;                             // candidate passes: 10 bits each
constexpr int kTopkPerThread = 16;                           // candidates (or row scores) a thread
constexpr int kTopkCand = kTopkThreads * kTopkPerThread;     // candidate positions held
constexpr int kTopkBinKeys = 2048;                           // threshold-bin keys held otherwise
constexpr int kTopkBinKeysW = kTopkBinKeys / kTopkWarps;     // per warp
constexpr int kTopkWin = kTopkBins1 * 32;                    // positions a candidate bitmap covers

struct TopkParams {
    const float* scores;         // [T, S]
    const int32_t* len;          // [T]: row t's causal history [0, len[t])
    const int32_t* block_table;  // [ceil(S / 64)] or null
    int32_t* out;                // [T, topk]
    int64_t S;
    int32_t T, topk;
};

// Order-preserving key: a larger score gives a larger unsigned key, and -0 the key of +0.
__device__ __forceinline__ uint32_t score_key(float x) {
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.f));  // -0 + 0 = +0; no other value moves
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The lowest score whose key's top 12 bits are b or more: for every score x that is not NaN,
// x >= bin_floor(b) exactly when score_key(x) >> 20 >= b.  Bins 0-7 hold -inf and NaN keys only,
// and their floor keys are NaN patterns, so those give -inf.
__device__ __forceinline__ float bin_floor(uint32_t b) {
    if (b <= 7u) return -INFINITY;
    const uint32_t key = b << 20;
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
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
    uint32_t tot_a[kTopkWarps], tot_b[kTopkWarps];  // four 16-byte reads, one wavefront each
#pragma unroll
    for (int q = 0; q < kTopkWarps / 4; ++q) {
        const uint4 x = reinterpret_cast<const uint4*>(s_warp)[q];
        const uint4 y = reinterpret_cast<const uint4*>(s_warp + kTopkWarps)[q];
        tot_a[4 * q] = x.x, tot_a[4 * q + 1] = x.y, tot_a[4 * q + 2] = x.z, tot_a[4 * q + 3] = x.w;
        tot_b[4 * q] = y.x, tot_b[4 * q + 1] = y.y, tot_b[4 * q + 2] = y.z, tot_b[4 * q + 3] = y.w;
    }
    uint32_t wa = 0, wb = 0, sa = 0, sb = 0;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
        const uint32_t va = tot_a[w], vb = tot_b[w];
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

// The bin of hist[0, nb) (nb = 16, 256, 1024 or 4096) where the count of keys, taken from the
// top bin down, reaches krem (1 <= krem <= the total): thread i covers nb / 256 bins (one when
// nb <= 256) from the top, a block-wide scan of the threads' totals finds the one thread whose
// bins hold the krem-th key, and that thread writes the bin, the count above it and the bin's
// own count to s_sel[0..2].  Every thread reads them after the closing barrier.  The threads of
// a warp sum their bins in rotated orders, so that each read of the warp hits 32 banks.
__device__ __forceinline__ void topk_find_bin(const uint32_t* hist, int nb, uint32_t krem, uint32_t* s_warp,
                                              uint32_t* s_sel) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nb > kTopkThreads ? nb / kTopkThreads : 1;
    const int top = nb - 1 - per * tid;  // this thread's highest bin
    const int rot = (lane * per) >> 5;   // per <= 16: lanes with equal per * lane mod 32 differ here
    uint32_t tot = 0;
    if (top >= 0)
        for (int j = 0; j < per; ++j) tot += hist[top - ((j + rot) & (per - 1))];
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
                s_sel[2] = c;
                break;
            }
            a += c;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads, 6) sparse_mla_topk_kernel(const TopkParams p) {
    __shared__ __align__(16) uint32_t buf[kTopkBins0];  // pass-1 histogram, then the candidates
    __shared__ uint32_t hist1[kTopkBins1];
    __shared__ __align__(16) uint32_t s_warp[2 * kTopkWarps];
    __shared__ uint32_t s_sel[3];
    __shared__ uint32_t s_cnt[kTopkWarps];  // threshold-bin keys per warp (each warp its own region)
    // launched as a programmatic dependent: the scores may be the previous launch's output
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int tid = threadIdx.x;
    const int64_t t = blockIdx.x;
    const float* row = p.scores + t * p.S;
    int32_t* orow = p.out + t * p.topk;
    int64_t n64 = p.len[t];
    n64 = n64 < 0 ? 0 : (n64 > p.S ? p.S : n64);  // a length outside [0, S] is clamped
    const int n = static_cast<int>(n64);
    const int k = n < p.topk ? n : p.topk;
    auto slot_of = [&](int i) -> int32_t { return p.block_table ? __ldg(p.block_table + (i >> 6)) * 64 + (i & 63) : i; };
    if (k == n) {  // the history is no longer than topk: all of it, then the padding
        for (int i = tid; i < p.topk; i += kTopkThreads) orow[i] = i < n ? slot_of(i) : -1;
        return;
    }

    // the scores at q .. q + 3; in a partial step (full false) those at or past n read as -inf
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    auto load4 = [&](int q, float* x, auto full) {
        if (vec && (decltype(full)::value || q + 4 <= n)) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(row + q));
            x[0] = v.x;
            x[1] = v.y;
            x[2] = v.z;
            x[3] = v.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                x[j] = (decltype(full)::value || q + j < n) ? __ldg(row + q + j) : -INFINITY;
        }
    };
    // one scan step: thread tid's scores of step c0 are c0 + 1024 g + 4 tid + j (g, j < 4);
    // visit(x, g, j, valid) for each
    auto scan_step = [&](int c0, auto full, auto&& visit) {
        float x[kTopkGroups][4];
#pragma unroll
        for (int g = 0; g < kTopkGroups; ++g) load4(c0 + 1024 * g + 4 * tid, x[g], full);
#pragma unroll
        for (int g = 0; g < kTopkGroups; ++g)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                visit(x[g][j], g, j, decltype(full)::value || c0 + 1024 * g + 4 * tid + j < n);
    };
    // every step of the row: the full ones unchecked, then the partial one
    auto scan_row = [&](auto&& step) {
        int c0 = 0;
        for (; c0 + kTopkChunk <= n; c0 += kTopkChunk) step(c0, std::true_type{});
        if (c0 < n) step(c0, std::false_type{});
    };

    // ---- pass 1: histogram of the top 12 key bits
    for (int i = tid; i < kTopkBins0 / 4; i += kTopkThreads) reinterpret_cast<uint4*>(buf)[i] = make_uint4(0, 0, 0, 0);
    if (tid < kTopkWarps) s_cnt[tid] = 0;
    __syncthreads();
    {
        // written out rather than through scan_step: 16 % fewer instructions in this pass
        int c0 = 0;
        if (vec) {
            const float4* row4 = reinterpret_cast<const float4*>(row);
            for (; c0 + kTopkChunk <= n; c0 += kTopkChunk) {
                const float4* src = row4 + (c0 >> 2) + tid;
                float4 v[kTopkGroups];
#pragma unroll
                for (int g = 0; g < kTopkGroups; ++g) v[g] = __ldg(src + 256 * g);
#pragma unroll
                for (int g = 0; g < kTopkGroups; ++g) {
                    atomicAdd(&buf[score_key(v[g].x) >> 20], 1u);
                    atomicAdd(&buf[score_key(v[g].y) >> 20], 1u);
                    atomicAdd(&buf[score_key(v[g].z) >> 20], 1u);
                    atomicAdd(&buf[score_key(v[g].w) >> 20], 1u);
                }
            }
        }
        for (int i = c0 + tid; i < n; i += kTopkThreads) atomicAdd(&buf[score_key(__ldg(row + i)) >> 20], 1u);
    }
    __syncthreads();
    uint32_t krem = static_cast<uint32_t>(k);
    topk_find_bin(buf, kTopkBins0, krem, s_warp, s_sel);
    const uint32_t bin = s_sel[0];
    krem -= s_sel[1];
    const bool few = s_sel[1] + s_sel[2] <= static_cast<uint32_t>(kTopkCand);
    __syncthreads();  // s_sel is rewritten below; buf is free

    if (few) {
        // ---- pass 2: a bitmap of the candidates (every score at or above bin's lowest) in
        // position order, then their positions in that order into buf, a window of kTopkWin
        // positions at a time.  Warp w of a scan step reads positions c0 + 512 w + 32 e + lane
        // (e < 16): one ballot per load gives 32 consecutive positions' bits.
        const float lo = bin_floor(bin);
        const int lane = tid & 31, warp = tid >> 5;
        uint32_t* bits = hist1;  // kTopkWin / 32 words, free until the candidate passes
        uint32_t nc = 0;
        for (int w0 = 0; w0 < n; w0 += kTopkWin) {
            const int wn = n - w0 < kTopkWin ? n - w0 : kTopkWin;
            auto ballot_step = [&](int c0, auto full) {  // c0: a multiple of kTopkChunk below wn
                const int q0 = w0 + c0 + 512 * warp + lane;
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    x[e] = (decltype(full)::value || q0 + 32 * e < n) ? __ldg(row + q0 + 32 * e) : -INFINITY;
                uint32_t mine = 0;  // lane e < 16 keeps word e and stores it
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const uint32_t wd =
                        __ballot_sync(0xffffffffu, (decltype(full)::value || q0 + 32 * e < n) && x[e] >= lo);
                    mine = lane == e ? wd : mine;
                }
                if (lane < 16) bits[(c0 + 512 * warp) / 32 + lane] = mine;
            };
            int c0 = 0;
            for (; c0 + kTopkChunk <= wn; c0 += kTopkChunk) ballot_step(c0, std::true_type{});
            if (c0 < wn) ballot_step(c0, std::false_type{});
            __syncthreads();
            // thread tid's words 4 tid .. 4 tid + 3: positions w0 + 128 tid .. + 127 (words past
            // the window's last step were not written this window: zero)
            uint4 v = make_uint4(0, 0, 0, 0);
            if (128 * tid < wn) v = reinterpret_cast<const uint4*>(bits)[tid];
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            const uint32_t cnt = __popc(wv[0]) + __popc(wv[1]) + __popc(wv[2]) + __popc(wv[3]);
            uint32_t off, off2, tot, tot2;
            block_scan2(cnt, 0u, off, off2, tot, tot2, s_warp);
            // always fits unless scores are NaN; a window that would not is dropped whole, so
            // buf[0, nc) always holds positions of the row
            if (nc + tot <= static_cast<uint32_t>(kTopkCand)) {
                uint32_t r = nc + off;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    for (uint32_t m = wv[q]; m != 0u; m &= m - 1u)
                        buf[r++] = static_cast<uint32_t>(w0 + 128 * tid + 32 * q + __ffs(m) - 1);
                nc += tot;
            }
            __syncthreads();  // bits is rewritten by the next window (or becomes hist1)
        }
        // ---- candidates 512 warp + 32 e + lane (e < 16), their keys gathered once
        uint32_t key[kTopkPerThread];
        uint32_t valid = 0;
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            const int c = 512 * warp + 32 * e + lane;
            key[e] = c < static_cast<int>(nc) ? score_key(__ldg(row + buf[c])) : 0u;
            valid |= static_cast<uint32_t>(c < static_cast<int>(nc)) << e;
        }
        // ---- key bits 19-10, then 9-0, over the candidates in bin
        uint32_t prefix = bin << 20, pmask = 0xFFF00000u;
#pragma unroll 1
        for (int shift = 10; shift >= 0; shift -= 10) {
            for (int i = tid; i < kTopkBins1; i += kTopkThreads) hist1[i] = 0;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kTopkPerThread; ++e)
                if (((valid >> e) & 1u) && (key[e] & pmask) == prefix)
                    atomicAdd(&hist1[(key[e] >> shift) & (kTopkBins1 - 1)], 1u);
            __syncthreads();
            topk_find_bin(hist1, kTopkBins1, krem, s_warp, s_sel);
            krem -= s_sel[1];
            prefix |= s_sel[0] << shift;
            pmask |= static_cast<uint32_t>(kTopkBins1 - 1) << shift;
            __syncthreads();  // hist1 and s_sel are rewritten by the next pass
        }
        // ---- every candidate above the threshold key and the first krem at it, in order: the
        // warps' counts scanned across the CTA, then within a warp one ballot per e
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            const bool v = (valid >> e) & 1u;
            gt |= static_cast<uint32_t>(v && key[e] > prefix) << e;
            eq |= static_cast<uint32_t>(v && key[e] == prefix) << e;
        }
        const uint32_t wgt = __reduce_add_sync(0xffffffffu, __popc(gt));
        const uint32_t weq = __reduce_add_sync(0xffffffffu, __popc(eq));
        if (lane == 0) {
            s_warp[warp] = wgt;
            s_warp[kTopkWarps + warp] = weq;
        }
        __syncthreads();
        uint32_t rgt = 0, req = 0;
#pragma unroll
        for (int w = 0; w < kTopkWarps; ++w)
            if (w < warp) {
                rgt += s_warp[w];
                req += s_warp[kTopkWarps + w];
            }
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            const uint32_t bg = __ballot_sync(0xffffffffu, (gt >> e) & 1u);
            const uint32_t be = __ballot_sync(0xffffffffu, (eq >> e) & 1u);
            const uint32_t g_before = rgt + __popc(bg & lt), e_before = req + __popc(be & lt);
            int slot_out = -1;
            if ((gt >> e) & 1u)
                slot_out = static_cast<int>(g_before + (e_before < krem ? e_before : krem));
            else if (((eq >> e) & 1u) && e_before < krem)
                slot_out = static_cast<int>(g_before + e_before);
            if (slot_out >= 0 && slot_out < k)  // always below k; the check keeps every store in the row
                orow[slot_out] = slot_of(static_cast<int>(buf[512 * warp + 32 * e + lane]));
            rgt += __popc(bg);
            req += __popc(be);
        }
        for (int i = k + tid; i < p.topk; i += kTopkThreads) orow[i] = -1;
        return;
    }

    // ---- many keys in bin: its keys alone into shared memory, each warp into its own region
    // through its own counter (one counter for the CTA serialised them); the counts go on past
    // the regions
    uint32_t prefix = bin << 20, pmask = 0xFFF00000u;
    {
        const int w = tid >> 5;
        scan_row([&](int c0, auto full) {
            scan_step(c0, full, [&](float x, int, int, bool valid) {
                const uint32_t key = score_key(x);
                if (valid && (key & pmask) == prefix) {
                    const uint32_t c = atomicAdd(&s_cnt[w], 1u);
                    if (c < kTopkBinKeysW) buf[w * kTopkBinKeysW + c] = key;
                }
            });
        });
    }
    __syncthreads();
    bool in_smem = true;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) in_smem = in_smem && s_cnt[w] <= static_cast<uint32_t>(kTopkBinKeysW);
    // key bits 19-12, 11-4 and 3-0, over those keys (over the row when they did not fit)
#pragma unroll 1
    for (int step = 0; step < 3; ++step) {
        const int shift = step == 0 ? 12 : (step == 1 ? 4 : 0);
        const int nb = step == 2 ? 16 : 256;
        for (int i = tid; i < nb; i += kTopkThreads) hist1[i] = 0;
        __syncthreads();
        auto count = [&](uint32_t key) {
            if ((key & pmask) == prefix) atomicAdd(&hist1[(key >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
        };
        if (in_smem) {
            for (int c = tid; c < kTopkBinKeys; c += kTopkThreads)
                if (static_cast<uint32_t>(c % kTopkBinKeysW) < s_cnt[c / kTopkBinKeysW]) count(buf[c]);
        } else {
            scan_row([&](int c0, auto full) {
                scan_step(c0, full, [&](float x, int, int, bool valid) {
                    if (valid) count(score_key(x));
                });
            });
        }
        __syncthreads();
        topk_find_bin(hist1, nb, krem, s_warp, s_sel);
        krem -= s_sel[1];
        prefix |= s_sel[0] << shift;
        pmask |= static_cast<uint32_t>(nb - 1) << shift;
        __syncthreads();  // hist1 and s_sel are rewritten by the next pass
    }

    // ---- every key above the threshold and the first krem at it, in position order: thread
    // tid takes 16 consecutive scores a step
    uint32_t base_gt = 0, base_eq = 0;
    for (int c0 = 0; c0 < n; c0 += kTopkCand) {
        const int i0 = c0 + tid * kTopkPerThread;
        float xs[kTopkPerThread];
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
        // bit e of gt / eq: score i0 + e is above the threshold / equal to it
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            if (i0 + e < n) {
                const uint32_t key = score_key(xs[e]);
                gt |= static_cast<uint32_t>(key > prefix) << e;
                eq |= static_cast<uint32_t>(key == prefix) << e;
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
                orow[slot_out] = slot_of(i);
        }
        base_gt += tgt;
        base_eq += teq;
    }
    for (int i = k + tid; i < p.topk; i += kTopkThreads) orow[i] = -1;
}

}  // namespace smla
