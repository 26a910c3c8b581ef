// Merge of the partial results of split top-k lists (the DCP merge).
//
// With decode context parallelism a token's top-k list is split across ranks; each rank runs
// the forward over its part and returns O_p (normalised over the part) and LSE_p, and the
// consumer merges them (vLLM PR #60220, Details: out and lse are "consumed by the v_up
// projection or the DCP merge"; vLLM PR #64510, Details: heads gathered by DCP).  The pages do
// not write the merge; it is the exact combination of softmax results over disjoint parts of
// one list:
//
//   M = max_p LSE_p,   LSE = M + ln sum_p exp(LSE_p - M),   O = sum_p exp(LSE_p - LSE) O_p
//
// an empty part (LSE_p = -inf) weighing 0 and a row with no non-empty part giving O = 0,
// LSE = -inf (what the forward returns for an empty list).
//
// The kernel is a stream over HBM: per (token, head) row it reads n LSEs and n x 1 KB of bf16
// O, and writes 1 KB + 4 bytes.  One warp per row: lanes 0..n-1 hold the parts' LSEs and their
// weights (warp shuffles for the max and the sum), then every lane accumulates two 16-byte
// chunks (dims 8c .. 8c+7 for c = lane, lane + 32) of every non-empty part in fp32 and stores
// them as bf16; each part's row is one coalesced 1 KB read.  A grid of a few CTAs per SM
// strides over the rows.
#pragma once

#include "sparse_mla_common.cuh"

namespace smla {

constexpr int kMergeMaxParts = 16;
constexpr int kMergeThreads = 256;  // eight rows in flight per CTA

struct MergeParams {
    const __nv_bfloat16* o_parts;  // [n][rows][512]
    const float* lse_parts;        // [n][rows]
    __nv_bfloat16* out;            // [rows][512]
    float* lse;                    // [rows]
    int64_t rows;                  // T * h
    int32_t n;                     // 1 .. kMergeMaxParts
};

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4 v, float w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += w * __uint_as_float(u[i] << 16);
        acc[2 * i + 1] += w * __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

__global__ void __launch_bounds__(kMergeThreads) sparse_mla_merge_kernel(const MergeParams mp) {
    // launched as a programmatic dependent: nothing before this reads global memory
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t first = (static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
    const int64_t stride = (static_cast<int64_t>(gridDim.x) * kMergeThreads) >> 5;
    constexpr float kLog2e = 1.4426950408889634f;
    for (int64_t row = first; row < mp.rows; row += stride) {
        const float lp = lane < mp.n ? __ldg(mp.lse_parts + lane * mp.rows + row) : -CUDART_INF_F;
        float m = lp;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float w = (lp != -CUDART_INF_F) ? ptx::ex2_approx((lp - m) * kLog2e) : 0.f;
        float sum = w;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) mp.lse[row] = sum > 0.f ? m + logf(sum) : -CUDART_INF_F;
        w = sum > 0.f ? w / sum : 0.f;

        float acc0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float acc1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int p0 = 0; p0 < mp.n; p0 += 4) {
            // four parts' chunks in flight before their weights are applied
            uint4 va[4], vb[4];
            float wp[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = p0 + u;
                wp[u] = __shfl_sync(0xffffffffu, w, p & 31);
                if (p < mp.n && wp[u] != 0.f) {
                    const uint4* src = reinterpret_cast<const uint4*>(mp.o_parts + (p * mp.rows + row) * kDV);
                    va[u] = __ldcs(src + lane);
                    vb[u] = __ldcs(src + lane + 32);
                } else {
                    wp[u] = 0.f;
                    va[u] = vb[u] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc_bf16x8(acc0, va[u], wp[u]);
                acc_bf16x8(acc1, vb[u], wp[u]);
            }
        }
        uint4 r0, r1;
        r0.x = pack_bf16x2(acc0[0], acc0[1]); r0.y = pack_bf16x2(acc0[2], acc0[3]);
        r0.z = pack_bf16x2(acc0[4], acc0[5]); r0.w = pack_bf16x2(acc0[6], acc0[7]);
        r1.x = pack_bf16x2(acc1[0], acc1[1]); r1.y = pack_bf16x2(acc1[2], acc1[3]);
        r1.z = pack_bf16x2(acc1[4], acc1[5]); r1.w = pack_bf16x2(acc1[6], acc1[7]);
        uint4* dst = reinterpret_cast<uint4*>(mp.out + row * kDV);
        __stcs(dst + lane, r0);
        __stcs(dst + lane + 32, r1);
    }
}

}  // namespace smla
