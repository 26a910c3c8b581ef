// Pieces shared by both forward kernels: sizes, launch parameters, the device error word,
// small helpers and the KV row gather run by the producer warps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "sm100_ptx.cuh"

namespace smla {

constexpr int kDQK = 576;                           // 512 latent + 64 rope dims per row
constexpr int kDV = 512;                            // value / output dims (the latent part)
constexpr int kPanels = kDQK / 64;                  // 9 panels of 64 bf16 = 128 bytes per row
constexpr int kMaxSplits = 8;                       // CTAs per token (one portable cluster)
constexpr int kMaxParts = 16;                       // CTAs sharing one token (balanced partition)
constexpr int kProducerWarps = 7;
constexpr int kFp8RowBytes = 656;
constexpr float kRescaleLog2 = 8.0f;                // rescale O only when max grows by > 2^8
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // bounded waits: 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;    // draining in-flight work after an abort

// device error word bits (read by sparse_mla_sync_status)
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrLayout = 2u;
constexpr unsigned int kErrIndexRange = 4u;         // checked mode: an entry other than -1 was invalid

struct FwdParams {
    const __nv_bfloat16* q;   // [T, h, 576]
    const void* kv;           // [num_slots] rows: 576 bf16, or 656 bytes of fp8 + scales + rope
    const int32_t* indices;   // [T, topk]
    __nv_bfloat16* out;       // [T, h, 512]
    float* lse;               // [T, h]
    int64_t num_slots;
    int32_t T, h, topk, splits;
    float sm_scale_log2;      // scale * log2(e)
    // balanced partition (small-head kernel): `grid` CTAs take equal contiguous ranges of the
    // token-major sequence of T * nblk row blocks; the parts of a list cut between CTAs go to
    // `part` ([grid][2] slots of 2h + 512h floats) and are merged after a grid-wide barrier on
    // the counter words `gbar` (cooperative launch).  part == nullptr: no list is cut.
    int32_t grid, nblk;
    float* part;
    unsigned int* gbar;
    // checked mode: list entries other than -1 outside [0, num_slots) are still masked, and the
    // producers also set kErrIndexRange in the device error word
    int32_t checked;
};

__device__ unsigned int g_smla_error;

// Checked mode: one warp-wide vote over the raw entries this warp's lanes hold (-1 never
// counts), and one atomic per warp that found an out-of-range entry.
__device__ __forceinline__ void flag_out_of_range(int raw, int slot) {
    const bool bad = raw != -1 && slot < 0;
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&g_smla_error, kErrIndexRange);
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(bf16_bits(lo)) | (static_cast<uint32_t>(bf16_bits(hi)) << 16);
}

// Raw list entry j of a row (-1 when j is past the CTA's range or pred is false).  The load is
// not checked here: the check reads the value, and a read right after the load would wait for
// it.  Callers hold raw entries in a ring and check them with valid_slot when they are used.
__device__ __forceinline__ int fetch_entry(const int32_t* idx_row, int j, int j1, bool pred) {
    int v = -1;
    if (pred && j < j1) v = __ldg(idx_row + j);
    return v;
}

// A list entry names a cache row when 0 <= entry < num_slots; anything else is masked (-1).
__device__ __forceinline__ int valid_slot(int raw, int64_t num_slots) {
    return (raw >= 0 && static_cast<int64_t>(raw) < num_slots) ? raw : -1;
}

// The KV row gather, run by producer warp pw (of NPW) for this CTA's nb blocks of
// ROWS list entries [j0, j1).  Block b goes to stage b % NST; a stage is a ROWS-row tile in the
// 128-byte-swizzled K-major operand layout: 9 panels of ROWS x 128 bytes, the 16-byte chunk c of
// row r in panel p at p * ROWS * 128 + r * 128 + ((c ^ (r & 7)) << 4).  Each producer thread
// arrives once per block on the stage's full barrier (expected count 32 * NPW) and a
// stage is refilled only after its empty barrier completes.
//   KVF 0: bf16 rows, copied with 16-byte cp.async, one warp instruction = 512 contiguous bytes
//          of a row; invalid entries are zero-filled without a read.
//   KVF 1: fp8 rows (656 bytes: [512 e4m3 | 4 fp32 scales, one per 128 latent values | 64 bf16
//          rope]); each lane loads 16 latent bytes, its tile scale and (lanes 0-7) 16 rope bytes
//          of a row into registers, dequantises (e4m3 -> f16 exactly, x scale in fp32, -> bf16
//          round to nearest even) and stores into the same bf16 tile.
template <int ROWS, int NST, int KVF, int NPW>
__device__ __forceinline__ void gather_rows(const FwdParams& p, const int32_t* idx_row, int j0, int j1,
                                            int nb, int pw, int lane, uint32_t sKV, uint32_t bar_full0,
                                            uint32_t bar_empty0, volatile int* sAbort) {
    constexpr int kRows = ROWS;
    constexpr int kPanelBytes = ROWS * 128;
    constexpr int kStageBytes = kPanels * kPanelBytes;
    constexpr int kPerWarp = (ROWS + NPW - 1) / NPW;
    auto wait_empty = [&](int s, uint32_t parity) -> bool {
        return ptx::mbar_wait(bar_empty0 + 8u * s, parity, sAbort, &g_smla_error, kErrTimeout,
                              kWaitLimitNs);
    };
    // warp pw copies rows pw, pw + NPW, pw + 2 NPW, ... of each block; lane i < kPerWarp
    // holds the slot of the warp's i-th row.
    const char* kv_bytes = reinterpret_cast<const char*>(p.kv);
    const int my_row = pw + NPW * lane;
    const bool row_owner = lane < kPerWarp && my_row < kRows;
    // The entries of this lane's row are loaded kAhead blocks (256 list entries) ahead into a
    // ring indexed by b % kAhead; the block loop is unrolled kAhead times so every ring index is
    // static and a load is first read kAhead blocks after it was issued.
    constexpr int kAhead = 256 / ROWS;
    int ring[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) ring[u] = fetch_entry(idx_row, j0 + u * kRows + my_row, j1, row_owner && u < nb);
    bool aborted = false;
    for (int b0 = 0; b0 < nb && !aborted; b0 += kAhead) {
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const int b = b0 + u;
            if (b >= nb) break;
            const int s = b % NST;
            const int my_slot = valid_slot(ring[u], p.num_slots);
            if (p.checked) flag_out_of_range(ring[u], my_slot);
            ring[u] = fetch_entry(idx_row, j0 + (b + kAhead) * kRows + my_row, j1, row_owner && b + kAhead < nb);
            if constexpr (KVF == 0) {
                if (b >= NST) {
                    bool ok = true;
                    if (lane == 0) ok = wait_empty(s, ((b / NST) - 1) & 1);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    __syncwarp();
                    if (!ok) {
                        aborted = true;
                        break;
                    }
                }
                const uint32_t st = sKV + s * kStageBytes;
#pragma unroll 1
                for (int i = 0; i < kPerWarp; ++i) {
                    const int r = pw + NPW * i;
                    if (r >= kRows) break;
                    const int slot = __shfl_sync(0xffffffffu, my_slot, i);
                    const char* src = kv_bytes + static_cast<int64_t>(slot < 0 ? 0 : slot) * (kDQK * 2);
                    const uint32_t nbytes = slot < 0 ? 0u : 16u;
                    const uint32_t dst_row = st + r * 128;
                    const uint32_t sw = static_cast<uint32_t>(r & 7);
#pragma unroll
                    for (int cc = 0; cc < 3; ++cc) {
                        const int c = lane + 32 * cc;  // 16-byte chunk of the 1152-byte row
                        if (c < 72) {
                            const uint32_t dst = dst_row + (c >> 3) * kPanelBytes + (((c & 7) ^ sw) << 4);
                            ptx::cp_async_16(dst, src + c * 16, nbytes);
                        }
                    }
                }
                ptx::cp_async_arrive_noinc(bar_full0 + 8u * s);
            } else {
                // fp8 rows: each lane of the warp takes 16 latent bytes of a row (dims 16*lane ..
                // 16*lane+15, tile scale lane/8); lanes 0-7 also take 16 bytes of the bf16 rope.
                // The loads of a block are issued before waiting for its stage to be free.
                const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
                uint4 lat[kPerWarp], rope[kPerWarp];
                float scl[kPerWarp];
#pragma unroll
                for (int i = 0; i < kPerWarp; ++i) {
                    const int r = pw + NPW * i;
                    const int slot = __shfl_sync(0xffffffffu, my_slot, i);
                    lat[i] = make_uint4(0u, 0u, 0u, 0u);
                    rope[i] = make_uint4(0u, 0u, 0u, 0u);
                    scl[i] = 0.f;
                    if (r < kRows && slot >= 0) {
                        const uint8_t* row = kv8 + static_cast<int64_t>(slot) * kFp8RowBytes;
                        lat[i] = ptx::ld_nc_v4(row + 16 * lane);
                        scl[i] = ptx::ld_nc_f32(row + 512 + 4 * (lane >> 3));
                        if (lane < 8) rope[i] = ptx::ld_nc_v4(row + 528 + 16 * lane);
                    }
                }
                if (b >= NST) {
                    bool ok = true;
                    if (lane == 0) ok = wait_empty(s, ((b / NST) - 1) & 1);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    __syncwarp();
                    if (!ok) {
                        aborted = true;
                        break;
                    }
                }
                const uint32_t st = sKV + s * kStageBytes;
#pragma unroll
                for (int i = 0; i < kPerWarp; ++i) {
                    const int r = pw + NPW * i;
                    if (r < kRows) {
                        const uint32_t sw = static_cast<uint32_t>(r & 7);
                        const uint32_t row_dst = st + r * 128;
                        // 16 e4m3 values -> 16 bf16 (two 16-byte chunks of panel lane/4)
                        uint4 v0, v1;
                        v0.x = ptx::e4m3x2_scaled_bf16x2(lat[i].x & 0xFFFFu, scl[i]);
                        v0.y = ptx::e4m3x2_scaled_bf16x2(lat[i].x >> 16, scl[i]);
                        v0.z = ptx::e4m3x2_scaled_bf16x2(lat[i].y & 0xFFFFu, scl[i]);
                        v0.w = ptx::e4m3x2_scaled_bf16x2(lat[i].y >> 16, scl[i]);
                        v1.x = ptx::e4m3x2_scaled_bf16x2(lat[i].z & 0xFFFFu, scl[i]);
                        v1.y = ptx::e4m3x2_scaled_bf16x2(lat[i].z >> 16, scl[i]);
                        v1.z = ptx::e4m3x2_scaled_bf16x2(lat[i].w & 0xFFFFu, scl[i]);
                        v1.w = ptx::e4m3x2_scaled_bf16x2(lat[i].w >> 16, scl[i]);
                        const uint32_t pan = row_dst + (lane >> 2) * kPanelBytes;
                        const uint32_t ch = static_cast<uint32_t>((lane & 3) * 2);
                        ptx::st_shared_v4(pan + ((ch ^ sw) << 4), v0);
                        ptx::st_shared_v4(pan + (((ch + 1) ^ sw) << 4), v1);
                        if (lane < 8)
                            ptx::st_shared_v4(row_dst + 8 * kPanelBytes + ((static_cast<uint32_t>(lane) ^ sw) << 4),
                                              rope[i]);
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(bar_full0 + 8u * s);
            }
        }
    }
    ptx::cp_async_wait_all();  // no copy may still be in flight when the CTA leaves
}

}  // namespace smla
