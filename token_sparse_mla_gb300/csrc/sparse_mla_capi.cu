// C ABI of libsparse_mla.so: argument validation, tensor-map encoding and launch.
// The declarations, argument meanings and error behaviour are documented in
// include/sparse_mla.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "sparse_mla.h"
#include "sparse_mla_kernel.cuh"
#include "sparse_mla_small_kernel.cuh"
#include "sparse_mla_merge.cuh"
#include "sparse_mla_v_up.cuh"
#include "sparse_mla_topk.cuh"
#include "sparse_mla_masked.cuh"

namespace {

constexpr int32_t kVersion = 10100;  // 1.1.0: checked mode, packed host buffers
constexpr int kMaxDevices = 64;

thread_local char g_last_error[512] = "";

smla_status fail(smla_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

smla_status cuda_fail(cudaError_t e, const char* what) {
    return fail(SMLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    std::once_flag once;
    cudaError_t init_error = cudaSuccess;
    int num_sms = 0;
    // the static merge scratch of sparse_mla_fwd_noalloc on this device (set once, under
    // g_static_mu)
    void* static_ptr = nullptr;
};

DeviceState g_dev[kMaxDevices];
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t set_kernel_attrs() {
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<8, 0, false>, smla::SmallLayout<8, 0>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<8, 1, false>, smla::SmallLayout<8, 1>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<16, 0, false>, smla::SmallLayout<16, 0>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<16, 1, false>, smla::SmallLayout<16, 1>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<8, 0, true>, smla::SmallLayout<8, 0>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<8, 1, true>, smla::SmallLayout<8, 1>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<16, 0, true>, smla::SmallLayout<16, 0>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_small_kernel<16, 1, true>, smla::SmallLayout<16, 1>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_v_up_kernel, smla::VupLayout::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_tc_kernel<32, 0>, smla::Layout<32>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_tc_kernel<32, 1>, smla::Layout<32>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_tc_kernel<64, 0>, smla::Layout<64>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_fwd_tc_kernel<64, 1>, smla::Layout<64>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_masked_mha_kernel<192, 128>, smla::MmLayout<192, 128>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_masked_mha_kernel<192, 256>, smla::MmLayout<192, 256>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_masked_mha_kernel<256, 128>, smla::MmLayout<256, 128>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_masked_mha_kernel<256, 256>, smla::MmLayout<256, 256>::kBytes);
    if (e == cudaSuccess) e = set_smem(smla::sparse_mla_scatter_mask_kernel, smla::kScatterMaxS / 32 * 4);
    return e;
}

smla_status device_state(int* dev_out, DeviceState** st_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SMLA_ERR_UNSUPPORTED, "device ordinal %d", dev);
    DeviceState& st = g_dev[dev];
    std::call_once(st.once, [&] {
        cudaDeviceProp prop;
        cudaError_t err = cudaGetDeviceProperties(&prop, dev);
        if (err == cudaSuccess && prop.major < 10) err = cudaErrorInvalidDeviceFunction;
        if (err == cudaSuccess) st.num_sms = prop.multiProcessorCount;
        if (err == cudaSuccess) err = set_kernel_attrs();
        st.init_error = err;
    });
    if (st.init_error != cudaSuccess) return cuda_fail(st.init_error, "device set-up");
    *dev_out = dev;
    *st_out = &st;
    return SMLA_OK;
}

smla_status encode_fn(EncodeTiledFn* fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!g_encode) return fail(SMLA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    *fn = g_encode;
    return SMLA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// 8 and 16 heads run the warp-MMA kernel (32-row stages); 32 and 64 the tcgen05 kernel.
bool small_heads(int h) { return h <= 16; }

// Split count: enough CTAs to cover the SMs once when there are few tokens.
int auto_splits(int64_t T, int nblk, int num_sms) {
    int s = 1;
    const int cand[3] = {8, 4, 2};
    for (int c : cand) {
        if (c <= nblk && T * c <= num_sms) {
            s = c;
            break;
        }
    }
    return s;
}

struct Plan {
    int hp = 16;
    int threads = 0;
    int splits = 1;       // tcgen05 kernel: CTAs (cluster) per token; small-head kernel: 0
    int64_t ctas = 0;
    int smem = 0;
    int nblk = 0;         // row blocks per token
    size_t scratch = 0;   // small-head kernel: bytes of merge scratch (0 = no token is cut)
};

// Scratch of the small-head kernel's balanced partition: the grid-barrier words (arrival count
// and generation, in a 256-byte head that starts zeroed) followed by grid x 2 partial slots of
// (2h + 512h) floats.
constexpr size_t kScratchHead = 256;
size_t small_scratch_bytes(int64_t grid, int h) {
    return kScratchHead + static_cast<size_t>(grid) * 2 * (2 * h + h * smla::kDV) * 4;
}

// File-scope merge scratch of sparse_mla_fwd_noalloc: sized for 16 heads on up to 160 CTAs (a
// launch that cuts lists never has more CTAs than SMs).  Zero-initialised when the module loads;
// its head (the grid-barrier words) is cleared once more per device at first use.
constexpr size_t kStaticScratchBytes = kScratchHead + static_cast<size_t>(160) * 2 * (2 * 16 + 16 * smla::kDV) * 4;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

smla_status check_args(const void* q, const void* kv, const int32_t* idx, int32_t T, int32_t h,
                       int32_t topk, int64_t num_slots, int32_t kv_format, float scale,
                       const void* out, const float* lse, int32_t splits) {
    if (T < 0) return fail(SMLA_ERR_INVALID_ARG, "T must be >= 0 (got %d)", T);
    if (!(h == 8 || h == 16 || h == 32 || h == 64))
        return fail(SMLA_ERR_UNSUPPORTED, "h must be 8, 16, 32 or 64 (got %d)", h);
    if (topk < 1) return fail(SMLA_ERR_INVALID_ARG, "topk must be >= 1 (got %d)", topk);
    if (num_slots < 1 || num_slots > 0x7fffffffLL)
        return fail(SMLA_ERR_INVALID_ARG, "num_slots must be in [1, 2^31-1] (got %lld)",
                    static_cast<long long>(num_slots));
    if (kv_format != SMLA_KV_BF16 && kv_format != SMLA_KV_FP8)
        return fail(SMLA_ERR_INVALID_ARG, "unknown kv_format %d", kv_format);
    if (!std::isfinite(scale)) return fail(SMLA_ERR_INVALID_ARG, "scale must be finite");
    if (!(splits == 0 || splits == 1 || splits == 2 || splits == 4 || splits == 8))
        return fail(SMLA_ERR_INVALID_ARG, "splits must be 0 (auto), 1, 2, 4 or 8 (got %d)", splits);
    if (T == 0) return SMLA_OK;
    if (!q || !kv || !idx || !out || !lse) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16))
        return fail(SMLA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
    if (!aligned(idx, 4) || !aligned(lse, 4))
        return fail(SMLA_ERR_INVALID_ARG, "indices and lse must be 4-byte aligned");
    if (static_cast<int64_t>(T) * 8 > 0x7fffffffLL)
        return fail(SMLA_ERR_INVALID_ARG, "T too large for one launch (%d)", T);
    if (topk > (1 << 20)) return fail(SMLA_ERR_INVALID_ARG, "topk above 2^20 (%d)", topk);
    return SMLA_OK;
}

Plan make_plan(int32_t T, int32_t h, int32_t topk, int32_t splits, int num_sms, bool fp8) {
    Plan pl;
    pl.hp = h;
    const int rows = small_heads(h) ? smla::kSmRows : smla::kRows;
    const int nblk = (topk + rows - 1) / rows;
    pl.nblk = nblk;
    if (small_heads(h)) {
        // The T * nblk row blocks are cut into `ctas` equal contiguous ranges.  Default: whole
        // lists (one CTA per token) once the tokens alone fill the SMs; otherwise s CTAs per
        // token, s the largest power of two that divides nblk with T * s <= #SMs and s <= 8,
        // so every range is an aligned part of one list: one thread-block cluster per token,
        // merged through distributed shared memory.  Given `splits`: T * splits CTAs; if the
        // cuts do not fall on whole parts, the parts are merged through the scratch after a
        // grid-wide barrier, so such a launch never has more CTAs than SMs.
        const int64_t W = static_cast<int64_t>(T) * nblk;
        int64_t want = T;
        if (splits > 0) {
            want = static_cast<int64_t>(T) * splits;
        } else {
            for (int c = smla::kMaxSplits; c > 1; c >>= 1) {
                if (nblk % c == 0 && static_cast<int64_t>(T) * c <= num_sms) {
                    want = static_cast<int64_t>(T) * c;
                    break;
                }
            }
        }
        pl.splits = 0;
        pl.ctas = W < want ? W : want;
        auto whole_lists = [&](int64_t g) { return W % g == 0 && (W / g) % nblk == 0; };
        const int64_t per_token = (T > 0 && pl.ctas % T == 0) ? pl.ctas / T : 0;
        const bool pow2 = per_token > 0 && (per_token & (per_token - 1)) == 0;
        if (pow2 && per_token >= 2 && per_token <= smla::kMaxSplits && nblk % per_token == 0) {
            // aligned parts, 2, 4 or 8 per list (so each CTA of the cluster owns 512 / parts
            // output dims, a multiple of 8): one thread-block cluster per token, merged through
            // distributed shared memory (no scratch, no grid barrier)
            pl.splits = static_cast<int>(per_token);
        } else {
            if (pl.ctas > num_sms && !whole_lists(pl.ctas)) pl.ctas = num_sms;
            if (pl.ctas > 0 && !whole_lists(pl.ctas)) pl.scratch = small_scratch_bytes(pl.ctas, h);
        }
    } else {
        pl.splits = splits > 0 ? splits : auto_splits(T, nblk, num_sms);
        pl.ctas = static_cast<int64_t>(T) * pl.splits;
    }
    pl.threads = small_heads(h) ? (fp8 ? smla::SmRoles<1>::kThreads : smla::SmRoles<0>::kThreads)
                               : (fp8 ? smla::TcRoles<1>::kThreads : smla::TcRoles<0>::kThreads);
    pl.smem = h == 8    ? (fp8 ? smla::SmallLayout<8, 1>::kBytes : smla::SmallLayout<8, 0>::kBytes)
              : h == 16 ? (fp8 ? smla::SmallLayout<16, 1>::kBytes : smla::SmallLayout<16, 0>::kBytes)
              : h == 32 ? smla::Layout<32>::kBytes
                        : smla::Layout<64>::kBytes;
    return pl;
}

// Library-owned merge scratch, one buffer per (device, stream), grown on demand.  Calls on one
// stream are ordered, so they can share it; calls on different streams get different buffers.
struct Scratch {
    int dev = 0;
    cudaStream_t stream = nullptr;
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_scratch_mu;
std::vector<Scratch> g_scratch;

smla_status stream_scratch(int dev, cudaStream_t stream, size_t need, void** ptr) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    Scratch* sc = nullptr;
    for (Scratch& x : g_scratch)
        if (x.dev == dev && x.stream == stream) sc = &x;
    if (!sc) {
        g_scratch.push_back(Scratch{});
        sc = &g_scratch.back();
        sc->dev = dev;
        sc->stream = stream;
    }
    if (sc->bytes < need) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
        if (cs != cudaStreamCaptureStatusNone)
            return fail(SMLA_ERR_INVALID_ARG,
                        "stream capture needs %zu bytes of merge scratch on this stream; make one call of "
                        "the same size on the stream before capturing", need);
        if (sc->ptr) {
            e = cudaStreamSynchronize(stream);  // earlier launches may still use the old buffer
            if (e == cudaSuccess) e = cudaFree(sc->ptr);
            sc->ptr = nullptr;
            sc->bytes = 0;
            if (e != cudaSuccess) return cuda_fail(e, "releasing the merge scratch");
        }
        void* p = nullptr;
        e = cudaMalloc(&p, need);
        if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, need, stream);
        if (e != cudaSuccess) {
            if (p) cudaFree(p);
            return cuda_fail(e, "allocating the merge scratch");
        }
        sc->ptr = p;
        sc->bytes = need;
    }
    *ptr = sc->ptr;
    return SMLA_OK;
}

// The device address of the static scratch, looked up (and its head cleared) once per device.
// That first call must not be inside a stream capture (it synchronises the device).
std::mutex g_static_mu;

smla_status static_scratch(DeviceState* ds, cudaStream_t stream, void** ptr) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!ds->static_ptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
        if (cs != cudaStreamCaptureStatusNone)
            return fail(SMLA_ERR_INVALID_ARG,
                        "the first sparse_mla_fwd_noalloc call on a device must not be captured");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e == cudaSuccess) e = cudaMemset(p, 0, kScratchHead);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "setting up the static merge scratch");
        ds->static_ptr = p;
    }
    *ptr = ds->static_ptr;
    return SMLA_OK;
}

enum class ScratchSource { kStream, kStatic };

smla_status launch(const void* q, const void* kv, const int32_t* idx, int32_t T, int32_t h,
                   int32_t topk, int64_t num_slots, int32_t kv_format, float scale, void* out,
                   float* lse, int32_t splits, cudaStream_t stream,
                   ScratchSource source = ScratchSource::kStream, bool checked = false) {
    smla_status st = check_args(q, kv, idx, T, h, topk, num_slots, kv_format, scale, out, lse, splits);
    if (st != SMLA_OK || T == 0) return st;
    int dev = 0;
    DeviceState* ds = nullptr;
    if ((st = device_state(&dev, &ds)) != SMLA_OK) return st;
    EncodeTiledFn enc = nullptr;
    if (!small_heads(h) && (st = encode_fn(&enc)) != SMLA_OK) return st;
    const Plan pl = make_plan(T, h, topk, splits, ds->num_sms, kv_format == SMLA_KV_FP8);

    alignas(64) CUtensorMap tm_q;
    if (!small_heads(h)) {  // the tcgen05 kernel loads Q^T with TMA
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(smla::kDQK), static_cast<cuuint64_t>(h),
                                    static_cast<cuuint64_t>(T)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(smla::kDQK) * 2,
                                       static_cast<cuuint64_t>(smla::kDQK) * 2 * h};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(h), 1};
        const cuuint32_t es[3] = {1, 1, 1};
        CUresult r = enc(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(SMLA_ERR_CUDA, "tensor map for q failed (%d)", (int)r);
    }

    smla::FwdParams prm;
    prm.q = reinterpret_cast<const __nv_bfloat16*>(q);
    prm.kv = kv;
    prm.indices = idx;
    prm.out = reinterpret_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.num_slots = num_slots;
    prm.T = T;
    prm.h = h;
    prm.topk = topk;
    prm.splits = pl.splits;
    prm.sm_scale_log2 = scale * 1.4426950408889634f;
    prm.grid = static_cast<int32_t>(pl.ctas);
    prm.nblk = pl.nblk;
    prm.part = nullptr;
    prm.gbar = nullptr;
    prm.checked = checked ? 1 : 0;
    if (pl.scratch > 0) {
        void* sp = nullptr;
        if (source == ScratchSource::kStatic) {
            if (pl.scratch > kStaticScratchBytes)
                return fail(SMLA_ERR_UNSUPPORTED, "this launch needs %zu bytes of merge scratch; the static scratch has %zu",
                            pl.scratch, kStaticScratchBytes);
            if ((st = static_scratch(ds, stream, &sp)) != SMLA_OK) return st;
        } else if ((st = stream_scratch(dev, stream, pl.scratch, &sp)) != SMLA_OK) {
            return st;
        }
        prm.gbar = static_cast<unsigned int*>(sp);
        prm.part = reinterpret_cast<float*>(static_cast<char*>(sp) + kScratchHead);
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(pl.threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    if (pl.splits > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(pl.splits);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    } else if (pl.scratch > 0) {
        // the merge of cut lists waits at a grid-wide barrier: all CTAs must be co-resident
        attr[nattr].id = cudaLaunchAttributeCooperative;
        attr[nattr].val.cooperative = 1;
        ++nattr;
    }
    if (pl.scratch == 0) {
        // programmatic dependent launch: this grid may be scheduled while the previous work on
        // the stream drains; the kernels wait (griddepcontrol.wait) before touching global memory
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = nattr ? attr : nullptr;
    cfg.numAttrs = nattr;
    cudaError_t e;
    const bool fp8 = kv_format == SMLA_KV_FP8;
    const bool cl = pl.splits > 1;  // small-head kernels: the cluster-merge instantiation
    if (h == 8 && cl)
        e = fp8 ? cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<8, 1, true>, prm)
                : cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<8, 0, true>, prm);
    else if (h == 8)
        e = fp8 ? cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<8, 1, false>, prm)
                : cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<8, 0, false>, prm);
    else if (h == 16 && cl)
        e = fp8 ? cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<16, 1, true>, prm)
                : cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<16, 0, true>, prm);
    else if (h == 16)
        e = fp8 ? cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<16, 1, false>, prm)
                : cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_small_kernel<16, 0, false>, prm);
    else if (h == 32)
        e = fp8 ? cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_tc_kernel<32, 1>, tm_q, prm)
                : cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_tc_kernel<32, 0>, tm_q, prm);
    else
        e = fp8 ? cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_tc_kernel<64, 1>, tm_q, prm)
                : cudaLaunchKernelEx(&cfg, smla::sparse_mla_fwd_tc_kernel<64, 0>, tm_q, prm);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return SMLA_OK;
}

}  // namespace

extern "C" {

smla_status sparse_mla_fwd(const void* q, const void* kv_cache, const int32_t* indices, int32_t T,
                           int32_t h, int32_t topk, int64_t num_slots, int32_t kv_format,
                           float scale, void* out, float* lse, void* stream) {
    return launch(q, kv_cache, indices, T, h, topk, num_slots, kv_format, scale, out, lse, 0,
                  static_cast<cudaStream_t>(stream));
}

smla_status sparse_mla_fwd_ex(const void* q, const void* kv_cache, const int32_t* indices,
                              int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                              int32_t kv_format, float scale, void* out, float* lse, int32_t splits,
                              void* stream) {
    return launch(q, kv_cache, indices, T, h, topk, num_slots, kv_format, scale, out, lse, splits,
                  static_cast<cudaStream_t>(stream));
}

smla_status sparse_mla_fwd_checked(const void* q, const void* kv_cache, const int32_t* indices,
                                   int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                                   int32_t kv_format, float scale, void* out, float* lse,
                                   int32_t splits, void* stream) {
    return launch(q, kv_cache, indices, T, h, topk, num_slots, kv_format, scale, out, lse, splits,
                  static_cast<cudaStream_t>(stream), ScratchSource::kStream, true);
}

smla_status sparse_mla_fwd_noalloc(const void* q, const void* kv_cache, const int32_t* indices,
                                   int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                                   int32_t kv_format, float scale, void* out, float* lse,
                                   int32_t splits, void* stream) {
    return launch(q, kv_cache, indices, T, h, topk, num_slots, kv_format, scale, out, lse, splits,
                  static_cast<cudaStream_t>(stream), ScratchSource::kStatic);
}

size_t sparse_mla_host_workspace_bytes(int32_t T, int32_t h, int32_t topk) {
    if (T <= 0 || h <= 0 || topk <= 0) return 0;
    const size_t t = static_cast<size_t>(T);
    return align256(t * h * smla::kDQK * 2) + align256(t * topk * 4) + align256(t * h * smla::kDV * 2) +
           align256(t * h * 4);
}

smla_status sparse_mla_fwd_host(const void* q_host, const void* kv_cache, const int32_t* indices_host,
                                int32_t T, int32_t h, int32_t topk, int64_t num_slots,
                                int32_t kv_format, float scale, void* out_host, float* lse_host,
                                void* workspace, size_t workspace_bytes, void* stream) {
    if (T == 0) return check_args(q_host, kv_cache, indices_host, T, h, topk, num_slots, kv_format,
                                  scale, out_host, lse_host, 0);
    if (T < 0 || h <= 0 || topk <= 0)
        return check_args(q_host, kv_cache, indices_host, T, h, topk, num_slots, kv_format, scale,
                          out_host, lse_host, 0);
    if (!q_host || !indices_host || !out_host || !lse_host || !workspace)
        return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(workspace, 256)) return fail(SMLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t need = sparse_mla_host_workspace_bytes(T, h, topk);
    if (workspace_bytes < need)
        return fail(SMLA_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes, need);
    const size_t t = static_cast<size_t>(T);
    const size_t q_bytes = t * h * smla::kDQK * 2, i_bytes = t * topk * 4;
    const size_t o_bytes = t * h * smla::kDV * 2, l_bytes = t * h * 4;
    char* w = static_cast<char*>(workspace);
    void* q_dev = w;
    int32_t* i_dev = reinterpret_cast<int32_t*>(w + align256(q_bytes));
    void* o_dev = w + align256(q_bytes) + align256(i_bytes);
    float* l_dev = reinterpret_cast<float*>(w + align256(q_bytes) + align256(i_bytes) + align256(o_bytes));
    smla_status st = check_args(q_dev, kv_cache, i_dev, T, h, topk, num_slots, kv_format, scale, o_dev,
                                l_dev, 0);
    if (st != SMLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(q_dev, q_host, q_bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(i_dev, indices_host, i_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    st = launch(q_dev, kv_cache, i_dev, T, h, topk, num_slots, kv_format, scale, o_dev, l_dev, 0, s);
    if (st != SMLA_OK) return st;
    e = cudaMemcpyAsync(out_host, o_dev, o_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(lse_host, l_dev, l_bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    return SMLA_OK;
}

smla_status sparse_mla_host_io_layout(int32_t T, int32_t h, int32_t topk, size_t* in_bytes,
                                      size_t* indices_offset, size_t* out_bytes, size_t* lse_offset) {
    if (T < 0 || h <= 0 || topk <= 0)
        return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d h=%d topk=%d", T, h, topk);
    const size_t t = static_cast<size_t>(T);
    const size_t q_bytes = t * h * smla::kDQK * 2, i_bytes = t * topk * 4;
    const size_t o_bytes = t * h * smla::kDV * 2, l_bytes = t * h * 4;
    if (in_bytes) *in_bytes = T == 0 ? 0 : align256(q_bytes) + i_bytes;
    if (indices_offset) *indices_offset = align256(q_bytes);
    if (out_bytes) *out_bytes = T == 0 ? 0 : align256(o_bytes) + l_bytes;
    if (lse_offset) *lse_offset = align256(o_bytes);
    return SMLA_OK;
}

smla_status sparse_mla_fwd_host_packed(const void* in_host, const void* kv_cache, int32_t T, int32_t h,
                                       int32_t topk, int64_t num_slots, int32_t kv_format, float scale,
                                       void* out_host, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    if (T < 0 || h <= 0 || topk <= 0)
        return check_args(in_host, kv_cache, static_cast<const int32_t*>(in_host), T, h, topk, num_slots,
                          kv_format, scale, out_host, static_cast<const float*>(out_host), 0);
    if (T == 0)
        return check_args(nullptr, kv_cache, nullptr, 0, h, topk, num_slots, kv_format, scale, nullptr,
                          nullptr, 0);
    if (!in_host || !out_host || !workspace) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(workspace, 256)) return fail(SMLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const size_t need = sparse_mla_host_workspace_bytes(T, h, topk);
    if (workspace_bytes < need)
        return fail(SMLA_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes, need);
    size_t in_bytes = 0, i_off = 0, out_bytes = 0, l_off = 0;
    sparse_mla_host_io_layout(T, h, topk, &in_bytes, &i_off, &out_bytes, &l_off);
    const size_t t = static_cast<size_t>(T);
    const size_t o_off = i_off + align256(t * topk * 4);  // device: [q | idx | out | lse]
    char* w = static_cast<char*>(workspace);
    const int32_t* i_dev = reinterpret_cast<const int32_t*>(w + i_off);
    float* l_dev = reinterpret_cast<float*>(w + o_off + l_off);
    smla_status st = check_args(w, kv_cache, i_dev, T, h, topk, num_slots, kv_format, scale, w + o_off, l_dev, 0);
    if (st != SMLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(w, in_host, in_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    st = launch(w, kv_cache, i_dev, T, h, topk, num_slots, kv_format, scale, w + o_off, l_dev, 0, s);
    if (st != SMLA_OK) return st;
    e = cudaMemcpyAsync(out_host, w + o_off, out_bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
    return SMLA_OK;
}

smla_status sparse_mla_sync_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, smla::g_smla_error, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(smla::g_smla_error, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        if (word & smla::kErrTimeout) {
            // a launch gave up part-way: its grid-barrier words may be left mid-count, so every
            // library-owned scratch of this device starts again from cleared words
            int dev = 0;
            if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess) {
                std::lock_guard<std::mutex> lock(g_scratch_mu);
                for (Scratch& x : g_scratch)
                    if (x.dev == dev && x.ptr) cudaMemset(x.ptr, 0, kScratchHead);
                std::lock_guard<std::mutex> lock2(g_static_mu);
                if (dev >= 0 && dev < kMaxDevices && g_dev[dev].static_ptr)
                    cudaMemset(g_dev[dev].static_ptr, 0, kScratchHead);
            }
            return fail(SMLA_ERR_TIMEOUT, "a kernel gave up on a bounded wait (error word 0x%x%s)", word,
                        (word & smla::kErrIndexRange) ? "; a checked launch also met out-of-range list entries" : "");
        }
        if (word & smla::kErrLayout)
            return fail(SMLA_ERR_CUDA, "kernel reported an error (error word 0x%x)", word);
        return fail(SMLA_ERR_INDEX_RANGE,
                    "a checked launch met list entries other than -1 outside [0, num_slots); they were masked");
    }
    return SMLA_OK;
}

smla_status sparse_mla_launch_info(int32_t T, int32_t h, int32_t topk, int32_t kv_format,
                                   int32_t* splits, int32_t* ctas, int32_t* smem_bytes,
                                   int32_t* launches) {
    if (T < 0 || topk < 1) return fail(SMLA_ERR_INVALID_ARG, "bad T or topk");
    if (!(h == 8 || h == 16 || h == 32 || h == 64))
        return fail(SMLA_ERR_UNSUPPORTED, "h must be 8, 16, 32 or 64 (got %d)", h);
    if (kv_format != SMLA_KV_BF16 && kv_format != SMLA_KV_FP8)
        return fail(SMLA_ERR_INVALID_ARG, "unknown kv_format %d", kv_format);
    int num_sms = 152;
    int dev = 0;
    DeviceState* ds = nullptr;
    if (device_state(&dev, &ds) == SMLA_OK) num_sms = ds->num_sms;
    const Plan pl = make_plan(T, h, topk, 0, num_sms, kv_format == SMLA_KV_FP8);
    if (splits) *splits = pl.splits;
    if (ctas) *ctas = static_cast<int32_t>(pl.ctas);
    if (smem_bytes) *smem_bytes = pl.smem;
    if (launches) *launches = T > 0 ? 1 : 0;
    return SMLA_OK;
}

const char* sparse_mla_last_error(void) { return g_last_error; }

int32_t sparse_mla_version(void) { return kVersion; }


smla_status sparse_mla_merge(const void* o_parts, const float* lse_parts, int32_t n_parts, int32_t T,
                             int32_t h, void* out, float* lse, void* stream) {
    if (n_parts < 1 || n_parts > smla::kMergeMaxParts)
        return fail(SMLA_ERR_INVALID_ARG, "n_parts must be in [1, %d] (got %d)", smla::kMergeMaxParts, n_parts);
    if (T < 0 || h < 1) return fail(SMLA_ERR_INVALID_ARG, "T must be >= 0 and h >= 1 (got %d, %d)", T, h);
    if (T == 0) return SMLA_OK;
    if (!o_parts || !lse_parts || !out || !lse) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(o_parts, 16) || !aligned(out, 16))
        return fail(SMLA_ERR_INVALID_ARG, "o_parts and out must be 16-byte aligned");
    if (!aligned(lse_parts, 4) || !aligned(lse, 4))
        return fail(SMLA_ERR_INVALID_ARG, "lse_parts and lse must be 4-byte aligned");
    int dev = 0;
    DeviceState* ds = nullptr;
    smla_status st = device_state(&dev, &ds);
    if (st != SMLA_OK) return st;
    smla::MergeParams mp;
    mp.o_parts = static_cast<const __nv_bfloat16*>(o_parts);
    mp.lse_parts = lse_parts;
    mp.out = static_cast<__nv_bfloat16*>(out);
    mp.lse = lse;
    mp.rows = static_cast<int64_t>(T) * h;
    mp.n = n_parts;
    // one warp per row, eight rows per CTA; a grid of the CTAs that fit on the device at once
    // strides over the rows (their count is asked of the runtime once per device; threads
    // that race here ask twice and store the same value)
    static std::atomic<int> resident[kMaxDevices];
    int per_dev = resident[dev].load(std::memory_order_relaxed);
    if (per_dev == 0) {
        int per_sm = 0;
        const cudaError_t oe =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, smla::sparse_mla_merge_kernel, smla::kMergeThreads, 0);
        if (oe != cudaSuccess) return cuda_fail(oe, "occupancy of the merge kernel");
        per_dev = per_sm > 0 ? per_sm : 1;
        resident[dev].store(per_dev, std::memory_order_relaxed);
    }
    const int64_t want = (mp.rows + 7) / 8;
    const int64_t cap = static_cast<int64_t>(ds->num_sms) * per_dev;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap), 1, 1);
    cfg.blockDim = dim3(smla::kMergeThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_merge_kernel, mp);
    if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
    return SMLA_OK;
}


smla_status sparse_mla_v_up(const void* o, const void* w, int32_t T, int32_t h, int32_t v, void* y,
                            void* stream) {
    if (T < 0 || h < 1) return fail(SMLA_ERR_INVALID_ARG, "T must be >= 0 and h >= 1 (got %d, %d)", T, h);
    if (!(v == 128 || v == 256)) return fail(SMLA_ERR_UNSUPPORTED, "v must be 128 or 256 (got %d)", v);
    if (T == 0) return SMLA_OK;
    if (!o || !w || !y) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(o, 16) || !aligned(w, 16) || !aligned(y, 16))
        return fail(SMLA_ERR_INVALID_ARG, "o, w and y must be 16-byte aligned");
    if (static_cast<int64_t>(h) * v > 0x7fffffffLL || static_cast<int64_t>(T) * h > 0x7fffffffLL)
        return fail(SMLA_ERR_INVALID_ARG, "T * h or h * v too large (%d, %d, %d)", T, h, v);
    int dev = 0;
    DeviceState* ds = nullptr;
    smla_status st = device_state(&dev, &ds);
    if (st != SMLA_OK) return st;
    EncodeTiledFn enc = nullptr;
    if ((st = encode_fn(&enc)) != SMLA_OK) return st;
    // O [T, h, 512]: boxes of 128 tokens x 64 dims of one head; W [h, v, 512]: 128 outputs x 64 dims
    alignas(64) CUtensorMap tm_o;
    alignas(64) CUtensorMap tm_w;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(smla::kDV), static_cast<cuuint64_t>(h),
                                    static_cast<cuuint64_t>(T)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(smla::kDV) * 2,
                                       static_cast<cuuint64_t>(smla::kDV) * 2 * h};
        const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(smla::kVupRows)};
        const cuuint32_t es[3] = {1, 1, 1};
        CUresult r = enc(&tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(o), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(SMLA_ERR_CUDA, "tensor map for o failed (%d)", (int)r);
    }
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(smla::kDV), static_cast<cuuint64_t>(v),
                                    static_cast<cuuint64_t>(h)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(smla::kDV) * 2,
                                       static_cast<cuuint64_t>(smla::kDV) * 2 * v};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(smla::kVupN), 1};
        const cuuint32_t es[3] = {1, 1, 1};
        CUresult r = enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(SMLA_ERR_CUDA, "tensor map for w failed (%d)", (int)r);
    }
    smla::VupParams vp;
    vp.y = static_cast<__nv_bfloat16*>(y);
    vp.T = T;
    vp.h = h;
    vp.v = v;
    vp.mtiles = (T + smla::kVupRows - 1) / smla::kVupRows;
    // one CTA per SM: the (head, 128-output) slices share the SMs, each slice's token tiles
    // split evenly over its CTAs (at least one tile each)
    const int64_t slices = static_cast<int64_t>(h) * (v / smla::kVupN);
    int64_t cpg = slices >= ds->num_sms ? 1 : ds->num_sms / slices;
    if (cpg > vp.mtiles) cpg = vp.mtiles;
    vp.cpg = static_cast<int32_t>(cpg);
    const int64_t grid = slices * cpg;
    if (grid > 0x7fffffffLL) return fail(SMLA_ERR_INVALID_ARG, "grid too large");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(smla::kVupThreads, 1, 1);
    cfg.dynamicSmemBytes = smla::VupLayout::kBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_v_up_kernel, tm_o, tm_w, vp);
    if (e != cudaSuccess) return cuda_fail(e, "v_up kernel launch");
    return SMLA_OK;
}


smla_status sparse_mla_topk(const float* scores, int32_t T, int64_t S, const int32_t* lengths, int32_t topk,
                            const int32_t* block_table, int32_t* indices, void* stream) {
    if (T < 0 || S < 1 || topk < 1 || topk > (1 << 20) || S > 0x7fffffffLL)
        return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d S=%lld topk=%d", T, static_cast<long long>(S), topk);
    if (T == 0) return SMLA_OK;
    if (!scores || !lengths || !indices) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(scores, 4) || !aligned(lengths, 4) || !aligned(indices, 4) || !aligned(block_table, 4))
        return fail(SMLA_ERR_INVALID_ARG, "scores, lengths, block_table and indices must be 4-byte aligned");
    int dev = 0;
    DeviceState* ds = nullptr;
    smla_status st = device_state(&dev, &ds);
    if (st != SMLA_OK) return st;
    smla::TopkParams tp;
    tp.scores = scores;
    tp.len = lengths;
    tp.block_table = block_table;
    tp.out = indices;
    tp.S = S;
    tp.T = T;
    tp.topk = topk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(T), 1, 1);
    cfg.blockDim = dim3(smla::kTopkThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_topk_kernel, tp);
    if (e != cudaSuccess) return cuda_fail(e, "top-k kernel launch");
    return SMLA_OK;
}


smla_status sparse_mla_scatter_mask(const int32_t* indices, int32_t T, int32_t topk, int64_t S, uint32_t* mask,
                                    void* stream) {
    if (T < 0 || topk < 1 || S < 1 || S > smla::kScatterMaxS)
        return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d topk=%d S=%lld (S <= %d)", T, topk,
                    static_cast<long long>(S), smla::kScatterMaxS);
    if (T == 0) return SMLA_OK;
    if (!indices || !mask) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(indices, 4) || !aligned(mask, 16))
        return fail(SMLA_ERR_INVALID_ARG, "indices must be 4-byte and mask 16-byte aligned");
    int dev = 0;
    DeviceState* ds = nullptr;
    smla_status st = device_state(&dev, &ds);
    if (st != SMLA_OK) return st;
    smla::ScatterParams sp;
    sp.idx = indices;
    sp.mask = mask;
    sp.S = S;
    sp.T = T;
    sp.topk = topk;
    sp.W = static_cast<int32_t>((S + 31) / 32);
    const int64_t cap = static_cast<int64_t>(ds->num_sms) * 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(T < cap ? T : cap), 1, 1);
    cfg.blockDim = dim3(smla::kScatterThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(sp.W) * 4;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_scatter_mask_kernel, sp);
    if (e != cudaSuccess) return cuda_fail(e, "scatter kernel launch");
    return SMLA_OK;
}

smla_status sparse_mla_masked_mha(const void* q, const void* k, const void* v, const uint32_t* mask, int32_t T,
                                  int64_t S, int32_t h, int32_t dqk, int32_t dv, float scale, void* out, float* lse,
                                  void* stream) {
    if (T < 0 || S < 1 || S > smla::kMmMaxS || h < 1)
        return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d S=%lld h=%d (1 <= S <= %d)", T, static_cast<long long>(S), h,
                    smla::kMmMaxS);
    if (!((dqk == 192 || dqk == 256) && (dv == 128 || dv == 256)))
        return fail(SMLA_ERR_UNSUPPORTED, "head dims (q/k %d, v %d): q/k must be 192 or 256 and v 128 or 256", dqk, dv);
    if (!std::isfinite(scale)) return fail(SMLA_ERR_INVALID_ARG, "scale must be finite");
    if (T == 0) return SMLA_OK;
    if (!q || !k || !v || !mask || !out || !lse) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return fail(SMLA_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    if (!aligned(mask, 4) || !aligned(lse, 4)) return fail(SMLA_ERR_INVALID_ARG, "mask and lse must be 4-byte aligned");
    const int64_t nq = (static_cast<int64_t>(T) + smla::kMmBM - 1) / smla::kMmBM;
    if (nq * h > 0x7fffffffLL || static_cast<int64_t>(T) * h > 0x7fffffffLL)
        return fail(SMLA_ERR_INVALID_ARG, "T * h too large (%d, %d)", T, h);
    int dev = 0;
    DeviceState* ds = nullptr;
    smla_status st = device_state(&dev, &ds);
    if (st != SMLA_OK) return st;
    EncodeTiledFn enc = nullptr;
    if ((st = encode_fn(&enc)) != SMLA_OK) return st;
    alignas(64) CUtensorMap tm_q;
    alignas(64) CUtensorMap tm_k;
    alignas(64) CUtensorMap tm_v;
    alignas(64) CUtensorMap tm_o;
    // [rows, h, d] viewed as (64 elements, rows, h, d / 64 panels): one box of (64, box_rows, 1,
    // d / 64) lands as d / 64 SW128 panels of box_rows x 128 bytes, one after another
    auto make = [&](CUtensorMap* tm, const void* base, int d, int64_t rows, uint32_t box_rows) -> CUresult {
        const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(h),
                                    static_cast<cuuint64_t>(d / 64)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2 * h, static_cast<cuuint64_t>(d) * 2, 128};
        const cuuint32_t box[4] = {64, box_rows, 1, static_cast<cuuint32_t>(d / 64)};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    CUresult r = make(&tm_q, q, dqk, T, smla::kMmBM);
    if (r == CUDA_SUCCESS) r = make(&tm_k, k, dqk, S, smla::kMmBN);
    if (r == CUDA_SUCCESS) r = make(&tm_v, v, dv, S, smla::kMmBN);
    if (r == CUDA_SUCCESS) r = make(&tm_o, out, dv, T, smla::kMmBM);
    if (r != CUDA_SUCCESS) return fail(SMLA_ERR_CUDA, "tensor maps for q/k/v/out failed (%d)", (int)r);
    smla::MmParams mp;
    mp.out = static_cast<__nv_bfloat16*>(out);
    mp.lse = lse;
    mp.mask = mask;
    mp.S = S;
    mp.T = T;
    mp.h = h;
    mp.W = static_cast<int32_t>((S + 31) / 32);
    mp.nq = static_cast<int32_t>(nq);
    mp.sm_scale_log2 = scale * 1.4426950408889634f;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nq * h), 1, 1);
    cfg.blockDim = dim3(smla::kMmThreads, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (dqk == 192 && dv == 128) {
        cfg.dynamicSmemBytes = smla::MmLayout<192, 128>::kBytes;
        e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_masked_mha_kernel<192, 128>, tm_q, tm_k, tm_v, tm_o, mp);
    } else if (dqk == 192) {
        cfg.dynamicSmemBytes = smla::MmLayout<192, 256>::kBytes;
        e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_masked_mha_kernel<192, 256>, tm_q, tm_k, tm_v, tm_o, mp);
    } else if (dv == 128) {
        cfg.dynamicSmemBytes = smla::MmLayout<256, 128>::kBytes;
        e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_masked_mha_kernel<256, 128>, tm_q, tm_k, tm_v, tm_o, mp);
    } else {
        cfg.dynamicSmemBytes = smla::MmLayout<256, 256>::kBytes;
        e = cudaLaunchKernelEx(&cfg, smla::sparse_mla_masked_mha_kernel<256, 256>, tm_q, tm_k, tm_v, tm_o, mp);
    }
    if (e != cudaSuccess) return cuda_fail(e, "masked MHA kernel launch");
    return SMLA_OK;
}

}  // extern "C"
