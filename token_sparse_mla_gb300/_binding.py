"""ctypes binding of libsparse_mla.so (argument marshalling only)."""

import contextlib
import ctypes
import functools
from pathlib import Path
from typing import Optional, Tuple

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libsparse_mla.so"
_lib = None

KV_FORMATS = {"bf16": 0, "fp8": 1}
D_QK, D_V, FP8_ROW_BYTES = 576, 512, 656

_STATUS = {0: "SMLA_OK", 1: "SMLA_ERR_INVALID_ARG", 2: "SMLA_ERR_UNSUPPORTED",
           3: "SMLA_ERR_CUDA", 4: "SMLA_ERR_TIMEOUT", 5: "SMLA_ERR_INDEX_RANGE"}
SMLA_ERR_INDEX_RANGE = 5

EXPORTED = ("sparse_mla_fwd", "sparse_mla_fwd_ex", "sparse_mla_fwd_checked", "sparse_mla_fwd_noalloc",
            "sparse_mla_fwd_host", "sparse_mla_fwd_host_packed", "sparse_mla_host_io_layout",
            "sparse_mla_host_workspace_bytes", "sparse_mla_merge",
            "sparse_mla_v_up", "sparse_mla_topk", "sparse_mla_scatter_mask", "sparse_mla_masked_mha",
            "sparse_mla_sync_status",
            "sparse_mla_launch_info", "sparse_mla_last_error", "sparse_mla_version")


class SparseMLAError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{_STATUS.get(status, status)}: {message}")


def lib_path() -> Path:
    return _LIB_PATH


def library() -> ctypes.CDLL:
    """Load libsparse_mla.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not _LIB_PATH.exists():
        raise ImportError(f"{_LIB_PATH} is missing: build it with "
                          "`python -m token_sparse_mla_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(str(_LIB_PATH))
    vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
    lib.sparse_mla_fwd.restype = ctypes.c_int
    lib.sparse_mla_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, f32, vp, vp, vp]
    lib.sparse_mla_fwd_ex.restype = ctypes.c_int
    lib.sparse_mla_fwd_ex.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, f32, vp, vp, i32, vp]
    lib.sparse_mla_fwd_checked.restype = ctypes.c_int
    lib.sparse_mla_fwd_checked.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, f32, vp, vp, i32, vp]
    lib.sparse_mla_fwd_noalloc.restype = ctypes.c_int
    lib.sparse_mla_fwd_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, f32, vp, vp, i32, vp]
    lib.sparse_mla_topk.restype = ctypes.c_int
    lib.sparse_mla_topk.argtypes = [vp, i32, i64, vp, i32, vp, vp, vp]
    lib.sparse_mla_v_up.restype = ctypes.c_int
    lib.sparse_mla_v_up.argtypes = [vp, vp, i32, i32, i32, vp, vp]
    lib.sparse_mla_merge.restype = ctypes.c_int
    lib.sparse_mla_merge.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    lib.sparse_mla_host_workspace_bytes.restype = sz
    lib.sparse_mla_host_workspace_bytes.argtypes = [i32, i32, i32]
    lib.sparse_mla_fwd_host.restype = ctypes.c_int
    lib.sparse_mla_fwd_host.argtypes = [vp, vp, vp, i32, i32, i32, i64, i32, f32, vp, vp, vp, sz, vp]
    lib.sparse_mla_scatter_mask.restype = ctypes.c_int
    lib.sparse_mla_scatter_mask.argtypes = [vp, i32, i32, i64, vp, vp]
    lib.sparse_mla_masked_mha.restype = ctypes.c_int
    lib.sparse_mla_masked_mha.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, f32, vp, vp, vp]
    lib.sparse_mla_host_io_layout.restype = ctypes.c_int
    lib.sparse_mla_host_io_layout.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    lib.sparse_mla_fwd_host_packed.restype = ctypes.c_int
    lib.sparse_mla_fwd_host_packed.argtypes = [vp, vp, i32, i32, i32, i64, i32, f32, vp, vp, sz, vp]
    lib.sparse_mla_sync_status.restype = ctypes.c_int
    lib.sparse_mla_sync_status.argtypes = [vp]
    lib.sparse_mla_launch_info.restype = ctypes.c_int
    lib.sparse_mla_launch_info.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
    lib.sparse_mla_last_error.restype = ctypes.c_char_p
    lib.sparse_mla_last_error.argtypes = []
    lib.sparse_mla_version.restype = ctypes.c_int32
    lib.sparse_mla_version.argtypes = []
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        msg = library().sparse_mla_last_error().decode(errors="replace")
        raise SparseMLAError(status, msg)


def _device_of(tensors) -> torch.device:
    """The one CUDA device that all (name, tensor) pairs live on; raises if there is none."""
    dev = None
    for name, t in tensors:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other tensors on {dev}")
    return dev


def _on(dev: torch.device):
    """Context that makes `dev` the current device: a no-op when it already is (entering
    torch.cuda.device costs several microseconds a call, a sizeable share of a decode step)."""
    return contextlib.nullcontext() if torch.cuda.current_device() == dev.index else torch.cuda.device(dev)


def _stream_handle(stream, device: Optional[torch.device] = None) -> Optional[int]:
    """Raw handle of `stream` (default: the current stream of `device`, else of the current
    device).  A stream object must belong to `device`; a raw int handle is passed as is."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return stream
    if device is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return stream.cuda_stream


def version() -> int:
    return int(library().sparse_mla_version())


def _dims(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor, kv_format: str):
    if q.dim() != 3 or q.shape[2] != D_QK or q.dtype != torch.bfloat16:
        raise ValueError(f"q must be [T, h, 576] bf16, got {tuple(q.shape)} {q.dtype}")
    T, h = int(q.shape[0]), int(q.shape[1])
    if indices.dim() != 2 or indices.shape[0] != T or indices.dtype != torch.int32:
        raise ValueError(f"indices must be [T, topk] int32, got {tuple(indices.shape)} {indices.dtype}")
    if kv_format not in KV_FORMATS:
        raise ValueError(f"kv_format must be one of {sorted(KV_FORMATS)}")
    if kv_format == "bf16":
        if kv_cache.dim() != 2 or kv_cache.shape[1] != D_QK or kv_cache.dtype != torch.bfloat16:
            raise ValueError(f"bf16 kv_cache must be [num_slots, 576] bf16, got "
                             f"{tuple(kv_cache.shape)} {kv_cache.dtype}")
    else:
        if kv_cache.dim() != 2 or kv_cache.shape[1] != FP8_ROW_BYTES or kv_cache.dtype != torch.uint8:
            raise ValueError(f"fp8 kv_cache must be [num_slots, 656] uint8, got "
                             f"{tuple(kv_cache.shape)} {kv_cache.dtype}")
    for name, t in (("q", q), ("kv_cache", kv_cache), ("indices", indices)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    return T, h, int(indices.shape[1]), int(kv_cache.shape[0])


def sparse_mla_fwd(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                   scale: Optional[float] = None, *, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, kv_format: str = "bf16",
                   splits: int = 0, checked: bool = False,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Token-sparse MLA forward on the GPU (see include/sparse_mla.h).

    scale defaults to 576 ** -0.5.  out / lse may be passed in (caller-owned
    buffers, [T, h, 512] bf16 and [T, h] fp32); otherwise they are allocated
    here.  splits = 0 lets the library choose how many CTAs share a token's
    list.  checked = True runs sparse_mla_fwd_checked: the same outputs, and list
    entries other than -1 outside [0, num_slots) make the next sync_status()
    raise SMLA_ERR_INDEX_RANGE.  Runs asynchronously on `stream` (default:
    torch's current stream).
    """
    T, h, topk, num_slots = _dims(q, kv_cache, indices, kv_format)
    dev = _device_of((("q", q), ("kv_cache", kv_cache), ("indices", indices)))
    if scale is None:
        scale = D_QK ** -0.5
    if out is None:
        out = torch.empty((T, h, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, h), dtype=torch.float32, device=dev)
    if out.shape != (T, h, D_V) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [T, h, 512] bf16 tensor")
    if lse.shape != (T, h) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [T, h] fp32 tensor")
    _device_of((("q", q), ("out", out), ("lse", lse)))
    with _on(dev):
        lib = library()
        fn = lib.sparse_mla_fwd_checked if checked else lib.sparse_mla_fwd_ex
        st = fn(
            q.data_ptr(), kv_cache.data_ptr(), indices.data_ptr(), T, h, topk, num_slots,
            KV_FORMATS[kv_format], float(scale), out.data_ptr(), lse.data_ptr(), int(splits),
            _stream_handle(stream, dev))
    _check(st)
    return out, lse


def sparse_mla_fwd_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                           scale: Optional[float] = None, *, out: torch.Tensor, lse: torch.Tensor,
                           kv_format: str = "bf16", splits: int = 0, stream=None) -> None:
    """sparse_mla_fwd with the library's static merge scratch: nothing is allocated, so out and
    lse are required (see include/sparse_mla.h for the rules on first call and streams)."""
    T, h, topk, num_slots = _dims(q, kv_cache, indices, kv_format)
    dev = _device_of((("q", q), ("kv_cache", kv_cache), ("indices", indices), ("out", out),
                      ("lse", lse)))
    if scale is None:
        scale = D_QK ** -0.5
    if out.shape != (T, h, D_V) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [T, h, 512] bf16 tensor")
    if lse.shape != (T, h) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [T, h] fp32 tensor")
    with _on(dev):
        st = library().sparse_mla_fwd_noalloc(
            q.data_ptr(), kv_cache.data_ptr(), indices.data_ptr(), T, h, topk, num_slots,
            KV_FORMATS[kv_format], float(scale), out.data_ptr(), lse.data_ptr(), int(splits),
            _stream_handle(stream, dev))
    _check(st)


def sparse_mla_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, *,
                     out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Merge the partial results of split token lists (the DCP merge; include/sparse_mla.h).

    o_parts [n, T, h, 512] bf16 and lse_parts [n, T, h] fp32 are what sparse_mla_fwd returned
    for each of the n parts (LSE -inf = empty part); returns out [T, h, 512] bf16 and
    lse [T, h] fp32 of the whole lists.
    """
    if o_parts.dim() != 4 or o_parts.shape[-1] != D_V or o_parts.dtype != torch.bfloat16:
        raise ValueError("o_parts must be [n, T, h, 512] bf16")
    n, T, h = int(o_parts.shape[0]), int(o_parts.shape[1]), int(o_parts.shape[2])
    if lse_parts.shape != (n, T, h) or lse_parts.dtype != torch.float32:
        raise ValueError("lse_parts must be [n, T, h] fp32")
    dev = _device_of((("o_parts", o_parts), ("lse_parts", lse_parts)))
    for name, t in (("o_parts", o_parts), ("lse_parts", lse_parts)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty((T, h, D_V), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, h), dtype=torch.float32, device=dev)
    if out.shape != (T, h, D_V) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [T, h, 512] bf16 tensor")
    if lse.shape != (T, h) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [T, h] fp32 tensor")
    _device_of((("o_parts", o_parts), ("out", out), ("lse", lse)))
    with _on(dev):
        st = library().sparse_mla_merge(o_parts.data_ptr(), lse_parts.data_ptr(), n, T, h,
                                        out.data_ptr(), lse.data_ptr(), _stream_handle(stream, dev))
    _check(st)
    return out, lse


def sparse_mla_v_up(o: torch.Tensor, w: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """The v_up projection of the attention output on the tensor cores (include/sparse_mla.h):
    y[t, h, n] = sum_k o[t, h, k] * w[h, n, k], o [T, h, 512] bf16, w [h, v, 512] bf16
    (v = 128 or 256); returns y [T, h, v] bf16."""
    if o.dim() != 3 or o.shape[-1] != D_V or o.dtype != torch.bfloat16:
        raise ValueError("o must be [T, h, 512] bf16")
    T, h = int(o.shape[0]), int(o.shape[1])
    if w.dim() != 3 or w.shape[0] != h or w.shape[2] != D_V or w.dtype != torch.bfloat16:
        raise ValueError("w must be [h, v, 512] bf16")
    v = int(w.shape[1])
    dev = _device_of((("o", o), ("w", w)))
    for name, t in (("o", o), ("w", w)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty((T, h, v), dtype=torch.bfloat16, device=dev)
    if out.shape != (T, h, v) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [T, h, v] bf16 tensor")
    _device_of((("o", o), ("out", out)))
    with _on(dev):
        st = library().sparse_mla_v_up(o.data_ptr(), w.data_ptr(), T, h, v, out.data_ptr(),
                                       _stream_handle(stream, dev))
    _check(st)
    return out


def sparse_mla_topk(scores: torch.Tensor, lengths: torch.Tensor, topk: int, *,
                    block_table: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """Index lists from per-position scores (include/sparse_mla.h): the top `topk` positions of
    scores[t, :lengths[t]] (ties to the lower position), ascending, mapped through block_table
    (64-slot blocks) when given, -1 padded.  scores [T, S] fp32, lengths [T] int32."""
    if scores.dim() != 2 or scores.dtype != torch.float32:
        raise ValueError("scores must be [T, S] fp32")
    T, S = int(scores.shape[0]), int(scores.shape[1])
    if lengths.shape != (T,) or lengths.dtype != torch.int32:
        raise ValueError("lengths must be [T] int32")
    tensors = [("scores", scores), ("lengths", lengths)]
    if block_table is not None:
        if block_table.dim() != 1 or block_table.dtype != torch.int32 or block_table.numel() * 64 < S:
            raise ValueError("block_table must be [ceil(S / 64)] int32")
        tensors.append(("block_table", block_table))
    dev = _device_of(tensors)
    for name, t in tensors:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty((T, topk), dtype=torch.int32, device=dev)
    if out.shape != (T, topk) or out.dtype != torch.int32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [T, topk] int32 tensor")
    _device_of((("scores", scores), ("out", out)))
    with _on(dev):
        st = library().sparse_mla_topk(scores.data_ptr(), T, S, lengths.data_ptr(), int(topk),
                                       None if block_table is None else block_table.data_ptr(),
                                       out.data_ptr(), _stream_handle(stream, dev))
    _check(st)
    return out


def sparse_mla_scatter_mask(indices: torch.Tensor, S: int, *, out: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """The lists of one request as a bit mask (include/sparse_mla.h): indices [T, topk] int32
    positions; returns mask [T, ceil(S / 32)] int32 whose bit s % 32 of word s / 32 is set iff s
    is listed (the words are uint32 bit patterns, held in an int32 tensor)."""
    if indices.dim() != 2 or indices.dtype != torch.int32:
        raise ValueError("indices must be [T, topk] int32")
    T, topk = int(indices.shape[0]), int(indices.shape[1])
    W = (int(S) + 31) // 32
    dev = _device_of((("indices", indices),))
    if not indices.is_contiguous():
        raise ValueError("indices must be contiguous")
    if out is None:
        out = torch.empty((T, W), dtype=torch.int32, device=dev)
    if out.shape != (T, W) or out.dtype != torch.int32 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous [T, {W}] int32 tensor")
    _device_of((("indices", indices), ("out", out)))
    with _on(dev):
        st = library().sparse_mla_scatter_mask(indices.data_ptr(), T, topk, int(S), out.data_ptr(),
                                               _stream_handle(stream, dev))
    _check(st)
    return out


def sparse_mla_masked_mha(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor,
                          scale: float, *, out: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Masked dense MHA (include/sparse_mla.h): q [T, h, dqk], k [S, h, dqk], v [S, h, dv] bf16,
    mask [T, ceil(S / 32)] int32 bit words; returns out [T, h, dv] bf16 and lse [T, h] fp32."""
    if q.dim() != 3 or q.dtype != torch.bfloat16:
        raise ValueError("q must be [T, h, dqk] bf16")
    T, h, dqk = (int(x) for x in q.shape)
    if k.dim() != 3 or k.dtype != torch.bfloat16 or k.shape[1] != h or k.shape[2] != dqk:
        raise ValueError("k must be [S, h, dqk] bf16")
    S = int(k.shape[0])
    if v.dim() != 3 or v.dtype != torch.bfloat16 or v.shape[0] != S or v.shape[1] != h:
        raise ValueError("v must be [S, h, dv] bf16")
    dv = int(v.shape[2])
    W = (S + 31) // 32
    if mask.shape != (T, W) or mask.dtype != torch.int32:
        raise ValueError(f"mask must be [T, {W}] int32")
    tensors = (("q", q), ("k", k), ("v", v), ("mask", mask))
    dev = _device_of(tensors)
    for name, t in tensors:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty((T, h, dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, h), dtype=torch.float32, device=dev)
    if out.shape != (T, h, dv) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous [T, h, {dv}] bf16 tensor")
    if lse.shape != (T, h) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [T, h] fp32 tensor")
    _device_of((("q", q), ("out", out), ("lse", lse)))
    with _on(dev):
        st = library().sparse_mla_masked_mha(q.data_ptr(), k.data_ptr(), v.data_ptr(), mask.data_ptr(), T, S, h,
                                             dqk, dv, float(scale), out.data_ptr(), lse.data_ptr(),
                                             _stream_handle(stream, dev))
    _check(st)
    return out, lse


def host_workspace_bytes(T: int, h: int, topk: int) -> int:
    return int(library().sparse_mla_host_workspace_bytes(T, h, topk))


def sparse_mla_fwd_host(q_host: torch.Tensor, kv_cache: torch.Tensor, indices_host: torch.Tensor,
                        scale: float, out_host: torch.Tensor, lse_host: torch.Tensor,
                        workspace: torch.Tensor, *, kv_format: str = "bf16", stream=None) -> None:
    """Forward pass with host-resident q/indices/out/lse (pinned for async copies);
    the library queues H2D copies, the kernel and D2H copies on `stream`."""
    T, h, topk, num_slots = _dims(q_host, kv_cache, indices_host, kv_format)
    if q_host.is_cuda or indices_host.is_cuda or out_host.is_cuda or lse_host.is_cuda:
        raise ValueError("q, indices, out and lse must be host tensors here")
    dev = _device_of((("kv_cache", kv_cache), ("workspace", workspace)))
    with _on(dev):
        st = library().sparse_mla_fwd_host(
            q_host.data_ptr(), kv_cache.data_ptr(), indices_host.data_ptr(), T, h, topk,
            num_slots, KV_FORMATS[kv_format], float(scale), out_host.data_ptr(),
            lse_host.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_handle(stream, dev))
    _check(st)


@functools.lru_cache(maxsize=256)
def _host_io_layout(T: int, h: int, topk: int) -> Tuple[int, int, int, int]:
    a, b, c, d = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(library().sparse_mla_host_io_layout(T, h, topk, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                               ctypes.byref(d)))
    return a.value, b.value, c.value, d.value


def host_io_layout(T: int, h: int, topk: int) -> dict:
    """Sizes and offsets of the packed host buffers of sparse_mla_fwd_host_packed (the library's
    answer, asked once per shape)."""
    a, b, c, d = _host_io_layout(int(T), int(h), int(topk))
    return {"in_bytes": a, "indices_offset": b, "out_bytes": c, "lse_offset": d}


def host_io_views(in_host: torch.Tensor, out_host: torch.Tensor, T: int, h: int, topk: int):
    """Views of q / indices inside a packed input buffer and of out / lse inside a packed output
    buffer (uint8 host tensors of the sizes host_io_layout gives)."""
    lay = host_io_layout(T, h, topk)
    if in_host.dtype != torch.uint8 or in_host.numel() < lay["in_bytes"]:
        raise ValueError(f"in_host must be a uint8 tensor of at least {lay['in_bytes']} bytes")
    if out_host.dtype != torch.uint8 or out_host.numel() < lay["out_bytes"]:
        raise ValueError(f"out_host must be a uint8 tensor of at least {lay['out_bytes']} bytes")
    i0, l0 = lay["indices_offset"], lay["lse_offset"]
    q = in_host[: T * h * D_QK * 2].view(torch.bfloat16).view(T, h, D_QK)
    idx = in_host[i0: i0 + T * topk * 4].view(torch.int32).view(T, topk)
    out = out_host[: T * h * D_V * 2].view(torch.bfloat16).view(T, h, D_V)
    lse = out_host[l0: l0 + T * h * 4].view(torch.float32).view(T, h)
    return q, idx, out, lse


def sparse_mla_fwd_host_packed(in_host: torch.Tensor, kv_cache: torch.Tensor, T: int, h: int, topk: int,
                               scale: float, out_host: torch.Tensor, workspace: torch.Tensor, *,
                               kv_format: str = "bf16", stream=None) -> None:
    """Forward pass from one packed host input buffer into one packed host output buffer
    (include/sparse_mla.h): one H2D copy, the kernel and one D2H copy queued on `stream`."""
    if in_host.is_cuda or out_host.is_cuda:
        raise ValueError("in_host and out_host must be host tensors")
    for name, t in (("in_host", in_host), ("out_host", out_host)):
        if t.dtype != torch.uint8 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous uint8 tensor")
    if kv_format not in KV_FORMATS:
        raise ValueError(f"kv_format must be one of {sorted(KV_FORMATS)}")
    in_bytes, _, out_bytes, _ = _host_io_layout(int(T), int(h), int(topk))
    if in_host.numel() < in_bytes or out_host.numel() < out_bytes:
        raise ValueError("in_host / out_host smaller than host_io_layout says")
    dev = _device_of((("kv_cache", kv_cache), ("workspace", workspace)))
    with _on(dev):
        st = library().sparse_mla_fwd_host_packed(
            in_host.data_ptr(), kv_cache.data_ptr(), T, h, topk, int(kv_cache.shape[0]),
            KV_FORMATS[kv_format], float(scale), out_host.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    _check(st)


def sync_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel reported a device-side error."""
    _check(library().sparse_mla_sync_status(_stream_handle(stream)))


def launch_info(T: int, h: int, topk: int, kv_format: str = "bf16") -> dict:
    s, c, m, n = (ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32())
    _check(library().sparse_mla_launch_info(T, h, topk, KV_FORMATS[kv_format], ctypes.byref(s),
                                            ctypes.byref(c), ctypes.byref(m), ctypes.byref(n)))
    return {"splits": s.value, "ctas": c.value, "smem_bytes": m.value, "launches": n.value}
