"""CPU oracle for the token-sparse MLA forward (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
may import this package.  The product path (token_sparse_mla_gb300) never loads
it, and it never loads the product path: the two share no code.

The arithmetic lives in sparse_mla_oracle.c (plain C, fp64, OpenMP over
(token, head) pairs); this module compiles it with gcc and marshals arrays.
See the C file's header for the definition it computes and the passages it
follows.
"""

import ctypes
import os
import subprocess
from pathlib import Path
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "sparse_mla_oracle.c"
_LIB_PATH = _HERE / "liboracle_smla.so"
_lib = None

KV_FORMATS = {"bf16": 0, "fp8": 1}


def build(force: bool = False) -> Path:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-o", str(tmp), str(_SRC), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        lib.oracle_sparse_mla_fwd.restype = ctypes.c_int
        lib.oracle_sparse_mla_fwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_e4m3_table.restype = None
        lib.oracle_e4m3_table.argtypes = [ctypes.c_void_p]
        lib.oracle_bf16_value.restype = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_row.restype = None
        lib.oracle_decode_row.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_void_p]
        lib.oracle_merge.restype = ctypes.c_int
        lib.oracle_merge.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                     ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_v_up.restype = ctypes.c_int
        lib.oracle_v_up.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_void_p]
        lib.oracle_topk.restype = ctypes.c_int
        lib.oracle_topk.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                    ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_scatter_mask.restype = ctypes.c_int
        lib.oracle_scatter_mask.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_int64, ctypes.c_void_p]
        lib.oracle_masked_mha.restype = ctypes.c_int
        lib.oracle_masked_mha.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        _lib = lib
    return _lib


def _as_np(x, dtype=None) -> np.ndarray:
    """torch CPU tensor or numpy array -> C-contiguous numpy array (bf16 as uint16 bits)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16)
            x = x.numpy()
    except ImportError:
        pass
    a = np.ascontiguousarray(x)
    if dtype is not None:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def sparse_mla_fwd(q, kv, indices, scale: float, kv_format: str = "bf16",
                   tokens: Optional[Sequence[int]] = None,
                   threads: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Exact sparse MLA forward in fp64.

    q        [T, h, 576] bf16 (torch bf16 tensor, or uint16 bit patterns)
    kv       bf16 [num_slots, 576], or uint8 [num_slots, 656] fp8 rows
    indices  [T, topk] int32
    tokens   optional token ids to evaluate (default: all)
    returns  out [n, h, 512] float64 and lse [n, h] float64 (n = len(tokens) or T)
    """
    lib = _load()
    qn = _as_np(q, np.uint16)
    kvn = _as_np(kv, np.uint16 if kv_format == "bf16" else np.uint8)
    idn = _as_np(indices, np.int32)
    T, h, d = qn.shape
    assert d == 576, qn.shape
    topk = idn.shape[1]
    assert idn.shape[0] == T
    num_slots = kvn.shape[0]
    if kv_format == "bf16":
        assert kvn.shape[1] == 576
    else:
        assert kvn.shape[1] == 656
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        n = tok.shape[0]
    out = np.empty((n, h, 512), dtype=np.float64)
    lse = np.empty((n, h), dtype=np.float64)
    rc = lib.oracle_sparse_mla_fwd(
        qn.ctypes.data, kvn.ctypes.data, KV_FORMATS[kv_format], idn.ctypes.data,
        T, h, topk, num_slots, float(scale),
        None if tok is None else tok.ctypes.data, n,
        out.ctypes.data, lse.ctypes.data, int(threads or 0))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out, lse


def e4m3_table() -> np.ndarray:
    t = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(t.ctypes.data)
    return t


def bf16_value(bits: int) -> float:
    return float(_load().oracle_bf16_value(int(bits) & 0xFFFF))


def decode_row(kv, kv_format: str, slot: int) -> np.ndarray:
    kvn = _as_np(kv, np.uint16 if kv_format == "bf16" else np.uint8)
    assert 0 <= slot < kvn.shape[0]
    row = np.empty(576, dtype=np.float64)
    _load().oracle_decode_row(kvn.ctypes.data, KV_FORMATS[kv_format], int(slot),
                              row.ctypes.data)
    return row


def merge(o_parts, lse_parts) -> Tuple[np.ndarray, np.ndarray]:
    """Exact merge of the partial results of a split list (the C file's oracle_merge), fp64.

    o_parts    [n, ..., 512]: a torch bf16 tensor (or uint16 bf16 bit patterns), or fp64 values
    lse_parts  [n, ...] natural-log LSE of each part (-inf = empty part), any float type
    returns    out [..., 512] float64 and lse [...] float64
    """
    lib = _load()
    ln = np.ascontiguousarray(_as_np(lse_parts).astype(np.float64))
    n = ln.shape[0]
    lead = ln.shape[1:]
    rows = int(np.prod(lead)) if len(lead) else 1
    on = _as_np(o_parts)
    if on.dtype == np.uint16 or on.dtype == np.int16:
        on, bf16 = np.ascontiguousarray(on.view(np.uint16)), 1
    else:
        on, bf16 = np.ascontiguousarray(on.astype(np.float64)), 0
    assert on.shape == (n,) + tuple(lead) + (512,), (on.shape, ln.shape)
    out = np.empty(tuple(lead) + (512,), dtype=np.float64)
    lse = np.empty(lead, dtype=np.float64)
    rc = lib.oracle_merge(on.ctypes.data, bf16, ln.ctypes.data, n, rows, out.ctypes.data,
                          lse.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out, lse


def v_up(o, w) -> np.ndarray:
    """The v_up projection (the C file's oracle_v_up), fp64.

    o  [T, h, 512] bf16 (torch bf16 tensor or uint16 bit patterns)
    w  [h, v, 512] bf16
    returns y [T, h, v] float64
    """
    lib = _load()
    on = _as_np(o, np.uint16)
    wn = _as_np(w, np.uint16)
    T, h, d = on.shape
    hw, v, dw = wn.shape
    assert d == 512 and dw == 512 and hw == h, (on.shape, wn.shape)
    y = np.empty((T, h, v), dtype=np.float64)
    rc = lib.oracle_v_up(on.ctypes.data, wn.ctypes.data, T, h, v, y.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return y


def topk(scores, lengths, k: int, block_table=None) -> np.ndarray:
    """Top-k index lists from scores (the C file's oracle_topk).

    scores [T, S] fp32, lengths [T] int32 (the causal history of each row), block_table
    optional [ceil(S / 64)] int32; returns [T, k] int32: selected slots (positions when no
    table) in ascending position order, -1 padding.
    """
    lib = _load()
    sn = np.ascontiguousarray(_as_np(scores).astype(np.float32))
    ln = np.ascontiguousarray(_as_np(lengths).astype(np.int32))
    T, S = sn.shape
    assert ln.shape == (T,)
    bt = None if block_table is None else np.ascontiguousarray(_as_np(block_table).astype(np.int32))
    out = np.empty((T, k), dtype=np.int32)
    rc = lib.oracle_topk(sn.ctypes.data, T, S, ln.ctypes.data, int(k),
                         None if bt is None else bt.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out


def _as_f64(x) -> np.ndarray:
    """torch tensor (any float dtype, bf16 included) or float array -> C-contiguous float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().cpu().double().numpy())  # exact widening
    except ImportError:
        pass
    a = np.asarray(x)
    assert a.dtype.kind == "f", a.dtype
    return np.ascontiguousarray(a.astype(np.float64))


def scatter_mask(indices, S: int) -> np.ndarray:
    """The lists scattered to a bit mask (the C file's oracle_scatter_mask).

    indices [T, topk] int32 positions in [0, S) (-1 and other values outside it set nothing);
    returns [T, ceil(S / 32)] uint32: bit s % 32 of word s // 32 is set iff s is listed.
    """
    lib = _load()
    idn = np.ascontiguousarray(_as_np(indices).astype(np.int32))
    T, k = idn.shape
    mask = np.empty((T, (int(S) + 31) // 32), dtype=np.uint32)
    rc = lib.oracle_scatter_mask(idn.ctypes.data, T, k, int(S), mask.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return mask


def masked_mha(q, k, v, mask, scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Masked dense MHA over per-head K and V (the C file's oracle_masked_mha), fp64.

    q [T, h, dqk], k [S, h, dqk], v [S, h, dv]: torch tensors (bf16 included) or float arrays;
    mask [T, ceil(S / 32)] uint32 bits as scatter_mask returns them.
    returns out [T, h, dv] float64 and lse [T, h] float64 (natural log; -inf for an empty row)
    """
    lib = _load()
    qn, kn, vn = _as_f64(q), _as_f64(k), _as_f64(v)
    T, h, dqk = qn.shape
    S = kn.shape[0]
    dv = vn.shape[2]
    assert kn.shape == (S, h, dqk) and vn.shape == (S, h, dv), (qn.shape, kn.shape, vn.shape)
    mn = np.ascontiguousarray(np.asarray(mask, dtype=np.uint32))
    assert mn.shape == (T, (S + 31) // 32), mn.shape
    out = np.empty((T, h, dv), dtype=np.float64)
    lse = np.empty((T, h), dtype=np.float64)
    rc = lib.oracle_masked_mha(qn.ctypes.data, kn.ctypes.data, vn.ctypes.data, mn.ctypes.data,
                               T, S, h, dqk, dv, float(scale), out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out, lse
