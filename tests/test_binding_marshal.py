"""The Python binding's argument marshalling, on the CPU.

Each wrapper is driven to its C-ABI call with stand-ins: CPU tensors that report a CUDA
device, a device guard and a current stream that only record what they are given, and a
library object that records its calls.  The checks: every wrapper passes the right pointers,
sizes and stream handle in the order include/sparse_mla.h declares, runs the call under a
guard for the tensors' device (entered only when another device is current), and rejects
tensors (or a stream) on another device, or a host tensor where device memory is expected,
before anything reaches the library.
"""

from types import SimpleNamespace

import pytest
import torch

import token_sparse_mla_gb300 as smla
from token_sparse_mla_gb300 import _binding

STREAM = 0xABC0


class _OnDevice:
    """A CPU tensor that reports itself as living on CUDA device `index`."""

    def __init__(self, t: torch.Tensor, index: int = 0):
        self._t = t
        self.is_cuda = True
        self.device = torch.device("cuda", index)

    def __getattr__(self, name):
        return getattr(self._t, name)


class _FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    lib = _FakeLib()
    entered = []

    class _Guard:
        def __init__(self, dev):
            self.dev = dev

        def __enter__(self):
            entered.append(self.dev)

        def __exit__(self, *exc):
            return False

    current = {"index": 1}  # another device is current: every call enters the guard
    monkeypatch.setattr(_binding, "library", lambda: lib)
    monkeypatch.setattr(torch.cuda, "device", _Guard)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: current["index"])
    monkeypatch.setattr(torch.cuda, "current_stream",
                        lambda device=None: SimpleNamespace(device=device, cuda_stream=STREAM))
    return SimpleNamespace(lib=lib, entered=entered, current=current)


def _d(shape, dtype, index=0):
    return _OnDevice(torch.zeros(shape, dtype=dtype), index)


def _fwd_args(T=3, h=8, topk=64, slots=100):
    return (_d((T, h, 576), torch.bfloat16), _d((slots, 576), torch.bfloat16),
            _d((T, topk), torch.int32), _d((T, h, 512), torch.bfloat16), _d((T, h), torch.float32))


CUDA0 = torch.device("cuda", 0)


def test_forward(fake):
    q, kv, idx, out, lse = _fwd_args()
    r = smla.sparse_mla_fwd(q, kv, idx, 0.1, out=out, lse=lse, splits=2)
    assert r == (out, lse)
    assert fake.lib.calls == [("sparse_mla_fwd_ex", (q.data_ptr(), kv.data_ptr(), idx.data_ptr(), 3, 8,
                                                     64, 100, 0, 0.1, out.data_ptr(), lse.data_ptr(), 2,
                                                     STREAM))]
    assert fake.entered == [CUDA0]


def test_forward_checked(fake):
    q, kv, idx, out, lse = _fwd_args()
    smla.sparse_mla_fwd(q, kv, idx, 0.1, out=out, lse=lse, splits=4, checked=True)
    assert fake.lib.calls == [("sparse_mla_fwd_checked", (q.data_ptr(), kv.data_ptr(), idx.data_ptr(), 3,
                                                          8, 64, 100, 0, 0.1, out.data_ptr(), lse.data_ptr(),
                                                          4, STREAM))]
    assert fake.entered == [CUDA0]


def test_forward_fp8_and_default_scale(fake):
    q, _, idx, out, lse = _fwd_args()
    kv = _d((100, 656), torch.uint8)
    smla.sparse_mla_fwd(q, kv, idx, out=out, lse=lse, kv_format="fp8")
    name, args = fake.lib.calls[0]
    assert name == "sparse_mla_fwd_ex" and args[7] == 1 and args[8] == 576 ** -0.5 and args[11] == 0


def test_forward_noalloc(fake):
    q, kv, idx, out, lse = _fwd_args(T=5, h=16, topk=2048, slots=4096)
    smla.sparse_mla_fwd_noalloc(q, kv, idx, 0.2, out=out, lse=lse, splits=4)
    assert fake.lib.calls == [("sparse_mla_fwd_noalloc", (q.data_ptr(), kv.data_ptr(), idx.data_ptr(), 5,
                                                          16, 2048, 4096, 0, 0.2, out.data_ptr(),
                                                          lse.data_ptr(), 4, STREAM))]
    assert fake.entered == [CUDA0]


def test_forward_host(fake):
    T, h, topk = 4, 8, 64
    q = torch.zeros(T, h, 576, dtype=torch.bfloat16)
    idx = torch.zeros(T, topk, dtype=torch.int32)
    out = torch.zeros(T, h, 512, dtype=torch.bfloat16)
    lse = torch.zeros(T, h, dtype=torch.float32)
    kv = _d((50, 576), torch.bfloat16)
    ws = _d((4096,), torch.uint8)
    smla.sparse_mla_fwd_host(q, kv, idx, 0.3, out, lse, ws)
    assert fake.lib.calls == [("sparse_mla_fwd_host", (q.data_ptr(), kv.data_ptr(), idx.data_ptr(), T, h,
                                                       topk, 50, 0, 0.3, out.data_ptr(), lse.data_ptr(),
                                                       ws.data_ptr(), 4096, STREAM))]
    assert fake.entered == [CUDA0]


def test_forward_host_packed(fake, monkeypatch):
    T, h, topk = 4, 8, 64
    monkeypatch.setattr(_binding, "_host_io_layout", lambda T_, h_, k_: (100, 64, 80, 48))
    inb = torch.zeros(100, dtype=torch.uint8)
    outb = torch.zeros(80, dtype=torch.uint8)
    kv = _d((50, 576), torch.bfloat16)
    ws = _d((4096,), torch.uint8)
    smla.sparse_mla_fwd_host_packed(inb, kv, T, h, topk, 0.3, outb, ws)
    assert fake.lib.calls == [("sparse_mla_fwd_host_packed", (inb.data_ptr(), kv.data_ptr(), T, h, topk, 50, 0,
                                                              0.3, outb.data_ptr(), ws.data_ptr(), 4096,
                                                              STREAM))]
    assert fake.entered == [CUDA0]
    with pytest.raises(ValueError):
        smla.sparse_mla_fwd_host_packed(torch.zeros(99, dtype=torch.uint8), kv, T, h, topk, 0.3, outb, ws)


def test_merge(fake):
    n, T, h = 3, 6, 8
    o, l = _d((n, T, h, 512), torch.bfloat16), _d((n, T, h), torch.float32)
    out, lse = _d((T, h, 512), torch.bfloat16), _d((T, h), torch.float32)
    assert smla.sparse_mla_merge(o, l, out=out, lse=lse) == (out, lse)
    assert fake.lib.calls == [("sparse_mla_merge", (o.data_ptr(), l.data_ptr(), n, T, h, out.data_ptr(),
                                                    lse.data_ptr(), STREAM))]
    assert fake.entered == [CUDA0]


def test_v_up(fake):
    T, h, v = 7, 8, 256
    o, w, y = _d((T, h, 512), torch.bfloat16), _d((h, v, 512), torch.bfloat16), _d((T, h, v), torch.bfloat16)
    assert smla.sparse_mla_v_up(o, w, out=y) is y
    assert fake.lib.calls == [("sparse_mla_v_up", (o.data_ptr(), w.data_ptr(), T, h, v, y.data_ptr(),
                                                   STREAM))]
    assert fake.entered == [CUDA0]


@pytest.mark.parametrize("with_table", [False, True])
def test_topk(fake, with_table):
    T, S, k = 5, 300, 16
    s, ln, out = _d((T, S), torch.float32), _d((T,), torch.int32), _d((T, k), torch.int32)
    bt = _d(((S + 63) // 64,), torch.int32) if with_table else None
    assert smla.sparse_mla_topk(s, ln, k, block_table=bt, out=out) is out
    assert fake.lib.calls == [("sparse_mla_topk", (s.data_ptr(), T, S, ln.data_ptr(), k,
                                                   bt.data_ptr() if with_table else None, out.data_ptr(),
                                                   STREAM))]
    assert fake.entered == [CUDA0]


def test_an_explicit_stream_is_passed_through(fake):
    q, kv, idx, out, lse = _fwd_args()
    smla.sparse_mla_fwd(q, kv, idx, 0.1, out=out, lse=lse, stream=SimpleNamespace(device=CUDA0, cuda_stream=77))
    smla.sparse_mla_fwd(q, kv, idx, 0.1, out=out, lse=lse, stream=99)
    assert [c[1][-1] for c in fake.lib.calls] == [77, 99]


def _mixed_device_calls():
    """(what, call) pairs, each with one tensor or the stream on another device."""
    T, h = 3, 8

    def fwd(**kw):
        q, kv, idx, out, lse = _fwd_args(T, h)
        a = dict(q=q, kv=kv, idx=idx, out=out, lse=lse)
        a.update(kw)
        return lambda: smla.sparse_mla_fwd(a["q"], a["kv"], a["idx"], 0.1, out=a["out"], lse=a["lse"],
                                           stream=a.get("stream"))

    def noalloc(**kw):
        q, kv, idx, out, lse = _fwd_args(T, h)
        a = dict(q=q, kv=kv, idx=idx, out=out, lse=lse)
        a.update(kw)
        return lambda: smla.sparse_mla_fwd_noalloc(a["q"], a["kv"], a["idx"], 0.1, out=a["out"], lse=a["lse"])

    o, l = _d((2, T, h, 512), torch.bfloat16), _d((2, T, h), torch.float32)
    mo, ml = _d((T, h, 512), torch.bfloat16), _d((T, h), torch.float32)
    w, y = _d((h, 128, 512), torch.bfloat16), _d((T, h, 128), torch.bfloat16)
    s, ln, ko = _d((T, 100), torch.float32), _d((T,), torch.int32), _d((T, 8), torch.int32)
    return [
        ("fwd kv on cuda:1", fwd(kv=_d((100, 576), torch.bfloat16, 1))),
        ("fwd out on cuda:1", fwd(out=_d((T, h, 512), torch.bfloat16, 1))),
        ("fwd out on the host", fwd(out=torch.zeros(T, h, 512, dtype=torch.bfloat16))),
        ("fwd lse on the host", fwd(lse=torch.zeros(T, h, dtype=torch.float32))),
        ("fwd stream on cuda:1", fwd(stream=SimpleNamespace(device=torch.device("cuda", 1), cuda_stream=5))),
        ("noalloc idx on cuda:1", noalloc(idx=_d((T, 64), torch.int32, 1))),
        ("noalloc lse on the host", noalloc(lse=torch.zeros(T, h, dtype=torch.float32))),
        ("merge lse_parts on cuda:1", lambda: smla.sparse_mla_merge(o, _d((2, T, h), torch.float32, 1),
                                                                    out=mo, lse=ml)),
        ("merge out on cuda:1", lambda: smla.sparse_mla_merge(o, l, out=_d((T, h, 512), torch.bfloat16, 1),
                                                              lse=ml)),
        ("v_up w on cuda:1", lambda: smla.sparse_mla_v_up(mo, _d((h, 128, 512), torch.bfloat16, 1), out=y)),
        ("v_up out on the host", lambda: smla.sparse_mla_v_up(mo, w, out=torch.zeros(T, h, 128,
                                                                                     dtype=torch.bfloat16))),
        ("topk lengths on cuda:1", lambda: smla.sparse_mla_topk(s, _d((T,), torch.int32, 1), 8, out=ko)),
        ("topk table on cuda:1", lambda: smla.sparse_mla_topk(s, ln, 8, block_table=_d((2,), torch.int32, 1),
                                                              out=ko)),
        ("topk out on cuda:1", lambda: smla.sparse_mla_topk(s, ln, 8, out=_d((T, 8), torch.int32, 1))),
        ("host path workspace on cuda:1", lambda: smla.sparse_mla_fwd_host(
            torch.zeros(T, h, 576, dtype=torch.bfloat16), _d((100, 576), torch.bfloat16),
            torch.zeros(T, 64, dtype=torch.int32), 0.1, torch.zeros(T, h, 512, dtype=torch.bfloat16),
            torch.zeros(T, h, dtype=torch.float32), _d((4096,), torch.uint8, 1))),
    ]


@pytest.mark.parametrize("what", [w for w, _ in _mixed_device_calls()])
def test_mixed_devices_are_rejected_before_the_library(fake, what):
    call = dict(_mixed_device_calls())[what]
    with pytest.raises(ValueError):
        call()
    assert fake.lib.calls == []


def test_no_guard_when_the_device_is_already_current(fake):
    fake.current["index"] = 0
    q, kv, idx, out, lse = _fwd_args()
    smla.sparse_mla_fwd(q, kv, idx, 0.5, out=out, lse=lse)
    assert fake.entered == []
    assert [c[0] for c in fake.lib.calls] == ["sparse_mla_fwd_ex"]
