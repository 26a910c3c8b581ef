"""CPU-side checks of the C ABI: the library loads, exports what the header
declares, and rejects bad arguments on the host before touching a device."""

import ctypes
import re
from pathlib import Path

import pytest
import torch

import token_sparse_mla_gb300 as smla
from token_sparse_mla_gb300 import _binding

ROOT = Path(__file__).resolve().parent.parent


def _declared_functions():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = h.read_text()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from token_sparse_mla_gb300 import build
    build.build()
    return smla.library()


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    assert "sparse_mla_fwd" in names and len(names) >= 7, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(_binding.EXPORTED) <= names


def test_version(lib):
    assert smla.version() == 10100


def test_workspace_bytes(lib):
    T, h, topk = 32, 8, 2048
    need = smla.host_workspace_bytes(T, h, topk)
    raw = T * h * 576 * 2 + T * topk * 4 + T * h * 512 * 2 + T * h * 4
    assert raw <= need <= raw + 4 * 256
    assert smla.host_workspace_bytes(0, 8, 2048) == 0


def test_host_io_layout(lib):
    T, h, topk = 32, 8, 2048
    lay = smla.host_io_layout(T, h, topk)
    q, i, o, l = T * h * 576 * 2, T * topk * 4, T * h * 512 * 2, T * h * 4
    assert lay["indices_offset"] >= q and lay["indices_offset"] % 256 == 0
    assert lay["in_bytes"] == lay["indices_offset"] + i
    assert lay["lse_offset"] >= o and lay["lse_offset"] % 256 == 0
    assert lay["out_bytes"] == lay["lse_offset"] + l
    # the device workspace holds both packed regions back to back
    assert lay["in_bytes"] + lay["out_bytes"] <= smla.host_workspace_bytes(T, h, topk)
    inb = torch.zeros(lay["in_bytes"], dtype=torch.uint8)
    outb = torch.zeros(lay["out_bytes"], dtype=torch.uint8)
    qv, iv, ov, lv = smla.host_io_views(inb, outb, T, h, topk)
    iv.fill_(-1)
    assert int(inb[lay["indices_offset"]:].sum()) == 255 * i and int(inb[:q].sum()) == 0
    lv.fill_(1.0)
    assert qv.shape == (T, h, 576) and ov.shape == (T, h, 512) and lv.shape == (T, h)
    assert outb[lay["lse_offset"]:].view(torch.float32).eq(1.0).all()


def _call(lib, **kw):
    args = dict(q=0x1000, kv=0x1000, idx=0x1000, T=4, h=8, topk=64, num_slots=256, fmt=0,
                scale=0.04, out=0x1000, lse=0x1000, splits=0)
    args.update(kw)
    return lib.sparse_mla_fwd_ex(args["q"], args["kv"], args["idx"], args["T"], args["h"],
                                 args["topk"], args["num_slots"], args["fmt"], args["scale"],
                                 args["out"], args["lse"], args["splits"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(h=12), 2), (dict(h=128), 2), (dict(topk=0), 1), (dict(T=-1), 1),
    (dict(num_slots=0), 1), (dict(num_slots=1 << 31), 1), (dict(fmt=7), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(splits=3), 1),
    (dict(splits=16), 1), (dict(q=0), 1), (dict(kv=0), 1), (dict(idx=0), 1), (dict(out=0), 1),
    (dict(lse=0), 1), (dict(q=0x1008), 1), (dict(kv=0x1004), 1), (dict(out=0x1002), 1),
    (dict(idx=0x1002), 1), (dict(lse=0x1001), 1),
])
def test_host_validation_rejects(lib, kw, status):
    assert _call(lib, **kw) == status
    assert lib.sparse_mla_last_error().decode()


def test_zero_tokens_is_a_noop(lib):
    assert _call(lib, T=0, q=0, kv=0, idx=0, out=0, lse=0) == 0


def test_launch_info_without_device(lib):
    # 8/16 heads: 32 tokens x 64 row blocks on 152 SMs (assumed without a device): a cluster
    # of four CTAs per token (the largest power of two dividing 64 with 32 x s <= 152)
    info = smla.launch_info(32, 8, 2048)
    assert info["launches"] == 1 and info["splits"] == 4 and info["ctas"] == 128
    # as many tokens as SMs: one CTA per token
    assert smla.launch_info(152, 8, 2048)["ctas"] == 152
    assert info["smem_bytes"] <= 232448
    # fewer blocks than SMs: one CTA per 32-entry block
    assert smla.launch_info(2, 16, 100)["ctas"] == 2 * 4
    # 32/64 heads: a cluster of `splits` CTAs per token
    info = smla.launch_info(32, 64, 2048)
    assert info["splits"] in (1, 2, 4, 8) and info["ctas"] == 32 * info["splits"]
    assert info["smem_bytes"] <= 232448
    assert smla.launch_info(0, 8, 2048)["launches"] == 0
    with pytest.raises(smla.SparseMLAError):
        smla.launch_info(4, 24, 64)


def test_binding_refuses_cpu_tensors():
    q = torch.zeros(2, 8, 576, dtype=torch.bfloat16)
    kv = torch.zeros(16, 576, dtype=torch.bfloat16)
    idx = torch.zeros(2, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        smla.sparse_mla_fwd(q, kv, idx)


def test_binding_shape_checks():
    q = torch.zeros(2, 8, 512, dtype=torch.bfloat16)
    kv = torch.zeros(16, 576, dtype=torch.bfloat16)
    idx = torch.zeros(2, 4, dtype=torch.int32)
    with pytest.raises(ValueError):
        smla.sparse_mla_fwd(q, kv, idx)
    with pytest.raises(ValueError):
        smla.sparse_mla_fwd(torch.zeros(2, 8, 576, dtype=torch.bfloat16), kv, idx.long())


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "_LIB_PATH", tmp_path / "absent.so")
    with pytest.raises(ImportError, match="missing"):
        _binding.library()


def test_product_package_does_not_import_the_oracle():
    pkg = ROOT / "token_sparse_mla_gb300"
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")):
        text = f.read_text()
        assert "oracle" not in text.replace("oracle-free", ""), f"{f} mentions the oracle"


def test_launch_plans_over_many_shapes(lib):
    # host-side plan (no device: 152 SMs assumed) for every head count and a spread of batch
    # sizes and list lengths: whole lists, aligned cluster parts (2/4/8 CTAs per token, never
    # more CTAs than SMs) or the tcgen05 kernel's clusters
    for h in (8, 16, 32, 64):
        for T in (1, 3, 19, 32, 76, 151, 152, 153, 1000):
            for topk in (1, 33, 100, 2048, 2049, 4096):
                nblk_small = (topk + 31) // 32
                info = smla.launch_info(T, h, topk)
                assert info["launches"] == 1 and info["smem_bytes"] <= 232448
                s, ctas = info["splits"], info["ctas"]
                if h <= 16:
                    if s == 0:
                        assert ctas == T  # whole lists, one CTA per token
                    else:
                        assert s in (2, 4, 8) and nblk_small % s == 0
                        assert ctas == T * s and ctas <= 152
                else:
                    assert s in (1, 2, 4, 8) and ctas == T * s
                    assert s == 1 or ctas <= 152
