"""sparse_mla_fwd_noalloc: the entry point whose merge scratch is a fixed array
inside the library.  It must give the same bytes as sparse_mla_fwd_ex on the
same arguments, call after call.  This file runs last: the first call on a
device sets up the array (it synchronises the device)."""

import subprocess
import sys
from pathlib import Path

import pytest
import torch

import token_sparse_mla_gb300 as smla

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ROOT = Path(__file__).resolve().parent.parent


def _inputs(seed, T, h, topk, S=8192, p_invalid=0.05):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, h, 576, generator=g) * 0.5).to(torch.bfloat16)
    kv = (torch.randn(S, 576, generator=g) * 0.5).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(S, generator=g)[:topk] for _ in range(T)])
    idx = idx.masked_fill(torch.rand(T, topk, generator=g) < p_invalid, -1).to(torch.int32)
    return q.to(DEV), kv.to(DEV), idx.to(DEV)


def _cuts_lists(T, h, topk, splits):
    """Whether the launch cuts lists at unaligned points, i.e. merges through the scratch:
    8/16 heads, and a split count that does not divide the list's 32-row blocks."""
    nblk = (topk + 31) // 32
    return h <= 16 and splits > 0 and T * splits <= T * nblk and nblk % splits != 0


@pytest.mark.parametrize("T,h,topk,splits", [(7, 8, 300, 4), (3, 16, 300, 8), (5, 16, 300, 4),
                                             (5, 16, 2048, 0), (200, 8, 2048, 2), (32, 8, 2048, 0),
                                             (4, 8, 64, 1)])
def test_noalloc_matches_the_stream_scratch_entry_point(T, h, topk, splits):
    q, kv, idx = _inputs(900 + T + topk, T, h, topk)
    for _ in range(2):  # two consecutive calls: the barrier words must be back at zero
        ref_o, ref_l = smla.sparse_mla_fwd(q, kv, idx, 0.05, splits=splits)
        out = torch.full_like(ref_o, 3.0)
        lse = torch.full_like(ref_l, 3.0)
        smla.sparse_mla_fwd_noalloc(q, kv, idx, 0.05, out=out, lse=lse, splits=splits)
        smla.sync_status()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_the_sixteen_head_cases_reach_the_static_array():
    # the 16-head slots ([grid][2] x (2h + 512h) floats) are only touched by cut lists
    assert _cuts_lists(3, 16, 300, 8) and _cuts_lists(5, 16, 300, 4) and _cuts_lists(7, 8, 300, 4)
    assert not _cuts_lists(5, 16, 2048, 0) and not _cuts_lists(200, 8, 2048, 2)


_FIRST_CALL_CAPTURED = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import token_sparse_mla_gb300 as smla
dev = "cuda:0"
g = torch.Generator().manual_seed(5)
q = (torch.randn(7, 8, 576, generator=g) * 0.5).to(torch.bfloat16).to(dev)
kv = (torch.randn(4096, 576, generator=g) * 0.5).to(torch.bfloat16).to(dev)
idx = torch.randint(0, 4096, (7, 300), generator=g, dtype=torch.int32).to(dev)
out = torch.empty(7, 8, 512, dtype=torch.bfloat16, device=dev)
lse = torch.empty(7, 8, dtype=torch.float32, device=dev)
s = torch.cuda.Stream()
with torch.cuda.stream(s):
    smla.sparse_mla_fwd(q, kv, idx, 0.05, splits=1, stream=s)  # device set-up, no scratch
torch.cuda.synchronize()
graph = torch.cuda.CUDAGraph()
status = None
try:
    with torch.cuda.graph(graph, stream=s):
        smla.sparse_mla_fwd_noalloc(q, kv, idx, 0.05, out=out, lse=lse, splits=4, stream=s)
except smla.SparseMLAError as e:
    status = e.status
torch.cuda.synchronize()
# outside a capture the same call sets the array up and runs
smla.sparse_mla_fwd_noalloc(q, kv, idx, 0.05, out=out, lse=lse, splits=4)
smla.sync_status()
ref_o, ref_l = smla.sparse_mla_fwd(q, kv, idx, 0.05, splits=4)
smla.sync_status()
ok = torch.equal(out, ref_o) and torch.equal(lse, ref_l)
print("STATUS", status, "OK", ok)
"""


def test_first_call_inside_a_capture_is_refused():
    # a fresh process, so the static array of the device is not set up yet
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_CAPTURED, str(ROOT)], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "STATUS 1 OK True" in r.stdout, r.stdout + r.stderr[-2000:]
