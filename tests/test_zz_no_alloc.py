"""sparse_mla_fwd_noalloc: the entry point whose merge scratch is a fixed array
inside the library.  It must give the same bytes as sparse_mla_fwd_ex on the
same arguments, call after call.  This file runs last: the first call on a
device sets up the array (it synchronises the device)."""

import pytest
import torch

import token_sparse_mla_gb300 as smla

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(seed, T, h, topk, S=8192, p_invalid=0.05):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, h, 576, generator=g) * 0.5).to(torch.bfloat16)
    kv = (torch.randn(S, 576, generator=g) * 0.5).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(S, generator=g)[:topk] for _ in range(T)])
    idx = idx.masked_fill(torch.rand(T, topk, generator=g) < p_invalid, -1).to(torch.int32)
    return q.to(DEV), kv.to(DEV), idx.to(DEV)


@pytest.mark.parametrize("T,h,topk,splits", [(7, 8, 300, 4), (5, 16, 2048, 0), (200, 8, 2048, 2),
                                             (32, 8, 2048, 0), (4, 8, 64, 1)])
def test_noalloc_matches_the_stream_scratch_entry_point(T, h, topk, splits):
    q, kv, idx = _inputs(900 + T + topk, T, h, topk)
    for _ in range(2):  # two consecutive calls: the barrier words must be back at zero
        ref_o, ref_l = smla.sparse_mla_fwd(q, kv, idx, 0.05, splits=splits)
        out = torch.full_like(ref_o, 3.0)
        lse = torch.full_like(ref_l, 3.0)
        smla.sparse_mla_fwd_noalloc(q, kv, idx, 0.05, out=out, lse=lse, splits=splits)
        smla.sync_status()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
