"""GPU parity of the masked dense route (through the C ABI) against the oracle.

The scatter of the lists into the bit mask is integer work: compared bit for bit with
oracle.scatter_mask.  The masked MHA is compared element by element with oracle.masked_mha at
the tolerance of tests/parity.py, for the three head geometries of the PR #55738 report's
`_is_masked_mha_available` table (q/k 192 or 256, v 128 or 256), ragged token counts and
request lengths (partial query and key tiles), full causal histories and sparse lists, empty
rows, key tiles that no row reaches, and sharp logits that make the running max grow.
"""

import numpy as np
import pytest
import torch

import oracle
import token_sparse_mla_gb300 as smla
from tests.parity import assert_parity
from workloads import causal_position_lists, make_masked_dense_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _mask_u32(m: torch.Tensor) -> np.ndarray:
    return m.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("T,S,topk", [(1, 1, 1), (5, 8, 3), (16, 100, 40), (3, 32, 32), (7, 65, 70),
                                      (40, 4096, 2048), (9, 70000, 300), (300, 512, 200)])
def test_scatter_is_bit_exact(T, S, topk):
    lists = causal_position_lists(T, S, topk, seed=T + S, p_empty=0.2)
    lists[0, 0] = S          # out of range: sets nothing
    lists[-1, -1] = -5       # negative: sets nothing
    if topk > 2:
        lists[T // 2, 1] = lists[T // 2, 0]   # a repeated position sets one bit
    got = smla.sparse_mla_scatter_mask(lists.to(DEV), S)
    smla.sync_status()
    assert np.array_equal(_mask_u32(got), oracle.scatter_mask(lists, S))


def test_scatter_writes_every_word():
    lists = torch.full((4, 16), -1, dtype=torch.int32)
    out = torch.full((4, 4), -1, dtype=torch.int32, device=DEV)   # stale bits everywhere
    smla.sparse_mla_scatter_mask(lists.to(DEV), 128, out=out)
    smla.sync_status()
    assert int(out.abs().sum()) == 0


def _check(T, S, h, dqk, dv, topk, seed, p_empty=0.0, qmul=1.0, what=""):
    q, k, v = make_masked_dense_inputs(T, S, h, dqk, dv, seed=seed)
    if qmul != 1.0:
        q = (q.float() * qmul).to(torch.bfloat16)
    lists = causal_position_lists(T, S, topk, seed=seed + 1, p_empty=p_empty)
    scale = dqk ** -0.5
    mask = smla.sparse_mla_scatter_mask(lists.to(DEV), S)
    out, lse = smla.sparse_mla_masked_mha(q.to(DEV), k.to(DEV), v.to(DEV), mask, scale)
    smla.sync_status()
    ref_o, ref_l = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), scale)
    return assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, what=what)


@pytest.mark.parametrize("h,dqk,dv", [(4, 192, 128), (2, 256, 256), (3, 256, 128), (2, 192, 256)])
@pytest.mark.parametrize("T,S,topk", [(1, 1, 1), (5, 70, 100), (130, 300, 512), (200, 200, 64),
                                      (257, 1000, 256)])
def test_masked_mha_matches_the_oracle(h, dqk, dv, T, S, topk):
    _check(T, S, h, dqk, dv, topk, seed=T * 7 + S, p_empty=0.1,
           what=f"masked T={T} S={S} h={h} dqk={dqk} dv={dv} topk={topk}")


@pytest.mark.parametrize("dqk,dv", [(192, 128), (256, 256)])
def test_sharp_logits_grow_the_running_max(dqk, dv):
    # q x 8: logits spread over ~+-30 in log2 units, so the running max of a row grows by more
    # than 2^8 between key tiles and O is rescaled in tensor memory
    _check(160, 700, 2, dqk, dv, 700, seed=31, qmul=8.0, what=f"sharp dqk={dqk}")


def test_empty_rows_and_single_positions():
    T, S, h = 6, 300, 2
    q, k, v = make_masked_dense_inputs(T, S, h, 256, 256, seed=5)
    lists = torch.full((T, 8), -1, dtype=torch.int32)
    lists[1, 0] = 7
    lists[2, 3] = 299
    lists[4, :2] = torch.tensor([64, 65], dtype=torch.int32)
    mask = smla.sparse_mla_scatter_mask(lists.to(DEV), S)
    out, lse = smla.sparse_mla_masked_mha(q.to(DEV), k.to(DEV), v.to(DEV), mask, 0.1)
    smla.sync_status()
    out, lse = out.cpu(), lse.cpu()
    for t in (0, 3, 5):
        assert torch.all(out[t].float() == 0) and torch.all(torch.isneginf(lse[t]))
    # one position: O is that position's V row exactly, LSE its scaled logit
    for t, s in ((1, 7), (2, 299)):
        assert torch.equal(out[t], v[s])
        ref = 0.1 * (q[t].double() * k[s].double()).sum(-1)
        assert torch.allclose(lse[t].double(), ref, atol=1e-3, rtol=0)


def test_sparse_lists_skip_unreached_key_tiles():
    # positions in three key tiles far apart: the other tiles are never loaded
    T, S, h = 150, 9000, 2
    q, k, v = make_masked_dense_inputs(T, S, h, 256, 128, seed=9)
    g = torch.Generator().manual_seed(3)
    lists = torch.stack([torch.tensor([0, 63, 4100, 8999], dtype=torch.int32)[torch.randperm(4, generator=g)]
                         for _ in range(T)])
    lists[::7, 2] = -1
    mask = smla.sparse_mla_scatter_mask(lists.to(DEV), S)
    out, lse = smla.sparse_mla_masked_mha(q.to(DEV), k.to(DEV), v.to(DEV), mask, 256 ** -0.5)
    smla.sync_status()
    ref_o, ref_l = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), 256 ** -0.5)
    assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, what="sparse tiles")


def test_repeated_calls_are_identical_and_graph_capturable():
    T, S, h = 140, 600, 2
    q, k, v = (x.to(DEV) for x in make_masked_dense_inputs(T, S, h, 256, 256, seed=12))
    lists = causal_position_lists(T, S, 300, seed=13).to(DEV)
    mask = smla.sparse_mla_scatter_mask(lists, S)
    o1, l1 = smla.sparse_mla_masked_mha(q, k, v, mask, 0.0625)
    s = torch.cuda.Stream()
    og, lg = torch.empty_like(o1), torch.empty_like(l1)
    mg = torch.empty_like(mask)
    with torch.cuda.stream(s):
        smla.sparse_mla_scatter_mask(lists, S, out=mg, stream=s)
        smla.sparse_mla_masked_mha(q, k, v, mg, 0.0625, out=og, lse=lg, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        smla.sparse_mla_scatter_mask(lists, S, out=mg, stream=s)
        smla.sparse_mla_masked_mha(q, k, v, mg, 0.0625, out=og, lse=lg, stream=s)
    for _ in range(3):
        og.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(og, o1) and torch.equal(lg, l1)
    smla.sync_status()


def test_full_size_glm5_prefill_sampled_tokens():
    # the bench workload: a 4096-token prefill chunk that is the whole request, GLM-5 geometry
    # (64 heads, q/k 192 + 64, v 256), top-2048 causal lists; sampled tokens against the oracle
    T = S = 4096
    h, dqk, dv = 64, 256, 256
    q, k, v = make_masked_dense_inputs(T, S, h, dqk, dv, seed=9400)
    lists = causal_position_lists(T, S, 2048, seed=9401)
    mask = smla.sparse_mla_scatter_mask(lists.to(DEV), S)
    out, lse = smla.sparse_mla_masked_mha(q.to(DEV), k.to(DEV), v.to(DEV), mask, dqk ** -0.5)
    smla.sync_status()
    assert np.array_equal(_mask_u32(mask), oracle.scatter_mask(lists, S))
    g = torch.Generator().manual_seed(4)
    toks = sorted(set([0, 127, 128, 2047, 2048, T - 1] + torch.randint(0, T, (10,), generator=g).tolist()))
    ref_o, ref_l = oracle.masked_mha(q[toks], k, v, oracle.scatter_mask(lists[toks], S), dqk ** -0.5)
    assert_parity(out.cpu()[toks], lse.cpu()[toks], ref_o, ref_l, what="glm5 full sampled")


def test_every_list_empty_writes_zeros_everywhere():
    # no query tile reaches any key tile: every CTA skips its loop, still drains the copy of Q it
    # started, and stores zeros over whatever the output held (two query tiles, the second ragged)
    T, S, h = 200, 500, 3
    q, k, v = (x.to(DEV) for x in make_masked_dense_inputs(T, S, h, 192, 256, seed=21))
    lists = torch.full((T, 16), -1, dtype=torch.int32, device=DEV)
    mask = smla.sparse_mla_scatter_mask(lists, S)
    out = torch.full((T, h, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, h), 3.0, dtype=torch.float32, device=DEV)
    smla.sparse_mla_masked_mha(q, k, v, mask, 0.05, out=out, lse=lse)
    smla.sync_status()
    assert int(out.float().abs().sum()) == 0
    assert torch.all(torch.isneginf(lse.cpu()))


def test_longest_request_reaches_the_last_key_tiles():
    # S at its maximum (65536 positions, 1024 key tiles): sparse lists over the whole range, so
    # the tile list holds indices up to 1023; two query tiles, the second ragged
    T, S, h = 130, 65536, 1
    q, k, v = make_masked_dense_inputs(T, S, h, 256, 128, seed=23)
    g = torch.Generator().manual_seed(24)
    lists = torch.randint(0, S, (T, 48), generator=g, dtype=torch.int32)
    lists[:, 0] = S - 1
    lists[:, 1] = 0
    lists[::5, 2:] = -1
    mask = smla.sparse_mla_scatter_mask(lists.to(DEV), S)
    out, lse = smla.sparse_mla_masked_mha(q.to(DEV), k.to(DEV), v.to(DEV), mask, 256 ** -0.5)
    smla.sync_status()
    assert np.array_equal(_mask_u32(mask), oracle.scatter_mask(lists, S))
    ref_o, ref_l = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), 256 ** -0.5)
    assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, what="S = 65536")
