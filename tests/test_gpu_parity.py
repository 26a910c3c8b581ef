"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Every comparison uses the tolerance in tests/parity.py.  Index handling is
checked exactly with closed-form probes: with q = 0 every logit is 0, so
LSE = ln(number of valid entries) and O is the mean of the listed V rows,
which identifies the rows the kernel actually used.
"""

import math
from functools import lru_cache

import numpy as np
import pytest
import torch

import oracle
import token_sparse_mla_gb300 as smla
from tests.parity import assert_parity, to_np
from workloads import make_workload, pad_heads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SPLITS = (0, 1, 2, 4, 8)


@lru_cache(maxsize=None)
def _wl(name, **kw):
    return make_workload(name, **kw)


def wl(name, **kw):
    return _wl(name, **dict(sorted(kw.items())))


def run_gpu(q, kv, idx, scale, splits=0, kv_format="bf16"):
    out, lse = smla.sparse_mla_fwd(q.to(DEV), kv.to(DEV), idx.to(DEV), scale, splits=splits,
                                   kv_format=kv_format)
    smla.sync_status()
    return out.cpu(), lse.cpu()


def check_case(q, kv, idx, scale, splits=0, kv_format="bf16", tokens=None, what=""):
    out, lse = run_gpu(q, kv, idx, scale, splits, kv_format)
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, scale, kv_format=kv_format, tokens=tokens)
    if tokens is not None:
        out, lse = out[list(tokens)], lse[list(tokens)]
    return assert_parity(out, lse, ref_o, ref_l, what=what)


# ----------------------------------------------------------------------------- small configs

@pytest.mark.parametrize("splits", SPLITS)
def test_tiny_config(splits):
    w = wl("tiny")
    check_case(w.q, w.kv, w.indices, w.scale, splits, what=f"tiny splits={splits}")


@pytest.mark.parametrize("h", [8, 16, 32, 64])
@pytest.mark.parametrize("splits", [0, 1, 4])
def test_sweep_reduced(h, splits):
    w = wl("sweep", n_seq=3, h=h)
    check_case(w.q, w.kv, w.indices, w.scale, splits, what=f"sweep h={h} splits={splits}")


@pytest.mark.parametrize("splits", SPLITS)
def test_decode_reduced(splits):
    w = wl("decode_bf16", n_seq=3)
    check_case(w.q, w.kv, w.indices, w.scale, splits, what=f"decode splits={splits}")


def test_prefill_reduced():
    w = wl("prefill", n_tokens=6)
    check_case(w.q, w.kv, w.indices, w.scale, 0, what="prefill prefix")


# ----------------------------------------------------------------------------- edge cases

def _rand(seed, T, h, topk, S, p_invalid=0.0, dup=False):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, h, 576, generator=g) * 0.5).to(torch.bfloat16)
    kv = (torch.randn(S, 576, generator=g) * 0.5).to(torch.bfloat16)
    if dup:
        idx = torch.randint(0, S, (T, topk), generator=g)
    else:
        idx = torch.stack([torch.randperm(S, generator=g)[:topk] for _ in range(T)])
    idx = idx.masked_fill(torch.rand(T, topk, generator=g) < p_invalid, -1)
    return q, kv, idx.to(torch.int32)


@pytest.mark.parametrize("topk", [1, 3, 37, 63, 65, 130, 2047, 2049])
@pytest.mark.parametrize("h", [8, 64])
def test_ragged_topk(topk, h):
    q, kv, idx = _rand(100 + topk, 5, h, topk, 4096, p_invalid=0.1)
    for splits in (0, 1, 2, 8):
        check_case(q, kv, idx, 576 ** -0.5, splits, what=f"topk={topk} h={h} splits={splits}")


@pytest.mark.parametrize("T,topk,splits", [(1, 4096, 0), (5, 2048, 0), (3, 33, 8), (7, 300, 4),
                                           (200, 2048, 2), (153, 300, 4)])
@pytest.mark.parametrize("h", [8, 16])
def test_balanced_partition_cuts_lists_anywhere(T, topk, splits, h):
    # 8/16 heads cut the T x ceil(topk/32) row blocks into equal ranges, one per CTA: aligned
    # (16 CTAs per list, one block per CTA) and unaligned (ranges that end inside one list and
    # start inside another, up to one CTA per SM); cut lists merge after the grid barrier
    q, kv, idx = _rand(300 + T + topk, T, h, topk, 8192, p_invalid=0.05)
    check_case(q, kv, idx, 576 ** -0.5, splits, what=f"balanced T={T} topk={topk} splits={splits} h={h}")


def test_balanced_partition_repeats_bit_for_bit():
    # the merge counters return to zero after every launch and partials are summed in CTA order:
    # repeated calls, a second stream and a replayed CUDA graph all give identical bytes
    q, kv, idx = _rand(77, 7, 8, 300, 8192, p_invalid=0.05)  # splits=4: unaligned cuts
    q, kv, idx = q.to(DEV), kv.to(DEV), idx.to(DEV)
    o1, l1 = smla.sparse_mla_fwd(q, kv, idx, 0.05, splits=4)
    o2, l2 = smla.sparse_mla_fwd(q, kv, idx, 0.05, splits=4)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o3, l3 = smla.sparse_mla_fwd(q, kv, idx, 0.05, splits=4, stream=s)  # sizes this stream's scratch
        g = torch.cuda.CUDAGraph()
        og = torch.empty_like(o1)
        lg = torch.empty_like(l1)
    with torch.cuda.graph(g, stream=s):
        smla.sparse_mla_fwd(q, kv, idx, 0.05, out=og, lse=lg, splits=4, stream=s)
    for _ in range(3):
        og.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(og, o1) and torch.equal(lg, l1)
    smla.sync_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
    ref_o, ref_l = oracle.sparse_mla_fwd(q.cpu(), kv.cpu(), idx.cpu(), 0.05)
    assert_parity(o1.cpu(), l1.cpu(), ref_o, ref_l, what="balanced repeat")


def test_out_of_range_and_negative_indices_are_masked():
    q, kv, idx = _rand(7, 4, 16, 200, 1000, p_invalid=0.2)
    idx[0, 3] = 1000          # == num_slots
    idx[1, 5] = 2_000_000_000
    idx[2, 7] = -5
    idx[3, :] = -1            # a list with no valid entry
    idx[3, 150] = -1
    check_case(q, kv, idx, 0.05, 0, what="masking")
    check_case(q, kv, idx, 0.05, 4, what="masking split")


@pytest.mark.parametrize("h,kv_format", [(8, "bf16"), (16, "bf16"), (32, "bf16"), (64, "bf16"),
                                         (8, "fp8"), (64, "fp8")])
def test_checked_mode_reports_out_of_range_entries(h, kv_format):
    # checked mode masks exactly what the default mode masks (same bytes out) and, for entries
    # other than -1 outside [0, num_slots), makes sync_status report SMLA_ERR_INDEX_RANGE once
    if kv_format == "fp8":
        q, kv, idx = _rand_fp8(17 + h, 4, h, 200, 1000, p_invalid=0.2)
    else:
        q, kv, idx = _rand(17 + h, 4, h, 200, 1000, p_invalid=0.2)
    clean = idx.clone()
    idx[0, 3] = 1000          # == num_slots
    idx[1, 5] = 2_000_000_000
    idx[2, 199] = -5          # last entry of a list
    qd, kvd, idd, cld = q.to(DEV), kv.to(DEV), idx.to(DEV), clean.to(DEV)
    for splits in (0, 1, 4):
        ref_o, ref_l = smla.sparse_mla_fwd(qd, kvd, idd, 0.05, splits=splits, kv_format=kv_format)
        smla.sync_status()  # the default mode masks silently
        o, l = smla.sparse_mla_fwd(qd, kvd, idd, 0.05, splits=splits, kv_format=kv_format, checked=True)
        with pytest.raises(smla.SparseMLAError) as e:
            smla.sync_status()
        assert e.value.status == 5
        smla.sync_status()  # read once, then cleared
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
        # -1 padding and in-range entries never count
        smla.sparse_mla_fwd(qd, kvd, cld, 0.05, splits=splits, kv_format=kv_format, checked=True)
        smla.sync_status()
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, 0.05, kv_format=kv_format)
    assert_parity(o.cpu(), l.cpu(), ref_o, ref_l, what=f"checked h={h} {kv_format}")


def test_all_invalid_lists():
    q, kv, idx = _rand(8, 6, 32, 300, 500)
    idx[:] = -1
    for splits in (1, 4):
        out, lse = run_gpu(q, kv, idx, 0.05, splits)
        assert torch.all(out.float() == 0)
        assert torch.all(torch.isneginf(lse))


def test_duplicates_and_topk_one():
    q, kv, _ = _rand(9, 4, 8, 1, 300)
    one = torch.tensor([[5], [17], [299], [0]], dtype=torch.int32)
    out1, lse1 = run_gpu(q, kv, one, 0.07)
    # topk = 1: O is that row's V (exactly, after bf16 rounding of a weight of 1)
    for t, s in enumerate([5, 17, 299, 0]):
        assert torch.equal(out1[t], kv[s, :512].unsqueeze(0).expand(8, 512))
    for k in (2, 7, 64, 65):
        outk, lsek = run_gpu(q, kv, one.repeat(1, k), 0.07)
        assert torch.equal(outk, out1)
        np.testing.assert_allclose(to_np(lsek), to_np(lse1) + math.log(k), atol=1e-3, rtol=0)
    check_case(q, kv, torch.randint(0, 300, (4, 500), dtype=torch.int32), 0.07, what="dups")


def test_permutation_invariance_on_gpu():
    q, kv, idx = _rand(10, 4, 16, 1024, 5000, p_invalid=0.05)
    o1, l1 = run_gpu(q, kv, idx, 576 ** -0.5)
    g = torch.Generator().manual_seed(3)
    perm = torch.stack([torch.randperm(1024, generator=g) for _ in range(4)])
    o2, l2 = run_gpu(q, kv, torch.gather(idx, 1, perm), 576 ** -0.5)
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, 576 ** -0.5)
    assert_parity(o2, l2, ref_o, ref_l, what="permuted")
    assert (to_np(o1) - to_np(o2)).__abs__().max() <= 8e-3


@pytest.mark.parametrize("h", [8, 64])
def test_count_and_mean_probe_selects_the_listed_rows(h):
    """q = 0: LSE = ln(n_valid) and O = mean of the listed V rows (small integers)."""
    T, topk, S = 6, 1000, 3000
    g = torch.Generator().manual_seed(11)
    vals = torch.randint(-8, 9, (S, 576), generator=g).float()
    kv = vals.to(torch.bfloat16)
    q = torch.zeros(T, h, 576, dtype=torch.bfloat16)
    idx = torch.stack([torch.randperm(S, generator=g)[:topk] for _ in range(T)])
    idx = idx.masked_fill(torch.rand(T, topk, generator=g) < 0.3, -1).to(torch.int32)
    for splits in (1, 8):
        out, lse = run_gpu(q, kv, idx, 0.1, splits)
        for t in range(T):
            sel = idx[t][idx[t] >= 0].long()
            n = sel.numel()
            assert abs(float(lse[t, 0]) - math.log(n)) <= 2e-5 * max(1.0, math.log(n))
            mean = vals[sel, :512].double().sum(0) / n
            got = out[t].double()
            assert torch.all((got - mean).abs() <= mean.abs() * 2.0 ** -7 + 1e-6), (t, splits)


def test_one_hot_logit_picks_the_row():
    T, h, S = 3, 16, 4096
    g = torch.Generator().manual_seed(12)
    kvf = torch.randn(S, 576, generator=g) * 0.5
    kvf[:, 575] = 0.0
    chosen = [100, 2000, 4095]
    for s in chosen:
        kvf[s, 575] = 8.0
    kv = kvf.to(torch.bfloat16)
    q = torch.zeros(T, h, 576)
    q[:, :, 575] = 8.0
    q = q.to(torch.bfloat16)
    idx = torch.stack([torch.randperm(S, generator=g)[:512] for _ in range(T)])
    for t, s in enumerate(chosen):
        idx[t][idx[t] == s] = -1   # list the chosen row exactly once
        idx[t, 333] = s
    idx = idx.to(torch.int32)
    out, lse = run_gpu(q, kv, idx, 1.0)
    for t, s in enumerate(chosen):
        assert torch.allclose(out[t].float(), kv[s, :512].float().expand(h, 512), atol=1e-2)


def test_peaked_distribution_tighter_gate():
    """q x 8 makes the logits ~8x sharper; compare with 2 % of max |ref| per (token, head)."""
    q, kv, idx = _rand(13, 8, 32, 2048, 20000, p_invalid=0.05)
    q = (q.float() * 8).to(torch.bfloat16)
    out, lse = run_gpu(q, kv, idx, 576 ** -0.5)
    ref_o, ref_l = oracle.sparse_mla_fwd(q, kv, idx, 576 ** -0.5)
    o = to_np(out)
    bound = 0.02 * np.abs(ref_o).max(axis=2, keepdims=True)
    assert np.all(np.abs(o - ref_o) <= bound)
    assert np.abs(to_np(lse) - ref_l).max() <= 1e-3


def test_zero_tokens_noop():
    q = torch.zeros(0, 8, 576, dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros(16, 576, dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros(0, 8, dtype=torch.int32, device=DEV)
    out, lse = smla.sparse_mla_fwd(q, kv, idx)
    smla.sync_status()
    assert out.shape == (0, 8, 512) and lse.shape == (0, 8)


def test_caller_owned_buffers_and_stream():
    w = wl("tiny")
    q, kv, idx = w.q.to(DEV), w.kv.to(DEV), w.indices.to(DEV)
    out = torch.full((w.T, 8, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((w.T, 8), 7.0, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = smla.sparse_mla_fwd(q, kv, idx, w.scale, out=out, lse=lse, stream=s)
    s.synchronize()
    assert o2.data_ptr() == out.data_ptr() and l2.data_ptr() == lse.data_ptr()
    ref_o, ref_l = oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale)
    assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, what="caller buffers")


def test_host_entry_point_matches_device_path():
    w = wl("decode_bf16", n_seq=4)
    kv = w.kv.to(DEV)
    out_d, lse_d = smla.sparse_mla_fwd(w.q.to(DEV), kv, w.indices.to(DEV), w.scale)
    qh, ih = w.q.pin_memory(), w.indices.pin_memory()
    oh = torch.empty((w.T, w.h, 512), dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((w.T, w.h), dtype=torch.float32).pin_memory()
    ws = torch.empty(smla.host_workspace_bytes(w.T, w.h, w.topk), dtype=torch.uint8, device=DEV)
    smla.sparse_mla_fwd_host(qh, kv, ih, w.scale, oh, lh, ws)
    smla.sync_status()
    assert torch.equal(oh, out_d.cpu()) and torch.equal(lh, lse_d.cpu())


def test_packed_host_entry_point_matches_device_path():
    w = wl("decode_bf16", n_seq=5)
    kv = w.kv.to(DEV)
    out_d, lse_d = smla.sparse_mla_fwd(w.q.to(DEV), kv, w.indices.to(DEV), w.scale)
    lay = smla.host_io_layout(w.T, w.h, w.topk)
    inb = torch.full((lay["in_bytes"],), 0xAB, dtype=torch.uint8).pin_memory()
    outb = torch.full((lay["out_bytes"],), 0xCD, dtype=torch.uint8).pin_memory()
    qv, iv, ov, lv = smla.host_io_views(inb, outb, w.T, w.h, w.topk)
    qv.copy_(w.q)
    iv.copy_(w.indices)
    ws = torch.empty(smla.host_workspace_bytes(w.T, w.h, w.topk), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    for _ in range(2):
        smla.sparse_mla_fwd_host_packed(inb, kv, w.T, w.h, w.topk, w.scale, outb, ws, stream=s)
        smla.sync_status(s)
        assert torch.equal(ov, out_d.cpu()) and torch.equal(lv, lse_d.cpu())


def test_padded_matches_native():
    w = wl("sweep", n_seq=3, h=8)
    q, kv, idx = w.q.to(DEV), w.kv.to(DEV), w.indices.to(DEV)
    o8, l8 = smla.sparse_mla_fwd(q, kv, idx, w.scale)
    o64, l64 = smla.sparse_mla_fwd(pad_heads(q, 64), kv, idx, w.scale)
    smla.sync_status()
    assert (o8.float() - o64[:, :8].float()).abs().max().item() <= 8e-3
    assert (l8 - l64[:, :8]).abs().max().item() <= 1e-3


# ----------------------------------------------------------------------------- full-size configs

def test_full_decode_bf16_all_tokens():
    w = wl("decode_bf16")
    check_case(w.q, w.kv, w.indices, w.scale, 0, what="decode_bf16 full")


@pytest.mark.parametrize("h", [8, 16, 32, 64])
def test_full_sweep(h):
    w = wl("sweep", h=h)
    toks = list(range(0, w.T, 4 if h == 64 else 2))
    check_case(w.q, w.kv, w.indices, w.scale, 0, tokens=toks, what=f"sweep full h={h}")
    qp = pad_heads(w.q, 64)
    out, lse = run_gpu(qp, w.kv, w.indices, w.scale)
    ref_o, ref_l = oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, tokens=toks[:16])
    assert_parity(out[toks[:16], :h], lse[toks[:16], :h], ref_o, ref_l, what=f"sweep padded h={h}")


def test_full_prefill_sampled_tokens():
    w = wl("prefill")
    g = torch.Generator().manual_seed(5)
    toks = sorted(set([0, 1, w.T - 1] + torch.randint(0, w.T, (29,), generator=g).tolist()))
    check_case(w.q, w.kv, w.indices, w.scale, 0, tokens=toks, what="prefill full")


# ----------------------------------------------------------------------------- fp8 KV rows

def _rand_fp8(seed, T, h, topk, S, p_invalid=0.05, dup=False):
    from workloads import quantize_fp8_rows
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, h, 576, generator=g) * 0.5).to(torch.bfloat16)
    kv = quantize_fp8_rows(torch.randn(S, 576, generator=g) * 0.5)
    if dup:
        idx = torch.randint(0, S, (T, topk), generator=g)
    else:
        idx = torch.stack([torch.randperm(S, generator=g)[:topk] for _ in range(T)])
    idx = idx.masked_fill(torch.rand(T, topk, generator=g) < p_invalid, -1)
    return q, kv, idx.to(torch.int32)


@pytest.mark.parametrize("h", [8, 16, 32, 64])
@pytest.mark.parametrize("splits", [0, 1, 4])
def test_fp8_random(h, splits):
    q, kv, idx = _rand_fp8(200 + h, 5, h, 777, 5000, dup=(h == 16))
    idx[0, 5] = 5000
    idx[1, :] = -1
    check_case(q, kv, idx, 576 ** -0.5, splits, kv_format="fp8", what=f"fp8 h={h} splits={splits}")


@pytest.mark.parametrize("h", [8, 16])
@pytest.mark.parametrize("splits", [0, 2])
def test_fp8_cluster_parts(h, splits):
    # topk 1000 = 32 row blocks: the list is cut into 8 (default) or 2 aligned parts, one
    # thread-block cluster per token, merged through distributed shared memory
    q, kv, idx = _rand_fp8(400 + h, 5, h, 1000, 6000)
    info = smla.launch_info(5, h, 1000, "fp8")
    assert splits != 0 or info["splits"] == 8
    check_case(q, kv, idx, 576 ** -0.5, splits, kv_format="fp8", what=f"fp8 clusters h={h} splits={splits}")


def test_fp8_reduced_config():
    w = wl("fp8_mixed", n_seq=1, n_tokens=48)
    check_case(w.q, w.kv, w.indices, w.scale, 0, kv_format="fp8", what="fp8_mixed prefix")


def test_fp8_single_entry_is_dequantised_row():
    q, kv, _ = _rand_fp8(300, 3, 8, 1, 64)
    idx = torch.tensor([[3], [40], [63]], dtype=torch.int32)
    out, lse = run_gpu(q, kv, idx, 0.1, kv_format="fp8")
    for t, s in enumerate([3, 40, 63]):
        row = oracle.decode_row(kv, "fp8", s)[:512]
        # e4m3 * scale is exact in fp64; the kernel rounds the fp32 product, then to bf16
        ref = torch.from_numpy(row).float().to(torch.bfloat16).float()
        assert torch.equal(out[t].float(), ref.expand(8, 512)), t


def test_full_fp8_mixed_sampled_tokens():
    w = wl("fp8_mixed")
    g = torch.Generator().manual_seed(6)
    toks = sorted(set([0, w.T - 1] + torch.randint(0, w.T, (30,), generator=g).tolist()))
    check_case(w.q, w.kv, w.indices, w.scale, 0, kv_format="fp8", tokens=toks, what="fp8 full")
    out, lse = run_gpu(pad_heads(w.q, 64), w.kv, w.indices, w.scale, kv_format="fp8")
    ref_o, ref_l = oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, kv_format="fp8",
                                         tokens=toks[:8])
    assert_parity(out[toks[:8], :8], lse[toks[:8], :8], ref_o, ref_l, what="fp8 padded")
