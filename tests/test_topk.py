"""Top-k selection of the index lists from per-position scores (the step before the sparse
attention): oracle pins on the CPU.

Row t keeps the topk positions with the largest scores among its causal history [0, len[t]),
ties to the lower position, in ascending position order, mapped to slots through a block table
of 64-slot blocks, -1 padded (vLLM PR #54951, Summary and Additional checks: int32 lists of
fixed width, only the set of selected rows matters).  Pins of the oracle, from outside it:

* set equality with torch.topk on distinct scores, rows in ascending position order;
* closed forms: a history shorter than topk selects all of it and pads with -1; equal scores
  select the lowest positions; a block table maps position p to table[p / 64] * 64 + p % 64;
* mutation: mutated copies (bottom-k, the history length ignored, ties to the higher
  position) each fail one of these.
"""

import ctypes
import math
import re
import subprocess
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle


def _scores(T, S, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(T, S, generator=g, dtype=torch.float32)


# ----------------------------------------------------------------------------- oracle pins

@pytest.mark.parametrize("T,S,k", [(4, 300, 16), (3, 5000, 2048), (2, 64, 64), (5, 1000, 1)])
def test_matches_torch_topk_as_sets(T, S, k):
    s = _scores(T, S, seed=S + k)
    g = torch.Generator().manual_seed(k)
    lens = torch.randint(k, S + 1, (T,), generator=g).to(torch.int32)
    out = oracle.topk(s, lens, k)
    for t in range(T):
        n = int(lens[t])
        ref = torch.topk(s[t, :n], k).indices.numpy()
        assert set(out[t].tolist()) == set(ref.tolist())
        assert np.all(np.diff(out[t]) > 0)


def test_short_history_selects_all_and_pads():
    s = _scores(3, 100, seed=1)
    out = oracle.topk(s, np.array([0, 7, 100], dtype=np.int32), 16)
    assert np.all(out[0] == -1)
    assert out[1].tolist() == list(range(7)) + [-1] * 9
    assert len(set(out[2].tolist())) == 16 and -1 not in out[2]


def test_signed_zeros_are_equal_scores():
    # -0 and +0 are the same real number: a tie, broken towards the lower position
    s = torch.tensor([[-0.0, 0.0, -0.0, 0.0, 1.0, -1.0], [0.0, -0.0, 2.0, -0.0, 0.0, 0.0]])
    out = oracle.topk(s, np.array([6, 6], dtype=np.int32), 3)
    assert out[0].tolist() == [0, 1, 4]
    assert out[1].tolist() == [0, 1, 2]


def test_ties_go_to_the_lower_positions():
    s = torch.zeros(2, 500)
    s[1, 300:] = 1.0  # 200 top scores tied, topk 50: the 50 lowest of them
    out = oracle.topk(s, np.array([500, 500], dtype=np.int32), 50)
    assert out[0].tolist() == list(range(50))
    assert out[1].tolist() == list(range(300, 350))


def test_block_table_maps_positions_to_slots():
    s = _scores(2, 640, seed=2)
    table = torch.randperm(10, generator=torch.Generator().manual_seed(3)).to(torch.int32) + 5
    pos = oracle.topk(s, np.array([640, 333], dtype=np.int32), 32)
    slots = oracle.topk(s, np.array([640, 333], dtype=np.int32), 32, block_table=table)
    tb = table.numpy()
    assert np.array_equal(slots, tb[pos // 64] * 64 + pos % 64)


_MUTANTS = {
    "bottom_k": (r"if \(x->score > y->score\) return -1;\n    if \(x->score < y->score\) return 1;",
                 "if (x->score < y->score) return -1;\n    if (x->score > y->score) return 1;"),
    "history_ignored": (r"const int64_t n = len\[t\];", "const int64_t n = S;"),
    "ties_to_higher_position": (r"return \(x->pos > y->pos\) - \(x->pos < y->pos\);\n\}\n\nstatic int oracle_by_pos",
                                "return (x->pos < y->pos) - (x->pos > y->pos);\n}\n\nstatic int oracle_by_pos"),
}


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_topk_mutants_fail_a_pin(tmp_path, monkeypatch, name):
    src = Path(oracle.__file__).with_name("sparse_mla_oracle.c").read_text()
    pat, rep = _MUTANTS[name]
    mutated, k = re.subn(pat, rep, src)
    assert k == 1, f"mutation {name} did not apply"
    c = tmp_path / f"{name}.c"
    c.write_text(mutated)
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    good = oracle._load()
    for fn in ("oracle_topk", "oracle_max_threads"):
        getattr(lib, fn).restype = getattr(good, fn).restype
        getattr(lib, fn).argtypes = getattr(good, fn).argtypes
    monkeypatch.setattr(oracle, "_lib", lib)
    pins = [lambda: test_matches_torch_topk_as_sets(4, 300, 16), test_short_history_selects_all_and_pads,
            test_ties_go_to_the_lower_positions, test_block_table_maps_positions_to_slots]
    failures = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught the mutant {name}"


# ----------------------------------------------------------------------------- C ABI (no GPU)

@pytest.fixture(scope="module")
def lib():
    import token_sparse_mla_gb300 as smla
    return smla.library()


@pytest.mark.parametrize("T,S,k", [(-1, 100, 8), (4, 0, 8), (4, 100, 0), (4, 100, (1 << 20) + 1)])
def test_topk_rejects_bad_sizes(lib, T, S, k):
    buf = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    assert lib.sparse_mla_topk(buf, T, S, buf, k, None, buf, None) == 1


def test_topk_rejects_null_and_misaligned(lib):
    good = ctypes.c_void_p(4096)
    assert lib.sparse_mla_topk(None, 4, 100, good, 8, None, good, None) == 1
    assert lib.sparse_mla_topk(ctypes.c_void_p(4098), 4, 100, good, 8, None, good, None) == 1
    assert lib.sparse_mla_topk(good, 4, 100, good, 8, ctypes.c_void_p(4097), good, None) == 1


def test_topk_zero_rows_is_a_noop(lib):
    assert lib.sparse_mla_topk(None, 0, 100, None, 8, None, None, None) == 0


# ----------------------------------------------------------------------------- GPU parity

DEV = "cuda:0"


@pytest.mark.gpu
@pytest.mark.parametrize("T,S,k,mode", [(4, 300, 16, "rand"), (3, 5000, 2048, "rand"), (6, 2047, 2048, "rand"),
                                        (5, 4096, 2048, "ties"), (2, 70000, 2048, "rand"), (8, 1000, 1, "rand"),
                                        (3, 3000, 777, "quant"), (16, 33000, 2048, "rand"),
                                        # more equal keys in the threshold's top-11-bit bin than the
                                        # shared-memory candidate buffer holds (the row-scan path)
                                        (3, 20000, 2048, "ties"), (2, 70000, 3000, "quant"),
                                        (4, 9000, 1000, "neg"),
                                        # equal +0 and -0 at the threshold, on the candidate path
                                        # (few keys in the threshold's bin) and the row-scan path
                                        (3, 3000, 1000, "zeros"), (3, 9000, 3000, "zeros"),
                                        # the threshold at -inf: candidates from the lowest bins
                                        (3, 3000, 1000, "neginf"), (3, 9000, 2048, "neginf"),
                                        (3, 3000, 777, "denorm"), (4, 20000, 2048, "rising"),
                                        # rows that do not start on a 16-byte boundary
                                        (5, 9999, 1500, "rand"), (3, 4097, 2048, "rand")])
def test_gpu_topk_matches_oracle_exactly(T, S, k, mode):
    import token_sparse_mla_gb300 as smla
    s = _scores(T, S, seed=S + k)
    if mode == "ties":
        s = torch.zeros(T, S)
        s[:, ::3] = 1.0  # many equal scores at the threshold
    elif mode == "quant":
        s = torch.round(s * 4) / 4  # few distinct values: ties everywhere
    elif mode == "neg":
        s = -s.abs() - 1.0  # every score negative: the low bins of the key
    elif mode == "zeros":
        z = torch.where(torch.rand(T, S, generator=torch.Generator().manual_seed(S)) < 0.5, -0.0, 0.0)
        s = torch.where(s < 0.5, z, s)  # about 69 % zeros of either sign
    elif mode == "neginf":
        s = torch.where(torch.rand(T, S, generator=torch.Generator().manual_seed(S)) < 0.9, -math.inf, s)
    elif mode == "denorm":
        s = s * 1e-39  # subnormal scores (and their zeros)
    elif mode == "rising":
        s = torch.arange(S, dtype=torch.float32) * 1e-3 + s * 1e-2  # the top near the row's end
    g = torch.Generator().manual_seed(T + k)
    lens = torch.randint(0, S + 1, (T,), generator=g).to(torch.int32)
    lens[0] = S
    if T > 1:
        lens[1] = min(S, k - 1)  # a short history
    table = (torch.randperm((S + 63) // 64, generator=g).to(torch.int32) + 3)
    for bt in (None, table):
        out = smla.sparse_mla_topk(s.to(DEV), lens.to(DEV), k, block_table=None if bt is None else bt.to(DEV))
        smla.sync_status()
        ref = oracle.topk(s, lens, k, block_table=bt)
        assert np.array_equal(out.cpu().numpy(), ref), f"T={T} S={S} k={k} {mode} table={bt is not None}"


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["rand", "zeros", "neginf", "denorm", "rising", "ties"])
@pytest.mark.parametrize("k", [1000, 2048])
def test_gpu_topk_long_rows_mixed_histories(mode, k):
    """Long rows (S = 40003, off the 16-byte boundary): histories short and long in one launch,
    each special score set, on both the candidate path and the row-scan path."""
    import token_sparse_mla_gb300 as smla
    S = 40000 + 3  # rows off the 16-byte boundary too
    lens = torch.tensor([S, 3000, 9000, k - 1, 33000, 4100], dtype=torch.int32)
    T = lens.numel()
    g = torch.Generator().manual_seed(k)
    s = torch.randn(T, S, generator=g)
    if mode == "zeros":
        z = torch.where(torch.rand(T, S, generator=g) < 0.5, -0.0, 0.0)
        s = torch.where(s < 0.5, z, s)
    elif mode == "neginf":
        s = torch.where(torch.rand(T, S, generator=g) < 0.9, -math.inf, s)
    elif mode == "denorm":
        s = s * 1e-39
    elif mode == "rising":
        s = torch.arange(S, dtype=torch.float32) * 1e-3 + s * 1e-2
    elif mode == "ties":
        s = torch.round(s * 4) / 4
    out = smla.sparse_mla_topk(s.to(DEV), lens.to(DEV), k)
    smla.sync_status()
    assert np.array_equal(out.cpu().numpy(), oracle.topk(s, lens, k)), mode


@pytest.mark.gpu
@pytest.mark.parametrize("in_bin", [2095, 2096, 2097])
def test_gpu_topk_candidate_capacity_edge(in_bin):
    """2000 scores above the threshold's 12-bit bin and in_bin in it, k = 2048: 4095 or 4096
    candidates take the candidate path, 4097 the row scan; both exact."""
    import token_sparse_mla_gb300 as smla
    T, S, k = 2, 12000, 2048
    g = torch.Generator().manual_seed(in_bin)
    s = torch.rand(T, S, generator=g) * 0.5  # below the bin [1, 1.125)
    for t in range(T):
        perm = torch.randperm(S, generator=g)
        s[t, perm[:2000]] = 10.0 + torch.rand(2000, generator=g)
        vals = 1.0 + torch.floor(torch.rand(in_bin, generator=g) * 300) / 2400  # ties inside the bin
        s[t, perm[2000:2000 + in_bin]] = vals
    lens = torch.full((T,), S, dtype=torch.int32)
    out = smla.sparse_mla_topk(s.to(DEV), lens.to(DEV), k)
    smla.sync_status()
    assert np.array_equal(out.cpu().numpy(), oracle.topk(s, lens, k))


@pytest.mark.gpu
def test_gpu_topk_feeds_the_forward():
    """Scores -> GPU top-k (slots through the block table) -> GPU forward, against the oracle
    forward on the oracle's lists: the lists must be identical and the outputs within the
    forward's tolerance."""
    import token_sparse_mla_gb300 as smla
    from tests.parity import assert_parity
    from workloads import make_workload
    w = make_workload("prefill", n_tokens=8)
    S = w.num_slots  # one sequence: positions 0 .. 32767
    g = torch.Generator().manual_seed(77)
    scores = torch.randn(w.T, S, generator=g)
    lens = torch.arange(S - w.T + 1, S + 1, dtype=torch.int32)[: w.T]  # causal histories
    table = torch.randperm(S // 64, generator=g).to(torch.int32)
    idx_gpu = smla.sparse_mla_topk(scores.to(DEV), lens.to(DEV), w.topk, block_table=table.to(DEV))
    out, lse = smla.sparse_mla_fwd(w.q.to(DEV), w.kv.to(DEV), idx_gpu, w.scale)
    smla.sync_status()
    idx_ref = oracle.topk(scores, lens, w.topk, block_table=table)
    assert np.array_equal(idx_gpu.cpu().numpy(), idx_ref)
    ref_o, ref_l = oracle.sparse_mla_fwd(w.q, w.kv, torch.from_numpy(idx_ref), w.scale)
    assert_parity(out.cpu(), lse.cpu(), ref_o, ref_l, "topk -> forward")
