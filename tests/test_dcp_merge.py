"""The merge of split-list partial results (the DCP merge): oracle pins on the CPU, C-ABI
validation, and GPU parity through sparse_mla_merge.

A token's top-k list split into disjoint parts, each part's (O_p, LSE_p) as the forward
returns them, merged: the result must be the forward of the whole list (vLLM PR #60220,
Details: out and lse are consumed by the DCP merge).  Pins of the oracle merge, each from
outside the merge itself:

* union: the forward oracle on the whole list equals the merge of the forward oracle on
  its parts, including an all-invalid part, to fp64 rounding;
* closed forms: one part comes back unchanged; two equal parts give the same O and
  LSE + ln 2; a row whose parts are all empty gives O = 0, LSE = -inf;
* the order of the parts does not matter;
* mutation: mutated copies of the merge (unnormalised weights, base-2 LSE, a part left out
  of the normaliser) each fail one of these.
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
from workloads import make_merge_parts, make_workload, split_lists

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _split_forward(w, n):
    """Forward oracle (fp64) of each part of w's lists: o [n, T, h, 512], lse [n, T, h]."""
    os_, ls_ = [], []
    for part in split_lists(w.indices, n):
        o, l = oracle.sparse_mla_fwd(w.q, w.kv, part, w.scale, kv_format=w.kv_format)
        os_.append(o)
        ls_.append(l)
    return np.stack(os_), np.stack(ls_)


# ----------------------------------------------------------------------------- oracle pins

@pytest.mark.parametrize("n", [2, 3, 8])
def test_merge_of_parts_equals_whole_list(n):
    w = make_workload("tiny")  # last 8 entries of each list are -1: with n = 8 a part is empty
    o_parts, l_parts = _split_forward(w, n)
    if n == 8:
        assert np.all(np.isneginf(l_parts[-1]))
    out, lse = oracle.merge(o_parts, l_parts)
    ref_out, ref_lse = oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale)
    assert np.allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_merge_of_parts_with_duplicates_and_fp8():
    g = torch.Generator().manual_seed(41)
    w = make_workload("tiny")
    # duplicates across parts are separate softmax terms, so the union still holds
    idx = torch.randint(0, w.num_slots, (w.T, 40), generator=g).to(torch.int32)
    idx[:, ::7] = -1
    o_parts, l_parts = [], []
    for part in split_lists(idx, 4):
        o, l = oracle.sparse_mla_fwd(w.q, w.kv, part, w.scale)
        o_parts.append(o)
        l_parts.append(l)
    out, lse = oracle.merge(np.stack(o_parts), np.stack(l_parts))
    ref_out, ref_lse = oracle.sparse_mla_fwd(w.q, w.kv, idx, w.scale)
    assert np.allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    wf = make_workload("fp8_mixed", n_seq=1, n_tokens=4)
    o_parts, l_parts = _split_forward(wf, 3)
    out, lse = oracle.merge(o_parts, l_parts)
    ref_out, ref_lse = oracle.sparse_mla_fwd(wf.q, wf.kv, wf.indices, wf.scale, kv_format="fp8")
    assert np.allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_single_part_is_returned_unchanged():
    o, l = make_merge_parts(1, 3, 8, seed=1)
    out, lse = oracle.merge(o, l)
    ref = o[0].float().double().numpy()
    assert np.array_equal(out, ref)
    assert np.array_equal(lse, l[0].double().numpy())


def test_two_equal_parts_add_ln2():
    o, l = make_merge_parts(1, 3, 8, seed=2, p_empty=0.0)
    o2, l2 = torch.cat([o, o]), torch.cat([l, l])
    out, lse = oracle.merge(o2, l2)
    ref_l = l[0].double().numpy()
    fin = np.isfinite(ref_l)
    assert np.allclose(out, o[0].float().double().numpy(), rtol=1e-15, atol=1e-15)
    assert np.allclose(lse[fin], ref_l[fin] + math.log(2.0), rtol=0, atol=1e-12)
    assert np.all(np.isneginf(lse[~fin]))


def test_all_empty_parts_give_zero_and_neg_inf():
    o, l = make_merge_parts(5, 2, 8, seed=3)
    l[:, 1] = float("-inf")
    o[:, 1] = 1.0  # whatever an empty part holds, it weighs nothing
    out, lse = oracle.merge(o, l)
    assert np.all(np.isneginf(lse[1])) and np.all(out[1] == 0.0)
    assert np.all(np.isneginf(lse[:, 0])) and np.all(out[:, 0] == 0.0)  # empty in every part


def test_part_order_does_not_matter():
    o, l = make_merge_parts(6, 3, 8, seed=4)
    perm = torch.tensor([3, 0, 5, 1, 4, 2])
    a_out, a_lse = oracle.merge(o, l)
    b_out, b_lse = oracle.merge(o[perm], l[perm])
    assert np.allclose(a_out, b_out, rtol=1e-13, atol=1e-15)
    fin = np.isfinite(a_lse)
    assert np.array_equal(fin, np.isfinite(b_lse))
    assert np.allclose(a_lse[fin], b_lse[fin], rtol=0, atol=1e-12)


_MUTANTS = {
    "merge_weights_unnormalised": (r"double w = exp\(l - total\);", "double w = exp(l - m);"),
    "merge_lse_base2": (r"double total = m \+ log\(sum\);", "double total = m + log2(sum);"),
    "merge_normaliser_skips_part0": (r"for \(int p = 0; p < n; \+\+p\) \{\n            double l = lse_parts\[p \* rows \+ r\];\n            if \(l != -INFINITY\) sum",
                                     "for (int p = 1; p < n; ++p) {\n            double l = lse_parts[p * rows + r];\n            if (l != -INFINITY) sum"),
}


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_merge_mutants_fail_a_pin(tmp_path, monkeypatch, name):
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
    for fn in ("oracle_sparse_mla_fwd", "oracle_merge", "oracle_max_threads"):
        getattr(lib, fn).restype = getattr(good, fn).restype
        getattr(lib, fn).argtypes = getattr(good, fn).argtypes
    monkeypatch.setattr(oracle, "_lib", lib)
    pins = [lambda: test_merge_of_parts_equals_whole_list(3), test_two_equal_parts_add_ln2,
            test_single_part_is_returned_unchanged, test_all_empty_parts_give_zero_and_neg_inf]
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


@pytest.mark.parametrize("n,T,h,status", [(0, 4, 8, 1), (17, 4, 8, 1), (4, -1, 8, 1), (4, 4, 0, 1)])
def test_merge_rejects_bad_arguments(lib, n, T, h, status):
    buf = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    assert lib.sparse_mla_merge(buf, buf, n, T, h, buf, buf, None) == status


def test_merge_rejects_null_and_misaligned(lib):
    good = ctypes.c_void_p(4096)
    assert lib.sparse_mla_merge(None, good, 2, 4, 8, good, good, None) == 1
    assert lib.sparse_mla_merge(ctypes.c_void_p(4104), good, 2, 4, 8, good, good, None) == 1
    assert lib.sparse_mla_merge(good, good, 2, 4, 8, ctypes.c_void_p(4100), good, None) == 1


def test_merge_zero_tokens_is_a_noop(lib):
    assert lib.sparse_mla_merge(None, None, 2, 0, 8, None, None, None) == 0


# ----------------------------------------------------------------------------- GPU parity

DEV = "cuda:0"


def _gpu_merge(o, l):
    import token_sparse_mla_gb300 as smla
    out, lse = smla.sparse_mla_merge(o.to(DEV), l.to(DEV))
    smla.sync_status()
    return out.cpu(), lse.cpu()


def _assert_merge_parity(out, lse, ref_out, ref_lse, what):
    o = out.float().double().numpy()
    l = lse.double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(l), ~fin), f"{what}: -inf pattern"
    assert np.all(o[~fin] == 0.0), f"{what}: empty rows must be 0"
    # fp32 weights and sums, one bf16 rounding of the result
    err = np.abs(o - ref_out)
    assert np.all(err <= 1e-5 + 2.0 ** -8 * np.abs(ref_out)), f"{what}: O max err {err.max()}"
    assert np.all(np.abs(l[fin] - ref_lse[fin]) <= 1e-5 * np.maximum(1.0, np.abs(ref_lse[fin]))), what


@pytest.mark.gpu
@pytest.mark.parametrize("n,T,h", [(1, 5, 8), (2, 3, 16), (4, 37, 8), (8, 9, 64), (16, 4, 32),
                                   (3, 1, 1), (5, 301, 8)])
def test_gpu_merge_matches_oracle(n, T, h):
    o, l = make_merge_parts(n, T, h, seed=100 + n * 7 + T)
    out, lse = _gpu_merge(o, l)
    ref_out, ref_lse = oracle.merge(o, l)
    _assert_merge_parity(out, lse, ref_out, ref_lse, f"n={n} T={T} h={h}")


@pytest.mark.gpu
def test_gpu_merge_single_part_is_exact():
    o, l = make_merge_parts(1, 7, 8, seed=5)
    out, lse = _gpu_merge(o, l)
    assert torch.equal(out, o[0]) and torch.equal(lse, l[0])


@pytest.mark.gpu
@pytest.mark.parametrize("name,kw,n", [("decode_bf16", {"n_seq": 4}, 4), ("sweep", {"h": 16, "n_seq": 3}, 2),
                                        ("sweep", {"h": 64, "n_seq": 2}, 8), ("fp8_mixed", {"n_seq": 1, "n_tokens": 6}, 3)])
def test_gpu_split_forward_then_merge_equals_whole_forward(name, kw, n):
    """The forward on each part of the lists, merged on the GPU, against the forward of the
    whole lists: the oracle's, and the GPU's own."""
    import token_sparse_mla_gb300 as smla
    from tests.parity import assert_parity
    w = make_workload(name, **kw)
    q, kv = w.q.to(DEV), w.kv.to(DEV)
    o_parts, l_parts = [], []
    for part in split_lists(w.indices, n):
        o, l = smla.sparse_mla_fwd(q, kv, part.to(DEV), w.scale, kv_format=w.kv_format)
        o_parts.append(o)
        l_parts.append(l)
    out, lse = smla.sparse_mla_merge(torch.stack(o_parts), torch.stack(l_parts))
    full_out, full_lse = smla.sparse_mla_fwd(q, kv, w.indices.to(DEV), w.scale, kv_format=w.kv_format)
    smla.sync_status()
    ref_out, ref_lse = oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, kv_format=w.kv_format)
    assert_parity(out.cpu(), lse.cpu(), ref_out, ref_lse, f"{name} merged")
    # against the unsplit GPU forward: both within the tolerance of the same reference
    assert_parity(full_out.cpu(), full_lse.cpu(), ref_out, ref_lse, f"{name} whole")
