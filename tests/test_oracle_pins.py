"""Pins for the CPU oracle: each check comes from outside the oracle itself.

* brute force: dense-mask attention over the whole cache (tests/bruteforce.py),
  decoded through torch's conversions;
* closed forms: a single entry gives its own V row; a slot listed k times gives
  LSE + ln k; zero queries give the plain mean of the listed V rows and
  LSE = ln(n_valid); two entries give the logistic closed form;
* format definitions: every e4m3 code against torch's float8_e4m3fn and the
  format's fixed points (max 448, smallest subnormal 2^-9, NaN codes);
* mutation: mutated copies of the oracle source (a dropped rope term, a shifted
  value slice, base-2 LSE, a lost scale, -1 read as a slot, a wrong fp8 tile)
  must each fail at least one of the pins above.
"""

import math
import re
import subprocess
import ctypes
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from tests.bruteforce import dense_attention, decode_cache
from workloads import make_workload, quantize_fp8_rows

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_case(seed, T, h, topk, num_slots, kv_format="bf16", p_invalid=0.1, dup=True):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(T, h, 576, generator=g) * 0.5).to(torch.bfloat16)
    x = torch.randn(num_slots, 576, generator=g) * 0.5
    kv = x.to(torch.bfloat16) if kv_format == "bf16" else quantize_fp8_rows(x)
    if dup:
        idx = torch.randint(0, num_slots, (T, topk), generator=g)
    else:
        idx = torch.stack([torch.randperm(num_slots, generator=g)[:topk] for _ in range(T)])
    drop = torch.rand(T, topk, generator=g) < p_invalid
    idx = idx.masked_fill(drop, -1)
    # a few out-of-range and other negative values: masked like -1
    if topk >= 4:
        idx[0, 0] = num_slots
        idx[-1, 1] = -7
    return q, kv, idx.to(torch.int32)


def _check(out, lse, ref_out, ref_lse, atol=1e-10):
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=atol)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.all(lse[~fin] == -np.inf)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=atol)


# ----------------------------------------------------------------------------- brute force

def test_tiny_config_matches_bruteforce():
    w = make_workload("tiny")
    out, lse = oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale)
    ref_out, ref_lse = dense_attention(w.q, w.kv, w.indices, w.scale)
    _check(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("seed,T,h,topk,S", [(1, 3, 8, 37, 50), (2, 5, 16, 64, 300),
                                             (3, 2, 64, 130, 1000), (4, 4, 32, 7, 5)])
def test_random_with_duplicates_and_invalid(seed, T, h, topk, S):
    q, kv, idx = _rand_case(seed, T, h, topk, S)
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 576 ** -0.5)
    ref_out, ref_lse = dense_attention(q, kv, idx, 576 ** -0.5)
    _check(out, lse, ref_out, ref_lse)


def test_fp8_rows_match_bruteforce():
    q, kv, idx = _rand_case(11, 4, 8, 96, 400, kv_format="fp8")
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 576 ** -0.5, kv_format="fp8")
    ref_out, ref_lse = dense_attention(q, kv, idx, 576 ** -0.5, kv_format="fp8")
    _check(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("name,kw", [("decode_bf16", dict(n_seq=2)),
                                     ("sweep", dict(n_seq=2, h=16)),
                                     ("prefill", dict(n_tokens=2, topk=256)),
                                     ("fp8_mixed", dict(n_seq=1, n_tokens=2, topk=256))])
def test_reduced_configs_match_bruteforce(name, kw):
    w = make_workload(name, **kw)
    out, lse = oracle.sparse_mla_fwd(w.q, w.kv, w.indices, w.scale, kv_format=w.kv_format)
    ref_out, ref_lse = dense_attention(w.q, w.kv, w.indices, w.scale, kv_format=w.kv_format)
    _check(out, lse, ref_out, ref_lse)


def test_token_subset_equals_full():
    q, kv, idx = _rand_case(5, 6, 8, 40, 90)
    full_o, full_l = oracle.sparse_mla_fwd(q, kv, idx, 0.1)
    sub_o, sub_l = oracle.sparse_mla_fwd(q, kv, idx, 0.1, tokens=[4, 1])
    assert np.array_equal(sub_o, full_o[[4, 1]])
    assert np.array_equal(sub_l, full_l[[4, 1]])


# ----------------------------------------------------------------------------- closed forms

def test_single_entry_returns_its_value_row():
    q, kv, _ = _rand_case(6, 3, 8, 4, 64)
    idx = torch.tensor([[17], [0], [63]], dtype=torch.int32)
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 576 ** -0.5)
    K = kv.float().double().numpy()
    for t, slot in enumerate([17, 0, 63]):
        assert np.array_equal(out[t], np.broadcast_to(K[slot, :512], (8, 512)))
    # LSE of a single logit is the logit itself; compare with the brute force's logit
    _, ref_lse = dense_attention(q, kv, idx, 576 ** -0.5)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12, rtol=0)


def test_duplicate_row_k_times():
    q, kv, _ = _rand_case(7, 2, 16, 4, 32)
    one = torch.tensor([[5], [9]], dtype=torch.int32)
    o1, l1 = oracle.sparse_mla_fwd(q, kv, one, 0.3)
    for k in (2, 3, 8):
        rep = one.repeat(1, k)
        ok, lk = oracle.sparse_mla_fwd(q, kv, rep, 0.3)
        np.testing.assert_allclose(ok, o1, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lk, l1 + math.log(k), atol=1e-12, rtol=0)
        # with invalid entries interleaved the answer does not change
        mixed = torch.cat([rep, torch.full_like(rep, -1)], dim=1)
        om, lm = oracle.sparse_mla_fwd(q, kv, mixed[:, torch.randperm(2 * k)], 0.3)
        np.testing.assert_allclose(om, o1, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lm, l1 + math.log(k), atol=1e-12, rtol=0)


def test_all_invalid_gives_zero_and_neg_inf():
    q, kv, _ = _rand_case(8, 2, 8, 4, 16)
    idx = torch.tensor([[-1] * 6, [-1, 16, -3, 99, -1, -1]], dtype=torch.int32)
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 0.5)
    assert np.all(out == 0.0)
    assert np.all(lse == -np.inf)


def test_permutation_invariance():
    q, kv, idx = _rand_case(9, 4, 8, 200, 500)
    o1, l1 = oracle.sparse_mla_fwd(q, kv, idx, 576 ** -0.5)
    g = torch.Generator().manual_seed(1)
    perm = torch.stack([torch.randperm(200, generator=g) for _ in range(4)])
    idx2 = torch.gather(idx, 1, perm)
    o2, l2 = oracle.sparse_mla_fwd(q, kv, idx2, 576 ** -0.5)
    np.testing.assert_allclose(o2, o1, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l2, l1, atol=1e-12, rtol=0)


def test_zero_query_gives_mean_and_log_count():
    """q = 0: every logit is 0, so O is the plain mean of the listed V rows
    (integers here, so the mean is exact) and LSE = ln(number of valid entries)."""
    S, topk = 40, 25
    g = torch.Generator().manual_seed(10)
    vals = torch.randint(-8, 9, (S, 576), generator=g).to(torch.float32)
    kv = vals.to(torch.bfloat16)
    q = torch.zeros(3, 8, 576, dtype=torch.bfloat16)
    idx = torch.randint(0, S, (3, topk), generator=g)
    idx[1, :10] = -1
    idx[2, :] = -1
    idx[2, 3] = 7
    idx = idx.to(torch.int32)
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 576 ** -0.5)
    V = vals.numpy().astype(np.int64)
    for t in range(3):
        sel = [int(s) for s in idx[t] if s >= 0]
        n = len(sel)
        exact_sum = V[sel, :512].sum(axis=0)              # integer arithmetic
        assert np.all(out[t] == np.broadcast_to(exact_sum / n, (8, 512)))
        assert np.all(np.abs(lse[t] - math.log(n)) <= 1e-15 * max(1.0, math.log(n)) + 1e-15)


def test_two_entries_logistic_closed_form():
    """q = a e_575 (a rope dim), rows r1 = b1 e_575 + V1, r2 = b2 e_575 + V2 with V in
    the first 512 dims: s_i = scale a b_i and O = sigma(s1 - s2) V1 + sigma(s2 - s1) V2,
    LSE = log(e^s1 + e^s2)."""
    g = torch.Generator().manual_seed(12)
    a, b1, b2, scale = 2.0, 3.0, -1.5, 0.25
    kvf = torch.zeros(2, 576)
    kvf[:, :512] = torch.randint(-4, 5, (2, 512), generator=g).float()
    kvf[0, 575], kvf[1, 575] = b1, b2
    kv = kvf.to(torch.bfloat16)
    q = torch.zeros(1, 8, 576)
    q[0, :, 575] = a
    q = q.to(torch.bfloat16)
    idx = torch.tensor([[0, 1]], dtype=torch.int32)
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, scale)
    s1, s2 = scale * a * b1, scale * a * b2
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    exp_o = w1 * kvf[0, :512].double().numpy() + (1 - w1) * kvf[1, :512].double().numpy()
    np.testing.assert_allclose(out[0], np.broadcast_to(exp_o, (8, 512)), atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse[0], np.logaddexp(s1, s2), atol=1e-14, rtol=0)


def test_rope_dims_enter_logits_not_values():
    """A query that only touches rope dims still changes the weights; a row that only
    differs in rope dims has the same value row."""
    kvf = torch.zeros(2, 576)
    kvf[0, :512] = 1.0
    kvf[1, :512] = 3.0
    kvf[0, 512:] = 0.5
    kvf[1, 512:] = -0.5
    kv = kvf.to(torch.bfloat16)
    q = torch.zeros(1, 8, 576)
    q[0, :, 512:] = 1.0
    q = q.to(torch.bfloat16)
    idx = torch.tensor([[0, 1]], dtype=torch.int32)
    out, lse = oracle.sparse_mla_fwd(q, kv, idx, 1.0)
    s1, s2 = 32.0, -32.0
    w1 = 1.0 / (1.0 + math.exp(s2 - s1))
    np.testing.assert_allclose(out[0, 0, 0], w1 * 1.0 + (1 - w1) * 3.0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.logaddexp(s1, s2), atol=1e-14)


# ----------------------------------------------------------------------------- number formats

def test_e4m3_table_matches_torch_and_format_points():
    tab = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan)
    assert sorted(np.nonzero(nan)[0].tolist()) == [0x7F, 0xFF]
    assert np.array_equal(tab[~nan], ref[~nan])
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0
    assert tab[0x01] == 2.0 ** -9
    assert tab[0x08] == 2.0 ** -6        # smallest normal
    assert tab[0x38] == 1.0
    assert np.nanmax(np.abs(tab)) == 448.0


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(13)
    bits = torch.randint(0, 65536, (4000,), generator=g, dtype=torch.int64)
    vals = bits.to(torch.int32).to(torch.int16).view(torch.bfloat16).float().double().numpy()
    for b, v in zip(bits.tolist()[:4000:7], vals[:4000:7]):
        got = oracle.bf16_value(b)
        if math.isnan(v):
            assert math.isnan(got)
        else:
            assert got == v


def test_fp8_row_decode_round_trip():
    g = torch.Generator().manual_seed(14)
    x = torch.randn(6, 576, generator=g) * 0.5
    x[2, 128:256] = 0.0                      # an all-zero tile takes scale 1
    rows = quantize_fp8_rows(x)
    dec_torch = decode_cache(rows, "fp8")
    for r in range(6):
        d = oracle.decode_row(rows, "fp8", r)
        assert np.array_equal(d, dec_torch[r])
        # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 of the tile max, per element
        lat = x[r, :512].double().numpy().reshape(4, 128)
        amax = np.abs(lat).max(axis=1, keepdims=True)
        err = np.abs(d[:512].reshape(4, 128) - lat)
        assert np.all(err <= np.maximum(amax, 1e-30) * 2.0 ** -4 + 1e-12)
        assert np.array_equal(d[512:], x[r, 512:].to(torch.bfloat16).double().numpy())
    assert np.all(oracle.decode_row(rows, "fp8", 2)[128:256] == 0.0)


# ----------------------------------------------------------------------------- mutation

_MUTANTS = {
    "rope_dropped": (r"for \(int d = 0; d < ORACLE_DQK; \+\+d\) dot \+=",
                     "for (int d = 0; d < ORACLE_DV; ++d) dot +="),
    "value_slice_shifted": (r"acc\[d\] \+= w \* row\[d\];", "acc[d] += w * row[d + 64];"),
    "lse_base2": (r"lse\[i \* h \+ hh\] = m \+ log\(l\);", "lse[i * h + hh] = m + log2(l);"),
    "scale_lost": (r"s\[j\] = scale \* dot;", "s[j] = dot;"),
    "minus_one_is_slot_zero": (r"if \(slot < 0 \|\| slot >= num_slots\) continue;",
                               "if (slot >= num_slots) continue; if (slot < 0) slot = 0;"),
    "fp8_tile_64": (r"tile_scale\[d / 128\]", "tile_scale[(d / 64) % 4]"),
    "max_not_subtracted_in_lse": (r"m \+ log\(l\)", "log(l)"),
}


def _build_mutant(tmp_path, name):
    src = Path(oracle.__file__).with_name("sparse_mla_oracle.c").read_text()
    pat, rep = _MUTANTS[name]
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation {name} did not apply"
    c = tmp_path / f"{name}.c"
    c.write_text(mutated)
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(c), "-lm"], check=True)
    return so


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_mutants_fail_a_pin(tmp_path, monkeypatch, name):
    so = _build_mutant(tmp_path, name)
    lib = ctypes.CDLL(str(so))
    lib.oracle_sparse_mla_fwd.restype = ctypes.c_int
    lib.oracle_sparse_mla_fwd.argtypes = oracle._load().oracle_sparse_mla_fwd.argtypes
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_e4m3_table.argtypes = [ctypes.c_void_p]
    lib.oracle_bf16_value.restype = ctypes.c_double
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_row.argtypes = oracle._load().oracle_decode_row.argtypes
    monkeypatch.setattr(oracle, "_lib", lib)
    pins = [test_tiny_config_matches_bruteforce, test_fp8_rows_match_bruteforce,
            test_two_entries_logistic_closed_form, test_zero_query_gives_mean_and_log_count,
            test_fp8_row_decode_round_trip, test_all_invalid_gives_zero_and_neg_inf,
            lambda: test_random_with_duplicates_and_invalid(2, 5, 16, 64, 300)]
    failures = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught the mutant {name}"
