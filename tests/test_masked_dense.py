"""The masked dense route for short prefill: oracle pins on the CPU.

The per-token lists are scattered into a bit mask over the request's positions and a dense
MHA runs over the decompressed per-head K and V under that mask (PR #55738 report, 实现拆解
(implementation breakdown) items 2 and 5: a scatter of the top-k lists and a `mask_mod`
masked MHA take the prefill instead of the per-token sparse kernel).  Pins of the two oracle
functions, each from outside them:

* the mask against numpy's own scatter and little-endian bit packing;
* the masked MHA against torch's float64 scaled_dot_product_attention with a boolean mask,
  and, for lists that hold whole causal histories, with torch's own causal mask;
* closed forms: one position returns its value row and its scaled logit as LSE; equal keys
  give the mean of the values and logit + ln(count); an empty row gives O = 0, LSE = -inf;
* the MLA absorption identity: attention over decompressed K = [W_UK c ; rope] and
  V = W_UV c equals the sparse forward oracle over the latent cache with the absorbed query,
  followed by W_UV, for the DeepSeek-V3.2, GLM-5 and NoPE geometries of the report's
  `_is_masked_mha_available` table; with every position listed twice the sparse LSE is
  ln 2 above the masked one (the mask holds a set, the sparse lists a multiset);
* mutation: mutated copies of the oracle each fail one of these.
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
from workloads import causal_position_lists, make_masked_dense_inputs


def _f64(x):
    return x.double().numpy()  # bf16 -> fp64 is exact


def _bool_mask(lists, S):
    """Dense boolean mask of the lists, built with numpy indexing."""
    li = lists.numpy().astype(np.int64)
    T = li.shape[0]
    m = np.zeros((T, S), dtype=bool)
    rows = np.repeat(np.arange(T), li.shape[1])
    cols = li.ravel()
    ok = (cols >= 0) & (cols < S)
    m[rows[ok], cols[ok]] = True
    return m


def _sdpa(q, k, v, allowed, scale):
    """torch float64 scaled_dot_product_attention, heads as the batch: [T, h, dv]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2)
    vt = torch.from_numpy(v).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(allowed), scale=scale)
    return o.permute(1, 0, 2).numpy()


# ----------------------------------------------------------------------------- the mask

@pytest.mark.parametrize("T,S,topk", [(5, 8, 3), (16, 100, 40), (3, 32, 32), (7, 65, 70)])
def test_mask_matches_numpy_scatter(T, S, topk):
    lists = causal_position_lists(T, S, topk, seed=T + S, p_empty=0.2)
    lists[0, 0] = S            # out of range: sets nothing
    lists[-1, -1] = -5         # negative: sets nothing
    mask = oracle.scatter_mask(lists, S)
    W = (S + 31) // 32
    packed = np.packbits(_bool_mask(lists, S), axis=1, bitorder="little")
    packed = np.pad(packed, ((0, 0), (0, 4 * W - packed.shape[1])))
    ref = packed.view("<u4")
    assert mask.shape == (T, W)
    assert np.array_equal(mask, ref)


def test_mask_of_a_repeated_position_is_one_bit():
    lists = torch.tensor([[3, 3, 3, -1], [0, 31, 32, 0]], dtype=torch.int32)
    mask = oracle.scatter_mask(lists, 40)
    assert mask.tolist() == [[1 << 3, 0], [1 | (1 << 31), 1]]


# ----------------------------------------------------------------------------- masked MHA

@pytest.mark.parametrize("T,S,h,dqk,dv,topk", [(12, 80, 3, 192, 128, 24), (9, 40, 2, 256, 256, 16),
                                              (20, 33, 4, 64, 32, 5)])
def test_masked_mha_matches_torch_sdpa(T, S, h, dqk, dv, topk):
    q, k, v = make_masked_dense_inputs(T, S, h, dqk, dv, seed=T * 7 + h)
    lists = causal_position_lists(T, S, topk, seed=S, p_empty=0.15)
    scale = dqk ** -0.5
    out, lse = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), scale)
    allowed = _bool_mask(lists, S)
    live = allowed.any(axis=1)
    assert live.any() and not live.all()
    ref = _sdpa(_f64(q), _f64(k), _f64(v), allowed, scale)
    assert np.allclose(out[live], ref[live], rtol=1e-11, atol=1e-13)
    assert np.all(out[~live] == 0.0)
    assert np.all(np.isneginf(lse[~live])) and np.all(np.isfinite(lse[live]))


@pytest.mark.parametrize("S,h,dqk,dv", [(48, 2, 192, 128), (70, 1, 256, 256)])
def test_full_histories_are_causal_attention(S, h, dqk, dv):
    """Short prefill: topk covers every history, so the lists are whole causal histories and
    the route is causal attention (torch's is_causal mask, T = S)."""
    q, k, v = make_masked_dense_inputs(S, S, h, dqk, dv, seed=S)
    lists = causal_position_lists(S, S, 2048, seed=S + 1)
    scale = dqk ** -0.5
    out, _ = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), scale)
    qt, kt, vt = (torch.from_numpy(_f64(x)).permute(1, 0, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                           scale=scale).permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_one_position_returns_its_value_row():
    T, S, h, dqk, dv = 6, 50, 3, 192, 128
    q, k, v = make_masked_dense_inputs(T, S, h, dqk, dv, seed=3)
    pick = [4, 49, 0, 17, 17, 32]
    lists = torch.full((T, 5), -1, dtype=torch.int32)
    lists[:, 2] = torch.tensor(pick, dtype=torch.int32)
    scale = 0.125
    out, lse = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), scale)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    for t, s in enumerate(pick):
        assert np.array_equal(out[t], vd[s])
        for hh in range(h):
            assert math.isclose(lse[t, hh], scale * float(np.dot(qd[t, hh], kd[s, hh])),
                                rel_tol=1e-13, abs_tol=1e-13)


def test_equal_keys_give_the_mean_of_the_values():
    T, S, h, dqk, dv = 5, 64, 2, 64, 48
    q, k, v = make_masked_dense_inputs(T, S, h, dqk, dv, seed=4)
    k[:] = k[7]
    lists = causal_position_lists(T, S, 20, seed=5)
    scale = 0.3
    out, lse = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), scale)
    allowed = _bool_mask(lists, S)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    for t in range(T):
        n = int(allowed[t].sum())
        for hh in range(h):
            assert np.allclose(out[t, hh], vd[allowed[t], hh].mean(axis=0), rtol=1e-12, atol=1e-14)
            logit = scale * float(np.dot(qd[t, hh], kd[0, hh]))
            assert math.isclose(lse[t, hh], logit + math.log(n), rel_tol=1e-12, abs_tol=1e-12)


# ----------------------------------------------------------------------------- absorption identity

def _absorbed_case(T, S, h, dn, dr, dv, topk, seed, repeat=1):
    """One MLA instance in both forms.  W_UK of head h maps latent dim sel[h, i] to key dim i
    with sign sgn[h, i] (a signed selection, so the absorbed query is exact in bf16); W_UV is
    dense.  Returns the masked route's result and the sparse route's, each (y, lse)."""
    g = torch.Generator().manual_seed(seed)
    c = (torch.randn(S, 576, generator=g) * 0.5).to(torch.bfloat16)
    sel = torch.stack([torch.randperm(512, generator=g)[:dn] for _ in range(h)])
    sgn = torch.where(torch.rand(h, dn, generator=g) < 0.5, -1.0, 1.0)
    q_nope = (torch.randn(T, h, dn, generator=g) * 0.5).to(torch.bfloat16)
    q_rope = (torch.randn(T, h, dr, generator=g) * 0.5).to(torch.bfloat16)
    w_uv = torch.randn(h, dv, 512, generator=g, dtype=torch.float64) / math.sqrt(512)

    cd = c.double()
    k = torch.empty(S, h, dn + dr, dtype=torch.float64)
    q_abs = torch.zeros(T, h, 576, dtype=torch.bfloat16)
    for hh in range(h):
        k[:, hh, :dn] = cd[:, sel[hh]] * sgn[hh]
        k[:, hh, dn:] = cd[:, 512:512 + dr]
        q_abs[:, hh, sel[hh]] = (q_nope[:, hh].double() * sgn[hh]).to(torch.bfloat16)
        q_abs[:, hh, 512:512 + dr] = q_rope[:, hh]
    v = torch.einsum("hvk,sk->shv", w_uv, cd[:, :512])
    q = torch.cat([q_nope, q_rope], dim=2)
    scale = (dn + dr) ** -0.5

    lists = causal_position_lists(T, S, topk, seed=seed + 1, p_empty=0.1)
    lists[1] = -1  # at least one empty row
    y_m, lse_m = oracle.masked_mha(q, k, v, oracle.scatter_mask(lists, S), scale)
    o_lat, lse_s = oracle.sparse_mla_fwd(q_abs, c, lists.repeat(1, repeat), scale)
    y_s = np.einsum("thk,hvk->thv", o_lat, w_uv.numpy())
    return (y_m, lse_m), (y_s, lse_s)


# (heads, qk_nope, qk_rope, v_head) of the report's geometry table, with fewer heads
GEOMETRIES = {"deepseek_v32": (4, 128, 64, 128), "glm5": (3, 192, 64, 256), "nope": (3, 256, 0, 256)}


@pytest.mark.parametrize("geom", sorted(GEOMETRIES))
@pytest.mark.parametrize("T,S,topk", [(10, 90, 32), (24, 24, 2048)])
def test_absorption_identity_with_the_sparse_oracle(geom, T, S, topk):
    h, dn, dr, dv = GEOMETRIES[geom]
    (y_m, lse_m), (y_s, lse_s) = _absorbed_case(T, S, h, dn, dr, dv, topk, seed=T + dn)
    empty = np.isneginf(lse_s)
    assert empty.any() and not empty.all()
    assert np.array_equal(np.isneginf(lse_m), empty)
    assert np.allclose(lse_m[~empty], lse_s[~empty], rtol=1e-12, atol=1e-12)
    assert np.allclose(y_m, y_s, rtol=1e-9, atol=1e-12)


def test_repeated_positions_weigh_once_in_the_mask():
    h, dn, dr, dv = GEOMETRIES["glm5"]
    (y_m, lse_m), (y_s, lse_s) = _absorbed_case(8, 60, h, dn, dr, dv, 16, seed=11, repeat=2)
    live = np.isfinite(lse_s)
    assert live.any()
    assert np.allclose(lse_s[live], lse_m[live] + math.log(2.0), rtol=1e-12, atol=1e-12)
    assert np.allclose(y_m, y_s, rtol=1e-9, atol=1e-12)


# ----------------------------------------------------------------------------- mutation

_MUTANTS = {
    # every head reads head 0's keys
    "key_head0": (r"const double \*kr = k \+ \(s \* h \+ hh\) \* \(int64_t\)dqk;",
                  "const double *kr = k + (s * h + 0) * (int64_t)dqk;"),
    # bits packed from the top of each word
    "mask_bit_reversed": (r"mask\[t \* W \+ s / 32\] \|= 1u << \(s % 32\);",
                          "mask[t * W + s / 32] |= 1u << (31 - s % 32);"),
    # LSE in base 2
    "lse_log2": (r"lse\[p\] = m \+ log\(l\);", "lse[p] = m + log2(l);"),
}


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_masked_dense_mutants_fail_a_pin(tmp_path, monkeypatch, name):
    src = Path(oracle.__file__).with_name("sparse_mla_oracle.c").read_text()
    pat, rep = _MUTANTS[name]
    mutated, n = re.subn(pat, rep, src)
    assert n == 1, f"mutation {name} did not apply"
    c = tmp_path / f"{name}.c"
    c.write_text(mutated)
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    good = oracle._load()
    for fn in ("oracle_scatter_mask", "oracle_masked_mha", "oracle_sparse_mla_fwd",
               "oracle_max_threads"):
        getattr(lib, fn).restype = getattr(good, fn).restype
        getattr(lib, fn).argtypes = getattr(good, fn).argtypes
    monkeypatch.setattr(oracle, "_lib", lib)
    pins = [lambda: test_mask_matches_numpy_scatter(16, 100, 40),
            lambda: test_masked_mha_matches_torch_sdpa(12, 80, 3, 192, 128, 24),
            test_equal_keys_give_the_mean_of_the_values,
            lambda: test_absorption_identity_with_the_sparse_oracle("glm5", 10, 90, 32)]
    failures = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught the mutant {name}"
