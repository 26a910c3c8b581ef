"""The v_up projection of the attention output: oracle pins on the CPU.

y[t, h, n] = sum_k O[t, h, k] W[h, n, k] with O [T, h, 512] bf16 and W [h, v, 512] bf16
(vLLM PR #60220, Details: the output is consumed by the v_up projection; v_head_dim 128 or
256 from the PR #55738 report's geometry table).  Pins of the oracle, each from outside it:

* numpy's float64 einsum over the exactly decoded bf16 values, on random cases;
* closed forms: identity weights return the first v latent dims exactly; weights that are
  zero except for one head leave every other head's output zero;
* mutation: mutated copies of the oracle (W read transposed, every head using head 0's
  weights, the sum cut at v dims) each fail one of these.
"""

import ctypes
import re
import subprocess
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from workloads import make_v_up_weights


def _rand_o(T, h, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(T, h, 512, generator=g) * 0.1).to(torch.bfloat16)


def _dec(x):
    return x.float().double().numpy()  # bf16 -> fp32 -> fp64 is exact


# ----------------------------------------------------------------------------- oracle pins

@pytest.mark.parametrize("T,h,v", [(3, 8, 128), (5, 2, 256), (1, 16, 128), (7, 1, 32)])
def test_matches_float64_einsum(T, h, v):
    o = _rand_o(T, h, seed=T * 100 + h)
    w = make_v_up_weights(h, v, seed=T + v)
    y = oracle.v_up(o, w)
    ref = np.einsum("thk,hnk->thn", _dec(o), _dec(w))
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-15)


def test_identity_weights_return_the_latent_dims():
    T, h, v = 4, 3, 128
    o = _rand_o(T, h, seed=5)
    w = torch.zeros(h, v, 512, dtype=torch.bfloat16)
    for n in range(v):
        w[:, n, n] = 1.0
    y = oracle.v_up(o, w)
    assert np.array_equal(y, _dec(o)[:, :, :v])


def test_heads_are_independent():
    T, h, v = 3, 4, 128
    o = _rand_o(T, h, seed=6)
    w = make_v_up_weights(h, v, seed=7)
    w[[0, 1, 3]] = 0
    y = oracle.v_up(o, w)
    assert np.all(y[:, [0, 1, 3]] == 0.0)
    assert np.all(np.abs(y[:, 2]) > 0.0)


_MUTANTS = {
    # W read as [h, 512, v]: element (n, k) taken from position k * v + n of the head's block
    "w_transposed": (r"acc \+= bf16_bits_to_double\(orow\[k\]\) \* bf16_bits_to_double\(wrow\[k\]\);",
                     "acc += bf16_bits_to_double(orow[k]) * "
                     "bf16_bits_to_double(w[(int64_t)hh * v * ORACLE_DV + (int64_t)k * v + n]);"),
    "head0_weights": (r"const uint16_t \*wrow = w \+ \(\(int64_t\)hh \* v \+ n\) \* ORACLE_DV;",
                      "const uint16_t *wrow = w + ((int64_t)0 * v + n) * ORACLE_DV;"),
    "sum_cut_at_v": (r"for \(int k = 0; k < ORACLE_DV; \+\+k\)\n                    acc \+= bf16_bits_to_double\(orow\[k\]\)",
                     "for (int k = 0; k < v; ++k)\n                    acc += bf16_bits_to_double(orow[k])"),
}


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_v_up_mutants_fail_a_pin(tmp_path, monkeypatch, name):
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
    for fn in ("oracle_v_up", "oracle_max_threads"):
        getattr(lib, fn).restype = getattr(good, fn).restype
        getattr(lib, fn).argtypes = getattr(good, fn).argtypes
    monkeypatch.setattr(oracle, "_lib", lib)
    pins = [lambda: test_matches_float64_einsum(3, 8, 128), lambda: test_matches_float64_einsum(5, 2, 256),
            test_identity_weights_return_the_latent_dims, test_heads_are_independent]
    failures = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught the mutant {name}"
