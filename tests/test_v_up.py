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


# ----------------------------------------------------------------------------- C ABI (no GPU)

@pytest.fixture(scope="module")
def lib():
    import token_sparse_mla_gb300 as smla
    return smla.library()


@pytest.mark.parametrize("T,h,v,status", [(4, 8, 64, 2), (4, 8, 512, 2), (4, 0, 128, 1), (-1, 8, 128, 1)])
def test_v_up_rejects_bad_arguments(lib, T, h, v, status):
    buf = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    assert lib.sparse_mla_v_up(buf, buf, T, h, v, buf, None) == status


def test_v_up_rejects_null_and_misaligned(lib):
    good = ctypes.c_void_p(4096)
    assert lib.sparse_mla_v_up(None, good, 4, 8, 128, good, None) == 1
    assert lib.sparse_mla_v_up(good, ctypes.c_void_p(4104), 4, 8, 128, good, None) == 1
    assert lib.sparse_mla_v_up(good, good, 4, 8, 128, ctypes.c_void_p(4098), None) == 1


def test_v_up_zero_tokens_is_a_noop(lib):
    assert lib.sparse_mla_v_up(None, None, 0, 8, 128, None, None) == 0


# ----------------------------------------------------------------------------- GPU parity

DEV = "cuda:0"


def _gpu_v_up(o, w):
    import token_sparse_mla_gb300 as smla
    y = smla.sparse_mla_v_up(o.to(DEV), w.to(DEV))
    smla.sync_status()
    return y.cpu()


def _assert_v_up_parity(y, ref, o, w, what):
    """fp32 accumulation over 512 products, one bf16 rounding of the result."""
    yv = y.float().double().numpy()
    scale = np.einsum("thk,hnk->thn", np.abs(_dec(o)), np.abs(_dec(w)))
    err = np.abs(yv - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * scale + 1e-30
    assert np.all(np.isfinite(yv)), what
    assert np.all(err <= bound), f"{what}: worst excess {(err - bound).max()}"


@pytest.mark.gpu
@pytest.mark.parametrize("T,h,v", [(1, 1, 128), (5, 8, 128), (128, 2, 128), (129, 3, 256), (300, 8, 128),
                                   (1000, 1, 256), (4096, 16, 128)])
def test_gpu_v_up_matches_oracle(T, h, v):
    o = _rand_o(T, h, seed=T + 7 * h)
    w = make_v_up_weights(h, v, seed=T + v)
    y = _gpu_v_up(o, w)
    ref = oracle.v_up(o, w)
    _assert_v_up_parity(y, ref, o, w, f"T={T} h={h} v={v}")


@pytest.mark.gpu
def test_gpu_v_up_identity_weights_are_exact():
    T, h, v = 257, 4, 256
    o = _rand_o(T, h, seed=9)
    w = torch.zeros(h, v, 512, dtype=torch.bfloat16)
    for n in range(v):
        w[:, n, n] = 1.0
    y = _gpu_v_up(o, w)
    assert torch.equal(y, o[:, :, :v])


@pytest.mark.gpu
@pytest.mark.parametrize("name,kw", [("decode_bf16", {"n_seq": 8}), ("sweep", {"h": 64, "n_seq": 3})])
def test_gpu_forward_then_v_up(name, kw):
    """The forward on the GPU, then v_up on the GPU: against the oracle v_up of the same
    output, and against the oracle chain within the forward's tolerance carried through W."""
    import token_sparse_mla_gb300 as smla
    from tests.parity import O_ATOL, O_RTOL
    from workloads import make_workload
    w_ = make_workload(name, **kw)
    out, _ = smla.sparse_mla_fwd(w_.q.to(DEV), w_.kv.to(DEV), w_.indices.to(DEV), w_.scale)
    W = make_v_up_weights(w_.h, 128, seed=3)
    y = smla.sparse_mla_v_up(out, W.to(DEV))
    smla.sync_status()
    o_gpu = out.cpu()
    _assert_v_up_parity(y.cpu(), oracle.v_up(o_gpu, W), o_gpu, W, f"{name} same input")
    ref_o, _ = oracle.sparse_mla_fwd(w_.q, w_.kv, w_.indices, w_.scale)
    ref_y = np.einsum("thk,hnk->thn", ref_o, _dec(W))
    carried = np.einsum("thk,hnk->thn", O_ATOL + O_RTOL * np.abs(ref_o), np.abs(_dec(W)))
    err = np.abs(y.cpu().float().double().numpy() - ref_y)
    assert np.all(err <= carried + 2.0 ** -8 * np.abs(ref_y) + 1e-6), f"{name} chain"
