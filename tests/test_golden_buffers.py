"""The padded arm's buffers against the sizes the pages measured.

tests/golden/padded_arm_buffers.txt holds the page's per-call allocation saved by staging
the head-padded q ([T, 64, 576] bf16) and the output ([T, 64, 512] bf16) in a workspace,
and the size of lse ([T, 64] fp32).  The padded arm of these tests and of bench.py builds
exactly those tensors (workloads.pad_heads and the binding's out/lse shapes), so their byte
counts must reproduce the page's figures to its printed precision.
"""

from pathlib import Path

import torch

from workloads import pad_heads

GOLDEN = Path(__file__).resolve().parent / "golden" / "padded_arm_buffers.txt"


def _rows():
    for line in GOLDEN.read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        t, saved, lse = line.split()
        yield int(t), float(saved), (None if lse == "-" else float(lse))


def test_golden_file_has_the_four_rows():
    assert [r[0] for r in _rows()] == [1024, 8192, 16384, 32768]


def test_padded_q_and_out_bytes_match_the_page():
    for T, saved_gib, lse_mib in _rows():
        q8 = torch.empty((T, 8, 576), dtype=torch.bfloat16, device="meta")
        qp = pad_heads(q8, 64)
        out = torch.empty((T, qp.shape[1], 512), dtype=torch.bfloat16, device="meta")
        lse = torch.empty((T, qp.shape[1]), dtype=torch.float32, device="meta")
        got = (qp.numel() * qp.element_size() + out.numel() * out.element_size()) / 2**30
        # the page prints GiB to three decimals (1.0625 -> 1.063)
        assert abs(got - saved_gib) <= 0.0005 + 1e-9, (T, got, saved_gib)
        if lse_mib is not None:
            assert lse.numel() * lse.element_size() / 2**20 == lse_mib
