"""The five synthetic workloads, with the shapes of the serving cases the pages describe.

Shapes follow the pages: the query is [T, h, 576] bf16 with 512 latent + 64 rope
dims and the output is [T, h, 512] (vLLM PR #60220, "Claims": padded q is
T x 64 x 576, out is T x 64 x 512); h is the per-rank head count under tensor
parallelism, 8/16/32 native or padded to 64 (vLLM PR #64510, "Overview",
"Details"); the per-token index list has index_topk = 2048 int32 columns
(vLLM PR #54951, "Summary"); the 16k-token prefill chunk comes from the
PR #55738 report, "功能与动机" (function and motivation).
"""

from dataclasses import dataclass, field
from typing import Optional, Tuple

D_QK = 576          # kv_lora_rank 512 + qk_rope 64 (PR #55738 report, geometry table)
D_V = 512           # V is the latent part of the same row
BLOCK_SIZE = 64     # paged-cache block size
FP8_ROW_BYTES = 656  # 512 e4m3 + 4 fp32 tile scales + 64 bf16 rope
BF16_ROW_BYTES = 1152


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    cfg_id: int
    n_seq: int                 # sequences in the paged cache
    seq_len: int               # cached tokens per sequence
    queries_per_seq: int       # query tokens per sequence (the last positions)
    h: int
    topk: int
    kv_format: str             # "bf16" or "fp8"
    index_mode: str            # "uniform" | "scores" (top-k of N(0,1) scores)
    invalid_tail: int = 0      # last entries of each list forced to -1
    invalid_prob: float = 0.0  # each entry independently -1 with this probability
    identity_blocks: bool = False
    sweep_h: Tuple[int, ...] = field(default_factory=tuple)

    @property
    def T(self) -> int:
        return self.n_seq * self.queries_per_seq

    @property
    def num_slots(self) -> int:
        return self.n_seq * self.seq_len

    @property
    def seed(self) -> int:
        return 1000 + self.cfg_id

    @property
    def row_bytes(self) -> int:
        return FP8_ROW_BYTES if self.kv_format == "fp8" else BF16_ROW_BYTES


CONFIGS = {
    # 1: tiny oracle case, one sequence of 256 tokens in 4 blocks, identity block table
    "tiny": WorkloadConfig("tiny", 1, n_seq=1, seq_len=256, queries_per_seq=4, h=8,
                           topk=64, kv_format="bf16", index_mode="uniform",
                           invalid_tail=8, identity_blocks=True),
    # 2: decode batch, bf16, 32 sequences x 16384 tokens, one query each
    "decode_bf16": WorkloadConfig("decode_bf16", 2, n_seq=32, seq_len=16384,
                                  queries_per_seq=1, h=8, topk=2048, kv_format="bf16",
                                  index_mode="uniform"),
    # 3: head-count sweep, decode, 128 sequences x 8192 tokens, ~5 % of entries -1
    "sweep": WorkloadConfig("sweep", 3, n_seq=128, seq_len=8192, queries_per_seq=1,
                            h=8, topk=2048, kv_format="bf16", index_mode="uniform",
                            invalid_prob=0.05, sweep_h=(8, 16, 32, 64)),
    # 4: long prefill chunk, the last 16384 of 32768 positions are queries, h=64
    "prefill": WorkloadConfig("prefill", 4, n_seq=1, seq_len=32768, queries_per_seq=16384,
                              h=64, topk=2048, kv_format="bf16", index_mode="scores"),
    # 5: fp8 KV mixed batch, 16 sequences x 65536 tokens, last 2048 positions are queries
    "fp8_mixed": WorkloadConfig("fp8_mixed", 5, n_seq=16, seq_len=65536,
                                queries_per_seq=2048, h=8, topk=2048, kv_format="fp8",
                                index_mode="uniform"),
}


def config_by_name(name: str) -> WorkloadConfig:
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")
    return CONFIGS[name]


def scale_for(d_qk: int = D_QK) -> float:
    """Softmax scale used by every workload: d_qk ** -0.5 with d_qk = 576."""
    return float(d_qk) ** -0.5


def describe(cfg: WorkloadConfig, h: Optional[int] = None) -> str:
    hh = cfg.h if h is None else h
    return (f"{cfg.name}: T={cfg.T} h={hh} topk={cfg.topk} kv={cfg.kv_format} "
            f"slots={cfg.num_slots} ({cfg.n_seq}x{cfg.seq_len}, block {BLOCK_SIZE})")
