"""Seeded generators for queries, paged latent KV caches and top-k slot lists.

Recipe (all draws come from torch CPU generators seeded from the config seed,
so the same seed gives the same bytes on any host):

* q[t, h, 0:576] = bf16(N(0, 1) * 0.5), i.e. mean 0, standard deviation 0.5.
* bf16 cache rows kv[slot, 0:576] = bf16(N(0, 1) * 0.5).
* fp8 cache rows (656 bytes): the 512 latent values x ~ N(0, 0.5) are split in
  four 128-value tiles; each tile stores scale = max|x| / 448 (1 when the tile is
  all zero) as fp32 and e4m3(x / scale) with round-to-nearest-even, saturated to
  +-448; the 64 rope values are stored as bf16.  Byte layout:
  [512 x e4m3 | 4 x fp32 scale | 64 x bf16 rope].
* Sequence s has seq_len cached positions in blocks of 64 slots.  A block table
  maps (s, pos // 64) to a physical block: a random permutation of all blocks
  (identity for the tiny case).  slot = block * 64 + pos % 64.
* Query tokens are the last `queries_per_seq` positions of each sequence.  The
  list of token t holds `topk` distinct causal positions (<= its own position)
  chosen as the top-k of i.i.d. keys (uniform, or N(0, 1) "indexer scores" for
  the prefill case), mapped to slots; -1 pads lists whose history is shorter than
  topk.  Some configs then force entries to -1 (a fixed tail, or each entry with
  a fixed probability).
"""

from dataclasses import dataclass
from typing import Optional

import torch

from .configs import (BLOCK_SIZE, D_QK, FP8_ROW_BYTES, WorkloadConfig, config_by_name,
                      scale_for)

_TOKEN_BATCH = 256
_ROW_CHUNK = 1 << 17


def _gen(seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 16 + stream)
    return g


@dataclass
class Workload:
    cfg: WorkloadConfig
    h: int
    q: torch.Tensor            # [T, h, 576] bf16
    kv: torch.Tensor           # [num_slots, 576] bf16, or [num_slots, 656] uint8 (fp8 rows)
    indices: torch.Tensor      # [T, topk] int32, -1 = invalid
    scale: float
    positions: torch.Tensor    # [T] int64, the query's own position in its sequence
    seq_of_token: torch.Tensor  # [T] int64
    block_table: torch.Tensor  # [n_seq, blocks_per_seq] int64

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])

    @property
    def num_slots(self) -> int:
        return int(self.kv.shape[0])

    @property
    def kv_format(self) -> str:
        return self.cfg.kv_format


def quantize_fp8_rows(x: torch.Tensor) -> torch.Tensor:
    """Pack fp32 rows [n, 576] into 656-byte fp8 cache rows (layout in the module doc)."""
    assert x.dim() == 2 and x.shape[1] == D_QK
    n = x.shape[0]
    lat = x[:, :512].float().reshape(n, 4, 128)
    amax = lat.abs().amax(dim=2, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (lat / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    out = torch.empty((n, FP8_ROW_BYTES), dtype=torch.uint8)
    out[:, 0:512] = codes.reshape(n, 512).view(torch.uint8)
    out[:, 512:528] = scale.reshape(n, 4).contiguous().view(torch.uint8)
    out[:, 528:656] = x[:, 512:].to(torch.bfloat16).contiguous().view(torch.uint8)
    return out


def _make_cache(cfg: WorkloadConfig, seed: int, num_slots: int) -> torch.Tensor:
    g = _gen(seed, 2)
    if cfg.kv_format == "bf16":
        kv = torch.empty((num_slots, D_QK), dtype=torch.bfloat16)
    else:
        kv = torch.empty((num_slots, FP8_ROW_BYTES), dtype=torch.uint8)
    for r0 in range(0, num_slots, _ROW_CHUNK):
        r1 = min(num_slots, r0 + _ROW_CHUNK)
        x = torch.randn((r1 - r0, D_QK), generator=g) * 0.5
        if cfg.kv_format == "bf16":
            kv[r0:r1] = x.to(torch.bfloat16)
        else:
            kv[r0:r1] = quantize_fp8_rows(x)
    return kv


def _make_block_table(cfg: WorkloadConfig, seed: int, n_seq: int) -> torch.Tensor:
    bps = cfg.seq_len // BLOCK_SIZE
    if cfg.identity_blocks:
        return torch.arange(n_seq * bps, dtype=torch.int64).reshape(n_seq, bps)
    g = _gen(seed, 4)
    return torch.randperm(n_seq * bps, generator=g).reshape(n_seq, bps)


def _make_indices(cfg: WorkloadConfig, seed: int, positions: torch.Tensor,
                  seq_of_token: torch.Tensor, block_table: torch.Tensor,
                  n_tokens: int) -> torch.Tensor:
    """Top-k of i.i.d. keys over each token's causal window, mapped to slots."""
    g = _gen(seed, 3)
    topk, width = cfg.topk, cfg.seq_len
    out = torch.empty((n_tokens, topk), dtype=torch.int32)
    cols = torch.arange(width, dtype=torch.int64)
    for t0 in range(0, n_tokens, _TOKEN_BATCH):
        t1 = min(n_tokens, t0 + _TOKEN_BATCH)
        # always draw a full batch so any prefix of tokens is generated identically
        if cfg.index_mode == "scores":
            keys = torch.randn((_TOKEN_BATCH, width), generator=g, dtype=torch.float64)
        else:
            keys = torch.rand((_TOKEN_BATCH, width), generator=g, dtype=torch.float64)
        keys = keys[: t1 - t0]
        pos = positions[t0:t1]
        keys.masked_fill_(cols[None, :] > pos[:, None], float("-inf"))
        k = min(topk, width)
        top = torch.topk(keys, k, dim=1)
        sel_pos = top.indices
        ok = torch.isfinite(top.values)
        seq = seq_of_token[t0:t1]
        blk = block_table[seq[:, None], sel_pos // BLOCK_SIZE]
        slots = blk * BLOCK_SIZE + sel_pos % BLOCK_SIZE
        slots = torch.where(ok, slots, torch.full_like(slots, -1))
        if k < topk:
            pad = torch.full((t1 - t0, topk - k), -1, dtype=slots.dtype)
            slots = torch.cat([slots, pad], dim=1)
        out[t0:t1] = slots.to(torch.int32)
    if cfg.invalid_tail:
        out[:, topk - cfg.invalid_tail:] = -1
    if cfg.invalid_prob > 0:
        drop = torch.rand((n_tokens, topk), generator=_gen(seed, 5)) < cfg.invalid_prob
        out.masked_fill_(drop, -1)
    return out


def _make_q(seed: int, n_tokens: int, h: int) -> torch.Tensor:
    g = _gen(seed, 1)
    q = torch.empty((n_tokens, h, D_QK), dtype=torch.bfloat16)
    for t0 in range(0, n_tokens, _TOKEN_BATCH):
        t1 = min(n_tokens, t0 + _TOKEN_BATCH)
        x = torch.randn((_TOKEN_BATCH, h, D_QK), generator=g) * 0.5
        q[t0:t1] = x[: t1 - t0].to(torch.bfloat16)
    return q


def make_workload(name: str, *, h: Optional[int] = None, seed: Optional[int] = None,
                  n_seq: Optional[int] = None, n_tokens: Optional[int] = None,
                  topk: Optional[int] = None) -> Workload:
    """Generate a workload.

    name      one of the five configs (tiny, decode_bf16, sweep, prefill, fp8_mixed)
    h         head count (defaults to the config's; the sweep takes 8/16/32/64)
    seed      defaults to 1000 + config number; other seeds give independent copies
    n_seq     fewer sequences than the config (a reduced cache for quick checks)
    n_tokens  only the first n query tokens (a prefix of the full workload)
    topk      shorter lists (still drawn the same way)
    """
    cfg = config_by_name(name)
    if topk is not None:
        cfg = WorkloadConfig(**{**cfg.__dict__, "topk": int(topk)})
    hh = cfg.h if h is None else int(h)
    sd = cfg.seed if seed is None else int(seed)
    ns = cfg.n_seq if n_seq is None else int(n_seq)
    T_full = ns * cfg.queries_per_seq
    T = T_full if n_tokens is None else min(int(n_tokens), T_full)
    num_slots = ns * cfg.seq_len

    block_table = _make_block_table(cfg, sd, ns)
    seq_of_token = torch.arange(T_full, dtype=torch.int64) // cfg.queries_per_seq
    positions = (cfg.seq_len - cfg.queries_per_seq
                 + torch.arange(T_full, dtype=torch.int64) % cfg.queries_per_seq)
    seq_of_token, positions = seq_of_token[:T], positions[:T]

    kv = _make_cache(cfg, sd, num_slots)
    q = _make_q(sd, T, hh)
    idx = _make_indices(cfg, sd, positions, seq_of_token, block_table, T)
    return Workload(cfg=cfg, h=hh, q=q, kv=kv, indices=idx, scale=scale_for(),
                    positions=positions, seq_of_token=seq_of_token,
                    block_table=block_table)


def pad_heads(q: torch.Tensor, heads: int = 64) -> torch.Tensor:
    """Zero-pad the head dimension of q [T, h, 576] to `heads` (the padded arm).

    This is the caller-side padding the pages describe for the SM90 kernels
    (vLLM PR #64510 "Overview"; vLLM PR #60220 "Details", root cause: the wrapper
    pads q to 64 heads with new_zeros).  The padded heads' outputs are discarded.
    """
    T, h, d = q.shape
    if h == heads:
        return q
    out = torch.zeros((T, heads, d), dtype=q.dtype, device=q.device)
    out[:, :h] = q
    return out


def gathered_bytes(indices: torch.Tensor, num_slots: int, row_bytes: int) -> int:
    """Algorithmic gathered KV bytes: valid list entries x row bytes."""
    valid = (indices >= 0) & (indices < num_slots)
    return int(valid.sum().item()) * int(row_bytes)


def split_lists(indices: torch.Tensor, n_parts: int) -> list:
    """Split every token's list into n_parts contiguous column ranges (the parts a decode-
    context-parallel split gives each rank): part p keeps columns [p*topk//n, (p+1)*topk//n)
    and holds -1 everywhere else, so the parts' valid entries are disjoint and their union is
    the list."""
    topk = indices.shape[1]
    parts = []
    for p in range(n_parts):
        a, b = p * topk // n_parts, (p + 1) * topk // n_parts
        part = torch.full_like(indices, -1)
        part[:, a:b] = indices[:, a:b]
        parts.append(part)
    return parts


def make_merge_parts(n_parts: int, T: int, h: int, seed: int = 6000, p_empty: float = 0.05):
    """Synthetic partial results of lists split into n_parts, in the layout the merge reads:
    o_parts [n, T, h, 512] bf16 = bf16(N(0, 1) * 0.1) (an attention output is a convex mix of
    value rows, smaller than the rows themselves) and lse_parts [n, T, h] fp32 = N(6, 1)
    (about ln 2048 / n), each part empty (LSE = -inf, O = 0) with probability p_empty, and
    the first row of every token empty in all parts."""
    g = _gen(seed, 11)
    o = (torch.randn(n_parts, T, h, 512, generator=g) * 0.1).to(torch.bfloat16)
    lse = torch.randn(n_parts, T, h, generator=g) + 6.0
    empty = torch.rand(n_parts, T, h, generator=g) < p_empty
    if T > 0:
        empty[:, :, 0] = True
    lse[empty] = float("-inf")
    o[empty] = 0
    return o, lse.to(torch.float32)


def make_v_up_weights(h: int, v: int, seed: int = 7000) -> torch.Tensor:
    """Synthetic value up-projection weights, W [h, v, 512] bf16 = bf16(N(0, 1) / sqrt(512))
    (row n of head h holds the 512 weights of output n), so the projected values keep about
    the scale of the latent output."""
    g = _gen(seed, 12)
    return (torch.randn(h, v, 512, generator=g) * 512 ** -0.5).to(torch.bfloat16)


def causal_position_lists(T: int, S: int, topk: int, seed: int = 8000,
                          p_empty: float = 0.0) -> torch.Tensor:
    """Position lists of a prefill chunk, [T, topk] int32: the chunk's T query tokens are the
    last T positions of an S-position request, so token t sees the causal history
    [0, S - T + 1 + t).  Its list holds min(topk, history) distinct positions of that history,
    the top-k of i.i.d. uniform keys (so in random order), -1 padded; a token's list is all -1
    with probability p_empty.  A topk at least S gives every token its full history: the
    short-prefill case."""
    assert 1 <= T <= S and topk >= 1
    g = _gen(seed, 13)
    out = torch.full((T, topk), -1, dtype=torch.int32)
    k = min(topk, S)
    pos = torch.arange(S)
    for t0 in range(0, T, _TOKEN_BATCH):
        t1 = min(T, t0 + _TOKEN_BATCH)
        hist = S - T + 1 + torch.arange(t0, t1)
        keys = torch.rand(t1 - t0, S, generator=g)
        keys[pos[None, :] >= hist[:, None]] = -1.0
        vals, sel = keys.topk(k, dim=1)
        sel = sel.to(torch.int32)
        sel[vals < 0] = -1
        out[t0:t1, :k] = sel
    if p_empty > 0:
        out[torch.rand(T, generator=g) < p_empty] = -1
    return out


def make_masked_dense_inputs(T: int, S: int, h: int, dqk: int, dv: int, seed: int = 9000):
    """Decompressed per-head inputs of the masked dense route: q [T, h, dqk], k [S, h, dqk]
    and v [S, h, dv], each bf16(N(0, 1) * 0.5) like the latent query and cache."""
    g = _gen(seed, 14)
    q = (torch.randn(T, h, dqk, generator=g) * 0.5).to(torch.bfloat16)
    k = (torch.randn(S, h, dqk, generator=g) * 0.5).to(torch.bfloat16)
    v = (torch.randn(S, h, dv, generator=g) * 0.5).to(torch.bfloat16)
    return q, k, v
