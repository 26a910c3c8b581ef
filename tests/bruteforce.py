"""Dense-mask brute force: ordinary attention over the whole cache.

This is the pin for the oracle.  Instead of walking each token's list, it builds
a dense [num_slots] multiplicity mask per token from the indices, scores every
cache row with one matrix product, adds log(multiplicity) (-inf for rows not in
the list) and runs a plain log-sum-exp softmax over all slots.  It decodes the
cache through torch's own bf16 / float8_e4m3fn conversions, not the oracle's.
This mirrors the SDPA-reference check the PR #55738 report describes for the
prefill paths (测试配套, test coverage).
"""

import numpy as np
import torch


def decode_cache(kv: torch.Tensor, kv_format: str) -> np.ndarray:
    if kv_format == "bf16":
        return kv.float().double().numpy()
    n = kv.shape[0]
    codes = kv[:, 0:512].contiguous().view(torch.float8_e4m3fn).float().double()
    scales = kv[:, 512:528].contiguous().view(torch.float32).double()     # [n, 4]
    lat = (codes.reshape(n, 4, 128) * scales[:, :, None]).reshape(n, 512)
    rope = kv[:, 528:656].contiguous().view(torch.bfloat16).float().double()
    return torch.cat([lat, rope], dim=1).numpy()


def dense_attention(q: torch.Tensor, kv: torch.Tensor, indices: torch.Tensor, scale: float,
                    kv_format: str = "bf16"):
    """Returns (out [T,h,512] float64, lse [T,h] float64)."""
    K = decode_cache(kv, kv_format)                    # [S, 576]
    S = K.shape[0]
    qd = q.float().double().numpy()                    # [T, h, 576]
    idx = indices.numpy().astype(np.int64)
    T, h, _ = qd.shape
    out = np.zeros((T, h, 512))
    lse = np.full((T, h), -np.inf)
    for t in range(T):
        sel = idx[t][(idx[t] >= 0) & (idx[t] < S)]
        if sel.size == 0:
            continue
        counts = np.bincount(sel, minlength=S).astype(np.float64)
        with np.errstate(divide="ignore"):
            bias = np.log(counts)                      # -inf where the slot is not listed
        z = scale * (K @ qd[t].T) + bias[:, None]      # [S, h]
        zmax = z.max(axis=0)
        e = np.exp(z - zmax)
        tot = e.sum(axis=0)
        lse[t] = zmax + np.log(tot)
        out[t] = (e / tot).T @ K[:, :512]
    return out, lse
