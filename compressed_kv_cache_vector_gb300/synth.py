"""Seeded synthetic inputs for the MosaicKV decode-time hot path.

This module only makes data. It holds no step of the compression method
(no rotation, no selection, no scoring, no attention): both the CUDA path and
the fp64 oracle receive the tensors it returns, and neither imports the other.

Key/value generator (low rank plus outliers): each (layer, sequence, kv head)
gets its own seed.  K = Z diag(s) Q^T with Z ~ N(0, 1) of shape [T, d],
s_i = decay**i and Q a Haar-random orthogonal d x d matrix (QR of a Gaussian
matrix with the signs of diag(R) folded into Q).  Four channels of the
original (unrotated) space, drawn without replacement, are multiplied by 8 on
round(0.02 T) tokens drawn without replacement.  The result is rounded to
bf16 (round to nearest even).  Queries are N(0, 1) rounded to bf16.

The pages measure on LongBench and RULER with LLaMA-3.1-8B; these generators
stand in for that data with the same attention shapes (d = 128, GQA 32q/8kv).
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch


def seed_for(*parts) -> int:
    """Stable 63-bit seed from any tuple of names and integers."""
    h = hashlib.sha256(repr(tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & 0x7FFF_FFFF_FFFF_FFFF


def haar_orthogonal(d: int, seed: int) -> np.ndarray:
    """Haar-distributed random orthogonal matrix (float64)."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((d, d))
    q, r = np.linalg.qr(a)
    q = q * np.sign(np.diag(r))[None, :]
    return q


def lowrank_outlier(T: int, d: int, decay: float, seed: int, device="cpu",
                    n_outlier_channels: int = 4, outlier_frac: float = 0.02,
                    outlier_scale: float = 8.0) -> torch.Tensor:
    """One head's K (or V) history, bf16 [T, d]."""
    Q = torch.as_tensor(haar_orthogonal(d, seed ^ 0x5A5A), dtype=torch.float32, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    Z = torch.randn(T, d, generator=g, device=device, dtype=torch.float32)
    s = torch.tensor([decay ** i for i in range(d)], dtype=torch.float32, device=device)
    X = (Z * s[None, :]) @ Q.T
    rng = np.random.default_rng(seed ^ 0xA5A5)
    n_out = int(round(outlier_frac * T))
    if n_out > 0 and n_outlier_channels > 0:
        ch = rng.choice(d, size=n_outlier_channels, replace=False)
        toks = rng.choice(T, size=n_out, replace=False)
        ti = torch.as_tensor(toks, device=device, dtype=torch.long)
        ci = torch.as_tensor(ch, device=device, dtype=torch.long)
        X[ti[:, None], ci[None, :]] *= outlier_scale
    return X.to(torch.bfloat16)


def query(n_seqs: int, n_q_heads: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """Decode queries, bf16 [n_seqs, n_q_heads, d], N(0, 1)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(n_seqs, n_q_heads, d, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def seq_lengths_loguniform(n: int, lo: int, hi: int, seed: int) -> list[int]:
    """Sequence lengths drawn log-uniform in [lo, hi] (floored)."""
    rng = np.random.default_rng(seed)
    u = rng.random(n)
    return [int(np.floor(np.exp(np.log(lo) + x * (np.log(hi) - np.log(lo))))) for x in u]


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor (on any device)."""
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_values(x: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor."""
    return x.detach().cpu().to(torch.float64).numpy()
