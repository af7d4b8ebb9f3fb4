"""The five synthetic workloads the hot path is tested and measured on.

Each entry gives the attention shape (LLaMA-3.1-8B: 32 query heads over 8 kv
heads, head dim 128, except the single-head correctness case), the context
length(s), and the compression strategy: sink tokens, recent window, token
block size, kept channels r per middle segment, and block retention.
Segments are given as (begin_permille, r, always): a segment starts at the
first block boundary at or after begin_permille/1000 of the prefill length,
keeps r channels per vector, and is either scored for top-k selection
(always = 0) or attended in full (always = 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class Workload:
    name: str
    n_q_heads: int
    n_kv_heads: int
    d: int
    seq_lens: list          # prefill length per sequence
    n_layers: int
    n_sink: int
    window: int
    block: int
    segments: list          # [(begin_permille, r, always)]
    topk_fixed: int = 0     # > 0: select exactly this many blocks
    retain_permille: int = 0
    meta_channels: int = 0        # > 0: channel-compressed per-block keys (a variant; 0 in every listed workload)
    elem_group: int = 0           # > 0: bitmap pages with this element-group size (a variant; 0 = uint8 indices)
    decay: float = 0.92
    append_per_step: int = 1
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n_seqs(self):
        return len(self.seq_lens)

    @property
    def group(self):
        return self.n_q_heads // self.n_kv_heads


def _loguniform_lens():
    from .synth import seq_lengths_loguniform, seed_for
    return seq_lengths_loguniform(64, 8192, 131072, seed_for("serving-mix-lengths"))


def get(name: str) -> Workload:
    if name == "c1":
        return Workload("c1-single-head-4k", 1, 1, 128, [4096], 1, 4, 64, 16,
                        [(0, 32, 0)], topk_fixed=64, decay=0.9, append_per_step=0,
                        description="single head, d=128, T=4096, r=32, block 16, top-64 blocks, "
                                    "4 sinks, 64-token window")
    if name == "c2":
        return Workload("c2-llama8b-layer-32k-b4", 32, 8, 128, [32768] * 4, 1, 4, 128, 16,
                        [(0, 38, 0)], retain_permille=100,
                        description="LLaMA-3.1-8B attention layer, T=32768, batch 4, r=38, "
                                    "block 16, 10% blocks, 4 sinks, 128-token window")
    if name == "c3":
        return Workload("c3-llama8b-128k-32layers", 32, 8, 128, [131072], 32, 4, 256, 32,
                        [(0, 38, 0)], retain_permille=100,
                        description="T=131072, batch 1, 32 layers, r=38, block 32, 10% blocks, "
                                    "4 sinks, 256-token window")
    if name == "c4":
        return Workload("c4-llama8b-1m-32layers", 32, 8, 128, [1048576], 32, 4, 512, 64,
                        [(0, 38, 0)], retain_permille=50,
                        description="T=1048576, batch 1, 32 layers, r=38, block 64, 5% blocks, "
                                    "4 sinks, 512-token window")
    if name == "c5":
        return Workload("c5-serving-mix-64seq", 32, 8, 128, _loguniform_lens(), 1, 4, 128, 16,
                        [(0, 32, 0), (350, 64, 1), (650, 32, 0)], retain_permille=100,
                        description="64 sequences, lengths log-uniform 8K..128K, one layer; "
                                    "middle 30% r=64 attended in full, rest r=32 with 10% blocks")
    raise KeyError(name)


ALL = ["c1", "c2", "c3", "c4", "c5"]
