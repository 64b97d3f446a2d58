"""Seeded synthetic workloads for the paged decode path.

This module only draws random inputs and describes how a pool is laid out;
it holds none of the method's arithmetic (no slot or table computation, no
attention, no quantisation).  Both the tests' oracle and the benchmark take
their inputs from here.

A workload is a batch of sequences for one decode layer-step:

* ``seq_lens``   lengths *after* this step's one-token append;
* a pool of ``pool_blocks`` physical blocks whose free order is a seeded
  permutation, so consecutive allocations land on scattered blocks;
* an op script (:func:`build_script`) that a block manager replays to reach
  the pre-step state (prompt appends, forks), after which each sequence
  appends one token.

Random tensors are standard normal, rounded to bf16; the long-context shape
multiplies each element independently by ``outlier_scale`` with probability
``outlier_prob`` before rounding.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seq_lens: list            # post-append lengths
    pool_blocks: int
    seed: int
    outlier_prob: float = 0.0
    outlier_scale: float = 1.0
    shared_prefix: int = 0     # tokens of a prefix shared by every sequence
    scale: float = field(default=0.0)
    scattered: bool = True     # False: blocks handed out in order 0, 1, 2, ...

    def __post_init__(self):
        if not self.scale:
            self.scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks_per_seq(self) -> int:
        return max(-(-n // self.block_size) for n in self.seq_lens)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _cdiv(a, b):
    return -(-a // b)


# ------------------------------------------------------------ workloads ---
def tiny() -> Workload:
    """B=4, lengths {7,16,33,50} before the append, Hq=4, Hkv=2, d=64, bs=16,
    32-block pool in a seeded permutation."""
    return Workload("tiny_paged_decode", 4, 4, 2, 64, 16,
                    seq_lens=[8, 17, 34, 51], pool_blocks=32, seed=1,
                    scale=1.0 / 8.0)


def llama32_1b(num_seqs: int = 64) -> Workload:
    """Llama-3.2-1B-shaped layer: Hq=32, Hkv=8, d=64, bs=16, B=64, lengths
    uniform in [128, 2048], pool 30% larger than needed."""
    g = _gen(2)
    lens = torch.randint(128, 2049, (num_seqs,), generator=g).tolist()
    need = sum(_cdiv(n, 16) for n in lens)
    return Workload("llama3.2-1b_decode_layer", num_seqs, 32, 8, 64, 16,
                    seq_lens=lens, pool_blocks=math.ceil(1.3 * need), seed=2)


def llama31_8b(num_seqs: int = 128) -> Workload:
    """Llama-3.1-8B-shaped layer: Hq=32, Hkv=8, d=128, bs=16, B=128; total
    length = prompt lognormal(median 256, sigma 1) + decoded lognormal(mean
    415, sigma 1), clipped to [16, 4096]; scattered blocks."""
    g = _gen(3)
    z1 = torch.randn(num_seqs, generator=g, dtype=torch.float64)
    z2 = torch.randn(num_seqs, generator=g, dtype=torch.float64)
    prompt = torch.exp(math.log(256.0) + 1.0 * z1)
    decoded = torch.exp(math.log(415.0) - 0.5 + 1.0 * z2)
    lens = (torch.round(prompt) + torch.round(decoded)).clamp(16, 4096)
    lens = [int(x) for x in lens.tolist()]
    need = sum(_cdiv(n, 16) for n in lens)
    return Workload("llama3.1-8b_decode_layer", num_seqs, 32, 8, 128, 16,
                    seq_lens=lens, pool_blocks=math.ceil(1.3 * need), seed=3)


def shared_prefix(block_size: int = 16, num_seqs: int = 256,
                  prefix: int = 2048) -> Workload:
    """8B shape; every sequence shares one 2048-token prefix (same physical
    blocks) plus a private suffix uniform in [1, 512]."""
    g = _gen(4)
    suffix = torch.randint(1, 513, (num_seqs,), generator=g).tolist()
    lens = [prefix + s for s in suffix]
    need = prefix // block_size + sum(
        _cdiv(prefix + s, block_size) - prefix // block_size for s in suffix)
    return Workload(f"shared_prefix_bs{block_size}", num_seqs, 32, 8, 128,
                    block_size, seq_lens=lens,
                    pool_blocks=math.ceil(1.3 * need), seed=4,
                    shared_prefix=prefix)


def llama31_70b_128k(num_seqs: int = 8, seq_len: int = 131072) -> Workload:
    """Llama-3.1-70B-shaped long-context layer: Hq=64, Hkv=8, d=128, bs=16,
    B=8 sequences of 131072 tokens; K/V N(0,1) with 1% outliers x20; the
    pool holds exactly the blocks needed."""
    need = num_seqs * _cdiv(seq_len, 16)
    return Workload("llama3.1-70b_128k_decode_layer", num_seqs, 64, 8, 128, 16,
                    seq_lens=[seq_len] * num_seqs, pool_blocks=need, seed=5,
                    outlier_prob=0.01, outlier_scale=20.0)


WORKLOADS = {
    "tiny": tiny,
    "llama3.2-1b": llama32_1b,
    "llama3.1-8b": llama31_8b,
    "shared_prefix_bs8": lambda: shared_prefix(8),
    "shared_prefix_bs16": lambda: shared_prefix(16),
    "shared_prefix_bs32": lambda: shared_prefix(32),
    "llama3.1-70b-128k": llama31_70b_128k,
}


# ------------------------------------------------------------- op script ---
def free_order(w: Workload) -> list:
    """Seeded permutation in which a freshly allocated pool is freed, so the
    LIFO free list hands blocks out in a scattered order (or, for a
    workload with ``scattered=False``, in order 0, 1, 2, ..., which gives
    every sequence contiguous physical blocks)."""
    if not w.scattered:
        return list(range(w.pool_blocks - 1, -1, -1))
    return torch.randperm(w.pool_blocks, generator=_gen(1000 + w.seed)).tolist()


def contiguous(w: Workload) -> Workload:
    """The same workload with every sequence's blocks physically contiguous
    (the paging tax is the difference between the two)."""
    from dataclasses import replace
    return replace(w, name=w.name + "_contiguous", scattered=False)


def build_script(w: Workload) -> list:
    """Ops that bring a block manager to the pre-step state.

    ("alloc", n) / ("free_list", ids) / ("append", seq, n) / ("fork", child,
    parent, ntok).  After the script, sequence b holds ``seq_lens[b] - 1``
    tokens; the step itself is one ("append", b, 1) per sequence.
    """
    ops = [("alloc", w.pool_blocks), ("free_list", free_order(w))]
    if w.shared_prefix:
        ops.append(("append", 0, w.shared_prefix))
        for b in range(1, w.num_seqs):
            ops.append(("fork", b, 0, w.shared_prefix))
        for b in range(w.num_seqs):
            ops.append(("append", b, w.seq_lens[b] - 1 - w.shared_prefix))
    else:
        for b in range(w.num_seqs):
            ops.append(("append", b, w.seq_lens[b] - 1))
    return ops


# --------------------------------------------------------- random values ---
def normal_bf16(shape, seed: int, device="cpu", outlier_prob: float = 0.0,
                outlier_scale: float = 1.0, chunk: int = 1 << 26):
    """Standard normal values rounded to bf16, optionally with outliers.

    Drawn in chunks of ``chunk`` elements from one seeded generator on
    ``device`` so that very large pools need no fp32 copy of the whole tensor.
    """
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        e = min(s + chunk, flat.numel())
        x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        if outlier_prob > 0:
            m = torch.rand(e - s, generator=g, device=device) < outlier_prob
            x = torch.where(m, x * outlier_scale, x)
        flat[s:e] = x.to(torch.bfloat16)
    return out


def distinct_slots(num_slots: int, count: int, seed: int) -> torch.Tensor:
    """``count`` distinct slot indices in [0, num_slots), seeded, int64."""
    return torch.randperm(num_slots, generator=_gen(seed))[:count].to(torch.int64)
