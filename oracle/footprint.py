"""KV footprint arithmetic (oracle; test infrastructure only).

The "Fragmentation" lesson page (section "Notes") gives the per-token KV
footprint of a decoder-only model as

    b_tok = 2 * L * H_kv * d_h * s

(2 for K and V, L layers, H_kv KV heads, head dimension d_h, s bytes per
scalar); a request of length T then needs T * b_tok bytes.  The page "Paged
Attention and KV Cache Fragmentation" (section "Quantization as a way to
stretch paged memory further") works it for Llama 3.1 70B at 128K tokens:
2 * 80 * 8 * 128 * 131072 * 2 B ~= 42.9 GB in BF16, half that in FP8.

For one decode layer-step the algorithmic KV bytes read are the footprint of
every cached token of every sequence at L = 1, plus, for FP8, the two fp32
per-(block, head) scales of every block touched.
"""
from __future__ import annotations


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                       bytes_per_scalar: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_scalar


def decode_step_kv_bytes(seq_lens, num_kv_heads: int, head_dim: int,
                         bytes_per_scalar: int, block_size: int = 0,
                         scale_bytes: int = 0) -> int:
    """Algorithmic KV bytes one layer's decode step reads.

    ``scale_bytes`` > 0 adds K and V scales (``scale_bytes`` each) for every
    (block, KV head) a sequence touches, ceil(n / block_size) blocks.
    """
    total = 0
    for n in seq_lens:
        n = int(n)
        total += n * kv_bytes_per_token(1, num_kv_heads, head_dim, bytes_per_scalar)
        if scale_bytes:
            total += 2 * (-(-n // block_size)) * num_kv_heads * scale_bytes
    return total


def nvfp4_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int) -> int:
    """NVFP4 cache bytes per token: half a byte per value plus one E4M3
    block scale per 16 values, for K and V of every layer.  (The page's
    "about 10.7 GB" for Llama 3.1 70B at 128K counts the 4-bit values alone.)"""
    return 2 * num_layers * num_kv_heads * (head_dim // 2 + head_dim // 16)
