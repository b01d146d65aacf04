"""Byte and bit accounting of the INT2 cache.

Test infrastructure only (see the package docstring).

[Escha log] part 2, fix 1: INT2 codes occupy 0.25 byte per element; the
supplementary table gives the INT2 KV cost per token as 8.0 KiB for 16
full-attention layers × 4 KV heads and 2.5 KiB for 10 layers × 2 KV heads
(head_dim 256, K and V, codes only).  [OSCAR news] "サービングシステム" section:
at 128K context the BF16 sink and recent windows are 0.24% of all tokens;
the intro quotes 2.28 bits per KV element.
"""


def code_bytes_per_token(num_layers, num_kv_heads, head_dim):
    """INT2 code bytes per token over layers, heads, K and V (scales excluded)."""
    return num_layers * num_kv_heads * head_dim * 2 * 0.25


def record_bytes(head_dim, group_size, scale_bits=16):
    """Bytes of one (slot, KV head) record: K and V codes and (s, z) per group;
    fp16 pairs (scale_bits 16) padded to 16 bytes, E4M3 pairs (8) to 8 bytes."""
    ng = head_dim // group_size
    raw = head_dim // 2 + 2 * 2 * (scale_bits // 8) * ng
    al = 16 if scale_bits == 16 else 8
    return (raw + al - 1) // al * al


def window_fraction(L, sink=64, recent=256):
    """Fraction of a request's L tokens held in the BF16 windows."""
    return min(L, sink + recent) / L


def bits_per_element(L, group_size, sink=64, recent=256, scale_bits=16):
    """Average stored bits per KV element at context L.

    BF16 windows cost 16 bits; an INT2 element costs 2 bits plus its share of
    the 2·scale_bits bits of (s, z) per group of G channels (fp16: 32, E4M3: 16).
    """
    w = min(L, sink + recent)
    return (16.0 * w + (2.0 + 2.0 * scale_bits / group_size) * (L - w)) / L
