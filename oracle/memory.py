"""KV cache memory arithmetic.

Test infrastructure only (see the package docstring).

Source: Flash-MoE "Context Optimization", Memory Budget Calculator: the KV bytes are
layers x 2 (K and V) x KV heads x head_dim x bytes per element x positions, where an
FP8 cache adds about 4 bytes of scale per position per cache (one binary32 scale per
position for K and one for V, in every layer: the reading of "For each position"
in FP8 KV Cache > How It Works).  positions = min(context, window) when a window is
set.

Parity: pinned by tests/test_oracle_memory.py against the page's own table values
(tests/golden/pages_figures.json).
"""

ELEM_BYTES = {"f32": 4, "bf16": 2, "e4m3": 1}


def kv_elements_per_position(layers, kv_heads, head_dim):
    return layers * 2 * kv_heads * head_dim


def kv_bytes_per_position(layers, kv_heads, head_dim, fmt):
    """Bytes one position occupies across all layers, K and V, scales included."""
    payload = kv_elements_per_position(layers, kv_heads, head_dim) * ELEM_BYTES[fmt]
    scales = layers * 2 * 4 if fmt == "e4m3" else 0
    return payload + scales


def kv_payload_bytes_per_position(layers, kv_heads, head_dim, fmt):
    """Bytes of K/V elements only (no scales), as in the page's first table."""
    return kv_elements_per_position(layers, kv_heads, head_dim) * ELEM_BYTES[fmt]


def kv_cache_bytes(layers, kv_heads, head_dim, fmt, context, window=0, with_scales=False):
    positions = min(context, window) if window else context
    per = (kv_bytes_per_position(layers, kv_heads, head_dim, fmt) if with_scales
           else kv_payload_bytes_per_position(layers, kv_heads, head_dim, fmt))
    return per * positions
