"""CPU oracle of the Qwen2 decoder forward -- TEST INFRASTRUCTURE ONLY.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``.  The product path (the ``qwen2_decoder_forward_gb300``
package and its CUDA library) never imports it and has no CPU fallback.

Parity status per function (what pins each one is in ``tests/``):
rms_norm, rope_neox, silu, softmax_rows, gqa_attention, Qwen2Oracle.forward
(head_dim 64 and 128, tied and untied LM head, f16 / Q8_0 / Q4_0 weights,
Q8_0 activations), Qwen2Oracle.greedy_generate, quantize_q8_0 /
dequantize_q8_0, q8_0_matmul, quantize_q4_0 / dequantize_q4_0 and the
nibble packing are all pinned.  End-to-end logits of a real Qwen2
checkpoint are parity unpinned (no checkpoint exists here).
"""
from .qwen2_oracle import (KVCache, OracleConfig, OracleWeights, PositionError,
                           Qwen2Oracle, gqa_attention, greedy_ids, rms_norm,
                           rope_inv_freq, rope_neox, silu, softmax_rows)
from .q4_0 import dequantize_q4_0, pack_nibbles, quantize_q4_0, unpack_nibbles
from .q8_0 import QK, dequantize_q8_0, q8_0_matmul, quantize_q8_0

__all__ = [
    "KVCache", "OracleConfig", "OracleWeights", "PositionError", "Qwen2Oracle",
    "gqa_attention", "greedy_ids", "rms_norm", "rope_inv_freq", "rope_neox",
    "silu", "softmax_rows", "QK", "dequantize_q8_0", "quantize_q8_0", "q8_0_matmul",
    "dequantize_q4_0", "quantize_q4_0", "pack_nibbles", "unpack_nibbles",
    "build_oracle",
]


def build_oracle(shape, weights: dict, n_ctx: int, weight_format: str = "f16",
                 **kw) -> Qwen2Oracle:
    """Convenience: an oracle for ``shape`` (a ``synth.ModelShape``)."""
    cfg = OracleConfig.from_shape(shape, n_ctx)
    return Qwen2Oracle(cfg, OracleWeights(weights, weight_format), **kw)
