"""Seeded synthetic inputs for the Qwen2 decoder forward.

This module makes model shapes, weights, prompts and positions from fixed
seeds.  It is the one module that both the CUDA path's tests/bench and the
CPU oracle draw their inputs from; it holds none of the forward's arithmetic
(no norm, projection, rotation, attention or quantisation), only random draws
and the shape tables.

Weight recipe (one ``numpy.random.Generator(PCG64(seed))`` stream, drawn in
the order embed; per layer attn_norm, wq, bq, wk, bk, wv, bv, wo, ffn_norm,
wg, wu, wd; then final_norm):

* matrices: ``0.02 * N(0,1)`` drawn in float32, then rounded to float16 -- the
  GPU-side storage type of the seven linear weights and the tied LM head
  (Module 7 -- Qwen2 / Qwen2.5, section 7.4: f16 linear weights and LM head,
  f32 bias and norm weights);
* biases ``bq, bk, bv``: ``0.02 * N(0,1)`` kept in float32;
* RMSNorm weights: ``1 + 0.1 * N(0,1)`` in float32.

Layouts follow the HF checkpoint convention ``[out_features][in_features]``
(Module 7 -- Qwen2 / Qwen2.5, Lab 7: q_proj [896, 896], k_proj [128, 896],
gate_proj [4864, 896]).
"""
from __future__ import annotations

import dataclasses
import functools

import numpy as np


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """The config fields of a Qwen2 decoder that size its tensors.

    Field names follow the config.json keys listed in Module 7 -- Qwen2 /
    Qwen2.5, section 7.1 (hidden_size, intermediate_size, num_hidden_layers,
    num_attention_heads, num_key_value_heads, vocab_size, rope_theta,
    rms_norm_eps, tie_word_embeddings).
    """

    name: str
    n_layer: int
    hidden: int
    n_head: int
    n_kv_head: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    tie_embeddings: bool = True   # False: a separate LM head matrix


SHAPES = {
    # Toy 2-layer Qwen2: hidden 256, 4 q heads / 2 kv heads of dim 64.
    "toy": ModelShape("toy", n_layer=2, hidden=256, n_head=4, n_kv_head=2,
                      head_dim=64, intermediate=1024, vocab=4096),
    # Qwen2.5-0.5B (nnterp encyclopedia qwen2, "Config" table; Module 7
    # section 7.1 table).
    "qwen2.5-0.5b": ModelShape("qwen2.5-0.5b", n_layer=24, hidden=896,
                               n_head=14, n_kv_head=2, head_dim=64,
                               intermediate=4864, vocab=151936),
    # A ragged shape for tail handling: 6 q heads over 2 kv heads (group 3),
    # a prime vocabulary, an intermediate that is not a multiple of 128.
    "ragged": ModelShape("ragged", n_layer=3, hidden=384, n_head=6,
                         n_kv_head=2, head_dim=64, intermediate=640,
                         vocab=5003),
    # Multi-head (no grouping) variant: num_key_value_heads == num_heads,
    # as on the Qwen1.5 0.5B/7B checkpoints.
    "toy-mha": ModelShape("toy-mha", n_layer=2, hidden=256, n_head=4,
                          n_kv_head=4, head_dim=64, intermediate=1024,
                          vocab=4096),
    # eight query heads per kv head, the widest group the kernels take
    "toy-g8": ModelShape("toy-g8", n_layer=2, hidden=512, n_head=8,
                         n_kv_head=1, head_dim=64, intermediate=1024,
                         vocab=4096),
    # head_dim 128, the head width of every size above 0.5B (nnterp
    # encyclopedia qwen2, "Grouped-query attention"): 4 q heads over 2 kv
    # heads, tied LM head (as 1.5B and 3B).
    "toy-hd128": ModelShape("toy-hd128", n_layer=2, hidden=512, n_head=4,
                            n_kv_head=2, head_dim=128, intermediate=1024,
                            vocab=4096),
    # head_dim 128 with 8 q heads over 4 kv heads and an untied LM head, the
    # layout of 7B (28 over 4, separate embedding and unembedding: nnterp
    # "Grouped-query attention" and "The readout is the plain projection").
    "toy-untied": ModelShape("toy-untied", n_layer=2, hidden=1024, n_head=8,
                             n_kv_head=4, head_dim=128, intermediate=1024,
                             vocab=4096, tie_embeddings=False),
    # The toy shape (head_dim 64) with an untied LM head: the separate
    # readout on the batch-1 persistent decode kernel.
    "toy-untied-hd64": ModelShape("toy-untied-hd64", n_layer=2, hidden=256,
                                  n_head=4, n_kv_head=2, head_dim=64,
                                  intermediate=1024, vocab=4096,
                                  tie_embeddings=False),
}


LAYER_KEYS = ("attn_norm", "wq", "bq", "wk", "bk", "wv", "bv", "wo",
              "ffn_norm", "wg", "wu", "wd")


def _draw(rng: np.random.Generator, shape, kind: str) -> np.ndarray:
    z = rng.standard_normal(size=shape, dtype=np.float32)
    if kind == "matrix":
        return (np.float32(0.02) * z).astype(np.float16)
    if kind == "bias":
        return np.float32(0.02) * z
    if kind == "norm":
        return np.float32(1.0) + np.float32(0.1) * z
    raise ValueError(kind)


def make_weights(shape: ModelShape, seed: int = 0) -> dict:
    """Seeded weights of ``shape``; see the module docstring for the recipe.

    Returns ``{"embed": f16 [V, H], "final_norm": f32 [H], "layers": [dict]}``
    where each layer dict has the keys of :data:`LAYER_KEYS`.  The LM head is
    tied to ``embed`` (no separate array) unless ``shape.tie_embeddings`` is
    False; then ``"lm_head"``, f16 [V, H], is drawn after every other array,
    so the tied arrays of a shape are the same draws either way.
    """
    return _make_weights_cached(shape, seed)


@functools.lru_cache(maxsize=2)
def _make_weights_cached(shape: ModelShape, seed: int) -> dict:
    rng = np.random.Generator(np.random.PCG64(seed))
    H, I, V = shape.hidden, shape.intermediate, shape.vocab
    q_out = shape.n_head * shape.head_dim
    kv_out = shape.n_kv_head * shape.head_dim
    w = {"embed": _draw(rng, (V, H), "matrix"), "layers": []}
    for _ in range(shape.n_layer):
        layer = {
            "attn_norm": _draw(rng, (H,), "norm"),
            "wq": _draw(rng, (q_out, H), "matrix"),
            "bq": _draw(rng, (q_out,), "bias"),
            "wk": _draw(rng, (kv_out, H), "matrix"),
            "bk": _draw(rng, (kv_out,), "bias"),
            "wv": _draw(rng, (kv_out, H), "matrix"),
            "bv": _draw(rng, (kv_out,), "bias"),
            "wo": _draw(rng, (H, q_out), "matrix"),
            "ffn_norm": _draw(rng, (H,), "norm"),
            "wg": _draw(rng, (I, H), "matrix"),
            "wu": _draw(rng, (I, H), "matrix"),
            "wd": _draw(rng, (H, I), "matrix"),
        }
        w["layers"].append(layer)
    w["final_norm"] = _draw(rng, (H,), "norm")
    if not shape.tie_embeddings:
        w["lm_head"] = _draw(rng, (V, H), "matrix")
    for arr in _iter_arrays(w):
        arr.setflags(write=False)
    return w


def _iter_arrays(w):
    yield w["embed"]
    yield w["final_norm"]
    if "lm_head" in w:
        yield w["lm_head"]
    for layer in w["layers"]:
        for k in LAYER_KEYS:
            yield layer[k]


def make_tokens(vocab: int, n: int, seed: int) -> np.ndarray:
    """``n`` uniform-random token ids in ``[0, vocab)`` as int32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def make_start_positions(n_seq: int, lo: int, hi_inclusive: int,
                         seed: int) -> np.ndarray:
    """``n_seq`` start positions drawn uniformly from ``[lo, hi_inclusive]``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi_inclusive + 1, size=n_seq,
                        dtype=np.int64).astype(np.int32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One measured or parity-checked run of the decoder forward."""

    name: str
    shape: str
    n_seq: int
    prompt_len: int          # tokens per sequence prefilled first (0: ragged)
    decode_steps: int
    n_ctx: int
    weight_format: str       # "f16" or "q8_0"
    prefill: str             # "f32" (SIMT, f32 activations) or "tensor" (f16 operands)
    token_seed: int
    weight_seed: int = 0
    ragged_lo: int = 0       # ragged prompt lengths drawn from [lo, hi]
    ragged_hi: int = 0
    ragged_seed: int = 0

    def prompt_lengths(self) -> np.ndarray:
        if self.prompt_len > 0:
            return np.full(self.n_seq, self.prompt_len, dtype=np.int32)
        return make_start_positions(self.n_seq, self.ragged_lo,
                                    self.ragged_hi, self.ragged_seed)

    def prompts(self, vocab: int) -> list:
        lens = self.prompt_lengths()
        total = int(lens.sum())
        toks = make_tokens(vocab, total, self.token_seed)
        out, off = [], 0
        for n in lens:
            out.append(toks[off:off + int(n)])
            off += int(n)
        return out


WORKLOADS = {
    # Toy model, one sequence: 16-token prompt, 16 greedy decode steps.
    "toy-decode": Workload("toy-decode", "toy", n_seq=1, prompt_len=16,
                           decode_steps=16, n_ctx=64, weight_format="f16",
                           prefill="f32", token_seed=1001),
    # Qwen2.5-0.5B shape, batch 1: 128-token prompt, 256 greedy steps.
    "0.5b-decode-b1": Workload("0.5b-decode-b1", "qwen2.5-0.5b", n_seq=1,
                               prompt_len=128, decode_steps=256, n_ctx=4096,
                               weight_format="f16", prefill="f32",
                               token_seed=1002),
    # Long-context batch-1 decode: 4000-token prompt, steps at 4000..4095.
    "0.5b-decode-b1-long": Workload("0.5b-decode-b1-long", "qwen2.5-0.5b",
                                    n_seq=1, prompt_len=4000,
                                    decode_steps=96, n_ctx=4096,
                                    weight_format="f16", prefill="f32",
                                    token_seed=1003),
    # Prefill-heavy: 8 sequences x 512 tokens, tensor-core prefill, tail cut.
    "0.5b-prefill-8x512": Workload("0.5b-prefill-8x512", "qwen2.5-0.5b",
                                   n_seq=8, prompt_len=512, decode_steps=0,
                                   n_ctx=4096, weight_format="f16",
                                   prefill="tensor", token_seed=1004),
    # Batched decode: 32 sequences at ragged start positions, Q8_0 weights.
    "0.5b-decode-b32-q8": Workload("0.5b-decode-b32-q8", "qwen2.5-0.5b",
                                   n_seq=32, prompt_len=0, decode_steps=64,
                                   n_ctx=4096, weight_format="q8_0",
                                   prefill="f32", token_seed=1005,
                                   ragged_lo=256, ragged_hi=4032,
                                   ragged_seed=2005),
}
