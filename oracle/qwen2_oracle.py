"""Plain float64 CPU forward of the Qwen2 decoder -- TEST INFRASTRUCTURE ONLY.

This is the oracle the CUDA path is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import,
call or execute it; the library never does.  It shares no code, table or
constant generator with the CUDA path: the two meet only in the seeded input
generators of the ``synth`` module.

Every step is the plain definition, in float64, in the order the pages give
it (minfer "Qwen2 / Qwen2.5 Architecture Support", section 1, the layer
diagram):

    h - RMSNorm - WQ/WK/WV matmuls + bias - RoPE(Q, K) - KV store
      - GQA attention (Q K^T scale -> softmax -> V) - WO matmul - + residual
      - RMSNorm - gate/up matmuls - SiLU(gate) * up - down matmul - + residual

then the final RMSNorm and the LM head (nnterp encyclopedia qwen2,
"The readout is the plain projection"; Module 7 section 7.3: tied, W_lm =
E, unless the weights carry a separate ``lm_head``).
A matrix product is a library primitive (numpy ``@``); there is no blocking,
fusion or reordering beyond the definition.

Readings of points the pages leave open (each also listed in the design
notes):

* storage: f16 weights and the f32 biases / norm weights are widened to
  float64 exactly; activations, the KV cache and all sums are float64;
* RMSNorm multiplies by ``w`` (not ``1 + w``) with eps inside the root;
* RoPE angles ``p * theta^(-2i/hd)`` in float64, NeoX ``rotate_half`` pairs
  ``(i, i + hd/2)``;
* greedy ids are the lowest index of the maximum of the float32-rounded
  logits (the precision the kernel decides it in);
* the KV store of a call happens before its attention; a row at position
  ``p`` attends to cache slots ``0..p`` of its own sequence.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import q4_0 as _q4
from . import q8_0 as _q8


class PositionError(ValueError):
    """A position outside ``[0, n_ctx)``: a hard error, never a truncation
    (minfer "Qwen2 / Qwen2.5 Architecture Support", section 6: positions[i] <
    n_ctx is enforced with a hard Err in the KV-store arm; section 7 item 5).
    """


@dataclasses.dataclass
class OracleConfig:
    n_layer: int
    hidden: int
    n_head: int
    n_kv_head: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float
    rope_theta: float
    n_ctx: int

    @classmethod
    def from_shape(cls, shape, n_ctx: int) -> "OracleConfig":
        return cls(shape.n_layer, shape.hidden, shape.n_head, shape.n_kv_head,
                   shape.head_dim, shape.intermediate, shape.vocab,
                   shape.rms_eps, shape.rope_theta, n_ctx)


# ---------------------------------------------------------------------------
# The per-step definitions.
# ---------------------------------------------------------------------------

def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm: ``x / sqrt(mean(x^2) + eps) * w`` over the last axis.

    Pre-norm with no mean subtraction and no bias (Module 7 -- Qwen2 /
    Qwen2.5, section 7.2 table, row "normalization"; eps = rms_norm_eps =
    1e-6, section 7.1).
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """``theta^(-2i/hd)`` for ``i < hd/2`` (the RoPE base is rope_theta,
    Module 7 section 7.1 table; 1e6 on Qwen2.5)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_neox(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """NeoX / ``rotate_half`` rotary embedding of ``x [T, heads, hd]``.

    Pairs are ``(i, i + hd/2)`` -- the NonInterleaved style of the Qwen2
    family (minfer page section 3; Module 7 section 7.2 "GPT-NeoX
    rotate_half").  With ``a = x_i``, ``b = x_{i+hd/2}`` and angle
    ``phi = p * theta^(-2i/hd)``:
    ``a' = a cos(phi) - b sin(phi)``, ``b' = b cos(phi) + a sin(phi)``.
    """
    hd = x.shape[-1]
    half = hd // 2
    phi = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(hd, theta)[None, :]
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    a = x[..., :half]
    b = x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z)) (hidden_act "silu", nnterp Config table)."""
    return z / (1.0 + np.exp(-z))


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted; ``-inf`` entries get 0."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def gqa_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                  positions: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention of rows ``q [T, nh, hd]`` against a
    sequence's cache ``K, V [P, nkv, hd]``.

    Query head ``h`` reads key/value head ``g = h // (nh / nkv)``, so kv head
    ``j`` serves query heads ``j*group .. j*group + group - 1`` (nnterp
    encyclopedia qwen2, "Grouped-query attention": an edit to kv head j
    reaches query heads 7j to 7j+6).  Scores are ``q.k * hd^-0.5``; a row at
    position ``p`` sees slots ``0..p`` -- full causal, no sliding window
    ("The sliding-window keys do nothing").
    """
    T, nh, hd = q.shape
    P, nkv, _ = K.shape
    group = nh // nkv
    scale = float(hd) ** -0.5
    visible = np.arange(P)[None, :] <= np.asarray(positions)[:, None]  # [T, P]
    out = np.empty((T, nh, hd), dtype=np.float64)
    for h in range(nh):
        g = h // group
        s = (q[:, h, :] @ K[:, g, :].T) * scale
        s = np.where(visible, s, -np.inf)
        out[:, h, :] = softmax_rows(s) @ V[:, g, :]
    return out


def greedy_ids(logits: np.ndarray) -> np.ndarray:
    """Lowest index of the maximum, decided on float32-rounded logits."""
    return np.argmax(logits.astype(np.float32), axis=-1).astype(np.int32)


# ---------------------------------------------------------------------------
# Weights and cache.
# ---------------------------------------------------------------------------

class _Layer:
    __slots__ = ("attn_norm", "wqkv", "bqkv", "wo", "ffn_norm", "wgu", "wd",
                 "wqkv_codes", "wo_codes", "wgu_codes", "wd_codes")


class OracleWeights:
    """float64 copies of one model's weights.

    ``weight_format`` "f16" widens the f16 matrices exactly; "q8_0" (or
    "q4_0") first quantises every linear matrix and the tied embedding with
    :func:`oracle.q8_0.quantize_q8_0` (:func:`oracle.q4_0.quantize_q4_0`)
    and widens the dequantised values (the
    embedding gather and the LM head then both read the quantised matrix,
    since it is one tied matrix, Module 7 section 7.3).  Q/K/V are stacked
    into one ``[(nh + 2 nkv) hd, H]`` matrix and gate/up into one
    ``[2I, H]`` matrix; the unfused forward reads row slices of them.  With
    "q8_0" each matrix also keeps its codes (``*_codes``: int8 values and
    f16 scales) for the Q8_0-activation products.
    """

    def __init__(self, weights: dict, weight_format: str = "f16"):
        if weight_format not in ("f16", "q8_0", "q4_0"):
            raise ValueError(weight_format)
        self.weight_format = weight_format

        def mat(a):
            """(float64 matrix, its Q8_0 codes or None)."""
            if weight_format == "q8_0":
                q, d = _q8.quantize_q8_0(a)
                return _q8.dequantize_q8_0(q, d), (q, d)
            if weight_format == "q4_0":
                q, d = _q4.quantize_q4_0(a)
                return _q4.dequantize_q4_0(q, d), None
            return np.asarray(a, dtype=np.float64), None

        def stack(parts):
            m = np.concatenate([p[0] for p in parts], axis=0)
            if any(p[1] is None for p in parts):
                return m, None
            return m, (np.concatenate([p[1][0] for p in parts], axis=0),
                       np.concatenate([p[1][1] for p in parts], axis=0))

        self.embed, self.embed_codes = mat(weights["embed"])
        # The readout matrix: the embedding itself when the LM head is tied
        # (0.5B to 3B), a separate matrix from 7B up (nnterp encyclopedia
        # qwen2, "The readout is the plain projection").
        lm = weights.get("lm_head")
        self.lm_head, self.lm_head_codes = (self.embed, self.embed_codes) if lm is None else mat(lm)
        self.final_norm = np.asarray(weights["final_norm"], dtype=np.float64)
        self.layers = []
        for lw in weights["layers"]:
            L = _Layer()
            L.attn_norm = np.asarray(lw["attn_norm"], dtype=np.float64)
            L.wqkv, L.wqkv_codes = stack([mat(lw["wq"]), mat(lw["wk"]), mat(lw["wv"])])
            L.bqkv = np.concatenate([lw["bq"], lw["bk"], lw["bv"]]).astype(np.float64)
            L.wo, L.wo_codes = mat(lw["wo"])
            L.ffn_norm = np.asarray(lw["ffn_norm"], dtype=np.float64)
            L.wgu, L.wgu_codes = stack([mat(lw["wg"]), mat(lw["wu"])])
            L.wd, L.wd_codes = mat(lw["wd"])
            self.layers.append(L)


class KVCache:
    """One sequence's key/value cache, ``[n_layer, n_ctx, n_kv_head, hd]``
    each, float64, zero-initialised; slot = position (minfer page section 6:
    KV positions are data)."""

    def __init__(self, cfg: OracleConfig):
        shp = (cfg.n_layer, cfg.n_ctx, cfg.n_kv_head, cfg.head_dim)
        self.K = np.zeros(shp, dtype=np.float64)
        self.V = np.zeros(shp, dtype=np.float64)


# ---------------------------------------------------------------------------
# The forward.
# ---------------------------------------------------------------------------

class Qwen2Oracle:
    """The plain Qwen2 decoder forward over one sequence's rows.

    ``fuse_qkv`` / ``fuse_ffn`` choose between one product with the stacked
    matrix and separate products with its row slices -- the two forms the
    minfer page (section 3, "Decode fusions") says are bit-identical.
    """

    def __init__(self, cfg: OracleConfig, weights: OracleWeights,
                 fuse_qkv: bool = True, fuse_ffn: bool = True, act_q8: bool = False):
        if act_q8 and (weights.weight_format != "q8_0" or not (fuse_qkv and fuse_ffn)):
            raise ValueError("Q8_0 activations need Q8_0 weights and the fused products")
        if cfg.hidden != cfg.n_head * cfg.head_dim:
            raise ValueError("head_dim must equal hidden / n_head")
        if cfg.n_head % cfg.n_kv_head:
            raise ValueError("n_head must be a multiple of n_kv_head")
        self.cfg = cfg
        self.w = weights
        self.fuse_qkv = fuse_qkv
        self.fuse_ffn = fuse_ffn
        self.act_q8 = act_q8

    def _lin(self, x: np.ndarray, W: np.ndarray, codes) -> np.ndarray:
        """x @ W^T; with ``act_q8`` the product of the Q8_0-quantised rows of x
        and W's Q8_0 codes (:func:`oracle.q8_0.q8_0_matmul`)."""
        if self.act_q8:
            return _q8.q8_0_matmul(x, *codes)
        return x @ W.T

    def new_cache(self) -> KVCache:
        return KVCache(self.cfg)

    # -- sub-steps ----------------------------------------------------------

    def _qkv(self, L: _Layer, n: np.ndarray):
        c = self.cfg
        nq, nk = c.n_head * c.head_dim, c.n_kv_head * c.head_dim
        if self.fuse_qkv:
            y = self._lin(n, L.wqkv, L.wqkv_codes) + L.bqkv
            q, k, v = y[:, :nq], y[:, nq:nq + nk], y[:, nq + nk:]
        else:
            q = n @ L.wqkv[:nq].T + L.bqkv[:nq]
            k = n @ L.wqkv[nq:nq + nk].T + L.bqkv[nq:nq + nk]
            v = n @ L.wqkv[nq + nk:].T + L.bqkv[nq + nk:]
        return q, k, v

    def _ffn(self, L: _Layer, m: np.ndarray):
        I = self.cfg.intermediate
        if self.fuse_ffn:
            gu = self._lin(m, L.wgu, L.wgu_codes)
            g, u = gu[:, :I], gu[:, I:]
        else:
            g = m @ L.wgu[:I].T
            u = m @ L.wgu[I:].T
        act = silu(g)
        neurons = act * u
        return act, neurons, self._lin(neurons, L.wd, L.wd_codes)

    # -- the whole forward ----------------------------------------------------

    def forward(self, cache: KVCache, tokens, positions, n_out: int | None = None,
                tail_cut: bool = True, probes: dict | None = None) -> dict:
        """Run rows ``tokens`` at ``positions`` of one sequence.

        Stores each row's rotated key and value at its position, attends
        causally over the cache, and returns, for the last ``n_out`` rows
        (all rows when ``None``): ``logits`` [n_out, V] float64,
        ``final_norm_output`` [n_out, H] and ``ids`` [n_out] int32.

        ``tail_cut`` keeps only the last ``n_out`` rows before the final
        layer's FFN (minfer page section 3, "G3 tail-row optimization"); the
        tail rows' results are the same either way.

        ``probes``, when a dict, receives the named intermediates of the
        nnterp encyclopedia ("02 . support()" value table), each a list over
        layers where per layer.
        """
        c = self.cfg
        tokens = np.asarray(tokens, dtype=np.int64)
        positions = np.asarray(positions, dtype=np.int64)
        T = tokens.shape[0]
        if positions.shape != (T,):
            raise ValueError("one position per token")
        if T == 0:
            raise ValueError("no rows")
        if np.any(positions < 0) or np.any(positions >= c.n_ctx):
            raise PositionError(f"position outside [0, {c.n_ctx})")
        if np.any(tokens < 0) or np.any(tokens >= c.vocab):
            raise ValueError("token id outside [0, vocab)")
        n_keep = T if n_out is None else int(n_out)
        if not 1 <= n_keep <= T:
            raise ValueError("n_out outside [1, T]")

        rec = probes is not None
        if rec:
            for key in ("layer_input", "attention_norm_output", "attention_queries",
                        "attention_keys", "attention_values", "attention_premix",
                        "attention_output", "layer_mid", "mlp_norm_output",
                        "mlp_activation", "mlp_neurons", "mlp_output", "layer_output"):
                probes[key] = []

        # token_embeddings: x = E[t] (embed_tokens, [151936, 896]).
        x = self.w.embed[tokens]
        if rec:
            probes["token_embeddings"] = x.copy()
        P = int(positions.max()) + 1
        for li, L in enumerate(self.w.layers):
            if rec:
                probes["layer_input"].append(x.copy())
            n = rms_norm(x, L.attn_norm, c.rms_eps)
            q, k, v = self._qkv(L, n)
            q = rope_neox(q.reshape(T, c.n_head, c.head_dim), positions, c.rope_theta)
            k = rope_neox(k.reshape(T, c.n_kv_head, c.head_dim), positions, c.rope_theta)
            v = v.reshape(T, c.n_kv_head, c.head_dim)
            cache.K[li, positions] = k
            cache.V[li, positions] = v
            o = gqa_attention(q, cache.K[li, :P], cache.V[li, :P], positions)
            o = o.reshape(T, c.n_head * c.head_dim)
            attn_out = self._lin(o, L.wo, L.wo_codes)
            if rec:
                probes["attention_norm_output"].append(n)
                probes["attention_queries"].append(q)
                probes["attention_keys"].append(k)
                probes["attention_values"].append(v)
                probes["attention_premix"].append(o)
                probes["attention_output"].append(attn_out)
            x = x + attn_out
            if li == c.n_layer - 1 and tail_cut and n_keep < T:
                x = x[T - n_keep:]
            if rec:
                probes["layer_mid"].append(x.copy())
            m = rms_norm(x, L.ffn_norm, c.rms_eps)
            act, neurons, mlp_out = self._ffn(L, m)
            x = x + mlp_out
            if rec:
                probes["mlp_norm_output"].append(m)
                probes["mlp_activation"].append(act)
                probes["mlp_neurons"].append(neurons)
                probes["mlp_output"].append(mlp_out)
                probes["layer_output"].append(x.copy())
        x = x[x.shape[0] - n_keep:]
        f = rms_norm(x, self.w.final_norm, c.rms_eps)
        logits = self._lin(f, self.w.lm_head, self.w.lm_head_codes)
        if rec:
            probes["final_norm_output"] = f
            probes["logits"] = logits
        return {"logits": logits, "final_norm_output": f, "ids": greedy_ids(logits)}

    # -- loops built on forward ---------------------------------------------

    def prefill(self, cache: KVCache, tokens, start: int = 0, **kw) -> dict:
        """Rows ``tokens`` at positions ``start, start+1, ...``; last row out."""
        pos = np.arange(start, start + len(tokens), dtype=np.int64)
        return self.forward(cache, tokens, pos, n_out=1, **kw)

    def greedy_decode(self, cache: KVCache, first_token: int, start_pos: int,
                      n_steps: int, keep_logits: bool = True) -> dict:
        """Feed ``first_token`` at ``start_pos`` and each step's id at the next
        position (positions are data, minfer page section 6); ``n_steps``
        rows.  Returns ``ids`` [n_steps] (the id produced by each step) and,
        if asked, ``logits`` [n_steps, V] and ``final_norm_output``."""
        tok = int(first_token)
        ids, logits, hidden = [], [], []
        for s in range(n_steps):
            r = self.forward(cache, [tok], [start_pos + s])
            tok = int(r["ids"][0])
            ids.append(tok)
            if keep_logits:
                logits.append(r["logits"][0])
                hidden.append(r["final_norm_output"][0])
        out = {"ids": np.asarray(ids, dtype=np.int32)}
        if keep_logits:
            out["logits"] = np.stack(logits)
            out["final_norm_output"] = np.stack(hidden)
        return out

    def greedy_generate(self, cache: KVCache, first_token: int, start_pos: int,
                        max_steps: int, stop_ids) -> dict:
        """Greedy generation that ends at a stop token: generation stops at
        the end-of-sequence id or the chat end-of-turn id (minfer page,
        section 5 "Tokenizer and chat", stop tokens eos and im_end; nnterp
        encyclopedia qwen2, "The chat template writes a system turn":
        <|endoftext|> 151643 and <|im_end|> 151645).  Steps as in
        greedy_decode; the first generated id that is in ``stop_ids`` is the
        last one kept.  Returns ``ids`` [max_steps] with -1 after that id
        and ``n_generated`` (the ids kept, the stop id included)."""
        stops = {int(t) for t in stop_ids}
        tok = int(first_token)
        ids = np.full(max_steps, -1, dtype=np.int32)
        n = 0
        for s in range(max_steps):
            r = self.forward(cache, [tok], [start_pos + s])
            tok = int(r["ids"][0])
            ids[s] = tok
            n = s + 1
            if tok in stops:
                break
        return {"ids": ids, "n_generated": n}
