"""Pins of the CPU oracle to facts that do not come from the oracle itself:
values printed on the pages, closed forms, invariants, special cases that
reduce to library routines, and brute force on tiny shapes.  CPU only."""
import dataclasses
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from conftest import read_golden

TINY = synth.ModelShape("tiny", n_layer=2, hidden=16, n_head=4, n_kv_head=2,
                        head_dim=4, intermediate=24, vocab=37, rope_theta=1e4)


def tiny_oracle(shape=TINY, n_ctx=32, seed=3, **kw):
    w = synth.make_weights(shape, seed)
    return oracle.build_oracle(shape, w, n_ctx, **kw), w


# ---------------------------------------------------------------------------
# Values the pages print.
# ---------------------------------------------------------------------------

def test_config_and_shapes_match_pages():
    g = read_golden("qwen2_0p5b_pages.txt")
    s = synth.SHAPES["qwen2.5-0.5b"]
    assert s.hidden == int(g["hidden_size"])
    assert s.intermediate == int(g["intermediate_size"])
    assert s.n_layer == int(g["num_hidden_layers"])
    assert s.n_head == int(g["num_attention_heads"])
    assert s.n_kv_head == int(g["num_key_value_heads"])
    assert s.vocab == int(g["vocab_size"])
    assert s.rope_theta == float(g["rope_theta"])
    assert s.rms_eps == float(g["rms_norm_eps"])
    # head_dim = H / n_heads; kv width = n_kv * hd; group = nh / nkv.
    assert s.hidden // s.n_head == int(g["head_dim"]) == s.head_dim
    assert s.n_kv_head * s.head_dim == int(g["kv_proj_out"])
    assert s.n_head // s.n_kv_head == int(g["kv_group"])


def test_weight_shapes_and_bytes_match_pages():
    """Shapes of the generated 0.5B weights and the f16 byte totals."""
    g = read_golden("qwen2_0p5b_pages.txt")
    w = synth.make_weights(synth.SHAPES["qwen2.5-0.5b"], 0)

    def shp(key):
        return tuple(int(t) for t in g[key].split())

    lw = w["layers"][0]
    assert lw["wq"].shape == shp("shape.q_proj")
    assert lw["wk"].shape == shp("shape.k_proj")
    assert lw["wv"].shape == shp("shape.v_proj")
    assert lw["wo"].shape == shp("shape.o_proj")
    assert lw["wg"].shape == shp("shape.gate_proj")
    assert lw["wu"].shape == shp("shape.up_proj")
    assert lw["wd"].shape == shp("shape.down_proj")
    assert w["embed"].shape == shp("shape.embed_tokens")
    assert len(w["layers"]) == int(g["num_hidden_layers"])
    assert w["embed"].dtype == np.float16
    assert w["embed"].nbytes == int(g["embed_f16_bytes"])
    f16 = w["embed"].nbytes + sum(lw[k].nbytes for lw in w["layers"]
                                  for k in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"))
    assert f16 == 987_922_432
    assert round(f16 / 2**20) == int(g["resident_f16_weights_mib"])
    s = synth.SHAPES["qwen2.5-0.5b"]
    kv_per_pos = s.n_layer * 2 * s.n_kv_head * s.head_dim * 4      # f32 K and V
    assert kv_per_pos == int(g["kv_bytes_per_position_kb"]) * 1024
    assert kv_per_pos * 4096 == int(g["kv_n_ctx_4096_mb"]) * 2**20


# ---------------------------------------------------------------------------
# RMSNorm, SiLU, softmax.
# ---------------------------------------------------------------------------

def test_rms_norm_matches_torch_library():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 16))
    w = 1 + 0.1 * rng.standard_normal(16)
    ref = F.rms_norm(torch.from_numpy(x), (16,), weight=torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, w, 1e-6), ref, rtol=1e-14, atol=1e-15)


def test_rms_norm_closed_form():
    # x = (3, 4): mean(x^2) = 12.5; eps 0 -> x / sqrt(12.5).
    out = oracle.rms_norm(np.array([3.0, 4.0]), np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(out, [3 / math.sqrt(12.5), 8 / math.sqrt(12.5)], rtol=1e-15)


def test_silu_matches_torch_library_and_values():
    z = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(oracle.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0


def test_softmax_rows_sum_to_one_and_mask():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((7, 11)) * 30
    s[:, 5:] = -np.inf
    p = oracle.softmax_rows(s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(p[:, 5:] == 0)


# ---------------------------------------------------------------------------
# RoPE (NeoX rotate_half, NonInterleaved).
# ---------------------------------------------------------------------------

def test_rope_identity_at_position_zero():
    x = np.random.default_rng(3).standard_normal((1, 3, 64))
    np.testing.assert_array_equal(oracle.rope_neox(x, np.array([0]), 1e6), x)


def test_rope_inverse_frequencies():
    f = oracle.rope_inv_freq(64, 1e6)
    assert f[0] == 1.0
    # i = hd/4 -> theta^(-1/2) = 1e-3 for theta 1e6.
    np.testing.assert_allclose(f[16], 1e-3, rtol=1e-14)
    np.testing.assert_allclose(f[31], 1e6 ** (-62 / 64), rtol=1e-14)


def test_rope_pairs_i_with_i_plus_half_and_sign():
    """A unit vector on index 0 turns in the (0, hd/2) plane only, towards +sin
    at hd/2 (rotate_half: the second half gains +a sin); index hd/2 goes to
    (-sin, cos).  An interleaved pairing (0, 1) fails this."""
    hd, p = 64, 5
    e0 = np.zeros((1, 1, hd)); e0[0, 0, 0] = 1
    eh = np.zeros((1, 1, hd)); eh[0, 0, hd // 2] = 1
    r0 = oracle.rope_neox(e0, np.array([p]), 1e6)[0, 0]
    rh = oracle.rope_neox(eh, np.array([p]), 1e6)[0, 0]
    expect0 = np.zeros(hd); expect0[0] = math.cos(p); expect0[hd // 2] = math.sin(p)
    expecth = np.zeros(hd); expecth[0] = -math.sin(p); expecth[hd // 2] = math.cos(p)
    np.testing.assert_allclose(r0, expect0, atol=1e-15)
    np.testing.assert_allclose(rh, expecth, atol=1e-15)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 2, 64))
    pos = np.array([0, 1, 7, 100, 4095, 32767])
    r = oracle.rope_neox(x, pos, 1e6)
    n_in = x[..., :32] ** 2 + x[..., 32:] ** 2
    n_out = r[..., :32] ** 2 + r[..., 32:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))

    def score(pq, pk):
        return float(np.sum(oracle.rope_neox(q, np.array([pq]), 1e6) *
                            oracle.rope_neox(k, np.array([pk]), 1e6)))

    base = score(10, 3)
    for d in (1, 17, 1000, 4000):
        assert abs(score(10 + d, 3 + d) - base) < 1e-10 * max(1, abs(base))
    assert abs(score(11, 3) - base) > 1e-6


# ---------------------------------------------------------------------------
# Attention.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("hd", [8, 128])
def test_gqa_attention_matches_sdpa_with_repeated_kv_heads(hd):
    rng = np.random.default_rng(6)
    T, nh, nkv = 9, 6, 2
    q = rng.standard_normal((T, nh, hd))
    K = rng.standard_normal((T, nkv, hd))
    V = rng.standard_normal((T, nkv, hd))
    out = oracle.gqa_attention(q, K, V, np.arange(T))
    qt = torch.from_numpy(q).transpose(0, 1)                     # [nh, T, hd]
    kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(nh // nkv, dim=0)
    vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(nh // nkv, dim=0)
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True).transpose(0, 1).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_gqa_with_kv_heads_equal_to_heads_is_mha_of_tiled_weights():
    """GQA (4 q heads over 2 kv heads) equals MHA whose k/v projections are
    the GQA ones tiled over contiguous groups (kv head j -> q heads 2j, 2j+1)."""
    shape = TINY
    w = synth.make_weights(shape, 7)
    mha_shape = dataclasses.replace(shape, name="tiny-mha", n_kv_head=shape.n_head)
    group, hd = shape.n_head // shape.n_kv_head, shape.head_dim
    w_mha = {"embed": w["embed"], "final_norm": w["final_norm"], "layers": []}
    for lw in w["layers"]:
        d = dict(lw)
        for key in ("wk", "wv", "bk", "bv"):
            a = lw[key].reshape(shape.n_kv_head, hd, *lw[key].shape[1:])
            d[key] = np.repeat(a, group, axis=0).reshape(shape.n_head * hd, *lw[key].shape[1:])
        w_mha["layers"].append(d)
    o_gqa = oracle.build_oracle(shape, w, 16)
    o_mha = oracle.build_oracle(mha_shape, w_mha, 16)
    toks = synth.make_tokens(shape.vocab, 10, 8)
    a = o_gqa.forward(o_gqa.new_cache(), toks, np.arange(10))
    b = o_mha.forward(o_mha.new_cache(), toks, np.arange(10))
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=0, atol=1e-13)
    # A wrong mapping (h % nkv) would break this: check the tiling matters.
    w_bad = {"embed": w["embed"], "final_norm": w["final_norm"], "layers": []}
    for lw in w["layers"]:
        d = dict(lw)
        for key in ("wk", "wv", "bk", "bv"):
            a_ = lw[key].reshape(shape.n_kv_head, hd, *lw[key].shape[1:])
            d[key] = np.tile(a_, (group,) + (1,) * (a_.ndim - 1)).reshape(shape.n_head * hd, *lw[key].shape[1:])
        w_bad["layers"].append(d)
    o_bad = oracle.build_oracle(mha_shape, w_bad, 16)
    c = o_bad.forward(o_bad.new_cache(), toks, np.arange(10))
    assert np.max(np.abs(c["logits"] - a["logits"])) > 1e-6


def test_zero_attention_input_falls_back_to_biases():
    """With the normed input zeroed, q, k, v are their biases: the keys are
    rope(b_k) and the attention output is o_proj(b_v) at every position
    (nnterp encyclopedia qwen2, "Queries, keys and values carry a bias")."""
    shape = TINY
    w = synth.make_weights(shape, 9)
    wz = {"embed": w["embed"], "final_norm": w["final_norm"], "layers": [dict(l) for l in w["layers"]]}
    wz["layers"][1]["attn_norm"] = np.zeros_like(w["layers"][1]["attn_norm"])
    o = oracle.build_oracle(shape, wz, 16)
    probes = {}
    T = 6
    o.forward(o.new_cache(), synth.make_tokens(shape.vocab, T, 10), np.arange(T), probes=probes)
    lw = wz["layers"][1]
    hd, nkv, nh = shape.head_dim, shape.n_kv_head, shape.n_head
    bk = np.broadcast_to(lw["bk"].astype(np.float64).reshape(1, nkv, hd), (T, nkv, hd))
    np.testing.assert_allclose(probes["attention_keys"][1],
                               oracle.rope_neox(bk, np.arange(T), shape.rope_theta), rtol=1e-14, atol=1e-16)
    assert np.max(np.abs(probes["attention_keys"][1])) > 0
    bv = lw["bv"].astype(np.float64).reshape(nkv, hd)
    premix = np.concatenate([bv[h // (nh // nkv)] for h in range(nh)])
    expect = lw["wo"].astype(np.float64) @ premix
    np.testing.assert_allclose(probes["attention_output"][1], np.broadcast_to(expect, (T, shape.hidden)),
                               rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# The whole forward.
# ---------------------------------------------------------------------------

def _rope_hf(x, pos, theta):
    """The HF formulation: cos/sin over duplicated frequencies and
    rotate_half(x) = cat(-x2, x1); a different arrangement of the rotation."""
    hd = x.shape[-1]
    inv = 1.0 / (theta ** (torch.arange(0, hd, 2, dtype=torch.float64) / hd))
    freqs = pos.to(torch.float64)[:, None] * inv[None, :]
    emb = torch.cat([freqs, freqs], dim=-1)
    cos, sin = emb.cos()[None], emb.sin()[None]
    x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
    return x * cos + torch.cat([-x2, x1], dim=-1) * sin


def _torch_library_forward(shape, w, tokens):
    """Tiny-shape forward built from torch float64 library routines
    (embedding, rms_norm, linear, scaled_dot_product_attention with repeated
    kv heads, silu) -- the independent restatement the oracle is pinned to."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    T = len(tokens)
    pos = torch.arange(T)
    H, nh, nkv, hd = shape.hidden, shape.n_head, shape.n_kv_head, shape.head_dim
    x = F.embedding(torch.from_numpy(np.asarray(tokens, dtype=np.int64)), t(w["embed"]))
    for lw in w["layers"]:
        n = F.rms_norm(x, (H,), weight=t(lw["attn_norm"]), eps=shape.rms_eps)
        q = F.linear(n, t(lw["wq"]), t(lw["bq"])).view(T, nh, hd).transpose(0, 1)
        k = F.linear(n, t(lw["wk"]), t(lw["bk"])).view(T, nkv, hd).transpose(0, 1)
        v = F.linear(n, t(lw["wv"]), t(lw["bv"])).view(T, nkv, hd).transpose(0, 1)
        q, k = _rope_hf(q, pos, shape.rope_theta), _rope_hf(k, pos, shape.rope_theta)
        k = k.repeat_interleave(nh // nkv, dim=0)
        v = v.repeat_interleave(nh // nkv, dim=0)
        a = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        x = x + F.linear(a.transpose(0, 1).reshape(T, H), t(lw["wo"]))
        m = F.rms_norm(x, (H,), weight=t(lw["ffn_norm"]), eps=shape.rms_eps)
        x = x + F.linear(F.silu(F.linear(m, t(lw["wg"]))) * F.linear(m, t(lw["wu"])), t(lw["wd"]))
    f = F.rms_norm(x, (H,), weight=t(w["final_norm"]), eps=shape.rms_eps)
    return F.linear(f, t(w["lm_head"] if "lm_head" in w else w["embed"])).numpy()


@pytest.mark.parametrize("shape", [TINY, dataclasses.replace(TINY, name="tiny-mha", n_kv_head=4),
                                   dataclasses.replace(TINY, name="tiny-g4", n_head=4, n_kv_head=1),
                                   dataclasses.replace(TINY, name="tiny-hd128", hidden=256, n_head=2,
                                                       n_kv_head=1, head_dim=128),
                                   dataclasses.replace(TINY, name="tiny-untied", tie_embeddings=False)])
def test_forward_matches_torch_library_brute_force(shape):
    o, w = tiny_oracle(shape)
    toks = synth.make_tokens(shape.vocab, 12, 11)
    r = o.forward(o.new_cache(), toks, np.arange(12))
    ref = _torch_library_forward(shape, w, toks)
    np.testing.assert_allclose(r["logits"], ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(r["ids"], np.argmax(ref.astype(np.float32), axis=1))


def test_residual_identity_and_readout():
    """layer_input + attention_output + mlp_output == layer_output (nnterp
    "01 . the residual stream"); logits == E . final_norm_output with no
    softcap or scale ("The readout is the plain projection")."""
    o, w = tiny_oracle()
    probes = {}
    r = o.forward(o.new_cache(), synth.make_tokens(TINY.vocab, 7, 12), np.arange(7), probes=probes)
    for i in range(TINY.n_layer):
        lhs = probes["layer_input"][i] + probes["attention_output"][i] + probes["mlp_output"][i]
        np.testing.assert_allclose(lhs, probes["layer_output"][i], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(r["logits"], probes["final_norm_output"] @ w["embed"].astype(np.float64).T,
                               rtol=1e-14, atol=1e-15)


def test_untied_lm_head_is_a_separate_readout():
    """From 7B up the embedding and the unembedding are separate matrices
    (nnterp "The readout is the plain projection"): the layers read the
    embedding only, the logits come from the LM head, and an LM head equal
    to the embedding is the tied model bit for bit."""
    untied = dataclasses.replace(TINY, name="tiny-untied", tie_embeddings=False)
    o_u, w_u = tiny_oracle(untied)
    assert w_u["lm_head"].shape == w_u["embed"].shape
    assert not np.array_equal(w_u["lm_head"], w_u["embed"])
    tied_w = {k: v for k, v in w_u.items() if k != "lm_head"}
    o_t = oracle.build_oracle(TINY, tied_w, 32)
    same_w = dict(tied_w, lm_head=np.array(w_u["embed"]))
    o_s = oracle.build_oracle(untied, same_w, 32)
    toks = synth.make_tokens(TINY.vocab, 9, 14)
    r_u = o_u.forward(o_u.new_cache(), toks, np.arange(9))
    r_t = o_t.forward(o_t.new_cache(), toks, np.arange(9))
    r_s = o_s.forward(o_s.new_cache(), toks, np.arange(9))
    np.testing.assert_array_equal(r_s["logits"], r_t["logits"])
    np.testing.assert_array_equal(r_u["final_norm_output"], r_t["final_norm_output"])
    np.testing.assert_allclose(r_u["logits"], r_u["final_norm_output"] @ w_u["lm_head"].astype(np.float64).T,
                               rtol=1e-14, atol=1e-15)
    assert not np.allclose(r_u["logits"], r_t["logits"])
    # The tied arrays are the same draws whether or not a head is drawn.
    for k in ("embed", "final_norm"):
        np.testing.assert_array_equal(w_u[k], synth.make_weights(TINY, 3)[k])


def test_kv_cache_decode_equals_full_recompute():
    """Positions are data: prefill then one-row decode steps give the same
    rows as one full-sequence forward (minfer page section 6)."""
    o, _ = tiny_oracle()
    toks = synth.make_tokens(TINY.vocab, 14, 13)
    full = o.forward(o.new_cache(), toks, np.arange(14))
    c = o.new_cache()
    o.forward(c, toks[:8], np.arange(8))
    for p in range(8, 14):
        r = o.forward(c, toks[p:p + 1], [p])
        np.testing.assert_allclose(r["logits"][0], full["logits"][p], rtol=1e-12, atol=1e-13)


def test_fused_and_unfused_are_identical():
    """One product with the stacked Q/K/V (gate/up) matrix equals separate
    products (minfer page section 3, "Decode fusions": bit-identical)."""
    toks = synth.make_tokens(TINY.vocab, 9, 14)
    outs = []
    for fq, ff in ((True, True), (False, False), (True, False), (False, True)):
        o, _ = tiny_oracle(fuse_qkv=fq, fuse_ffn=ff)
        outs.append(o.forward(o.new_cache(), toks, np.arange(9))["logits"])
    for x in outs[1:]:
        np.testing.assert_allclose(x, outs[0], rtol=0, atol=1e-14)


def test_tail_cut_keeps_last_rows():
    """Cutting to the last n_out rows before the final layer's FFN leaves
    their logits unchanged (minfer page section 3, "G3 tail-row")."""
    o, _ = tiny_oracle()
    toks = synth.make_tokens(TINY.vocab, 11, 15)
    full = o.forward(o.new_cache(), toks, np.arange(11))
    cut = o.forward(o.new_cache(), toks, np.arange(11), n_out=2, tail_cut=True)
    nocut = o.forward(o.new_cache(), toks, np.arange(11), n_out=2, tail_cut=False)
    np.testing.assert_allclose(cut["logits"], full["logits"][-2:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(nocut["logits"], full["logits"][-2:], rtol=0, atol=1e-14)


def test_position_beyond_n_ctx_is_an_error_and_writes_nothing():
    o, _ = tiny_oracle(n_ctx=8)
    c = o.new_cache()
    with pytest.raises(oracle.PositionError):
        o.forward(c, [1, 2], [7, 8])
    assert not np.any(c.K) and not np.any(c.V)
    o.forward(c, [1], [7])
    assert np.any(c.K[:, 7])


# ---------------------------------------------------------------------------
# Q8_0.
# ---------------------------------------------------------------------------

def test_q8_0_special_blocks():
    w = np.zeros((4, 64), dtype=np.float16)
    w[1, :32] = 0.5                       # constant block -> all q = 127, d = 0.5/127
    w[2, 3] = -2.0                        # one-hot negative -> q = -127 at 3, 0 elsewhere
    w[3, :32] = np.arange(32) - 16        # ramp -> extremes map to -127
    q, d = oracle.quantize_q8_0(w)
    assert q.dtype == np.int8 and d.dtype == np.float16 and d.shape == (4, 2)
    assert np.all(q[0] == 0) and np.all(d[0] == 0)
    assert np.all(q[1, :32] == 127) and d[1, 0] == np.float16(np.float32(0.5) / np.float32(127))
    assert q[2, 3] == -127 and np.count_nonzero(q[2]) == 1
    assert q[3, 0] == -127 and q[3, 16] == 0
    assert np.all(np.diff(q[3, :32].astype(int)) >= 0)


def test_q8_0_rounds_half_away_from_zero():
    """Reading of the unnamed Q8_0 rounding (minfer page "Qwen2 / Qwen2.5
    Architecture Support", sections 3 and 6): round half away from zero.
    A block whose largest magnitude is 127 has d = 1 exactly, so x / d is x
    and every half case is decided by the rounding rule alone: half-even
    would give 0, 2, 2 where half-away gives 1, 2, 3."""
    w = np.zeros((1, 32), dtype=np.float16)
    w[0, :7] = [127.0, 0.5, -0.5, 1.5, -1.5, 2.5, -2.5]
    q, d = oracle.quantize_q8_0(w)
    assert d[0, 0] == 1.0
    np.testing.assert_array_equal(q[0, :7], [127, 1, -1, 2, -2, 3, -3])
    # The largest float32 below one half rounds to 0.  No float16 weight
    # reaches this quotient; float32 activation rows (the Q8_0 activation
    # product) can, and floor(|v| + 0.5) in float32 would give 1 here.
    below = np.nextafter(np.float32(0.5), np.float32(0))
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :3] = [127.0, below, -below]
    q, d = oracle.quantize_q8_0(x)
    assert d[0, 0] == 1.0
    np.testing.assert_array_equal(q[0, :3], [127, 0, 0])
    # Just above one half, and a large quotient just below a half step.
    x[0, 1:3] = [np.nextafter(np.float32(0.5), np.float32(1)), np.float32(126.49999)]
    q, _ = oracle.quantize_q8_0(x)
    np.testing.assert_array_equal(q[0, 1:3], [1, 126])


def test_greedy_ids_take_the_lowest_index_of_a_tie():
    """Greedy argmax keeps the lowest index among equal maxima, decided on
    the float32 logits both sides hold (xinfer "Module 7", section 7.3, the
    on-device argmax; the reading of ties is the lowest index)."""
    row = np.array([0.25, 3.0, -1.0, 3.0, 3.0], dtype=np.float64)
    assert oracle.greedy_ids(row[None])[0] == 1
    assert oracle.greedy_ids(row[None, ::-1].copy())[0] == 0
    # Two logits that differ in float64 but round to the same float32: a
    # tie in float32, so the lower index wins although the later one is
    # larger in float64.
    a = 1.0
    b = 1.0 + 2.0 ** -30
    assert np.float32(a) == np.float32(b) and b > a
    assert oracle.greedy_ids(np.array([[0.0, a, b]]))[0] == 1
    # A row of equal values, and a batch of rows with ties at different places.
    assert oracle.greedy_ids(np.zeros((1, 7)))[0] == 0
    rows = np.zeros((3, 6))
    rows[0, [2, 5]] = 1.0
    rows[1, [4, 1]] = 2.0
    rows[2, [5]] = 0.5
    np.testing.assert_array_equal(oracle.greedy_ids(rows), [2, 1, 5])


def test_q8_0_round_trip_bound_and_exact_dequant():
    rng = np.random.default_rng(16)
    w = (0.02 * rng.standard_normal((64, 256))).astype(np.float16)
    q, d = oracle.quantize_q8_0(w)
    deq = oracle.dequantize_q8_0(q, d)
    x = w.astype(np.float64).reshape(64, 8, 32)
    dd = np.max(np.abs(x), axis=2) / 127          # unrounded scale
    dh = d.astype(np.float64)
    bound = dd / 2 + 127 * np.abs(dd - dh) + 1e-12
    err = np.abs(x - deq.reshape(64, 8, 32))
    assert np.all(err <= bound[:, :, None])
    # Dequant is exact in float32: scale (11-bit significand) times |q| <= 127.
    f32 = (d.astype(np.float32)[:, :, None] * q.reshape(64, 8, 32).astype(np.float32)).reshape(64, 256)
    np.testing.assert_array_equal(f32.astype(np.float64), deq)
    # Sign symmetry.
    q2, d2 = oracle.quantize_q8_0(-w)
    np.testing.assert_array_equal(q2, -q)
    np.testing.assert_array_equal(d2, d)


def test_q8_0_oracle_forward_is_close_to_f16():
    shape = dataclasses.replace(TINY, hidden=64, head_dim=16, intermediate=96)
    w = synth.make_weights(shape, 17)
    a = oracle.build_oracle(shape, w, 16)
    b = oracle.build_oracle(shape, w, 16, weight_format="q8_0")
    toks = synth.make_tokens(shape.vocab, 5, 18)
    la = a.forward(a.new_cache(), toks, np.arange(5))["logits"]
    lb = b.forward(b.new_cache(), toks, np.arange(5))["logits"]
    assert 0 < np.max(np.abs(la - lb)) < 0.05 * np.max(np.abs(la))


def test_generation_stops_at_the_first_stop_id():
    """Stop tokens end generation (minfer page section 5, eos and im_end):
    the stop-aware generation is the plain greedy decode cut right after the
    first generated id that is a stop id, the stop id kept, -1 after it."""
    o, _ = tiny_oracle(n_ctx=32)
    prompt = synth.make_tokens(TINY.vocab, 5, 21)
    pre = o.forward(o.new_cache(), prompt, np.arange(5))
    first = int(pre["ids"][-1])

    def primed():
        c = o.new_cache()
        o.forward(c, prompt, np.arange(5))
        return c

    n = 20
    ref = o.greedy_decode(primed(), first, 5, n, keep_logits=False)["ids"]
    # A stop id first generated at step k: ids up to and including k.
    for k in (0, 3, n - 1):
        stop = int(ref[k])
        k_first = int(np.flatnonzero(ref == stop)[0])
        r = o.greedy_generate(primed(), first, 5, n, [stop])
        assert r["n_generated"] == k_first + 1
        np.testing.assert_array_equal(r["ids"][:k_first + 1], ref[:k_first + 1])
        assert np.all(r["ids"][k_first + 1:] == -1)
    # Stop ids that are never generated (or none): the plain greedy decode.
    never = [t for t in range(TINY.vocab) if t not in set(ref.tolist())][:2]
    for stops in ([], never):
        r = o.greedy_generate(primed(), first, 5, n, stops)
        assert r["n_generated"] == n
        np.testing.assert_array_equal(r["ids"], ref)
    # The earliest of several stop ids wins.
    r = o.greedy_generate(primed(), first, 5, n, [int(ref[9]), int(ref[2])])
    k_first = min(int(np.flatnonzero(ref == ref[9])[0]), int(np.flatnonzero(ref == ref[2])[0]))
    assert r["n_generated"] == k_first + 1


# ---------------------------------------------------------------------------
# Q4_0 (the reading in oracle/q4_0.py: blocks of 32 along K, d = amax / 7,
# codes c + 8 in nibbles, element 2j low / 2j + 1 high).
# ---------------------------------------------------------------------------

def test_q4_0_special_blocks_rounding_and_nibble_order():
    w = np.zeros((4, 64), dtype=np.float16)
    w[1, :32] = 0.5                       # constant block -> c = 7 everywhere
    w[2, 3] = -2.0                        # one-hot negative -> c = -7 at 3
    w[3, :4] = [7.0, 2.5, -2.5, 0.5]      # d = 1 exactly: halves round away from zero
    packed, d = oracle.quantize_q4_0(w)
    assert packed.dtype == np.uint8 and packed.shape == (4, 32)
    assert d.dtype == np.float16 and d.shape == (4, 2)
    codes = oracle.unpack_nibbles(packed)
    assert np.all(codes[0] == 8) and np.all(d[0] == 0)
    assert np.all(codes[1, :32] == 15) and np.all(codes[1, 32:] == 8)
    assert d[1, 0] == np.float16(np.float32(0.5) / np.float32(7))
    assert codes[2, 3] == 1 and np.count_nonzero(codes[2] - 8) == 1
    assert d[3, 0] == 1.0
    np.testing.assert_array_equal(codes[3, :4], [15, 11, 5, 9])   # 7, 3, -3, 1 (+8)
    assert packed[3, 0] == 0xBF and packed[3, 1] == 0x95          # low nibble = even element
    assert np.all(codes >= 1) and np.all(codes <= 15)
    # Float32 rows: the largest float32 below one half rounds to 0 (code 8).
    below = np.nextafter(np.float32(0.5), np.float32(0))
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :3] = [7.0, below, -below]
    packed, d = oracle.quantize_q4_0(x)
    assert d[0, 0] == 1.0
    np.testing.assert_array_equal(oracle.unpack_nibbles(packed)[0, :3], [15, 8, 8])


def test_q4_0_round_trip_bound_exact_dequant_and_size():
    rng = np.random.default_rng(31)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float16)
    packed, d = oracle.quantize_q4_0(w)
    assert packed.nbytes + d.nbytes == (w.size // 32) * 18           # 4.5 bits an element
    deq = oracle.dequantize_q4_0(packed, d)
    x = w.astype(np.float64).reshape(8, 8, 32)
    dd = (np.max(np.abs(w.astype(np.float32).reshape(8, 8, 32)), axis=2) / np.float32(7)).astype(np.float64)
    dh = d.astype(np.float64)
    bound = dd / 2 + 7 * np.abs(dd - dh) + 1e-12
    assert np.all(np.abs(x - deq.reshape(8, 8, 32)) <= bound[:, :, None])
    c = oracle.unpack_nibbles(packed).astype(np.float32) - 8
    f32 = (d.astype(np.float32).repeat(32, axis=1) * c)              # the float32 product
    np.testing.assert_array_equal(f32.astype(np.float64), deq)
    codes = rng.integers(0, 16, size=(3, 64)).astype(np.uint8)
    np.testing.assert_array_equal(oracle.unpack_nibbles(oracle.pack_nibbles(codes)), codes)


def test_q4_0_oracle_forward_tracks_f16():
    shape = dataclasses.replace(TINY, hidden=64, head_dim=16, intermediate=96)
    w = synth.make_weights(shape, 17)
    a = oracle.build_oracle(shape, w, 16)
    b4 = oracle.build_oracle(shape, w, 16, weight_format="q4_0")
    b8 = oracle.build_oracle(shape, w, 16, weight_format="q8_0")
    toks = synth.make_tokens(shape.vocab, 8, 18)
    la = a.forward(a.new_cache(), toks, np.arange(8))["logits"]
    l4 = b4.forward(b4.new_cache(), toks, np.arange(8))["logits"]
    l8 = b8.forward(b8.new_cache(), toks, np.arange(8))["logits"]
    e4, e8 = np.max(np.abs(l4 - la)), np.max(np.abs(l8 - la))
    assert 0 < e8 < e4                       # 4-bit codes are coarser than 8-bit ones
    assert np.corrcoef(l4.ravel(), la.ravel())[0, 1] > 0.95


# ---------------------------------------------------------------------------
# Products with Q8_0 activations (the reading in oracle.q8_0.q8_0_matmul).
# ---------------------------------------------------------------------------

def test_q8_0_matmul_is_the_product_of_the_dequantised_operands():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((5, 96)).astype(np.float32) * 3
    w = (rng.standard_normal((7, 96)) * 0.02).astype(np.float16)
    wq, wd = oracle.quantize_q8_0(w)
    xq, xd = oracle.quantize_q8_0(x)
    ref = torch.from_numpy(oracle.dequantize_q8_0(xq, xd)) @ torch.from_numpy(oracle.dequantize_q8_0(wq, wd)).T
    out = oracle.q8_0_matmul(x, wq, wd)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_q8_0_matmul_is_lossless_on_q8_0_activations_and_bounded_otherwise():
    rng = np.random.default_rng(42)
    w = (rng.standard_normal((6, 64)) * 0.02).astype(np.float16)
    wq, wd = oracle.quantize_q8_0(w)
    wdeq = oracle.dequantize_q8_0(wq, wd)
    # Rows already on the Q8_0 grid (|code| reaching 127 in every block):
    # quantising them again gives back the same values.
    codes = rng.integers(-127, 128, size=(3, 2, 32))
    codes[:, :, 0] = 127
    scale = rng.uniform(0.01, 1.0, size=(3, 2)).astype(np.float16).astype(np.float32)
    x = (scale[:, :, None] * codes).reshape(3, 64).astype(np.float32)
    np.testing.assert_allclose(oracle.q8_0_matmul(x, wq, wd), x.astype(np.float64) @ wdeq.T, rtol=1e-13, atol=1e-15)
    # Any rows: the error is within the activations' quantisation bound.
    x = rng.standard_normal((4, 64)).astype(np.float32)
    xb = x.reshape(4, 2, 32)
    d = (np.max(np.abs(xb), axis=2) / np.float32(127)).astype(np.float64)
    dh = d.astype(np.float32).astype(np.float16).astype(np.float64)
    elem = (d / 2 + 127 * np.abs(d - dh))[:, :, None] * np.ones((1, 1, 32))
    bound = elem.reshape(4, 64) @ np.abs(wdeq).T + 1e-12
    err = np.abs(oracle.q8_0_matmul(x, wq, wd) - x.astype(np.float64) @ wdeq.T)
    assert np.all(err <= bound) and np.max(err) > 0


def test_q8_0_activation_forward_tracks_the_q8_0_weight_forward():
    shape = dataclasses.replace(TINY, hidden=64, head_dim=16, intermediate=96)
    w = synth.make_weights(shape, 17)
    cfg = oracle.OracleConfig.from_shape(shape, 16)
    wq8 = oracle.OracleWeights(w, "q8_0")
    a = oracle.Qwen2Oracle(cfg, wq8)
    b = oracle.Qwen2Oracle(cfg, wq8, act_q8=True)
    toks = synth.make_tokens(shape.vocab, 8, 18)
    la = a.forward(a.new_cache(), toks, np.arange(8))["logits"]
    lb = b.forward(b.new_cache(), toks, np.arange(8))["logits"]
    assert 0 < np.max(np.abs(la - lb)) < 0.05 * np.max(np.abs(la))
    assert np.corrcoef(la.ravel(), lb.ravel())[0, 1] > 0.99
    with pytest.raises(ValueError):
        oracle.Qwen2Oracle(cfg, oracle.OracleWeights(w, "f16"), act_q8=True)
