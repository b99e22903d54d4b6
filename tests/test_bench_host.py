"""Host logic of bench.py on the CPU: the algorithmic bytes and FLOPs behind
every roofline fraction, each checked against a count made another way, and
the clock-sample parser that decides whether a run was throttled."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

S05 = synth.SHAPES["qwen2.5-0.5b"]
MATS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
SMALL = ("bq", "bk", "bv", "attn_norm", "ffn_norm")


def test_decode_bytes_f16_match_the_weight_arrays():
    """Weights once (the arrays' own sizes), f32 biases and norms, one f16
    embedding row per sequence, and per sequence the KV read of positions
    0..p plus the write of p (f32 K and V of every layer and kv head)."""
    w = synth.make_weights(S05, 0)
    mats = w["embed"].nbytes + sum(L[k].nbytes for L in w["layers"] for k in MATS)
    small = w["final_norm"].nbytes + sum(L[k].nbytes for L in w["layers"] for k in SMALL)
    assert mats == 987_922_432 and small == 286_208
    kv_pos = S05.n_layer * 2 * S05.n_kv_head * S05.head_dim * 4
    for pos in ([128], [383], [4000, 256, 1000]):
        want = mats + small + sum(S05.hidden * 2 + kv_pos * (p + 1) + kv_pos for p in pos)
        assert bench.decode_bytes_per_step(S05, pos) == want


def test_decode_bytes_q8_0_match_the_quantised_sizes():
    """Q8_0: each matrix stored as int8 values plus one f16 scale per 32
    (the oracle's quantiser output sizes, on a small shape so it runs fast),
    embedding rows read in the same format."""
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    mats = 0
    for a in [w["embed"]] + [L[k] for L in w["layers"] for k in MATS]:
        q, d = oracle.quantize_q8_0(a)
        mats += q.nbytes + d.nbytes
    small = w["final_norm"].nbytes + sum(L[k].nbytes for L in w["layers"] for k in SMALL)
    row = shape.hidden + shape.hidden // 32 * 2
    kv_pos = shape.n_layer * 2 * shape.n_kv_head * shape.head_dim * 4
    pos = [5, 40]
    want = mats + small + sum(row + kv_pos * (p + 2) for p in pos)
    assert bench.decode_bytes_per_step(shape, pos, q8=True) == want
    # The 0.5B Q8_0 weight total: 1 + 2/32 bytes per element.
    n_elem = 987_922_432 // 2
    assert n_elem * (1 + 2 / 32) == 524_833_792


def test_prefill_flops_match_a_row_by_row_count():
    """2 flops per multiply-add, counted row by row: every row through the
    first L-1 layers and the last layer's Q/K/V; causal attention (q.k and
    p.v over keys 0..i, all heads) of every row in the first L-1 layers and
    of the kept rows in the last; o_proj, the FFN and the LM head of the
    kept rows only (the tail cut)."""
    s = S05
    H, I, V, L = s.hidden, s.intermediate, s.vocab, s.n_layer
    nq, nkv = s.n_head * s.head_dim, s.n_kv_head * s.head_dim
    for lens, keep in (([512] * 8, 1), ([300, 17, 64], 1), ([40, 9], 3)):
        total = 0
        for n in lens:
            for layer in range(L):
                last = layer == L - 1
                for i in range(n):
                    kept = i >= n - keep
                    total += 2 * (nq + 2 * nkv) * H                     # Q/K/V
                    if last and not kept:
                        continue
                    total += 2 * 2 * (i + 1) * s.head_dim * s.n_head    # q.k and p.v
                    total += 2 * H * nq + 2 * 2 * I * H + 2 * H * I     # o_proj, gate/up, down
            total += keep * 2 * V * H                                   # LM head
        assert bench.prefill_flops(s, lens, keep) == total
    # 8 x 512 with one kept row per sequence: the figure the bench divides by.
    assert abs(bench.prefill_flops(s, [512] * 8, 1) / 1e12 - 2.907) < 5e-4


def test_clock_sampler_summary_flags_throttle_reasons():
    cs = bench.ClockSampler(0)
    cs.lines = [
        "2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "1980, 2070, 1400.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    out = cs.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0).summary()
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_peaks_come_from_the_measured_file():
    hbm, tf, src = bench.peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        import json
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        assert (hbm, tf, src) == (float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured")
    else:
        assert (hbm, tf, src) == (6800.0, 1900.0, "fallback")
