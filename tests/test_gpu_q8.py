"""GPU parity of the Q8_0 and Q4_0 weight paths (minfer "Qwen2 / Qwen2.5
Architecture Support", sections 3 and 6 name both formats): the library
quantises the f16 weights itself, the oracle dequantises the same blocks
exactly, and the batched decode product (up to 32 sequences per step) is
compared with the oracle row by row."""
import numpy as np
import pytest

import oracle
import synth
from parity import check_free_running, check_hidden, check_kv, check_logits_ids

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import qwen2_decoder_forward_gb300 as m
    from qwen2_decoder_forward_gb300 import build
    build.build()
    return m


def _prompts(shape, lens, seed):
    return [synth.make_tokens(shape.vocab, n, seed + i) for i, n in enumerate(lens)]


@pytest.mark.parametrize("shape_name,lens,n_ctx,fmt", [
    ("toy", [20, 45, 33], 128, "q8_0"), ("ragged", [20, 45, 33], 128, "q8_0"),
    ("toy", list(range(5, 25)), 128, "q8_0"),
    # one query head per kv head (group 1) through the batched attention
    ("toy-mha", [20, 45, 33], 128, "q8_0"),
    # long rows: many 64-key chunks, segments split across CTAs
    ("toy", [2500, 40, 1200, 700], 4096, "q8_0"),
    # n_ctx above 4096: the batched decode falls back to the split-k attention
    ("toy", [70, 130], 4160, "q8_0"),
    # Q4_0 weights through the same kernels (nibble codes instead of int8)
    ("toy", [20, 45, 33], 128, "q4_0"), ("ragged", [20, 45, 33], 128, "q4_0"),
    ("toy", list(range(5, 25)), 128, "q4_0"), ("toy-untied", [20, 45, 33], 128, "q4_0")])
def test_q8_prefill_and_teacher_forced_batched_decode(q2, shape_name, lens, n_ctx, fmt):
    """3 sequences (one 16-row M-tile) or 20 (two M-tiles): prefill on the f32
    path with Q8_0 weights, then teacher-forced decode steps of all rows at
    once, each row against the oracle on the same Q8_0 blocks."""
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 0)
    n_steps = 4
    prompts = _prompts(shape, lens, 300)
    orc = oracle.build_oracle(shape, w, n_ctx, weight_format=fmt)
    refs = []
    for p in prompts:
        cache = orc.new_cache()
        pre = orc.prefill(cache, p)
        refs.append((pre, orc.greedy_decode(cache, int(pre["ids"][0]), len(p), n_steps), cache))
    S = len(prompts)
    wf = q2.WEIGHTS_Q4_0 if fmt == "q4_0" else q2.WEIGHTS_Q8_0
    with q2.Qwen2Model(shape, w, n_ctx=n_ctx, max_seqs=S, max_tokens=sum(lens), weight_format=wf) as m:
        logits, ids = m.prefill(list(range(S)), prompts)
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        hid = m.final_hidden(S).cpu().numpy()
        for s in range(S):
            check_logits_ids(lg[s:s + 1], ig[s:s + 1], refs[s][0]["logits"], f"q8 prefill seq {s}")
            check_hidden(hid[s:s + 1], refs[s][0]["final_norm_output"], f"q8 prefill seq {s}")
        toks = [int(r[0]["ids"][0]) for r in refs]
        for step in range(n_steps):
            pos = [len(p) + step for p in prompts]
            lgt, idt = m.decode_step(list(range(S)), toks, pos)
            lgt, idt = lgt.cpu().numpy(), idt.cpu().numpy()
            hid = m.final_hidden(S).cpu().numpy()
            for s in range(S):
                dec = refs[s][1]
                check_logits_ids(lgt[s:s + 1], idt[s:s + 1], dec["logits"][step:step + 1], f"step {step} seq {s}")
                check_hidden(hid[s:s + 1], dec["final_norm_output"][step:step + 1], f"step {step} seq {s}")
            toks = [int(r[1]["ids"][step]) for r in refs]
        kv = m.kv_cache().cpu().numpy()
        m.synchronize()
    for s in range(S):
        check_kv(kv[s], refs[s][2], np.arange(len(prompts[s]) + n_steps), f"q8 KV seq {s}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_q8_free_running_decode_steps_batch_20(q2, fmt):
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    lens = list(range(3, 23))
    prompts = _prompts(shape, lens, 500)
    n_steps = 12
    orc = oracle.build_oracle(shape, w, 64, weight_format=fmt)
    refs = []
    for p in prompts:
        cache = orc.new_cache()
        pre = orc.prefill(cache, p)
        refs.append((int(pre["ids"][0]), orc.greedy_decode(cache, int(pre["ids"][0]), len(p), n_steps)))
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=20, max_tokens=sum(lens),
                       weight_format=q2.WEIGHTS_Q4_0 if fmt == "q4_0" else q2.WEIGHTS_Q8_0) as m:
        _, first = m.prefill(list(range(20)), prompts)
        first = [int(t) for t in first.cpu().numpy()]
        assert first == [r[0] for r in refs]
        out = m.decode_steps(list(range(20)), first, lens, n_steps).cpu().numpy()
        m.synchronize()
    for s in range(20):
        check_free_running(out[:, s], refs[s][1]["ids"], refs[s][1]["logits"], f"q8 seq {s}")
