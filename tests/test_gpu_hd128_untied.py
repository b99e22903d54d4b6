"""GPU parity of head_dim 128 and of untied LM heads (nnterp encyclopedia
qwen2: every size above 0.5B has head_dim 128, "Grouped-query attention";
from 7B up the embedding and the unembedding are separate matrices, "The
readout is the plain projection").  The shapes are small ones with those
properties (the pages print no intermediate sizes or vocabularies for the
larger models): toy-hd128 (4 q heads over 2 kv heads of 128, tied),
toy-untied (8 over 4 of 128, untied) and toy-untied-hd64 (the toy shape
with an untied head, which runs the batch-1 persistent kernel).  Each is
compared with the oracle: prefill, teacher-forced decode, free-running
greedy decode, the KV cache, on f16 and on Q8_0 weights."""
import numpy as np
import pytest

import oracle
import synth
from parity import check_free_running, check_hidden, check_kv, check_logits_ids

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = ["toy-hd128", "toy-untied", "toy-untied-hd64"]


@pytest.fixture(scope="module")
def q2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import qwen2_decoder_forward_gb300 as m
    from qwen2_decoder_forward_gb300 import build
    build.build()
    return m


def _refs(shape, w, prompts, n_steps, n_ctx, fmt):
    orc = oracle.build_oracle(shape, w, n_ctx, weight_format=fmt)
    out = []
    for p in prompts:
        cache = orc.new_cache()
        pre = orc.forward(cache, p, np.arange(len(p)), n_out=1)
        dec = orc.greedy_decode(cache, int(pre["ids"][-1]), len(p), n_steps)
        out.append((pre, dec, cache))
    return out


@pytest.mark.parametrize("fmt", ["f16", "q8_0"])
@pytest.mark.parametrize("shape_name", SHAPES)
def test_prefill_and_teacher_forced_decode(q2, shape_name, fmt):
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 0)
    assert ("lm_head" in w) == (not shape.tie_embeddings)
    n_ctx, n_steps = 160, 12
    prompts = [synth.make_tokens(shape.vocab, 37, 71), synth.make_tokens(shape.vocab, 70, 72)]
    ref = _refs(shape, w, prompts, n_steps, n_ctx, fmt)
    wf = q2.WEIGHTS_Q8_0 if fmt == "q8_0" else q2.WEIGHTS_F16
    with q2.Qwen2Model(shape, w, n_ctx=n_ctx, max_seqs=2, max_tokens=128, weight_format=wf) as m:
        logits, ids = m.prefill([0, 1], prompts)
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        hid = m.final_hidden(2).cpu().numpy()
        for s in range(2):
            check_logits_ids(lg[s:s + 1], ig[s:s + 1], ref[s][0]["logits"], f"{fmt} prefill seq {s}")
            check_hidden(hid[s:s + 1], ref[s][0]["final_norm_output"], f"{fmt} prefill seq {s}")
        toks = [int(ref[s][0]["ids"][-1]) for s in range(2)]
        for step in range(n_steps):
            pos = [len(prompts[0]) + step, len(prompts[1]) + step]
            lgt, idt = m.decode_step([0, 1], toks, pos)
            lgt, idt = lgt.cpu().numpy(), idt.cpu().numpy()
            hid = m.final_hidden(2).cpu().numpy()
            for s in range(2):
                dec = ref[s][1]
                check_logits_ids(lgt[s:s + 1], idt[s:s + 1], dec["logits"][step:step + 1], f"step {step} seq {s}")
                check_hidden(hid[s:s + 1], dec["final_norm_output"][step:step + 1], f"step {step} seq {s}")
            toks = [int(ref[s][1]["ids"][step]) for s in range(2)]
        kv = m.kv_cache().cpu().numpy()
        m.synchronize()
    for s in range(2):
        check_kv(kv[s], ref[s][2], np.arange(len(prompts[s]) + n_steps), f"{fmt} KV seq {s}")


@pytest.mark.parametrize("shape_name", SHAPES)
def test_free_running_batch1_decode(q2, shape_name):
    """qwen2_decode_steps at batch 1 (the persistent kernel where it applies:
    head_dim 64; the per-step graph for head_dim 128)."""
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 0)
    prompt = synth.make_tokens(shape.vocab, 16, 1001)
    n_steps = 24
    (pre, dec, cache), = _refs(shape, w, [prompt], n_steps, 64, "f16")
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        if shape.head_dim == 64:
            assert m.features & q2.FEATURE_PERSISTENT_DECODE, q2.lib().qwen2_last_error(m._h).decode()
        else:
            assert not m.features & q2.FEATURE_PERSISTENT_DECODE
        logits, ids = m.prefill([0], [prompt])
        check_logits_ids(logits.cpu().numpy(), ids.cpu().numpy(), pre["logits"], "prefill")
        out = m.decode_steps([0], [int(ids[0])], [16], n_steps).cpu().numpy()[:, 0]
        # Teacher-forced rows through decode_step at batch 1 as well.
        tok = int(pre["ids"][0])
        for s in range(n_steps):
            lg, idt = m.decode_step([0], [tok], [16 + s])
            check_logits_ids(lg.cpu().numpy(), idt.cpu().numpy(), dec["logits"][s:s + 1], f"b1 step {s}")
            check_hidden(m.final_hidden(1).cpu().numpy(), dec["final_norm_output"][s:s + 1], f"b1 step {s}")
            tok = int(dec["ids"][s])
        kv = m.kv_cache()[0].cpu().numpy()
        m.synchronize()
    n_ok = check_free_running(out, dec["ids"], dec["logits"], f"{shape_name} greedy")
    print(f"{shape_name}: free-running greedy ids equal the oracle's for {n_ok} of {n_steps} steps")
    check_kv(kv, cache, np.arange(16 + n_steps), f"{shape_name} KV")


def test_untied_head_is_the_readout_and_tied_embedding_the_input(q2):
    """With lm_head equal to the embedding the untied model gives the tied
    model's logits bit for bit; with a different head only the readout
    changes (the hidden state is the same)."""
    tied = synth.SHAPES["toy"]
    untied = synth.SHAPES["toy-untied-hd64"]
    w = dict(synth.make_weights(tied, 0))
    prompt = synth.make_tokens(tied.vocab, 20, 5)
    outs = []
    for head in (None, w["embed"], synth.make_weights(untied, 0)["lm_head"]):
        ww = dict(w)
        shp = tied
        if head is not None:
            ww["lm_head"] = head
            shp = untied
        with q2.Qwen2Model(shp, ww, n_ctx=64, max_seqs=1, max_tokens=32) as m:
            lg, _ = m.prefill([0], [prompt])
            h = m.final_hidden(1).cpu().numpy()
            lg2, _ = m.decode_step([0], [7], [20])
            outs.append((lg.cpu().numpy(), h, lg2.cpu().numpy()))
            m.synchronize()
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert np.array_equal(outs[0][2].view(np.uint32), outs[1][2].view(np.uint32))
    assert np.array_equal(outs[0][1].view(np.uint32), outs[2][1].view(np.uint32))
    assert not np.array_equal(outs[0][0], outs[2][0])
