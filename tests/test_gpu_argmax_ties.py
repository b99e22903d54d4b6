"""The greedy argmax keeps the lowest index of an exact tie on every LM-head
path of the GPU (xinfer "Module 7 -- Qwen2 / Qwen2.5", section 7.3: the
argmax over the tied head's logits runs on the device; ties go to the
lowest index).

Synthetic logits never tie by chance, so each test makes one: it runs a
decode step, takes the picked id m, copies the embedding row E[m] into a
lower row l that no input token uses (so the hidden state is unchanged),
and runs the same step again.  Rows l and m then hold the same bytes and
give bit-identical logits; the id must be l.  l is the lowest unused row
(near the start of the vocabulary) and m falls wherever the maximum is, so
the tie is usually settled by the merge across the head kernel's blocks."""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import qwen2_decoder_forward_gb300 as m
    from qwen2_decoder_forward_gb300 import build
    build.build()
    return m


def _step(q2, shape, w, prompts, kw):
    """Prefill, then one decode step of every sequence; logits and ids."""
    seqs = list(range(len(prompts)))
    with q2.Qwen2Model(shape, w, n_ctx=128, max_seqs=len(prompts),
                       max_tokens=sum(len(p) for p in prompts), **kw) as m:
        _, first = m.prefill(seqs, prompts)
        first = [int(t) for t in first.cpu().numpy()]
        lg, ids = m.decode_step(seqs, first, [len(p) for p in prompts])
        out = lg.cpu().numpy(), ids.cpu().numpy(), first
        m.synchronize()
    return out


def _tie_row(shape, prompts, first, m):
    used = set(int(t) for p in prompts for t in p) | set(first)
    return next(t for t in range(m) if t not in used)


@pytest.mark.parametrize("shape_name,batch,kw", [
    # batch 1: the persistent decode kernel's LM-head phase
    ("toy", 1, {}),
    ("ragged", 1, {}),
    # batch 2, and batch 1 with the persistent kernel switched off: the
    # per-step LM-head kernel with its two-stage argmax
    ("toy", 2, {}),
    ("ragged", 1, {"flags": "FLAG_NO_MEGAKERNEL"}),
    # Q8_0 weights: the batched product's tile-walking LM head
    ("toy", 3, {"weight_format": "WEIGHTS_Q8_0"}),
    ("ragged", 1, {"weight_format": "WEIGHTS_Q8_0"}),
])
def test_exact_tie_takes_the_lowest_index(q2, shape_name, batch, kw):
    kw = {k: getattr(q2, v) for k, v in kw.items()}
    shape = synth.SHAPES[shape_name]
    w = dict(synth.make_weights(shape, 4))
    prompts = [synth.make_tokens(shape.vocab, 9 + 4 * b, 700 + b) for b in range(batch)]
    lg, ids, first = _step(q2, shape, w, prompts, kw)
    b = batch - 1
    m = int(ids[b])
    assert m > 0 and lg[b, m] == lg[b].max()
    l = _tie_row(shape, prompts, first, m)
    w["embed"] = np.array(w["embed"], copy=True)
    w["embed"][l] = w["embed"][m]
    lg2, ids2, first2 = _step(q2, shape, w, prompts, kw)
    # A prefill row whose own greedy id was m now ties rows l and m as well:
    # it must pick l, and the decode step then reads E[l] = E[m] (the same
    # hidden state).
    assert first2 == [l if f == m else f for f in first]
    assert lg2[b, l].view(np.uint32) == lg2[b, m].view(np.uint32)
    assert lg2[b, m].view(np.uint32) == lg[b, m].view(np.uint32)
    assert int(ids2[b]) == l
    # Rows other than l are untouched: every other logit keeps its bits.
    keep = np.ones(shape.vocab, dtype=bool)
    keep[l] = False
    assert np.array_equal(lg2[:, keep].view(np.uint32), lg[:, keep].view(np.uint32))


@pytest.mark.parametrize("shape_name", ["toy", "ragged"])
def test_exact_tie_in_the_tensor_core_prefill_head(q2, shape_name):
    """The tensor-core prefill's LM head (tcgen05, E streamed as the MMA's M
    operand, per-CTA bests merged by the last CTA): copy E[m] of the last
    kept row's id m into an unused lower row l; the prefill's id must become
    l, with bit-identical logits for l and m."""
    shape = synth.SHAPES[shape_name]
    w = dict(synth.make_weights(shape, 5))
    prompts = [synth.make_tokens(shape.vocab, 40, 810), synth.make_tokens(shape.vocab, 23, 811)]

    def run(weights):
        with q2.Qwen2Model(shape, weights, n_ctx=128, max_seqs=2, max_tokens=64,
                           prefill_mode=q2.PREFILL_TENSOR) as m:
            assert m.features & q2.FEATURE_TENSOR_PREFILL
            lg, ids = m.prefill([0, 1], prompts, n_out=3)
            out = lg.cpu().numpy(), ids.cpu().numpy()
            m.synchronize()
        return out

    lg, ids = run(w)
    m = int(ids[-1])
    assert m > 0 and lg[-1, m] == lg[-1].max()
    used = set(int(t) for p in prompts for t in p)
    l = next(t for t in range(m) if t not in used)
    w["embed"] = np.array(w["embed"], copy=True)
    w["embed"][l] = w["embed"][m]
    lg2, ids2 = run(w)
    assert lg2[-1, l].view(np.uint32) == lg2[-1, m].view(np.uint32)
    assert lg2[-1, m].view(np.uint32) == lg[-1, m].view(np.uint32)
    assert int(ids2[-1]) == l
    # Every row whose maximum was m now picks l; the others keep their ids.
    assert list(ids2) == [l if int(i) == m else int(i) for i in ids]
