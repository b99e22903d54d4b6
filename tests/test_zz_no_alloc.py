"""GPU test of qwen2_lm_head_argmax_noalloc, the context-free LM head +
argmax whose scratch is a static device array: two calls in a row, each
compared with qwen2_decode_step's own logits and ids for the same rows
(the final RMSNorm output read back with qwen2_final_hidden).  Named to run
after the other GPU tests; it passes alone as well."""
import numpy as np
import pytest

import synth
from parity import LOGIT_TOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPE = synth.SHAPES["ragged"]   # V = 5003: a ragged last block of the head


@pytest.fixture(scope="module")
def q2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import qwen2_decoder_forward_gb300 as m
    from qwen2_decoder_forward_gb300 import build
    build.build()
    return m


def _same_pick(ids_a, ids_b, logits_b):
    """ids_a agrees with ids_b, or picks a logit within the test tolerance of
    ids_b's maximum."""
    for r in range(len(ids_b)):
        a, b = int(ids_a[r]), int(ids_b[r])
        assert a == b or logits_b[r, a] >= logits_b[r, b] - LOGIT_TOL, f"row {r}: id {a} vs {b}"


def test_no_alloc_head_matches_decode_step_twice(q2):
    w = synth.make_weights(SHAPE, 0)
    prompts = [synth.make_tokens(SHAPE.vocab, n, seed=91 + n) for n in (12, 7, 30)]
    embed = torch.from_numpy(np.ascontiguousarray(w["embed"])).cuda()
    with q2.Qwen2Model(SHAPE, w, n_ctx=64, max_seqs=3, max_tokens=64) as m:
        _, ids = m.prefill([0, 1, 2], prompts)
        toks = [int(t) for t in ids.cpu().numpy()]
        pos = [len(p) for p in prompts]
        for call in range(2):
            lg, idd = m.decode_step([0, 1, 2], toks, pos)
            hid = m.final_hidden(3)
            nl, ni = q2.lm_head_argmax_noalloc(embed, hid)
            lg_np, nl_np = lg.cpu().numpy(), nl.cpu().numpy()
            d = float(np.abs(nl_np.astype(np.float64) - lg_np).max())
            assert d <= LOGIT_TOL, f"call {call}: max |dlogit| {d:.3e}"
            _same_pick(ni.cpu().numpy(), idd.cpu().numpy(), lg_np)
            # One row, no logits: the id alone.
            _, n1 = q2.lm_head_argmax_noalloc(embed, hid[1:2].contiguous(), want_logits=False)
            _same_pick(n1.cpu().numpy(), idd.cpu().numpy()[1:2], lg_np[1:2])
            toks = [int(t) for t in idd.cpu().numpy()]
            pos = [p + 1 for p in pos]
        m.synchronize()


def test_no_alloc_head_rejects_rows_beyond_its_scratch(q2):
    embed = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    hid = torch.zeros((9, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(q2.Qwen2Error) as e:
        q2.lm_head_argmax_noalloc(embed, hid)
    assert e.value.code == 1 and "n_rows" in str(e.value)
