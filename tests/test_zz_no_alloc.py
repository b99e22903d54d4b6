"""GPU test of qwen2_lm_head_argmax_noalloc, the LM head + greedy argmax for
callers that cannot let a library allocate device memory (its only scratch
is a static device array).  Two calls in a row are each compared with
qwen2_decode_step for the same rows (the final RMSNorm output read back
with qwen2_final_hidden): logits bit for bit and ids exactly, as the header
promises, and the logits against E . h computed in float64 on the host.
Named to run after the other GPU tests; it passes alone as well."""
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


def test_no_alloc_head_matches_decode_step_twice(q2):
    w = synth.make_weights(SHAPE, 0)
    prompts = [synth.make_tokens(SHAPE.vocab, n, seed=91 + n) for n in (12, 7, 30)]
    e_host = np.array(w["embed"], dtype=np.float16, copy=True)
    embed = torch.from_numpy(e_host).cuda()
    e64 = e_host.astype(np.float64)
    with q2.Qwen2Model(SHAPE, w, n_ctx=64, max_seqs=3, max_tokens=64) as m:
        _, ids = m.prefill([0, 1, 2], prompts)
        toks = [int(t) for t in ids.cpu().numpy()]
        pos = [len(p) for p in prompts]
        for call in range(2):
            lg, idd = m.decode_step([0, 1, 2], toks, pos)
            hid = m.final_hidden(3)
            nl, ni = q2.lm_head_argmax_noalloc(embed, hid)
            lg_np, nl_np = lg.cpu().numpy(), nl.cpu().numpy()
            assert np.array_equal(nl_np.view(np.uint32), lg_np.view(np.uint32)), f"call {call}: logits differ"
            np.testing.assert_array_equal(ni.cpu().numpy(), idd.cpu().numpy())
            # The head itself against its definition, logits = E . h.
            ref = hid.cpu().numpy().astype(np.float64) @ e64.T
            d = float(np.abs(nl_np - ref).max())
            assert d <= LOGIT_TOL, f"call {call}: max |dlogit| {d:.3e} against E . h"
            np.testing.assert_array_equal(ni.cpu().numpy(), np.argmax(nl_np, axis=1))
            # One row, no logits: the id alone.
            _, n1 = q2.lm_head_argmax_noalloc(embed, hid[1:2].contiguous(), want_logits=False)
            assert int(n1[0]) == int(idd[1])
            toks = [int(t) for t in idd.cpu().numpy()]
            pos = [p + 1 for p in pos]
        m.synchronize()


def test_no_alloc_head_nan_rows_give_an_index_inside_the_vocabulary(q2):
    """A NaN hidden row makes every logit of the row NaN; NaN orders above
    every number, so the id is the first index (0), never a sentinel."""
    w = synth.make_weights(SHAPE, 0)
    embed = torch.from_numpy(np.array(w["embed"], dtype=np.float16, copy=True)).cuda()
    g = torch.Generator().manual_seed(5)
    hid = torch.randn((3, SHAPE.hidden), generator=g, dtype=torch.float32).cuda()
    hid[1, 17] = float("nan")
    logits, ids = q2.lm_head_argmax_noalloc(embed, hid)
    lg, ii = logits.cpu().numpy(), ids.cpu().numpy()
    assert np.all(np.isnan(lg[1])) and int(ii[1]) == 0
    np.testing.assert_array_equal(ii[[0, 2]], np.argmax(lg[[0, 2]], axis=1))


def test_no_alloc_head_rejects_rows_beyond_its_scratch(q2):
    embed = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    hid = torch.zeros((9, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(q2.Qwen2Error) as e:
        q2.lm_head_argmax_noalloc(embed, hid)
    assert e.value.code == 1 and "n_rows" in str(e.value)
