"""GPU parity at the full Qwen2.5-0.5B shape, in the launch configuration the
benchmark times (prefill, then greedy decode through qwen2_decode_steps'
CUDA graph), on outputs the oracle computes one row at a time."""
import numpy as np
import pytest

import oracle
import synth
from parity import check_free_running, check_hidden, check_kv, check_logits_ids

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPE = synth.SHAPES["qwen2.5-0.5b"]


@pytest.fixture(scope="module")
def q2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import qwen2_decoder_forward_gb300 as m
    from qwen2_decoder_forward_gb300 import build
    build.build()
    return m


@pytest.fixture(scope="module")
def weights():
    return synth.make_weights(SHAPE, 0)


@pytest.fixture(scope="module")
def orc(weights):
    return oracle.build_oracle(SHAPE, weights, 4096)


def test_decode_batch1_prompt128_256_steps(q2, weights, orc):
    wl = synth.WORKLOADS["0.5b-decode-b1"]
    prompt = wl.prompts(SHAPE.vocab)[0]
    cache = orc.new_cache()
    pre = orc.prefill(cache, prompt)
    ref = orc.greedy_decode(cache, int(pre["ids"][0]), len(prompt), wl.decode_steps)
    with q2.Qwen2Model(SHAPE, weights, n_ctx=wl.n_ctx, max_seqs=1, max_tokens=len(prompt)) as m:
        assert m.weight_bytes >= 987_922_432
        assert m.features & q2.FEATURE_PERSISTENT_DECODE, q2.lib().qwen2_last_error(m._h).decode()
        logits, ids = m.prefill([0], [prompt])
        check_logits_ids(logits.cpu().numpy(), ids.cpu().numpy(), pre["logits"], "prefill")
        check_hidden(m.final_hidden(1).cpu().numpy(), pre["final_norm_output"], "prefill")
        out = m.decode_steps([0], [int(pre["ids"][0])], [len(prompt)], wl.decode_steps).cpu().numpy()[:, 0]
        n_ok = check_free_running(out, ref["ids"], ref["logits"], "0.5B greedy")
        assert n_ok >= 32, f"greedy sequences diverged at a near-tie after {n_ok} steps"
        # Teacher-forced rows at sampled steps: feed the oracle's ids.
        tok = int(pre["ids"][0])
        for s in range(8):
            lg, idt = m.decode_step([0], [tok], [len(prompt) + s])
            check_logits_ids(lg.cpu().numpy(), idt.cpu().numpy(), ref["logits"][s:s + 1], f"step {s}")
            check_hidden(m.final_hidden(1).cpu().numpy(), ref["final_norm_output"][s:s + 1], f"step {s}")
            tok = int(ref["ids"][s])
        kv = m.kv_cache()[0].cpu().numpy()
        m.synchronize()
    check_kv(kv, cache, np.arange(0, len(prompt) + 8), "0.5B KV")


def test_decode_batch1_long_context(q2, weights, orc):
    wl = synth.WORKLOADS["0.5b-decode-b1-long"]
    prompt = wl.prompts(SHAPE.vocab)[0]
    cache = orc.new_cache()
    pre = orc.prefill(cache, prompt)
    ref = orc.greedy_decode(cache, int(pre["ids"][0]), len(prompt), wl.decode_steps)
    with q2.Qwen2Model(SHAPE, weights, n_ctx=wl.n_ctx, max_seqs=1, max_tokens=len(prompt)) as m:
        logits, ids = m.prefill([0], [prompt])
        check_logits_ids(logits.cpu().numpy(), ids.cpu().numpy(), pre["logits"], "long prefill")
        out = m.decode_steps([0], [int(pre["ids"][0])], [len(prompt)], wl.decode_steps).cpu().numpy()[:, 0]
        n_ok = check_free_running(out, ref["ids"], ref["logits"], "long greedy")
        assert n_ok >= 16
        kv = m.kv_cache()[0].cpu().numpy()
        m.synchronize()
    sample = np.r_[0:8, 1000:1008, 3990:4000 + n_ok]
    check_kv(kv, cache, sample, "long KV")


def test_prefill_8x512_tail_cut(q2, weights, orc):
    wl = synth.WORKLOADS["0.5b-prefill-8x512"]
    prompts = wl.prompts(SHAPE.vocab)
    refs = []
    for i in (0, 5):
        refs.append(orc.prefill(orc.new_cache(), prompts[i]))
    with q2.Qwen2Model(SHAPE, weights, n_ctx=wl.n_ctx, max_seqs=8, max_tokens=8 * 512) as m:
        logits, ids = m.prefill(list(range(8)), prompts, n_out=1)
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        hid = m.final_hidden(8).cpu().numpy()
        m.synchronize()
    for j, i in enumerate((0, 5)):
        check_logits_ids(lg[i:i + 1], ig[i:i + 1], refs[j]["logits"], f"prefill seq {i}")
        check_hidden(hid[i:i + 1], refs[j]["final_norm_output"], f"prefill seq {i}")


def test_prefill_8x512_tensor_cores(q2, weights, orc):
    """Config 4 as the benchmark runs it: tcgen05 GEMMs on f16 operands."""
    wl = synth.WORKLOADS["0.5b-prefill-8x512"]
    prompts = wl.prompts(SHAPE.vocab)
    caches = {i: orc.new_cache() for i in (0, 3, 7)}
    refs = {i: orc.prefill(caches[i], prompts[i]) for i in caches}
    with q2.Qwen2Model(SHAPE, weights, n_ctx=wl.n_ctx, max_seqs=8, max_tokens=8 * 512,
                       prefill_mode=q2.PREFILL_TENSOR) as m:
        assert m.features & q2.FEATURE_TENSOR_PREFILL
        logits, ids = m.prefill(list(range(8)), prompts, n_out=1)
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        hid = m.final_hidden(8).cpu().numpy()
        kv3 = m.kv_cache()[3].cpu().numpy()
        m.synchronize()
    for i, r in refs.items():
        check_logits_ids(lg[i:i + 1], ig[i:i + 1], r["logits"], f"tensor prefill seq {i}")
        check_hidden(hid[i:i + 1], r["final_norm_output"], f"tensor prefill seq {i}")
    check_kv(kv3, caches[3], np.r_[0:8, 250:258, 504:512], "tensor prefill KV seq 3")


def test_batched_decode_32_ragged_q8(q2, weights):
    """Config 5: 32 sequences at ragged positions (prompt lengths U{256..4032}),
    Q8_0 weights, 64 greedy steps of all 32 rows per launch.  The oracle
    continues four of the sequences (the shortest, the longest and two
    others) from the KV cache the GPU prefill wrote, teacher-forced at step 0
    and free-running over the 64 steps; the shortest prompt's KV rows are
    checked against the oracle's own prefill."""
    wl = synth.WORKLOADS["0.5b-decode-b32-q8"]
    prompts = wl.prompts(SHAPE.vocab)
    lens = [len(p) for p in prompts]
    orc = oracle.build_oracle(SHAPE, weights, wl.n_ctx, weight_format="q8_0")
    sample = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 5, 17})
    with q2.Qwen2Model(SHAPE, weights, n_ctx=wl.n_ctx, max_seqs=32, max_tokens=sum(lens),
                       weight_format=q2.WEIGHTS_Q8_0) as m:
        _, first = m.prefill(list(range(32)), prompts)
        first = [int(t) for t in first.cpu().numpy()]
        kv = {s: m.kv_cache()[s].cpu().numpy() for s in sample}
        lg0, id0 = m.decode_step(list(range(32)), first, lens)
        lg0, id0 = lg0.cpu().numpy(), id0.cpu().numpy()
        out = m.decode_steps(list(range(32)), first, lens, wl.decode_steps).cpu().numpy()
        m.synchronize()
    assert (out[0] == id0).all()
    s0 = sample[0]
    own = orc.new_cache()
    pre = orc.prefill(own, prompts[s0])
    assert int(pre["ids"][0]) == first[s0] or abs(pre["logits"][0][first[s0]] - pre["logits"][0].max()) < 2e-2
    check_kv(kv[s0], own, np.arange(lens[s0]), f"q8 prefill KV seq {s0}")
    for s in sample:
        cache = orc.new_cache()
        n = lens[s]
        cache.K[:, :n] = np.transpose(kv[s][:, 0, :, :n], (0, 2, 1, 3))
        cache.V[:, :n] = np.transpose(kv[s][:, 1, :, :n], (0, 2, 1, 3))
        ref = orc.greedy_decode(cache, first[s], n, wl.decode_steps)
        check_logits_ids(lg0[s:s + 1], id0[s:s + 1], ref["logits"][:1], f"q8 step 0 seq {s}")
        n_ok = check_free_running(out[:, s], ref["ids"], ref["logits"], f"q8 greedy seq {s}")
        assert n_ok >= 8, f"seq {s} diverged at a near-tie after {n_ok} steps"
