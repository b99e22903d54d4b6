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


def _teacher_forced(m, first, start, ref, what):
    """Feed the oracle's ids one decode_step at a time (batch 1 runs the
    persistent kernel) and compare every row's logits, greedy id and
    final_norm_output with the oracle's."""
    tok = int(first)
    worst = 0.0
    for s in range(len(ref["ids"])):
        lg, idt = m.decode_step([0], [tok], [start + s])
        worst = max(worst, check_logits_ids(lg.cpu().numpy(), idt.cpu().numpy(), ref["logits"][s:s + 1],
                                            f"{what} step {s}"))
        check_hidden(m.final_hidden(1).cpu().numpy(), ref["final_norm_output"][s:s + 1], f"{what} step {s}")
        tok = int(ref["ids"][s])
    return worst


def test_decode_batch1_prompt128_256_steps(q2, weights, orc):
    """Config 2: every one of the 256 decode rows teacher-forced and compared
    element by element; the free-running greedy sequence as well, up to its
    first near-tie."""
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
        print(f"free-running greedy ids equal the oracle's for {n_ok} of {wl.decode_steps} steps")
        # Teacher forcing rewrites positions 128.. with the oracle's tokens.
        _teacher_forced(m, pre["ids"][0], len(prompt), ref, "0.5B")
        kv = m.kv_cache()[0].cpu().numpy()
        m.synchronize()
    check_kv(kv, cache, np.arange(0, len(prompt) + wl.decode_steps), "0.5B KV")


def test_decode_batch1_long_context(q2, weights, orc):
    """Config 3: all 96 rows at positions 4000..4095 teacher-forced and
    compared element by element (the persistent kernel's long-context
    attention split and per-head merge)."""
    wl = synth.WORKLOADS["0.5b-decode-b1-long"]
    prompt = wl.prompts(SHAPE.vocab)[0]
    cache = orc.new_cache()
    pre = orc.prefill(cache, prompt)
    ref = orc.greedy_decode(cache, int(pre["ids"][0]), len(prompt), wl.decode_steps)
    with q2.Qwen2Model(SHAPE, weights, n_ctx=wl.n_ctx, max_seqs=1, max_tokens=len(prompt)) as m:
        logits, ids = m.prefill([0], [prompt])
        check_logits_ids(logits.cpu().numpy(), ids.cpu().numpy(), pre["logits"], "long prefill")
        check_hidden(m.final_hidden(1).cpu().numpy(), pre["final_norm_output"], "long prefill")
        out = m.decode_steps([0], [int(pre["ids"][0])], [len(prompt)], wl.decode_steps).cpu().numpy()[:, 0]
        n_ok = check_free_running(out, ref["ids"], ref["logits"], "long greedy")
        print(f"free-running greedy ids equal the oracle's for {n_ok} of {wl.decode_steps} steps")
        _teacher_forced(m, pre["ids"][0], len(prompt), ref, "long")
        kv = m.kv_cache()[0].cpu().numpy()
        m.synchronize()
    sample = np.r_[0:8, 1000:1008, 3990:4096]
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
    """Config 5: 32 sequences at ragged positions (prompt lengths
    U{256..4032}), Q8_0 weights, every step a batch of 32 rows.  The oracle
    continues each sequence from the KV cache the GPU prefill wrote (its own
    prefill of the shortest prompt checks that cache).  Step 0 is compared
    for all 32 rows; 8 sequences (the shortest, the longest and six others)
    are teacher-forced through all 64 steps and compared at every step; the
    free-running greedy sequences are compared up to their first near-tie."""
    wl = synth.WORKLOADS["0.5b-decode-b32-q8"]
    prompts = wl.prompts(SHAPE.vocab)
    lens = [len(p) for p in prompts]
    S, T = len(prompts), wl.decode_steps
    orc = oracle.build_oracle(SHAPE, weights, wl.n_ctx, weight_format="q8_0")
    forced = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 1, 5, 11, 20, 23, 30})
    assert len(forced) == 8
    with q2.Qwen2Model(SHAPE, weights, n_ctx=wl.n_ctx, max_seqs=S, max_tokens=sum(lens),
                       weight_format=q2.WEIGHTS_Q8_0) as m:
        _, first = m.prefill(list(range(S)), prompts)
        first = [int(t) for t in first.cpu().numpy()]
        s0 = int(np.argmin(lens))
        own = orc.new_cache()
        pre = orc.prefill(own, prompts[s0])
        check_kv(m.kv_cache()[s0].cpu().numpy(), own, np.arange(lens[s0]), f"q8 prefill KV seq {s0}")
        # The oracle continues every sequence from the GPU's prefix cache.
        step0, refs = {}, {}
        for s in range(S):
            kv = m.kv_cache()[s, :, :, :, :lens[s]].cpu().numpy()
            cache = orc.new_cache()
            cache.K[:, :lens[s]] = np.transpose(kv[:, 0], (0, 2, 1, 3))
            cache.V[:, :lens[s]] = np.transpose(kv[:, 1], (0, 2, 1, 3))
            del kv
            if s in forced:
                refs[s] = orc.greedy_decode(cache, first[s], lens[s], T)
                step0[s] = (refs[s]["logits"][:1], refs[s]["final_norm_output"][:1])
            else:
                r = orc.forward(cache, [first[s]], [lens[s]])
                step0[s] = (r["logits"], r["final_norm_output"])
        assert int(pre["ids"][0]) == first[s0] or \
            pre["logits"][0][first[s0]] >= pre["logits"][0].max() - 2e-2
        out = m.decode_steps(list(range(S)), first, lens, T).cpu().numpy()
        # Teacher forcing: the forced rows take the oracle's ids, the others
        # their own greedy ids.
        toks = list(first)
        for step in range(T):
            lg, ids = m.decode_step(list(range(S)), toks, [n + step for n in lens])
            lg, ids = lg.cpu().numpy(), ids.cpu().numpy()
            hid = m.final_hidden(S).cpu().numpy()
            rows = range(S) if step == 0 else forced
            for s in rows:
                if step == 0:
                    rl, rh = step0[s]
                else:
                    rl = refs[s]["logits"][step:step + 1]
                    rh = refs[s]["final_norm_output"][step:step + 1]
                check_logits_ids(lg[s:s + 1], ids[s:s + 1], rl, f"q8 step {step} seq {s}")
                check_hidden(hid[s:s + 1], rh, f"q8 step {step} seq {s}")
            if step == 0:
                assert (out[0] == ids).all()
            toks = [int(refs[s]["ids"][step]) if s in forced else int(ids[s]) for s in range(S)]
        m.synchronize()
    for s in forced:
        n_ok = check_free_running(out[:, s], refs[s]["ids"], refs[s]["logits"], f"q8 greedy seq {s}")
        print(f"seq {s}: free-running greedy ids equal the oracle's for {n_ok} of {T} steps")
