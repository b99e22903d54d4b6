"""GPU parity of the CUDA path against the oracle on shapes the oracle runs
in seconds (toy, ragged, multi-head), element by element, plus the path's
invariants: fused == unfused and graph == no-graph bit for bit, batch
invariance, the position error, and KV save / restore."""
import numpy as np
import pytest

import oracle
import synth
from parity import (check_free_running, check_hidden, check_kv, check_logits_ids)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q2():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import qwen2_decoder_forward_gb300 as m
    from qwen2_decoder_forward_gb300 import build
    build.build()
    return m


def run_oracle(shape, w, prompts, n_steps, n_ctx, n_out=1):
    orc = oracle.build_oracle(shape, w, n_ctx)
    out = []
    for p in prompts:
        cache = orc.new_cache()
        pre = orc.forward(cache, p, np.arange(len(p)), n_out=n_out)
        dec = orc.greedy_decode(cache, int(pre["ids"][-1]), len(p), n_steps)
        out.append((pre, dec, cache))
    return orc, out


@pytest.mark.parametrize("shape_name", ["toy", "ragged", "toy-mha", "toy-g8"])
def test_prefill_and_teacher_forced_decode(q2, shape_name):
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 0)
    n_ctx, n_steps = 160, 16
    prompts = [synth.make_tokens(shape.vocab, 37, 7), synth.make_tokens(shape.vocab, 70, 8)]
    _, ref = run_oracle(shape, w, prompts, n_steps, n_ctx, n_out=2)
    with q2.Qwen2Model(shape, w, n_ctx=n_ctx, max_seqs=2, max_tokens=128) as m:
        logits, ids = m.prefill([0, 1], prompts, n_out=2)
        hid = m.final_hidden(4).cpu().numpy()
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        for s in range(2):
            pre = ref[s][0]
            check_logits_ids(lg[2 * s:2 * s + 2], ig[2 * s:2 * s + 2], pre["logits"], f"prefill seq {s}")
            check_hidden(hid[2 * s:2 * s + 2], pre["final_norm_output"], f"prefill seq {s}")
        # Teacher-forced batch decode: both sequences each step, fed the
        # oracle's ids.
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
            check_kv(kv[s], ref[s][2], np.arange(len(prompts[s]) + n_steps), f"seq {s}")


def test_free_running_decode_steps_matches_oracle(q2):
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    prompt = synth.make_tokens(shape.vocab, 16, 1001)
    _, ref = run_oracle(shape, w, [prompt], 16, 64)
    pre, dec, _ = ref[0]
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        _, ids = m.prefill([0], [prompt])
        assert int(ids[0]) == int(pre["ids"][0])
        out = m.decode_steps([0], [int(ids[0])], [16], 16).cpu().numpy()[:, 0]
        # Host output buffer path (the call synchronises).
        host = np.zeros((16, 1), dtype=np.int32)
        m.decode_steps([0], [int(ids[0])], [16], 16, ids_out=host)
        m.synchronize()
    assert check_free_running(out, dec["ids"], dec["logits"], "toy greedy") == 16
    np.testing.assert_array_equal(host[:, 0], out)


@pytest.mark.parametrize("shape_name,batch", [("toy", 1), ("ragged", 3)])
def test_generation_stops_at_stop_ids(q2, shape_name, batch):
    """Stop tokens (minfer page section 5): after each sequence's first
    generated stop id the ids are -1 and n_generated counts the stop id.
    Batch 1 runs the persistent kernel, batch 3 the step graph.  The result
    must be the GPU's own plain greedy sequence cut at the stop (exact), and
    the oracle's stop-aware generation wherever the two greedy sequences
    agree up to the stop."""
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 0)
    n, n_ctx = 24, 64
    prompts = [synth.make_tokens(shape.vocab, 6 + 5 * b, 600 + b) for b in range(batch)]
    orc, ref = run_oracle(shape, w, prompts, n, n_ctx)
    seqs = list(range(batch))
    with q2.Qwen2Model(shape, w, n_ctx=n_ctx, max_seqs=batch, max_tokens=sum(len(p) for p in prompts)) as m:
        _, ids0 = m.prefill(seqs, prompts)
        first = [int(t) for t in ids0.cpu().numpy()]
        starts = [len(p) for p in prompts]
        plain = m.decode_steps(seqs, first, starts, n).cpu().numpy()
        # Stop ids that occur: one early in the first sequence, one later in
        # the last, and one that never occurs in the batch's plain output.
        never = next(t for t in range(shape.vocab) if t not in set(plain.reshape(-1).tolist()))
        stops = [int(plain[4, 0]), int(plain[13, batch - 1]), never]
        ids, n_gen = m.generate(seqs, first, starts, n, stops)
        ids, n_gen = ids.cpu().numpy(), n_gen.cpu().numpy()
        # Host outputs give the same.
        h_ids = np.zeros((n, batch), dtype=np.int32)
        h_n = np.zeros((batch,), dtype=np.int32)
        m.generate(seqs, first, starts, n, stops, ids_out=h_ids, n_generated_out=h_n)
        # No stop ids: nothing masked, every step counted.
        ids_all, n_all = m.generate(seqs, first, starts, n, [])
        with pytest.raises(q2.Qwen2Error) as e:
            m.generate(seqs, first, starts, n, [shape.vocab])
        assert e.value.code == q2.QWEN2_E_ARG
        with pytest.raises(q2.Qwen2Error) as e:
            m.generate(seqs, first, starts, n, list(range(9)))
        assert e.value.code == q2.QWEN2_E_ARG
        m.synchronize()
    np.testing.assert_array_equal(h_ids, ids)
    np.testing.assert_array_equal(h_n, n_gen)
    np.testing.assert_array_equal(ids_all.cpu().numpy(), plain)
    assert np.all(n_all.cpu().numpy() == n)
    for b in range(batch):
        hit = [s for s in range(n) if int(plain[s, b]) in stops]
        k = hit[0] if hit else n - 1
        assert int(n_gen[b]) == k + 1
        np.testing.assert_array_equal(ids[:k + 1, b], plain[:k + 1, b])
        assert np.all(ids[k + 1:, b] == -1)
        # Against the oracle: the GPU's plain sequence matches the oracle's
        # up to a near-tie (checked); up to there the stop must agree too.
        pre, dec, _ = ref[b]
        if first[b] != int(pre["ids"][-1]):
            continue
        agree = check_free_running(plain[:, b], dec["ids"], dec["logits"], f"seq {b}")
        if agree > k:
            cache = orc.new_cache()
            orc.forward(cache, prompts[b], np.arange(len(prompts[b])))
            r = orc.greedy_generate(cache, first[b], len(prompts[b]), n, stops)
            assert r["n_generated"] == int(n_gen[b])
            np.testing.assert_array_equal(r["ids"], ids[:, b])


@pytest.mark.parametrize("shape_name", ["ragged", "toy"])
@pytest.mark.parametrize("flags", ["fuse", "graph"])
def test_variants_are_bit_identical(q2, flags, shape_name):
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 1)
    prompt = synth.make_tokens(shape.vocab, 40, 9)
    # Batch-1 decode runs the persistent kernel by default; the unfused flags
    # and FLAG_NO_MEGAKERNEL select the per-step kernels.
    variants = ([0, q2.FLAG_NO_MEGAKERNEL, q2.FLAG_NO_FUSE_QKV | q2.FLAG_NO_FUSE_FFN, q2.FLAG_NO_FUSE_QKV,
                 q2.FLAG_NO_FUSE_FFN]
                if flags == "fuse" else [0, q2.FLAG_NO_GRAPH, q2.FLAG_NO_GRAPH | q2.FLAG_NO_MEGAKERNEL])
    outs = []
    for f in variants:
        with q2.Qwen2Model(shape, w, n_ctx=128, max_seqs=1, max_tokens=64, flags=f) as m:
            if f == 0:
                assert m.features & q2.FEATURE_PERSISTENT_DECODE, q2.lib().qwen2_last_error(m._h).decode()
            m.prefill([0], [prompt])
            rows = []
            tok = 5
            for s in range(6):
                lg, ids = m.decode_step([0], [tok], [40 + s])
                rows.append(lg.cpu().numpy().copy())
                rows.append(m.final_hidden(1).cpu().numpy()[0].copy())
                tok = int(ids[0])
            ids = m.decode_steps([0], [tok], [46], 70).cpu().numpy()
            m.synchronize()
            outs.append((np.concatenate([r.ravel() for r in rows]), ids))
    for o in outs[1:]:
        assert np.array_equal(o[0].view(np.uint32), outs[0][0].view(np.uint32))
        np.testing.assert_array_equal(o[1], outs[0][1])


def test_batch_invariance(q2):
    """A sequence's decode row gives the same bits alone or in a batch."""
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 2)
    prompts = [synth.make_tokens(shape.vocab, n, 20 + n) for n in (5, 9, 13)]
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=3, max_tokens=32) as m:
        m.prefill([0, 1, 2], prompts)
        kv0 = m.kv_cache().clone()
        lb, _ = m.decode_step([0, 1, 2], [1, 2, 3], [5, 9, 13])
        lb = lb.cpu().numpy()
        m.kv_cache().copy_(kv0)
        for s in range(3):
            ls, _ = m.decode_step([s], [s + 1], [[5, 9, 13][s]])
            assert np.array_equal(ls.cpu().numpy()[0].view(np.uint32), lb[s].view(np.uint32))


def test_position_outside_n_ctx_is_an_error_and_writes_nothing(q2):
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    with q2.Qwen2Model(shape, w, n_ctx=32, max_seqs=1, max_tokens=8) as m:
        m.prefill([0], [[1, 2, 3]])
        before = m.kv_cache().clone()
        with pytest.raises(q2.Qwen2Error) as e:
            m.decode_step([0], [4], [32])
        assert e.value.code == q2.QWEN2_E_POS
        with pytest.raises(q2.Qwen2Error) as e:
            m.decode_steps([0], [4], [30], 3)
        assert e.value.code == q2.QWEN2_E_POS
        with pytest.raises(q2.Qwen2Error) as e:
            m.prefill([0], [[1, 2]], positions=[[31, 32]])
        assert e.value.code == q2.QWEN2_E_POS
        with pytest.raises(q2.Qwen2Error) as e:
            m.decode_step([0], [shape.vocab], [3])
        assert e.value.code == q2.QWEN2_E_ARG
        m.synchronize()
        assert torch.equal(m.kv_cache(), before)
        m.decode_steps([0], [4], [29], 3)      # the last allowed position
        m.synchronize()


def test_kv_cache_save_and_restore(q2):
    """Decode, save the caller-visible cache, destroy, recreate, restore and
    continue: the ids equal an uninterrupted run."""
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 3)
    prompt = synth.make_tokens(shape.vocab, 12, 30)
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        _, ids = m.prefill([0], [prompt])
        full = m.decode_steps([0], [int(ids[0])], [12], 20).cpu().numpy()[:, 0]
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        _, ids = m.prefill([0], [prompt])
        first = m.decode_steps([0], [int(ids[0])], [12], 10).cpu().numpy()[:, 0]
        saved = m.kv_cache().cpu().clone()
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        m.kv_cache().copy_(saved.cuda())
        rest = m.decode_steps([0], [int(first[-1])], [22], 10).cpu().numpy()[:, 0]
        m.synchronize()
    np.testing.assert_array_equal(np.concatenate([first, rest]), full)


@pytest.mark.parametrize("shape_name", ["toy", "ragged", "toy-mha", "toy-g8"])
def test_tensor_core_prefill(q2, shape_name):
    """QWEN2_PREFILL_TENSOR (tcgen05 GEMMs on f16 operands): two sequences of
    37 and 150 rows (two 128-row tiles, the second ragged) with the tail cut,
    then one 60-row prompt with every row kept (no cut: all layers on tensor
    cores), against the oracle; KV cache rows too."""
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 0)
    n_ctx = 192
    prompts = [synth.make_tokens(shape.vocab, 37, 17), synth.make_tokens(shape.vocab, 150, 18)]
    orc = oracle.build_oracle(shape, w, n_ctx)
    ref = []
    for p in prompts:
        cache = orc.new_cache()
        ref.append((orc.forward(cache, p, np.arange(len(p)), n_out=2), None, cache))
    full = synth.make_tokens(shape.vocab, 60, 19)
    fcache = orc.new_cache()
    fref = orc.forward(fcache, full, np.arange(len(full)), n_out=len(full))
    with q2.Qwen2Model(shape, w, n_ctx=n_ctx, max_seqs=2, max_tokens=192,
                       prefill_mode=q2.PREFILL_TENSOR) as m:
        assert m.features & q2.FEATURE_TENSOR_PREFILL
        logits, ids = m.prefill([0, 1], prompts, n_out=2)
        hid = m.final_hidden(4).cpu().numpy()
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        kv = m.kv_cache().cpu().numpy()
        for s in range(2):
            pre = ref[s][0]
            check_logits_ids(lg[2 * s:2 * s + 2], ig[2 * s:2 * s + 2], pre["logits"], f"tensor prefill seq {s}")
            check_hidden(hid[2 * s:2 * s + 2], pre["final_norm_output"], f"tensor prefill seq {s}")
            check_kv(kv[s], ref[s][2], np.arange(len(prompts[s])), f"tensor prefill KV seq {s}")
        logits, ids = m.prefill([0], [full], n_out=len(full))
        hid = m.final_hidden(len(full)).cpu().numpy()
        check_logits_ids(logits.cpu().numpy(), ids.cpu().numpy(), fref["logits"], "tensor prefill, no cut")
        check_hidden(hid, fref["final_norm_output"], "tensor prefill, no cut")
        m.synchronize()


@pytest.mark.parametrize("shape_name", ["toy", "ragged", "toy-g8"])
def test_tensor_core_prefill_in_chunks(q2, shape_name):
    """Chunked prefill on the tensor-core path: the second call's rows attend
    to keys an earlier call stored (prefixes of 70 and 31 positions, neither
    a whole 64-key tile; n_ctx 200 is not a multiple of 64 either), against
    the oracle run in the same chunks; KV cache rows too."""
    shape = synth.SHAPES[shape_name]
    w = synth.make_weights(shape, 0)
    n_ctx = 200
    a = synth.make_tokens(shape.vocab, 150, 21)
    b = synth.make_tokens(shape.vocab, 100, 22)
    cut = (70, 31)
    orc = oracle.build_oracle(shape, w, n_ctx)
    caches, refs = [], []
    for t, c in zip((a, b), cut):
        cache = orc.new_cache()
        orc.forward(cache, t[:c], np.arange(c), n_out=1)
        refs.append(orc.forward(cache, t[c:], np.arange(c, len(t)), n_out=2))
        caches.append(cache)
    with q2.Qwen2Model(shape, w, n_ctx=n_ctx, max_seqs=2, max_tokens=192,
                       prefill_mode=q2.PREFILL_TENSOR) as m:
        m.prefill([0, 1], [a[:cut[0]], b[:cut[1]]], n_out=1)
        logits, ids = m.prefill([0, 1], [a[cut[0]:], b[cut[1]:]],
                                positions=[np.arange(cut[0], len(a)), np.arange(cut[1], len(b))], n_out=2)
        hid = m.final_hidden(4).cpu().numpy()
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        kv = m.kv_cache().cpu().numpy()
        for s, t in enumerate((a, b)):
            what = f"chunked tensor prefill seq {s}"
            check_logits_ids(lg[2 * s:2 * s + 2], ig[2 * s:2 * s + 2], refs[s]["logits"], what)
            check_hidden(hid[2 * s:2 * s + 2], refs[s]["final_norm_output"], what)
            check_kv(kv[s], caches[s], np.arange(len(t)), what + " KV")
        m.synchronize()


def test_tensor_core_prefill_at_unordered_positions(q2):
    """Positions are data: one sequence's rows at the positions 69..0 in
    reverse, another's at 0..29 and 40..69 (a gap that holds the cache's
    zeros on both sides).  The tensor-core prefill then converts every key
    up to each sequence's last position from the f32 cache (its rows are not
    consecutive), against the oracle given the same positions."""
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    n_ctx = 128
    a = synth.make_tokens(shape.vocab, 70, 31)
    b = synth.make_tokens(shape.vocab, 60, 32)
    pa = np.arange(69, -1, -1)
    pb = np.r_[0:30, 40:70]
    orc = oracle.build_oracle(shape, w, n_ctx)
    ca, cb = orc.new_cache(), orc.new_cache()
    ra = orc.forward(ca, a, pa, n_out=2)
    rb = orc.forward(cb, b, pb, n_out=2)
    with q2.Qwen2Model(shape, w, n_ctx=n_ctx, max_seqs=2, max_tokens=192,
                       prefill_mode=q2.PREFILL_TENSOR) as m:
        logits, ids = m.prefill([0, 1], [a, b], positions=[pa, pb], n_out=2)
        hid = m.final_hidden(4).cpu().numpy()
        lg, ig = logits.cpu().numpy(), ids.cpu().numpy()
        kv = m.kv_cache().cpu().numpy()
        m.synchronize()
    for s, (r, cache, pos) in enumerate(((ra, ca, pa), (rb, cb, pb))):
        what = f"unordered tensor prefill seq {s}"
        check_logits_ids(lg[2 * s:2 * s + 2], ig[2 * s:2 * s + 2], r["logits"], what)
        check_hidden(hid[2 * s:2 * s + 2], r["final_norm_output"], what)
        check_kv(kv[s], cache, np.sort(pos), what + " KV")


def test_canary_check_finds_a_write_past_a_buffer(q2):
    """The guard words around the context's device buffers: a clean run
    passes the check; four bytes written just past the end of the KV cache
    (into its trailing guard region, which is allocated memory) make the
    check fail with QWEN2_E_DEVICE_GUARD; restoring them makes it pass."""
    import torch
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    prompt = synth.make_tokens(shape.vocab, 16, 1002)
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        _, ids = m.prefill([0], [prompt])
        m.decode_steps([0], [int(ids[0])], [16], 4)
        m.check_canaries()
        kv = m.kv_cache()
        end = kv.data_ptr() + kv.numel() * 4
        tail = torch.as_tensor(q2._CudaArray(end, [1], "<i4"), device="cuda")
        canary = int(np.array([0xA5A5A5A5], dtype=np.uint32).view(np.int32)[0])
        assert int(tail.item()) == canary
        tail.fill_(0)
        torch.cuda.synchronize()
        with pytest.raises(q2.Qwen2Error) as e:
            m.check_canaries()
        assert e.value.code == q2.QWEN2_E_DEVICE_GUARD
        assert "canary after device buffer" in str(e.value)
        tail.fill_(canary)
        torch.cuda.synchronize()
        m.check_canaries()


def test_device_guard_is_reported_once_and_decoding_continues(q2):
    """Failure detection without a GPU fault: the test hook writes the
    device guard word the way a kernel's bounded wait does when it gives up.
    synchronize reports QWEN2_E_DEVICE_GUARD once, clears the word and resets
    the persistent kernel's exchange state, and the next decode gives the
    same ids as before."""
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    prompt = synth.make_tokens(shape.vocab, 16, 1001)
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        _, ids = m.prefill([0], [prompt])
        first = int(ids[0])
        ref = m.decode_steps([0], [first], [16], 8).cpu().numpy()
        m.test_raise_guard(4)
        with pytest.raises(q2.Qwen2Error) as e:
            m.synchronize()
        assert e.value.code == q2.QWEN2_E_DEVICE_GUARD
        assert "bounded wait timed out" in str(e.value)
        m.synchronize()
        again = m.decode_steps([0], [first], [16], 8).cpu().numpy()
        m.synchronize()
        with pytest.raises(q2.Qwen2Error) as e:
            m.test_raise_guard(0)
        assert e.value.code == q2.QWEN2_E_ARG
    np.testing.assert_array_equal(again, ref)


def test_a_bounded_wait_that_runs_out_is_reported_and_decoding_recovers(q2):
    """Failure detection without a GPU fault: the test hook makes one
    persistent decode launch wait on an arrival counter that no CTA arrives
    at, with a 1 ms limit on its bounded waits.  The wait runs out, every
    CTA stops (the feeding lane waits for its copies in flight), the launch
    raises the guard word; synchronize reports QWEN2_E_DEVICE_GUARD once,
    resets the exchange state, and the same decode then gives the ids of an
    undisturbed run."""
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    prompt = synth.make_tokens(shape.vocab, 16, 1001)
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        assert m.features & q2.FEATURE_PERSISTENT_DECODE
        _, ids = m.prefill([0], [prompt])
        first = int(ids[0])
        ref = m.decode_steps([0], [first], [16], 8).cpu().numpy()
        m.synchronize()
        for _ in range(2):
            m.test_stall_decode(1000)
            m.decode_steps([0], [first], [16], 1)
            with pytest.raises(q2.Qwen2Error) as e:
                m.synchronize()
            assert e.value.code == q2.QWEN2_E_DEVICE_GUARD
            assert "bounded wait timed out" in str(e.value)
            m.synchronize()
            again = m.decode_steps([0], [first], [16], 8).cpu().numpy()
            m.synchronize()
            np.testing.assert_array_equal(again, ref)
        with pytest.raises(q2.Qwen2Error) as e:
            m.test_stall_decode(10)
        assert e.value.code == q2.QWEN2_E_ARG
    for kw in ({"flags": q2.FLAG_NO_MEGAKERNEL}, {"weight_format": q2.WEIGHTS_Q8_0}):
        with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16, **kw) as m:
            with pytest.raises(q2.Qwen2Error) as e:
                m.test_stall_decode(1000)
            assert e.value.code == q2.QWEN2_E_UNSUPPORTED


def test_oversized_kv_cache_is_an_allocation_error(q2):
    """A KV cache larger than the device (65,536 sequences x 32,768
    positions of the toy model: 4 TB) is QWEN2_E_OOM from create, and the
    device stays usable."""
    shape = synth.SHAPES["toy"]
    w = synth.make_weights(shape, 0)
    with pytest.raises(q2.Qwen2Error) as e:
        q2.Qwen2Model(shape, w, n_ctx=32768, max_seqs=65536, max_tokens=16)
    assert e.value.code == q2.QWEN2_E_OOM
    with q2.Qwen2Model(shape, w, n_ctx=64, max_seqs=1, max_tokens=16) as m:
        m.prefill([0], [synth.make_tokens(shape.vocab, 8, 3)])
        m.synchronize()
