"""The C ABI library without a GPU: it loads, exports every symbol the
header declares, validates configs before touching the device, and its Q8_0
packer matches the oracle's quantiser byte for byte."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth
from conftest import ROOT

q2 = pytest.importorskip("qwen2_decoder_forward_gb300")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(q2.LIB_PATH):
        from qwen2_decoder_forward_gb300 import build
        build.build()
    return q2.lib()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "qwen2.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(qwen2_[a-z0-9_]+)\s*\(", src))


def test_every_declared_symbol_is_exported(L):
    syms = header_symbols()
    assert syms == set(q2.EXPORTS)
    for s in syms:
        assert hasattr(L, s), s


def test_kv_bytes_per_position_matches_page_figure(L):
    s = synth.SHAPES["qwen2.5-0.5b"]
    assert q2.kv_bytes_per_seq(s, 1) == 24 * 1024
    assert q2.kv_bytes_per_seq(s, 4096) == 96 * 2**20


def _create(L, **over):
    s = synth.SHAPES["toy"]
    cfg = q2._Config(s.n_layer, s.hidden, s.n_head, s.n_kv_head, s.head_dim, s.intermediate, s.vocab,
                     s.rms_eps, s.rope_theta, 0, 0, 64, 1, 16, 0)
    for k, v in over.items():
        setattr(cfg, k, v)
    dummy = np.zeros(16, dtype=np.float32)
    layers = (q2._LayerWeights * max(cfg.n_layer, 1))()
    for i in range(len(layers)):
        for f, _ in q2._LayerWeights._fields_:
            setattr(layers[i], f, dummy.ctypes.data)
    w = q2._Weights(dummy.ctypes.data, None, dummy.ctypes.data, layers)
    h = ctypes.c_void_p()
    rc = L.qwen2_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
    return rc, L.qwen2_last_error(None).decode(), h


@pytest.mark.parametrize("over,code", [
    ({"head_dim": 96, "hidden": 384}, q2.QWEN2_E_UNSUPPORTED),
    ({"head_dim": 128, "hidden": 512, "prefill_mode": 1}, q2.QWEN2_E_UNSUPPORTED),
    ({"hidden": 320}, q2.QWEN2_E_UNSUPPORTED),
    ({"intermediate": 1000}, q2.QWEN2_E_UNSUPPORTED),
    ({"n_kv_head": 3}, q2.QWEN2_E_UNSUPPORTED),
    ({"prefill_mode": 2}, q2.QWEN2_E_UNSUPPORTED),           # Q8_0 activations need Q8_0 weights
    ({"prefill_mode": 2, "weight_format": 2}, q2.QWEN2_E_UNSUPPORTED),
    ({"n_ctx": 0}, q2.QWEN2_E_ARG),
    ({"vocab": 1}, q2.QWEN2_E_ARG),
])
def test_create_rejects_bad_configs_without_a_device(L, over, code):
    rc, msg, h = _create(L, **over)
    assert rc == code and msg
    assert not h.value


def test_null_arguments_are_rejected(L):
    h = ctypes.c_void_p()
    assert L.qwen2_create(None, None, ctypes.byref(h)) == q2.QWEN2_E_ARG
    assert L.qwen2_create(None, None, None) == q2.QWEN2_E_ARG
    # The debug checks of a context refuse a null context on the host.
    assert L.qwen2_check_canaries(None) == q2.QWEN2_E_ARG


def test_q8_0_packer_matches_oracle_bytes(L):
    rng = np.random.default_rng(0)
    w = (0.02 * rng.standard_normal((96, 256))).astype(np.float16)
    w[3, :32] = 0                       # an all-zero block
    w[5, 40] = np.float16(-1.5)         # a block dominated by one value
    w[7, 64:96] = np.float16(0.25)      # a constant block
    q_lib, d_lib = q2.quantize_q8_0(w)
    q_orc, d_orc = oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(q_lib, q_orc)
    np.testing.assert_array_equal(d_lib.view(np.uint16), d_orc.view(np.uint16))


def test_q8_0_packer_rounds_half_away_like_the_oracle(L):
    """Half cases decided by the rounding rule alone (a block whose largest
    magnitude is 127 has d = 1): the packer and the oracle both round half
    away from zero."""
    w = np.zeros((2, 64), dtype=np.float16)
    w[0, :7] = [127.0, 0.5, -0.5, 1.5, -1.5, 2.5, -2.5]
    w[1, 32:39] = [-127.0, 126.5, -126.5, 3.5, -3.5, 4.5, -4.5]
    q_lib, d_lib = q2.quantize_q8_0(w)
    q_orc, d_orc = oracle.quantize_q8_0(w)
    np.testing.assert_array_equal(q_lib[0, :7], [127, 1, -1, 2, -2, 3, -3])
    np.testing.assert_array_equal(q_lib[1, 32:39], [-127, 127, -127, 4, -4, 5, -5])
    np.testing.assert_array_equal(q_lib, q_orc)
    np.testing.assert_array_equal(d_lib.view(np.uint16), d_orc.view(np.uint16))


def test_q4_0_packer_matches_oracle_bytes(L):
    """The library's Q4_0 packer and the oracle's quantiser give the same
    nibbles and scales (reading of the unnamed format: blocks of 32 along K,
    d = max|x| / 7, codes round-half-away(x / d) + 8, element 2j in the low
    nibble of byte j)."""
    rng = np.random.default_rng(4)
    w = (0.02 * rng.standard_normal((64, 256))).astype(np.float16)
    w[3, :32] = 0                                   # an all-zero block
    w[5, 40] = np.float16(-1.5)                     # one dominant value
    w[7, 64:96] = np.float16(0.25)                  # a constant block
    w[9, :6] = [7.0, 0.5, -0.5, 2.5, -2.5, 6.5]     # d = 1: half cases
    p_lib, d_lib = q2.quantize_q4_0(w)
    p_orc, d_orc = oracle.quantize_q4_0(w)
    np.testing.assert_array_equal(p_lib, p_orc)
    np.testing.assert_array_equal(d_lib.view(np.uint16), d_orc.view(np.uint16))
    np.testing.assert_array_equal(oracle.unpack_nibbles(p_lib)[9, :6], [15, 9, 7, 11, 5, 15])


def test_q8_0_packer_rejects_ragged_k(L):
    w = np.zeros((2, 48), dtype=np.float16)
    q = np.empty((2, 48), dtype=np.int8)
    d = np.empty((2, 2), dtype=np.uint16)
    assert L.qwen2_quantize_q8_0(w.ctypes.data, 2, 48, q.ctypes.data, d.ctypes.data) == q2.QWEN2_E_ARG


def test_no_alloc_head_rejects_bad_sizes_before_any_cuda_call(L):
    # Non-null dummy pointers: argument checks come before any CUDA call.
    fake = ctypes.c_void_p(16)
    assert L.qwen2_lm_head_argmax_noalloc(fake, fake, 9, 896, 151936, None, fake, None) == 1
    assert b"n_rows" in L.qwen2_last_error(None)
    assert L.qwen2_lm_head_argmax_noalloc(fake, fake, 1, 1032, 151936, None, fake, None) == 1
    assert b"hidden_size" in L.qwen2_last_error(None)
    assert L.qwen2_lm_head_argmax_noalloc(fake, fake, 1, 896, 151936, None, None, None) == 1
    # A 2-byte-aligned embedding (a pool sub-allocation) is refused on the
    # host: the rows are read with 16-byte vector loads.
    assert L.qwen2_lm_head_argmax_noalloc(ctypes.c_void_p(16 + 2), fake, 1, 896, 151936, None, fake, None) == 1
    assert b"16-byte" in L.qwen2_last_error(None)


def test_untied_shape_without_a_head_matrix_is_rejected_before_any_device_work():
    """A shape that declares an untied LM head must bring the head matrix;
    the binding refuses it before any library call otherwise."""
    shape = synth.SHAPES["toy-untied"]
    w = dict(synth.make_weights(shape, 0))
    del w["lm_head"]
    with pytest.raises(q2.Qwen2Error) as e:
        q2.Qwen2Model(shape, w, n_ctx=32)
    assert e.value.code == q2.QWEN2_E_ARG


def test_weights_struct_carries_the_lm_head_between_embed_and_final_norm():
    names = [f for f, _ in q2._Weights._fields_]
    assert names == ["embed", "lm_head", "final_norm", "layers"]


def test_stop_id_constants_match_the_pages():
    from conftest import read_golden
    g = read_golden("qwen2_0p5b_pages.txt")
    assert q2.ENDOFTEXT_ID == int(g["endoftext_id"])
    assert q2.IM_END_ID == int(g["im_end_id"])
    assert max(q2.ENDOFTEXT_ID, q2.IM_END_ID) < synth.SHAPES["qwen2.5-0.5b"].vocab
