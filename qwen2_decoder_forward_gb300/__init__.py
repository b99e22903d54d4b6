"""Python binding of libqwen2, the GB300 (sm_103a) Qwen2 decoder forward.

Argument marshalling only: every step of the forward runs in the CUDA
kernels of ``libqwen2.so`` behind the C ABI of ``include/qwen2.h``.  There
is no CPU fallback; if the library is missing or fails to load, every call
raises.  PyTorch supplies device memory (output tensors) and streams.

    import qwen2_decoder_forward_gb300 as q2
    m = q2.Qwen2Model(shape, weights, n_ctx=4096, max_seqs=1, max_tokens=128)
    logits, ids = m.prefill([0], [prompt], n_out=1)
    ids = m.decode_steps([0], [int(ids[0])], [len(prompt)], n_steps=256)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqwen2.so")

QWEN2_OK = 0
QWEN2_E_ARG = 1
QWEN2_E_POS = 2
QWEN2_E_UNSUPPORTED = 3
QWEN2_E_OOM = 4
QWEN2_E_CUDA = 5
QWEN2_E_DEVICE_GUARD = 6

# Stop ids of the Qwen2 / Qwen2.5 tokenizers for generate(): base
# checkpoints end generation on <|endoftext|>, instruct checkpoints on
# <|im_end|> (nnterp encyclopedia qwen2, "The chat template writes a system
# turn"; minfer "Qwen2 / Qwen2.5 Architecture Support", section 5).
ENDOFTEXT_ID = 151643
IM_END_ID = 151645

WEIGHTS_F16 = 0
WEIGHTS_Q8_0 = 1
WEIGHTS_Q4_0 = 2
PREFILL_F32 = 0
PREFILL_TENSOR = 1
PREFILL_Q8_ACT = 2

FLAG_NO_FUSE_QKV = 0x1
FLAG_NO_FUSE_FFN = 0x2
FLAG_NO_GRAPH = 0x4
FLAG_NO_MEGAKERNEL = 0x8
FLAG_PROFILE = 0x10
FEATURE_PERSISTENT_DECODE = 0x1
FEATURE_TENSOR_PREFILL = 0x2

# Every symbol include/qwen2.h declares.
EXPORTS = (
    "qwen2_create", "qwen2_destroy", "qwen2_last_error", "qwen2_kv_cache",
    "qwen2_prefill", "qwen2_decode_step", "qwen2_decode_steps", "qwen2_decode_steps_stop",
    "qwen2_final_hidden", "qwen2_synchronize", "qwen2_weight_bytes",
    "qwen2_kv_bytes_per_seq", "qwen2_quantize_q8_0", "qwen2_quantize_q4_0", "qwen2_features", "qwen2_profile_marks",
    "qwen2_lm_head_argmax_noalloc", "qwen2_test_raise_guard", "qwen2_test_stall_decode",
    "qwen2_check_canaries",
)


class Qwen2Error(RuntimeError):
    """A libqwen2 call returned an error code."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"libqwen2 error {code}: {msg}")
        self.code = code


class _Config(ctypes.Structure):
    _fields_ = [
        ("n_layer", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_head", ctypes.c_int32),
        ("n_kv_head", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
        ("weight_format", ctypes.c_int32), ("prefill_mode", ctypes.c_int32), ("n_ctx", ctypes.c_int32),
        ("max_seqs", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32),
    ]


_P = ctypes.c_void_p


class _LayerWeights(ctypes.Structure):
    _fields_ = [(k, _P) for k in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "bq", "bk", "bv",
                                  "attn_norm", "ffn_norm")]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", _P), ("lm_head", _P), ("final_norm", _P), ("layers", ctypes.POINTER(_LayerWeights))]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libqwen2.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m qwen2_decoder_forward_gb300.build` (no CPU fallback exists)")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    pi32 = ctypes.POINTER(ctypes.c_int32)
    L.qwen2_create.argtypes = [ctypes.POINTER(_Config), ctypes.POINTER(_Weights), ctypes.POINTER(_P)]
    L.qwen2_create.restype = ctypes.c_int
    L.qwen2_destroy.argtypes = [_P]
    L.qwen2_destroy.restype = None
    L.qwen2_last_error.argtypes = [_P]
    L.qwen2_last_error.restype = ctypes.c_char_p
    L.qwen2_kv_cache.argtypes = [_P, ctypes.POINTER(_P), ctypes.POINTER(i64)]
    L.qwen2_kv_cache.restype = ctypes.c_int
    L.qwen2_prefill.argtypes = [_P, i32, pi32, pi32, pi32, pi32, i32, _P, _P, _P]
    L.qwen2_prefill.restype = ctypes.c_int
    L.qwen2_decode_step.argtypes = [_P, i32, pi32, pi32, pi32, _P, _P, _P]
    L.qwen2_decode_step.restype = ctypes.c_int
    L.qwen2_decode_steps.argtypes = [_P, i32, pi32, pi32, pi32, i32, _P, _P]
    L.qwen2_decode_steps.restype = ctypes.c_int
    L.qwen2_decode_steps_stop.argtypes = [_P, i32, pi32, pi32, pi32, i32, pi32, i32, _P, _P, _P]
    L.qwen2_decode_steps_stop.restype = ctypes.c_int
    L.qwen2_test_raise_guard.argtypes = [_P, i32, _P]
    L.qwen2_test_raise_guard.restype = ctypes.c_int
    L.qwen2_test_stall_decode.argtypes = [_P, i32]
    L.qwen2_test_stall_decode.restype = ctypes.c_int
    L.qwen2_check_canaries.argtypes = [_P]
    L.qwen2_check_canaries.restype = ctypes.c_int
    L.qwen2_final_hidden.argtypes = [_P, _P, i32, _P]
    L.qwen2_final_hidden.restype = ctypes.c_int
    L.qwen2_synchronize.argtypes = [_P, _P]
    L.qwen2_synchronize.restype = ctypes.c_int
    L.qwen2_weight_bytes.argtypes = [_P]
    L.qwen2_weight_bytes.restype = i64
    L.qwen2_kv_bytes_per_seq.argtypes = [ctypes.POINTER(_Config)]
    L.qwen2_kv_bytes_per_seq.restype = i64
    L.qwen2_quantize_q8_0.argtypes = [_P, i64, i64, _P, _P]
    L.qwen2_quantize_q8_0.restype = ctypes.c_int
    L.qwen2_quantize_q4_0.argtypes = [_P, i64, i64, _P, _P]
    L.qwen2_quantize_q4_0.restype = ctypes.c_int
    L.qwen2_features.argtypes = [_P]
    L.qwen2_features.restype = ctypes.c_uint32
    L.qwen2_profile_marks.argtypes = [_P, _P, i64, pi32, pi32]
    L.qwen2_profile_marks.restype = ctypes.c_int
    L.qwen2_lm_head_argmax_noalloc.argtypes = [_P, _P, i32, i32, i32, _P, _P, _P]
    L.qwen2_lm_head_argmax_noalloc.restype = ctypes.c_int
    _lib = L
    return L


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def quantize_q8_0(w: np.ndarray):
    """Q8_0-quantise an f16 matrix [rows, K] with the library's packer
    (host code; needs no GPU).  Returns (q int8 [rows, K], d f16 [rows, K/32])."""
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float16))
    rows, k = w.shape
    q = np.empty((rows, k), dtype=np.int8)
    d = np.empty((rows, k // 32), dtype=np.uint16)
    rc = lib().qwen2_quantize_q8_0(w.ctypes.data, rows, k, q.ctypes.data, d.ctypes.data)
    if rc:
        raise Qwen2Error(rc, "qwen2_quantize_q8_0 rejected its arguments")
    return q, d.view(np.float16)


def quantize_q4_0(w: np.ndarray):
    """Q4_0-quantise an f16 matrix [rows, K] with the library's packer
    (host code; needs no GPU).  Returns (packed uint8 [rows, K/2], element
    2j in the low nibble of byte j; d f16 [rows, K/32])."""
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float16))
    rows, k = w.shape
    packed = np.empty((rows, k // 2), dtype=np.uint8)
    d = np.empty((rows, k // 32), dtype=np.uint16)
    rc = lib().qwen2_quantize_q4_0(w.ctypes.data, rows, k, packed.ctypes.data, d.ctypes.data)
    if rc:
        raise Qwen2Error(rc, "qwen2_quantize_q4_0 rejected its arguments")
    return packed, d.view(np.float16)


def lm_head_argmax_noalloc(embed, hidden, logits=None, ids=None, want_logits: bool = True, stream=None):
    """Tied LM head + greedy argmax on normalised rows through
    qwen2_lm_head_argmax_noalloc (no context, no device allocation by the
    library).  embed: CUDA f16 [V, H]; hidden: CUDA f32 [rows, H].  Output
    tensors are allocated here by torch unless passed in.  Returns
    (logits f32 [rows, V] or None, ids int32 [rows])."""
    import torch
    if embed.dtype != torch.float16 or hidden.dtype != torch.float32 or not (embed.is_cuda and hidden.is_cuda):
        raise ValueError("embed must be CUDA f16 and hidden CUDA f32")
    rows, h = hidden.shape
    v = embed.shape[0]
    if embed.shape[1] != h:
        raise ValueError("embed and hidden disagree on the hidden size")
    if want_logits and logits is None:
        logits = torch.empty((rows, v), dtype=torch.float32, device=hidden.device)
    if ids is None:
        ids = torch.empty((rows,), dtype=torch.int32, device=hidden.device)
    rc = lib().qwen2_lm_head_argmax_noalloc(_data_ptr(embed), _data_ptr(hidden), rows, h, v,
                                            _data_ptr(logits if want_logits else None), _data_ptr(ids),
                                            _stream_ptr(stream))
    if rc:
        raise Qwen2Error(rc, lib().qwen2_last_error(None).decode())
    return (logits if want_logits else None), ids


def kv_bytes_per_seq(shape, n_ctx: int) -> int:
    c = _Config(n_layer=shape.n_layer, n_kv_head=shape.n_kv_head, head_dim=shape.head_dim, n_ctx=n_ctx)
    return int(lib().qwen2_kv_bytes_per_seq(ctypes.byref(c)))


class _CudaArray:
    """Exposes a raw device pointer to torch through __cuda_array_interface__."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(int(s) for s in shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


class Qwen2Model:
    """One libqwen2 context on the current CUDA device.

    ``shape`` has the fields of ``synth.ModelShape``; ``weights`` is
    ``{"embed": f16 [V, H], "final_norm": f32 [H], "layers": [ {wq, wk, wv,
    wo, wg, wu, wd (f16, [out, in]), bq, bk, bv, attn_norm, ffn_norm (f32)} ]}``.
    """

    def __init__(self, shape, weights: dict, n_ctx: int, max_seqs: int = 1, max_tokens: int = 128,
                 weight_format: int = WEIGHTS_F16, prefill_mode: int = PREFILL_F32, flags: int = 0):
        # A separate LM head (untied, 7B and up) is passed as its own
        # matrix; a shape that declares an untied head must bring one.
        if weights.get("lm_head") is None and not getattr(shape, "tie_embeddings", True):
            raise Qwen2Error(QWEN2_E_ARG, "the shape declares an untied LM head but the weights have no lm_head")
        L = lib()
        self.shape = shape
        self.n_ctx, self.max_seqs, self.max_tokens = n_ctx, max_seqs, max_tokens
        self.vocab, self.hidden = shape.vocab, shape.hidden
        self._cfg = _Config(shape.n_layer, shape.hidden, shape.n_head, shape.n_kv_head, shape.head_dim,
                            shape.intermediate, shape.vocab, float(shape.rms_eps), float(shape.rope_theta),
                            weight_format, prefill_mode, n_ctx, max_seqs, max_tokens, flags)
        keep = []

        def p(a, dt):
            a = np.ascontiguousarray(np.asarray(a, dtype=dt))
            keep.append(a)
            return a.ctypes.data

        layers = (_LayerWeights * shape.n_layer)()
        for i, lw in enumerate(weights["layers"]):
            for k in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
                setattr(layers[i], k, p(lw[k], np.float16))
            for k in ("bq", "bk", "bv", "attn_norm", "ffn_norm"):
                setattr(layers[i], k, p(lw[k], np.float32))
        head = weights.get("lm_head")
        w = _Weights(p(weights["embed"], np.float16), p(head, np.float16) if head is not None else None,
                     p(weights["final_norm"], np.float32), layers)
        h = _P()
        rc = L.qwen2_create(ctypes.byref(self._cfg), ctypes.byref(w), ctypes.byref(h))
        if rc:
            raise Qwen2Error(rc, L.qwen2_last_error(None).decode())
        self._h = h
        del keep

    # -- helpers ------------------------------------------------------------
    def _check(self, rc: int):
        if rc:
            raise Qwen2Error(rc, lib().qwen2_last_error(self._h).decode())

    def close(self):
        if getattr(self, "_h", None):
            lib().qwen2_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def weight_bytes(self) -> int:
        return int(lib().qwen2_weight_bytes(self._h))

    @property
    def features(self) -> int:
        """QWEN2_FEATURE_* bits: which kernels this context runs."""
        return int(lib().qwen2_features(self._h))

    def profile_marks(self) -> np.ndarray:
        """Per-phase timestamps (ns) of the last persistent decode launch,
        [n_cta, n_marks] (context created with FLAG_PROFILE)."""
        n_cta, n_marks = ctypes.c_int32(), ctypes.c_int32()
        cap = 4096 * 256
        buf = np.zeros(cap, dtype=np.int64)
        self._check(lib().qwen2_profile_marks(self._h, buf.ctypes.data, cap, ctypes.byref(n_cta),
                                              ctypes.byref(n_marks)))
        return buf[:n_cta.value * n_marks.value].reshape(n_cta.value, n_marks.value)

    # -- the entry points ----------------------------------------------------
    def prefill(self, seq_ids, tokens, positions=None, n_out: int = 1, want_logits: bool = True,
                logits_out=None, ids_out=None, stream=None):
        """Prefill the token lists of ``seq_ids``; ``positions`` default to
        0..n-1 per sequence.  Returns ``(logits [n_seq*n_out, V] | None,
        ids [n_seq*n_out])`` as CUDA tensors unless outputs are given."""
        import torch
        seq_ids = _i32(seq_ids)
        toks = [_i32(t) for t in tokens]
        if positions is None:
            positions = [np.arange(len(t), dtype=np.int32) for t in toks]
        poss = [_i32(p) for p in positions]
        n_tok = _i32([len(t) for t in toks])
        flat_t = _i32(np.concatenate(toks))
        flat_p = _i32(np.concatenate(poss))
        rows = len(seq_ids) * n_out
        if want_logits and logits_out is None:
            logits_out = torch.empty((rows, self.vocab), dtype=torch.float32, device="cuda")
        if ids_out is None:
            ids_out = torch.empty((rows,), dtype=torch.int32, device="cuda")
        self._check(lib().qwen2_prefill(
            self._h, len(seq_ids), _ptr_i32(seq_ids), _ptr_i32(n_tok), _ptr_i32(flat_t), _ptr_i32(flat_p),
            n_out, _data_ptr(logits_out) if want_logits else None, _data_ptr(ids_out), _stream_ptr(stream)))
        return (logits_out if want_logits else None), ids_out

    def decode_step(self, seq_ids, tokens, positions, want_logits: bool = True, logits_out=None,
                    ids_out=None, stream=None):
        """One decode row per sequence; returns ``(logits | None, ids)``."""
        import torch
        seq_ids, tokens, positions = _i32(seq_ids), _i32(tokens), _i32(positions)
        n = len(seq_ids)
        if want_logits and logits_out is None:
            logits_out = torch.empty((n, self.vocab), dtype=torch.float32, device="cuda")
        if ids_out is None:
            ids_out = torch.empty((n,), dtype=torch.int32, device="cuda")
        self._check(lib().qwen2_decode_step(
            self._h, n, _ptr_i32(seq_ids), _ptr_i32(tokens), _ptr_i32(positions),
            _data_ptr(logits_out) if want_logits else None, _data_ptr(ids_out), _stream_ptr(stream)))
        return (logits_out if want_logits else None), ids_out

    def decode_steps(self, seq_ids, first_tokens, start_positions, n_steps: int, ids_out=None, stream=None):
        """Greedy decode ``n_steps`` steps on the device; returns ids
        [n_steps, n_seq] (a CUDA tensor unless ``ids_out`` is given)."""
        import torch
        seq_ids, first_tokens, start_positions = _i32(seq_ids), _i32(first_tokens), _i32(start_positions)
        n = len(seq_ids)
        if ids_out is None:
            ids_out = torch.empty((n_steps, n), dtype=torch.int32, device="cuda")
        self._check(lib().qwen2_decode_steps(
            self._h, n, _ptr_i32(seq_ids), _ptr_i32(first_tokens), _ptr_i32(start_positions), n_steps,
            _data_ptr(ids_out), _stream_ptr(stream)))
        return ids_out

    def generate(self, seq_ids, first_tokens, start_positions, max_steps: int, stop_ids, ids_out=None,
                 n_generated_out=None, stream=None):
        """Greedy decode of up to ``max_steps`` tokens per sequence that ends
        at the first generated id in ``stop_ids`` (at most 8): returns
        (ids [max_steps, n_seq] with -1 after each sequence's stop id,
        n_generated [n_seq] counting the stop id), CUDA tensors unless the
        outputs are given."""
        import torch
        seq_ids, first_tokens, start_positions = _i32(seq_ids), _i32(first_tokens), _i32(start_positions)
        stops = _i32(stop_ids)
        n = len(seq_ids)
        if ids_out is None:
            ids_out = torch.empty((max_steps, n), dtype=torch.int32, device="cuda")
        if n_generated_out is None:
            n_generated_out = torch.empty((n,), dtype=torch.int32, device="cuda")
        self._check(lib().qwen2_decode_steps_stop(
            self._h, n, _ptr_i32(seq_ids), _ptr_i32(first_tokens), _ptr_i32(start_positions), max_steps,
            _ptr_i32(stops), len(stops), _data_ptr(ids_out), _data_ptr(n_generated_out), _stream_ptr(stream)))
        return ids_out, n_generated_out

    def final_hidden(self, rows: int, stream=None):
        """final_norm_output rows of the last call, [rows, H] CUDA tensor."""
        import torch
        out = torch.empty((rows, self.hidden), dtype=torch.float32, device="cuda")
        self._check(lib().qwen2_final_hidden(self._h, _data_ptr(out), rows, _stream_ptr(stream)))
        return out

    def kv_cache(self):
        """The KV cache as a CUDA tensor sharing the library's memory:
        [max_seqs, n_layer, 2, n_kv_head, n_ctx, head_dim] f32."""
        import torch
        base = _P()
        dims = (ctypes.c_int64 * 6)()
        self._check(lib().qwen2_kv_cache(self._h, ctypes.byref(base), dims))
        return torch.as_tensor(_CudaArray(base.value, list(dims), "<f4"), device="cuda")

    def test_raise_guard(self, code: int, stream=None):
        """Test hook: write ``code`` into the device guard word (as a kernel's
        bounded wait does when it gives up); the next synchronize reports it."""
        self._check(lib().qwen2_test_raise_guard(self._h, code, _stream_ptr(stream)))

    def test_stall_decode(self, wait_us: int = 1000):
        """Test hook: the next persistent decode launch waits on a counter
        nothing arrives at, with its bounded waits limited to wait_us; the
        next synchronize reports the timeout."""
        self._check(lib().qwen2_test_stall_decode(self._h, int(wait_us)))

    def synchronize(self, stream=None):
        self._check(lib().qwen2_synchronize(self._h, _stream_ptr(stream)))

    def check_canaries(self):
        """Debug check: raises Qwen2Error (QWEN2_E_DEVICE_GUARD) if a kernel
        wrote into the guard words around any of the context's device
        buffers."""
        self._check(lib().qwen2_check_canaries(self._h))


def _data_ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        if not t.flags["C_CONTIGUOUS"]:
            raise ValueError("output arrays must be contiguous")
        return ctypes.c_void_p(t.ctypes.data)
    if not t.is_contiguous():
        raise ValueError("output tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())
