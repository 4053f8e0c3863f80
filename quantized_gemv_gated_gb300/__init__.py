"""Python binding of libqg.so, the C ABI declared in include/qg.h.

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  Functions carry the C names (qg_gemv_q4k, qg_decode_token, ...)
and take device pointers as ints (torch `data_ptr()`) or torch tensors, host
buffers as numpy arrays, streams as ints or torch streams.  There is no CPU
fallback: if the library cannot be built or loaded, import fails.
"""
import ctypes
import os

import numpy as np

from . import _build

QG_OK = 0
QG_ERR_SHAPE, QG_ERR_QTYPE, QG_ERR_EMPTY, QG_ERR_POS, QG_ERR_TOKEN = -1, -2, -3, -4, -5
QG_ERR_LAYER_KIND, QG_ERR_CUDA, QG_ERR_TIMEOUT, QG_ERR_ARG, QG_ERR_OOM = -6, -7, -8, -9, -10
QG_QTYPE_Q4_K, QG_QTYPE_Q6_K = 12, 14
QG_LAYER_DELTANET, QG_LAYER_ATTENTION = 0, 1

ERROR_NAMES = {0: "QG_OK", -1: "QG_ERR_SHAPE", -2: "QG_ERR_QTYPE", -3: "QG_ERR_EMPTY", -4: "QG_ERR_POS",
               -5: "QG_ERR_TOKEN", -6: "QG_ERR_LAYER_KIND", -7: "QG_ERR_CUDA", -8: "QG_ERR_TIMEOUT",
               -9: "QG_ERR_ARG", -10: "QG_ERR_OOM"}

# Symbols exported by the library (every function declared in include/qg.h).
EXPORTS = [
    "qg_model_create", "qg_model_destroy", "qg_state_create", "qg_state_destroy", "qg_state_reset",
    "qg_state_upload_layer", "qg_state_upload_kv", "qg_state_download_layer", "qg_state_download_hidden",
    "qg_state_kv_len", "qg_state_stream", "qg_state_stats", "qg_state_set_token_mask",
    "qg_gemv_q4k", "qg_gemv_q6k", "qg_gemv_q6k_planar", "qg_q6k_planar_bytes", "qg_q4k_planar_bytes", "qg_q4k_to_planar",
    "qg_gemv_q4k_planar",
    "qg_q6k_to_planar", "qg_lmhead_argmax_workspace_bytes", "qg_lmhead_argmax", "qg_lmhead_argmax_noalloc",
    "qg_argmax_f32",
    "qg_deltanet_step", "qg_attn_decode_step", "qg_decode_token", "qg_decode_token_eager",
    "qg_decode_greedy", "qg_device_status", "qg_last_error",
    "qg_state_create_kv", "qg_state_kv_format", "qg_state_download_kv_records", "qg_prefill",
    "qg_decode_batch", "qg_batch_create", "qg_batch_step", "qg_batch_destroy", "qg_bench_kernel",
]


# kernel kinds of the decode step (qg_bench_kernel)
KERNEL_DN_IN, KERNEL_DELTA, KERNEL_SSM_OUT, KERNEL_ATTN_IN, KERNEL_ATTN, KERNEL_ATTN_OUT = 0, 1, 2, 3, 4, 5
KERNEL_FFN_UP, KERNEL_FFN_DOWN, KERNEL_LMHEAD = 6, 7, 8
KERNEL_NAMES = {0: "dn_in", 1: "delta", 2: "ssm_out", 3: "attn_in", 4: "attn", 5: "attn_out", 6: "ffn_up",
                7: "ffn_down", 8: "lmhead"}
KV_F32, KV_Q8_0_Q5_1 = 0, 1  # qg_state_create_kv
K_RECORD_BYTES, V_RECORD_BYTES = 272, 192  # per (kv head, position) of a quantized cache


class QgError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class QgConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "ffn", "vocab", "n_k_heads", "n_v_heads", "head_k_dim", "head_v_dim",
        "conv_kernel", "n_heads", "n_kv_heads", "head_dim", "n_rot")] + [
        ("eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("layer_kinds", ctypes.POINTER(ctypes.c_int32))]


class QgQTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("qtype", ctypes.c_int32), ("n", ctypes.c_int32),
                ("k", ctypes.c_int32)]


_F = ctypes.c_void_p


class QgLayerWeights(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("attn_norm", _F), ("post_attention_norm", _F),
                ("ffn_gate", QgQTensor), ("ffn_up", QgQTensor), ("ffn_down", QgQTensor),
                ("ssm_conv1d", _F), ("ssm_a_log", _F), ("ssm_dt_bias", _F), ("ssm_norm", _F),
                ("attn_qkv", QgQTensor), ("ssm_alpha", QgQTensor), ("ssm_beta", QgQTensor),
                ("attn_gate", QgQTensor), ("ssm_out", QgQTensor),
                ("attn_q_norm", _F), ("attn_k_norm", _F),
                ("attn_q", QgQTensor), ("attn_k", QgQTensor), ("attn_v", QgQTensor),
                ("attn_output", QgQTensor)]


class QgHostWeights(ctypes.Structure):
    _fields_ = [("token_embd", _F), ("output_norm", _F), ("lm_head", QgQTensor),
                ("layers", ctypes.POINTER(QgLayerWeights))]


class QgStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "device_allocs", "h2d_bytes", "d2h_bytes", "graph_launches", "graph_captures",
        "graph_kernel_nodes", "steps")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lib = None


def lib():
    """The loaded libqg.so (built in-tree on first use)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i, p, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        sigs = {
            "qg_model_create": [ctypes.POINTER(QgConfig), ctypes.POINTER(QgHostWeights), i, ctypes.POINTER(p)],
            "qg_model_destroy": [p],
            "qg_state_create": [p, i, ctypes.POINTER(p)],
            "qg_state_create_kv": [p, i, i, ctypes.POINTER(p)],
            "qg_prefill": [p, p, p, i, i, ctypes.POINTER(ctypes.c_uint32)],
            "qg_decode_batch": [p, p, i, p, p, p],
            "qg_batch_create": [p, p, i, ctypes.POINTER(p)],
            "qg_batch_step": [p, p, p, p],
            "qg_batch_destroy": [p],
            "qg_state_kv_format": [p, ctypes.POINTER(i)],
            "qg_state_download_kv_records": [p, i, p, p, ctypes.POINTER(sz), ctypes.POINTER(sz)],
            "qg_state_destroy": [p],
            "qg_state_reset": [p],
            "qg_state_upload_layer": [p, i, p, p],
            "qg_state_upload_kv": [p, i, p, p, i],
            "qg_state_download_layer": [p, i, p, p, ctypes.POINTER(sz)],
            "qg_state_download_hidden": [p, p],
            "qg_state_kv_len": [p, ctypes.POINTER(i)],
            "qg_state_stream": [p, ctypes.POINTER(p)],
            "qg_state_stats": [p, ctypes.POINTER(QgStats)],
            "qg_state_set_token_mask": [p, p, i],
            "qg_gemv_q4k": [p, p, p, i, i, p],
            "qg_gemv_q6k": [p, p, p, i, i, p],
            "qg_gemv_q6k_planar": [p, p, p, i, i, p],
            "qg_q6k_to_planar": [p, p, i, i, p],
            "qg_q4k_to_planar": [p, p, i, i, p],
            "qg_gemv_q4k_planar": [p, p, p, i, i, p],
            "qg_lmhead_argmax": [p, p, i, i, p, p, p],
            "qg_lmhead_argmax_noalloc": [p, p, i, i, p, p],
            "qg_argmax_f32": [p, i, p, p],
            "qg_deltanet_step": [p, p, i, p, p],
            "qg_attn_decode_step": [p, p, i, p, i, p],
            "qg_bench_kernel": [p, p, i, i, p],
            "qg_decode_token": [p, p, ctypes.c_uint32, i, ctypes.POINTER(ctypes.c_uint32)],
            "qg_decode_token_eager": [p, p, ctypes.c_uint32, i, ctypes.POINTER(ctypes.c_uint32)],
            "qg_decode_greedy": [p, p, i, i, p],
            "qg_device_status": [],
        }
        for name, args in sigs.items():
            if not hasattr(L, name):  # reported by the export test
                continue
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = i
        L.qg_q6k_planar_bytes.argtypes = [i, i]
        L.qg_q6k_planar_bytes.restype = sz
        L.qg_q4k_planar_bytes.argtypes = [i, i]
        L.qg_q4k_planar_bytes.restype = sz
        L.qg_lmhead_argmax_workspace_bytes.argtypes = []
        L.qg_lmhead_argmax_workspace_bytes.restype = sz
        L.qg_last_error.argtypes = []
        L.qg_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def library_path():
    return _build.LIB


def _check(rc):
    if rc != QG_OK:
        raise QgError(rc, lib().qg_last_error().decode(errors="replace"))
    return rc


def _dev(x):
    """Device pointer of a torch tensor or an int."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return ctypes.c_void_p(x.data_ptr())
    return ctypes.c_void_p(int(x))


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return ctypes.c_void_p(s.cuda_stream)
    return ctypes.c_void_p(int(s))


def _host(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------ building blocks

def qg_gemv_q4k(w, x, y, n, k, stream=None):
    return _check(lib().qg_gemv_q4k(_dev(w), _dev(x), _dev(y), n, k, _stream(stream)))


def qg_gemv_q6k(w, x, y, n, k, stream=None):
    return _check(lib().qg_gemv_q6k(_dev(w), _dev(x), _dev(y), n, k, _stream(stream)))


def qg_gemv_q6k_planar(w_planar, x, y, n, k, stream=None):
    return _check(lib().qg_gemv_q6k_planar(_dev(w_planar), _dev(x), _dev(y), n, k, _stream(stream)))


def qg_gemv_q4k_planar(w_planar, x, y, n, k, stream=None):
    return _check(lib().qg_gemv_q4k_planar(_dev(w_planar), _dev(x), _dev(y), n, k, _stream(stream)))


def qg_q4k_planar_bytes(n, k):
    return int(lib().qg_q4k_planar_bytes(n, k))


def qg_q4k_to_planar(src, dst, n, k, stream=None):
    return _check(lib().qg_q4k_to_planar(_dev(src), _dev(dst), n, k, _stream(stream)))


def qg_q6k_planar_bytes(n, k):
    return int(lib().qg_q6k_planar_bytes(n, k))


def qg_q6k_to_planar(src, dst, n, k, stream=None):
    return _check(lib().qg_q6k_to_planar(_dev(src), _dev(dst), n, k, _stream(stream)))


def qg_lmhead_argmax_workspace_bytes():
    return int(lib().qg_lmhead_argmax_workspace_bytes())


def qg_lmhead_argmax(w_planar, x, n_vocab, k, workspace, tok, stream=None):
    return _check(lib().qg_lmhead_argmax(_dev(w_planar), _dev(x), n_vocab, k, _dev(workspace), _dev(tok),
                                         _stream(stream)))


def qg_lmhead_argmax_noalloc(w_planar, x, n_vocab, k, tok, stream=None):
    return _check(lib().qg_lmhead_argmax_noalloc(_dev(w_planar), _dev(x), n_vocab, k, _dev(tok), _stream(stream)))


def qg_argmax_f32(x, n, idx, stream=None):
    return _check(lib().qg_argmax_f32(_dev(x), n, _dev(idx), _stream(stream)))


def qg_device_status():
    return _check(lib().qg_device_status())


def qg_last_error():
    return lib().qg_last_error().decode(errors="replace")


# -------------------------------------------------------------- model / state

def _qt(t):
    if t is None:
        return QgQTensor(None, 0, 0, 0)
    return QgQTensor(ctypes.c_void_p(t.data.ctypes.data), t.qtype, t.n, t.k)


class Model:
    """Device-resident weights (qg_model).  `weights` has the attributes of
    include/qg.h's qg_host_weights (cfg, token_embd, output_norm, lm_head,
    layers[...] with the qg_layer_weights field names); host arrays are
    copied to the device by qg_model_create."""

    def __init__(self, weights, device=0):
        c = weights.cfg
        self.cfg = c
        self._kinds = (ctypes.c_int32 * c.n_layers)(*c.kinds())
        self._cfg = QgConfig(c.n_layers, c.hidden, c.ffn, c.vocab, c.n_k_heads, c.n_v_heads, c.head_k_dim,
                             c.head_v_dim, c.conv_kernel, c.n_heads, c.n_kv_heads, c.head_dim, c.n_rot,
                             c.eps, c.rope_theta, self._kinds)
        layers = (QgLayerWeights * c.n_layers)()
        for il, L in enumerate(weights.layers):
            o = layers[il]
            o.kind = L.kind
            o.attn_norm, o.post_attention_norm = _host(L.attn_norm).value, _host(L.post_attention_norm).value
            o.ffn_gate, o.ffn_up, o.ffn_down = _qt(L.ffn_gate), _qt(L.ffn_up), _qt(L.ffn_down)
            if L.kind == QG_LAYER_DELTANET:
                o.ssm_conv1d, o.ssm_a_log = _host(L.ssm_conv1d).value, _host(L.ssm_a_log).value
                o.ssm_dt_bias, o.ssm_norm = _host(L.ssm_dt_bias).value, _host(L.ssm_norm).value
                o.attn_qkv, o.ssm_alpha, o.ssm_beta = _qt(L.attn_qkv), _qt(L.ssm_alpha), _qt(L.ssm_beta)
                o.attn_gate, o.ssm_out = _qt(L.attn_gate), _qt(L.ssm_out)
            else:
                o.attn_q_norm, o.attn_k_norm = _host(L.attn_q_norm).value, _host(L.attn_k_norm).value
                o.attn_q, o.attn_k, o.attn_v = _qt(L.attn_q), _qt(L.attn_k), _qt(L.attn_v)
                o.attn_output = _qt(L.attn_output)
        hw = QgHostWeights(_host(weights.token_embd).value, _host(weights.output_norm).value,
                           _qt(weights.lm_head), layers)
        h = ctypes.c_void_p()
        _check(lib().qg_model_create(ctypes.byref(self._cfg), ctypes.byref(hw), device, ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) and self.handle.value:
            lib().qg_model_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class State:
    """Per-sequence decode state (qg_state)."""

    def __init__(self, model: Model, max_seq_len: int, kv_format: int = KV_F32):
        self.model = model
        self.cfg = model.cfg
        self.max_seq_len = max_seq_len
        self.kv_format = kv_format
        h = ctypes.c_void_p()
        _check(lib().qg_state_create_kv(model.handle, max_seq_len, kv_format, ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) and self.handle.value:
            lib().qg_state_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        _check(lib().qg_state_reset(self.handle))

    def upload_layer(self, il, conv, ssm):
        conv = np.ascontiguousarray(conv, np.float32)
        ssm = np.ascontiguousarray(ssm, np.float32)
        _check(lib().qg_state_upload_layer(self.handle, il, _host(conv), _host(ssm)))

    def upload_kv(self, il, k, v):
        k = np.ascontiguousarray(k, np.float32)
        v = np.ascontiguousarray(v, np.float32)
        rows = k.shape[0] if k.ndim == 2 else k.size // self.cfg.kv_dim
        _check(lib().qg_state_upload_kv(self.handle, il, _host(k), _host(v), rows))

    def download_layer(self, il):
        c = self.cfg
        if c.kinds()[il] == QG_LAYER_DELTANET:
            conv = np.empty((c.conv_dim, c.conv_kernel - 1), np.float32)
            ssm = np.empty((c.n_v_heads, c.head_v_dim, c.head_k_dim), np.float32)
            n = ctypes.c_size_t()
            _check(lib().qg_state_download_layer(self.handle, il, _host(conv), _host(ssm), ctypes.byref(n)))
            return conv, ssm
        n = ctypes.c_size_t()
        _check(lib().qg_state_download_layer(self.handle, il, None, None, ctypes.byref(n)))
        k = np.empty(n.value, np.float32)
        v = np.empty(n.value, np.float32)
        if n.value:
            _check(lib().qg_state_download_layer(self.handle, il, _host(k), _host(v), ctypes.byref(n)))
        return k.reshape(-1, c.kv_dim), v.reshape(-1, c.kv_dim)

    def download_kv_records(self, il):
        """Quantized cache of attention layer il: (K records [n_kv][kv_len][272],
        V records [n_kv][kv_len][192]) as uint8 arrays."""
        kb, vb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().qg_state_download_kv_records(self.handle, il, None, None, ctypes.byref(kb), ctypes.byref(vb)))
        k = np.empty(kb.value, np.uint8)
        v = np.empty(vb.value, np.uint8)
        if kb.value:
            _check(lib().qg_state_download_kv_records(self.handle, il, _host(k), _host(v), ctypes.byref(kb),
                                                      ctypes.byref(vb)))
        nkv = self.cfg.n_kv_heads
        return k.reshape(nkv, -1, K_RECORD_BYTES), v.reshape(nkv, -1, V_RECORD_BYTES)

    def download_hidden(self):
        h = np.empty(self.cfg.hidden, np.float32)
        _check(lib().qg_state_download_hidden(self.handle, _host(h)))
        return h

    @property
    def kv_len(self):
        v = ctypes.c_int()
        _check(lib().qg_state_kv_len(self.handle, ctypes.byref(v)))
        return v.value

    @property
    def stream(self):
        """The state's CUDA stream handle (int)."""
        v = ctypes.c_void_p()
        _check(lib().qg_state_stream(self.handle, ctypes.byref(v)))
        return v.value or 0

    def stats(self):
        st = QgStats()
        _check(lib().qg_state_stats(self.handle, ctypes.byref(st)))
        return st.as_dict()

    def set_token_mask(self, allow_words=None):
        """Token mask of the whole-token calls (qg_state_set_token_mask):
        `allow_words` a uint32 array of ceil(vocab/32) words, bit i & 31 of
        word i >> 5 set = token i allowed; None clears it."""
        if allow_words is None:
            _check(lib().qg_state_set_token_mask(self.handle, None, 0))
            return
        a = np.ascontiguousarray(allow_words, dtype=np.uint32)
        _check(lib().qg_state_set_token_mask(self.handle, a.ctypes.data, int(a.size)))


def qg_deltanet_step(model, state, il, hidden, stream=None):
    return _check(lib().qg_deltanet_step(model.handle, state.handle, il, _dev(hidden), _stream(stream)))


def qg_attn_decode_step(model, state, il, hidden, pos, stream=None):
    return _check(lib().qg_attn_decode_step(model.handle, state.handle, il, _dev(hidden), pos, _stream(stream)))


def qg_bench_kernel(model, state, kind, launches, stream=None):
    """`launches` PDL-chained launches of one kernel kind of the decode step
    (KERNEL_*), over the layers that have it; leaves the state meaningless."""
    return _check(lib().qg_bench_kernel(model.handle, state.handle, int(kind), int(launches), _stream(stream)))


def qg_decode_token(model, state, token, pos):
    out = ctypes.c_uint32()
    _check(lib().qg_decode_token(model.handle, state.handle, int(token), int(pos), ctypes.byref(out)))
    return out.value


def qg_prefill(model, state, tokens, pos0=0):
    """Batched prompt prefill of `tokens` at positions pos0.. (qg_prefill);
    returns the first generated token."""
    t = np.ascontiguousarray(tokens, np.uint32).reshape(-1)
    out = ctypes.c_uint32()
    _check(lib().qg_prefill(model.handle, state.handle, _host(t), int(t.size), int(pos0), ctypes.byref(out)))
    return out.value


def qg_decode_batch(model, states, tokens, positions):
    """One lockstep decode step of len(states) sequences (qg_decode_batch);
    returns their next tokens."""
    n = len(states)
    hs = (ctypes.c_void_p * n)(*[st.handle.value for st in states])
    t = np.ascontiguousarray(tokens, np.uint32).reshape(-1)
    p = np.ascontiguousarray(positions, np.int32).reshape(-1)
    assert t.size == n and p.size == n
    out = np.zeros(n, np.uint32)
    _check(lib().qg_decode_batch(model.handle, ctypes.cast(hs, ctypes.c_void_p), n, _host(t), _host(p), _host(out)))
    return [int(x) for x in out]


class Batch:
    """A fixed set of sequences decoded in lockstep through one captured graph
    (qg_batch_create / qg_batch_step / qg_batch_destroy)."""

    def __init__(self, model, states):
        self.model, self.states = model, list(states)
        hs = (ctypes.c_void_p * len(self.states))(*[st.handle.value for st in self.states])
        h = ctypes.c_void_p()
        _check(lib().qg_batch_create(model.handle, ctypes.cast(hs, ctypes.c_void_p), len(self.states),
                                     ctypes.byref(h)))
        self.handle = h

    def step(self, tokens, positions):
        n = len(self.states)
        t = np.ascontiguousarray(tokens, np.uint32).reshape(-1)
        p = np.ascontiguousarray(positions, np.int32).reshape(-1)
        assert t.size == n and p.size == n
        out = np.zeros(n, np.uint32)
        _check(lib().qg_batch_step(self.handle, _host(t), _host(p), _host(out)))
        return [int(x) for x in out]

    def close(self):
        if getattr(self, "handle", None) and self.handle.value:
            lib().qg_batch_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def qg_decode_token_eager(model, state, token, pos):
    out = ctypes.c_uint32()
    _check(lib().qg_decode_token_eager(model.handle, state.handle, int(token), int(pos), ctypes.byref(out)))
    return out.value


def qg_decode_greedy(model, state, pos0, n_steps):
    out = np.empty(n_steps, np.uint32)
    _check(lib().qg_decode_greedy(model.handle, state.handle, int(pos0), int(n_steps), _host(out)))
    return out
