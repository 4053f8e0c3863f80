"""CPU oracle of the decode step -- TEST INFRASTRUCTURE.

Only the tests, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` use this package; the CUDA library and its Python binding never
import it.  The arithmetic lives in qg_oracle.c (plain C, f32 as the pages fix
it); this module compiles it, marshals numpy arrays into its structs and
keeps the model/state objects alive.

Every function of qg_oracle.c is pinned by tests/test_oracle_pins.py and
tests/test_oracle_kvq.py against closed forms, invariants, hand-worked
examples or brute force; the layer and whole-token compositions are pinned by
tests/test_oracle_compose.py, which restates them from those primitives and
checks that planted wiring mistakes are detected.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np

import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qg_oracle.c")
_LIB = os.path.join(_HERE, "libqg_oracle.so")
_lib = None

Q4_K, Q6_K = 12, 14
DELTANET, ATTENTION = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, no FMA contraction, OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class OrConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "hidden", "ffn", "vocab", "n_k_heads", "n_v_heads", "head_k_dim",
        "head_v_dim", "conv_kernel", "n_heads", "n_kv_heads", "head_dim", "n_rot")] + [
        ("eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("max_seq_len", ctypes.c_int)]


class OrQt(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("qtype", ctypes.c_int), ("n", ctypes.c_int),
                ("k", ctypes.c_int)]


_FP = ctypes.POINTER(ctypes.c_float)


class OrLayer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("attn_norm", _FP), ("post_norm", _FP),
                ("ffn_gate", OrQt), ("ffn_up", OrQt), ("ffn_down", OrQt),
                ("conv1d", _FP), ("a_log", _FP), ("dt_bias", _FP), ("ssm_norm", _FP),
                ("qkv", OrQt), ("alpha", OrQt), ("beta", OrQt), ("gate", OrQt), ("ssm_out", OrQt),
                ("q_norm", _FP), ("k_norm", _FP),
                ("wq", OrQt), ("wk", OrQt), ("wv", OrQt), ("wo", OrQt)]


class OrModel(ctypes.Structure):
    _fields_ = [("cfg", OrConfig), ("embd", _FP), ("out_norm", _FP), ("lm_head", OrQt),
                ("layers", ctypes.POINTER(OrLayer))]


class OrState(ctypes.Structure):
    _fields_ = [("conv", ctypes.POINTER(_FP)), ("ssm", ctypes.POINTER(_FP)),
                ("kc", ctypes.POINTER(_FP)), ("vc", ctypes.POINTER(_FP)), ("kv_len", ctypes.c_int),
                ("kv_format", ctypes.c_int), ("kq", ctypes.POINTER(ctypes.c_void_p)),
                ("vq", ctypes.POINTER(ctypes.c_void_p))]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        f, i, p = ctypes.c_float, ctypes.c_int, ctypes.c_void_p
        sig = {
            "or_set_threads": (None, [i]),
            "or_max_threads": (i, []),
            "or_f16": (f, [ctypes.c_uint16]),
            "or_q4k_scale_min": (None, [p, i, p, p]),
            "or_dequant_q4k_block": (None, [p, p]),
            "or_dequant_q6k_block": (None, [p, p]),
            "or_dequant_row": (None, [OrQt, i, p]),
            "or_gemv": (None, [OrQt, p, p]),
            "or_gemv_f64": (None, [OrQt, p, p]),
            "or_gemv_rows": (None, [OrQt, p, p, i, p]),
            "or_silu": (f, [f]),
            "or_sigmoid": (f, [f]),
            "or_softplus": (f, [f]),
            "or_rmsnorm": (None, [p, p, p, i, f]),
            "or_l2norm_heads": (None, [p, i, i, f]),
            "or_conv1d_silu": (None, [p, p, p, p, i, i]),
            "or_gates": (None, [p, p, p, p, p, p, i]),
            "or_delta_rule": (None, [p, p, p, p, p, p, p, i, i, i, i]),
            "or_gated_rmsnorm": (None, [p, p, p, p, i, i, f]),
            "or_swiglu": (None, [p, p, p, i]),
            "or_split_q_gate": (None, [p, p, p, i, i]),
            "or_rmsnorm_heads": (None, [p, p, p, i, i, f]),
            "or_theta_scale": (f, [f, i]),
            "or_rope_neox": (None, [p, i, i, i, i, f]),
            "or_attention": (None, [p, p, p, p, i, i, i, i]),
            "or_sigmoid_gate": (None, [p, p, i]),
            "or_f32_to_f16": (ctypes.c_uint16, [f]),
            "or_f32_to_f16_n": (None, [p, i, p]),
            "or_kv_prescaled": (None, [p, i, i, p]),
            "or_quantize_q8_0": (None, [p, i, p]),
            "or_dequantize_q8_0": (None, [p, i, p]),
            "or_quantize_q5_1": (None, [p, i, p]),
            "or_dequantize_q5_1": (None, [p, i, p]),
            "or_argmax": (i, [p, i]),
            "or_top2": (None, [p, i, p, p]),
            "or_deltanet_layer": (None, [ctypes.POINTER(OrModel), ctypes.POINTER(OrState), i, p]),
            "or_attention_layer": (None, [ctypes.POINTER(OrModel), ctypes.POINTER(OrState), i, p, i]),
            "or_forward_token": (i, [ctypes.POINTER(OrModel), ctypes.POINTER(OrState), i, i, p, p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def fptr(a):
    if a is None:
        return None
    assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_FP)


def set_threads(n: int):
    lib().or_set_threads(int(n))


def max_threads() -> int:
    return int(lib().or_max_threads())


# ----------------------------------------------------------- single ops

def qt(t: "synth.QTensor") -> OrQt:
    if t is None:
        return OrQt(None, 0, 0, 0)
    return OrQt(ctypes.c_void_p(t.data.ctypes.data), t.qtype, t.n, t.k)


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def dequant_block(block: np.ndarray, qtype: int) -> np.ndarray:
    out = np.empty(256, np.float32)
    b = np.ascontiguousarray(block, dtype=np.uint8)
    if qtype == Q4_K:
        lib().or_dequant_q4k_block(ptr(b), ptr(out))
    else:
        lib().or_dequant_q6k_block(ptr(b), ptr(out))
    return out


def dequant(t) -> np.ndarray:
    out = np.empty((t.n, t.k), np.float32)
    for r in range(t.n):
        lib().or_dequant_row(qt(t), r, ptr(out[r]))
    return out


def q4k_scale_min(scale_bytes: np.ndarray, j: int):
    sc, m = ctypes.c_int(), ctypes.c_int()
    b = np.ascontiguousarray(scale_bytes, dtype=np.uint8)
    lib().or_q4k_scale_min(ptr(b), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def gemv(t, x) -> np.ndarray:
    x = f32(x)
    y = np.empty(t.n, np.float32)
    lib().or_gemv(qt(t), ptr(x), ptr(y))
    return y


def gemv_f64(t, x) -> np.ndarray:
    x = f32(x)
    y = np.empty(t.n, np.float64)
    lib().or_gemv_f64(qt(t), ptr(x), ptr(y))
    return y


def gemv_rows(t, x, rows) -> np.ndarray:
    x = f32(x)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    y = np.empty(len(rows), np.float32)
    lib().or_gemv_rows(qt(t), ptr(x), ptr(rows), len(rows), ptr(y))
    return y


def rmsnorm(x, w, eps=1e-6):
    x, w = f32(x), f32(w)
    y = np.empty_like(x)
    lib().or_rmsnorm(ptr(x), ptr(w), ptr(y), x.size, eps)
    return y


def l2norm_heads(x, dk, eps=1e-6):
    x = f32(x).copy()
    lib().or_l2norm_heads(ptr(x), dk, x.size // dk, eps)
    return x


def conv1d_silu(xin, win, wconv):
    """Returns (out, rolled window); `win` [C, K-1] is not modified."""
    xin, wconv = f32(xin), f32(wconv)
    win = f32(win).copy()
    C, K = wconv.shape
    out = np.empty(C, np.float32)
    lib().or_conv1d_silu(ptr(xin), ptr(win), ptr(wconv), ptr(out), C, K)
    return out, win


def gates(alpha, dt_bias, a, beta_raw):
    alpha, dt_bias, a, beta_raw = f32(alpha), f32(dt_bias), f32(a), f32(beta_raw)
    dt, be = np.empty_like(alpha), np.empty_like(alpha)
    lib().or_gates(ptr(alpha), ptr(dt_bias), ptr(a), ptr(beta_raw), ptr(dt), ptr(be), alpha.size)
    return dt, be


def delta_rule(q, k, v, beta, dt, S, nk, dk, nv, dv):
    """Returns (o, updated S); `S` [nv, dv, dk] is not modified."""
    q, k, v, beta, dt = f32(q), f32(k), f32(v), f32(beta), f32(dt)
    S = f32(S).copy()
    o = np.empty(nv * dv, np.float32)
    lib().or_delta_rule(ptr(q), ptr(k), ptr(v), ptr(beta), ptr(dt), ptr(S), ptr(o), nk, dk, nv, dv)
    return o, S


def gated_rmsnorm(o, z, w, dv, eps=1e-6):
    o, z, w = f32(o), f32(z), f32(w)
    u = np.empty_like(o)
    lib().or_gated_rmsnorm(ptr(o), ptr(z), ptr(w), ptr(u), dv, o.size // dv, eps)
    return u


def swiglu(g, up):
    g, up = f32(g), f32(up)
    act = np.empty_like(g)
    lib().or_swiglu(ptr(g), ptr(up), ptr(act), g.size)
    return act


def split_q_gate(qf, nh, hd):
    qf = f32(qf)
    q, gate = np.empty(nh * hd, np.float32), np.empty(nh * hd, np.float32)
    lib().or_split_q_gate(ptr(qf), ptr(q), ptr(gate), nh, hd)
    return q, gate


def rmsnorm_heads(x, w, hd, eps=1e-6):
    x, w = f32(x), f32(w)
    y = np.empty_like(x)
    lib().or_rmsnorm_heads(ptr(x), ptr(w), ptr(y), hd, x.size // hd, eps)
    return y


def theta_scale(rope_theta, n_rot):
    return float(lib().or_theta_scale(rope_theta, n_rot))


def rope_neox(x, hd, n_rot, pos, ts):
    x = f32(x).copy()
    lib().or_rope_neox(ptr(x), x.size // hd, hd, n_rot, pos, ts)
    return x


def attention(q, kc, vc, nh, nkv, hd, t_len):
    q, kc, vc = f32(q), f32(kc), f32(vc)
    out = np.empty(nh * hd, np.float32)
    lib().or_attention(ptr(q), ptr(kc), ptr(vc), ptr(out), nh, nkv, hd, t_len)
    return out


# ------------------------------------------------- quantized KV cache blocks
KV_F32, KV_Q8_0_Q5_1 = 0, 1
Q8_0_BYTES, Q5_1_BYTES = 34, 24  # per 32 values


def f32_to_f16_bits(x) -> np.ndarray:
    x = f32(np.atleast_1d(x)).copy()
    out = np.empty(x.size, np.uint16)
    lib().or_f32_to_f16_n(ptr(x), x.size, ptr(out))
    return out


def kv_prescaled(x, which: int) -> np.ndarray:
    """The f32 values the codes round (which: 0 = q8_0, 1 = q5_1)."""
    x = f32(x).copy()
    pre = np.empty_like(x)
    lib().or_kv_prescaled(ptr(x), x.size, int(which), ptr(pre))
    return pre


def _kvq(fn, x, nbytes):
    x = f32(x).copy()
    assert x.size % 32 == 0
    out = np.empty(x.size // 32 * nbytes, np.uint8)
    fn(ptr(x), x.size, ptr(out))
    return out


def _kvd(fn, b, nbytes):
    b = np.ascontiguousarray(b, np.uint8)
    n = b.size // nbytes * 32
    out = np.empty(n, np.float32)
    fn(ptr(b), n, ptr(out))
    return out


def quantize_q8_0(x) -> np.ndarray:
    return _kvq(lib().or_quantize_q8_0, x, Q8_0_BYTES)


def dequantize_q8_0(b) -> np.ndarray:
    return _kvd(lib().or_dequantize_q8_0, b, Q8_0_BYTES)


def quantize_q5_1(x) -> np.ndarray:
    return _kvq(lib().or_quantize_q5_1, x, Q5_1_BYTES)


def dequantize_q5_1(b) -> np.ndarray:
    return _kvd(lib().or_dequantize_q5_1, b, Q5_1_BYTES)


def sigmoid_gate(x, gate):
    x = f32(x).copy()
    gate = f32(gate)
    lib().or_sigmoid_gate(ptr(x), ptr(gate), x.size)
    return x


def argmax(x) -> int:
    x = f32(x)
    return int(lib().or_argmax(ptr(x), x.size))


def argmax_masked(x, allow_words) -> int:
    """First-index argmax under the decode session's grammar mask (memra
    decode.rs, GraphSession mask_dev / decode_step_dc_cap_masked): a token
    whose bit (i & 31 of word i >> 5) is unset in the packed allow bitset has
    its logit replaced by -FLT_MAX before the argmax reads the row."""
    x = f32(x).copy()
    words = np.asarray(allow_words, dtype=np.uint32)
    i = np.arange(x.size)
    allowed = (words[i >> 5] >> (i & 31).astype(np.uint32)) & np.uint32(1)
    x[allowed == 0] = -np.finfo(np.float32).max
    return argmax(x)


def top2(x):
    x = f32(x)
    a, b = ctypes.c_float(), ctypes.c_float()
    lib().or_top2(ptr(x), x.size, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def silu(x):
    return float(lib().or_silu(x))


def sigmoid(x):
    return float(lib().or_sigmoid(x))


def softplus(x):
    return float(lib().or_softplus(x))


# ----------------------------------------------------------- whole model

class Model:
    """Oracle view of a synth.ModelWeights (arrays are borrowed, not copied)."""

    def __init__(self, w: "synth.ModelWeights"):
        self.w = w
        c = w.cfg
        self.cfg = c
        self._cfg = OrConfig(c.n_layers, c.hidden, c.ffn, c.vocab, c.n_k_heads, c.n_v_heads,
                             c.head_k_dim, c.head_v_dim, c.conv_kernel, c.n_heads, c.n_kv_heads,
                             c.head_dim, c.n_rot, c.eps, c.rope_theta, c.max_seq_len)
        layers = (OrLayer * c.n_layers)()
        for il, L in enumerate(w.layers):
            o = layers[il]
            o.kind = L.kind
            o.attn_norm, o.post_norm = fptr(L.attn_norm), fptr(L.post_attention_norm)
            o.ffn_gate, o.ffn_up, o.ffn_down = qt(L.ffn_gate), qt(L.ffn_up), qt(L.ffn_down)
            if L.kind == DELTANET:
                o.conv1d, o.a_log = fptr(L.ssm_conv1d), fptr(L.ssm_a_log)
                o.dt_bias, o.ssm_norm = fptr(L.ssm_dt_bias), fptr(L.ssm_norm)
                o.qkv, o.alpha, o.beta = qt(L.attn_qkv), qt(L.ssm_alpha), qt(L.ssm_beta)
                o.gate, o.ssm_out = qt(L.attn_gate), qt(L.ssm_out)
            else:
                o.q_norm, o.k_norm = fptr(L.attn_q_norm), fptr(L.attn_k_norm)
                o.wq, o.wk, o.wv, o.wo = qt(L.attn_q), qt(L.attn_k), qt(L.attn_v), qt(L.attn_output)
        self._layers = layers
        self._m = OrModel(self._cfg, fptr(w.token_embd), fptr(w.output_norm), qt(w.lm_head), layers)


class State:
    """Oracle decode state: conv windows, recurrent states, K/V caches."""

    def __init__(self, model: Model, kv_format: int = KV_F32):
        c = model.cfg
        self.cfg = c
        self.kv_format = int(kv_format)
        assert self.kv_format in (KV_F32, KV_Q8_0_Q5_1)
        n = c.n_layers
        self.conv, self.ssm, self.kc, self.vc = [None] * n, [None] * n, [None] * n, [None] * n
        self.kq, self.vq = [None] * n, [None] * n
        for il, kind in enumerate(c.kinds()):
            if kind == DELTANET:
                self.conv[il] = np.zeros((c.conv_dim, c.conv_kernel - 1), np.float32)
                self.ssm[il] = np.zeros((c.n_v_heads, c.head_v_dim, c.head_k_dim), np.float32)
            else:
                self.kc[il] = np.zeros((c.max_seq_len, c.kv_dim), np.float32)
                self.vc[il] = np.zeros((c.max_seq_len, c.kv_dim), np.float32)
                if self.kv_format == KV_Q8_0_Q5_1:
                    self.kq[il] = np.zeros((c.max_seq_len, c.kv_dim // 32 * Q8_0_BYTES), np.uint8)
                    self.vq[il] = np.zeros((c.max_seq_len, c.kv_dim // 32 * Q5_1_BYTES), np.uint8)
        arr = lambda lst: (_FP * n)(*[fptr(a) if a is not None else None for a in lst])  # noqa: E731
        barr = lambda lst: (ctypes.c_void_p * n)(*[a.ctypes.data if a is not None else None for a in lst])  # noqa
        self._s = OrState(arr(self.conv), arr(self.ssm), arr(self.kc), arr(self.vc), 0, self.kv_format,
                          barr(self.kq), barr(self.vq))

    def set_kv_rows(self, il: int, k, v):
        """Rows 0..len(k)-1 of layer il's cache from f32 K/V rows: stored as
        they are (f32 cache), or quantized to q8_0 / q5_1 blocks with the
        dequantized values as the rows the attention reads."""
        k, v = f32(k), f32(v)
        t = k.shape[0]
        if self.kv_format == KV_F32:
            self.kc[il][:t] = k
            self.vc[il][:t] = v
            return
        kb, vb = quantize_q8_0(k.reshape(-1)), quantize_q5_1(v.reshape(-1))
        self.kq[il][:t] = kb.reshape(t, -1)
        self.vq[il][:t] = vb.reshape(t, -1)
        self.kc[il][:t] = dequantize_q8_0(kb).reshape(t, -1)
        self.vc[il][:t] = dequantize_q5_1(vb).reshape(t, -1)

    @property
    def kv_len(self):
        return self._s.kv_len

    @kv_len.setter
    def kv_len(self, v):
        self._s.kv_len = int(v)


def deltanet_layer(model: Model, state: State, il: int, h) -> np.ndarray:
    h = f32(h).copy()
    lib().or_deltanet_layer(ctypes.byref(model._m), ctypes.byref(state._s), il, ptr(h))
    return h


def attention_layer(model: Model, state: State, il: int, h, pos: int) -> np.ndarray:
    h = f32(h).copy()
    lib().or_attention_layer(ctypes.byref(model._m), ctypes.byref(state._s), il, ptr(h), pos)
    return h


def forward_token(model: Model, state: State, token: int, pos: int, want_logits: bool = False):
    """Returns (token id, final hidden state, logits or None)."""
    H, V = model.cfg.hidden, model.cfg.vocab
    hidden = np.empty(H, np.float32)
    logits = np.empty(V, np.float32) if want_logits else None
    tok = lib().or_forward_token(ctypes.byref(model._m), ctypes.byref(state._s), int(token),
                                 int(pos), ptr(hidden), ptr(logits) if want_logits else None)
    if tok < 0:
        raise ValueError(f"token {token} or position {pos} out of range")
    return int(tok), hidden, logits


if __name__ == "__main__":
    build(force="--force" in sys.argv)
    print(_LIB)
