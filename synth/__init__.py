"""Seeded synthetic inputs shared by the oracle and the CUDA path.

The C core (qg_synth.c) draws SplitMix64 streams; this module turns them into
numpy arrays: f32 tensors, token ids and raw GGUF Q4_K / Q6_K block bytes.  It
holds none of the decode step's arithmetic.  Per-tensor seeds are
SplitMix64(master XOR FNV-1a(name)).

Recipe (per tensor of a model workload):
  Q4_K projections  random 4-bit quants, uniform 6-bit scales and mins,
                    fp16 d and dmin uniform in [0, 0.02)
  Q6_K projections  (ffn_down, lm_head) uniform 6-bit quants, uniform int8
                    scales, fp16 d uniform in [0, 0.02)
  norm weights      1 + N(0, 0.1)
  A_log             U(-1, 1)          dt_bias   N(0, 0.5)
  conv1d weight     N(0, 0.1)         embedding N(0, 1)
"""
import ctypes
import os
import subprocess
import sys
from dataclasses import dataclass
from typing import List, Optional

import numpy as np

from .configs import (ATTENTION, DELTANET, MASTER_SEED, ModelConfig, WORKLOADS,  # noqa: F401
                      CFG_LAYER, CFG_0P8B, CFG_4B, CFG_4B_LONG, CFG_TINY,
                      PROMPT_LEN, DECODE_LEN, LONG_PREFILL, LONG_DECODE)

QTYPE_Q4_K = 12
QTYPE_Q6_K = 14
Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qg_synth.c")
_LIB = os.path.join(_HERE, "libqg_synth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator core (plain C, no FMA contraction, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, f32, i64, p = ctypes.c_uint64, ctypes.c_float, ctypes.c_int64, ctypes.c_void_p
        L.qs_subseed.restype = u64
        L.qs_subseed.argtypes = [u64, ctypes.c_char_p]
        L.qs_u64.restype = u64
        L.qs_u64.argtypes = [u64, u64]
        L.qs_normal_f64.restype = ctypes.c_double
        L.qs_normal_f64.argtypes = [u64, u64]
        L.qs_ln.restype = ctypes.c_double
        L.qs_ln.argtypes = [ctypes.c_double]
        L.qs_f16_bits.restype = ctypes.c_uint16
        L.qs_f16_bits.argtypes = [f32]
        for name in ("qs_normal_f32", "qs_uniform_f32"):
            getattr(L, name).restype = None
            getattr(L, name).argtypes = [u64, f32, f32, p, i64]
        L.qs_bytes.restype = None
        L.qs_bytes.argtypes = [u64, p, i64]
        L.qs_tokens.restype = None
        L.qs_tokens.argtypes = [u64, ctypes.c_uint32, p, i64]
        for name in ("qs_q4k_blocks", "qs_q6k_blocks"):
            getattr(L, name).restype = None
            getattr(L, name).argtypes = [u64, f32, p, i64]
        _lib = L
    return _lib


def subseed(master: int, name: str) -> int:
    return int(lib().qs_subseed(master & 0xFFFFFFFFFFFFFFFF, name.encode()))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def normal(seed: int, shape, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().qs_normal_f32(seed, mu, sigma, _ptr(out), out.size)
    return out


def uniform(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().qs_uniform_f32(seed, lo, hi, _ptr(out), out.size)
    return out


def random_bytes(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    lib().qs_bytes(seed, _ptr(out), n)
    return out


def tokens(seed: int, vocab: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    lib().qs_tokens(seed, vocab, _ptr(out), n)
    return out


@dataclass
class QTensor:
    """Raw GGUF k-quant tensor: `n` rows of `k` weights, row-major blocks."""
    data: np.ndarray  # uint8, n * (k // 256) * block bytes
    qtype: int
    n: int
    k: int


def q4k_tensor(seed: int, n: int, k: int, dmax: float = 0.02) -> QTensor:
    assert k % 256 == 0
    nb = n * (k // 256)
    out = np.empty(nb * Q4K_BLOCK_BYTES, dtype=np.uint8)
    lib().qs_q4k_blocks(seed, dmax, _ptr(out), nb)
    return QTensor(out, QTYPE_Q4_K, n, k)


def q6k_tensor(seed: int, n: int, k: int, dmax: float = 0.02) -> QTensor:
    assert k % 256 == 0
    nb = n * (k // 256)
    out = np.empty(nb * Q6K_BLOCK_BYTES, dtype=np.uint8)
    lib().qs_q6k_blocks(seed, dmax, _ptr(out), nb)
    return QTensor(out, QTYPE_Q6_K, n, k)


@dataclass
class LayerWeights:
    kind: int
    attn_norm: np.ndarray
    post_attention_norm: np.ndarray
    ffn_gate: QTensor
    ffn_up: QTensor
    ffn_down: QTensor
    # Gated DeltaNet
    ssm_conv1d: Optional[np.ndarray] = None   # [conv_dim, conv_kernel]
    ssm_a_log: Optional[np.ndarray] = None    # [n_v_heads]
    ssm_dt_bias: Optional[np.ndarray] = None  # [n_v_heads]
    ssm_norm: Optional[np.ndarray] = None     # [head_v_dim]
    attn_qkv: Optional[QTensor] = None
    ssm_alpha: Optional[QTensor] = None
    ssm_beta: Optional[QTensor] = None
    attn_gate: Optional[QTensor] = None
    ssm_out: Optional[QTensor] = None
    # full attention
    attn_q_norm: Optional[np.ndarray] = None  # [head_dim]
    attn_k_norm: Optional[np.ndarray] = None
    attn_q: Optional[QTensor] = None
    attn_k: Optional[QTensor] = None
    attn_v: Optional[QTensor] = None
    attn_output: Optional[QTensor] = None


@dataclass
class ModelWeights:
    cfg: ModelConfig
    token_embd: np.ndarray  # [vocab, hidden] f32
    output_norm: np.ndarray
    lm_head: QTensor        # Q6_K [vocab x hidden]
    layers: List[LayerWeights]


def make_model_weights(cfg: ModelConfig, master: int = MASTER_SEED, dmax: float = 0.02) -> ModelWeights:
    """Seeded random-init weights of a model config.  `dmax` bounds the fp16
    super-block scales d / dmin of every quantized matrix (uniform in
    [0, dmax)); the model workloads use 0.02."""
    s = lambda name: subseed(master, name)  # noqa: E731
    H, F = cfg.hidden, cfg.ffn
    layers = []
    for il, kind in enumerate(cfg.kinds()):
        p = f"blk.{il}."
        common = dict(
            attn_norm=normal(s(p + "attn_norm"), H, 1.0, 0.1),
            post_attention_norm=normal(s(p + "post_attention_norm"), H, 1.0, 0.1),
            ffn_gate=q4k_tensor(s(p + "ffn_gate"), F, H, dmax),
            ffn_up=q4k_tensor(s(p + "ffn_up"), F, H, dmax),
            ffn_down=q6k_tensor(s(p + "ffn_down"), H, F, dmax),
        )
        if kind == DELTANET:
            lw = LayerWeights(
                kind=kind, **common,
                ssm_conv1d=normal(s(p + "ssm_conv1d"), (cfg.conv_dim, cfg.conv_kernel), 0.0, 0.1),
                ssm_a_log=uniform(s(p + "ssm_a_log"), cfg.n_v_heads, -1.0, 1.0),
                ssm_dt_bias=normal(s(p + "ssm_dt_bias"), cfg.n_v_heads, 0.0, 0.5),
                ssm_norm=normal(s(p + "ssm_norm"), cfg.head_v_dim, 1.0, 0.1),
                attn_qkv=q4k_tensor(s(p + "attn_qkv"), cfg.conv_dim, H, dmax),
                ssm_alpha=q4k_tensor(s(p + "ssm_alpha"), cfg.n_v_heads, H, dmax),
                ssm_beta=q4k_tensor(s(p + "ssm_beta"), cfg.n_v_heads, H, dmax),
                attn_gate=q4k_tensor(s(p + "attn_gate"), cfg.v_dim, H, dmax),
                ssm_out=q4k_tensor(s(p + "ssm_out"), H, cfg.v_dim, dmax),
            )
        else:
            lw = LayerWeights(
                kind=kind, **common,
                attn_q_norm=normal(s(p + "attn_q_norm"), cfg.head_dim, 1.0, 0.1),
                attn_k_norm=normal(s(p + "attn_k_norm"), cfg.head_dim, 1.0, 0.1),
                attn_q=q4k_tensor(s(p + "attn_q"), 2 * cfg.q_dim, H, dmax),
                attn_k=q4k_tensor(s(p + "attn_k"), cfg.kv_dim, H, dmax),
                attn_v=q4k_tensor(s(p + "attn_v"), cfg.kv_dim, H, dmax),
                attn_output=q4k_tensor(s(p + "attn_output"), H, cfg.q_dim, dmax),
            )
        layers.append(lw)
    return ModelWeights(
        cfg=cfg,
        token_embd=normal(s("token_embd"), (cfg.vocab, H), 0.0, 1.0),
        output_norm=normal(s("output_norm"), H, 1.0, 0.1),
        lm_head=q6k_tensor(s("output"), cfg.vocab, H, dmax),
        layers=layers,
    )


def initial_deltanet_state(cfg: ModelConfig, il: int, master: int = MASTER_SEED):
    """Conv window [conv_dim, conv_kernel-1] and recurrent state
    [n_v_heads, head_v_dim, head_k_dim], both N(0, 0.1)."""
    conv = normal(subseed(master, f"state.{il}.conv"), (cfg.conv_dim, cfg.conv_kernel - 1), 0.0, 0.1)
    ssm = normal(subseed(master, f"state.{il}.ssm"),
                 (cfg.n_v_heads, cfg.head_v_dim, cfg.head_k_dim), 0.0, 0.1)
    return conv, ssm


def layer_inputs(cfg: ModelConfig, n_steps: int, master: int = MASTER_SEED) -> np.ndarray:
    """Hidden-state inputs of the single-layer workload, N(0, 1), one per step."""
    return normal(subseed(master, "layer.hidden"), (n_steps, cfg.hidden), 0.0, 1.0)


def prompt_tokens(cfg: ModelConfig, n: int = PROMPT_LEN, master: int = MASTER_SEED) -> np.ndarray:
    return tokens(subseed(master, "prompt"), cfg.vocab, n)


def long_context_kv(cfg: ModelConfig, il: int, rows: int, master: int = MASTER_SEED):
    """K and V cache rows [rows, n_kv_heads * head_dim], N(0, 1)."""
    k = normal(subseed(master, f"kv.{il}.k"), (rows, cfg.kv_dim), 0.0, 1.0)
    v = normal(subseed(master, f"kv.{il}.v"), (rows, cfg.kv_dim), 0.0, 1.0)
    return k, v


if __name__ == "__main__":
    build(force="--force" in sys.argv)
    print(_LIB)
