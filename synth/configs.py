"""Named workloads: model dimensions and the synthetic-input recipe.

Dimensions follow the decode step of a hybrid Gated-DeltaNet / full-attention
model (forward_qwen35_cuda.rs, struct Qwen35CudaDims): hidden, FFN width,
DeltaNet key/value heads of 128, a 4-tap causal conv, attention heads of 256
with a [q | gate] query projection and partial NEOX rope on a quarter of each
head.  Layer `il` is full attention when il % 4 == 3 (three DeltaNet layers to
one attention layer); the single-layer workload is one DeltaNet layer.
"""
from dataclasses import dataclass, field, asdict
from typing import List

DELTANET = 0
ATTENTION = 1

MASTER_SEED = 0x5147


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    hidden: int
    ffn: int
    vocab: int
    n_k_heads: int
    n_v_heads: int
    head_k_dim: int = 128
    head_v_dim: int = 128
    conv_kernel: int = 4
    n_heads: int = 8
    n_kv_heads: int = 2
    head_dim: int = 256
    n_rot: int = 64
    eps: float = 1e-6
    rope_theta: float = 1.0e7
    max_seq_len: int = 1024
    layer_kinds: tuple = field(default=())

    @property
    def k_dim(self):
        return self.n_k_heads * self.head_k_dim

    @property
    def v_dim(self):
        return self.n_v_heads * self.head_v_dim

    @property
    def conv_dim(self):
        return 2 * self.k_dim + self.v_dim

    @property
    def q_dim(self):
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim

    def kinds(self) -> List[int]:
        if self.layer_kinds:
            return list(self.layer_kinds)
        return [ATTENTION if il % 4 == 3 else DELTANET for il in range(self.n_layers)]

    def as_dict(self):
        d = asdict(self)
        d["layer_kinds"] = self.kinds()
        return d


# One Gated DeltaNet layer (the 8-step single-layer workload).
CFG_LAYER = ModelConfig(name="deltanet-layer", n_layers=1, hidden=1024, ffn=3072, vocab=256,
                        n_k_heads=16, n_v_heads=16, layer_kinds=(DELTANET,))

# 0.8B-shaped hybrid: 24 layers (18 DeltaNet + 6 attention).
CFG_0P8B = ModelConfig(name="0.8b", n_layers=24, hidden=1024, ffn=3584, vocab=248320,
                       n_k_heads=16, n_v_heads=16, n_heads=8, n_kv_heads=2)

# 4B-shaped hybrid: 32 layers (24 DeltaNet + 8 attention), 32 value heads over 16 key heads.
CFG_4B = ModelConfig(name="4b", n_layers=32, hidden=2560, ffn=9216, vocab=248320,
                     n_k_heads=16, n_v_heads=32, n_heads=16, n_kv_heads=4)

# 4B-shaped with a KV cache of 8192 positions (decode from position 8000).
CFG_4B_LONG = ModelConfig(name="4b-long", n_layers=32, hidden=2560, ffn=9216, vocab=248320,
                          n_k_heads=16, n_v_heads=32, n_heads=16, n_kv_heads=4,
                          max_seq_len=8192)

# Small hybrid used by the parity tests: same structure, every dimension a few
# tiles wide, a vocabulary that is not a multiple of any tile.
CFG_TINY = ModelConfig(name="tiny", n_layers=4, hidden=512, ffn=768, vocab=3000,
                       n_k_heads=2, n_v_heads=4, n_heads=4, n_kv_heads=2, max_seq_len=96)

WORKLOADS = {c.name: c for c in (CFG_LAYER, CFG_0P8B, CFG_4B, CFG_4B_LONG, CFG_TINY)}

# Decode schedule of the model workloads: prompt tokens fed one per step, then
# greedy tokens.
PROMPT_LEN = 850
DECODE_LEN = 128
LONG_PREFILL = 8000
LONG_DECODE = 64
