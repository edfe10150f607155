"""Workload shapes of the decode QKV stage (pure data, no arithmetic).

Shapes are those of Qwen2.5 0.5B / 7B / 14B attention inputs, the models the
pages measure ("73 · D3-8 — G4 FusedQKV ported to CUDA", §2: 14B od 7168 x
id 5120, 7B od 4608 x id 3584; "07 · The allocator: liveness, buffer reuse,
and the KV cache", §2.5: 0.5B KV width 128).  Weights, bias and inputs are
seeded synthetic values (``qkv_rope_kv_gb300.synth``), not trained weights.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_head: int
    n_head_kv: int
    head_dim: int
    w_dtype: str            # "f32" or "bf16"
    kv_dtype: str           # "f32" or "f16"
    n_ctx: int
    n_layers: int
    positions: tuple        # decode positions (one step per entry)
    mixed_layers: tuple = field(default=())  # layer indices of the mixed class
    theta: float = 1.0e6
    freq_scale: float = 1.0
    nt: int = 1             # tokens per step (prefill when > 1)
    rmsnorm: bool = False   # decode input is the hidden state; its RMSNorm runs in the projection kernel
    rms_eps: float = 1.0e-6
    qknorm: bool = False    # FusedQkvNorm: every q / k head RMS-normalised (weights of hd values) before RoPE
    qk_eps: float = 1.0e-6

    @property
    def nqt(self) -> int:
        return self.n_head * self.head_dim

    @property
    def nkt(self) -> int:
        return self.n_head_kv * self.head_dim

    @property
    def rows(self) -> int:
        return self.nqt + 2 * self.nkt

    def w_bytes(self) -> int:
        return self.rows * self.hidden * (4 if self.w_dtype == "f32" else 2)

    def kv_elem_bytes(self) -> int:
        return 4 if self.kv_dtype == "f32" else 2

    def algo_bytes_per_layer(self) -> int:
        """Bytes one decode layer must move: W, x, bias read; q|k|v and one cache row per region written."""
        return (self.w_bytes() + 4 * self.hidden + 4 * self.rows + 4 * self.rows
                + 2 * self.nkt * self.kv_elem_bytes() + (4 * self.hidden if self.rmsnorm else 0)
                + (2 * 4 * self.head_dim if self.qknorm else 0))


QWEN05_SINGLE = Workload("qwen2.5-0.5b-single-layer", 896, 14, 2, 64, "f32", "f32", 512, 1, (17,))
QWEN05_SWEEP = Workload("qwen2.5-0.5b-24layer-sweep", 896, 14, 2, 64, "f32", "f16", 2048, 24,
                        tuple(range(128)))
QWEN7B = Workload("qwen2.5-7b-28layer", 3584, 28, 4, 128, "bf16", "f16", 4096, 28, (1641,))
QWEN14B = Workload("qwen2.5-14b-48layer-mixed", 5120, 40, 8, 128, "bf16", "f16", 4096, 48, (3254,),
                   mixed_layers=tuple(range(24, 48)))
QWEN14B_PREFILL = Workload("qwen2.5-14b-prefill-nt128", 5120, 40, 8, 128, "bf16", "f16", 4096, 48,
                           tuple(range(128)), nt=128)

# The same decode steps with each layer's RMSNorm fused in front (eps 1e-6, the public
# Qwen2.5 configuration; the pages give no value).
QWEN7B_NORM = Workload("qwen2.5-7b-28layer-rmsnorm", 3584, 28, 4, 128, "bf16", "f16", 4096, 28, (1641,),
                       rmsnorm=True)
QWEN14B_NORM = Workload("qwen2.5-14b-48layer-mixed-rmsnorm", 5120, 40, 8, 128, "bf16", "f16", 4096, 48, (3254,),
                        mixed_layers=tuple(range(24, 48)), rmsnorm=True)

# Qwen3-14B attention input (H 5120, 40 q / 8 kv heads of 128, per-head q/k norm), the model
# family the pages name for FusedQkvNorm; synthetic weights, and a bias (the stage's own op
# carries one; zero-free here so the bias path stays exercised).
QWEN3_14B_QKNORM = Workload("qwen3-14b-48layer-qknorm", 5120, 40, 8, 128, "bf16", "f16", 4096, 48, (3254,),
                            qknorm=True)

WORKLOADS = {w.name: w for w in (QWEN05_SINGLE, QWEN05_SWEEP, QWEN7B, QWEN14B, QWEN14B_PREFILL, QWEN7B_NORM,
                                 QWEN14B_NORM, QWEN3_14B_QKNORM)}


@dataclass(frozen=True)
class FfnWorkload:
    """Decode FusedFFN (gate|up projection + SwiGLU) over n_layers layers of one shape."""
    name: str
    hidden: int
    n_ff: int
    w_dtype: str            # "f32" or "bf16"
    n_layers: int

    def w_bytes(self) -> int:
        return 2 * self.n_ff * self.hidden * (4 if self.w_dtype == "f32" else 2)

    def algo_bytes_per_layer(self) -> int:
        """Bytes one layer must move: the gate|up weight and x read, nf outputs written."""
        return self.w_bytes() + 4 * self.hidden + 4 * self.n_ff


# Intermediate sizes: 4864 for 0.5B is printed on page 06 (§2.2); 13824 (14B) and
# 18944 (7B) are the public Qwen2.5 model configurations.
QWEN05_FFN = FfnWorkload("qwen2.5-0.5b-ffn-24layer", 896, 4864, "f32", 24)
QWEN7B_FFN = FfnWorkload("qwen2.5-7b-ffn-28layer", 3584, 18944, "bf16", 28)
QWEN14B_FFN = FfnWorkload("qwen2.5-14b-ffn-48layer", 5120, 13824, "bf16", 48)

FFN_WORKLOADS = {w.name: w for w in (QWEN05_FFN, QWEN7B_FFN, QWEN14B_FFN)}
