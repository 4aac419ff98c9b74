"""Geometry and workload descriptions for the DSpark draft-and-verify step.

This module holds sizes and seeds only (no arithmetic of the method). It is
shared by the oracle and by the GPU path so that both read the same seeded
synthetic inputs.

Geometry sources (Kimi-K3-DSpark model cards):
  * hidden 7168, vocab 163,840, q_lora 1536, kv_lora 512, block size 7
    -- "kimi-k3-dspark-gguf", section "GGUF metadata";
  * 5 dense layers, non-causal, 7 tokens per pass, Markov head, confidence
    head -- "Kimi-K3-DSpark-NVFP4", "Original model card / Model Overview";
  * 5 captured states into fc, Markov rank 256, YaRN-16 from 65,536 --
    "Kimi K3 DSpark Q8_0 GGUF", section "Architecture metadata";
  * MLA split dims (nope 128, rope 64, v 128), 64 heads, SwiGLU 14336 -- the
    workload statement of this path (the cards fix only the ranks above).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple

# Purposes of the counter-based uniforms (part of the sampling spec's keying).
PURPOSE_DRAFT = 1
PURPOSE_ACCEPT = 2
PURPOSE_RESID = 3
PURPOSE_BONUS = 4

FORMAT_BF16 = 0
FORMAT_FP8 = 1
FORMAT_NVFP4 = 2
FORMAT_MXFP4 = 3


@dataclass(frozen=True)
class Geometry:
    hidden: int
    n_aux: int
    n_layers: int
    n_heads: int
    q_lora: int
    kv_lora: int
    d_nope: int
    d_rope: int
    d_v: int
    inter: int
    vocab: int
    rank: int
    block: int = 7
    rope_theta: float = 10000.0
    eps: float = 1e-6
    yarn_factor: float = 1.0  # 1.0 means plain RoPE
    yarn_orig_ctx: int = 65536
    yarn_alpha: float = 1.0
    yarn_beta: float = 32.0
    page_size: int = 64

    @property
    def kv_dim(self) -> int:
        """Latent KV entry per token per layer: kv_lora normalised latent + d_rope roped key."""
        return self.kv_lora + self.d_rope

    @property
    def qkv_a_out(self) -> int:
        return self.q_lora + self.kv_lora + self.d_rope

    @property
    def q_head_dim(self) -> int:
        return self.d_nope + self.d_rope

    # --- parameter counts (sizes of the weight set) -------------------------------
    def layer_params(self) -> dict:
        H, nh = self.hidden, self.n_heads
        return {
            "q_a": self.q_lora * H,
            "kv_a": (self.kv_lora + self.d_rope) * H,
            "q_b": nh * self.q_head_dim * self.q_lora,
            "kv_b": nh * (self.d_nope + self.d_v) * self.kv_lora,
            "o": H * nh * self.d_v,
            "gate": self.inter * H,
            "up": self.inter * H,
            "down": H * self.inter,
            "norms": 2 * H + self.q_lora + self.kv_lora,
        }

    def param_counts(self) -> dict:
        per = self.layer_params()
        layers = self.n_layers * sum(per.values())
        fc = self.hidden * self.n_aux * self.hidden
        markov = 2 * self.vocab * self.rank
        conf = self.hidden + 1
        final_norm = self.hidden
        embed = self.vocab * self.hidden
        drafter = fc + layers + markov + conf + final_norm
        quantised = fc + self.n_layers * (per["q_b"] + per["o"] + per["gate"] + per["up"] + per["down"])
        return {
            "fc": fc,
            "layers": layers,
            "markov": markov,
            "confidence": conf,
            "final_norm": final_norm,
            "embed": embed,
            "lm_head": embed,
            "drafter_no_embed": drafter,
            "drafter_with_embed": drafter + embed,
            "quantised": quantised,
        }


FULL = Geometry(hidden=7168, n_aux=5, n_layers=5, n_heads=64, q_lora=1536, kv_lora=512,
                d_nope=128, d_rope=64, d_v=128, inter=14336, vocab=163840, rank=256)

TINY = Geometry(hidden=512, n_aux=5, n_layers=2, n_heads=8, q_lora=128, kv_lora=64,
                d_nope=32, d_rope=16, d_v=32, inter=1024, vocab=4096, rank=16)

# YaRN factor 16 from 65,536 ("Context metadata: 1,048,576 with YaRN-16 from 65,536").
FULL_YARN = replace(FULL, yarn_factor=16.0)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: geometry plus how the inputs are drawn."""
    name: str
    geom: Geometry
    bs: int
    ctx: Tuple[int, ...]          # per-sequence context lengths (or a single value)
    weight_seed: int
    input_seed: int
    weight_std: float = 0.02
    aux_dist: str = "normal"      # "normal" or "student_t3_unit_rms"
    aux_std: float = 1.0
    kv_std: float = 1.0
    draft_mode: int = 0           # 0 greedy, 1 probabilistic
    verify_mode: int = 0
    temperature: float = 1.0
    top_p: float = 1.0
    target_noise: float = 0.5     # target logits = drafter logits + N(0, target_noise^2)
    weight_format: int = FORMAT_BF16
    random_pages: bool = True
    extra: dict = field(default_factory=dict)


# The five workloads. The first is the small case the oracle finishes in seconds.
TINY_STEP = Workload("tiny", TINY, bs=1, ctx=(128,), weight_seed=0, input_seed=0,
                     aux_std=0.02, kv_std=0.02)
FULL_STEP = Workload("full_bs1_ctx4096", FULL, bs=1, ctx=(4096,), weight_seed=1, input_seed=1)
LONG_STEP = Workload("full_bs1_ctx95000_yarn", FULL_YARN, bs=1, ctx=(95000,), weight_seed=1,
                     input_seed=3, aux_dist="student_t3_unit_rms", draft_mode=1, verify_mode=1,
                     temperature=1.0, top_p=0.95)
BATCH_STEP = Workload("full_bs32_paged", FULL, bs=32, ctx=(), weight_seed=1, input_seed=4,
                      extra={"ctx_lo": 1024, "ctx_hi": 16384})
FP8_STEP = Workload("full_bs1_ctx4096_fp8", FULL, bs=1, ctx=(4096,), weight_seed=1, input_seed=5,
                    weight_format=FORMAT_FP8)
NVFP4_STEP = Workload("full_bs1_ctx4096_nvfp4", FULL, bs=1, ctx=(4096,), weight_seed=1,
                      input_seed=5, weight_format=FORMAT_NVFP4)
MXFP4_STEP = Workload("full_bs1_ctx4096_mxfp4", FULL, bs=1, ctx=(4096,), weight_seed=1,
                      input_seed=5, weight_format=FORMAT_MXFP4)

WORKLOADS = {w.name: w for w in (TINY_STEP, FULL_STEP, LONG_STEP, BATCH_STEP, FP8_STEP, NVFP4_STEP, MXFP4_STEP)}
