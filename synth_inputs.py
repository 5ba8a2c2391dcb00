"""Seeded synthetic inputs for the fused MoE layer (forward + backward).

This module is the one piece of code that both the CPU oracle (``oracle/``) and
the CUDA library's tests and benchmark use.  It only draws random numbers and
shapes them; it holds none of the layer's arithmetic (no routing, no GEMM, no
activation).

Workloads stand in for the Qwen3-shaped layers that the Prime Mega MoE pages
benchmark (Qwen3-30B-A3B and Qwen3-235B-A22B, 128 experts, top-8 routing,
16,384-token sequences); the real models, weights and datasets are not needed.

Recipe (every tensor is drawn in fp32 from a seeded ``torch.Generator`` on the
requested device and then rounded to bf16 with round-to-nearest-even):

* x ~ N(0, 1)                  [T, H]
* W_r ~ N(0, 0.02)             [H, E]   router
* W_gate, W_up ~ N(0, 0.02)    [E, H, F]
* W_down ~ N(0, 0.02)          [E, F, H]
* dY ~ N(0, 1)                 [T, H]   upstream gradient
* logit_bias (skewed workload only) [E] fp32:
  bias_e = -alpha * s * ln(rank_e), rank a seeded permutation of 1..E (Zipf with
  exponent s = 1.1); the four experts with the largest rank get -30 so that
  they receive no tokens.  alpha = 0.25 puts the largest expert load at about
  5.5x the mean load for the 30B shape at T = 16384.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoeShape:
    name: str
    T: int
    H: int
    F: int
    E: int
    top_k: int
    seed: int
    skew: bool = False          # add the Zipf per-expert logit bias
    precision: str = "bf16"     # "bf16", "mxfp8" or "fp8_bwd"
    keep_fp32: bool = False     # also return the un-rounded fp32 draws

    @property
    def P(self) -> int:
        """Number of (token, slot) pairs, i.e. rows of the permuted layout."""
        return self.T * self.top_k


# The workloads.  Seeds: 0 for the tiny layer (as specified), 1, 2 and 3 for the
# 30B, skewed 30B and 235B shapes; the MXFP8 workloads reuse the 235B seed, and
# the skewed MXFP8 one adds the Zipf bias to it.
WORKLOADS: Dict[str, MoeShape] = {
    "tiny": MoeShape("tiny", T=128, H=256, F=128, E=8, top_k=2, seed=0, keep_fp32=True),
    "qwen3_30b": MoeShape("qwen3_30b", T=4096, H=2048, F=768, E=128, top_k=8, seed=1),
    "qwen3_30b_skew": MoeShape("qwen3_30b_skew", T=16384, H=2048, F=768, E=128, top_k=8,
                               seed=2, skew=True),
    "qwen3_235b": MoeShape("qwen3_235b", T=16384, H=4096, F=1536, E=128, top_k=8, seed=3),
    "qwen3_235b_mxfp8": MoeShape("qwen3_235b_mxfp8", T=16384, H=4096, F=1536, E=128, top_k=8,
                                 seed=3, precision="mxfp8"),
    "qwen3_235b_fp8_bwd": MoeShape("qwen3_235b_fp8_bwd", T=16384, H=4096, F=1536, E=128,
                                   top_k=8, seed=3, precision="fp8_bwd"),
    # the MXFP8 layer once more with the skewed routing of the 30B-skew workload
    "qwen3_235b_mxfp8_skew": MoeShape("qwen3_235b_mxfp8_skew", T=16384, H=4096, F=1536, E=128,
                                      top_k=8, seed=3, skew=True, precision="mxfp8"),
}

ZIPF_S = 1.1
ZIPF_ALPHA = 0.25
ZIPF_ZERO_EXPERTS = 4
ZIPF_ZERO_BIAS = -30.0
WEIGHT_STD = 0.02


def shape(name: str, **overrides) -> MoeShape:
    """Look up a named workload, optionally overriding fields (e.g. T=...)."""
    base = WORKLOADS[name]
    return dataclasses.replace(base, **overrides) if overrides else base


def custom_shape(T: int, H: int, F: int, E: int, top_k: int, seed: int = 0,
                 skew: bool = False, precision: str = "bf16", name: str = "custom") -> MoeShape:
    return MoeShape(name, T=T, H=H, F=F, E=E, top_k=top_k, seed=seed, skew=skew,
                    precision=precision)


def _normal(gen: torch.Generator, shape, std: float, device) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def zipf_logit_bias(E: int, seed: int, alpha: float = ZIPF_ALPHA, s: float = ZIPF_S,
                    n_zero: int = ZIPF_ZERO_EXPERTS) -> torch.Tensor:
    """Per-expert logit bias whose ranks follow a seeded permutation (CPU, fp32)."""
    gen = torch.Generator(device="cpu").manual_seed(seed + 1000)
    rank = torch.randperm(E, generator=gen) + 1                       # 1..E
    bias = torch.tensor([-alpha * s * math.log(float(r)) for r in rank.tolist()],
                        dtype=torch.float32)
    if n_zero > 0:
        worst = torch.argsort(rank, descending=True)[:n_zero]
        bias[worst] = ZIPF_ZERO_BIAS
    return bias


def make_inputs(sh: MoeShape, device="cpu", with_grad: bool = True,
                with_weights: bool = True) -> Dict[str, Optional[torch.Tensor]]:
    """Draw one seeded set of inputs for workload ``sh`` on ``device``.

    Returns bf16 tensors ``x, W_r, W_gate, W_up, W_down`` (and ``dY`` when
    ``with_grad``), an fp32 ``logit_bias`` or None, and, when the workload keeps
    them, the fp32 draws under ``*_f32`` keys.  The same seed on the same device
    type gives the same bits.
    """
    device = torch.device(device)
    T, H, F, E = sh.T, sh.H, sh.F, sh.E
    out: Dict[str, Optional[torch.Tensor]] = {}
    draws = {"x": ((T, H), 1.0), "W_r": ((H, E), WEIGHT_STD)}
    if with_weights:
        draws.update({"W_gate": ((E, H, F), WEIGHT_STD), "W_up": ((E, H, F), WEIGHT_STD),
                      "W_down": ((E, F, H), WEIGHT_STD)})
    if with_grad:
        draws["dY"] = ((T, H), 1.0)
    # each tensor has its own generator stream, so leaving one out changes no other
    for stream, key in enumerate(("x", "W_r", "W_gate", "W_up", "W_down", "dY")):
        if key not in draws:
            continue
        shp, std = draws[key]
        gen = torch.Generator(device=device).manual_seed(sh.seed * 64 + stream)
        f32 = _normal(gen, shp, std, device)
        out[key] = f32.to(torch.bfloat16)
        if sh.keep_fp32:
            out[key + "_f32"] = f32
        else:
            del f32
    out["logit_bias"] = zipf_logit_bias(E, sh.seed).to(device) if sh.skew else None
    return out
