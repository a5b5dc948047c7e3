"""Seeded synthetic inputs for the FP8 block-scaled linear layer.

This module holds no arithmetic of the method: it only draws BF16 tensors
with the shapes and value distributions of the decoder-layer linears the
Puro-2B pages train in blockwise FP8 ("Puro-2B: Poor Lab's Qwen2-1.5B
Trained on RTX 5090 within $5090", part 1/7, section 2.1: a Qwen3-1.7B-shaped
dense decoder, hidden 2048).  The pages measure on their own pretraining
corpus, which is not available; these tensors stand in for its activations,
weights and gradients.  Both the CUDA path's tests and the oracle take their
inputs from here.

Recipe (all workloads): a CPU ``torch.Generator`` seeded per workload draws
FP32 values in a fixed order, which are then rounded to BF16 (round to
nearest even).  "N(0, s)" means standard deviation s.  Outlier channels are
whole input columns (feature channels) multiplied by a factor; their indices
come from ``randperm`` of the same generator.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import torch


@dataclasses.dataclass(frozen=True)
class Linear:
    """One linear layer y = x W^T with x [tokens, k] and W [n, k]."""
    name: str
    tokens: int      # M
    in_features: int  # K
    out_features: int  # N
    ops: tuple        # subset of ("fprop", "dgrad", "wgrad")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    linears: tuple
    x_dist: str       # "normal", "normal_outliers", "silu_gate", "student_t3"
    outliers: int = 0
    outlier_factor: float = 1.0
    description: str = ""


WORKLOADS: Dict[str, Workload] = {
    "tiny_fprop_256x512x512": Workload(
        "tiny_fprop_256x512x512", 0,
        (Linear("tiny", 256, 512, 512, ("fprop",)),),
        "normal_outliers", outliers=4, outlier_factor=50.0,
        description="X[256,512] ~N(0,1) with 4 outlier columns x50; W[512,512] ~N(0,0.02); fprop"),
    "attn_qkv_fprop_8192x3072x2048": Workload(
        "attn_qkv_fprop_8192x3072x2048", 1,
        (Linear("qkv", 8192, 2048, 3072, ("fprop",)),),
        "normal_outliers", outliers=20, outlier_factor=30.0,
        description="attention QKV projection (16 q heads + 2x4 kv heads of dim 128): "
                    "X[8192,2048] ~N(0,1) with 1% (20) outlier columns x30; W[3072,2048] ~N(0,0.02); fprop"),
    "mlp_gate_up_16384x11264x2048": Workload(
        "mlp_gate_up_16384x11264x2048", 2,
        (Linear("gate_up", 16384, 2048, 11264, ("fprop", "dgrad")),),
        "normal",
        description="MLP gate+up: X[16384,2048] ~N(0,1); W[11264,2048] ~N(0,0.02); "
                    "dY[16384,11264] ~N(0,1e-3); fprop + dgrad"),
    "mlp_down_16384x2048x5632": Workload(
        "mlp_down_16384x2048x5632", 3,
        (Linear("down", 16384, 5632, 2048, ("fprop", "dgrad", "wgrad")),),
        "silu_gate",
        description="MLP down projection: X = silu(g)*u, g,u ~N(0,1) [16384,5632]; "
                    "W[2048,5632] ~N(0,0.02); dY[16384,2048] ~N(0,1e-3); fprop + dgrad + wgrad"),
    "decoder_layer_32768": Workload(
        "decoder_layer_32768", 7,
        (Linear("qkv", 32768, 2048, 3072, ("fprop", "dgrad", "wgrad")),
         Linear("o", 32768, 2048, 2048, ("fprop", "dgrad", "wgrad")),
         Linear("gate_up", 32768, 2048, 11264, ("fprop", "dgrad", "wgrad")),
         Linear("down", 32768, 5632, 2048, ("fprop", "dgrad", "wgrad"))),
        "student_t3",
        description="one decoder layer's four linears at 32768 tokens; X ~ t(3)/sqrt(3) "
                    "(unit variance); W ~N(0,0.02); dY ~N(0,1e-3); fprop + dgrad + wgrad"),
}

# The decoder layer at fewer tokens (same recipe and seed): small cases for
# profiler captures whose DRAM traffic is scaled to 32768 tokens.
for _tokens in (8192, 16384):
    _name = f"decoder_layer_{_tokens}"
    WORKLOADS[_name] = dataclasses.replace(
        WORKLOADS["decoder_layer_32768"], name=_name,
        linears=tuple(dataclasses.replace(lin, tokens=_tokens) for lin in WORKLOADS["decoder_layer_32768"].linears),
        description=f"the decoder layer's four linears at {_tokens} tokens (profiling cases)")

# The five configurations of the benchmark's metric, in order.
CONFIGS = ("tiny_fprop_256x512x512", "attn_qkv_fprop_8192x3072x2048", "mlp_gate_up_16384x11264x2048",
           "mlp_down_16384x2048x5632", "decoder_layer_32768")

WEIGHT_STD = 0.02
GRAD_STD = 1e-3


def _gen(seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _draw_x(wl: Workload, lin: Linear, g: torch.Generator, device: str) -> torch.Tensor:
    m, k = lin.tokens, lin.in_features
    if wl.x_dist in ("normal", "normal_outliers"):
        x = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
        if wl.outliers:
            idx = torch.randperm(k, generator=g, device=device)[: wl.outliers]
            x[:, idx] *= wl.outlier_factor
    elif wl.x_dist == "silu_gate":
        gate = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
        up = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
        x = torch.nn.functional.silu(gate) * up
        del gate, up
    elif wl.x_dist == "student_t3":
        # t(3) = Z / sqrt(chi2_3 / 3); divided by sqrt(3) for unit variance.
        z = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
        chi2 = torch.zeros(m, k, device=device, dtype=torch.float32)
        for _ in range(3):
            e = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
            chi2.addcmul_(e, e)
            del e
        x = z / torch.sqrt(chi2)  # = t3 / sqrt(3)
        del z, chi2
    else:
        raise ValueError(wl.x_dist)
    return x.to(torch.bfloat16)


def make_linear_inputs(wl: Workload, device: str = "cpu") -> List[Dict[str, torch.Tensor]]:
    """Draw (x, w[, dy]) BF16 tensors for every linear of a workload, in order.

    The draw order per linear is x, w, dy.  Drawing on device="cpu" is the
    reference recipe that parity tests use; device="cuda" draws the same
    distributions from CUDA's generator (different values), which the
    benchmark may use to skip host generation of multi-GB tensors."""
    g = _gen(wl.seed, device)
    out = []
    for lin in wl.linears:
        x = _draw_x(wl, lin, g, device)
        w = (torch.randn(lin.out_features, lin.in_features, generator=g, device=device,
                         dtype=torch.float32) * WEIGHT_STD).to(torch.bfloat16)
        d = {"x": x, "w": w}
        if "dgrad" in lin.ops or "wgrad" in lin.ops:
            d["dy"] = (torch.randn(lin.tokens, lin.out_features, generator=g, device=device,
                                   dtype=torch.float32) * GRAD_STD).to(torch.bfloat16)
        out.append(d)
    return out


def random_bf16(shape, seed: int, std: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """Plain N(0, std) BF16 tensor for shape/edge-case tests."""
    g = _gen(seed, device)
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def sample_rows(total: int, seed: int, count: int = 256) -> torch.Tensor:
    """Seeded row sample for checking large outputs: randperm(total)[:count]
    under a generator seeded with `seed`, sorted."""
    g = _gen(seed, "cpu")
    idx = torch.randperm(total, generator=g)[: min(count, total)]
    return torch.sort(idx).values
