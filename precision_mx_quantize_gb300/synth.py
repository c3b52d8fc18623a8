"""Seeded synthetic inputs shaped like the workloads the MX path serves.

Only random draws and the bf16 storage cast live here (none of the
quantization, rotation or GEMM arithmetic), so the tests, the benchmark and
the CPU oracle can all draw the same tensors.

Distributions (the pages train Llama 3.1-8B on C4, "AMD顛覆行業認知！終于攻克FP4
大模型訓練致命難題", §03; no dataset or weights are used, these stand in):

* activations: Student-t with 3 degrees of freedom times a per-channel
  LogNormal(0, 1) scale (heavy tails plus outlier channels);
* weights: N(0, 0.02);
* output gradients: N(0, 1e-3) times a per-column LogNormal(0, 2) scale;
* the small quantize/dequantize case: N(0, 1) with 1% of entries x100.

Every tensor is drawn in fp32 from a torch CPU generator seeded explicitly
and rounded to bf16 (round to nearest even).
"""

from __future__ import annotations

import torch

# Llama-3.1-8B linear layers as (name, in_features, out_features)
LLAMA8B_LINEARS = (
    ("qkv", 4096, 6144),
    ("o", 4096, 4096),
    ("gate_up", 4096, 28672),
    ("down", 14336, 4096),
)
LLAMA8B_TOKENS = 8192


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    g = _gen(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def normal_with_outliers(shape, seed: int, frac: float = 0.01, mult: float = 100.0) -> torch.Tensor:
    g = _gen(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    hit = torch.rand(shape, generator=g) < frac
    return torch.where(hit, x * mult, x).to(torch.bfloat16)


def _student_t3(shape, g: torch.Generator) -> torch.Tensor:
    # t(3) = Z / sqrt(V / 3) with V a chi-square of 3 degrees (3 squared normals)
    z = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.zeros(shape, dtype=torch.float32)
    for _ in range(3):
        n = torch.randn(shape, generator=g, dtype=torch.float32)
        v.addcmul_(n, n)
    return z / torch.sqrt(v / 3.0)


def activation(tokens: int, channels: int, seed: int) -> torch.Tensor:
    """[tokens, channels]: Student-t(3) times a per-channel LogNormal(0, 1) scale."""
    g = _gen(seed)
    t = _student_t3((tokens, channels), g)
    col = torch.exp(torch.randn((1, channels), generator=g, dtype=torch.float32))
    return (t * col).to(torch.bfloat16)


def weight(out_features: int, in_features: int, seed: int) -> torch.Tensor:
    """[out, in] (PyTorch Linear layout): N(0, 0.02)."""
    return normal((out_features, in_features), seed, 0.02)


def out_grad(tokens: int, channels: int, seed: int) -> torch.Tensor:
    """[tokens, channels]: N(0, 1e-3) times a per-column LogNormal(0, 2) scale."""
    g = _gen(seed)
    z = torch.randn((tokens, channels), generator=g, dtype=torch.float32) * 1e-3
    col = torch.exp(2.0 * torch.randn((1, channels), generator=g, dtype=torch.float32))
    return (z * col).to(torch.bfloat16)


# ---- the named workloads ------------------------------------------------------

def quantize_dequantize_small():
    """256x1024, N(0,1) with 1% x100 outliers, seed 0 (E4M3 row-wise round trip)."""
    return {"x": normal_with_outliers((256, 1024), 0)}


def hadamard_dual_activation(rows: int = 8192, cols: int = 4096):
    """8192x4096 activation for the fused Hadamard + E2M1 row-and-column quantizer."""
    return {"x": activation(rows, cols, 0)}


def mlp_up_forward(tokens: int = 8192, hidden: int = 4096, ffn: int = 14336):
    """X [tokens, hidden] ~ N(0,1), W [hidden, ffn] ~ N(0,0.02) (K x N as stored)."""
    return {"x": normal((tokens, hidden), 0), "w": normal((hidden, ffn), 1, 0.02)}


def mlp_wgrad(tokens: int = 16384, ffn: int = 14336, hidden: int = 4096):
    """dY [tokens, ffn] gradient and X [tokens, hidden] activation for dW = dY^T X."""
    g = _gen(1)
    x = (_student_t3((tokens, hidden), g)).to(torch.bfloat16)
    return {"dy": out_grad(tokens, ffn, 0), "x": x}


def decoder_block_layer(in_f: int, out_f: int, tokens: int, layer_index: int):
    """Inputs of one linear layer of the decoder-block pass, seeds 3*i .. 3*i+2."""
    s = 3 * layer_index
    return {
        "x": activation(tokens, in_f, s),
        "w": weight(out_f, in_f, s + 1),
        "dy": out_grad(tokens, out_f, s + 2),
    }


def sweep_tensor(n_elems: int, seed: int = 0) -> torch.Tensor:
    """[n/4096, 4096] N(0,1) for the quantizer bandwidth sweep."""
    return normal((n_elems // 4096, 4096), seed)
