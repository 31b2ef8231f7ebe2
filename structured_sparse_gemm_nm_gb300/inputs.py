"""Seeded synthetic inputs shaped like the workloads the source pages discuss.

This module draws random numbers and nothing else: no pruning, packing or
multiplication happens here.  Every tensor is drawn on the host with a CPU
``torch.Generator`` in float32 and then cast (round-to-nearest-even) to the
storage type, so the GPU path and the CPU oracle can be fed bit-identical
data.  Standard deviations are given as the second argument of ``N(0, s)``.

Workloads (sizes follow the pages' layers):

* ``tiny``: 2:4 round trip, W f16 64x128 ~ U(-1, 1), X f16 128x32 ~ N(0, 1)
  (cuSPARSELt blog, "Structured sparse matrix-matrix multiplication code
  example": prune, check, compress, matmul).
* ``mlp``: SparseLinear 512->256 f16 (PyTorch issue #126420, the MNIST
  model) with W ~ N(0, 0.05), X 4096x512 = relu(N(0, 1)), dY 4096x256 ~
  N(0, 0.01).
* ``bert``: BERT-Large-shaped GEMMs (cuSPARSELt blog, Table 1) with 32x128
  tokens; W ~ N(0, 0.02), activations ~ N(0, 1); int8 variants are uniform
  integers in [-127, 127].
* ``nm``: arbitrary N:M (apex PR #1631), W f16 4096x4096 ~ N(0, 0.02),
  x f16 [b][4096] ~ N(0, 1).
* ``gptneo``: GPT-neo-125M-shaped linears (microsoft/mttl PR #108), bf16,
  12 layers of QKV 768->2304, O 768->768, FC1 768->3072, FC2 3072->768,
  W ~ N(0, 0.02), 16384 tokens of activations ~ N(0, 1).
"""
from __future__ import annotations

import torch

# Seeds per tensor role.
SEED_W, SEED_X, SEED_DY, SEED_C, SEED_VEC = 0, 1, 2, 3, 4

# GPT-neo-125M block linears as (name, out_features, in_features).
GPTNEO_LINEARS = (("qkv", 2304, 768), ("o", 768, 768), ("fc1", 3072, 768), ("fc2", 768, 3072))
GPTNEO_LAYERS = 12
GPTNEO_TOKENS = 16384

# BERT-Large-shaped pruned GEMMs as (M, N, K) with N = 32 sequences x 128 tokens.
BERT_SHAPES = ((1024, 4096, 1024), (4096, 4096, 1024), (1024, 4096, 4096))

_TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, dtype: str = "f16", device="cpu") -> torch.Tensor:
    """N(0, std) drawn in float32, cast to ``dtype`` (f16, bf16 or f32).

    ``device`` selects where the numbers are drawn (large benchmark inputs are
    drawn on the GPU; CPU and GPU draws of one seed differ)."""
    x = torch.randn(*shape, generator=_gen(seed, device), dtype=torch.float32, device=device) * float(std)
    return x.to(_TORCH_DT[dtype])


def relu_normal(shape, seed: int, dtype: str = "f16") -> torch.Tensor:
    """max(N(0, 1), 0) drawn in float32 (post-ReLU activations), cast to ``dtype``."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32).clamp_min_(0.0)
    return x.to(_TORCH_DT[dtype])


def uniform(shape, lo: float, hi: float, seed: int, dtype: str = "f16") -> torch.Tensor:
    """U(lo, hi) drawn in float32, cast to ``dtype``."""
    x = torch.rand(*shape, generator=_gen(seed), dtype=torch.float32) * (hi - lo) + lo
    return x.to(_TORCH_DT[dtype])


def uniform_int8(shape, seed: int, lo: int = -127, hi: int = 127) -> torch.Tensor:
    """Integers uniform on [lo, hi] inclusive, stored as int8."""
    return torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed), dtype=torch.int16).to(torch.int8)


def gptneo_seed(layer: int, linear: int, role: int) -> int:
    """Distinct seed per (layer, linear, tensor role) of the GPT-neo-shaped workload."""
    return 1000 * (layer + 1) + 10 * linear + role


def as_numpy_bits(t: torch.Tensor):
    """Host numpy view of a CPU tensor's storage: uint16 bit patterns for f16/bf16, int8 for int8."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.int8:
        return t.numpy()
    if t.dtype in (torch.float32, torch.int32, torch.uint8, torch.int16, torch.int64):
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
