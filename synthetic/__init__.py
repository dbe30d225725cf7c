"""Seeded synthetic inputs for the tensor/sequence-parallel MLP block.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds none of the block's arithmetic: it only draws random
numbers, scales them to the stated distributions and stores them in the
requested element type.

Workload shapes are the pages' model widths (all activations sequence-first
``[s, b, h]``):

* tiny TP MLP: ``[16, 2, 64]``, f = 256, tp = 2, fp32, tanh-GeLU;
* TP+SP MLP: ``[512, 4, 1024]``, f = 4096, tp = 4, SP on, bf16;
* 8.3B width (Megatron-LM 8.3B model, h = 3072, "Megatron-LM tensor parallel"
  reading, Table 1): ``[1024, 8, 3072]``, f = 12288, tp = 8, SP off, fp16;
* 22B width ("Sequence Parallel 与 Context Parallel", §SP memory, 22B
  configuration h = 6144, s = 4096, t = 8): ``[4096, 1, 6144]``, f = 24576,
  tp = 8, SP on, bf16;
* Llama-70B-like SwiGLU ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）",
  §6 numbers, H = 8192, s = 4096, b = 1, TP = 8): ``[4096, 1, 8192]``,
  ffn_hidden F = 28672 (fc1 produces 2F), tp = 8, SP on, bf16.

Distribution: X and dZ ~ N(0, 1); weights ~ N(0, 0.02) (0.02 is the standard
deviation).  Draw order X, W1, W2, dZ from one CPU ``torch.Generator`` seeded
with the config seed, in fp32, then rounded to the storage type.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class BlockConfig:
    """One MLP-block workload.  ``f`` is the ffn width (F for SwiGLU)."""

    name: str
    s: int
    b: int
    h: int
    f: int
    tp: int
    sp: bool
    dtype: str  # "f32" | "f16" | "bf16"
    act: str  # "gelu" | "swiglu" | "identity" | "relu"
    seed: int = 0

    @property
    def M(self) -> int:
        return self.s * self.b

    @property
    def fc1_rows(self) -> int:
        """Rows of W1 (= fc1 output features): 2F for SwiGLU, else f."""
        return 2 * self.f if self.act == "swiglu" else self.f

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.dtype]

    def flops_fwd_bwd(self) -> int:
        """Matmul FLOPs of one forward+backward (element-wise work excluded).

        GeLU-style block: six GEMMs of M*h*f multiply-adds = 12*M*h*f.
        SwiGLU: fc1 and its two backward GEMMs are twice as wide: 18*M*h*F.
        """
        if self.act == "swiglu":
            return 18 * self.M * self.h * self.f
        return 12 * self.M * self.h * self.f

    def with_(self, **kw) -> "BlockConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny_tp2_f32": BlockConfig("tiny_tp2_f32", 16, 2, 64, 256, 2, False, "f32", "gelu"),
    "tpsp4_bf16": BlockConfig("tpsp4_bf16", 512, 4, 1024, 4096, 4, True, "bf16", "gelu"),
    "w8p3b_tp8_f16": BlockConfig("w8p3b_tp8_f16", 1024, 8, 3072, 12288, 8, False, "f16", "gelu"),
    "w22b_tpsp8_bf16": BlockConfig("w22b_tpsp8_bf16", 4096, 1, 6144, 24576, 8, True, "bf16", "gelu"),
    "llama70b_swiglu_tpsp8_bf16": BlockConfig(
        "llama70b_swiglu_tpsp8_bf16", 4096, 1, 8192, 28672, 8, True, "bf16", "swiglu"
    ),
}


def block_inputs(cfg: BlockConfig, seed: int | None = None) -> dict[str, torch.Tensor]:
    """CPU tensors X [s,b,h], W1 [fc1_rows,h], W2 [h,f], dZ [s,b,h] in cfg.dtype."""
    g = torch.Generator().manual_seed(cfg.seed if seed is None else seed)
    dt = cfg.torch_dtype
    X = torch.randn(cfg.s, cfg.b, cfg.h, generator=g)
    W1 = torch.randn(cfg.fc1_rows, cfg.h, generator=g).mul_(0.02)
    W2 = torch.randn(cfg.h, cfg.f, generator=g).mul_(0.02)
    dZ = torch.randn(cfg.s, cfg.b, cfg.h, generator=g)
    return {"X": X.to(dt), "W1": W1.to(dt), "W2": W2.to(dt), "dZ": dZ.to(dt)}


def integer_tensor(shape, lo: int, hi: int, seed: int, dtype: str = "f32") -> torch.Tensor:
    """Uniform integers in [lo, hi] stored as floats (exact in every dtype here)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, tuple(shape), generator=g).to(TORCH_DTYPES[dtype])


def integer_block_inputs(s, b, h, f, act, seed, dtype="f32", lo=-3, hi=3) -> dict[str, torch.Tensor]:
    """Small-integer X, W1, W2, dZ so that every product and sum is exact in fp32."""
    rows = 2 * f if act == "swiglu" else f
    return {
        "X": integer_tensor((s, b, h), lo, hi, seed, dtype),
        "W1": integer_tensor((rows, h), lo, hi, seed + 1, dtype),
        "W2": integer_tensor((h, f), lo, hi, seed + 2, dtype),
        "dZ": integer_tensor((s, b, h), lo, hi, seed + 3, dtype),
    }


def fp32_partials(tp: int, rows: int, cols: int, seed: int) -> torch.Tensor:
    """Random fp32 partial sums [tp, rows, cols] ~ N(0, 1) for the shard-sum kernels."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(tp, rows, cols, generator=g)


def sp_region_inputs(s: int, b: int, h: int, p: float, seed: int, dtype: str = "bf16") -> dict[str, torch.Tensor]:
    """Residual stream R [s,b,h] ~ N(0,1)·2 + 0.5, LayerNorm γ ~ 1 + N(0,0.1), β ~ N(0,0.1),
    and a dropout keep-mask (uint8, 1 = kept with probability 1 - p) for the
    sequence-parallel region around the block."""
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DTYPES[dtype]
    return {
        "R": (torch.randn(s, b, h, generator=g) * 2 + 0.5).to(dt),
        "gamma": (1 + 0.1 * torch.randn(h, generator=g)).to(dt),
        "beta": (0.1 * torch.randn(h, generator=g)).to(dt),
        "keep": (torch.rand(s, b, h, generator=g) >= p).to(torch.uint8),
        "dOut": torch.randn(s, b, h, generator=g).to(dt),
    }


@dataclass(frozen=True)
class AttnConfig:
    """One tensor-parallel self-attention workload: h = heads·d with head width
    d = 128 ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §6 numbers:
    heads = 64, head_dim = 128 at H = 8192) or 96 (the 22B model of "Sequence
    Parallel 与 Context Parallel", h = 6144, a = 64; the 8.3B model's 96 per
    head), and ``kv_heads`` key/value heads (grouped-query attention, 8 × 128 at
    the Llama-70B-like width; 0 means one per query head, i.e. multi-head)."""

    name: str
    s: int
    b: int
    h: int
    heads: int
    tp: int
    sp: bool
    dtype: str
    causal: bool
    seed: int = 0
    kv_heads: int = 0

    @property
    def M(self) -> int:
        return self.s * self.b

    @property
    def d(self) -> int:
        return self.h // self.heads

    @property
    def groups(self) -> int:
        """Key/value heads (query groups)."""
        return self.kv_heads or self.heads

    @property
    def h_kv(self) -> int:
        return self.groups * self.d

    @property
    def qkv_rows(self) -> int:
        """Rows of the fused Wqkv: h + 2·h_kv."""
        return self.h + 2 * self.h_kv

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.dtype]

    def flops_fwd_bwd(self) -> int:
        """Matmul FLOPs of one forward+backward, without recomputation.

        Projections: QKV 2·M·h·(h + 2h_kv) and output 2·M·h·h forward, twice that
        backward (input and weight gradients): 12·M·h·(h + h_kv) (24·M·h² for
        multi-head attention).  Core per sequence and query head: QKᵀ and P·V
        forward (2·s²·d each), dV, dP, dQ, dK backward (2·s²·d each): 12·s²·d,
        i.e. 12·b·s²·h over all query heads — halved (to the visible pairs,
        ≈ s²/2) with the causal mask."""
        core = 12 * self.b * self.s * self.s * self.h
        if self.causal:
            core = 12 * self.b * (self.s * (self.s + 1) // 2) * self.h
        return 12 * self.M * self.h * (self.h + self.h_kv) + core

    def with_(self, **kw) -> "AttnConfig":
        return replace(self, **kw)


ATTN_CONFIGS = {
    "attn_tiny_tp2_bf16": AttnConfig("attn_tiny_tp2_bf16", 192, 2, 512, 4, 2, True, "bf16", False),
    "llama70b_attn_tpsp8_bf16": AttnConfig("llama70b_attn_tpsp8_bf16", 4096, 1, 8192, 64, 8, True, "bf16", True),
    "llama70b_attn_unmasked_tpsp8_bf16": AttnConfig(
        "llama70b_attn_unmasked_tpsp8_bf16", 4096, 1, 8192, 64, 8, True, "bf16", False
    ),
    # grouped-query attention at the Llama-70B-like width: 64 query heads, 8 KV heads of 128
    "llama70b_gqa_attn_tpsp8_bf16": AttnConfig(
        "llama70b_gqa_attn_tpsp8_bf16", 4096, 1, 8192, 64, 8, True, "bf16", True, kv_heads=8
    ),
    # the 22B model: h = 6144, 64 heads of 96, s = 4096, t = 8, SP
    "w22b_attn_tpsp8_bf16": AttnConfig("w22b_attn_tpsp8_bf16", 4096, 1, 6144, 64, 8, True, "bf16", True),
}


def attn_inputs(cfg: AttnConfig, seed: int | None = None) -> dict[str, torch.Tensor]:
    """CPU tensors X [s,b,h], Wqkv [h+2h_kv,h], Wo [h,h], dZ [s,b,h] in cfg.dtype:
    X, dZ ~ N(0, 1), weights ~ N(0, 0.02), drawn in that order from one generator."""
    g = torch.Generator().manual_seed(cfg.seed if seed is None else seed)
    dt = cfg.torch_dtype
    X = torch.randn(cfg.s, cfg.b, cfg.h, generator=g)
    Wqkv = torch.randn(cfg.qkv_rows, cfg.h, generator=g).mul_(0.02)
    Wo = torch.randn(cfg.h, cfg.h, generator=g).mul_(0.02)
    dZ = torch.randn(cfg.s, cfg.b, cfg.h, generator=g)
    return {"X": X.to(dt), "Wqkv": Wqkv.to(dt), "Wo": Wo.to(dt), "dZ": dZ.to(dt)}
