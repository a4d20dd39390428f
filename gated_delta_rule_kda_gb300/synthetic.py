"""Seeded synthetic inputs shaped like the KDA workloads.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic beyond the input recipe itself (unit-normalising q and k
before they are rounded, and mapping a normal draw x to a log-decay in
(-5, 0) the way the workloads are specified).  Both the CUDA path and the
CPU oracle consume exactly the tensors returned here (the oracle widens the
rounded bf16/fp32 values to fp64).

Workloads (d_k = d_v = 128):
  1 oracle-scale      B=1, H=2, T=256, fp32 q/k/v, x~N(0,1), S0 = 0
  2 prefill           B=1, H=96, T=8192, bf16 q/k/v, x~N(0,2), S0 = 0
  3 decode            B=256 requests, H=96, S~N(0,0.1), bf16, x~N(0,2)
  4 long prefill      B=1, H=96, T=131072, bf16, x~N(1,1), S0~N(0,0.1)
  5 varlen layer core 16 sequences, lengths log-uniform in [1K, 64K], H=96,
                      pre-projection q^p/k^p/v^p ~N(0,1), conv w~N(0,0.5),
                      A~N(0,0.5), z~N(0,1), b=0, beta logit~N(0,1), g~N(0,1)
"N(m, s)" is read as mean m and standard deviation s.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

D = 128
BASE_SEED = 0x4B4441


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen, device, mean=0.0, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


@dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, H, 128] dtype
    k: torch.Tensor            # [T, H, 128] dtype
    v: torch.Tensor            # [T, H, 128] dtype
    log_alpha: torch.Tensor    # [T, H, 128] fp32, in (-5, 0)
    beta: torch.Tensor         # [T, H] fp32
    S0: Optional[torch.Tensor]  # [N, H, 128, 128] fp32 or None (zeros)
    cu_seqlens: torch.Tensor   # [N+1] int32

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.shape[0]) - 1


def cu_from_lengths(lengths: Sequence[int], device="cpu") -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def prefill_inputs(lengths: Sequence[int], H: int, dtype=torch.bfloat16, seed: int = BASE_SEED,
                   x_mean: float = 0.0, x_std: float = 2.0, s0_std: Optional[float] = None,
                   device="cpu", head_decay: bool = False) -> PrefillInputs:
    """q,k ~ N(0,1) unit-normalised per head, v ~ N(0,1), log_alpha = -5 sigmoid(x),
    beta = sigmoid(N(0,1)); all rounded to ``dtype`` (log_alpha, beta stay fp32).
    head_decay: one log_alpha per (token, head), shape [T, H] (the Gated DeltaNet case)."""
    g = _gen(seed, device)
    T = int(sum(lengths))
    N = len(lengths)
    q = _unit_rows(_randn((T, H, D), g, device)).to(dtype)
    k = _unit_rows(_randn((T, H, D), g, device)).to(dtype)
    v = _randn((T, H, D), g, device).to(dtype)
    la_shape = (T, H) if head_decay else (T, H, D)
    la = torch.sigmoid(_randn(la_shape, g, device, x_mean, x_std)).mul_(-5.0)
    beta = torch.sigmoid(_randn((T, H), g, device))
    S0 = None
    if s0_std is not None:
        S0 = _randn((N, H, D, D), g, device, 0.0, s0_std)
    return PrefillInputs(q, k, v, la.contiguous(), beta.contiguous(), S0,
                         cu_from_lengths(lengths, device))


@dataclass
class DecodeInputs:
    q: torch.Tensor          # [B, H, 128]
    k: torch.Tensor
    v: torch.Tensor
    log_alpha: torch.Tensor  # [B, H, 128] fp32
    beta: torch.Tensor       # [B, H] fp32
    S: torch.Tensor          # [B, H, 128, 128] fp32


def decode_inputs(B: int, H: int, dtype=torch.bfloat16, seed: int = BASE_SEED + 3,
                  x_mean: float = 0.0, x_std: float = 2.0, s_std: float = 0.1,
                  device="cpu", head_decay: bool = False) -> DecodeInputs:
    g = _gen(seed, device)
    q = _unit_rows(_randn((B, H, D), g, device)).to(dtype)
    k = _unit_rows(_randn((B, H, D), g, device)).to(dtype)
    v = _randn((B, H, D), g, device).to(dtype)
    la_shape = (B, H) if head_decay else (B, H, D)
    la = torch.sigmoid(_randn(la_shape, g, device, x_mean, x_std)).mul_(-5.0)
    beta = torch.sigmoid(_randn((B, H), g, device))
    S = _randn((B, H, D, D), g, device, 0.0, s_std)
    return DecodeInputs(q, k, v, la, beta, S)


@dataclass
class LayerInputs:
    qp: torch.Tensor          # [T, H, 128] bf16 pre-conv projections
    kp: torch.Tensor
    vp: torch.Tensor
    conv_w: torch.Tensor      # [3, H*128, 4] fp32; tap 0 multiplies the current token
    z: torch.Tensor           # [T, H, 128] bf16
    A: torch.Tensor           # [H] fp32
    b: torch.Tensor           # [H, 128] fp32
    beta_logit: torch.Tensor  # [T, H] bf16
    g: torch.Tensor           # [T, H, 128] bf16 output-gate pre-activation
    S0: Optional[torch.Tensor]
    cu_seqlens: torch.Tensor  # [N+1] int32


def varlen_lengths(n: int = 16, lo: int = 1024, hi: int = 65536, seed: int = BASE_SEED + 5):
    """n lengths log-uniform in [lo, hi] (rounded)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    u = torch.rand((n,), generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))))
            for x in u]


def layer_inputs(lengths: Sequence[int], H: int, seed: int = BASE_SEED + 5,
                 s0_std: Optional[float] = None, device="cpu") -> LayerInputs:
    g = _gen(seed, device)
    T = int(sum(lengths))
    bf = torch.bfloat16
    qp = _randn((T, H, D), g, device).to(bf)
    kp = _randn((T, H, D), g, device).to(bf)
    vp = _randn((T, H, D), g, device).to(bf)
    conv_w = _randn((3, H * D, 4), g, device, 0.0, 0.5)
    z = _randn((T, H, D), g, device).to(bf)
    A = _randn((H,), g, device, 0.0, 0.5)
    b = torch.zeros((H, D), dtype=torch.float32, device=device)
    beta_logit = _randn((T, H), g, device).to(bf)
    gg = _randn((T, H, D), g, device).to(bf)
    S0 = None
    if s0_std is not None:
        S0 = _randn((len(lengths), H, D, D), g, device, 0.0, s0_std)
    return LayerInputs(qp, kp, vp, conv_w, z, A, b, beta_logit, gg, S0,
                       cu_from_lengths(lengths, device))


@dataclass
class DecodeLayerInputs:
    qp: torch.Tensor          # [B, H, 128] bf16, this token's pre-convolution projections
    kp: torch.Tensor
    vp: torch.Tensor
    conv_w: torch.Tensor      # [3, H*128, 4] fp32
    z: torch.Tensor           # [B, H, 128] bf16
    A: torch.Tensor           # [H] fp32
    b: torch.Tensor           # [H, 128] fp32 (zero)
    beta_logit: torch.Tensor  # [B, H] bf16
    g: torch.Tensor           # [B, H, 128] bf16
    slot: torch.Tensor        # [B] int32, distinct rows of the pools
    S_pool: torch.Tensor      # [P, H, 128, 128] fp32
    conv_pool: torch.Tensor   # [P, 3, 3, H, 128] bf16 (previous pre-convolution inputs)


def decode_layer_inputs(B: int, H: int, P: int, seed: int = BASE_SEED + 6,
                        s_std: float = 0.1, device="cpu") -> DecodeLayerInputs:
    """One decode token per request, with the distributions of the layer-core workload
    (pre-projection inputs ~N(0,1) bf16, conv w ~N(0,0.5), A ~N(0,0.5), b = 0,
    beta logit ~N(0,1), g ~N(0,1)); the requests sit in B distinct, shuffled rows of
    pools of P rows (state ~N(0, s_std), convolution history ~N(0,1) bf16)."""
    if P < B:
        raise ValueError("the pools need at least one row per request")
    g = _gen(seed, device)
    bf = torch.bfloat16
    qp = _randn((B, H, D), g, device).to(bf)
    kp = _randn((B, H, D), g, device).to(bf)
    vp = _randn((B, H, D), g, device).to(bf)
    conv_w = _randn((3, H * D, 4), g, device, 0.0, 0.5)
    z = _randn((B, H, D), g, device).to(bf)
    A = _randn((H,), g, device, 0.0, 0.5)
    b = torch.zeros((H, D), dtype=torch.float32, device=device)
    beta_logit = _randn((B, H), g, device).to(bf)
    gg = _randn((B, H, D), g, device).to(bf)
    slot = torch.randperm(P, generator=g, device=device)[:B].to(torch.int32)
    S_pool = _randn((P, H, D, D), g, device, 0.0, s_std)
    conv_pool = _randn((P, 3, 3, H, D), g, device).to(bf)
    return DecodeLayerInputs(qp, kp, vp, conv_w, z, A, b, beta_logit, gg, slot, S_pool, conv_pool)


@dataclass
class DecodeLayerTokensInputs:
    qp: torch.Tensor          # [T, H, 128] bf16, the requests' tokens packed
    kp: torch.Tensor
    vp: torch.Tensor
    conv_w: torch.Tensor      # [3, H*128, 4] fp32
    z: torch.Tensor           # [T, H, 128] bf16
    A: torch.Tensor           # [H] fp32
    b: torch.Tensor           # [H, 128] fp32 (zero)
    beta_logit: torch.Tensor  # [T, H] bf16
    g: torch.Tensor           # [T, H, 128] bf16
    cu_tokens: torch.Tensor   # [B+1] int32
    slot: torch.Tensor        # [B] int32, distinct shuffled rows of the pools
    S_pool: torch.Tensor      # [P, H, 128, 128] fp32
    conv_pool: torch.Tensor   # [P, 3, 3, H, 128] bf16


def decode_layer_tokens_inputs(lengths: Sequence[int], H: int, P: int, seed: int = BASE_SEED + 8,
                               s_std: float = 0.1, device="cpu") -> DecodeLayerTokensInputs:
    """A few tokens per request through the layer core, with the layer-core workload's
    distributions (as decode_layer_inputs), the requests in shuffled rows of P-row pools."""
    B = len(lengths)
    if P < B:
        raise ValueError("the pools need at least one row per request")
    g = _gen(seed, device)
    T = int(sum(lengths))
    bf = torch.bfloat16
    qp = _randn((T, H, D), g, device).to(bf)
    kp = _randn((T, H, D), g, device).to(bf)
    vp = _randn((T, H, D), g, device).to(bf)
    conv_w = _randn((3, H * D, 4), g, device, 0.0, 0.5)
    z = _randn((T, H, D), g, device).to(bf)
    A = _randn((H,), g, device, 0.0, 0.5)
    b = torch.zeros((H, D), dtype=torch.float32, device=device)
    beta_logit = _randn((T, H), g, device).to(bf)
    gg = _randn((T, H, D), g, device).to(bf)
    slot = torch.randperm(P, generator=g, device=device)[:B].to(torch.int32)
    S_pool = _randn((P, H, D, D), g, device, 0.0, s_std)
    conv_pool = _randn((P, 3, 3, H, D), g, device).to(bf)
    return DecodeLayerTokensInputs(qp, kp, vp, conv_w, z, A, b, beta_logit, gg,
                                   cu_from_lengths(lengths, device), slot, S_pool, conv_pool)


@dataclass
class DecodeTokensInputs:
    q: torch.Tensor           # [T, H, 128] dtype, the requests' tokens packed
    k: torch.Tensor
    v: torch.Tensor
    log_alpha: torch.Tensor   # [T, H, 128] fp32, in (-5, 0)
    beta: torch.Tensor        # [T, H] fp32
    cu_tokens: torch.Tensor   # [B+1] int32
    slot: torch.Tensor        # [B] int32, distinct shuffled rows of the pool
    S_pool: torch.Tensor      # [P, H, 128, 128] fp32


def decode_tokens_inputs(lengths: Sequence[int], H: int, P: int, dtype=torch.bfloat16,
                         seed: int = BASE_SEED + 7, x_std: float = 2.0, s_std: float = 0.1,
                         device="cpu") -> DecodeTokensInputs:
    """A few tokens per request (a speculative draft), with the decode workload's
    distributions; request b has lengths[b] tokens and its state in row slot[b] of a
    P-row pool (state ~N(0, s_std))."""
    B = len(lengths)
    if P < B:
        raise ValueError("the pool needs at least one row per request")
    g = _gen(seed, device)
    T = int(sum(lengths))
    q = _unit_rows(_randn((T, H, D), g, device)).to(dtype)
    k = _unit_rows(_randn((T, H, D), g, device)).to(dtype)
    v = _randn((T, H, D), g, device).to(dtype)
    la = torch.sigmoid(_randn((T, H, D), g, device, 0.0, x_std)).mul_(-5.0)
    beta = torch.sigmoid(_randn((T, H), g, device))
    slot = torch.randperm(P, generator=g, device=device)[:B].to(torch.int32)
    S_pool = _randn((P, H, D, D), g, device, 0.0, s_std)
    return DecodeTokensInputs(q, k, v, la.contiguous(), beta.contiguous(),
                              cu_from_lengths(lengths, device), slot, S_pool)


def workload(index: int, device="cpu"):
    """The five named workloads (see the module docstring)."""
    seed = BASE_SEED + index
    if index == 1:
        return prefill_inputs([256], 2, torch.float32, seed, 0.0, 1.0, None, device)
    if index == 2:
        return prefill_inputs([8192], 96, torch.bfloat16, seed, 0.0, 2.0, None, device)
    if index == 3:
        return decode_inputs(256, 96, torch.bfloat16, seed, 0.0, 2.0, 0.1, device)
    if index == 4:
        return prefill_inputs([131072], 96, torch.bfloat16, seed, 1.0, 1.0, 0.1, device)
    if index == 5:
        return layer_inputs(varlen_lengths(seed=seed), 96, seed, None, device)
    raise ValueError(f"unknown workload {index}")
