"""Seeded synthetic inputs for the outer-product associative-memory layers.

This module only draws random tensors: it holds none of the layers' arithmetic,
so both the CUDA path and the float64 oracle can be fed from it.  Every
generator uses a torch CPU ``Generator`` so a seed gives the same tensors on
any machine.  Draw order is fixed: q, k, v, then per-token / per-head scalars.

Recipes (one per workload of the pages):

* Tensor Cache layer (gist.science 2605.22884, "Tensor Cache", Methodology 1):
  q and k are standard Gaussian rows scaled to unit L2 norm, v is standard
  Gaussian; per-head decay lambda ~ U[0.9, 0.999], write rate eta ~ U[0.1, 1],
  gate g ~ N(0, 1) (or fixed values when given).
* DeltaNet delta rule (molayo1419.me, "DeltaNet: writing the prediction
  error"): k unit-norm Gaussian, q and v Gaussian, beta_t = logistic(N(0,1))
  per token and head, so beta lies in (0, 1) as the page requires.  Decode
  steps draw tokens the same way and start from a Gaussian state with
  entries of variance 1/d_k.
* BDH-style linear attention (ainews.random.gg BDH post, "low-rank
  factorisation plus ReLU thresholding"): k = ReLU(x U_h - theta) and
  q = ReLU(x' U_h - theta) with x, x' ~ N(0, I_256) per token, one
  U_h ~ N(0, 1/256)^{256 x N} per head shared by q and k, and theta the 95th
  percentile of N(0,1) so about 5% of the entries are non-zero.

bf16 inputs are drawn in float32 and rounded to bf16 (round to nearest even);
the oracle then reads the rounded values, so a tolerance measures kernel error
only.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# 95th percentile of the standard normal: x U_h has N(0,1) entries, so
# thresholding at this value keeps about 5% of them.
BDH_THETA_5PCT = 1.6448536269514722

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    """Scale each last-dim row of a Gaussian draw to unit L2 norm (input prep)."""
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def _round(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(_DT[dtype]).contiguous()


# ---------------------------------------------------------------- Tensor Cache
@dataclass
class TCInputs:
    q: torch.Tensor          # [B,H,T,d_k] dtype
    k: torch.Tensor          # [B,H,T,d_k]
    v: torch.Tensor          # [B,H,T,d_v]
    lam: torch.Tensor        # [H] float32, decay lambda
    eta: torch.Tensor        # [H] float32, write rate eta
    gate: torch.Tensor       # [H] float32, gate logit g
    W: int
    dtype: str


def tc_inputs(B, H, T, d_k, d_v, W, dtype="bf16", seed=0, lam=None, eta=None,
              gate=None) -> TCInputs:
    g = _gen(seed)
    q = _unit_rows(torch.randn(B, H, T, d_k, generator=g))
    k = _unit_rows(torch.randn(B, H, T, d_k, generator=g))
    v = torch.randn(B, H, T, d_v, generator=g)
    lam_t = (torch.empty(H).uniform_(0.9, 0.999, generator=g) if lam is None
             else torch.full((H,), float(lam)))
    eta_t = (torch.empty(H).uniform_(0.1, 1.0, generator=g) if eta is None
             else torch.full((H,), float(eta)))
    gate_t = (torch.randn(H, generator=g) if gate is None
              else torch.full((H,), float(gate)))
    return TCInputs(_round(q, dtype), _round(k, dtype), _round(v, dtype),
                    lam_t.float().contiguous(), eta_t.float().contiguous(),
                    gate_t.float().contiguous(), int(W), dtype)


@dataclass
class TCDecodeInputs:
    q: torch.Tensor          # [steps, S, H, d_k]
    k: torch.Tensor          # [steps, S, H, d_k]
    v: torch.Tensor          # [steps, S, H, d_v]
    dtype: str


def tc_decode_inputs(steps, S, H, d_k, d_v, dtype="bf16", seed=103) -> TCDecodeInputs:
    g = _gen(seed)
    q = _unit_rows(torch.randn(steps, S, H, d_k, generator=g))
    k = _unit_rows(torch.randn(steps, S, H, d_k, generator=g))
    v = torch.randn(steps, S, H, d_v, generator=g)
    return TCDecodeInputs(_round(q, dtype), _round(k, dtype), _round(v, dtype), dtype)


def tc_decode_state(S, H, W, d_k, d_v, pos, dtype="bf16", seed=104) -> dict:
    """A full Tensor Cache streaming state to start decode steps from, for
    timing: ring keys unit rows and ring values Gaussian (as tokens are drawn),
    A Gaussian with entries of variance 1/d_k, every sequence at position
    ``pos`` (>= W, so the ring is full and every step evicts)."""
    g = _gen(seed)
    ring_k = _unit_rows(torch.randn(S, H, W, d_k, generator=g))
    ring_v = torch.randn(S, H, W, d_v, generator=g)
    A = torch.randn(S, H, d_k, d_v, generator=g) / math.sqrt(d_k)
    return dict(ring_k=_round(ring_k, dtype), ring_v=_round(ring_v, dtype), A=A.float().contiguous(),
                pos=torch.full((S,), int(pos), dtype=torch.int64))


# ---------------------------------------------------------------- DeltaNet
@dataclass
class DeltaInputs:
    q: torch.Tensor          # [B,H,T,d_k]
    k: torch.Tensor          # [B,H,T,d_k]  unit rows
    v: torch.Tensor          # [B,H,T,d_v]
    beta: torch.Tensor       # [B,H,T] float32 in (0,1)
    dtype: str


def delta_inputs(B, H, T, d_k, d_v, dtype="bf16", seed=2) -> DeltaInputs:
    g = _gen(seed)
    q = torch.randn(B, H, T, d_k, generator=g)
    k = _unit_rows(torch.randn(B, H, T, d_k, generator=g))
    v = torch.randn(B, H, T, d_v, generator=g)
    beta = torch.sigmoid(torch.randn(B, H, T, generator=g))
    return DeltaInputs(_round(q, dtype), _round(k, dtype), _round(v, dtype),
                       beta.float().contiguous(), dtype)


@dataclass
class DeltaDecodeInputs:
    q: torch.Tensor          # [steps, S, H, d_k]
    k: torch.Tensor          # [steps, S, H, d_k]  unit rows
    v: torch.Tensor          # [steps, S, H, d_v]
    beta: torch.Tensor       # [steps, S, H] float32 in (0,1)
    S0: torch.Tensor         # [S, H, d_k, d_v] float32 key-major start state
    dtype: str


def delta_decode_inputs(steps, S, H, d_k, d_v, dtype="bf16", seed=104) -> DeltaDecodeInputs:
    """Single-token DeltaNet steps for S sequences: tokens drawn as in
    ``delta_inputs``; the start state is Gaussian with entries of variance
    1/d_k, the scale at which a unit-norm key reads out a unit-variance value."""
    g = _gen(seed)
    q = torch.randn(steps, S, H, d_k, generator=g)
    k = _unit_rows(torch.randn(steps, S, H, d_k, generator=g))
    v = torch.randn(steps, S, H, d_v, generator=g)
    beta = torch.sigmoid(torch.randn(steps, S, H, generator=g))
    S0 = torch.randn(S, H, d_k, d_v, generator=g) / math.sqrt(d_k)
    return DeltaDecodeInputs(_round(q, dtype), _round(k, dtype), _round(v, dtype),
                             beta.float().contiguous(), S0.float().contiguous(), dtype)


# ---------------------------------------------------------------- BDH
@dataclass
class SparseInputs:
    q: torch.Tensor          # [B,H,T,N] float32, non-negative, ~5% non-zero
    k: torch.Tensor          # [B,H,T,N]
    v: torch.Tensor          # [B,H,T,d_v]
    theta: float


def sparse_inputs(B, H, T, N, d_v, seed=4, rank=256, theta=BDH_THETA_5PCT) -> SparseInputs:
    g = _gen(seed)
    xq = torch.randn(B, H, T, rank, generator=g)
    xk = torch.randn(B, H, T, rank, generator=g)
    v = torch.randn(B, H, T, d_v, generator=g)
    U = torch.randn(H, rank, N, generator=g) / math.sqrt(rank)
    q = torch.relu(torch.einsum("bhtr,hrn->bhtn", xq, U) - theta)
    k = torch.relu(torch.einsum("bhtr,hrn->bhtn", xk, U) - theta)
    return SparseInputs(q.contiguous(), k.contiguous(), v.contiguous(), float(theta))


@dataclass
class KeygenInputs:
    xq: torch.Tensor         # [B,H,T,R] bf16 query-side token inputs
    xk: torch.Tensor         # [B,H,T,R] bf16 key-side token inputs
    U: torch.Tensor          # [H,R,N] bf16, one factor per head
    v: torch.Tensor          # [B,H,T,d_v] float32
    theta: float


def sparse_keygen_inputs(B, H, T, N, d_v, seed=5, rank=256, theta=BDH_THETA_5PCT) -> KeygenInputs:
    """The inputs of the BDH recipe before the ReLU threshold: x, x' ~ N(0, I_R)
    per token, U_h ~ N(0, 1/R)^{R x N} per head, v Gaussian; x and U rounded
    to bf16 (the tensor-core operand type) so that both sides read the same
    values.  The activations themselves are not formed here."""
    g = _gen(seed)
    xq = torch.randn(B, H, T, rank, generator=g)
    xk = torch.randn(B, H, T, rank, generator=g)
    v = torch.randn(B, H, T, d_v, generator=g)
    U = torch.randn(H, rank, N, generator=g) / math.sqrt(rank)
    return KeygenInputs(_round(xq, "bf16"), _round(xk, "bf16"), _round(U, "bf16"), v.contiguous(), float(theta))


# ---------------------------------------------------------------- workloads
@dataclass
class Workload:
    name: str
    kind: str                # "tc" | "tc_decode" | "delta" | "delta_decode" | "sparse"
    dims: dict = field(default_factory=dict)
    seed: int = 0


WORKLOADS = {
    # Tensor Cache layer forward, fp32, one head.
    "tc_fp32_T256_d32_W32": Workload(
        "tc_fp32_T256_d32_W32", "tc",
        dict(B=1, H=1, T=256, d_k=32, d_v=32, W=32, dtype="f32",
             lam=0.99, eta=0.5, gate=0.0), seed=0),
    # Tensor Cache layer prefill, bf16 inputs / fp32 state.
    "tc_bf16_B4_H8_T4096_d64_W512": Workload(
        "tc_bf16_B4_H8_T4096_d64_W512", "tc",
        dict(B=4, H=8, T=4096, d_k=64, d_v=64, W=512, dtype="bf16"), seed=1),
    # DeltaNet chunked prefill, bf16 inputs / fp32 state.
    "delta_bf16_B8_H16_T8192_d128_C64": Workload(
        "delta_bf16_B8_H16_T8192_d128_C64", "delta",
        dict(B=8, H=16, T=8192, d_k=128, d_v=128, chunk=64, dtype="bf16"), seed=2),
    # Long-context Tensor Cache prefill, then 64-sequence decode.
    "tc_bf16_B1_H16_T32768_d128_W2048": Workload(
        "tc_bf16_B1_H16_T32768_d128_W2048", "tc",
        dict(B=1, H=16, T=32768, d_k=128, d_v=128, W=2048, dtype="bf16"), seed=3),
    "tc_decode_bf16_S64_H16_d128_W2048_steps256": Workload(
        "tc_decode_bf16_S64_H16_d128_W2048_steps256", "tc_decode",
        dict(S=64, H=16, d_k=128, d_v=128, W=2048, steps=256, dtype="bf16",
             prefill="tc_bf16_B1_H16_T32768_d128_W2048"), seed=103),
    # DeltaNet single-token decode from a stored state (state 256 MiB, above L2).
    "delta_decode_bf16_S256_H16_d128_steps64": Workload(
        "delta_decode_bf16_S256_H16_d128_steps64", "delta_decode",
        dict(S=256, H=16, d_k=128, d_v=128, steps=64, dtype="bf16"), seed=104),
    # BDH-style linear attention, wide sparse non-negative keys, fp32.
    "bdh_fp32_B2_H4_T2048_N16384_dv256": Workload(
        "bdh_fp32_B2_H4_T2048_N16384_dv256", "sparse",
        dict(B=2, H=4, T=2048, N=16384, d_v=256), seed=4),
    # The same attention with the keys and queries generated on the GPU from
    # their 256-wide inputs (bf16 x and U, fp32 accumulation and state).
    "bdh_keygen_B2_H4_T2048_R256_N16384_dv256": Workload(
        "bdh_keygen_B2_H4_T2048_R256_N16384_dv256", "sparse_keygen",
        dict(B=2, H=4, T=2048, R=256, N=16384, d_v=256), seed=5),
}
