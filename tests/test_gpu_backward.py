"""Backward passes on the GPU vs the float64 oracle's reverse-mode gradients.

tc_layer_backward and delta_rule_backward are compared gradient by gradient
with oracle.tc_backward / oracle.delta_backward on the same seeded inputs and
upstream gradient dy.  Bars as for the forward: fp32 inputs -> relative L2
<= 1e-5 per gradient tensor; bf16 inputs (fp32 arithmetic, bf16 gradients)
-> RMS(error) <= 2e-2 of the gradient's RMS.  The per-head scalars (dlambda,
deta, dgate) are fp32 in both cases and held to the fp32 bar.  Cases cover
ragged tails, one to several chunks, windows of 1, around the chunk length
and past the sequence (no eviction), lambda at 0 and 1, unequal d_k / d_v,
and the headline and DeltaNet head sizes over long sequences.
"""
import numpy as np
import pytest
import torch

from helpers import TOL_F32_REL_L2, check_parity, rel_l2, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status(cuda_lib):
    cuda_lib.check_device_errors()
    yield
    cuda_lib.check_device_errors()


def _dy(shape, dtype, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed)).to(dtype).contiguous()


def _scalars_ok(got, ref, what):
    err = rel_l2(got, ref)
    print(f"parity {what}: rel L2 {err:.3e} (bar {TOL_F32_REL_L2 * 10})")
    # sums over every token of the batch, accumulated in fp32 in a different
    # order than the oracle: one decade above the per-element fp32 bar
    assert err <= TOL_F32_REL_L2 * 10, f"{what}: rel L2 {err:.3e}"


TC_CASES = [
    # dtype, B, H, T, d_k, d_v, W, lam, eta
    ("f32", 1, 1, 1, 32, 32, 1, None, None),
    ("f32", 1, 2, 37, 32, 64, 1, None, None),
    ("f32", 2, 1, 70, 64, 64, 16, None, None),
    ("f32", 1, 1, 200, 64, 32, 64, None, None),
    ("f32", 1, 2, 300, 32, 32, 65, 1.0, 1.0),
    ("f32", 1, 1, 130, 128, 128, 129, None, None),
    ("f32", 1, 1, 257, 64, 64, 1, 0.0, 0.5),
    ("f32", 2, 2, 100, 32, 32, 300, None, None),     # W > T: no eviction, L2 gradient 0
    ("bf16", 1, 2, 333, 64, 64, 63, None, None),
    ("bf16", 2, 1, 500, 128, 128, 100, None, None),
    ("bf16", 1, 1, 777, 64, 128, 300, None, None),
    ("bf16", 3, 1, 129, 128, 64, 64, None, None),
    # bf16 d = 64 takes the tensor-core dK/dV kernel: W a multiple of the
    # 128-key tile with a ragged tail, a single token, and W > T
    ("bf16", 2, 1, 300, 64, 64, 128, None, None),
    ("bf16", 1, 1, 1, 64, 64, 1, None, None),
    ("bf16", 1, 2, 200, 64, 64, 256, None, None),
]


@pytest.mark.parametrize("dtype,B,H,T,dk,dv,W,lam,eta", TC_CASES)
def test_tc_backward_matches_oracle(cuda_lib, oracle_mod, dtype, B, H, T, dk, dv, W, lam, eta):
    inp = synth.tc_inputs(B, H, T, dk, dv, W, dtype=dtype, seed=T + W, lam=lam, eta=eta)
    dy = _dy((B, H, T, dv), inp.q.dtype, 7 + T)
    g = cuda_lib.tc_layer_backward(*[x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)], W,
                                   dy.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.tc_backward(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, dy)
    for got, name in zip(g[:3], ("dq", "dk", "dv")):
        check_parity(to_np(got), ref[name], dtype, f"tc backward {name} {dtype} B{B} H{H} T{T} d{dk}/{dv} W{W}")
    for got, name in zip(g[3:], ("dlam", "deta", "dgate")):
        if np.all(ref[name] == 0.0):
            assert np.all(to_np(got) == 0.0), name
        else:
            _scalars_ok(to_np(got), ref[name], f"tc backward {name}")


def test_tc_backward_headline_heads_full_length(cuda_lib, oracle_mod):
    """Two heads of the headline workload at its full length (T = 4096,
    d = 64, W = 512, 64 chunks): every gradient element checked."""
    d = synth.WORKLOADS["tc_bf16_B4_H8_T4096_d64_W512"].dims
    inp = synth.tc_inputs(1, 2, d["T"], 64, 64, d["W"], dtype="bf16", seed=77)
    dy = _dy((1, 2, d["T"], 64), torch.bfloat16, 78)
    g = cuda_lib.tc_layer_backward(*[x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)],
                                   d["W"], dy.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.tc_backward(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, d["W"], dy)
    for got, name in zip(g[:3], ("dq", "dk", "dv")):
        check_parity(to_np(got), ref[name], "bf16", f"tc backward headline heads {name}")
    for got, name in zip(g[3:], ("dlam", "deta", "dgate")):
        _scalars_ok(to_np(got), ref[name], f"tc backward headline heads {name}")


DELTA_CASES = [
    # dtype, B, H, T, d_k, d_v, with S0, with dS_T
    ("f32", 1, 1, 1, 32, 32, False, False),
    ("f32", 2, 1, 45, 64, 32, True, False),
    ("f32", 1, 2, 130, 32, 64, False, True),
    ("f32", 1, 1, 300, 128, 128, True, True),
    ("bf16", 2, 2, 200, 64, 64, True, False),
    ("bf16", 1, 1, 257, 128, 64, False, False),
    ("bf16", 1, 2, 100, 32, 128, True, True),
]


@pytest.mark.parametrize("dtype,B,H,T,dk,dv,with_S0,with_dST", DELTA_CASES)
def test_delta_backward_matches_oracle(cuda_lib, oracle_mod, dtype, B, H, T, dk, dv, with_S0, with_dST):
    inp = synth.delta_inputs(B, H, T, dk, dv, dtype=dtype, seed=T + dk)
    gen = torch.Generator().manual_seed(T)
    S0 = torch.randn(B, H, dk, dv, generator=gen) / np.sqrt(dk) if with_S0 else None
    dST = torch.randn(B, H, dk, dv, generator=gen) if with_dST else None
    dy = _dy((B, H, T, dv), inp.q.dtype, 11 + T)
    g = cuda_lib.delta_rule_backward(*[x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)], dy.cuda(),
                                     S0=None if S0 is None else S0.cuda(),
                                     dS_T=None if dST is None else dST.cuda(), want_dS0=True)
    torch.cuda.synchronize()
    ref = oracle_mod.delta_backward(inp.q, inp.k, inp.v, inp.beta, dy, S0=S0, dS_T=dST)
    for got, name in zip(g[:3], ("dq", "dk", "dv")):
        check_parity(to_np(got), ref[name], dtype, f"delta backward {name} {dtype} T{T} d{dk}/{dv}")
    check_parity(to_np(g[3]), ref["dbeta"], "f32" if dtype == "f32" else "bf16", "delta backward dbeta")
    check_parity(to_np(g[4]), ref["dS0"], "f32" if dtype == "f32" else "bf16", "delta backward dS0")


def test_delta_backward_long_sequence_d128(cuda_lib, oracle_mod):
    """The DeltaNet workload's head size over a long sequence (T = 2048,
    d = 128): the reverse walk reconstructs 2048 states from the last one."""
    inp = synth.delta_inputs(1, 2, 2048, 128, 128, dtype="bf16", seed=91)
    dy = _dy((1, 2, 2048, 128), torch.bfloat16, 92)
    g = cuda_lib.delta_rule_backward(*[x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)], dy.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.delta_backward(inp.q, inp.k, inp.v, inp.beta, dy)
    for got, name in zip(g[:4], ("dq", "dk", "dv", "dbeta")):
        check_parity(to_np(got), ref[name], "bf16", f"delta backward long {name}")


def test_delta_backward_fp32_long_sequence(cuda_lib, oracle_mod):
    """fp32 over 1024 tokens: the rounding of the exact state reversal stays
    inside the fp32 bar."""
    inp = synth.delta_inputs(1, 1, 1024, 64, 64, dtype="f32", seed=93)
    dy = _dy((1, 1, 1024, 64), torch.float32, 94)
    g = cuda_lib.delta_rule_backward(*[x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)], dy.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.delta_backward(inp.q, inp.k, inp.v, inp.beta, dy)
    for got, name in zip(g[:4], ("dq", "dk", "dv", "dbeta")):
        check_parity(to_np(got), ref[name], "f32", f"delta backward fp32 long {name}")
