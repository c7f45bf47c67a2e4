"""DeltaNet delta rule on the GPU vs the float64 oracle.

Small cases cover ragged chunk tails, every supported chunk length and head
size, odd B*H, start states and aliasing S_out = S0; the page-sized workload
(B=8, H=16, T=8192, d=128, chunk 64) runs at full size and is checked on
sampled heads replayed in full by the oracle.
"""
import numpy as np
import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


def _gpu(inp):
    return [x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)]


@pytest.mark.parametrize("dtype,B,H,T,dk,dv,chunk,with_S0", [
    ("f32", 1, 1, 1, 32, 32, 64, False),
    ("f32", 1, 3, 15, 64, 64, 16, True),
    ("f32", 3, 1, 64, 128, 128, 64, False),
    ("f32", 1, 1, 65, 32, 64, 32, True),
    ("f32", 2, 1, 200, 64, 32, 64, True),
    ("bf16", 1, 1, 17, 128, 128, 16, False),
    ("bf16", 1, 3, 130, 128, 128, 64, True),
    ("bf16", 2, 2, 257, 64, 64, 32, False),
])
def test_small_parity(cuda_lib, oracle_mod, dtype, B, H, T, dk, dv, chunk, with_S0):
    inp = synth.delta_inputs(B, H, T, dk, dv, dtype=dtype, seed=T + dk)
    q, k, v, beta = _gpu(inp)
    S0 = None
    if with_S0:
        S0 = (torch.randn(B, H, dk, dv, generator=torch.Generator().manual_seed(3)) * 0.1)
    S_out = torch.empty(B, H, dk, dv, device="cuda")
    y = cuda_lib.delta_rule_forward(q, k, v, beta, chunk=chunk, S0=None if S0 is None else S0.cuda(),
                                    S_out=S_out)
    torch.cuda.synchronize()
    ref = oracle_mod.delta(inp.q, inp.k, inp.v, inp.beta, S0=S0, want_state=True)
    check_parity(to_np(y), ref["y"], dtype, "delta y")
    check_parity(to_np(S_out), ref["S"], dtype, "delta S")


# Shapes served by the tensor-core path (bf16, chunk 64, d_v 64 or 128): ragged
# tails, a single token, exact chunk multiples, both key and value widths,
# start states (updated in place).
@pytest.mark.parametrize("B,H,T,dk,dv,with_S0", [
    (1, 1, 1, 128, 128, False),
    (1, 2, 63, 128, 128, True),
    (2, 1, 64, 128, 128, False),
    (1, 1, 65, 64, 128, True),
    (1, 3, 200, 128, 128, True),
    (2, 2, 333, 64, 128, False),
    (1, 1, 1024, 128, 128, True),
    (1, 1, 1, 64, 64, False),
    (1, 2, 63, 64, 64, True),
    (2, 2, 333, 128, 64, True),
    (1, 1, 1024, 64, 64, True),
])
def test_tensor_core_shapes(cuda_lib, oracle_mod, B, H, T, dk, dv, with_S0):
    inp = synth.delta_inputs(B, H, T, dk, dv, dtype="bf16", seed=T + 7 * dk + dv)
    q, k, v, beta = _gpu(inp)
    S0 = (torch.randn(B, H, dk, dv, generator=torch.Generator().manual_seed(9)) * 0.1) if with_S0 else None
    S = None if S0 is None else S0.clone().cuda()
    S_out = S if S is not None else torch.empty(B, H, dk, dv, device="cuda")  # in place when given
    y = cuda_lib.delta_rule_forward(q, k, v, beta, chunk=64, S0=S, S_out=S_out)
    torch.cuda.synchronize()
    cuda_lib.check_device_errors()
    ref = oracle_mod.delta(inp.q, inp.k, inp.v, inp.beta, S0=S0, want_state=True)
    check_parity(to_np(y), ref["y"], "bf16", "delta y (tensor cores)")
    check_parity(to_np(S_out), ref["S"], "bf16", "delta S (tensor cores)")


def test_in_place_state_and_chunk_independence(cuda_lib, oracle_mod):
    inp = synth.delta_inputs(2, 2, 150, 64, 64, dtype="f32", seed=5)
    q, k, v, beta = _gpu(inp)
    S0 = torch.randn(2, 2, 64, 64, generator=torch.Generator().manual_seed(4)) * 0.1
    ys = []
    for chunk in (16, 32, 64):
        S = S0.clone().cuda()
        ys.append(to_np(cuda_lib.delta_rule_forward(q, k, v, beta, chunk=chunk, S0=S, S_out=S)))
    torch.cuda.synchronize()
    ref = oracle_mod.delta(inp.q, inp.k, inp.v, inp.beta, S0=S0, want_state=True)
    for y in ys:
        check_parity(y, ref["y"], "f32", "chunk independence")
    check_parity(to_np(S), ref["S"], "f32", "in-place S")


def test_full_size_workload_sampled(cuda_lib, oracle_mod):
    w = synth.WORKLOADS["delta_bf16_B8_H16_T8192_d128_C64"]
    d = w.dims
    inp = synth.delta_inputs(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], dtype=d["dtype"], seed=w.seed)
    q, k, v, beta = _gpu(inp)
    y = cuda_lib.delta_rule_forward(q, k, v, beta, chunk=d["chunk"])
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    for b, h in [(0, 0), (5, 11)]:
        sl = lambda x: x[b:b + 1, h:h + 1]  # noqa: E731
        ref = oracle_mod.delta(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.beta))["y"]
        check_parity(to_np(y[b:b + 1, h:h + 1]), ref, "bf16", f"delta unit {b},{h}")
