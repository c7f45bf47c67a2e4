"""DeltaNet single-token decode on the GPU vs the float64 oracle.

A decode step is the delta rule applied to one token from a stored state, so
the oracle for `steps` decode calls is its delta-rule recurrence run over the
same `steps` tokens from the same start state.  Cases: every head-size pair
in both element types with odd sequence and head counts, a hand-off from a
GPU prefill, beta = 0 (state untouched bit for bit), beta = 1 with a
unit-norm key (the state then maps k to v), and the 256-sequence workload at
full size on sampled (sequence, head) units.
"""
import numpy as np
import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


def _run_decode(cuda_lib, dec, S):
    """All steps of `dec` on the GPU, S updated in place; y stacked [S,H,steps,d_v]."""
    ys = []
    for i in range(dec.q.shape[0]):
        ys.append(cuda_lib.delta_decode_step(S, dec.q[i].cuda(), dec.k[i].cuda(), dec.v[i].cuda(),
                                             dec.beta[i].cuda()))
    torch.cuda.synchronize()
    return torch.stack(ys, dim=2)


def _seq(x):
    """[steps, S, H, ...] -> [S, H, steps, ...] (the oracle's token axis)."""
    return x.movedim(0, 2).contiguous()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128), (32, 128), (128, 32), (64, 64)])
def test_decode_matches_oracle(cuda_lib, oracle_mod, dtype, dk, dv):
    dec = synth.delta_decode_inputs(5, 3, 5, dk, dv, dtype=dtype, seed=dk + 3 * dv)
    S = dec.S0.clone().cuda()
    y = _run_decode(cuda_lib, dec, S)
    ref = oracle_mod.delta(_seq(dec.q), _seq(dec.k), _seq(dec.v), _seq(dec.beta), S0=dec.S0,
                           want_state=True)
    check_parity(to_np(y), ref["y"], dtype, f"delta decode y d_k={dk} d_v={dv}")
    check_parity(to_np(S), ref["S"], dtype, f"delta decode S d_k={dk} d_v={dv}")


def test_decode_continues_a_gpu_prefill(cuda_lib, oracle_mod):
    T0, n, B, H, d = 130, 4, 2, 3, 128
    inp = synth.delta_inputs(B, H, T0 + n, d, d, dtype="bf16", seed=11)
    q, k, v, beta = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.beta)]
    S = torch.empty(B, H, d, d, device="cuda")
    y0 = cuda_lib.delta_rule_forward(q[:, :, :T0].contiguous(), k[:, :, :T0].contiguous(),
                                     v[:, :, :T0].contiguous(), beta[:, :, :T0].contiguous(), chunk=64,
                                     S_out=S)
    ys = [cuda_lib.delta_decode_step(S, q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                     v[:, :, t].contiguous(), beta[:, :, t].contiguous())
          for t in range(T0, T0 + n)]
    torch.cuda.synchronize()
    cuda_lib.check_device_errors()
    ref = oracle_mod.delta(inp.q, inp.k, inp.v, inp.beta, want_state=True)
    check_parity(to_np(y0), ref["y"][:, :, :T0], "bf16", "prefill part")
    check_parity(to_np(torch.stack(ys, dim=2)), ref["y"][:, :, T0:], "bf16", "decode part")
    check_parity(to_np(S), ref["S"], "bf16", "state after prefill + decode")


def test_beta_zero_leaves_state_bitwise(cuda_lib, oracle_mod):
    dec = synth.delta_decode_inputs(1, 2, 3, 64, 64, dtype="f32", seed=5)
    beta = torch.zeros(2, 3, device="cuda")
    S = dec.S0.clone().cuda()
    y = cuda_lib.delta_decode_step(S, dec.q[0].cuda(), dec.k[0].cuda(), dec.v[0].cuda(), beta)
    torch.cuda.synchronize()
    assert torch.equal(S.cpu(), dec.S0)
    ref = oracle_mod.delta(_seq(dec.q), _seq(dec.k), _seq(dec.v), np.zeros((2, 3, 1)), S0=dec.S0)
    check_parity(to_np(y), ref["y"][:, :, 0], "f32", "beta = 0 read")


def test_beta_one_unit_key_maps_key_to_value(cuda_lib):
    """Page property: with beta = 1 the written key reads back its value."""
    dec = synth.delta_decode_inputs(1, 4, 2, 128, 64, dtype="f32", seed=8)
    beta = torch.ones(4, 2, device="cuda")
    S = dec.S0.clone().cuda()
    k = dec.k[0].cuda()
    cuda_lib.delta_decode_step(S, dec.q[0].cuda(), k, dec.v[0].cuda(), beta)
    torch.cuda.synchronize()
    readback = torch.einsum("shd,shde->she", k.double(), S.double())
    err = (readback.cpu() - dec.v[0].double()).norm() / dec.v[0].double().norm()
    assert err < 1e-5, float(err)


def test_full_size_workload_sampled(cuda_lib, oracle_mod):
    w = synth.WORKLOADS["delta_decode_bf16_S256_H16_d128_steps64"]
    d = w.dims
    dec = synth.delta_decode_inputs(3, d["S"], d["H"], d["d_k"], d["d_v"], dtype=d["dtype"], seed=w.seed)
    S = dec.S0.clone().cuda()
    y = _run_decode(cuda_lib, dec, S)
    assert torch.isfinite(y.float()).all()
    for s, h in [(0, 0), (137, 9), (255, 15)]:
        sl = lambda x: _seq(x)[s:s + 1, h:h + 1]  # noqa: E731
        ref = oracle_mod.delta(sl(dec.q), sl(dec.k), sl(dec.v), sl(dec.beta), S0=dec.S0[s:s + 1, h:h + 1],
                               want_state=True)
        check_parity(to_np(y[s:s + 1, h:h + 1]), ref["y"], "bf16", f"decode unit {s},{h}")
        check_parity(to_np(S[s:s + 1, h:h + 1]), ref["S"], "bf16", f"decode state {s},{h}")
