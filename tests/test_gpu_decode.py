"""Tensor Cache decode step on the GPU vs the float64 oracle.

Each case prefills T0 tokens (on the GPU through tc_layer_forward, in the
oracle through its own prefill), then runs single-token decode steps and
compares every step's output and the final state.  Covers rings that are not
yet full, rings that wrap during decode, W = 1, and the full-width decode
batch (64 sequences x 16 heads, W = 2048, d = 128) checked on sampled
sequences.
"""
import numpy as np
import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


def _prefill_state(cuda_lib, inp, S):
    """GPU prefill of a B=1 batch, then the state replicated to S sequences."""
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    B, H, T, dk = inp.q.shape
    dv = inp.v.shape[-1]
    st1 = cuda_lib.TCState(B, H, inp.W, dk, dv, dtype=q.dtype)
    cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, inp.W, state=st1)
    st = cuda_lib.TCState(S, H, inp.W, dk, dv, dtype=q.dtype)
    st.ring_k.copy_(st1.ring_k.expand(S, -1, -1, -1))
    st.ring_v.copy_(st1.ring_v.expand(S, -1, -1, -1))
    st.A.copy_(st1.A.expand(S, -1, -1, -1))
    st.pos.fill_(T)
    return st, (lam, eta, gate)


def _oracle_state(oracle_mod, inp, S):
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, inp.W, want_state=True)
    rep = lambda x: np.ascontiguousarray(np.repeat(x, S, axis=0))  # noqa: E731
    return dict(ring_k=rep(ref["ring_k"]), ring_v=rep(ref["ring_v"]), A=rep(ref["A"]),
                pos=np.full(S, inp.q.shape[2], dtype=np.int64))


@pytest.mark.parametrize("dtype,T0,steps,W,d,S,H", [
    ("f32", 5, 6, 8, 32, 3, 2),        # ring fills up during decode
    ("f32", 40, 5, 16, 64, 2, 1),
    ("f32", 9, 4, 1, 32, 2, 2),        # W = 1
    ("bf16", 100, 8, 64, 128, 3, 2),
    ("bf16", 600, 6, 256, 64, 5, 3),
    ("bf16", 1, 12, 8, 128, 2, 1),
])
def test_decode_matches_oracle(cuda_lib, oracle_mod, dtype, T0, steps, W, d, S, H):
    inp = synth.tc_inputs(1, H, T0, d, d, W, dtype=dtype, seed=T0 + W)
    dec = synth.tc_decode_inputs(steps, S, H, d, d, dtype=dtype, seed=T0 + 1)
    st, (lam, eta, gate) = _prefill_state(cuda_lib, inp, S)
    ys = []
    for i in range(steps):
        ys.append(cuda_lib.tc_decode_step(st, dec.q[i].cuda(), dec.k[i].cuda(), dec.v[i].cuda(),
                                          lam, eta, gate))
    torch.cuda.synchronize()
    y = np.stack([to_np(t) for t in ys])
    ref_y, ref_st = oracle_mod.tc_decode(_oracle_state(oracle_mod, inp, S), dec.q, dec.k, dec.v,
                                         inp.lam, inp.eta, inp.gate)
    check_parity(y, ref_y, dtype, "decode outputs")
    np.testing.assert_array_equal(to_np(st.ring_k), ref_st["ring_k"])
    np.testing.assert_array_equal(to_np(st.ring_v), ref_st["ring_v"])
    check_parity(to_np(st.A), ref_st["A"], dtype, "decode A")
    assert np.array_equal(st.pos.cpu().numpy(), ref_st["pos"])


def test_decode_full_width_batch_sampled(cuda_lib, oracle_mod):
    """64 sequences x 16 heads, W = 2048, d = 128 (the decode workload's
    per-step shape) from a prefill that has wrapped the ring; two sequences
    are replayed in the oracle."""
    H, W, d, S, T0, steps = 16, 2048, 128, 64, 2300, 3
    inp = synth.tc_inputs(1, H, T0, d, d, W, dtype="bf16", seed=77)
    dec = synth.tc_decode_inputs(steps, S, H, d, d, dtype="bf16", seed=78)
    st, (lam, eta, gate) = _prefill_state(cuda_lib, inp, S)
    ys = [cuda_lib.tc_decode_step(st, dec.q[i].cuda(), dec.k[i].cuda(), dec.v[i].cuda(), lam, eta, gate)
          for i in range(steps)]
    torch.cuda.synchronize()
    y = np.stack([to_np(t) for t in ys])
    pick = [0, 37]
    ost = _oracle_state(oracle_mod, inp, len(pick))
    ref_y, ref_st = oracle_mod.tc_decode(ost, dec.q[:, pick], dec.k[:, pick], dec.v[:, pick], inp.lam,
                                         inp.eta, inp.gate)
    check_parity(y[:, pick], ref_y, "bf16", "full-width decode")
    check_parity(to_np(st.A[pick]), ref_st["A"], "bf16", "full-width decode A")
