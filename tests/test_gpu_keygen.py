"""BDH attention with the keys and queries generated on the GPU
(sparse_linattn_keygen_forward) vs the float64 oracle: keys and queries from
oracle.bdh_keys (max(0, x U_h - theta) from the same bf16 x and U), then
oracle.sparse_linattn.  Bar: the fp32 path's relative L2 <= 1e-5 on y (and on
the final state when one is returned).  The GPU takes the threshold decision
on an fp32 accumulation of exact bf16 products; an entry that lands on the
other side of theta than in float64 is within rounding of theta, so its
value, and its effect on y, is below the bar.
"""
import numpy as np
import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status(cuda_lib):
    cuda_lib.check_device_errors()
    yield
    cuda_lib.check_device_errors()


CASES = [
    # B, H, T, R, N, d_v, theta (None: the 5% threshold)
    (1, 1, 1, 64, 128, 32, None),
    (1, 2, 200, 64, 512, 64, None),
    (2, 1, 129, 128, 1024, 32, None),
    (1, 2, 300, 256, 4096, 256, None),
    (1, 1, 257, 256, 2048, 128, None),
    (1, 1, 70, 64, 256, 32, -0.5),     # most entries kept: lists near their capacity
    (1, 2, 350, 128, 1024, 64, 0.6745),  # a quarter kept: 128 x 128 tiles of about 4096 entries, some more
    (1, 1, 50, 64, 128, 64, 40.0),     # no entry passes: y = 0
]


def _oracle(oracle_mod, kg, theta, S0=None, want_state=False):
    q = oracle_mod.bdh_keys(kg.xq, kg.U, theta)
    k = oracle_mod.bdh_keys(kg.xk, kg.U, theta)
    return oracle_mod.sparse_linattn(q, k, kg.v, S0=S0, want_state=want_state)


@pytest.mark.parametrize("B,H,T,R,N,dv,theta", CASES)
def test_keygen_forward_matches_oracle(cuda_lib, oracle_mod, B, H, T, R, N, dv, theta):
    kg = synth.sparse_keygen_inputs(B, H, T, N, dv, seed=T + N, rank=R)
    th = kg.theta if theta is None else theta
    y = cuda_lib.sparse_linattn_keygen_forward(kg.xq.cuda(), kg.xk.cuda(), kg.U.cuda(), th, kg.v.cuda())
    torch.cuda.synchronize()
    ref = _oracle(oracle_mod, kg, th)["y"]
    if np.all(ref == 0.0):
        assert torch.all(y == 0.0)
    else:
        check_parity(to_np(y), ref, "f32", f"keygen y B{B} H{H} T{T} R{R} N{N} dv{dv} theta {th:.3f}")


def test_keygen_forward_with_state(cuda_lib, oracle_mod):
    B, H, T, R, N, dv = 1, 2, 150, 128, 1024, 64
    kg = synth.sparse_keygen_inputs(B, H, T, N, dv, seed=31, rank=R)
    S0 = torch.randn(B, H, N, dv, generator=torch.Generator().manual_seed(2)) * 0.1
    S = S0.clone().cuda()
    y = cuda_lib.sparse_linattn_keygen_forward(kg.xq.cuda(), kg.xk.cuda(), kg.U.cuda(), kg.theta, kg.v.cuda(),
                                               S0=S, S_out=S)   # in place
    torch.cuda.synchronize()
    ref = _oracle(oracle_mod, kg, kg.theta, S0=S0, want_state=True)
    check_parity(to_np(y), ref["y"], "f32", "keygen y with S0")
    check_parity(to_np(S), ref["S"], "f32", "keygen final state")


def test_keygen_full_workload_sampled(cuda_lib, oracle_mod):
    """The full workload (B=2, H=4, T=2048, R=256, N=16384, d_v=256) on the
    GPU; two units checked at sampled positions by the oracle's closed form
    over keys and queries it generates itself."""
    d = synth.WORKLOADS["bdh_keygen_B2_H4_T2048_R256_N16384_dv256"].dims
    kg = synth.sparse_keygen_inputs(d["B"], d["H"], d["T"], d["N"], d["d_v"],
                                    seed=synth.WORKLOADS["bdh_keygen_B2_H4_T2048_R256_N16384_dv256"].seed)
    y = cuda_lib.sparse_linattn_keygen_forward(kg.xq.cuda(), kg.xk.cuda(), kg.U.cuda(), kg.theta, kg.v.cuda())
    torch.cuda.synchronize()
    ts = [0, 1, 127, 128, 1000, 2047]
    for b, h in ((0, 0), (1, 3)):
        q = oracle_mod.bdh_keys(kg.xq[b:b + 1, h:h + 1], kg.U[h:h + 1], kg.theta)[0, 0]
        k = oracle_mod.bdh_keys(kg.xk[b:b + 1, h:h + 1], kg.U[h:h + 1], kg.theta)[0, 0]
        ref = oracle_mod.sparse_linattn_output_at(q, k, kg.v[b, h], ts)
        check_parity(to_np(y[b, h, ts]), ref, "f32", f"keygen full workload b={b} h={h}")
