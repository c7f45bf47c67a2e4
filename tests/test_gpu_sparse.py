"""BDH-style sparse linear attention on the GPU vs the float64 oracle (fp32
path, relative L2 <= 1e-5).  Small cases cover ragged chunks, start states,
S_out aliasing S0, every supported d_v, fully dense and all-zero rows; the
page-sized workload (B=2, H=4, T=2048, N=16384, d_v=256, ~5% density) runs at
full size and is checked at sampled positions the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,T,N,dv,with_S0", [
    (1, 1, 1, 40, 32, False),
    (1, 3, 17, 256, 64, True),
    (2, 1, 64, 1000, 128, False),
    (1, 1, 65, 512, 256, True),
    (1, 2, 150, 2048, 64, True),
])
def test_small_parity(cuda_lib, oracle_mod, B, H, T, N, dv, with_S0):
    inp = synth.sparse_inputs(B, H, T, N, dv, seed=T + N)
    S0 = torch.randn(B, H, N, dv, generator=torch.Generator().manual_seed(2)) if with_S0 else None
    S_out = torch.empty(B, H, N, dv, device="cuda")
    y = cuda_lib.sparse_linattn_forward(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(),
                                        S0=None if S0 is None else S0.cuda(), S_out=S_out)
    torch.cuda.synchronize()
    ref = oracle_mod.sparse_linattn(inp.q, inp.k, inp.v, S0=S0, want_state=True)
    check_parity(to_np(y), ref["y"], "f32", "bdh y")
    check_parity(to_np(S_out), ref["S"], "f32", "bdh S")


# Without a start state or a returned state the library takes the pairwise
# form (coordinate lists per 128-token block): ragged blocks, one and several
# blocks, every supported d_v.
@pytest.mark.parametrize("B,H,T,N,dv", [
    (1, 1, 1, 40, 32),
    (1, 2, 129, 300, 64),
    (2, 1, 300, 1000, 128),
    (1, 1, 257, 512, 256),
    (1, 3, 150, 2048, 32),
    (1, 1, 640, 4096, 256),
    (1, 2, 200, 320, 64),     # N a multiple of 64 but not of 128
])
def test_pairwise_form_parity(cuda_lib, oracle_mod, B, H, T, N, dv):
    inp = synth.sparse_inputs(B, H, T, N, dv, seed=3 * T + N)
    y = cuda_lib.sparse_linattn_forward(inp.q.cuda(), inp.k.cuda(), inp.v.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.sparse_linattn(inp.q, inp.k, inp.v)
    check_parity(to_np(y), ref["y"], "f32", f"bdh pairwise T={T} N={N} dv={dv}")


def test_pairwise_form_dense_and_empty_rows(cuda_lib, oracle_mod):
    inp = synth.sparse_inputs(1, 2, 200, 300, 64, seed=19)
    q, k = inp.q.clone(), inp.k.clone()
    k[0, 0, 5] = torch.rand(300)           # a fully dense key
    q[0, 1, 150] = torch.rand(300)         # a fully dense query in the second block
    k[0, 1, :10] = 0.0                     # keys with empty support
    q[0, 0, 120:140] = 0.0                 # queries with empty support across a block edge
    y = cuda_lib.sparse_linattn_forward(q.cuda(), k.cuda(), inp.v.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.sparse_linattn(q, k, inp.v)
    check_parity(to_np(y), ref["y"], "f32", "pairwise edge rows")


def test_pairwise_form_overflowing_key_lists(cuda_lib, oracle_mod):
    # A key block of fully dense rows: every window's key lists exceed the
    # shared-memory buffer and are read from global memory; the second block
    # stays sparse (buffered), and dense queries walk every coordinate.
    inp = synth.sparse_inputs(1, 1, 250, 700, 128, seed=23)
    q, k = inp.q.clone(), inp.k.clone()
    k[0, 0, :128] = torch.rand(128, 700, generator=torch.Generator().manual_seed(2))
    q[0, 0, 130:140] = torch.rand(10, 700, generator=torch.Generator().manual_seed(3))
    y = cuda_lib.sparse_linattn_forward(q.cuda(), k.cuda(), inp.v.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.sparse_linattn(q, k, inp.v)
    check_parity(to_np(y), ref["y"], "f32", "pairwise overflowing key lists")


def test_pairwise_form_dense_tiles_from_dense_rows(cuda_lib, oracle_mod):
    # N a multiple of 128: the coordinate lists come straight from the dense
    # rows, 128 x 128 tiles at a time.  A block of fully dense keys gives
    # tiles with more entries than the shared-memory stage (written in
    # place); the sparse block and a few dense queries are staged.
    inp = synth.sparse_inputs(1, 1, 250, 384, 64, seed=29)
    q, k = inp.q.clone(), inp.k.clone()
    k[0, 0, :128] = torch.rand(128, 384, generator=torch.Generator().manual_seed(4))
    q[0, 0, 130:135] = torch.rand(5, 384, generator=torch.Generator().manual_seed(5))
    y = cuda_lib.sparse_linattn_forward(q.cuda(), k.cuda(), inp.v.cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.sparse_linattn(q, k, inp.v)
    check_parity(to_np(y), ref["y"], "f32", "pairwise dense tiles from dense rows")


def test_dense_and_empty_rows_in_place_state(cuda_lib, oracle_mod):
    inp = synth.sparse_inputs(1, 2, 70, 300, 32, seed=9)
    q, k = inp.q.clone(), inp.k.clone()
    k[0, 0, 5] = torch.rand(300)           # a fully dense key
    q[0, 1, 9] = torch.rand(300)           # a fully dense query
    k[0, 1, :10] = 0.0                     # keys with empty support
    q[0, 0, 20:30] = 0.0                   # queries with empty support
    S0 = torch.randn(1, 2, 300, 32, generator=torch.Generator().manual_seed(1))
    S = S0.clone().cuda()
    y = cuda_lib.sparse_linattn_forward(q.cuda(), k.cuda(), inp.v.cuda(), S0=S, S_out=S)
    torch.cuda.synchronize()
    ref = oracle_mod.sparse_linattn(q, k, inp.v, S0=S0, want_state=True)
    check_parity(to_np(y), ref["y"], "f32", "edge rows y")
    check_parity(to_np(S), ref["S"], "f32", "edge rows S")


def test_full_size_workload_sampled(cuda_lib, oracle_mod):
    w = synth.WORKLOADS["bdh_fp32_B2_H4_T2048_N16384_dv256"]
    d = w.dims
    inp = synth.sparse_inputs(d["B"], d["H"], d["T"], d["N"], d["d_v"], seed=w.seed)
    y = cuda_lib.sparse_linattn_forward(inp.q.cuda(), inp.k.cuda(), inp.v.cuda())
    torch.cuda.synchronize()
    ts = [0, 1, 63, 64, 1000, 2047]
    got, ref = [], []
    for b, h in [(0, 0), (1, 3)]:
        got.append(to_np(y[b, h, ts]))
        ref.append(oracle_mod.sparse_linattn_output_at(inp.q[b, h], inp.k[b, h], inp.v[b, h], ts))
    check_parity(np.stack(got), np.stack(ref), "f32", "bdh full size")
