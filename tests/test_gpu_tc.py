"""Tensor Cache prefill on the GPU vs the float64 oracle.

Bars: fp32 inputs -> relative L2 <= 1e-5 over the whole output; bf16 inputs /
fp32 state -> RMS(error) <= 2e-2 of the output RMS.  Small cases cover ragged
tails, windows around the chunk length, head sizes 32/64/128, unequal d_k /
d_v and odd B*H; the two page-sized workloads run at full size on the GPU and
are checked on sampled heads and positions the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from helpers import canary_intact, check_parity, guarded, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_timeouts(cuda_lib):
    """Every case must leave its calls' device status clean (no bounded wait
    ran out, no CUDA error)."""
    cuda_lib.check_device_errors()
    yield
    cuda_lib.check_device_errors()


def _gpu(inp):
    return [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]


SMALL = [
    # dtype, B, H, T, d_k, d_v, W
    ("f32", 1, 1, 1, 32, 32, 1),
    ("f32", 1, 3, 2, 64, 64, 1),
    ("f32", 3, 1, 3, 32, 64, 2),
    ("f32", 1, 1, 15, 128, 128, 4),
    ("f32", 2, 1, 16, 64, 32, 16),
    ("f32", 1, 3, 17, 32, 32, 63),
    ("f32", 1, 1, 63, 64, 64, 64),
    ("f32", 1, 2, 64, 128, 64, 65),
    ("f32", 1, 1, 65, 32, 32, 64),
    ("f32", 1, 1, 200, 64, 64, 63),
    ("f32", 1, 1, 200, 128, 128, 65),
    ("f32", 2, 3, 200, 32, 32, 300),
    ("f32", 1, 1, 257, 64, 64, 1),
    ("bf16", 1, 1, 1, 64, 64, 1),
    ("bf16", 3, 1, 17, 64, 64, 2),
    ("bf16", 1, 3, 65, 128, 128, 64),
    ("bf16", 1, 1, 200, 64, 64, 63),
    ("bf16", 2, 1, 333, 128, 128, 129),
    ("bf16", 1, 2, 640, 64, 64, 128),
    ("bf16", 1, 1, 700, 128, 128, 256),
    ("bf16", 1, 1, 150, 32, 128, 50),
    # d = 64/64 (one-row-per-thread kernel): windows that are not a multiple
    # of the 128-key tile, shorter than a tile, and sequences ending mid-tile
    ("bf16", 1, 1, 300, 64, 64, 1),
    ("bf16", 1, 2, 1100, 64, 64, 512),
    ("bf16", 2, 1, 777, 64, 64, 300),
    ("bf16", 1, 1, 1024, 64, 64, 129),
    ("bf16", 1, 1, 900, 64, 64, 640),
    ("bf16", 1, 1, 515, 64, 64, 100),
]


@pytest.mark.parametrize("dtype,B,H,T,dk,dv,W", SMALL)
def test_small_parity(cuda_lib, oracle_mod, dtype, B, H, T, dk, dv, W):
    inp = synth.tc_inputs(B, H, T, dk, dv, W, dtype=dtype, seed=T * 7 + W)
    q, k, v, lam, eta, gate = _gpu(inp)
    y, buf = guarded((B, H, T, dv), q.dtype)
    cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, W, out=y)
    torch.cuda.synchronize()
    assert canary_intact(buf, (B, H, T, dv))
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W)["y"]
    check_parity(to_np(y), ref, dtype, f"T={T} W={W} d={dk}/{dv}")


@pytest.mark.parametrize("dtype,T,W,d", [("f32", 100, 7, 32), ("f32", 20, 50, 64),
                                         ("bf16", 300, 64, 128), ("bf16", 130, 129, 64)])
def test_state_export(cuda_lib, oracle_mod, dtype, T, W, d):
    B, H = 2, 2
    inp = synth.tc_inputs(B, H, T, d, d, W, dtype=dtype, seed=11)
    q, k, v, lam, eta, gate = _gpu(inp)
    st = cuda_lib.TCState(B, H, W, d, d, dtype=q.dtype)
    st.pos.fill_(-5)
    cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, W, state=st)
    torch.cuda.synchronize()
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, want_state=True)
    np.testing.assert_array_equal(to_np(st.ring_k), ref["ring_k"])   # copies are exact
    np.testing.assert_array_equal(to_np(st.ring_v), ref["ring_v"])
    assert torch.all(st.pos.cpu() == T)
    check_parity(to_np(st.A), ref["A"], "f32" if dtype == "f32" else "bf16", "A")


def test_fp32_workload_T256_d32_W32(cuda_lib, oracle_mod):
    w = synth.WORKLOADS["tc_fp32_T256_d32_W32"]
    inp = synth.tc_inputs(**{k: w.dims[k] for k in ("B", "H", "T", "d_k", "d_v", "W", "dtype", "lam",
                                                    "eta", "gate")}, seed=w.seed)
    q, k, v, lam, eta, gate = _gpu(inp)
    y = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, inp.W)
    torch.cuda.synchronize()
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, inp.W)["y"]
    err = check_parity(to_np(y), ref, "f32", "fp32 workload")
    assert err < 1e-5


@pytest.mark.parametrize("lam,scale", [(0.0, 0.0), (1.0, 0.0), (-0.8, 0.0), (0.95, 25.0)])
def test_decay_and_scale_extremes(cuda_lib, oracle_mod, lam, scale):
    """lambda = 0 (only the latest eviction counts), 1 (no decay), negative
    (alternating signs), and a softmax scale large enough that the running
    maximum moves by many binades within a row."""
    B, H, T, d, W = 1, 2, 700, 64, 200
    inp = synth.tc_inputs(B, H, T, d, d, W, dtype="bf16", seed=31, lam=lam)
    q, k, v, lam_t, eta, gate = _gpu(inp)
    y = cuda_lib.tc_layer_forward(q, k, v, lam_t, eta, gate, W, softmax_scale=scale)
    torch.cuda.synchronize()
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W,
                                scale=None if scale == 0.0 else scale)["y"]
    check_parity(to_np(y), ref, "bf16", f"lambda={lam} scale={scale}")


def test_cuda_graph_replay_matches_eager(cuda_lib):
    """A call captured into a CUDA graph and replayed gives the eager result bit for bit."""
    inp = synth.tc_inputs(2, 2, 1000, 64, 64, 256, dtype="bf16", seed=5)
    q, k, v, lam, eta, gate = _gpu(inp)
    ws = torch.empty(cuda_lib.tc_layer_forward_workspace_size(2, 2, 1000, 64, 64, 256, q.dtype),
                     dtype=torch.uint8, device="cuda")
    y_eager = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, 256, workspace=ws)
    y = torch.empty_like(y_eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, 256, out=y, workspace=ws)
    y.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)


def test_multi_chunk_segments_full_tensor(cuda_lib, oracle_mod):
    """Every output element of a batch whose state recurrence is split into
    segments of several chunks: at d = 64 the library sizes the state pass to
    one CTA per SM, so 64 (batch, head) units leave two segments per head on a
    148-SM GPU and T = 2048 (16 chunks of 128) gives segments of eight chunks;
    the carry lambda^(C (j - gL)) A_{gL} and the local states A_j^loc are both
    exercised at every chunk."""
    B, H, T, d, W = 8, 8, 2048, 64, 256
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nch = -(-T // 128)
    want = max(1, min(nch, sms // (B * H)))
    chunks_per_segment = -(-nch // want)
    assert chunks_per_segment > 1 and -(-nch // chunks_per_segment) < nch
    inp = synth.tc_inputs(B, H, T, d, d, W, dtype="bf16", seed=55)
    q, k, v, lam, eta, gate = _gpu(inp)
    st = cuda_lib.TCState(B, H, W, d, d, dtype=torch.bfloat16)
    y = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, W, state=st)
    torch.cuda.synchronize()
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, want_state=True)
    check_parity(to_np(y), ref["y"], "bf16", f"multi-chunk segments ({chunks_per_segment} chunks each)")
    check_parity(to_np(st.A), ref["A"], "bf16", "multi-chunk segments, final A")


def _sampled_positions(T, W):
    ts = {0, 1, W - 1, W, W + 1, T // 2, T - 2, T - 1}
    ts |= set(np.random.default_rng(T).integers(0, T, 8).tolist())
    return sorted(t for t in ts if 0 <= t < T)


@pytest.mark.parametrize("name,units", [("tc_bf16_B4_H8_T4096_d64_W512", [(0, 0), (3, 7), (1, 4)]),
                                        ("tc_bf16_B1_H16_T32768_d128_W2048", [(0, 0), (0, 9), (0, 15)])])
def test_full_size_workload_sampled(cuda_lib, oracle_mod, name, units):
    w = synth.WORKLOADS[name]
    d = w.dims
    inp = synth.tc_inputs(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], dtype=d["dtype"], seed=w.seed)
    q, k, v, lam, eta, gate = _gpu(inp)
    y = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, inp.W)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    ts = _sampled_positions(d["T"], d["W"])
    got, ref = [], []
    for b, h in units:
        got.append(to_np(y[b, h, ts]))
        ref.append(oracle_mod.tc_output_at(inp.q[b, h], inp.k[b, h], inp.v[b, h], float(inp.lam[h]),
                                           float(inp.eta[h]), float(inp.gate[h]), inp.W, ts))
    check_parity(np.stack(got), np.stack(ref), "bf16", name)


# Window-only variant: the same kernels with the L2 part off.  Its reference
# is the oracle layer with eta = 0 (A stays 0, so y is the window softmax).
@pytest.mark.parametrize("dtype,B,H,T,dk,dv,W", [
    ("bf16", 2, 3, 700, 64, 64, 512),     # row kernel: blocks with and without a shifted first tile
    ("bf16", 1, 2, 1000, 64, 64, 129),
    ("bf16", 1, 1, 300, 64, 64, 1),
    ("bf16", 1, 1, 400, 64, 64, 1000),    # window longer than the sequence
    ("bf16", 1, 2, 520, 128, 128, 300),   # split-key-half kernel
    ("bf16", 2, 1, 333, 64, 128, 129),
    ("f32", 1, 2, 333, 32, 32, 77),       # CUDA-core kernel
    ("f32", 2, 1, 200, 64, 128, 64),
    ("bf16", 1, 1, 150, 32, 128, 50),     # bf16 on the CUDA-core kernel
])
def test_window_only_matches_eta_zero(cuda_lib, oracle_mod, dtype, B, H, T, dk, dv, W):
    inp = synth.tc_inputs(B, H, T, dk, dv, W, dtype=dtype, seed=T + W)
    y, buf = guarded((B, H, T, dv), inp.q.dtype)
    cuda_lib.tc_window_forward(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), W, out=y)
    torch.cuda.synchronize()
    assert canary_intact(buf, (B, H, T, dv))
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, torch.zeros(H), inp.gate, W)["y"]
    check_parity(to_np(y), ref, dtype, f"window only {dtype} T={T} d={dk}/{dv} W={W}")


def test_window_only_headline_workload_sampled(cuda_lib, oracle_mod):
    w = synth.WORKLOADS["tc_bf16_B4_H8_T4096_d64_W512"]
    d = w.dims
    inp = synth.tc_inputs(d["B"], d["H"], d["T"], d["d_k"], d["d_v"], d["W"], dtype=d["dtype"], seed=w.seed)
    y = cuda_lib.tc_window_forward(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.W)
    torch.cuda.synchronize()
    ts = _sampled_positions(d["T"], d["W"])
    got, ref = [], []
    for b, h in [(0, 0), (2, 5), (3, 7)]:
        got.append(to_np(y[b, h, ts]))
        ref.append(oracle_mod.tc_output_at(inp.q[b, h], inp.k[b, h], inp.v[b, h], float(inp.lam[h]), 0.0,
                                           float(inp.gate[h]), inp.W, ts))
    check_parity(np.stack(got), np.stack(ref), "bf16", "window only, headline workload")
