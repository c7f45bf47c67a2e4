"""tc_layer_forward_noalloc: the Tensor Cache prefill for callers that cannot
allocate device memory (plugins inside an application that owns all device
memory, services that forbid allocation after start-up).  It takes its scratch
from an array built into the library instead of a caller workspace.

Through the C ABI: calls in a row must give exactly what tc_layer_forward
gives with its own workspace (the same kernels on the same inputs), one call
is checked against the oracle, a call whose chunk and segment layout differs
from the previous call's must not pick up that call's leftover scratch, and a
problem larger than the built-in scratch must be rejected with a clear
message.  This file is collected last on purpose, so a failure here cannot
stop the rest of the suite from running first.
"""
import ctypes

import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import binding, synth

pytestmark = pytest.mark.gpu


def _gpu(inp):
    return [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]


def test_two_calls_match_workspace_entry_point(cuda_lib, oracle_mod):
    # The headline shape needs about 11.5 MB of scratch on a 148-SM GPU (the
    # segment count, and with it the size, follows the SM count).
    B, H, T, d, W = 4, 8, 4096, 64, 512
    need = cuda_lib.tc_layer_forward_workspace_size(B, H, T, d, d, W, torch.bfloat16)
    assert 0 < need <= cuda_lib.STATIC_SCRATCH_BYTES
    for seed in (21, 22):                          # two calls in a row, different inputs
        inp = synth.tc_inputs(B, H, T, d, d, W, dtype="bf16", seed=seed)
        q, k, v, lam, eta, gate = _gpu(inp)
        ref = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, W)
        out = torch.full_like(ref, float("nan"))
        cuda_lib.tc_layer_forward_noalloc(q, k, v, lam, eta, gate, W, out)
        cuda_lib.check_device_error(None)
        assert torch.equal(out, ref), f"seed {seed}: no-alloc result differs from the workspace call"
    # one of them against the oracle, on sampled heads and positions
    ts = [0, 511, 512, 513, 2047, 4095]
    for b, h in ((0, 0), (3, 7)):
        ref_o = oracle_mod.tc_output_at(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.lam[h], inp.eta[h],
                                        inp.gate[h], W, ts)
        check_parity(to_np(out[b, h, ts]), ref_o, "bf16", f"no-alloc vs oracle b={b} h={h}")


def test_layout_change_between_calls(cuda_lib):
    """A long d=128 call leaves its per-chunk states in the array; a short
    d=64 call after it has a different chunk and segment layout and must
    equal tc_layer_forward run with a NaN-filled workspace."""
    first = synth.tc_inputs(1, 4, 8192, 128, 128, 1024, dtype="bf16", seed=31)
    q, k, v, lam, eta, gate = _gpu(first)
    out1 = torch.empty(1, 4, 8192, 128, dtype=torch.bfloat16, device="cuda")
    cuda_lib.tc_layer_forward_noalloc(q, k, v, lam, eta, gate, 1024, out1)
    second = synth.tc_inputs(2, 3, 300, 64, 64, 100, dtype="bf16", seed=32)
    q, k, v, lam, eta, gate = _gpu(second)
    out2 = torch.full((2, 3, 300, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    cuda_lib.tc_layer_forward_noalloc(q, k, v, lam, eta, gate, 100, out2)
    cuda_lib.check_device_error(None)
    need = cuda_lib.tc_layer_forward_workspace_size(2, 3, 300, 64, 64, 100, torch.bfloat16)
    ws = torch.full((need // 4 + 1,), float("nan"), dtype=torch.float32, device="cuda")
    ref = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, 100, workspace=ws.view(torch.uint8))
    cuda_lib.check_device_error(ws)
    assert torch.equal(out2, ref)


def test_state_export_and_fp32(cuda_lib):
    inp = synth.tc_inputs(2, 3, 300, 32, 32, 40, dtype="f32", seed=23)
    q, k, v, lam, eta, gate = _gpu(inp)
    st_ref = cuda_lib.TCState(2, 3, 40, 32, 32, dtype=torch.float32)
    st = cuda_lib.TCState(2, 3, 40, 32, 32, dtype=torch.float32)
    ref = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, 40, state=st_ref)
    out = torch.empty_like(ref)
    cuda_lib.tc_layer_forward_noalloc(q, k, v, lam, eta, gate, 40, out, state=st)
    cuda_lib.check_device_error(None)
    assert torch.equal(out, ref)
    assert torch.equal(st.A, st_ref.A)
    assert torch.equal(st.ring_k, st_ref.ring_k) and torch.equal(st.pos, st_ref.pos)


def test_oversized_problem_is_rejected(cuda_lib):
    L = cuda_lib.lib()
    B, H, T, d, W = 1, 16, 32768, 128, 2048       # needs ~270 MB of scratch
    assert L.tc_layer_forward_workspace_size(B, H, T, d, d, W, 1) > cuda_lib.STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)               # never touched: the size check comes first
    rc = L.tc_layer_forward_noalloc(fake, fake, fake, 1, B, H, T, d, d, W, fake, fake, fake, 0.0, fake,
                                    None, None)
    assert rc == binding.OPAM_ERR_WORKSPACE
    msg = cuda_lib.last_error()
    assert "scratch" in msg and "tc_layer_forward" in msg
