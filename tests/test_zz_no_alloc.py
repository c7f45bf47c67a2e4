"""tc_layer_forward_noalloc: the Tensor Cache prefill for callers that cannot
allocate device memory (plugins inside an application that owns all device
memory, services that forbid allocation after start-up).  It takes its scratch
from an array built into the library instead of a caller workspace.

Through the C ABI: two calls in a row must match tc_layer_forward (run with
its own workspace) within the parity tolerance, and a problem larger than the
built-in scratch must be rejected with a clear message.  This file is
collected last on purpose, so a failure here cannot stop the rest of the
suite from running first.
"""
import ctypes

import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import synth

pytestmark = pytest.mark.gpu


def test_two_calls_match_workspace_entry_point(cuda_lib):
    B, H, T, d, W = 4, 8, 4096, 64, 512          # scratch need ~34 MB, inside the 64 MiB array
    need = cuda_lib.tc_layer_forward_workspace_size(B, H, T, d, d, W, torch.bfloat16)
    assert 0 < need <= cuda_lib.STATIC_SCRATCH_BYTES
    for seed in (21, 22):                          # two calls in a row, different inputs
        inp = synth.tc_inputs(B, H, T, d, d, W, dtype="bf16", seed=seed)
        q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
        ref = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, W)
        out = torch.full_like(ref, float("nan"))
        cuda_lib.tc_layer_forward_noalloc(q, k, v, lam, eta, gate, W, out)
        torch.cuda.synchronize()
        check_parity(to_np(out), to_np(ref), "bf16", f"no-alloc call seed={seed}")


def test_state_export_and_fp32(cuda_lib):
    inp = synth.tc_inputs(2, 3, 300, 32, 32, 40, dtype="f32", seed=23)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    st_ref = cuda_lib.TCState(2, 3, 40, 32, 32, dtype=torch.float32)
    st = cuda_lib.TCState(2, 3, 40, 32, 32, dtype=torch.float32)
    ref = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, 40, state=st_ref)
    out = torch.empty_like(ref)
    cuda_lib.tc_layer_forward_noalloc(q, k, v, lam, eta, gate, 40, out, state=st)
    torch.cuda.synchronize()
    check_parity(to_np(out), to_np(ref), "f32", "no-alloc fp32")
    check_parity(to_np(st.A), to_np(st_ref.A), "f32", "no-alloc state A")
    assert torch.equal(st.ring_k, st_ref.ring_k) and torch.equal(st.pos, st_ref.pos)


def test_oversized_problem_is_rejected(cuda_lib):
    L = cuda_lib.lib()
    B, H, T, d, W = 1, 16, 32768, 128, 2048       # needs ~270 MB of scratch
    assert L.tc_layer_forward_workspace_size(B, H, T, d, d, W, 1) > cuda_lib.STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)               # never touched: the size check comes first
    rc = L.tc_layer_forward_noalloc(fake, fake, fake, 1, B, H, T, d, d, W, fake, fake, fake, 0.0, fake,
                                    None, None)
    assert rc == -4
    msg = cuda_lib.last_error()
    assert "scratch" in msg and "tc_layer_forward" in msg
