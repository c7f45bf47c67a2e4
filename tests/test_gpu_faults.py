"""The bounded waits report instead of hanging (no GPU fault is caused).

The tensor-core kernels wait on mbarriers with a cycle limit; a wait that runs
out sets a bit in the status word at the head of the call's workspace, the
CTA abandons its work, and opam_check_device_error(workspace, stream) returns
OPAM_ERR_TIMEOUT.  The self-test kernel makes that happen on purpose with a
barrier that nothing completes and a limit of about half a millisecond.  Two
calls on two streams with two workspaces, one timing out and one not, must be
told apart; the next call on the same workspace clears the word; and the
context still computes correctly afterwards.
"""
import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import binding, synth

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_for_its_own_call_only(cuda_lib, oracle_mod):
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = torch.full((binding.STATUS_BYTES,), 0xFF, dtype=torch.uint8, device="cuda")   # garbage on entry
    ws2 = torch.full((binding.STATUS_BYTES,), 0xFF, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    cuda_lib.selftest_bounded_wait(arrive=False, limit_cycles=1_000_000, workspace=ws1, stream=s1)
    cuda_lib.selftest_bounded_wait(arrive=True, limit_cycles=1_000_000, workspace=ws2, stream=s2)
    with pytest.raises(binding.OpamError) as err:
        cuda_lib.check_device_error(ws1, stream=s1)
    assert err.value.status == binding.OPAM_ERR_TIMEOUT
    assert "self-test" in str(err.value)
    cuda_lib.check_device_error(ws2, stream=s2)            # the other call is clean
    with pytest.raises(binding.OpamError):                 # reading does not clear it
        cuda_lib.check_device_error(ws1, stream=s1)

    # the next call that uses ws1 zeroes the word before its kernels
    cuda_lib.selftest_bounded_wait(arrive=True, limit_cycles=1_000_000, workspace=ws1, stream=s1)
    cuda_lib.check_device_error(ws1, stream=s1)

    # the context is still usable: a tensor-core prefill on the timed-out
    # workspace's stream matches the oracle and reports clean
    inp = synth.tc_inputs(1, 2, 300, 64, 64, 129, dtype="bf16", seed=21)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    need = cuda_lib.tc_layer_forward_workspace_size(1, 2, 300, 64, 64, 129, torch.bfloat16)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(s1):
        y = cuda_lib.tc_layer_forward(q, k, v, lam, eta, gate, 129, workspace=ws)
    cuda_lib.check_device_error(ws, stream=s1)
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, 129)["y"]
    check_parity(to_np(y), ref, "bf16", "prefill after a reported timeout")
