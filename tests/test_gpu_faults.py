"""The bounded waits report instead of hanging (no GPU fault is caused).

The tensor-core kernels wait on mbarriers with a cycle limit; a wait that runs
out sets a status bit, the CTA abandons its work, and opam_device_status()
returns OPAM_ERR_TIMEOUT.  The self-test kernel makes that happen on purpose
with a barrier that nothing completes and a limit of about half a millisecond,
then the test checks the status, that it clears, and that the context still
computes correctly.
"""
import pytest
import torch

from helpers import check_parity, to_np
from outer_product_associative_chunked_b300 import binding, synth

pytestmark = pytest.mark.gpu

OPAM_ERR_TIMEOUT = -5


def test_wait_that_runs_out_is_reported_and_cleared(cuda_lib, oracle_mod):
    cuda_lib.device_status(clear=True)
    cuda_lib.selftest_bounded_wait(arrive=False, limit_cycles=1_000_000)
    with pytest.raises(binding.OpamError) as err:
        cuda_lib.device_status(clear=False)
    assert err.value.status == OPAM_ERR_TIMEOUT
    with pytest.raises(binding.OpamError):
        cuda_lib.device_status(clear=True)   # reports once more, then clears
    cuda_lib.device_status(clear=True)       # clean now

    # a wait whose barrier completes does not report
    cuda_lib.selftest_bounded_wait(arrive=True, limit_cycles=1_000_000)
    cuda_lib.device_status(clear=True)

    # the context is still usable: a tensor-core prefill matches the oracle
    inp = synth.tc_inputs(1, 2, 300, 64, 64, 129, dtype="bf16", seed=21)
    y = cuda_lib.tc_layer_forward(*[x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)], 129)
    torch.cuda.synchronize()
    cuda_lib.device_status(clear=True)
    ref = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, 129)["y"]
    check_parity(to_np(y), ref, "bf16", "prefill after a reported timeout")
