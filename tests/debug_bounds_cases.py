"""Small cases of every entry point, run by tests/test_gpu_debug_bounds.py in
a child process whose OPAM_LIBRARY names the debug-bounds build of the library
(index checks that record a status bit instead of trapping).  Every call is
compared with the float64 oracle at the usual bars and its device status must
come back clean.  Prints one line per case and "all cases clean" at the end.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import torch  # noqa: E402

from helpers import check_parity, to_np  # noqa: E402
from oracle import oracle  # noqa: E402
from outer_product_associative_chunked_b300 import binding, synth  # noqa: E402


def main():
    torch.cuda.set_device(0)
    oracle.build()
    assert binding.LIB_PATH.endswith("libopam_debug.so"), binding.LIB_PATH
    assert binding.debug_bounds_build(), "the loaded library is not the debug-bounds build"
    # the checks report: a failed index check comes back as INVALID_ARG
    ws = binding.selftest_bounds(5)
    try:
        binding.check_device_error(ws)
        raise SystemExit("a failed index check was not reported")
    except binding.OpamError as e:
        assert e.status == -1, e
    binding.check_device_error(binding.selftest_bounds(32))

    def done(what):
        binding.check_device_errors()
        print("clean:", what, flush=True)

    g = lambda x: x.cuda()  # noqa: E731
    for dt, B, H, T, dk, dv, W in [("bf16", 1, 2, 300, 64, 64, 100), ("bf16", 1, 1, 260, 128, 128, 129),
                                   ("f32", 2, 1, 130, 32, 64, 40)]:
        inp = synth.tc_inputs(B, H, T, dk, dv, W, dtype=dt, seed=T)
        st = binding.TCState(B, H, W, dk, dv, dtype=inp.q.dtype)
        y = binding.tc_layer_forward(*map(g, (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)), W, state=st)
        ref = oracle.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, want_state=True)
        check_parity(to_np(y), ref["y"], dt, f"prefill {dt} d{dk}/{dv}")
        dec = synth.tc_decode_inputs(2, B, H, dk, dv, dtype=dt, seed=1)
        yd = [binding.tc_decode_step(st, g(dec.q[i]), g(dec.k[i]), g(dec.v[i]), g(inp.lam), g(inp.eta),
                                     g(inp.gate)) for i in range(2)]
        rd, _ = oracle.tc_decode(ref, dec.q, dec.k, dec.v, inp.lam, inp.eta, inp.gate)
        check_parity(to_np(torch.stack(yd)), rd, dt, "decode")
        yw = binding.tc_window_forward(*map(g, (inp.q, inp.k, inp.v)), W)
        rw = oracle.tc_prefill(inp.q, inp.k, inp.v, inp.lam, torch.zeros(H), inp.gate, W)["y"]
        check_parity(to_np(yw), rw, dt, "window only")
        dy = torch.randn(B, H, T, dv, generator=torch.Generator().manual_seed(3)).to(inp.q.dtype)
        gr = binding.tc_layer_backward(*map(g, (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)), W, g(dy))
        rb = oracle.tc_backward(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, W, dy)
        for got, name in zip(gr[:3], ("dq", "dk", "dv")):
            check_parity(to_np(got), rb[name], dt, f"tc backward {name}")
        done(f"Tensor Cache {dt} d{dk}/{dv}")
    for dt, dk, dv in [("bf16", 128, 128), ("bf16", 64, 32), ("f32", 32, 64)]:
        inp = synth.delta_inputs(1, 2, 150, dk, dv, dtype=dt, seed=dk)
        y = binding.delta_rule_forward(*map(g, (inp.q, inp.k, inp.v, inp.beta)))
        check_parity(to_np(y), oracle.delta(inp.q, inp.k, inp.v, inp.beta)["y"], dt, "delta")
        dy = torch.randn(1, 2, 150, dv, generator=torch.Generator().manual_seed(4)).to(inp.q.dtype)
        gr = binding.delta_rule_backward(*map(g, (inp.q, inp.k, inp.v, inp.beta)), g(dy))
        rb = oracle.delta_backward(inp.q, inp.k, inp.v, inp.beta, dy)
        for got, name in zip(gr[:3], ("dq", "dk", "dv")):
            check_parity(to_np(got), rb[name], dt, f"delta backward {name}")
        dd = synth.delta_decode_inputs(1, 2, 3, dk, dv, dtype=dt, seed=5)
        S = dd.S0.cuda()
        yd = binding.delta_decode_step(S, g(dd.q[0]), g(dd.k[0]), g(dd.v[0]), g(dd.beta[0]))
        rd = oracle.delta(dd.q.movedim(0, 2), dd.k.movedim(0, 2), dd.v.movedim(0, 2), dd.beta.movedim(0, 2),
                          S0=dd.S0)["y"][:, :, 0]
        check_parity(to_np(yd), rd, dt, "delta decode")
        done(f"DeltaNet {dt} d{dk}/{dv}")
    sp = synth.sparse_inputs(1, 2, 200, 512, 64, seed=3)
    y = binding.sparse_linattn_forward(*map(g, (sp.q, sp.k, sp.v)))
    check_parity(to_np(y), oracle.sparse_linattn(sp.q, sp.k, sp.v)["y"], "f32", "sparse pairwise")
    S = torch.zeros(1, 2, 512, 64, device="cuda")
    y = binding.sparse_linattn_forward(*map(g, (sp.q, sp.k, sp.v)), S_out=S)
    check_parity(to_np(y), oracle.sparse_linattn(sp.q, sp.k, sp.v)["y"], "f32", "sparse recurrent")
    kg = synth.sparse_keygen_inputs(1, 2, 200, 1024, 64, seed=6, rank=128)
    y = binding.sparse_linattn_keygen_forward(g(kg.xq), g(kg.xk), g(kg.U), kg.theta, g(kg.v))
    ref = oracle.sparse_linattn(oracle.bdh_keys(kg.xq, kg.U, kg.theta), oracle.bdh_keys(kg.xk, kg.U, kg.theta),
                                kg.v)["y"]
    check_parity(to_np(y), ref, "f32", "keygen pairwise")
    S = torch.zeros(1, 2, 1024, 64, device="cuda")
    y = binding.sparse_linattn_keygen_forward(g(kg.xq), g(kg.xk), g(kg.U), kg.theta, g(kg.v), S_out=S)
    check_parity(to_np(y), ref, "f32", "keygen recurrent")
    done("BDH")
    print("all cases clean", flush=True)


if __name__ == "__main__":
    main()
