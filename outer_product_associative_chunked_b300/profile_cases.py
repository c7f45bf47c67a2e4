"""Small, self-contained invocations of each entry point for profiler captures.

Each case allocates a few hundred MB at most, runs the call four times on
cuda:0 and checks the device status, so an ``ncu`` capture of one launch
(``-s 2 -c 1``) sees warm caches and ends quickly:

    python -m outer_product_associative_chunked_b300.profile_cases prefill
    python -m outer_product_associative_chunked_b300.profile_cases prefill_long
    python -m outer_product_associative_chunked_b300.profile_cases decode
    python -m outer_product_associative_chunked_b300.profile_cases delta
    python -m outer_product_associative_chunked_b300.profile_cases delta_decode
    python -m outer_product_associative_chunked_b300.profile_cases sparse
    python -m outer_product_associative_chunked_b300.profile_cases sparse_keygen
    python -m outer_product_associative_chunked_b300.profile_cases tc_backward
    python -m outer_product_associative_chunked_b300.profile_cases delta_backward

Inputs come from the seeded generators in ``synth``; the shapes are the
page workloads with fewer sequences or heads.
"""
from __future__ import annotations

import sys

import torch

from . import binding, synth


def prefill(B=4, H=8, T=4096, d=64, W=512, reps=4):
    """Tensor Cache prefill, bf16 (the B=4 H=8 T=4096 d=64 W=512 workload)."""
    inp = synth.tc_inputs(B, H, T, d, d, W, dtype="bf16", seed=1)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    y = torch.empty_like(v)
    ws = torch.empty(binding.tc_layer_forward_workspace_size(B, H, T, d, d, W, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    for _ in range(reps):
        binding.tc_layer_forward(q, k, v, lam, eta, gate, W, out=y, workspace=ws)


def prefill_long(B=1, H=4, T=8192, d=128, W=2048, reps=4):
    """Tensor Cache prefill, bf16, the long-context shape with fewer heads and tokens."""
    prefill(B, H, T, d, W, reps)


def decode(S=16, H=16, W=2048, d=128, reps=4):
    """Decode steps for S sequences x H heads from a full ring (W slots)."""
    st = binding.TCState(S, H, W, d, d, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(0)
    st.ring_k.copy_(torch.randn(S, H, W, d, generator=g).to(torch.bfloat16))
    st.ring_v.copy_(torch.randn(S, H, W, d, generator=g).to(torch.bfloat16))
    st.A.copy_(torch.randn(S, H, d, d, generator=g) * 0.01)
    st.pos.fill_(5000)
    dec = synth.tc_decode_inputs(reps, S, H, d, d, dtype="bf16", seed=1)
    lam = torch.full((H,), 0.99, device="cuda")
    eta = torch.full((H,), 0.5, device="cuda")
    gate = torch.zeros(H, device="cuda")
    for i in range(reps):
        binding.tc_decode_step(st, dec.q[i].cuda(), dec.k[i].cuda(), dec.v[i].cuda(), lam, eta, gate)


def delta(B=1, H=16, T=8192, d=128, reps=4):
    """DeltaNet forward, chunk 64, bf16 inputs."""
    inp = synth.delta_inputs(B, H, T, d, d, dtype="bf16", seed=2)
    q, k, v, beta = inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.beta.cuda()
    y = torch.empty_like(v)
    ws = torch.empty(binding.delta_rule_forward_workspace_size(B, H, T, d, d, 64, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    for _ in range(reps):
        binding.delta_rule_forward(q, k, v, beta, chunk=64, out=y, workspace=ws)


def delta_decode(S=128, H=16, d=128, reps=4):
    """DeltaNet decode steps for S sequences x H heads (128 MiB state), bf16 tokens."""
    dec = synth.delta_decode_inputs(reps, S, H, d, d, dtype="bf16", seed=5)
    St = dec.S0.cuda()
    for i in range(reps):
        binding.delta_decode_step(St, dec.q[i].cuda(), dec.k[i].cuda(), dec.v[i].cuda(), dec.beta[i].cuda())


def sparse(B=1, H=2, T=2048, N=16384, dv=256, reps=4):
    """BDH sparse linear attention, ~5% dense keys and queries, fp32."""
    inp = synth.sparse_inputs(B, H, T, N, dv, seed=4)
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    y = torch.empty_like(v)
    ws = torch.empty(binding.sparse_linattn_forward_workspace_size(B, H, T, N, dv), dtype=torch.uint8,
                     device="cuda")
    for _ in range(reps):
        binding.sparse_linattn_forward(q, k, v, out=y, workspace=ws)


def sparse_keygen(B=1, H=2, T=2048, R=256, N=16384, dv=256, reps=4):
    """BDH attention with the keys and queries generated on the GPU."""
    kg = synth.sparse_keygen_inputs(B, H, T, N, dv, seed=5, rank=R)
    xq, xk, U, v = kg.xq.cuda(), kg.xk.cuda(), kg.U.cuda(), kg.v.cuda()
    y = torch.empty_like(v)
    ws = torch.empty(binding.sparse_linattn_keygen_forward_workspace_size(B, H, T, R, N, dv), dtype=torch.uint8,
                     device="cuda")
    for _ in range(reps):
        binding.sparse_linattn_keygen_forward(xq, xk, U, kg.theta, v, out=y, workspace=ws)


def tc_backward(B=4, H=8, T=4096, d=64, W=512, reps=4):
    """Tensor Cache backward on the headline shape, bf16."""
    inp = synth.tc_inputs(B, H, T, d, d, W, dtype="bf16", seed=1)
    q, k, v, lam, eta, gate = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate)]
    dy = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).cuda()
    ws = torch.empty(binding.tc_layer_backward_workspace_size(B, H, T, d, d, W, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    for _ in range(reps):
        binding.tc_layer_backward(q, k, v, lam, eta, gate, W, dy, workspace=ws)


def delta_backward(B=1, H=16, T=2048, d=128, reps=4):
    """DeltaNet backward, bf16, the DeltaNet head size over 2048 tokens."""
    inp = synth.delta_inputs(B, H, T, d, d, dtype="bf16", seed=2)
    q, k, v, beta = inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.beta.cuda()
    dy = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(10)).to(torch.bfloat16).cuda()
    ws = torch.empty(binding.delta_rule_backward_workspace_size(B, H, T, d, d, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    for _ in range(reps):
        binding.delta_rule_backward(q, k, v, beta, dy, workspace=ws)


CASES = {"prefill": prefill, "prefill_long": prefill_long, "decode": decode, "delta": delta,
         "delta_decode": delta_decode, "sparse": sparse, "sparse_keygen": sparse_keygen,
         "tc_backward": tc_backward, "delta_backward": delta_backward}


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    if len(argv) != 1 or argv[0] not in CASES:
        raise SystemExit(f"usage: python -m {__package__}.profile_cases {{{','.join(CASES)}}}")
    torch.cuda.set_device(0)
    CASES[argv[0]]()
    torch.cuda.synchronize()
    binding.check_device_errors()
    print(f"{argv[0]} ok")


if __name__ == "__main__":
    main()
