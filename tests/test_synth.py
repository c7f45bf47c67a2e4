"""The seeded generators: determinism and the stated input distributions."""
import torch

from outer_product_associative_chunked_b300 import synth


def test_tc_inputs_deterministic_and_unit_norm():
    a = synth.tc_inputs(2, 3, 17, 8, 8, 4, dtype="f32", seed=5)
    b = synth.tc_inputs(2, 3, 17, 8, 8, 4, dtype="f32", seed=5)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.lam, b.lam)):
        assert torch.equal(x, y)
    assert torch.allclose(a.q.norm(dim=-1), torch.ones(2, 3, 17), atol=1e-6)
    assert torch.all((a.lam >= 0.9) & (a.lam <= 0.999))
    assert torch.all((a.eta >= 0.1) & (a.eta <= 1.0))


def test_bf16_inputs_are_rounded_copies():
    a = synth.tc_inputs(1, 1, 9, 16, 16, 4, dtype="bf16", seed=6)
    f = synth.tc_inputs(1, 1, 9, 16, 16, 4, dtype="f32", seed=6)
    assert a.q.dtype == torch.bfloat16
    assert torch.equal(a.q, f.q.to(torch.bfloat16))


def test_delta_beta_in_open_unit_interval():
    d = synth.delta_inputs(1, 2, 50, 8, 8, dtype="f32", seed=2)
    assert torch.all((d.beta > 0) & (d.beta < 1))
    assert torch.allclose(d.k.norm(dim=-1), torch.ones(1, 2, 50), atol=1e-6)


def test_delta_decode_inputs_shapes_and_ranges():
    a = synth.delta_decode_inputs(3, 2, 4, 16, 8, dtype="f32", seed=7)
    b = synth.delta_decode_inputs(3, 2, 4, 16, 8, dtype="f32", seed=7)
    assert a.q.shape == (3, 2, 4, 16) and a.v.shape == (3, 2, 4, 8) and a.beta.shape == (3, 2, 4)
    assert a.S0.shape == (2, 4, 16, 8) and a.S0.dtype == torch.float32
    assert torch.equal(a.S0, b.S0) and torch.equal(a.k, b.k)
    assert torch.all((a.beta > 0) & (a.beta < 1))
    assert torch.allclose(a.k.norm(dim=-1), torch.ones(3, 2, 4), atol=1e-6)
    big = synth.delta_decode_inputs(1, 8, 8, 64, 64, dtype="f32", seed=1)
    assert abs(float(big.S0.var()) * 64 - 1.0) < 0.05
