"""Pins for the Tensor Cache oracle (CPU only).

Page: "Tensor Cache: Eviction-conditioned Associative Memory for Transformers"
(gist.science 2605.22884).  Methodology 1 defines the layer (L1 ring of the W
most recent tokens with exact softmax; eviction write A <- lambda A +
eta (k (x) v); read m_t = q_t A using q (k (x) v) = <q,k> v; fuse
y = y_local + sigmoid(g) m).  Methodology 2 states that the parallel
weighted-sum scan equals the sequential per-token writes (relative error below
1e-7 in float32) and that chunk-averaging adds C^2 - C spurious cross terms.
Main contributions: every token is either resident in L1 or compressed in L2.

Each test ties the oracle to something other than itself: hand-worked
fixtures, a library routine (torch SDPA), closed forms in matrix form,
invariants, or a pure-Python brute force.
"""
import math

import numpy as np
import pytest
import torch

from helpers import load_golden, rel_l2
from outer_product_associative_chunked_b300 import synth


def _logistic(x):
    return 1.0 / (1.0 + math.exp(-x))


def _unit(B, H, T, d, seed, unit=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, H, T, d, generator=g, dtype=torch.float64)
    if unit:
        x = x / x.norm(dim=-1, keepdim=True)
    return x.numpy()


@pytest.mark.parametrize("name", ["tc_w1_d2_t3.txt", "tc_w2_d2_t4.txt"])
def test_hand_worked_fixture(oracle_mod, name):
    g = load_golden(name)
    q, k, v = (np.asarray(g[x])[None, None] for x in ("q", "k", "v"))
    one = lambda x: np.array([x])  # noqa: E731
    out = oracle_mod.tc_prefill(q, k, v, one(g["lambda"]), one(g["eta"]), one(g["gate"]),
                                int(g["W"]), scale=g["scale"])
    np.testing.assert_allclose(out["y"][0, 0], g["y"], rtol=0, atol=1e-14)


def _brute_tc(q, k, v, lam, eta, gate, W, scale):
    """Pure-Python double sums straight from the definitions (T <= 16)."""
    T, dk = len(q), len(q[0])
    dv = len(v[0])
    dot = lambda a, b: sum(x * y for x, y in zip(a, b))  # noqa: E731
    ys = []
    for t in range(T):
        win = list(range(max(0, t - W + 1), t + 1))
        sc = [scale * dot(q[t], k[s]) for s in win]
        mx = max(sc)
        e = [math.exp(x - mx) for x in sc]
        z = sum(e)
        y = [sum(e[i] * v[s][b] for i, s in enumerate(win)) / z for b in range(dv)]
        for s in range(0, t - W + 1):  # tokens already evicted into A
            w = _logistic(gate) * eta * lam ** (t - W - s) * dot(q[t], k[s])
            for b in range(dv):
                y[b] += w * v[s][b]
        ys.append(y)
    return np.array(ys)


@pytest.mark.parametrize("T,W,dk,dv", [(16, 1, 3, 2), (16, 3, 4, 5), (13, 4, 2, 3),
                                       (16, 8, 4, 4), (16, 16, 3, 3), (9, 16, 2, 2), (1, 1, 2, 2)])
def test_bruteforce_small(oracle_mod, T, W, dk, dv):
    rng = np.random.default_rng(T * 100 + W)
    q = rng.standard_normal((1, 1, T, dk))
    k = rng.standard_normal((1, 1, T, dk))
    v = rng.standard_normal((1, 1, T, dv))
    lam, eta, gate, scale = 0.8, 0.7, 0.3, 0.9
    out = oracle_mod.tc_prefill(q, k, v, [lam], [eta], [gate], W, scale=scale)
    ref = _brute_tc(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), lam, eta, gate, W, scale)
    np.testing.assert_allclose(out["y"][0, 0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("T,W", [(40, 7), (33, 1), (64, 64), (20, 50)])
def test_eta_zero_is_band_softmax_sdpa(oracle_mod, T, W):
    """eta = 0 leaves A at zero, so the layer is softmax attention over the
    band t-W < s <= t: compare with torch SDPA (float64) and a band mask."""
    B, H, d = 2, 3, 8
    q, k, v = _unit(B, H, T, d, 1), _unit(B, H, T, d, 2), _unit(B, H, T, d, 3, unit=False)
    gate = np.array([0.5, -1.0, 2.0])
    out = oracle_mod.tc_prefill(q, k, v, [0.9] * H, [0.0] * H, gate, W)
    t = torch.arange(T)
    band = (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - W)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=band,
        scale=1.0 / math.sqrt(d))
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_window_covering_sequence_is_causal_sdpa(oracle_mod):
    """W >= T: nothing is ever evicted, the L2 read stays zero and the layer is
    causal softmax attention."""
    B, H, T, d = 1, 2, 24, 16
    q, k, v = _unit(B, H, T, d, 4), _unit(B, H, T, d, 5), _unit(B, H, T, d, 6, unit=False)
    out = oracle_mod.tc_prefill(q, k, v, [0.95, 0.9], [1.0, 0.3], [0.1, 0.2], T, want_m=True)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=True)
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-13)
    assert np.all(out["m"] == 0.0)


def test_single_eviction_reads_inner_product_times_value(oracle_mod):
    """One evicted pair: A = eta k0 v0^T and m = q A = eta <q,k0> v0 (the
    identity q (k (x) v) = <q,k> v).  d_k != d_v so a transposed A cannot even
    be formed by mistake, and a read of A q instead of q A would give k0."""
    W, dk, dv = 5, 3, 4
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, W + 1, dk))
    k = rng.standard_normal((1, 1, W + 1, dk))
    v = rng.standard_normal((1, 1, W + 1, dv))
    out = oracle_mod.tc_prefill(q, k, v, [0.3], [1.7], [0.0], W, want_m=True, want_state=True)
    qW, k0, v0 = q[0, 0, W], k[0, 0, 0], v[0, 0, 0]
    np.testing.assert_allclose(out["m"][0, 0, W], 1.7 * float(qW @ k0) * v0, rtol=1e-13)
    np.testing.assert_allclose(out["A"][0, 0], 1.7 * np.outer(k0, v0), rtol=1e-13)
    assert np.all(out["m"][0, 0, :W] == 0.0)


def _l2_closed_form_matrix(q, k, v, lam, eta, W):
    """m = (D o Q K^T) V with D[t,s] = eta lambda^(t-W-s) for s <= t-W: the
    parallel weighted-sum form of the evicted-token read, as one dense product."""
    T = q.shape[0]
    t = np.arange(T)[:, None]
    s = np.arange(T)[None, :]
    e = t - W - s
    D = np.where(e >= 0, eta * lam ** np.maximum(e, 0), 0.0)
    return ((q @ k.T) * D) @ v


@pytest.mark.parametrize("T,W,lam", [(100, 10, 0.97), (64, 1, 0.5), (90, 31, 1.0)])
def test_l2_read_matches_dense_weighted_sum(oracle_mod, T, W, lam):
    B, H, d = 1, 2, 8
    q, k, v = _unit(B, H, T, d, 8), _unit(B, H, T, d, 9), _unit(B, H, T, d, 10, unit=False)
    eta = [0.6, 1.3]
    out = oracle_mod.tc_prefill(q, k, v, [lam] * H, eta, [0.0] * H, W, want_m=True)
    for h in range(H):
        ref = _l2_closed_form_matrix(q[0, h], k[0, h], v[0, h], lam, eta[h], W)
        np.testing.assert_allclose(out["m"][0, h], ref, rtol=1e-11, atol=1e-12)


def test_lambda_eta_one_is_offset_causal_linear_attention(oracle_mod):
    """lambda = eta = 1: m_t = sum_{s <= t-W} <q_t,k_s> v_s, i.e. tril(QK^T, -W) V."""
    T, W, d = 50, 6, 5
    q, k, v = _unit(1, 1, T, d, 11), _unit(1, 1, T, d, 12), _unit(1, 1, T, d, 13, unit=False)
    out = oracle_mod.tc_prefill(q, k, v, [1.0], [1.0], [0.0], W, want_m=True)
    ref = np.tril(q[0, 0] @ k[0, 0].T, -W) @ v[0, 0]
    np.testing.assert_allclose(out["m"][0, 0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("T,W", [(37, 5), (10, 10), (10, 20), (64, 1)])
def test_each_token_written_once_at_eviction(oracle_mod, T, W):
    """Every token is either in L1 or compressed in L2: token s is written
    exactly once, at step s + W, iff s + W < T."""
    q, k, v = _unit(1, 2, T, 4, 14), _unit(1, 2, T, 4, 15), _unit(1, 2, T, 4, 16, unit=False)
    out = oracle_mod.tc_prefill(q, k, v, [0.9, 0.8], [1.0, 1.0], [0.0, 0.0], W, want_writes=True)
    s = np.arange(T)
    for h in range(2):
        expect_count = (s + W < T).astype(np.int32)
        np.testing.assert_array_equal(out["write_count"][0, h], expect_count)
        np.testing.assert_array_equal(out["write_time"][0, h], np.where(s + W < T, s + W, -1))


@pytest.mark.parametrize("T0,n,W", [(40, 9, 8), (5, 12, 8), (16, 3, 16), (0, 7, 3)])
def test_prefill_then_decode_equals_longer_prefill(oracle_mod, T0, n, W):
    B, H, dk, dv = 2, 2, 6, 5
    T = T0 + n
    q, k, v = _unit(B, H, T, dk, 17), _unit(B, H, T, dk, 18), _unit(B, H, T, dv, 19, unit=False)
    lam, eta, gate = [0.9, 0.7], [0.5, 1.1], [0.2, -0.4]
    full = oracle_mod.tc_prefill(q, k, v, lam, eta, gate, W, want_state=True)
    if T0 > 0:
        st = oracle_mod.tc_prefill(q[:, :, :T0], k[:, :, :T0], v[:, :, :T0], lam, eta, gate, W,
                                   want_state=True)
    else:
        st = dict(ring_k=np.zeros((B, H, W, dk)), ring_v=np.zeros((B, H, W, dv)),
                  A=np.zeros((B, H, dk, dv)), pos=np.zeros(B, dtype=np.int64))
    step = lambda x: np.ascontiguousarray(x[:, :, T0:].transpose(2, 0, 1, 3))  # noqa: E731
    y, st2 = oracle_mod.tc_decode(st, step(q), step(k), step(v), lam, eta, gate)
    np.testing.assert_allclose(y.transpose(1, 2, 0, 3), full["y"][:, :, T0:], rtol=1e-12, atol=1e-13)
    for key in ("ring_k", "ring_v", "A"):
        np.testing.assert_allclose(st2[key], full[key], rtol=1e-12, atol=1e-13)
    assert np.all(st2["pos"] == T)


def test_closed_form_positions_match_recurrence(oracle_mod):
    T, W, dk, dv = 150, 20, 6, 7
    q, k, v = _unit(1, 1, T, dk, 20), _unit(1, 1, T, dk, 21), _unit(1, 1, T, dv, 22, unit=False)
    out = oracle_mod.tc_prefill(q, k, v, [0.93], [0.8], [0.7], W)
    ts = [0, 1, 19, 20, 21, 77, 149]
    y = oracle_mod.tc_output_at(q[0, 0], k[0, 0], v[0, 0], 0.93, 0.8, 0.7, W, ts)
    np.testing.assert_allclose(y, out["y"][0, 0, ts], rtol=1e-12, atol=1e-13)


def _evicted_stream(k, v, W):
    T = k.shape[0]
    kp = np.zeros_like(k)
    vp = np.zeros_like(v)
    kp[W:] = k[:T - W]
    vp[W:] = v[:T - W]
    return kp, vp


def _scan_sequential(q, kp, vp, lam, eta, dt):
    A = np.zeros((q.shape[1], vp.shape[1]), dtype=dt)
    m = np.zeros((q.shape[0], vp.shape[1]), dtype=dt)
    lam, eta = dt(lam), dt(eta)
    for u in range(q.shape[0]):
        A = lam * A + eta * np.outer(kp[u], vp[u]).astype(dt)
        m[u] = q[u] @ A
    return m


def _scan_chunked(q, kp, vp, lam, eta, C, dt):
    """Parallel weighted-sum scan over chunks of C steps: inside a chunk each
    read is lambda^(i+1) q A_prev + sum_{j<=i} eta lambda^(i-j) <q_i,k'_j> v'_j,
    and the chunk folds into the carried state as lambda^n A + K'^T diag(w) V'."""
    T = q.shape[0]
    A = np.zeros((q.shape[1], vp.shape[1]), dtype=dt)
    m = np.zeros((T, vp.shape[1]), dtype=dt)
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        i = np.arange(n)
        D = np.where(i[:, None] >= i[None, :], eta * np.power(lam, np.maximum(i[:, None] - i[None, :], 0)), 0).astype(dt)
        Qc, Kc, Vc = q[c0:c0 + n], kp[c0:c0 + n], vp[c0:c0 + n]
        m[c0:c0 + n] = (np.power(lam, i + 1)[:, None].astype(dt) * (Qc @ A)) + ((Qc @ Kc.T) * D) @ Vc
        w = (eta * np.power(lam, n - 1 - i)).astype(dt)
        A = dt(lam ** n) * A + (Kc * w[:, None]).T @ Vc
    return m


def test_parallel_scan_equals_sequential_writes(oracle_mod):
    """Methodology 2: the parallel weighted-sum scan reproduces the per-token
    writes.  float64: chunked form vs the oracle's L2 read to 1e-12 for every
    chunk size -- this is the exact gate.  float32, on the fp32 workload
    (T=256, d=32, W=32, lambda=0.99, eta=0.5): the two forms differ by about
    2.7e-7 relative, above the page's 1e-7, because the sequential float32
    scan is itself about 2.3e-7 from the exact result (the chunked one about
    1.4e-7); the float32 check therefore bounds both at 5e-7 and the exact
    equality is held in float64."""
    inp = synth.tc_inputs(1, 1, 256, 32, 32, 32, dtype="f32", seed=0, lam=0.99, eta=0.5, gate=0.0)
    q, k, v = (x[0, 0].double().numpy() for x in (inp.q, inp.k, inp.v))
    out = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, 32, want_m=True)
    kp, vp = _evicted_stream(k, v, 32)
    lam = float(inp.lam[0])            # lambda as the layer receives it (float32 0.99)
    for C in (1, 16, 64, 100, 256):
        m64 = _scan_chunked(q, kp, vp, lam, 0.5, C, np.float64)
        assert rel_l2(m64, out["m"][0, 0]) < 1e-12
    q32, kp32, vp32 = (x.astype(np.float32) for x in (q, kp, vp))
    seq32 = _scan_sequential(q32, kp32, vp32, lam, 0.5, np.float32)
    par32 = _scan_chunked(q32, kp32, vp32, np.float32(lam), np.float32(0.5), 64, np.float32)
    err = rel_l2(par32, seq32)
    assert err < 5e-7, err
    # Both float32 forms stay within float32 rounding of the float64 oracle.
    assert rel_l2(seq32, out["m"][0, 0]) < 5e-7
    assert rel_l2(par32, out["m"][0, 0]) < 5e-7


def test_chunk_averaging_negative_control(oracle_mod):
    """Methodology 2: summarising a chunk by k_bar (x) v_bar adds C^2 - C cross
    terms k_i (x) v_j.  That shortcut must miss the oracle by far more than
    the 1e-5 parity bar, so the parity tests can tell the two apart."""
    inp = synth.tc_inputs(1, 1, 256, 32, 32, 32, dtype="f32", seed=0, lam=0.99, eta=0.5, gate=0.0)
    q, k, v = (x[0, 0].double().numpy() for x in (inp.q, inp.k, inp.v))
    out = oracle_mod.tc_prefill(inp.q, inp.k, inp.v, inp.lam, inp.eta, inp.gate, 32, want_m=True)
    kp, vp = _evicted_stream(k, v, 32)
    C, lam, eta = 16, float(inp.lam[0]), 0.5
    A = np.zeros((32, 32))
    ends, m_avg = [], []
    for c0 in range(0, 256, C):
        kb, vb = kp[c0:c0 + C].mean(0), vp[c0:c0 + C].mean(0)
        A = lam ** C * A + eta * C * np.outer(kb, vb)
        u = c0 + C - 1                      # read after the chunk's writes
        ends.append(u)
        m_avg.append(q[u] @ A)
    assert rel_l2(np.array(m_avg), out["m"][0, 0, ends]) > 1e-2
