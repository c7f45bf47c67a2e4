"""Pins for the DeltaNet delta-rule oracle (CPU only).

Page: molayo1419.me, "DeltaNet-family linear attention variants".
- "DeltaNet: write the prediction error instead of the value":
  e_t = beta_t (v_t - S_{t-1} k_t), S_t = S_{t-1} + e_t k_t^T, beta in [0,1];
  re-reading with the same key gives (1 - beta) S_{t-1} k_t + beta v_t, which
  is exactly v_t when beta = 1.
- "The update is local in key space": a query orthogonal to k_t sees no change.
- "Derivation from a reconstruction loss": the update is one gradient step of
  size beta on 1/2 ||S k_t - v_t||^2.
Each pin compares the oracle with something computed another way: a
hand-worked fixture, torch autograd, identities of the page, a closed form for
orthonormal keys, the chunked (WY) algebra, or pure-Python brute force.
"""
import numpy as np
import pytest
import torch

from helpers import load_golden


def _inputs(B, H, T, dk, dv, seed, unit_k=True):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, T, dk, generator=g, dtype=torch.float64)
    k = torch.randn(B, H, T, dk, generator=g, dtype=torch.float64)
    if unit_k:
        k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, H, T, dv, generator=g, dtype=torch.float64)
    beta = torch.sigmoid(torch.randn(B, H, T, generator=g, dtype=torch.float64))
    return q.numpy(), k.numpy(), v.numpy(), beta.numpy()


def _S(keymajor):
    """Key-major storage [d_k, d_v] -> the page's S in R^{d_v x d_k}."""
    return np.asarray(keymajor).T


def test_hand_worked_fixture(oracle_mod):
    g = load_golden("delta_d2_t3.txt")
    out = oracle_mod.delta(g["q"][None, None], g["k"][None, None], g["v"][None, None],
                           g["beta"].reshape(1, 1, -1), want_state=True)
    np.testing.assert_allclose(out["y"][0, 0], g["y"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(out["S"][0, 0], g["S_final_keymajor"], rtol=0, atol=1e-14)


def _brute_delta(q, k, v, beta):
    T, dk, dv = len(q), len(q[0]), len(v[0])
    S = [[0.0] * dk for _ in range(dv)]
    ys = []
    for t in range(T):
        pred = [sum(S[i][j] * k[t][j] for j in range(dk)) for i in range(dv)]
        e = [beta[t] * (v[t][i] - pred[i]) for i in range(dv)]
        for i in range(dv):
            for j in range(dk):
                S[i][j] += e[i] * k[t][j]
        ys.append([sum(S[i][j] * q[t][j] for j in range(dk)) for i in range(dv)])
    return np.array(ys)


@pytest.mark.parametrize("T,dk,dv", [(16, 3, 2), (16, 4, 5), (1, 2, 2), (7, 6, 3)])
def test_bruteforce_small(oracle_mod, T, dk, dv):
    q, k, v, beta = _inputs(1, 1, T, dk, dv, T + dk, unit_k=False)
    out = oracle_mod.delta(q, k, v, beta)
    ref = _brute_delta(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), beta[0, 0].tolist())
    np.testing.assert_allclose(out["y"][0, 0], ref, rtol=1e-12, atol=1e-12)


def _states(oracle_mod, q, k, v, beta, t):
    """S_{t-1} and S_t (page orientation) for unit (0, 0)."""
    prev = oracle_mod.delta(q[:, :, :t], k[:, :, :t], v[:, :, :t], beta[:, :, :t], want_state=True)
    cur = oracle_mod.delta(q[:, :, :t + 1], k[:, :, :t + 1], v[:, :, :t + 1], beta[:, :, :t + 1],
                           want_state=True)
    return _S(prev["S"][0, 0]), _S(cur["S"][0, 0])


def test_beta_one_reread_returns_value(oracle_mod):
    q, k, v, beta = _inputs(1, 1, 12, 8, 6, 30)
    beta[0, 0, 11] = 1.0
    _, St = _states(oracle_mod, q, k, v, beta, 11)
    np.testing.assert_allclose(St @ k[0, 0, 11], v[0, 0, 11], rtol=0, atol=1e-14)


@pytest.mark.parametrize("t", [0, 5, 9])
def test_general_beta_reread_interpolates(oracle_mod, t):
    q, k, v, beta = _inputs(1, 1, 10, 8, 6, 31)
    Sp, St = _states(oracle_mod, q, k, v, beta, t)
    kt, vt, bt = k[0, 0, t], v[0, 0, t], beta[0, 0, t]
    np.testing.assert_allclose(St @ kt, (1 - bt) * (Sp @ kt) + bt * vt, rtol=1e-13, atol=1e-14)


def test_orthogonal_query_unchanged(oracle_mod):
    q, k, v, beta = _inputs(1, 1, 9, 8, 5, 32, unit_k=False)
    Sp, St = _states(oracle_mod, q, k, v, beta, 8)
    kt = k[0, 0, 8]
    rng = np.random.default_rng(3)
    for _ in range(3):
        x = rng.standard_normal(8)
        x -= (x @ kt) / (kt @ kt) * kt
        np.testing.assert_allclose(St @ x, Sp @ x, rtol=1e-13, atol=1e-13)


def test_update_is_gradient_step_on_reconstruction_loss(oracle_mod):
    """S_t = S_{t-1} - beta_t grad_S 1/2 ||S k_t - v_t||^2, gradient by autograd."""
    q, k, v, beta = _inputs(1, 1, 7, 6, 4, 33, unit_k=False)
    Sp, St = _states(oracle_mod, q, k, v, beta, 6)
    S = torch.tensor(Sp, requires_grad=True)
    kt, vt = torch.tensor(k[0, 0, 6]), torch.tensor(v[0, 0, 6])
    loss = 0.5 * ((S @ kt - vt) ** 2).sum()
    loss.backward()
    np.testing.assert_allclose(St, Sp - beta[0, 0, 6] * S.grad.numpy(), rtol=1e-13, atol=1e-14)


def test_beta_zero_keeps_initial_state(oracle_mod):
    q, k, v, beta = _inputs(2, 1, 11, 5, 4, 34)
    beta[:] = 0.0
    S0 = np.random.default_rng(4).standard_normal((2, 1, 5, 4))
    out = oracle_mod.delta(q, k, v, beta, S0=S0, want_state=True)
    np.testing.assert_array_equal(out["S"], S0)
    np.testing.assert_allclose(out["y"], np.einsum("bhtj,bhji->bhti", q, S0), rtol=1e-13)


def test_orthonormal_keys_beta_one_store_every_pair(oracle_mod):
    """With orthonormal keys and beta = 1 each write replaces exactly its own
    association: S = sum_t v_t k_t^T, and reading k_s returns v_s."""
    d, T = 8, 6
    Qm, _ = np.linalg.qr(np.random.default_rng(5).standard_normal((d, d)))
    k = Qm[:T][None, None]
    v = np.random.default_rng(6).standard_normal((1, 1, T, 3))
    q = np.random.default_rng(7).standard_normal((1, 1, T, d))
    out = oracle_mod.delta(q, k, v, np.ones((1, 1, T)), want_state=True)
    np.testing.assert_allclose(_S(out["S"][0, 0]), v[0, 0].T @ k[0, 0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(_S(out["S"][0, 0]) @ k[0, 0].T, v[0, 0].T, rtol=1e-12, atol=1e-13)


def delta_chunked_wy(q, k, v, beta, C, S0=None):
    """Chunked form of the same recurrence (row i = token i of a chunk,
    S0 = state at chunk start):  (I + diag(beta) strict_lower(K K^T)) U =
    diag(beta)(V - K S0^T), so U = T diag(beta) V - T diag(beta) K S0^T with
    T the inverse of that unit-lower matrix; O = Q S0^T + (Q K^T masked to
    j <= i) U; S_end = S0 + U^T K."""
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, dtype=np.float64)
    y = np.zeros((T, dv))
    for c0 in range(0, T, C):
        K, V, Q, b = k[c0:c0 + C], v[c0:c0 + C], q[c0:c0 + C], beta[c0:c0 + C]
        n = K.shape[0]
        Tm = np.linalg.inv(np.eye(n) + b[:, None] * np.tril(K @ K.T, -1))
        Wt, Ut = Tm @ (b[:, None] * K), Tm @ (b[:, None] * V)
        U = Ut - Wt @ S.T
        y[c0:c0 + n] = Q @ S.T + np.tril(Q @ K.T) @ U
        S = S + U.T @ K
    return y, S


@pytest.mark.parametrize("T,C", [(200, 64), (64, 64), (65, 16), (37, 1), (50, 8)])
def test_chunked_wy_form_equals_recurrence(oracle_mod, T, C):
    q, k, v, beta = _inputs(1, 2, T, 16, 12, 35 + T)
    S0 = np.random.default_rng(8).standard_normal((1, 2, 16, 12)) * 0.3
    out = oracle_mod.delta(q, k, v, beta, S0=S0, want_state=True)
    for h in range(2):
        y, S = delta_chunked_wy(q[0, h], k[0, h], v[0, h], beta[0, h], C, S0=_S(S0[0, h]))
        np.testing.assert_allclose(y, out["y"][0, h], rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(S, _S(out["S"][0, h]), rtol=1e-11, atol=1e-11)


def test_split_sequence_through_exported_state(oracle_mod):
    q, k, v, beta = _inputs(2, 2, 30, 6, 5, 36)
    full = oracle_mod.delta(q, k, v, beta, want_state=True)
    a = oracle_mod.delta(q[:, :, :13], k[:, :, :13], v[:, :, :13], beta[:, :, :13], want_state=True)
    b = oracle_mod.delta(q[:, :, 13:], k[:, :, 13:], v[:, :, 13:], beta[:, :, 13:], S0=a["S"],
                         want_state=True)
    np.testing.assert_allclose(b["y"], full["y"][:, :, 13:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["S"], full["S"], rtol=1e-12, atol=1e-13)


def test_token_by_token_decode_equals_whole_sequence(oracle_mod):
    """Decode reading: one-token calls chained through the exported state give
    the same outputs and final state as one call over the whole sequence."""
    q, k, v, beta = _inputs(2, 3, 9, 8, 5, 41)
    S0 = np.random.default_rng(3).standard_normal((2, 3, 8, 5)) * 0.3
    full = oracle_mod.delta(q, k, v, beta, S0=S0, want_state=True)
    S = S0
    for t in range(9):
        one = oracle_mod.delta(q[:, :, t:t + 1], k[:, :, t:t + 1], v[:, :, t:t + 1], beta[:, :, t:t + 1],
                               S0=S, want_state=True)
        np.testing.assert_allclose(one["y"][:, :, 0], full["y"][:, :, t], rtol=1e-12, atol=1e-13)
        S = one["S"]
    np.testing.assert_allclose(S, full["S"], rtol=1e-12, atol=1e-13)
