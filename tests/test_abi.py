"""C-ABI checks that need no GPU: the library loads, exports every function
the header declares, sizes workspaces, and rejects bad arguments on the host
before anything is enqueued (each call below fails validation, so no kernel
launches and no pointer is dereferenced)."""
import ctypes
import os
import re

import pytest

from outer_product_associative_chunked_b300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "opam.h")
FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call here fails validation first


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_binding_exports():
    assert sorted(binding.EXPORTS) == _declared_functions()


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def _enum_values():
    text = open(HEADER).read()
    body = re.search(r"typedef enum \{([^{}]*)\} opam_status;", text).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"(OPAM_\w+)\s*=\s*(-?\d+)", body)}


def test_status_values_match_the_boundary_contract():
    # the boundary's status codes: timeout -4, workspace -5
    assert _enum_values() == {"OPAM_OK": 0, "OPAM_ERR_INVALID_ARG": -1, "OPAM_ERR_UNSUPPORTED": -2,
                              "OPAM_ERR_CUDA": -3, "OPAM_ERR_TIMEOUT": -4, "OPAM_ERR_WORKSPACE": -5}
    assert binding.OPAM_ERR_TIMEOUT == -4 and binding.OPAM_ERR_WORKSPACE == -5
    m = re.search(r"#define OPAM_STATUS_BYTES (\d+)u", open(HEADER).read())
    assert int(m.group(1)) == binding.STATUS_BYTES


def test_every_workspace_holds_the_status_block(L):
    sb = binding.STATUS_BYTES
    assert L.tc_window_forward_workspace_size(1, 1, 16, 64, 64, 4, 1) == sb
    assert L.tc_window_forward_workspace_size(1, 1, 0, 64, 64, 4, 1) == 0
    assert L.tc_layer_forward_workspace_size(1, 1, 16, 64, 64, 4, 1) > sb
    assert L.tc_layer_forward_workspace_size(1, 1, 16, 32, 32, 4, 0) > sb
    assert L.delta_rule_forward_workspace_size(1, 1, 16, 64, 64, 0, 0) > sb
    assert L.sparse_linattn_forward_workspace_size(1, 1, 16, 512, 64) > sb
    st = binding.TCStateStruct(FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 32, 32, 0)
    assert L.tc_decode_step_workspace_size(ctypes.byref(st)) > sb


def test_check_and_selftest_reject_bad_workspace(L):
    assert L.opam_check_device_error(FAKE + 4, None) == -1      # misaligned, rejected before any sync
    assert L.opam_selftest_bounded_wait(0, 1000, None, None) == -1
    assert L.opam_selftest_bounded_wait(0, 1000, FAKE + 8, None) == -1


def test_workspace_sizes(L):
    assert binding.tc_layer_forward_workspace_size(4, 8, 4096, 64, 64, 512, __import__("torch").bfloat16) > 0
    assert L.tc_layer_forward_workspace_size(1, 1, 16, 96, 96, 4, 0) == 0       # unsupported head
    assert L.tc_layer_forward_workspace_size(1, 1, 0, 64, 64, 4, 0) == 0        # empty sequence
    assert L.delta_rule_forward_workspace_size(8, 16, 8192, 128, 128, 64, 1) > 0
    assert L.delta_rule_forward_workspace_size(1, 1, 8, 64, 64, 48, 1) == 0     # bad chunk
    assert L.sparse_linattn_forward_workspace_size(2, 4, 2048, 16384, 256) > 0
    assert L.sparse_linattn_forward_workspace_size(1, 1, 8, 100000, 64) == 0    # N too wide
    st = binding.TCStateStruct(FAKE, FAKE, FAKE, FAKE, 64, 16, 2048, 128, 128, 1)
    assert L.tc_decode_step_workspace_size(ctypes.byref(st)) > 0


def _tc(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=1, B=1, H=1, T=16, dk=64, dv=64, W=4, lam=FAKE, eta=FAKE,
             gate=FAKE, scale=0.0, y=FAKE, state=None, ws=FAKE, wsb=0, stream=None)
    a.update(kw)
    a["wsb"] = kw.get("wsb", L.tc_layer_forward_workspace_size(a["B"], a["H"], a["T"], a["dk"], a["dv"],
                                                               a["W"], a["dtype"]))
    rc = L.tc_layer_forward(a["q"], a["k"], a["v"], a["dtype"], a["B"], a["H"], a["T"], a["dk"], a["dv"],
                            a["W"], a["lam"], a["eta"], a["gate"], a["scale"], a["y"], a["state"],
                            a["ws"], a["wsb"], a["stream"])
    return rc, binding.last_error()


def test_tc_forward_rejects_bad_arguments(L):
    assert _tc(L, q=None)[0] == -1
    assert _tc(L, y=FAKE + 4)[0] == -1            # misaligned
    assert _tc(L, T=0)[0] == -1
    assert _tc(L, W=0)[0] == -1
    assert _tc(L, dtype=7)[0] == -1
    assert _tc(L, dk=96, dv=96)[0] == -2
    rc, msg = _tc(L, wsb=16)
    assert rc == -5 and "workspace" in msg
    assert _tc(L, ws=None)[0] == -5
    bad_state = binding.TCStateStruct(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 64, 64, 1)  # W mismatch
    assert _tc(L, state=ctypes.byref(bad_state))[0] == -1


def test_decode_rejects_bad_arguments(L):
    st = binding.TCStateStruct(FAKE, FAKE, FAKE, FAKE, 2, 2, 16, 64, 64, 1)
    need = L.tc_decode_step_workspace_size(ctypes.byref(st))
    call = lambda st, ws=need, q=FAKE: L.tc_decode_step(  # noqa: E731
        ctypes.byref(st), q, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, FAKE, FAKE, ws, None)
    assert call(st, q=None) == -1
    assert call(st, ws=need - 1) == -5
    st2 = binding.TCStateStruct(None, FAKE, FAKE, FAKE, 2, 2, 16, 64, 64, 1)
    assert call(st2) == -1
    st3 = binding.TCStateStruct(FAKE, FAKE, FAKE, FAKE, 2, 2, 16, 48, 48, 1)
    assert call(st3) == -2
    assert L.tc_decode_step(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, FAKE, FAKE, need, None) == -1


def test_delta_and_sparse_reject_bad_arguments(L):
    ws = L.delta_rule_forward_workspace_size(1, 1, 16, 64, 64, 0, 1)
    d = lambda **kw: L.delta_rule_forward(  # noqa: E731
        kw.get("q", FAKE), FAKE, FAKE, kw.get("beta", FAKE), 1, 1, 1, 16, 64, 64, kw.get("chunk", 0),
        kw.get("S0", None), None, FAKE, FAKE, kw.get("ws", ws), None)
    assert d(q=None) == -1
    assert d(beta=None) == -1
    assert d(chunk=48) == -2
    assert d(S0=FAKE + 8) == -1
    assert d(ws=ws - 1) == -5
    wss = L.sparse_linattn_forward_workspace_size(1, 1, 16, 512, 64)
    s = lambda **kw: L.sparse_linattn_forward(  # noqa: E731
        FAKE, kw.get("k", FAKE), FAKE, 1, 1, 16, kw.get("N", 512), kw.get("dv", 64), None, None, FAKE,
        FAKE, kw.get("ws", wss), None)
    assert s(k=None) == -1
    assert s(dv=48) == -2
    assert s(N=0) == -1
    assert s(ws=wss - 1) == -5


def test_delta_decode_rejects_bad_arguments(L):
    call = lambda **kw: L.delta_decode_step(  # noqa: E731
        kw.get("S", FAKE), kw.get("q", FAKE), FAKE, FAKE, kw.get("beta", FAKE), kw.get("dtype", 1),
        kw.get("B", 2), 3, kw.get("dk", 64), kw.get("dv", 128), kw.get("y", FAKE), None)
    assert call(S=None) == -1
    assert call(q=FAKE + 4) == -1                 # misaligned
    assert call(beta=None) == -1
    assert call(y=None) == -1
    assert call(B=0) == -1
    assert call(dtype=5) == -1
    assert call(dk=96) == -2
    assert call(dv=16) == -2
    assert call(B=70000) == -2                    # B*H above the grid limit
    assert "delta_decode_step" in binding.last_error()


def test_window_forward_rejects_bad_arguments(L):
    call = lambda **kw: L.tc_window_forward(  # noqa: E731
        kw.get("q", FAKE), FAKE, FAKE, kw.get("dtype", 1), 1, 2, kw.get("T", 16), kw.get("dk", 64), 64,
        kw.get("W", 4), 0.0, kw.get("y", FAKE), kw.get("ws", FAKE), kw.get("wsb", 256), None)
    assert call(q=None) == -1
    assert call(ws=None) == -5
    assert call(wsb=255) == -5
    assert call(y=FAKE + 8) == -1                 # misaligned
    assert call(T=0) == -1
    assert call(W=0) == -1
    assert call(dtype=3) == -1
    assert call(dk=96) == -2
    assert "tc_window_forward" in binding.last_error()


def test_binding_rejects_mismatched_tensors():
    """The binding checks every tensor against q (and the state) before the
    C call: the ABI takes all extents from q, so a mismatched k, v, scalar,
    state or output would otherwise be accessed out of bounds on the device.
    CPU tensors with a patched placement check stand in for device tensors;
    every case raises before any pointer reaches the library."""
    import torch
    orig = binding._dev
    binding._dev = lambda *ts: None   # placement is checked elsewhere; shapes here
    try:
        bf, f32 = torch.bfloat16, torch.float32
        q = torch.zeros(2, 3, 16, 64, dtype=bf)
        v = torch.zeros(2, 3, 16, 32, dtype=bf)
        h = torch.zeros(3)
        bad = [
            dict(k=torch.zeros(2, 3, 16, 64, dtype=f32)),           # dtype differs from q
            dict(k=torch.zeros(2, 3, 15, 64, dtype=bf)),            # T differs
            dict(v=torch.zeros(2, 3, 16, 32, dtype=f32)),
            dict(lam=torch.zeros(4)),                               # not [H]
            dict(gate=torch.zeros(3, dtype=torch.float64)),
            dict(out=torch.zeros(2, 3, 16, 64, dtype=bf)),          # d_v of out differs from v
        ]
        for kw in bad:
            a = dict(q=q, k=q, v=v, lam=h, eta=h, gate=h)
            a.update(kw)
            with pytest.raises(ValueError):
                binding.tc_layer_forward(a["q"], a["k"], a["v"], a["lam"], a["eta"], a["gate"], 4,
                                         out=kw.get("out"))
        st = binding.TCState.__new__(binding.TCState)
        st.B, st.H, st.W, st.d_k, st.d_v, st.dtype = 2, 3, 8, 64, 32, bf   # W differs from the call
        with pytest.raises(ValueError):
            binding.tc_layer_forward(q, q, v, h, h, h, 4, state=st)
        with pytest.raises(ValueError):
            binding.tc_window_forward(q, q[:, :, :8], v, 4)
        st.W = 4
        st.ring_k = torch.zeros(2, 3, 4, 64, dtype=bf)
        st.ring_v = torch.zeros(2, 3, 4, 32, dtype=bf)
        st.A = torch.zeros(2, 3, 64, 32)
        st.pos = torch.zeros(2, dtype=torch.int32)                  # pos must be int64
        with pytest.raises(ValueError):
            binding.tc_decode_step(st, q[:, :, 0], q[:, :, 0], v[:, :, 0], h, h, h)
        st.pos = torch.zeros(2, dtype=torch.int64)
        with pytest.raises(ValueError):                             # v has d_k columns, not d_v
            binding.tc_decode_step(st, q[:, :, 0], q[:, :, 0], q[:, :, 0], h, h, h)
        beta = torch.zeros(2, 3, 16)
        with pytest.raises(ValueError):
            binding.delta_rule_forward(q, q, v, beta[:, :, :8])
        with pytest.raises(ValueError):
            binding.delta_rule_forward(q, q, v, beta, S0=torch.zeros(2, 3, 32, 64))
        with pytest.raises(ValueError):
            binding.delta_decode_step(torch.zeros(2, 3, 64, 32), q[:, :, 0], q[:, :, 0], v[:, :, 0],
                                      torch.zeros(2, 4))
        qs = torch.zeros(1, 2, 8, 512)
        with pytest.raises(ValueError):
            binding.sparse_linattn_forward(qs, qs[..., :256], torch.zeros(1, 2, 8, 64))
        with pytest.raises(ValueError):
            binding.sparse_linattn_forward(qs.to(bf), qs.to(bf), torch.zeros(1, 2, 8, 64, dtype=bf))
        with pytest.raises(ValueError):
            binding.sparse_linattn_forward(qs, qs, torch.zeros(1, 2, 8, 64), S_out=torch.zeros(1, 2, 64, 512))
    finally:
        binding._dev = orig
