"""Small helpers shared by the tests (fixture parsing, error measures)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    """Parse a ``key: value`` fixture; ';' separates matrix rows."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            rows = [r.split() for r in val.split(";")]
            arr = np.array([[float(x) for x in r] for r in rows], dtype=np.float64)
            out[key.strip()] = arr if arr.size > 1 else float(arr.reshape(-1)[0])
    return out


def rel_l2(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def rms_rel(x, ref):
    """RMS(x - ref) / RMS(ref): the bf16-path parity measure."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.mean(ref ** 2))
    return float(np.sqrt(np.mean((x - ref) ** 2)) / (den if den > 0 else 1.0))


# Parity bars for the CUDA path against the float64 oracle.
TOL_F32_REL_L2 = 1e-5      # fp32 inputs / fp32 state
TOL_BF16_RMS = 2e-2        # bf16 inputs / fp32 state, relative to output RMS


def to_np(t):
    """float64 numpy copy of a (device) tensor."""
    return t.detach().to("cpu").double().numpy()


def check_parity(y, ref, dtype, what=""):
    """Apply the parity bar of the given input dtype; return the measured error
    (also printed, so `pytest -s` lists every measured error)."""
    if dtype in ("f32", "float32"):
        err = rel_l2(y, ref)
        print(f"parity {what}: rel L2 {err:.3e} (bar {TOL_F32_REL_L2})")
        assert err <= TOL_F32_REL_L2, f"{what}: rel L2 {err:.3e} > {TOL_F32_REL_L2}"
    else:
        err = rms_rel(y, ref)
        print(f"parity {what}: RMS {err:.3e} of output RMS (bar {TOL_BF16_RMS})")
        assert err <= TOL_BF16_RMS, f"{what}: RMS err {err:.3e} > {TOL_BF16_RMS} of output RMS"
    return err


def guarded(shape, dtype, device="cuda", pad=4096):
    """Output tensor followed by a canary tail; returns (view, full buffer)."""
    import torch
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + pad,), 1234.5, dtype=dtype, device=device)
    return buf[:n].view(*shape), buf


def canary_intact(buf, shape):
    import torch
    n = 1
    for s in shape:
        n *= s
    return bool(torch.all(buf[n:] == 1234.5))
