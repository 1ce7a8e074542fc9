"""Helpers shared by the GPU parity tests: device runs through the C ABI and
the tolerance checks (oracle on the host, float64)."""

import numpy as np
import torch

import selective_state_space_130_b300 as ss

# max |y_gpu - y_ref| <= REL[in_dtype] * rms(y_ref); bf16 outputs add one bf16
# rounding of the reference value (2^-8 |y_ref| bounds half an ulp with margin).
REL = {torch.float32: 1e-4, torch.bfloat16: 5e-3}
BF16_OUT_REL = 2.0 ** -8


def to_dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_scan(x, out_dtype=torch.float32, sg=0, chunk=0, check_status=True, workers=0):
    """Run ss_scan_fwd on the GPU for host inputs x; returns float64 numpy (y, h_last)."""
    y, h = run_scan_dev(x, out_dtype, sg, chunk, check_status, workers)
    return y.double().cpu().numpy(), h.double().cpu().numpy()


def run_scan_dev(x, out_dtype=torch.float32, sg=0, chunk=0, check_status=True, workers=0):
    """Run ss_scan_fwd on the GPU for host inputs x; returns the device tensors (y, h_last)."""
    d = to_dev(x)
    Bt, L, Dm = d["u"].shape
    ss.ss_scan_set_tuning(sg, chunk, workers)
    try:
        ws_bytes = ss.ss_scan_fwd_workspace_size(Bt, L, Dm, 16)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
        y, h = ss.ss_scan_fwd(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d.get("D"), d.get("z"),
                              d.get("delta_bias"), d.get("h0"), out_dtype=out_dtype, workspace=ws)
        if check_status:
            ss.ss_scan_status(ws)
        torch.cuda.synchronize()
    finally:
        ss.ss_scan_set_tuning(0, 0)
    return y, h


def assert_close(got, ref, in_dtype, out_bf16=False, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    lim = REL[in_dtype] * rms + (BF16_OUT_REL * np.abs(ref) if out_bf16 else 0.0)
    err = np.abs(got - ref)
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err - lim), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; max err {err.max():.3e}, "
                             f"rms(ref) {rms:.3e}, worst at {i}: got {got[i]:.6e} ref {ref[i]:.6e}")
    return float(err.max() / rms) if rms else 0.0


def sample_channels(batch, dim, n, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, batch, size=n)
    d = rng.integers(0, dim, size=n)
    # always include the first and last channel of the first and last batch element
    extra = np.array([[0, 0], [batch - 1, dim - 1], [0, dim - 1]])
    ch = np.concatenate([np.stack([b, d], axis=1), extra])
    return np.unique(ch, axis=0)
