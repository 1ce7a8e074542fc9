"""GPU parity on the full-size workloads, in the launch configuration the
benchmark times. The oracle recomputes sampled channels over the whole
sequence (and, for decode, every step of the sampled channels); the rest of
the output is checked for properties that hold at any size."""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close, run_scan_dev, sample_channels, to_dev
from workloads import configs, gen

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


def _check_sampled(w, x, y, h, out_bf16, nsample, seed):
    """y, h: device tensors of the whole problem; the sampled channels go to the host."""
    assert bool(torch.isfinite(y).all()) and bool(torch.isfinite(h).all())
    ch = sample_channels(w.batch, w.dim, nsample, seed)
    yr, hr = oracle.scan(x, channels=ch)
    ib = torch.tensor(ch[:, 0], device=y.device)
    idd = torch.tensor(ch[:, 1], device=y.device)
    yg = y[ib, :, idd].double().cpu().numpy()   # [n, L]
    hg = h[ib, idd].double().cpu().numpy()      # [n, N]
    in_dt = torch.float32 if w.in_dtype == "f32" else BF16
    e1 = assert_close(yg, yr, in_dt, out_bf16=out_bf16, what=f"{w.name} sampled y")
    e2 = assert_close(hg, hr, in_dt, what=f"{w.name} sampled h_last")
    return e1, e2


@pytest.mark.parametrize("name,nsample", [("mamba130m_layer", 48), ("mamba2p8b_layer", 48)])
@pytest.mark.parametrize("out", [torch.float32, BF16])
def test_layer_configs(name, nsample, out):
    w = configs.get_config(name)
    x = gen.make_scan_inputs(w)
    y, h = run_scan_dev(x, out)
    _check_sampled(w, x, y, h, out == BF16, nsample, seed={"mamba130m_layer": 11, "mamba2p8b_layer": 22}[name])


def test_dna_1m_config():
    w = configs.DNA_1M
    x = gen.make_scan_inputs(w)
    assert ss.ss_scan_fwd_workspace_size(w.batch, w.seqlen, w.dim) > 0  # the cross-chunk carry path is used
    y, h = run_scan_dev(x, BF16)
    _check_sampled(w, x, y, h, True, 20, seed=3)


def test_decode_config():
    w = configs.DECODE256
    pre = gen.make_scan_inputs(w.prefix)
    # prefix scan on the GPU gives the initial state of the 256 streams
    d = to_dev(pre)
    _, h = ss.ss_scan_fwd(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"])
    del d["u"], d["delta_raw"], d["z"]
    steps = gen.make_decode_steps(w, 0, w.steps)
    ch = sample_channels(w.streams, w.dim, 40, seed=4)
    idx_b = torch.tensor(ch[:, 0], device="cuda")
    idx_d = torch.tensor(ch[:, 1], device="cuda")
    su = {k: v.cuda() for k, v in steps.items()}
    ys = torch.empty((w.steps, len(ch)), dtype=torch.float32, device="cuda")
    y = torch.empty((w.streams, w.dim), dtype=BF16, device="cuda")
    for k in range(w.steps):
        ss.ss_state_update(h, su["u"][k], su["delta_raw"][k], d["A"], su["B"][k], su["C"][k], d["D"], su["z"][k],
                           d["delta_bias"], y=y)
        ys[k] = y[idx_b, idx_d].float()
    torch.cuda.synchronize()
    hg = h.double().cpu().numpy()
    assert np.isfinite(hg).all()
    # oracle: its own prefix scan, then every step, for the sampled channels
    _, h_pre = oracle.scan(pre, channels=ch)
    hs = np.zeros((w.streams, w.dim, 16))
    for i, (b, dd) in enumerate(ch):
        hs[b, dd] = h_pre[i]
    yr = np.empty((w.steps, len(ch)))
    for k in range(w.steps):
        step = {key: steps[key][k] for key in ("u", "delta_raw", "z", "B", "C")}
        step.update(A=pre["A"], D=pre["D"], delta_bias=pre["delta_bias"])
        yr[k] = oracle.state_update(hs, step, channels=ch)
    assert_close(ys.double().cpu().numpy(), yr, BF16, out_bf16=True, what="decode y (every step)")
    assert_close(np.stack([hg[b, dd] for b, dd in ch]), np.stack([hs[b, dd] for b, dd in ch]), BF16,
                 what="decode final state")
