"""GPU parity where the element offsets of a [batch, seqlen, dim] tensor pass
2^31 and 2^32: the scan in its chunked mode (few channel blocks, long
sequences) and in its stream-K mode (more channel blocks than SMs), and the
convolution front-end. The inputs are symbol tables (workloads.gen.
symbol_scan_inputs), expanded on the device by an index copy; the oracle
recomputes sampled channels from the same tables, among them channels of the
last batch elements, whose offsets lie past 2^32. A 32-bit wrap of an offset
would read batch element b - 4 (chunked shape) or an earlier timestep, with
other symbols, and fail the comparison."""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close
from workloads import gen

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16
KEYS = ("u", "delta_raw", "z")


def _host_channels(x, b, ds):
    """The scan inputs of channels ds of batch element b, as a [1, L, len(ds)] problem."""
    ds = torch.as_tensor(ds)
    out = {k: gen.gather_symbols(x["tables"][k][:, ds], x["symbols"][k][b:b + 1]) for k in KEYS}
    out.update(B=x["B"][b:b + 1].contiguous(), C=x["C"][b:b + 1].contiguous(), A=x["A"][ds].contiguous(),
               D=x["D"][ds].contiguous(), delta_bias=x["delta_bias"][ds].contiguous(), h0=None)
    return out


def _sample(batch, dim, seed):
    rng = np.random.default_rng(seed)
    ch = {(0, 0), (batch - 1, dim - 1), (batch - 1, 0), (batch // 2, dim // 2)}
    for _ in range(8):
        ch.add((int(rng.integers(0, batch)), int(rng.integers(0, dim))))
    by_b = {}
    for b, d in sorted(ch):
        by_b.setdefault(b, []).append(d)
    return by_b


# (batch, seqlen, dim): 5 x 2^20 x 1024 takes the chunked mode (40 channel
# blocks), 4 x 2^18 x 5120 the stream-K mode (160 blocks); both 5.37e9 elements
SHAPES = [(5, 1 << 20, 1024), (4, 1 << 18, 5120)]


@pytest.mark.parametrize("shape", SHAPES, ids=["chunked", "streamk"])
def test_scan_and_conv1d_offsets_beyond_2_32(shape):
    Bt, L, Dm = shape
    n = Bt * L * Dm
    assert n > 1 << 32
    need = 5 * n * 2 + (8 << 30)  # u, delta_raw, z, y and the convolution's y in bf16, plus slack
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB of free device memory, {free / 1e9:.0f} GB free")
    x = gen.symbol_scan_inputs(Bt, L, Dm, seed=5)
    dev = torch.device("cuda", 0)
    full = {k: gen.gather_symbols(x["tables"][k].to(dev), x["symbols"][k].to(dev)) for k in KEYS}
    B, C = x["B"].to(dev), x["C"].to(dev)
    A, Dk, bias = x["A"].to(dev), x["D"].to(dev), x["delta_bias"].to(dev)
    y, h = ss.ss_scan_fwd(full["u"], full["delta_raw"], A, B, C, Dk, full["z"], bias)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(h).all())
    assert not bool(torch.isnan(y).any())
    by_b = _sample(Bt, Dm, seed=Bt + Dm)
    for b, ds in by_b.items():
        yr, hr = oracle.scan(_host_channels(x, b, ds))
        idx = torch.tensor(ds, device=dev)
        yg = y[b][:, idx].double().cpu().numpy()  # [L, k]
        hg = h[b][idx].double().cpu().numpy()     # [k, N]
        assert_close(yg, yr[0], BF16, out_bf16=True, what=f"scan y, batch {b}, channels {ds}")
        assert_close(hg, hr[0], BF16, what=f"scan h_last, batch {b}, channels {ds}")
    del y, h, full["delta_raw"], full["z"]
    # the convolution front-end over u
    g = torch.Generator().manual_seed(Bt * 7 + 1)
    w = (0.5 * torch.randn(Dm, 4, generator=g)).contiguous()
    cb = (0.1 * torch.randn(Dm, generator=g)).contiguous()
    yc, _ = ss.ss_conv1d_fwd(full["u"], w.to(dev), cb.to(dev), None)
    torch.cuda.synchronize()
    assert not bool(torch.isnan(yc).any())
    for b, ds in by_b.items():
        dst = torch.as_tensor(ds)
        xu = gen.gather_symbols(x["tables"]["u"][:, dst], x["symbols"]["u"][b:b + 1])
        yr, _ = oracle.conv1d({"x": xu, "weight": w[dst].contiguous(), "bias": cb[dst].contiguous(), "state": None})
        yg = yc[b][:, torch.tensor(ds, device=dev)].double().cpu().numpy()
        assert_close(yg, yr[0], BF16, out_bf16=True, what=f"conv1d y, batch {b}, channels {ds}")
