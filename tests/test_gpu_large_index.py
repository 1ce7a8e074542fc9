"""GPU parity where element offsets pass 2^31 and 2^32, for every kernel:
- the scan in its chunked mode (few channel blocks, long sequences) and in its
  stream-K mode (more channel blocks than SMs), and the convolution front-end;
- the generalised scan (d_state 64, zero-order hold);
- the backward pass;
- the state-space-dual layer;
- the decode step (a state of 5.37e9 elements).

The inputs are symbol tables (workloads.gen.symbol_tensor), expanded on the
device by an index copy. The oracle recomputes sampled channels, heads or
streams from the same tables, among them those of the last batch elements,
whose offsets lie past 2^32. A 32-bit wrap of an offset would read another
batch element or timestep, with other symbols, and fail the comparison."""

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


def _need(nbytes):
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes:
        pytest.skip(f"needs {nbytes / 1e9:.0f} GB of free device memory, {free / 1e9:.0f} GB free")


def _expand(tables, symbols, dev):
    return {k: gen.gather_symbols(tables[k].to(dev), symbols[k].to(dev)) for k in tables}


def test_general_offsets_beyond_2_32():
    # d_state 64, one group, zero-order hold: the CTA kernel with persistent shares
    Bt, L, Dm, N = 4, 1 << 18, 5120, 64
    n = Bt * L * Dm
    _need(4 * n * 2 + (8 << 30))
    x = gen.symbol_scan_inputs(Bt, L, Dm, dstate=N, seed=6)
    dev = torch.device("cuda", 0)
    full = _expand(x["tables"], x["symbols"], dev)
    y, h = ss.ss_scan_fwd_general(full["u"], full["delta_raw"], x["A"].to(dev), x["B"].to(dev), x["C"].to(dev),
                                  x["D"].to(dev), full["z"], x["delta_bias"].to(dev), None, disc="zoh")
    torch.cuda.synchronize()
    assert bool(torch.isfinite(h).all())
    assert not bool(torch.isnan(y).any())
    for b, ds in _sample(Bt, Dm, seed=61).items():
        yr, hr = oracle.scan_general(_host_channels(x, b, ds), 1, "zoh")
        idx = torch.tensor(ds, device=dev)
        assert_close(y[b][:, idx].double().cpu().numpy(), yr[0], BF16, out_bf16=True,
                     what=f"general y, batch {b}, channels {ds}")
        assert_close(h[b][idx].double().cpu().numpy(), hr[0], BF16, what=f"general h_last, batch {b}, channels {ds}")
    del y, h, full
    torch.cuda.empty_cache()


def test_scan_bwd_offsets_beyond_2_32():
    # output gradients zero outside the sampled channels S: every other
    # channel's adjoint is exactly zero, so dB and dC are sums over S, which the
    # oracle computes on the channel slice (all batch elements, the whole sequence)
    Bt, L, Dm = 4, 1 << 18, 5120
    n = Bt * L * Dm
    _need(7 * n * 2 + 4 * n + (8 << 30))  # u, delta_raw, z, dy; du, ddelta_raw, dz; the saved states
    S = [0, 17, 2560, 4095, Dm - 1]
    x = gen.symbol_scan_inputs(Bt, L, Dm, seed=7)
    tdy, sdy = gen.symbol_tensor((Bt, L), (Dm,), 7, slot=3)
    mask = torch.zeros(Dm)
    mask[S] = 1.0
    tdy = (tdy.float() * mask).to(BF16)  # exact: zero outside S
    dh = torch.zeros(Bt, Dm, 16)
    dh[:, S] = gen.randn_blocks(Bt * len(S) * 16, 7, 98).view(Bt, len(S), 16)
    dev = torch.device("cuda", 0)
    full = _expand(x["tables"], x["symbols"], dev)
    dyf = gen.gather_symbols(tdy.to(dev), sdy.to(dev))
    g = ss.ss_scan_bwd(full["u"], full["delta_raw"], x["A"].to(dev), x["B"].to(dev), x["C"].to(dev), dyf,
                       x["D"].to(dev), full["z"], x["delta_bias"].to(dev), None, dh.to(dev))
    torch.cuda.synchronize()
    del full, dyf
    st = torch.as_tensor(S)
    xs = {k: gen.gather_symbols(x["tables"][k][:, st], x["symbols"][k]) for k in KEYS}
    xs.update(B=x["B"], C=x["C"], A=x["A"][st].contiguous(), D=x["D"][st].contiguous(),
              delta_bias=x["delta_bias"][st].contiguous(), h0=None)
    ref = oracle.scan_bwd(xs, gen.gather_symbols(tdy[:, st], sdy), dh[:, st].contiguous())
    idx = torch.tensor(S, device=dev)
    for k in ("du", "ddelta_raw", "dz"):
        assert_close(g[k][:, :, idx].double().cpu().numpy(), ref[k], BF16, out_bf16=True, what=f"bwd {k} on S")
        g[k][:, :, idx] = 0
        assert not bool(g[k].ne(0).any()), f"bwd {k}: nonzero outside S"
    for k in ("dB", "dC"):
        assert_close(g[k].double().cpu().numpy(), ref[k], BF16, what=f"bwd {k}")
    assert_close(g["dA"][idx].double().cpu().numpy(), ref["dA"], BF16, what="bwd dA on S")
    assert_close(g["dD"][idx].double().cpu().numpy(), ref["dD"], BF16, what="bwd dD on S")
    assert_close(g["ddelta_bias"][idx].double().cpu().numpy(), ref["ddelta_bias"], BF16, what="bwd ddelta_bias on S")
    assert_close(g["dh0"][:, idx].double().cpu().numpy(), ref["dh0"], BF16, what="bwd dh0 on S")
    del g
    torch.cuda.empty_cache()


def test_ssd_offsets_beyond_2_32():
    # 5 x 2^18 steps x 80 heads x 64: x and y hold 6.7e9 elements. The oracle
    # runs the first 2048 steps of sampled heads of the first and the last batch
    # element (the outputs of a prefix depend on the prefix alone)
    Bt, L, H, P, N, T = 5, 1 << 18, 80, 64, 128, 2048
    n = Bt * L * H * P
    _need(2 * n * 2 + (8 << 30))
    par = gen.random_ssd_inputs(1, 1, H, P, N, seed=8)  # per-head A, D, dt_bias
    tx, sx = gen.symbol_tensor((Bt, L), (H, P), 8, slot=0)
    tdt, sdt = gen.symbol_tensor((Bt, L), (H,), 8, slot=1, scale=0.5)
    tb, sb = gen.symbol_tensor((Bt, L), (1, N), 8, slot=2)
    tc, sc = gen.symbol_tensor((Bt, L), (1, N), 8, slot=3)
    dev = torch.device("cuda", 0)
    xf = gen.gather_symbols(tx.to(dev), sx.to(dev))
    dtf = gen.gather_symbols(tdt.to(dev), sdt.to(dev))
    Bf, Cf = gen.gather_symbols(tb.to(dev), sb.to(dev)), gen.gather_symbols(tc.to(dev), sc.to(dev))
    y, hl = ss.ss_ssd_fwd(xf, dtf, par["A"].to(dev), Bf, Cf, par["D"].to(dev), par["dt_bias"].to(dev), None)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(hl).all())
    assert not bool(torch.isnan(y).any())
    heads = [0, 41, H - 1]
    hs = torch.as_tensor(heads)
    for b in (0, Bt - 1):
        pre = {"x": gen.gather_symbols(tx[:, hs], sx[b:b + 1, :T]), "dt": gen.gather_symbols(tdt[:, hs], sdt[b:b + 1, :T]),
               "B": gen.gather_symbols(tb, sb[b:b + 1, :T]), "C": gen.gather_symbols(tc, sc[b:b + 1, :T]),
               "A": par["A"][hs].contiguous(), "D": par["D"][hs].contiguous(),
               "dt_bias": par["dt_bias"][hs].contiguous(), "h0": None}
        yr, _ = oracle.ssd(pre)
        yg = y[b, :T][:, torch.tensor(heads, device=dev)].double().cpu().numpy()  # [T, k, P]
        assert_close(yg, yr[0], BF16, out_bf16=True, what=f"ssd y, batch {b}, heads {heads}, first {T} steps")
    del y, hl, xf, dtf, Bf, Cf
    torch.cuda.empty_cache()


def test_decode_offsets_beyond_2_32():
    # 65536 streams x 5120 channels x 16 states: the state holds 5.37e9 fp32
    Sn, Dm = 65536, 5120
    n = Sn * Dm * 16
    _need(n * 4 + (8 << 30))
    w = gen.ScanWorkload("decode_large", 1, 1, Dm, 16, "bf16", 9, 1.0, 0.0)
    A, Dk, bias = gen.make_params(w)
    th, sh = gen.symbol_tensor((Sn,), (Dm, 16), 9, slot=0, dtype="f32", scale=0.5)
    tabs = {}
    syms = {}
    for i, k in enumerate(KEYS):
        tabs[k], syms[k] = gen.symbol_tensor((Sn,), (Dm,), 9, slot=1 + i)
    tb, sb = gen.symbol_tensor((Sn,), (16,), 9, slot=4)
    tc, sc = gen.symbol_tensor((Sn,), (16,), 9, slot=5)
    dev = torch.device("cuda", 0)
    h = gen.gather_symbols(th.to(dev), sh.to(dev))
    full = _expand(tabs, syms, dev)
    Bf, Cf = gen.gather_symbols(tb.to(dev), sb.to(dev)), gen.gather_symbols(tc.to(dev), sc.to(dev))
    y = ss.ss_state_update(h, full["u"], full["delta_raw"], A.to(dev), Bf, Cf, Dk.to(dev), full["z"], bias.to(dev))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(h).all()) and bool(torch.isfinite(y.float()).all())
    for s, ds in _sample(Sn, Dm, seed=91).items():
        dt_ = torch.as_tensor(ds)
        h_np = gen.gather_symbols(th[:, dt_], sh[s:s + 1]).double().numpy().copy()  # [1, k, 16]
        step = {k: gen.gather_symbols(tabs[k][:, dt_], syms[k][s:s + 1]) for k in KEYS}
        step.update(B=gen.gather_symbols(tb, sb[s:s + 1]), C=gen.gather_symbols(tc, sc[s:s + 1]),
                    A=A[dt_].contiguous(), D=Dk[dt_].contiguous(), delta_bias=bias[dt_].contiguous())
        yr = oracle.state_update(h_np, step)
        idx = torch.tensor(ds, device=dev)
        assert_close(y[s][idx].double().cpu().numpy()[None], yr, BF16, out_bf16=True, what=f"decode y, stream {s}")
        assert_close(h[s][idx].double().cpu().numpy()[None], h_np, BF16, what=f"decode state, stream {s}")
    del h, y, full, Bf, Cf
    torch.cuda.empty_cache()
