"""GPU parity of ss_scan_fwd / ss_state_update against the float64 oracle, on
small and ragged problems (every output compared), through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close, run_scan, run_scan_dev, to_dev
from workloads import configs, gen

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def _dt(name):
    return F32 if name == "f32" else BF16


def test_config0_tiny_fp32_full():
    x = gen.make_scan_inputs(configs.TINY_FP32)
    x["h0"] = None
    yr, hr = oracle.scan(x)
    for sg in (1, 2):
        y, h = run_scan(x, F32, sg=sg)
        assert_close(y, yr, F32, what=f"c0 y sg={sg}")
        assert_close(h, hr, F32, what=f"c0 h_last sg={sg}")


# (in_dtype, batch, L, D, h0, z, D_skip, bias)
SHAPES = [
    ("f32", 1, 1, 16, False, True, True, True),
    ("bf16", 2, 1, 64, True, True, True, True),
    ("bf16", 1, 7, 100, False, True, True, True),    # D*2 not a multiple of 16: plain-load staging
    ("f32", 3, 33, 130, True, False, True, True),   # ragged channel block, no gate
    ("bf16", 2, 513, 72, True, True, False, True),  # no skip term
    ("f32", 1, 1000, 5, True, True, True, False),   # no bias
    ("bf16", 1, 64, 1, False, True, True, True),
    ("bf16", 2, 257, 520, True, True, True, True),
    ("f32", 2, 95, 64, True, True, True, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}-b{s[1]}-L{s[2]}-D{s[3]}" for s in SHAPES])
@pytest.mark.parametrize("sg", [1, 2])
def test_ragged_shapes(shape, sg):
    dt, Bt, L, Dm, h0, hz, hd, hb = shape
    x = gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype=dt, seed=1000 + L + Dm, with_h0=h0, has_z=hz, has_d=hd,
                               a_log_jitter=0.2)
    if not hb:
        x["delta_bias"] = None
    yr, hr = oracle.scan(x)
    y, h = run_scan(x, F32, sg=sg)
    assert_close(y, yr, _dt(dt), what="y")
    assert_close(h, hr, _dt(dt), what="h_last")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_bf16_output(dt):
    x = gen.random_scan_inputs(2, 300, 96, 16, in_dtype=dt, seed=7, with_h0=True)
    yr, hr = oracle.scan(x)
    y, h = run_scan(x, BF16)
    assert_close(y, yr, _dt(dt), out_bf16=True, what="bf16 y")
    assert_close(h, hr, _dt(dt), what="h_last")


# Chunked scan: cross-block carries by look-back plus head recompute.
CHUNKED = [
    # (in_dtype, batch, L, D, chunk, sg, dt_min, dt_max, h0)
    ("f32", 1, 1000, 64, 64, 2, 1e-3, 1e-1, True),      # slow decay: recompute spans whole chunks
    ("bf16", 2, 2000, 40, 128, 1, 1e-3, 1e-1, False),
    ("f32", 1, 1500, 32, 96, 1, 0.5, 2.0, True),         # fast decay: recompute stops early
    ("bf16", 1, 4099, 136, 256, 2, 0.05, 1.0, True),     # ragged tail chunk
    ("f32", 3, 700, 8, 32, 2, 1e-2, 0.5, False),         # one-tile chunks
]


@pytest.mark.parametrize("case", CHUNKED, ids=[f"{c[0]}-L{c[2]}-D{c[3]}-ch{c[4]}-sg{c[5]}" for c in CHUNKED])
def test_chunked_lookback(case):
    dt, Bt, L, Dm, chunk, sg, lo, hi, h0 = case
    x = gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype=dt, seed=L + chunk, with_h0=h0, dt_min=lo, dt_max=hi,
                               a_log_jitter=0.3)
    yr, hr = oracle.scan(x)
    y, h = run_scan(x, F32, sg=sg, chunk=chunk)
    assert_close(y, yr, _dt(dt), what="chunked y")
    assert_close(h, hr, _dt(dt), what="chunked h_last")


# Stream-K split: equal ranges of the (channel block, tile) space per CTA, with
# states handed over where a range boundary falls inside a channel block. It
# engages once there are more channel blocks (128 channels with one lane per
# channel, 64 with two) than CTA slots (one per SM, or the max_workers cap).
STREAMK = [
    # (in_dtype, batch, L, D, sg, max_workers, h0, z)
    ("bf16", 19, 100, 1000, 1, 0, True, True),     # 152 blocks of 2 tiles on one CTA per SM: most ranges hand over
    ("bf16", 19, 100, 1000, 2, 0, False, True),    # 304 blocks
    ("bf16", 19, 100, 1000, 2, 100, True, True),   # 304 blocks on 100 CTAs: three blocks per range
    ("f32", 19, 33, 1000, 1, 0, True, False),      # two tiles per block, the second ragged
    ("f32", 20, 1000, 960, 2, 0, False, True),     # 32 tiles per block, 300 blocks
    ("bf16", 3, 100, 640, 1, 4, True, True),       # 15 blocks on 4 CTAs
]


@pytest.mark.parametrize("case", STREAMK, ids=[f"{c[0]}-b{c[1]}-L{c[2]}-D{c[3]}-sg{c[4]}-w{c[5]}" for c in STREAMK])
def test_streamk_handover(case):
    dt, Bt, L, Dm, sg, workers, h0, hz = case
    x = gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype=dt, seed=3 * L + Dm + sg, with_h0=h0, has_z=hz,
                               a_log_jitter=0.2)
    ss.ss_scan_set_tuning(sg, 0, workers)
    try:
        assert ss.ss_scan_fwd_workspace_size(Bt, L, Dm) > 0  # the split mode needs its hand-over buffer
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    yr, hr = oracle.scan(x)
    y, h = run_scan(x, F32, sg=sg, workers=workers)
    assert_close(y, yr, _dt(dt), what="stream-K y")
    assert_close(h, hr, _dt(dt), what="stream-K h_last")


def test_streamk_matches_static():
    # the split changes no arithmetic: each state sees the same operations in
    # the same order, so the outputs are bit-identical to one CTA per block
    x = gen.random_scan_inputs(19, 100, 1000, 16, in_dtype="bf16", seed=12, with_h0=True)
    y1, h1 = run_scan(x, F32, sg=1, chunk=1 << 30)  # one chunk: one CTA per block, whole sequence
    y2, h2 = run_scan(x, F32, sg=1, workers=7)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)


@pytest.mark.parametrize("sg", [1, 2])
def test_chunked_many_chunks_long_sequence(sg):
    # eight chunks per channel block: look-back walks over predecessors whose
    # flags move from aggregate to inclusive while they are read (the whole
    # warp must take one decision per flag); sampled channels against the oracle
    L, Dm = 1 << 16, 1024
    x = gen.random_scan_inputs(1, L, Dm, 16, in_dtype="bf16", seed=21, dt_min=1e-3, dt_max=0.1)
    ss.ss_scan_set_tuning(sg, 0, 0)
    try:
        assert ss.ss_scan_fwd_workspace_size(1, L, Dm) > 0
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    y, h = run_scan_dev(x, F32, sg=sg)
    ch = np.array([[0, c] for c in (0, 1, 31, 32, 500, 511, 512, 1000, 1023)])
    yr, hr = oracle.scan(x, channels=ch)
    yg = y[0, :, ch[:, 1]].T.double().cpu().numpy()
    hg = h[0, ch[:, 1]].double().cpu().numpy()
    assert_close(yg, yr, BF16, what="many-chunk y")
    assert_close(hg, hr, BF16, what="many-chunk h_last")


def test_chunked_matches_unchunked():
    # chunking changes only the rounding (P = exp(A * sum delta) vs a product of
    # Abar, and the 2^-24 stop of the head recompute): within the fp32-input bound
    x = gen.random_scan_inputs(1, 3000, 48, 16, in_dtype="bf16", seed=5, with_h0=True)
    y1, h1 = run_scan(x, F32, sg=2)
    y2, h2 = run_scan(x, F32, sg=2, chunk=160)
    assert_close(y2, y1, F32, what="chunked vs unchunked y")
    assert_close(h2, h1, F32, what="chunked vs unchunked h_last")


def test_empty_and_zero_length():
    x = gen.random_scan_inputs(2, 4, 32, 16, in_dtype="f32", seed=3, with_h0=True)
    d = to_dev(x)
    h_last = torch.full((2, 32, 16), 7.0, device="cuda")
    y = torch.empty((2, 0, 32), device="cuda")
    ss.ss_scan_fwd(d["u"][:, :0].contiguous(), d["delta_raw"][:, :0].contiguous(), d["A"],
                   d["B"][:, :0].contiguous(), d["C"][:, :0].contiguous(), d["D"], d["z"][:, :0].contiguous(),
                   d["delta_bias"], d["h0"], y=y, h_last=h_last)
    torch.cuda.synchronize()
    assert torch.equal(h_last, d["h0"])  # L = 0: the state passes through unchanged
    ss.ss_scan_fwd(d["u"][:, :0].contiguous(), d["delta_raw"][:, :0].contiguous(), d["A"],
                   d["B"][:, :0].contiguous(), d["C"][:, :0].contiguous(), y=y, h_last=h_last)
    torch.cuda.synchronize()
    assert torch.count_nonzero(h_last).item() == 0


def test_workspace_too_small_is_rejected():
    x = to_dev(gen.random_scan_inputs(1, 1000, 64, 16, in_dtype="f32", seed=9))
    ss.ss_scan_set_tuning(2, 64)
    try:
        need = ss.ss_scan_fwd_workspace_size(1, 1000, 64)
        small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
        with pytest.raises(ss.SSError) as ei:
            ss.ss_scan_fwd(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], workspace=small)
        assert ei.value.status == ss._lib.SS_ERR_INVALID_ARG
    finally:
        ss.ss_scan_set_tuning(0, 0)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("out", [F32, BF16])
def test_state_update_matches_oracle(dt, out):
    Bt, Dm, steps = 5, 300, 12
    x = gen.random_scan_inputs(Bt, steps, Dm, 16, in_dtype=dt, seed=77, with_h0=True, a_log_jitter=0.2)
    h = x["h0"].cuda().clone()
    hr = x["h0"].double().numpy().copy()
    d = to_dev(x)
    for t in range(steps):
        step = {k: x[k][:, t].contiguous() for k in ("u", "delta_raw", "z", "B", "C")}
        step.update(A=x["A"], D=x["D"], delta_bias=x["delta_bias"])
        yr = oracle.state_update(hr, step)
        y = ss.ss_state_update(h, d["u"][:, t].contiguous(), d["delta_raw"][:, t].contiguous(), d["A"],
                               d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), d["D"],
                               d["z"][:, t].contiguous(), d["delta_bias"], out_dtype=out)
        assert_close(y.double().cpu().numpy(), yr, _dt(dt), out_bf16=(out == BF16), what=f"decode y step {t}")
    assert_close(h.double().cpu().numpy(), hr, _dt(dt), what="decode h")


def test_decode_steps_equal_scan_on_gpu():
    x = gen.random_scan_inputs(3, 40, 128, 16, in_dtype="bf16", seed=11, with_h0=True)
    ys, hs = run_scan(x, F32)
    d = to_dev(x)
    h = d["h0"].clone()
    for t in range(40):
        y = ss.ss_state_update(h, d["u"][:, t].contiguous(), d["delta_raw"][:, t].contiguous(), d["A"],
                               d["B"][:, t].contiguous(), d["C"][:, t].contiguous(), d["D"],
                               d["z"][:, t].contiguous(), d["delta_bias"], out_dtype=F32)
        yt = y.double().cpu().numpy()
        rms = np.sqrt(np.mean(ys[:, t] ** 2))
        assert np.max(np.abs(yt - ys[:, t])) <= 2e-5 * max(rms, 1e-30)
    hh = h.double().cpu().numpy()
    assert np.max(np.abs(hh - hs)) <= 2e-5 * np.sqrt(np.mean(hs ** 2))


def test_state_update_odd_sizes():
    # channel count not a multiple of the warp's 16 channels; single stream
    for Bt, Dm in [(1, 1), (3, 7), (1, 33)]:
        x = gen.random_scan_inputs(Bt, 1, Dm, 16, in_dtype="f32", seed=Dm, with_h0=True)
        hr = x["h0"].double().numpy().copy()
        step = {k: x[k][:, 0].contiguous() for k in ("u", "delta_raw", "z", "B", "C")}
        step.update(A=x["A"], D=x["D"], delta_bias=x["delta_bias"])
        yr = oracle.state_update(hr, step)
        d = to_dev(x)
        h = d["h0"].clone()
        y = ss.ss_state_update(h, d["u"][:, 0].contiguous(), d["delta_raw"][:, 0].contiguous(), d["A"],
                               d["B"][:, 0].contiguous(), d["C"][:, 0].contiguous(), d["D"],
                               d["z"][:, 0].contiguous(), d["delta_bias"])
        assert_close(y.double().cpu().numpy(), yr, F32, what=f"odd decode y {Bt}x{Dm}")
        assert_close(h.double().cpu().numpy(), hr, F32, what=f"odd decode h {Bt}x{Dm}")
