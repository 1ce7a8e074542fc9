"""GPU parity of the scan's backward pass (ss_scan_bwd) against the float64
oracle's reverse sweep of the adjoint state, through the C ABI: every gradient
compared on small and ragged problems; at the Mamba-2.8B layer size, the
per-channel gradients on sampled channels and the channel-summed dB, dC
exactly through a property that holds at any size (output gradients that
vanish outside a channel set make dB, dC sums over that set alone)."""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close, to_dev
from workloads import configs, gen

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16
PER_CHANNEL = ("du", "ddelta_raw", "dz")
SUMMED = ("dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


def _run_bwd(x, dy, dh_last, sg=0):
    d = to_dev(x)
    ss.ss_scan_set_tuning(sg, 0, 0)
    try:
        g = ss.ss_scan_bwd(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], dy.cuda(), d.get("D"), d.get("z"),
                           d.get("delta_bias"), d.get("h0"), dh_last.cuda() if dh_last is not None else None)
        torch.cuda.synchronize()
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    return g


def _np(t):
    return t.double().cpu().numpy()


def _compare(g, ref, in_dt, has_z, what):
    for k in PER_CHANNEL:
        if k == "dz" and not has_z:
            assert g["dz"] is None
            continue
        assert_close(_np(g[k]), ref[k], in_dt, out_bf16=(in_dt == BF16), what=f"{what} {k}")
    for k in SUMMED:
        assert_close(_np(g[k]), ref[k], in_dt, what=f"{what} {k}")


# (in_dtype, dy_dtype, batch, L, D, h0, z, D_skip, bias, dh_last)
SHAPES = [
    ("f32", "f32", 1, 1, 16, False, True, True, True, False),    # one step
    ("f32", "f32", 2, 17, 40, True, True, True, True, True),     # ragged sub-tile and channel block
    ("bf16", "bf16", 2, 33, 72, True, True, False, True, True),  # no skip term
    ("bf16", "f32", 1, 100, 5, False, False, True, False, True),  # no gate, no bias, 5 channels
    ("f32", "bf16", 3, 64, 130, True, True, True, True, False),  # whole sub-tiles
    ("bf16", "bf16", 1, 513, 33, True, True, True, True, True),
    ("f32", "f32", 1, 1000, 64, True, True, True, True, True),   # long chain of saved states
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}-dy{s[1]}-b{s[2]}-L{s[3]}-D{s[4]}" for s in SHAPES])
@pytest.mark.parametrize("sg", [1, 2])
def test_scan_bwd_matches_oracle(shape, sg):
    dt, dyt, Bt, L, Dm, h0, hz, hd, hb, hdh = shape
    in_dt = BF16 if dt == "bf16" else F32
    x = gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype=dt, seed=L + Dm, with_h0=h0, has_z=hz, has_d=hd,
                               a_log_jitter=0.3)
    if not hb:
        x["delta_bias"] = None
    dy, dh = gen.random_output_grads(Bt, L, Dm, 16, dyt, seed=L * 3 + Dm, with_dh_last=hdh)
    ref = oracle.scan_bwd(x, dy, dh)
    g = _run_bwd(x, dy, dh, sg)
    _compare(g, ref, in_dt, hz, f"bwd {shape} sg={sg}")


def test_scan_bwd_mid_size_every_output():
    # 2 x 512 x 1024 bf16: 64 channel blocks, 32 saved states per block, every gradient compared
    x = gen.random_scan_inputs(2, 512, 1024, 16, in_dtype="bf16", seed=21, with_h0=True, a_log_jitter=0.3)
    dy, dh = gen.random_output_grads(2, 512, 1024, 16, "bf16", seed=22)
    ref = oracle.scan_bwd(x, dy, dh)
    for sg in (1, 2):
        g = _run_bwd(x, dy, dh, sg)
        _compare(g, ref, BF16, True, f"bwd mid sg={sg}")


def _slice_channels(x, S):
    idx = torch.as_tensor(S, dtype=torch.long)
    out = dict(x)
    for k in ("u", "delta_raw", "z"):
        if x.get(k) is not None:
            out[k] = x[k][:, :, idx].contiguous()
    out["A"] = x["A"][idx].contiguous()
    for k in ("D", "delta_bias"):
        if x.get(k) is not None:
            out[k] = x[k][idx].contiguous()
    if x.get("h0") is not None:
        out["h0"] = x["h0"][:, idx].contiguous()
    return out


@pytest.fixture(scope="module")
def layer():
    x = gen.make_scan_inputs(configs.MAMBA2P8B_LAYER)
    x["h0"] = None
    Bt, L, Dm = x["u"].shape
    S = sorted({0, 1, 31, 32, 63, 2047, 2048, 4000, Dm - 33, Dm - 2, Dm - 1})
    return x, S


@pytest.mark.parametrize("sg", [1, 2])
def test_scan_bwd_layer_sampled_channels(layer, sg):
    # Mamba-2.8B layer (4 x 2048 x 5120, bf16): dense output gradients; the
    # per-channel gradients of sampled channels depend on those channels alone
    x, S = layer
    Bt, L, Dm = x["u"].shape
    dy, dh = gen.random_output_grads(Bt, L, Dm, 16, "bf16", seed=5)
    g = _run_bwd(x, dy, dh, sg)
    idx = torch.as_tensor(S, dtype=torch.long)
    ref = oracle.scan_bwd(_slice_channels(x, S), dy[:, :, idx].contiguous(), dh[:, idx].contiguous())
    for k in PER_CHANNEL:
        assert_close(_np(g[k][:, :, idx.cuda()]), ref[k], BF16, out_bf16=True, what=f"layer {k}")
    assert_close(_np(g["dA"][idx.cuda()]), ref["dA"], BF16, what="layer dA")
    assert_close(_np(g["dD"][idx.cuda()]), ref["dD"], BF16, what="layer dD")
    assert_close(_np(g["ddelta_bias"][idx.cuda()]), ref["ddelta_bias"], BF16, what="layer ddelta_bias")
    assert_close(_np(g["dh0"][:, idx.cuda()]), ref["dh0"], BF16, what="layer dh0")


@pytest.mark.parametrize("sg", [1, 2])
def test_scan_bwd_layer_channel_sums(layer, sg):
    # output gradients zero outside S: every other channel's adjoint is exactly
    # zero, so dB and dC are the sums over S, which the oracle computes on the
    # channel slice; the kernel still runs over all 5120 channels
    x, S = layer
    Bt, L, Dm = x["u"].shape
    dy, dh = gen.random_output_grads(Bt, L, Dm, 16, "bf16", seed=6, channels=S)
    g = _run_bwd(x, dy, dh, sg)
    idx = torch.as_tensor(S, dtype=torch.long)
    ref = oracle.scan_bwd(_slice_channels(x, S), dy[:, :, idx].contiguous(), dh[:, idx].contiguous())
    assert_close(_np(g["dB"]), ref["dB"], BF16, what="layer dB")
    assert_close(_np(g["dC"]), ref["dC"], BF16, what="layer dC")
    assert_close(_np(g["du"][:, :, idx.cuda()]), ref["du"], BF16, out_bf16=True, what="layer du (sparse)")
    rest = torch.ones(Dm, dtype=torch.bool)
    rest[idx] = False
    rest = rest.cuda()
    for k in ("du", "ddelta_raw", "dz"):
        assert torch.count_nonzero(g[k][:, :, rest]) == 0, k
    assert torch.count_nonzero(g["dA"][rest]) == 0


def test_scan_bwd_per_channel_outputs_deterministic():
    x = gen.random_scan_inputs(2, 200, 96, 16, in_dtype="bf16", seed=4, with_h0=True)
    dy, dh = gen.random_output_grads(2, 200, 96, 16, "bf16", seed=4)
    for sg in (1, 2):
        g1 = _run_bwd(x, dy, dh, sg)
        g2 = _run_bwd(x, dy, dh, sg)
        for k in ("du", "ddelta_raw", "dz", "dh0"):
            assert torch.equal(g1[k], g2[k]), (k, sg)


def test_scan_bwd_sequence_split_chains():
    # gradients through two calls (the second's dh0 is the first's dh_last, the
    # first's h_last the second's h0) equal the one-call gradients
    Bt, L, Dm, m = 2, 150, 64, 70
    x = gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype="f32", seed=12, with_h0=True, a_log_jitter=0.3)
    dy, dh = gen.random_output_grads(Bt, L, Dm, 16, "f32", seed=13)
    g = _run_bwd(x, dy, dh)
    d = to_dev(x)
    first = {k: (v[:, :m].contiguous() if k in ("u", "delta_raw", "z", "B", "C") and v is not None else v)
             for k, v in x.items()}
    second = {k: (v[:, m:].contiguous() if k in ("u", "delta_raw", "z", "B", "C") and v is not None else v)
              for k, v in x.items()}
    df = to_dev(first)
    _, h_mid = ss.ss_scan_fwd(df["u"], df["delta_raw"], df["A"], df["B"], df["C"], df["D"], df["z"],
                              df["delta_bias"], df["h0"])
    second["h0"] = h_mid.cpu()
    g2 = _run_bwd(second, dy[:, m:].contiguous(), dh)
    g1 = _run_bwd(first, dy[:, :m].contiguous(), g2["dh0"].cpu())
    for k in ("du", "ddelta_raw", "dz", "dB", "dC"):
        whole = _np(g[k])
        assert_close(np.concatenate([_np(g1[k]), _np(g2[k])], axis=1), whole, F32, what=f"split {k}")
    for k in ("dA", "dD", "ddelta_bias"):
        assert_close(_np(g1[k]) + _np(g2[k]), _np(g[k]), F32, what=f"split {k}")
    assert_close(_np(g1["dh0"]), _np(g["dh0"]), F32, what="split dh0")
    del d


def test_scan_bwd_empty_and_errors():
    x = gen.random_scan_inputs(2, 3, 16, 16, in_dtype="f32", seed=1, with_h0=True)
    d = to_dev(x)
    dy, dh = gen.random_output_grads(2, 3, 16, 16, "f32", seed=1)
    dy, dh = dy.cuda(), dh.cuda()
    # L = 0: the state gradient passes through, the sums are zero
    e = {k: d[k][:, :0].contiguous() for k in ("u", "delta_raw", "z", "B", "C")}
    out = {"dA": torch.full((16, 16), 3.0, device="cuda"), "dh0": torch.full((2, 16, 16), 3.0, device="cuda")}
    g = ss.ss_scan_bwd(e["u"], e["delta_raw"], d["A"], e["B"], e["C"], dy[:, :0].contiguous(), d["D"], e["z"],
                       d["delta_bias"], d["h0"], dh, out=out)
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"], dh)
    assert torch.count_nonzero(g["dA"]) == 0
    # z given without dz
    args = [2, 3, 16, 16, ss.SS_F32, ss.SS_F32] + [t.data_ptr() if t is not None else None for t in (
        d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], d["h0"], dy, dh)]
    outs = {k: torch.empty(sh, device="cuda") for k, sh in [("du", (2, 3, 16)), ("ddelta_raw", (2, 3, 16)),
                                                               ("dA", (16, 16)), ("dB", (2, 3, 16)),
                                                               ("dC", (2, 3, 16))]}
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(2, 3, 16), dtype=torch.uint8, device="cuda")
    L = ss.lib()
    st = L.ss_scan_bwd(*args, outs["du"].data_ptr(), outs["ddelta_raw"].data_ptr(), None, outs["dA"].data_ptr(),
                       outs["dB"].data_ptr(), outs["dC"].data_ptr(), None, None, None, ws.data_ptr(), ws.numel(),
                       None)
    assert st == ss._lib.SS_ERR_INVALID_ARG and "dz" in ss.ss_last_error()
    # workspace too small
    dz = torch.empty(2, 3, 16, device="cuda")
    st = L.ss_scan_bwd(*args, outs["du"].data_ptr(), outs["ddelta_raw"].data_ptr(), dz.data_ptr(),
                       outs["dA"].data_ptr(), outs["dB"].data_ptr(), outs["dC"].data_ptr(), None, None, None,
                       ws.data_ptr(), 64, None)
    assert st == ss._lib.SS_ERR_INVALID_ARG and "workspace" in ss.ss_last_error()
    # dstate other than 16
    args_n8 = list(args)
    args_n8[3] = 8
    st = L.ss_scan_bwd(*args_n8, outs["du"].data_ptr(), outs["ddelta_raw"].data_ptr(), dz.data_ptr(),
                       outs["dA"].data_ptr(), outs["dB"].data_ptr(), outs["dC"].data_ptr(), None, None, None,
                       ws.data_ptr(), ws.numel(), None)
    assert st == ss._lib.SS_ERR_UNSUPPORTED


def _run_bwd_shares(x, dy, dh_last, sg, share):
    ss.ss_scan_set_tuning(sg, share, 0)
    try:
        return _run_bwd_tuned(x, dy, dh_last)
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)


def _run_bwd_tuned(x, dy, dh_last):
    d = to_dev(x)
    g = ss.ss_scan_bwd(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], dy.cuda(), d.get("D"), d.get("z"),
                       d.get("delta_bias"), d.get("h0"), dh_last.cuda() if dh_last is not None else None)
    torch.cuda.synchronize()
    return g


# (in_dtype, batch, L, D, sg, share length in steps): the blocks' 16-step
# sub-tiles cut into contiguous shares, one per warp. Where a share starts
# inside a block, the state comes from the share before and the adjoint goes
# back to it. One-sub-tile shares make chains of hand-overs both ways; shares
# of 3 and 7 sub-tiles cross block ends (a warp runs the next block's forward
# sweep first and its reverse sweep last); 400-step shares hold whole blocks
BWD_SPLITS = [("f32", 2, 300, 64, 2, 16), ("bf16", 2, 300, 64, 2, 48), ("f32", 3, 200, 96, 1, 112),
              ("bf16", 1, 1000, 64, 1, 400), ("bf16", 2, 333, 130, 2, 48)]


@pytest.mark.parametrize("case", BWD_SPLITS, ids=[f"{c[0]}-b{c[1]}-L{c[2]}-D{c[3]}-sg{c[4]}-share{c[5]}"
                                                  for c in BWD_SPLITS])
def test_scan_bwd_split_shares(case):
    dt, Bt, L, Dm, sg, share = case
    in_dt = BF16 if dt == "bf16" else F32
    x = gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype=dt, seed=L + share, with_h0=True, a_log_jitter=0.3)
    dy, dh = gen.random_output_grads(Bt, L, Dm, 16, dt, seed=L + Dm)
    ref = oracle.scan_bwd(x, dy, dh)
    g = _run_bwd_shares(x, dy, dh, sg, share)
    ss.ss_scan_status(None)
    _compare(g, ref, in_dt, True, f"bwd split {case}")


def test_scan_bwd_withheld_hand_over_times_out():
    # shares of two sub-tiles: share 0 (block 0, sub-tiles 0-1) hands nothing
    # on, so the share after it gives up waiting for its state (and share 0
    # for the adjoint it would have got back); the call finishes, the status
    # reports the timeout once, and a clean call is correct again
    x = gen.random_scan_inputs(1, 200, 32, 16, in_dtype="f32", seed=44, with_h0=True)
    dy, dh = gen.random_output_grads(1, 200, 32, 16, "f32", seed=45)
    ss.ss_scan_set_tuning(2, 32, 0)
    try:
        ss.ss_scan_set_wait_limit(2_000_000, 0)
        try:
            _run_bwd_tuned(x, dy, dh)
        finally:
            ss.ss_scan_set_wait_limit(0, -1)
        with pytest.raises(ss.SSError) as ei:
            ss.ss_scan_status(None)
        assert ei.value.status == ss._lib.SS_ERR_TIMEOUT
        ss.ss_scan_status(None)
        g = _run_bwd_tuned(x, dy, dh)
        ss.ss_scan_status(None)
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    _compare(g, oracle.scan_bwd(x, dy, dh), F32, True, "bwd after a timed-out hand-over")


def test_scan_bwd_shares_beyond_resident_warps_fall_back():
    # one-sub-tile shares of 64 blocks x 32 sub-tiles = 2048 shares, more than
    # the resident warps a cooperative launch allows: the call runs one warp
    # per block instead, with the same gradients
    x = gen.random_scan_inputs(1, 512, 1024, 16, in_dtype="bf16", seed=46, with_h0=True)
    dy, dh = gen.random_output_grads(1, 512, 1024, 16, "bf16", seed=47)
    ref = oracle.scan_bwd(x, dy, dh)
    g = _run_bwd_shares(x, dy, dh, 2, 16)
    ss.ss_scan_status(None)
    _compare(g, ref, BF16, True, "bwd, shares past the resident warps")
