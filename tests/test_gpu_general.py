"""GPU parity of the generalised scan (ss_scan_fwd_general: d_state 16-128, B and
C in groups, first-order or zero-order-hold Bbar) against the float64 oracle,
through the C ABI: every output on small and ragged problems, sampled channels
over the whole sequence at the Mamba-2.8B layer size."""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close, sample_channels, to_dev
from workloads import configs, gen

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def _run(x, disc, out_dtype):
    d = to_dev(x)
    y, h = ss.ss_scan_fwd_general(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d.get("D"), d.get("z"),
                                  d.get("delta_bias"), d.get("h0"), disc=disc, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y.double().cpu().numpy(), h.double().cpu().numpy()


# (in_dtype, batch, L, D, N, G, h0, z, D_skip, bias)
SHAPES = [
    ("f32", 1, 1, 16, 16, 1, False, True, True, True),
    ("bf16", 2, 17, 40, 32, 1, True, True, True, True),      # ragged sub-tile and channel block
    ("f32", 2, 33, 24, 16, 3, True, False, True, True),      # groups of 8 channels: three per warp
    ("f32", 1, 45, 24, 32, 2, True, True, True, True),       # groups of 12: a warp straddles two
    ("bf16", 2, 33, 24, 64, 3, True, False, True, True),     # groups of 8 = one warp's channels
    ("bf16", 1, 100, 64, 128, 8, True, True, False, True),   # 4 channels per warp, 8 groups
    ("f32", 3, 64, 6, 16, 6, False, True, True, False),      # one B/C per channel
    ("bf16", 1, 40, 5, 64, 1, True, True, True, True),       # rows of 10 bytes: element-wise staging
    ("bf16", 2, 21, 6, 128, 2, True, True, True, True),      # rows of 8 bytes: 4-byte copies
    ("f32", 1, 513, 130, 32, 2, True, True, True, True),
    ("bf16", 1, 1000, 96, 64, 4, True, True, True, True),
    ("f32", 1, 20, 1000, 16, 1000, True, True, True, True),  # one B/C per channel, ragged last block at channel 992
    ("bf16", 2, 30, 200, 32, 40, True, True, True, True),    # groups of 5 channels, ragged last block
    # shapes the CTA-cooperative kernel takes (every CTA's channels in one group,
    # 16-byte rows): 64, 32 or 16 channels per CTA, sequences ending inside a tile
    ("bf16", 2, 100, 64, 32, 1, True, True, True, True),
    ("f32", 1, 77, 64, 64, 2, True, True, True, True),
    ("bf16", 3, 65, 48, 128, 3, False, True, False, True),
    ("bf16", 1, 300, 128, 64, 1, True, False, True, True),
    ("f32", 2, 40, 32, 128, 1, True, True, True, False),
]


def test_cta_shapes_take_the_cta_kernel():
    # the new shapes above are the ones whose CTAs (4 warps of 32 / (N / 16)
    # channels) each hold channels of one group
    for dt, Bt, L, Dm, N, G, *_ in SHAPES[-5:]:
        cc = 4 * (32 // (N // 16))
        assert (Dm // G) % cc == 0 and (Dm * (2 if dt == "bf16" else 4)) % 16 == 0


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}-b{s[1]}-L{s[2]}-D{s[3]}-N{s[4]}-G{s[5]}" for s in SHAPES])
@pytest.mark.parametrize("disc", ["first_order", "zoh"])
def test_general_matches_oracle(shape, disc):
    dt, Bt, L, Dm, N, G, h0, hz, hd, hb = shape
    in_dt = BF16 if dt == "bf16" else F32
    x = gen.random_general_inputs(Bt, L, Dm, N, G, in_dtype=dt, seed=L + Dm + N, with_h0=h0, has_z=hz,
                                  has_d=hd, a_log_jitter=0.3)
    if not hb:
        x["delta_bias"] = None
    yr, hr = oracle.scan_general(x, G, "zoh" if disc == "zoh" else "euler")
    for out in (F32, BF16):
        y, h = _run(x, disc, out)
        assert_close(y, yr, in_dt, out_bf16=(out == BF16), what=f"general y {shape} {disc}")
        assert_close(h, hr, in_dt, what=f"general h_last {shape} {disc}")


def test_general_first_order_matches_scan():
    # d_state 16, one group, first order: the specialised scan's problem
    x = gen.random_scan_inputs(2, 300, 200, 16, in_dtype="bf16", seed=7, with_h0=True)
    d = to_dev(x)
    y1, h1 = ss.ss_scan_fwd(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"], d["h0"],
                            out_dtype=F32)
    y2, h2 = ss.ss_scan_fwd_general(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                    d["h0"], out_dtype=F32)
    torch.cuda.synchronize()
    assert_close(y2.double().cpu().numpy(), y1.double().cpu().numpy(), F32, what="general vs scan y")
    assert_close(h2.double().cpu().numpy(), h1.double().cpu().numpy(), F32, what="general vs scan h")


@pytest.mark.parametrize("N,G,disc", [(64, 1, "zoh"), (128, 8, "first_order")])
def test_general_layer_sampled(N, G, disc):
    # Mamba-2.8B layer shape (4 x 2048 x 5120, bf16), larger state: sampled channels over the whole sequence
    w = configs.MAMBA2P8B_LAYER
    x = gen.random_general_inputs(w.batch, w.seqlen, w.dim, N, G, in_dtype="bf16", seed=N + G)
    ch = sample_channels(w.batch, w.dim, 24, seed=N)
    yr, hr = oracle.scan_general(x, G, "zoh" if disc == "zoh" else "euler", channels=ch)
    y, h = _run(x, disc, BF16)
    assert_close(y[ch[:, 0], :, ch[:, 1]], yr, BF16, out_bf16=True, what=f"layer N={N} G={G} y")
    assert_close(h[ch[:, 0], ch[:, 1]], hr, BF16, what=f"layer N={N} G={G} h_last")


def test_general_zoh_with_zero_a():
    # zero-order hold where some A_n are 0: Bbar = delta B there (the CTA
    # kernel's shape: 32 channels of one group per CTA)
    x = gen.random_general_inputs(2, 90, 64, 64, 1, in_dtype="bf16", seed=12, with_h0=True)
    A = x["A"].clone()
    A[:, ::5] = 0.0
    x["A"] = A.contiguous()
    yr, hr = oracle.scan_general(x, 1, "zoh")
    y, h = _run(x, "zoh", F32)
    assert_close(y, yr, BF16, what="general zoh y, some A = 0")
    assert_close(h, hr, BF16, what="general zoh h_last, some A = 0")


def test_general_errors_and_empty():
    x = gen.random_general_inputs(1, 4, 8, 32, 2, in_dtype="f32", seed=1, with_h0=True)
    d = to_dev(x)
    lib = ss.lib()
    args = lambda N, G, disc: [1, 4, 8, N, G, disc, ss.SS_F32, ss.SS_F32] + [  # noqa: E731
        t.data_ptr() if t is not None else None for t in (d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"],
                                                          d["z"], d["delta_bias"], d["h0"])]
    y = torch.empty(1, 4, 8, device="cuda")
    for N, G, disc, code in [(48, 2, 0, ss._lib.SS_ERR_UNSUPPORTED), (32, 3, 0, ss._lib.SS_ERR_INVALID_ARG),
                             (32, 2, 2, ss._lib.SS_ERR_UNSUPPORTED), (32, 0, 0, ss._lib.SS_ERR_INVALID_ARG)]:
        st = lib.ss_scan_fwd_general(*args(N, G, disc), y.data_ptr(), None, None, 0, None)
        assert st == code, (N, G, disc, st, ss.ss_last_error())
    # L = 0: h_last = h0
    e = {k: d[k][:, :0].contiguous() for k in ("u", "delta_raw", "z", "B", "C")}
    hl = torch.full((1, 8, 32), 5.0, device="cuda")
    ss.ss_scan_fwd_general(e["u"], e["delta_raw"], d["A"], e["B"], e["C"], d["D"], e["z"], d["delta_bias"], d["h0"],
                           y=torch.empty(1, 0, 8, device="cuda"), h_last=hl)
    torch.cuda.synchronize()
    assert torch.equal(hl, d["h0"])
    np.testing.assert_array_equal(hl.cpu().numpy(), x["h0"].numpy())


# (in_dtype, batch, L, D, N, G, disc, share length in steps): the CTA kernel's
# 32-step tiles of all channel blocks cut into contiguous shares, one per CTA,
# the state handed on through the workspace where a share starts inside a
# block's sequence. One-tile shares make chains of hand-overs; shares of 3 and
# 13 tiles start and end inside sequences and cross block ends, so a CTA runs
# the next block's head before the tail it takes over; 20-tile shares hold two
# whole blocks
GEN_SPLITS = [("f32", 2, 200, 64, 128, 2, "first_order", 32), ("bf16", 2, 300, 128, 64, 1, "zoh", 96),
              ("bf16", 3, 300, 128, 32, 2, "zoh", 416), ("bf16", 3, 300, 128, 32, 2, "first_order", 640),
              ("f32", 1, 333, 64, 64, 1, "zoh", 96)]


@pytest.mark.parametrize("case", GEN_SPLITS, ids=[f"{c[0]}-b{c[1]}-L{c[2]}-D{c[3]}-N{c[4]}-G{c[5]}-{c[6]}-share{c[7]}"
                                                  for c in GEN_SPLITS])
def test_general_split_shares(case):
    dt, Bt, L, Dm, N, G, disc, share = case
    x = gen.random_general_inputs(Bt, L, Dm, N, G, in_dtype=dt, seed=L + share, with_h0=True)
    yr, hr = oracle.scan_general(x, G, "zoh" if disc == "zoh" else "euler")
    in_dt = BF16 if dt == "bf16" else F32
    ss.ss_scan_set_tuning(0, share, 0)
    try:
        for out in (F32, BF16):
            y, h = _run(x, disc, out)
            ss.ss_scan_status(None)
            assert_close(y, yr, in_dt, out_bf16=(out == BF16), what=f"split general y {case}")
            assert_close(h, hr, in_dt, what=f"split general h_last {case}")
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)


# (batch, L, D, N, G, disc): more channel blocks than resident CTAs. 8 x 160
# blocks of 32 channels at d_state 64 (ZOH, three CTAs per SM); 2 x 320 blocks
# of 16 channels at d_state 128 with the first-order rule (raw bf16 rows, four
# CTAs per SM)
MANY_BLOCKS = [(8, 100, 5120, 64, 1, "zoh"), (2, 300, 5120, 128, 8, "first_order")]


@pytest.mark.parametrize("case", MANY_BLOCKS, ids=[f"b{c[0]}-L{c[1]}-N{c[3]}-G{c[4]}-{c[5]}" for c in MANY_BLOCKS])
def test_general_more_blocks_than_slots(case):
    # the automatic plan gives every slot an equal share of all blocks' tiles,
    # with hand-overs between CTAs; every output checked
    Bt, L, Dm, N, G, disc = case
    x = gen.random_general_inputs(Bt, L, Dm, N, G, in_dtype="bf16", seed=Bt * Dm // 32 + N, with_h0=True)
    yr, hr = oracle.scan_general(x, G, "zoh" if disc == "zoh" else "euler")
    y, h = _run(x, disc, BF16)
    ss.ss_scan_status(None)
    assert_close(y, yr, BF16, out_bf16=True, what=f"general y {case}")
    assert_close(h, hr, BF16, what=f"general h_last {case}")


def test_general_withheld_hand_over_times_out():
    # shares of two tiles: share 0 (block 0, tiles 0-1) never hands its state
    # on, so the shares after it in that block give up after the short limit,
    # the call finishes, the status reports the timeout once, and a clean call
    # is correct again
    x = gen.random_general_inputs(1, 300, 64, 64, 1, in_dtype="bf16", seed=43, with_h0=True)
    d = to_dev(x)
    ss.ss_scan_set_tuning(0, 64, 0)
    try:
        ss.ss_scan_set_wait_limit(2_000_000, 0)
        try:
            ss.ss_scan_fwd_general(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                   d["h0"], disc="zoh", out_dtype=F32)
        finally:
            ss.ss_scan_set_wait_limit(0, -1)
        torch.cuda.synchronize()
        with pytest.raises(ss.SSError) as ei:
            ss.ss_scan_status(None)
        assert ei.value.status == ss._lib.SS_ERR_TIMEOUT
        ss.ss_scan_status(None)
        y, h = _run(x, "zoh", F32)
        ss.ss_scan_status(None)
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    yr, hr = oracle.scan_general(x, 1, "zoh")
    assert_close(y, yr, BF16, what="general y after a timed-out hand-over")
    assert_close(h, hr, BF16, what="general h_last after a timed-out hand-over")
