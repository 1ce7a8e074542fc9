"""GPU parity of the state-space-dual (Mamba-2) layer (ss_ssd_fwd, tensor-core
chunked form) against the float64 oracle (the recurrence with a scalar decay
per head), through the C ABI: every output on small and ragged problems,
sampled head channels over the whole sequence at a Mamba-2 2.7B-shaped layer."""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close, to_dev
from workloads import gen

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def _run(x, out_dtype):
    d = to_dev(x)
    y, h = ss.ss_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d.get("D"), d.get("dt_bias"), d.get("h0"),
                         out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y.double().cpu().numpy(), h.double().cpu().numpy()


# (batch, L, heads, N, groups, h0)
SHAPES = [
    (1, 1, 1, 64, 1, False),      # one step
    (2, 65, 4, 64, 2, True),      # one step past a chunk
    (1, 64, 2, 128, 1, False),    # exactly one chunk
    (1, 130, 3, 128, 1, True),    # ragged third chunk
    (2, 200, 8, 128, 4, True),    # two heads per group
    (1, 1000, 2, 64, 2, True),    # 16 chunks of carried state
    (1, 128, 2, 128, 1, True),    # exactly one 128-step chunk of the d_state 128 kernel
    (1, 129, 2, 128, 2, False),   # one step past it
    (1, 1000, 2, 128, 2, True),   # eight chunks of carried state, ragged tail
    (3, 384, 6, 128, 3, True),    # three full chunks, two heads per group
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{s[0]}-L{s[1]}-H{s[2]}-N{s[3]}-G{s[4]}" for s in SHAPES])
def test_ssd_matches_oracle(shape):
    Bt, L, H, N, G, h0 = shape
    x = gen.random_ssd_inputs(Bt, L, H, 64, N, G, in_dtype="bf16", seed=L + H + N, with_h0=h0)
    yr, hr = oracle.ssd(x, G)
    for out in (F32, BF16):
        y, h = _run(x, out)
        assert_close(y, yr, BF16, out_bf16=(out == BF16), what=f"ssd y {shape}")
        assert_close(h, hr, BF16, what=f"ssd h_last {shape}")
    # the products carry about 16 significant bits: the float32 output also
    # meets the float32-input bound
    y, h = _run(x, F32)
    assert_close(y, yr, F32, what=f"ssd y {shape} (float32 bound)")
    assert_close(h, hr, F32, what=f"ssd h_last {shape} (float32 bound)")


def test_ssd_without_skip_and_bias():
    x = gen.random_ssd_inputs(1, 100, 2, 64, 64, 1, in_dtype="bf16", seed=3, with_h0=True)
    x["D"] = None
    x["dt_bias"] = None
    yr, hr = oracle.ssd(x, 1)
    y, h = _run(x, F32)
    assert_close(y, yr, BF16, what="ssd y (no D, no bias)")
    assert_close(h, hr, BF16, what="ssd h_last (no D, no bias)")


def test_ssd_layer_sampled():
    # Mamba-2 2.7B-shaped layer: batch 4, L 2048, 80 heads of 64 channels (d_inner 5120), d_state 128
    Bt, L, H, N = 4, 2048, 80, 128
    x = gen.random_ssd_inputs(Bt, L, H, 64, N, 1, in_dtype="bf16", seed=11)
    rng = np.random.default_rng(2)
    ch = np.stack([rng.integers(0, Bt, 24), rng.integers(0, H, 24), rng.integers(0, 64, 24)], axis=1)
    ch = np.concatenate([ch, [[0, 0, 0], [Bt - 1, H - 1, 63]]])
    yr, hr = oracle.ssd(x, 1, channels=ch)
    y, h = _run(x, BF16)
    assert_close(y[ch[:, 0], :, ch[:, 1], ch[:, 2]], yr, BF16, out_bf16=True, what="layer ssd y")
    assert_close(h[ch[:, 0], ch[:, 1], ch[:, 2]], hr, BF16, what="layer ssd h_last")


def test_ssd_chunk_continuity():
    # two calls chained through the state equal one call
    x = gen.random_ssd_inputs(2, 300, 4, 64, 128, 2, in_dtype="bf16", seed=5, with_h0=True)
    y, h = _run(x, F32)
    m = 100
    a = dict(x, x=x["x"][:, :m].contiguous(), dt=x["dt"][:, :m].contiguous(), B=x["B"][:, :m].contiguous(),
             C=x["C"][:, :m].contiguous())
    ya, ha = _run(a, F32)
    bb = dict(x, x=x["x"][:, m:].contiguous(), dt=x["dt"][:, m:].contiguous(), B=x["B"][:, m:].contiguous(),
              C=x["C"][:, m:].contiguous(), h0=torch.tensor(ha, dtype=torch.float32))
    yb, hb = _run(bb, F32)
    # the two runs cut the sequence into chunks at different steps; both are
    # held to the bound of their bf16 inputs
    assert_close(np.concatenate([ya, yb], axis=1), y, BF16, what="chained y")
    assert_close(hb, h, BF16, what="chained h_last")


def test_ssd_errors_and_empty():
    x = gen.random_ssd_inputs(1, 4, 2, 64, 64, 1, in_dtype="bf16", seed=1, with_h0=True)
    d = to_dev(x)
    lib = ss.lib()
    y = torch.empty(1, 4, 2, 64, dtype=torch.bfloat16, device="cuda")
    ptrs = [t.data_ptr() if t is not None else None for t in (d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                                                              d["dt_bias"], d["h0"])]
    for (P, N, G, dt_code, code) in [(32, 64, 1, ss.SS_BF16, ss._lib.SS_ERR_UNSUPPORTED),
                                     (64, 96, 1, ss.SS_BF16, ss._lib.SS_ERR_UNSUPPORTED),
                                     (64, 64, 3, ss.SS_BF16, ss._lib.SS_ERR_INVALID_ARG),
                                     (64, 64, 1, ss.SS_F32, ss._lib.SS_ERR_UNSUPPORTED)]:
        st = lib.ss_ssd_fwd(1, 4, 2, P, N, G, dt_code, ss.SS_BF16, *ptrs, y.data_ptr(), None, None, 0, None)
        assert st == code, (P, N, G, st, ss.ss_last_error())
    e = {k: d[k][:, :0].contiguous() for k in ("x", "dt", "B", "C")}
    hl = torch.full((1, 2, 64, 64), 3.0, device="cuda")
    ss.ss_ssd_fwd(e["x"], e["dt"], d["A"], e["B"], e["C"], d["D"], d["dt_bias"], d["h0"],
                  y=torch.empty(1, 0, 2, 64, dtype=torch.bfloat16, device="cuda"), h_last=hl)
    torch.cuda.synchronize()
    assert torch.equal(hl, d["h0"])


@pytest.mark.parametrize("dt_level,a_scale", [(4.0, 1.0), (-6.0, 0.01), (2.0, 8.0)],
                         ids=["strong-decay", "almost-no-decay", "decay-underflows"])
def test_ssd_decay_extremes(dt_level, a_scale):
    # delta ~ softplus(dt_level) with A scaled by a_scale: a decay so strong
    # that the state forgets within a few steps (the factors of the decay
    # between steps underflow to zero), and one so weak that a chunk carries
    # almost all of it; both must stay finite and within the bound
    x = gen.random_ssd_inputs(2, 300, 4, 64, 128, 2, in_dtype="bf16", seed=17, with_h0=True)
    x["dt_bias"] = torch.full_like(x["dt_bias"], dt_level)
    x["A"] = (x["A"] * a_scale).contiguous()
    yr, hr = oracle.ssd(x, 2)
    y, h = _run(x, F32)
    assert_close(y, yr, BF16, what=f"ssd y, dt level {dt_level}, A x {a_scale}")
    assert_close(h, hr, BF16, what=f"ssd h_last, dt level {dt_level}, A x {a_scale}")


# (batch, L, heads, groups, h0, share length in steps): the chunks of all
# sequences cut into contiguous shares, one per CTA, the state handed on
# through the workspace where a share starts inside a sequence. Shares of one
# chunk make chains of hand-overs; shares of 3 and 11 chunks (sequences of 8)
# cross sequence ends, so a CTA runs the next sequence's head before the
# tail it takes over; shares of 20 chunks hold two whole sequences each.
SPLITS = [(1, 1000, 2, 2, True, 128), (2, 1000, 3, 1, False, 256), (1, 1100, 4, 2, True, 384),
          (3, 700, 2, 1, True, 512), (2, 1000, 3, 1, True, 384), (2, 1000, 3, 3, False, 1408),
          (2, 1000, 3, 1, True, 2560)]


@pytest.mark.parametrize("case", SPLITS, ids=[f"b{c[0]}-L{c[1]}-H{c[2]}-G{c[3]}-share{c[5]}" for c in SPLITS])
def test_ssd_split_sequences(case):
    Bt, L, H, G, h0, share = case
    x = gen.random_ssd_inputs(Bt, L, H, 64, 128, G, in_dtype="bf16", seed=L + share, with_h0=h0)
    yr, hr = oracle.ssd(x, G)
    ss.ss_scan_set_tuning(0, share, 0)
    try:
        for out in (F32, BF16):
            y, h = _run(x, out)
            ss.ss_scan_status(None)
            assert_close(y, yr, BF16, out_bf16=(out == BF16), what=f"split ssd y {case}")
            assert_close(h, hr, BF16, what=f"split ssd h_last {case}")
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)


def test_ssd_more_sequences_than_sms():
    # 2 x 80 heads = 160 sequences of 3 chunks: the automatic plan gives every
    # SM an equal share of the 480 chunks, with hand-overs between CTAs; every
    # output checked
    x = gen.random_ssd_inputs(2, 300, 80, 64, 128, 4, in_dtype="bf16", seed=160, with_h0=True)
    yr, hr = oracle.ssd(x, 4)
    y, h = _run(x, BF16)
    ss.ss_scan_status(None)
    assert_close(y, yr, BF16, out_bf16=True, what="ssd y, 160 sequences")
    assert_close(h, hr, BF16, what="ssd h_last, 160 sequences")


def test_ssd_without_workspace():
    # no workspace: one CTA per (batch, head), the whole sequence in order
    x = gen.random_ssd_inputs(2, 1000, 3, 64, 128, 1, in_dtype="bf16", seed=9, with_h0=True)
    yr, hr = oracle.ssd(x, 1)
    d = to_dev(x)
    y, h = ss.ss_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], d["h0"],
                         out_dtype=F32, workspace=False)
    torch.cuda.synchronize()
    assert_close(y.double().cpu().numpy(), yr, BF16, what="ssd y without workspace")
    assert_close(h.double().cpu().numpy(), hr, BF16, what="ssd h_last without workspace")


def test_ssd_withheld_hand_over_times_out():
    # shares of two chunks: share 0 (sequence 0, chunks 0-1) never hands its
    # state on, so share 1 of that sequence gives up after the short limit
    # (and share 2 after it), the call finishes, the status reports the
    # timeout once, and a clean call is correct again
    x = gen.random_ssd_inputs(1, 1000, 2, 64, 128, 1, in_dtype="bf16", seed=41, with_h0=True)
    d = to_dev(x)
    ss.ss_scan_set_tuning(0, 256, 0)
    try:
        ss.ss_scan_set_wait_limit(2_000_000, 0)
        try:
            ss.ss_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["dt_bias"], d["h0"], out_dtype=F32)
        finally:
            ss.ss_scan_set_wait_limit(0, -1)
        torch.cuda.synchronize()
        with pytest.raises(ss.SSError) as ei:
            ss.ss_scan_status(None)
        assert ei.value.status == ss._lib.SS_ERR_TIMEOUT
        ss.ss_scan_status(None)
        y, h = _run(x, F32)
        ss.ss_scan_status(None)
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    yr, hr = oracle.ssd(x, 1)
    assert_close(y, yr, BF16, what="ssd y after a timed-out hand-over")
    assert_close(h, hr, BF16, what="ssd h_last after a timed-out hand-over")


def test_ssd_split_sequences_dstate64():
    # d_state 64 runs with B and C zero-padded to 128 columns; split into
    # shares of two chunks, with an initial state
    x = gen.random_ssd_inputs(2, 900, 3, 64, 64, 3, in_dtype="bf16", seed=64, with_h0=True)
    yr, hr = oracle.ssd(x, 3)
    ss.ss_scan_set_tuning(0, 256, 0)
    try:
        y, h = _run(x, F32)
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    ss.ss_scan_status(None)
    assert_close(y, yr, BF16, what="split ssd y, d_state 64")
    assert_close(h, hr, BF16, what="split ssd h_last, d_state 64")
    assert_close(y, yr, F32, what="split ssd y, d_state 64 (float32 bound)")
