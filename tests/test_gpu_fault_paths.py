"""The scan's bounded device-side waits, made to run out on purpose.

Cross-CTA waits (the stream-K hand-over of a state, the look-back over chunk
carries) poll a flag that another CTA publishes, with a time limit. Here a flag
is withheld through the library's test knob (ss_scan_set_wait_limit): nothing
ever sets it, so the waiting CTAs give up after a short limit, record the
timeout in the fault word and return. The call must finish, ss_scan_status must
report SS_ERR_TIMEOUT once (and clear it), and the next clean call must be
correct. No trap, fault or unbounded wait is involved: every wait ends.
"""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close, to_dev
from selective_state_space_130_b300 import _lib
from workloads import gen

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000  # 2 ms


def _run(d, Bt, L, Dm, ws):
    y, h = ss.ss_scan_fwd(d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                          d["h0"], out_dtype=torch.float32, workspace=ws)
    return y, h


def _expect_timeout_then_clean(x, tuning, withhold):
    d = to_dev(x)
    Bt, L, Dm = d["u"].shape
    ss.ss_scan_set_tuning(*tuning)
    try:
        nb = ss.ss_scan_fwd_workspace_size(Bt, L, Dm)
        assert nb > 0, "the forced split must use the workspace"
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        ss.ss_scan_set_wait_limit(LIMIT_NS, withhold)
        try:
            _run(d, Bt, L, Dm, ws)
        finally:
            ss.ss_scan_set_wait_limit(0, -1)
        torch.cuda.synchronize()  # the call finished: every wait ended
        with pytest.raises(ss.SSError) as ei:
            ss.ss_scan_status(ws)
        assert ei.value.status == _lib.SS_ERR_TIMEOUT
        ss.ss_scan_status(ws)  # the fault record was cleared by the read
        # a clean call on the same workspace is correct again
        y, h = _run(d, Bt, L, Dm, ws)
        ss.ss_scan_status(ws)
        torch.cuda.synchronize()
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    yr, hr = oracle.scan(x)
    assert_close(y.double().cpu().numpy(), yr, torch.bfloat16, what="clean call after a timeout: y")
    assert_close(h.double().cpu().numpy(), hr, torch.bfloat16, what="clean call after a timeout: h_last")


@pytest.mark.parametrize("sg", [1, 2])
def test_lookback_wait_times_out(sg):
    # chunks of 64 steps; chunk 0 of block 0 never publishes its carry, so every
    # later chunk of that block waits for it and gives up
    x = gen.random_scan_inputs(1, 1000, 64, 16, in_dtype="bf16", seed=31, with_h0=True)
    _expect_timeout_then_clean(x, (sg, 64, 0), withhold=0)


def test_handover_wait_times_out():
    # 3 x 640 channels in blocks of 128 = 15 blocks of 2 tiles on 4 CTAs: the
    # range of CTA 1 starts inside a block, so it waits for the state CTA 0
    # hands over, which is withheld
    x = gen.random_scan_inputs(3, 100, 640, 16, in_dtype="bf16", seed=32, with_h0=True)
    _expect_timeout_then_clean(x, (1, 0, 4), withhold=1)


def test_wait_limit_does_not_change_results():
    # a clean call under a short limit (nothing is withheld) is unaffected
    x = gen.random_scan_inputs(1, 1000, 64, 16, in_dtype="bf16", seed=33)
    d = to_dev(x)
    ss.ss_scan_set_tuning(1, 64, 0)
    try:
        ws = torch.empty(ss.ss_scan_fwd_workspace_size(1, 1000, 64), dtype=torch.uint8, device="cuda")
        ss.ss_scan_set_wait_limit(200_000_000, -1)
        try:
            y, h = _run(d, 1, 1000, 64, ws)
        finally:
            ss.ss_scan_set_wait_limit(0, -1)
        ss.ss_scan_status(ws)
        torch.cuda.synchronize()
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    yr, hr = oracle.scan(x)
    assert_close(y.double().cpu().numpy(), yr, torch.bfloat16, what="y")
    assert np.isfinite(h.cpu().numpy()).all()
