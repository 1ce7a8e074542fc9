"""The scan entry point that allocates nothing (ss_scan_fwd_noalloc), called
through the C ABI and checked against ss_scan_fwd with a caller-provided
workspace.

Some callers cannot call cudaMalloc: a plugin given only its input and output
buffers by a host framework, or a serving loop that must not allocate (an
allocation can synchronise the device) once it runs. They use the variant whose
cross-block scratch is a fixed array inside the library. The comparison uses
the parity tolerance of the other GPU tests, on two calls in a row, so a
scratch left dirty by the first call would show up in the second. This file is
named so that pytest collects it last.
"""

import pytest
import torch

import selective_state_space_130_b300 as ss
from parity import REL, assert_close, to_dev
from selective_state_space_130_b300 import _lib
from workloads import gen

pytestmark = pytest.mark.gpu


def _args(d):
    return (d["u"], d["delta_raw"], d["A"], d["B"], d["C"], d.get("D"), d.get("z"), d.get("delta_bias"), d.get("h0"))


def _with_workspace(d, out_dtype):
    Bt, L, Dm = d["u"].shape
    nb = ss.ss_scan_fwd_workspace_size(Bt, L, Dm)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    y, h = ss.ss_scan_fwd(*_args(d), out_dtype=out_dtype, workspace=ws)
    ss.ss_scan_status(ws)
    return y, h


# (in_dtype, batch, L, dim, h0): the first two need cross-block scratch
# (the sequence is split into chunks), the last one does not
CASES = [("bf16", 2, 20000, 64, True), ("f32", 1, 17000, 40, False), ("bf16", 2, 300, 96, True)]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-b{c[1]}-L{c[2]}-D{c[3]}" for c in CASES])
def test_noalloc_matches_workspace_call(case):
    dt, Bt, L, Dm, h0 = case
    in_dt = torch.bfloat16 if dt == "bf16" else torch.float32
    if L > 10000:  # these shapes do use the scratch
        assert ss.ss_scan_fwd_workspace_size(Bt, L, Dm) > 0
    for call, seed in enumerate((101, 202)):  # two calls in a row on different inputs
        x = gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype=dt, seed=seed + L, with_h0=h0)
        d = to_dev(x)
        y_ref, h_ref = _with_workspace(d, torch.float32)
        y, h = ss.ss_scan_fwd_noalloc(*_args(d), out_dtype=torch.float32)
        ss.ss_scan_status(None)  # device-side waits of the no-allocation call report here
        torch.cuda.synchronize()
        assert_close(y.double().cpu().numpy(), y_ref.double().cpu().numpy(), in_dt, what=f"call {call} y")
        assert_close(h.double().cpu().numpy(), h_ref.double().cpu().numpy(), in_dt, what=f"call {call} h_last")


def test_noalloc_rejects_problems_beyond_its_scratch():
    # forcing 32-step chunks on a long sequence needs far more scratch than the
    # fixed array holds: the call must refuse before launching anything
    x = to_dev(gen.random_scan_inputs(1, 64, 32, 16, in_dtype="bf16", seed=7))
    L_big = 1 << 22
    ss.ss_scan_set_tuning(0, 32)
    try:
        need = ss.ss_scan_fwd_workspace_size(1, L_big, 1024)
        assert need > _lib.SS_SCAN_NOALLOC_SCRATCH_BYTES
        st = _lib.lib().ss_scan_fwd_noalloc(1, L_big, 1024, 16, _lib.SS_BF16, _lib.SS_BF16, x["u"].data_ptr(),
                                            x["delta_raw"].data_ptr(), x["A"].data_ptr(), x["B"].data_ptr(),
                                            x["C"].data_ptr(), None, None, None, None, x["u"].data_ptr(), None,
                                            torch.cuda.current_stream().cuda_stream)
    finally:
        ss.ss_scan_set_tuning(0, 0)
    assert st == _lib.SS_ERR_INVALID_ARG
    assert "scratch" in ss.ss_last_error()
    torch.cuda.synchronize()


def test_noalloc_allocates_nothing():
    # the entry point exists for callers that cannot allocate: after one
    # warm-up call (which resolves the scratch array's address and loads the
    # kernels), a call with preallocated outputs leaves the device's free
    # memory and torch's allocation count unchanged
    x = gen.random_scan_inputs(2, 20000, 64, 16, in_dtype="bf16", seed=5, with_h0=True)
    d = to_dev(x)
    assert ss.ss_scan_fwd_workspace_size(2, 20000, 64) > 0  # this shape does use the scratch
    y = torch.empty((2, 20000, 64), dtype=torch.float32, device="cuda")
    h = torch.empty((2, 64, 16), dtype=torch.float32, device="cuda")
    ss.ss_scan_fwd_noalloc(*_args(d), y=y, h_last=h)
    ss.ss_scan_status(None)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    n0 = torch.cuda.memory_stats()["allocation.all.allocated"]
    ss.ss_scan_fwd_noalloc(*_args(d), y=y, h_last=h)
    ss.ss_scan_status(None)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    n1 = torch.cuda.memory_stats()["allocation.all.allocated"]
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert n1 == n0, "torch allocated during the call"
    y_ref, h_ref = _with_workspace(d, torch.float32)
    assert_close(y.double().cpu().numpy(), y_ref.double().cpu().numpy(), torch.bfloat16, what="y")
