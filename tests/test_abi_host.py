"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/ss_scan.h declares, and rejects bad arguments before
touching the device."""

import ctypes
import os
import re

import pytest
import torch

import selective_state_space_130_b300 as ss
from selective_state_space_130_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include"))) if f.endswith(".h")]


def declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(ss_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("ss_scan_fwd", "ss_state_update", "ss_scan_fwd_workspace_size", "ss_scan_status", "ss_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no binding signature"


def test_version():
    assert ss.ss_version() >= 10000


def _scan(**kw):
    args = dict(batch=1, seqlen=8, dim=8, dstate=16, in_dtype=0, out_dtype=0)
    args.update({k: v for k, v in kw.items() if k in args})
    ptrs = dict(u=0x1000, delta_raw=0x2000, A=0x3000, B=0x4000, C=0x5000, D=None, z=None, delta_bias=None,
                h0=None, y=0x6000, h_last=None, workspace=None)
    ptrs.update({k: v for k, v in kw.items() if k in ptrs})
    return ss.lib().ss_scan_fwd(args["batch"], args["seqlen"], args["dim"], args["dstate"], args["in_dtype"],
                                 args["out_dtype"], ptrs["u"], ptrs["delta_raw"], ptrs["A"], ptrs["B"], ptrs["C"],
                                 ptrs["D"], ptrs["z"], ptrs["delta_bias"], ptrs["h0"], ptrs["y"], ptrs["h_last"],
                                 ptrs["workspace"], kw.get("ws_bytes", 0), None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(dstate=8), _lib.SS_ERR_UNSUPPORTED, "dstate"),
    (dict(dstate=32), _lib.SS_ERR_UNSUPPORTED, "dstate"),
    (dict(in_dtype=5), _lib.SS_ERR_UNSUPPORTED, "dtype"),
    (dict(out_dtype=-1), _lib.SS_ERR_UNSUPPORTED, "dtype"),
    (dict(batch=-1), _lib.SS_ERR_INVALID_ARG, "negative"),
    (dict(seqlen=-3), _lib.SS_ERR_INVALID_ARG, "negative"),
    (dict(seqlen=1 << 31), _lib.SS_ERR_INVALID_ARG, "2^31"),
    (dict(u=None), _lib.SS_ERR_INVALID_ARG, "u must not be NULL"),
    (dict(delta_raw=None), _lib.SS_ERR_INVALID_ARG, "delta_raw"),
    (dict(A=None), _lib.SS_ERR_INVALID_ARG, "A must not"),
    (dict(B=None), _lib.SS_ERR_INVALID_ARG, "B must not"),
    (dict(C=None), _lib.SS_ERR_INVALID_ARG, "C must not"),
    (dict(y=None), _lib.SS_ERR_INVALID_ARG, "y must not"),
    (dict(u=0x1002), _lib.SS_ERR_INVALID_ARG, "aligned"),
    (dict(B=0x4008), _lib.SS_ERR_INVALID_ARG, "aligned"),
    (dict(h0=0x7004), _lib.SS_ERR_INVALID_ARG, "aligned"),
    (dict(z=0x7001), _lib.SS_ERR_INVALID_ARG, "aligned"),
])
def test_scan_rejects_bad_arguments(kw, code, msg):
    st = _scan(**kw)
    assert st == code
    assert msg in ss.ss_last_error()


def test_empty_problem_is_ok_without_device():
    assert _scan(batch=0) == _lib.SS_OK
    assert _scan(dim=0) == _lib.SS_OK
    assert ss.ss_last_error() == ""


def test_state_update_rejects_bad_arguments():
    L = ss.lib()
    ok = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, None, None, None, 0x7000]
    st = L.ss_state_update(4, 8, 15, 0, 0, *ok, None)
    assert st == _lib.SS_ERR_UNSUPPORTED and "dstate" in ss.ss_last_error()
    bad = list(ok)
    bad[0] = None  # h
    assert L.ss_state_update(4, 8, 16, 0, 0, *bad, None) == _lib.SS_ERR_INVALID_ARG
    bad = list(ok)
    bad[3] = 0x3004  # A misaligned
    assert L.ss_state_update(4, 8, 16, 1, 0, *bad, None) == _lib.SS_ERR_INVALID_ARG
    assert L.ss_state_update(0, 8, 16, 1, 0, *ok, None) == _lib.SS_OK


def test_workspace_size_queries():
    assert ss.ss_scan_fwd_workspace_size(1, 512, 256) == 0             # few blocks, short: one warp per block
    assert ss.ss_scan_fwd_workspace_size(4, 2048, 5120) > 0            # equal-range split hands states over
    ws = ss.ss_scan_fwd_workspace_size(1, 1 << 20, 1024)
    assert ws > 0                                                     # long sequences are split into chunks
    assert ss.ss_scan_fwd_workspace_size(1, 1 << 20, 1024, 8) == 0     # unsupported dstate
    ss.ss_scan_set_tuning(2, 64)
    try:
        forced = ss.ss_scan_fwd_workspace_size(1, 1000, 64)
    finally:
        ss.ss_scan_set_tuning(0, 0)
    assert forced > 0
    assert ss.ss_scan_fwd_workspace_size(1, 1000, 64) == 0


def test_binding_raises_typed_errors():
    with pytest.raises(ss.SSError) as ei:
        ss._lib._check(_scan(dstate=4))
    assert ei.value.status == _lib.SS_ERR_UNSUPPORTED


# ---------------------------------------------------------------- backward, generalised scan, SSD layer
def _bwd(**kw):
    a = dict(batch=1, seqlen=8, dim=8, dstate=16, in_dtype=0, dy_dtype=0)
    a.update({k: v for k, v in kw.items() if k in a})
    p = dict(u=0x1000, delta_raw=0x2000, A=0x3000, B=0x4000, C=0x5000, D=None, z=None, delta_bias=None, h0=None,
             dy=0x6000, dh_last=None, du=0x7000, ddelta_raw=0x8000, dz=None, dA=0x9000, dB=0xa000, dC=0xb000,
             dD=None, ddelta_bias=None, dh0=None, workspace=0xc000)
    p.update({k: v for k, v in kw.items() if k in p})
    order = ("u", "delta_raw", "A", "B", "C", "D", "z", "delta_bias", "h0", "dy", "dh_last", "du", "ddelta_raw",
             "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0", "workspace")
    return ss.lib().ss_scan_bwd(a["batch"], a["seqlen"], a["dim"], a["dstate"], a["in_dtype"], a["dy_dtype"],
                                *[p[k] for k in order], kw.get("ws_bytes", 1 << 20), None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(dstate=32), _lib.SS_ERR_UNSUPPORTED, "dstate"),
    (dict(dy_dtype=3), _lib.SS_ERR_UNSUPPORTED, "dtype"),
    (dict(seqlen=-1), _lib.SS_ERR_INVALID_ARG, "negative"),
    (dict(dy=None), _lib.SS_ERR_INVALID_ARG, "dy must not"),
    (dict(dB=None), _lib.SS_ERR_INVALID_ARG, "dB must not"),
    (dict(dA=None), _lib.SS_ERR_INVALID_ARG, "dA must not"),
    (dict(z=0xd000), _lib.SS_ERR_INVALID_ARG, "dz must not"),
    (dict(dh0=0xe008), _lib.SS_ERR_INVALID_ARG, "aligned"),
    (dict(ws_bytes=16), _lib.SS_ERR_INVALID_ARG, "workspace"),
    (dict(workspace=None), _lib.SS_ERR_INVALID_ARG, "workspace"),
])
def test_scan_bwd_rejects_bad_arguments(kw, code, msg):
    assert _bwd(**kw) == code
    assert msg in ss.ss_last_error()


def test_scan_bwd_workspace_and_empty():
    assert _bwd(batch=0) == _lib.SS_OK
    # the saved states, 2 KB per 32 channels per 16 steps (either lane layout),
    # padded to 256 bytes; then the hand-over area of a split over warps: two
    # flags per block of 16 channels (two lanes per channel, the larger case),
    # each array padded to 256 bytes, and two 2 KB slots per block
    def size(batch, seqlen, dim):
        blocks = batch * dim // 16
        ckpt = batch * dim // 32 * ((seqlen + 15) // 16) * 2048
        return (ckpt + 255) // 256 * 256 + 2 * ((blocks * 4 + 255) // 256 * 256) + 2 * blocks * 2048
    assert ss.ss_scan_bwd_workspace_size(1, 16, 32) == size(1, 16, 32) == 2048 + 512 + 8192
    assert ss.ss_scan_bwd_workspace_size(4, 2048, 5120) == size(4, 2048, 5120)
    assert size(4, 2048, 5120) == 4 * 160 * 128 * 2048 + 2 * 5120 + 2 * 1280 * 2048
    assert ss.ss_scan_bwd_workspace_size(1, 16, 32, 8) == 0


def _gen(**kw):
    a = dict(batch=1, seqlen=8, dim=8, dstate=32, ngroups=2, disc=0, in_dtype=0, out_dtype=0)
    a.update({k: v for k, v in kw.items() if k in a})
    p = [kw.get(k, v) for k, v in (("u", 0x1000), ("delta_raw", 0x2000), ("A", 0x3000), ("B", 0x4000),
                                   ("C", 0x5000), ("D", None), ("z", None), ("delta_bias", None), ("h0", None),
                                   ("y", 0x6000), ("h_last", None), ("workspace", None))]
    return ss.lib().ss_scan_fwd_general(a["batch"], a["seqlen"], a["dim"], a["dstate"], a["ngroups"], a["disc"],
                                        a["in_dtype"], a["out_dtype"], *p, kw.get("workspace_bytes", 0), None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(dstate=48), _lib.SS_ERR_UNSUPPORTED, "dstate"),
    (dict(dstate=256), _lib.SS_ERR_UNSUPPORTED, "dstate"),
    (dict(disc=2), _lib.SS_ERR_UNSUPPORTED, "discretisation"),
    (dict(ngroups=3), _lib.SS_ERR_INVALID_ARG, "multiple of ngroups"),
    (dict(ngroups=0), _lib.SS_ERR_INVALID_ARG, "ngroups"),
    (dict(B=None), _lib.SS_ERR_INVALID_ARG, "B must not"),
    (dict(u=0x1004), _lib.SS_ERR_INVALID_ARG, "aligned"),
])
def test_scan_general_rejects_bad_arguments(kw, code, msg):
    assert _gen(**kw) == code
    assert msg in ss.ss_last_error()


def test_scan_general_workspace_size_and_checks():
    # the CTA kernel's split: a ticket counter (256 bytes), one flag per
    # channel block (padded to 256 bytes), one 2048-float state per block;
    # blocks are 32, 16 and 64 channels at d_state 64, 128 and 32
    ws = ss.ss_scan_fwd_general_workspace_size
    assert ws(4, 2048, 5120, 64, 1, "zoh") == 256 + 2560 + 640 * 2048 * 4
    assert ws(4, 2048, 5120, 128, 8) == 256 + 5120 + 1280 * 2048 * 4
    assert ws(2, 100, 256, 32, 2) == 256 + 256 + 8 * 2048 * 4
    assert ws(4, 2048, 5120, 16, 1) == 0       # the scan kernel's static split
    assert ws(4, 2048, 5120, 16, 4) == 0       # the one-warp kernel
    assert ws(1, 32, 256, 64, 1) == 0          # one tile: nothing to split
    assert ws(2, 100, 40, 64, 1) == 0          # 40 channels: not whole 32-channel blocks
    assert ws(2, 100, 256, 64, 1, in_dtype=torch.float32) == ws(2, 100, 256, 64, 1)
    need = ws(1, 300, 64, 64, 1, "first_order", torch.float32)
    kw = dict(seqlen=300, dim=64, dstate=64, ngroups=1)
    assert _gen(workspace=0x10000, workspace_bytes=need - 1, **kw) == _lib.SS_ERR_INVALID_ARG
    assert "workspace" in ss.ss_last_error()
    assert _gen(workspace=0x10008, workspace_bytes=need, **kw) == _lib.SS_ERR_INVALID_ARG
    assert "workspace" in ss.ss_last_error()


def _ssd(**kw):
    a = dict(batch=1, seqlen=8, nheads=4, headdim=64, dstate=128, ngroups=2, in_dtype=1, out_dtype=1)
    a.update({k: v for k, v in kw.items() if k in a})
    p = [kw.get(k, v) for k, v in (("x", 0x1000), ("dt", 0x2000), ("A", 0x3000), ("B", 0x4000), ("C", 0x5000),
                                   ("D", None), ("dt_bias", None), ("h0", None), ("y", 0x6000),
                                   ("h_last", None), ("workspace", None))]
    return ss.lib().ss_ssd_fwd(a["batch"], a["seqlen"], a["nheads"], a["headdim"], a["dstate"], a["ngroups"],
                               a["in_dtype"], a["out_dtype"], *p, kw.get("workspace_bytes", 0), None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(in_dtype=0), _lib.SS_ERR_UNSUPPORTED, "bf16"),
    (dict(headdim=128), _lib.SS_ERR_UNSUPPORTED, "headdim"),
    (dict(dstate=16), _lib.SS_ERR_UNSUPPORTED, "dstate"),
    (dict(ngroups=3), _lib.SS_ERR_INVALID_ARG, "multiple of ngroups"),
    (dict(x=None), _lib.SS_ERR_INVALID_ARG, "x must not"),
    (dict(dt=0x2002), _lib.SS_ERR_INVALID_ARG, "aligned"),
])
def test_ssd_rejects_bad_arguments(kw, code, msg):
    assert _ssd(**kw) == code
    assert msg in ss.ss_last_error()


def test_ssd_workspace_size_and_checks():
    # one ticket counter (256 bytes), one flag per (batch, head) padded to 256
    # bytes, one 64 x 128 fp32 state per (batch, head) (d_state 64 runs padded
    # to 128); nothing for a single chunk, which never splits
    assert ss.ss_ssd_fwd_workspace_size(4, 2048, 80, 128) == 256 + 1280 + 320 * 64 * 128 * 4
    assert ss.ss_ssd_fwd_workspace_size(1, 300, 3, 128) == 256 + 256 + 3 * 64 * 128 * 4
    assert ss.ss_ssd_fwd_workspace_size(4, 2048, 80, 64) == ss.ss_ssd_fwd_workspace_size(4, 2048, 80, 128)
    assert ss.ss_ssd_fwd_workspace_size(4, 2048, 80, 32) == 0
    assert ss.ss_ssd_fwd_workspace_size(2, 128, 8, 128) == 0
    assert ss.ss_ssd_fwd_workspace_size(-1, 128, 8, 128) == 0
    need = ss.ss_ssd_fwd_workspace_size(1, 300, 4, 128)
    assert _ssd(seqlen=300, workspace=0x10000, workspace_bytes=need - 1) == _lib.SS_ERR_INVALID_ARG
    assert "workspace" in ss.ss_last_error()
    assert _ssd(seqlen=300, workspace=0x10008, workspace_bytes=need) == _lib.SS_ERR_INVALID_ARG
    assert "workspace" in ss.ss_last_error()


def _conv(**kw):
    a = dict(batch=2, seqlen=16, dim=64, width=4, in_dtype=1, out_dtype=1)
    a.update({k: v for k, v in kw.items() if k in a})
    p = [kw.get(k, v) for k, v in (("x", 0x10000), ("weight", 0x1000), ("bias", None), ("state_in", None))]
    q = [kw.get(k, v) for k, v in (("y", 0x40000), ("state_out", None))]
    return ss.lib().ss_conv1d_fwd(a["batch"], a["seqlen"], a["dim"], a["width"], a["in_dtype"], a["out_dtype"],
                                  *p, 1, *q, None)


# x spans 2 * 16 * 64 * 2 = 4096 bytes from 0x10000 in bf16
@pytest.mark.parametrize("kw,code,msg", [
    (dict(width=5), _lib.SS_ERR_UNSUPPORTED, "width"),
    (dict(weight=None), _lib.SS_ERR_INVALID_ARG, "weight"),
    (dict(y=0x10008), _lib.SS_ERR_INVALID_ARG, "aligned"),
    (dict(y=0x10000), _lib.SS_ERR_INVALID_ARG, "overlap"),
    (dict(y=0x10ff0), _lib.SS_ERR_INVALID_ARG, "overlap"),
    (dict(y=0x10000 - 4096 + 16), _lib.SS_ERR_INVALID_ARG, "overlap"),
    (dict(y=0x10000 - 2 * 4096 + 16, out_dtype=0), _lib.SS_ERR_INVALID_ARG, "overlap"),
    (dict(state_in=0x8000, state_out=0x8000), _lib.SS_ERR_INVALID_ARG, "state_out"),
])
def test_conv1d_rejects_bad_arguments(kw, code, msg):
    assert _conv(**kw) == code
    assert msg in ss.ss_last_error()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the call would launch on made-up addresses")
def test_conv1d_adjacent_buffers_pass_the_overlap_check():
    # y ending where x starts, or starting where x ends, is no overlap: the
    # call gets past the argument checks to the device check, which fails here
    for y in (0x10000 - 4096, 0x10000 + 4096):
        _conv(y=y)
        assert "overlap" not in ss.ss_last_error()


def test_new_entry_points_empty_problems_without_device():
    assert _gen(batch=0) == _lib.SS_OK
    assert _ssd(nheads=0) == _lib.SS_OK


# ---------------------------------------------------------------- the scan planner (no device: sizes only)
HDR = 64 * 4  # workspace header bytes


def _ws(batch, seqlen, dim, tuning=(0, 0, 0)):
    ss.ss_scan_set_tuning(*tuning)
    try:
        return ss.ss_scan_fwd_workspace_size(batch, seqlen, dim)
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)


def test_plan_follows_the_number_of_cta_slots():
    # one lane per channel: blocks of 128 channels. 2 x 1000 channels = 16
    # blocks. With at least 16 CTA slots every block gets its own CTA (no
    # workspace); with fewer, the equal-range split hands states over between
    # CTAs through a workspace of one flag and one 128 x 16 fp32 state per CTA.
    assert _ws(2, 100, 1000, (1, 0, 16)) == 0
    assert _ws(2, 100, 1000, (1, 0, 148)) == 0
    for w in (1, 4, 15):
        flags = (w * 4 + 255) // 256 * 256
        assert _ws(2, 100, 1000, (1, 0, w)) == HDR + flags + w * 128 * 16 * 4
    # two lanes per channel: blocks of 64 channels, 32 blocks
    assert _ws(2, 100, 1000, (2, 0, 32)) == 0
    assert _ws(2, 100, 1000, (2, 0, 31)) == HDR + 256 + 31 * 64 * 16 * 4


def test_plan_chunked_workspace():
    # forced chunks of 64 steps (bf16 tiles of 64): 1000 steps -> 16 chunks per
    # block; each (block, chunk) keeps a flag and a 48-float carry per channel
    need = _ws(1, 1000, 64, (1, 64, 0))
    items = 1 * 16
    assert need >= HDR + 256 + items * 128 * 48 * 4


# ---------------------------------------------------------------- the no-allocation scan: argument checks
def _noalloc(**kw):
    args = dict(batch=1, seqlen=8, dim=8, dstate=16, in_dtype=0, out_dtype=0)
    args.update({k: v for k, v in kw.items() if k in args})
    ptrs = dict(u=0x1000, delta_raw=0x2000, A=0x3000, B=0x4000, C=0x5000, D=None, z=None, delta_bias=None,
                h0=None, y=0x6000, h_last=None)
    ptrs.update({k: v for k, v in kw.items() if k in ptrs})
    return ss.lib().ss_scan_fwd_noalloc(args["batch"], args["seqlen"], args["dim"], args["dstate"], args["in_dtype"],
                                        args["out_dtype"], ptrs["u"], ptrs["delta_raw"], ptrs["A"], ptrs["B"],
                                        ptrs["C"], ptrs["D"], ptrs["z"], ptrs["delta_bias"], ptrs["h0"], ptrs["y"],
                                        ptrs["h_last"], None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(dstate=8), _lib.SS_ERR_UNSUPPORTED, "dstate"),
    (dict(in_dtype=7), _lib.SS_ERR_UNSUPPORTED, "dtype"),
    (dict(batch=-2), _lib.SS_ERR_INVALID_ARG, "negative"),
    (dict(dim=1 << 31), _lib.SS_ERR_INVALID_ARG, "2^31"),
    (dict(u=None), _lib.SS_ERR_INVALID_ARG, "u must not be NULL"),
    (dict(y=None), _lib.SS_ERR_INVALID_ARG, "y must not be NULL"),
    (dict(B=0x4004), _lib.SS_ERR_INVALID_ARG, "aligned"),
    (dict(h_last=0x8008), _lib.SS_ERR_INVALID_ARG, "aligned"),
])
def test_noalloc_rejects_bad_arguments_without_device(kw, code, msg):
    assert _noalloc(**kw) == code
    assert msg in ss.ss_last_error()


def test_noalloc_rejects_oversized_scratch_without_device():
    # chunks of one 64-step tile over 2^22 steps need far more scratch than the
    # fixed array: refused before any device call
    ss.ss_scan_set_tuning(0, 32, 0)
    try:
        st = _noalloc(batch=1, seqlen=1 << 22, dim=1024, in_dtype=1, out_dtype=1)
    finally:
        ss.ss_scan_set_tuning(0, 0, 0)
    assert st == _lib.SS_ERR_INVALID_ARG
    assert "scratch" in ss.ss_last_error()


def test_noalloc_empty_problem_is_ok_without_device():
    assert _noalloc(batch=0) == _lib.SS_OK
    assert _noalloc(dim=0) == _lib.SS_OK
