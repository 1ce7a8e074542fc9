"""The entry points inside a captured CUDA graph: each call is captured once
with its outputs and workspace allocated beforehand, the graph is replayed
twice, and the results equal those of the same call made eagerly. The
workspace clears are stream memsets and every other piece of a call's setup
(tensor maps, the launch shape, the cooperative launch of the backward) is
host-side, so the graph holds the whole call and a replay starts from a clean
workspace. Results that do not depend on the order in which CTAs meet are
bit-identical; two kinds agree to rounding: the chunked scan's output (its
look-back may take a carry from an aggregate or from an inclusive prefix) and
the backward's sums over channels and time (dA, dB, dC, dD, ddelta_bias, added
up by atomics in the order the CTAs reach them)."""

import pytest
import torch

import selective_state_space_130_b300 as ss
from parity import to_dev
from workloads import gen

pytestmark = pytest.mark.gpu


def _scan_case(Bt, L, Dm, seed):
    x = to_dev(gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype="bf16", seed=seed))
    y = torch.empty((Bt, L, Dm), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((Bt, Dm, 16), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(ss.ss_scan_fwd_workspace_size(Bt, L, Dm), 16), dtype=torch.uint8, device="cuda")

    def call():
        ss.ss_scan_fwd(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], None, y=y,
                       h_last=h, workspace=ws)
    return call, [y, h], [], ws


def _general_case():
    Bt, L, Dm, N = 4, 1024, 5120, 64
    x = to_dev(gen.random_general_inputs(Bt, L, Dm, N, 1, in_dtype="bf16", seed=41))
    y = torch.empty((Bt, L, Dm), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((Bt, Dm, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(ss.ss_scan_fwd_general_workspace_size(Bt, L, Dm, N, 1, "zoh"), 16), dtype=torch.uint8,
                     device="cuda")

    def call():
        ss.ss_scan_fwd_general(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], None,
                               disc="zoh", y=y, h_last=h, workspace=ws)
    return call, [y, h], [], ws


def _ssd_case():
    Bt, L, H, P, N = 4, 1024, 80, 64, 128
    x = to_dev(gen.random_ssd_inputs(Bt, L, H, P, N, 1, in_dtype="bf16", seed=42))
    y = torch.empty((Bt, L, H, P), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((Bt, H, P, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(ss.ss_ssd_fwd_workspace_size(Bt, L, H, N), 16), dtype=torch.uint8, device="cuda")

    def call():
        ss.ss_ssd_fwd(x["x"], x["dt"], x["A"], x["B"], x["C"], x["D"], x["dt_bias"], None, y=y, h_last=h,
                      workspace=ws)
    return call, [y, h], [], None


def _conv_case():
    x = to_dev(gen.random_conv_inputs(4, 2048, 5120, 4, "bf16", seed=43, with_state=True))
    y = torch.empty((4, 2048, 5120), dtype=torch.bfloat16, device="cuda")
    st = torch.empty((4, 5120, 3), dtype=torch.bfloat16, device="cuda")

    def call():
        ss.ss_conv1d_fwd(x["x"], x["weight"], x["bias"], x["state"], y=y, state_out=st)
    return call, [y, st], [], None


def _bwd_case():
    Bt, L, Dm = 4, 512, 5120  # 1280 channel blocks: the shares and the cooperative launch
    x = to_dev(gen.random_scan_inputs(Bt, L, Dm, 16, in_dtype="bf16", seed=44))
    dy, dh = gen.random_output_grads(Bt, L, Dm, 16, "bf16", seed=44)
    dy, dh = dy.cuda(), dh.cuda()
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bt, L, Dm), dtype=torch.uint8, device="cuda")
    out = ss.ss_scan_bwd(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], dy, x["D"], x["z"], x["delta_bias"], None,
                         dh, workspace=ws)
    torch.cuda.synchronize()

    def call():  # (the library clears the summed outputs itself, by memsets that the graph holds)
        ss.ss_scan_bwd(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], dy, x["D"], x["z"], x["delta_bias"], None, dh,
                       out=out, workspace=ws)
    per_channel = [out[k] for k in ("du", "ddelta_raw", "dz", "dh0")]
    sums = [out[k] for k in ("dA", "dB", "dC", "dD", "ddelta_bias")]
    return call, per_channel, sums, None


def _chunked_case():
    call, outs, _, ws = _scan_case(1, 65536, 1024, 46)
    return call, [], outs, ws


CASES = {
    "scan stream-K": lambda: _scan_case(4, 1024, 5120, 45),
    "scan chunked": _chunked_case,
    "general": _general_case,
    "ssd": _ssd_case,
    "conv1d": _conv_case,
    "backward": _bwd_case,
}


@pytest.mark.parametrize("name", list(CASES))
def test_graph_replay_matches_eager_call(name):
    call, exact, rounded, ws = CASES[name]()
    outs = exact + rounded
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        call()  # the eager call: the reference, and the library's one-time setup
    st.synchronize()
    if ws is not None:
        ss.ss_scan_status(ws, stream=st)
    ref = [t.clone() for t in outs]
    for t in outs:
        t.fill_(float("nan")) if t.is_floating_point() else t.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        call()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    if ws is not None:
        ss.ss_scan_status(ws)
    for i, (got, want) in enumerate(zip(outs, ref)):
        if i < len(exact):
            assert torch.equal(got, want), f"{name}: output {i} of the graph replay differs from the eager call"
        else:
            gf, wf = got.float(), want.float()
            lim = 2.0 ** -7 * wf.abs() + 1e-5 * float(wf.pow(2).mean().sqrt())
            assert bool(((gf - wf).abs() <= lim).all()), f"{name}: output {i} of the graph replay outside rounding"
