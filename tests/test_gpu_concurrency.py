"""Calls from several host threads at once, each on its own stream with its own
buffers and workspace, give the results of the same calls made one by one.
This covers the library's shared host state (the per-device plan inputs, the
fault word's address, the tensor-map encoder) and kernels whose CTAs wait on
one another (stream-K and look-back hand-overs, persistent shares with tickets)
running beside each other on the same SMs. Every such wait is on a CTA that has
already started, so the kernels make progress whatever else is resident.

The backward pass is left out: its cooperative launch needs all of its CTAs
resident at once, so it does not share the SMs with kernels on other streams
the way these do."""

import threading

import pytest
import torch

import selective_state_space_130_b300 as ss
from parity import to_dev
from workloads import gen

pytestmark = pytest.mark.gpu

BF16 = torch.bfloat16


def _scan(x):
    Bt, L, Dm = x["u"].shape
    ws = torch.empty(max(ss.ss_scan_fwd_workspace_size(Bt, L, Dm), 16), dtype=torch.uint8, device="cuda")
    y, h = ss.ss_scan_fwd(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], None,
                          workspace=ws)
    return [y, h], ws


def _general(x, N):
    Bt, L, Dm = x["u"].shape
    ws = torch.empty(max(ss.ss_scan_fwd_general_workspace_size(Bt, L, Dm, N, 1, "zoh"), 16), dtype=torch.uint8,
                     device="cuda")
    y, h = ss.ss_scan_fwd_general(x["u"], x["delta_raw"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                                  None, disc="zoh", workspace=ws)
    return [y, h], ws


def _ssd(x):
    y, h = ss.ss_ssd_fwd(x["x"], x["dt"], x["A"], x["B"], x["C"], x["D"], x["dt_bias"], None)
    return [y, h], None


def _conv(x):
    y, st = ss.ss_conv1d_fwd(x["x"], x["weight"], x["bias"], x["state"])
    return [y, st], None


def _decode(x, h0):
    h = h0.clone()
    y = ss.ss_state_update(h, x["u"], x["delta_raw"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    return [y, h], None


def _problems():
    """(name, call, exact): exact problems give bit-identical results however
    the CTAs interleave; the chunked scan's look-back may combine a carry from
    an aggregate or from an inclusive prefix, so its results agree to rounding."""
    out = []
    # stream-K scan: 160 channel blocks of the 2.8B layer width
    xs = to_dev(gen.random_scan_inputs(4, 1024, 5120, 16, in_dtype="bf16", seed=31))
    out.append(("scan stream-K", lambda: _scan(xs), True))
    # chunked scan: 8 channel blocks, a long sequence
    xc = to_dev(gen.random_scan_inputs(1, 65536, 1024, 16, in_dtype="bf16", seed=32))
    out.append(("scan chunked", lambda: _scan(xc), False))
    # generalised scan with persistent shares (640 units)
    xg = to_dev(gen.random_general_inputs(4, 1024, 5120, 64, 1, in_dtype="bf16", seed=33))
    out.append(("general", lambda: _general(xg, 64), True))
    # SSD with persistent shares (320 sequences)
    xd = to_dev(gen.random_ssd_inputs(4, 1024, 80, 64, 128, 1, in_dtype="bf16", seed=34))
    out.append(("ssd", lambda: _ssd(xd), True))
    xv = to_dev(gen.random_conv_inputs(4, 2048, 5120, 4, "bf16", seed=35, with_state=True))
    out.append(("conv1d", lambda: _conv(xv), True))
    w = gen.random_scan_inputs(256, 1, 5120, 16, in_dtype="bf16", seed=36)
    step = to_dev({k: (w[k][:, 0].contiguous() if k in ("u", "delta_raw", "z", "B", "C") else w[k])
                   for k in ("u", "delta_raw", "z", "B", "C", "A", "D", "delta_bias")})
    h0 = (0.5 * gen.randn_blocks(256 * 5120 * 16, 36, 97)).view(256, 5120, 16).cuda()
    out.append(("decode", lambda: _decode(step, h0), True))
    return out


def _same(name, got, ref, exact):
    for g, r in zip(got, ref):
        if exact:
            assert torch.equal(g, r), f"{name}: concurrent result differs from the serial one"
        else:
            gf, rf = g.float(), r.float()
            lim = 2.0 ** -7 * rf.abs() + 1e-6 * float(rf.pow(2).mean().sqrt())
            assert bool(((gf - rf).abs() <= lim).all()), f"{name}: concurrent result outside rounding"


def test_threads_on_separate_streams_match_serial_calls():
    probs = _problems()
    ref = []
    for name, call, _ in probs:
        outs, ws = call()
        torch.cuda.synchronize()
        if ws is not None:
            ss.ss_scan_status(ws)
        ref.append([t.clone() for t in outs])
    reps = 3
    results = [None] * len(probs)
    errors = []
    barrier = threading.Barrier(len(probs), timeout=60)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                barrier.wait()
                for _ in range(reps):
                    outs, ws = probs[i][1]()
                st.synchronize()
                if ws is not None:
                    ss.ss_scan_status(ws, stream=st)
                results[i] = outs
        except Exception as e:  # reported below, with the problem's name
            errors.append(f"{probs[i][0]}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,), daemon=True) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors
    for (name, _, exact), got, r in zip(probs, results, ref):
        _same(name, got, r, exact)
