"""Pins for the float64 CPU oracle: checks against results that the pages and
the mathematics fix independently of the oracle's own loop.

Each `pin_*` function runs the oracle (optionally a given build of it, so the
mutant test can run the same pins against deliberately broken copies) and
raises AssertionError when the oracle disagrees with the independent result.

Independent restatements used here (none calls the oracle's arithmetic):
- brute-force unrolled sum y_t = sum_{s<=t} C_t (prod_{s<k<=t} Abar_k) Bbar_s u_s
  + C_t (prod_{k<=t} Abar_k) h0 + D u_t, from the product form dh_t/dh_0 =
  prod Abar_k ("外文文献精读：Mamba - 线性时间序列建模与结构化状态空间模型",
  section 6.1) and the recurrence ("Transformer时代终结？Mamba的状态空间革命
  重塑AI底层架构", section 二.1);
- LTI case = causal 1-D convolution with kernel K_k = sum_n C_n Abar_n^k Bbar_n
  (same page, section 二.1 "卷积视角"; mlqm.cn tutorial section 3.3), checked
  by direct convolution and by FFT;
- small delta keeps the state, large delta overwrites it (mlqm.cn tutorial
  section 5.2; review page, method step 1);
- chunking with the carry pair (P, S), (P1,S1)o(P2,S2) = (P1 P2, P2 S1 + S2),
  equals the unsplit scan exactly up to rounding ("Transformer时代终结？"
  section 二.3 "无近似"; "外文文献精读" section 2.2 block combination);
- closed forms (geometric series), a hand-evaluated single step, exact zeros,
  linearity in u, channel/batch independence, decode x L = scan;
- generalised scan: scipy's zero-order-hold discretisation (cont2discrete) and
  simulation (dlsim) of the same linear system, the exact discretisation of
  h' = A h + B x for a step-wise constant input ("外文文献精读" section 1.2;
  mlqm.cn tutorial section 3.2); the brute-force sum on the first-order case at
  any state size; per-group channel slices;
- state-space-dual layer: the selective scan with a scalar decay per head is
  multiplication by the semiseparable matrix M[t, s] = (C_t . B_s) delta_s
  exp(sum_{s<k<=t} delta_k A) for s <= t ("AI 推理系列（十四）", section on
  Mamba-2 reorganising the SSM as matrix computation; mlqm.cn tutorial,
  section 8), built densely here.
"""

import math

import numpy as np
import torch
from scipy.special import expit

import oracle
from workloads.gen import random_general_inputs, random_scan_inputs, random_ssd_inputs


# ----------------------------------------------------------------- helpers

def _np(t):
    return None if t is None else t.double().numpy()


def _softplus_ref(x):
    # log(1 + e^x) via logaddexp: a different evaluation from the oracle's
    return np.logaddexp(0.0, x)


def brute_force(x):
    """O(L^2 N) unrolled sum with explicit products over Abar."""
    u, dr, z = _np(x["u"]), _np(x["delta_raw"]), _np(x.get("z"))
    B, C, A = _np(x["B"]), _np(x["C"]), _np(x["A"])
    Dk, bias, h0 = _np(x.get("D")), _np(x.get("delta_bias")), _np(x.get("h0"))
    Bt, L, Dm = u.shape
    N = B.shape[-1]
    y = np.zeros((Bt, L, Dm))
    hl = np.zeros((Bt, Dm, N))
    for b in range(Bt):
        for d in range(Dm):
            delta = _softplus_ref(dr[b, :, d] + (bias[d] if bias is not None else 0.0))  # [L]
            abar = np.exp(delta[:, None] * A[d][None, :])                              # [L, N]
            bx = delta[:, None] * B[b] * u[b, :, d][:, None]                            # [L, N]
            for t in range(L + 1):
                # state after step t-1 (t == L gives h_last)
                tt = t if t < L else L - 1
                h = np.zeros(N)
                if h0 is not None:
                    h += np.prod(abar[: tt + 1], axis=0) * h0[b, d]
                for s in range(tt + 1):
                    h += np.prod(abar[s + 1: tt + 1], axis=0) * bx[s]
                if t == L:
                    hl[b, d] = h
                    break
                yt = float(np.dot(C[b, t], h))
                if Dk is not None:
                    yt += Dk[d] * u[b, t, d]
                if z is not None:
                    yt *= z[b, t, d] * expit(z[b, t, d])
                y[b, t, d] = yt
    return y, hl


def _close(a, b, rtol, atol=0.0, what=""):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    bad = err > lim
    assert not bad.any(), f"{what}: max err {err.max():.3e} (worst rel {(err / np.maximum(np.abs(b), 1e-300)).max():.3e})"


def _f32(a):
    return torch.tensor(np.ascontiguousarray(a, dtype=np.float32))


# -------------------------------------------------------------------- pins

def pin_brute_force(lib=None):
    for seed, dtype, with_h0, shape in [(11, "f32", True, (2, 23, 3, 4)), (12, "bf16", True, (1, 17, 5, 3)),
                                        (13, "f32", False, (2, 9, 4, 16))]:
        x = random_scan_inputs(*shape, in_dtype=dtype, seed=seed, with_h0=with_h0, a_log_jitter=0.3)
        y, h = oracle.scan(x, lib_path=lib)
        yb, hb = brute_force(x)
        _close(y, yb, 1e-11, 1e-13, "brute force y")
        _close(h, hb, 1e-11, 1e-13, "brute force h_last")


def pin_lti_convolution(lib=None):
    rng = np.random.default_rng(21)
    Bt, L, Dm, N = 1, 96, 3, 5
    dr_c = rng.normal(size=Dm) * 0.5
    Bc, Cc = rng.normal(size=N), rng.normal(size=N)
    A = -np.exp(np.log(np.arange(1, N + 1))[None, :] + 0.2 * rng.normal(size=(Dm, N)))
    bias = np.log(np.expm1(np.exp(rng.uniform(np.log(1e-2), np.log(0.5), size=Dm))))
    Dk = rng.normal(size=Dm)
    u = rng.normal(size=(Bt, L, Dm))
    x = {
        "u": _f32(u), "delta_raw": _f32(np.broadcast_to(dr_c, (Bt, L, Dm)).copy()), "z": None,
        "B": _f32(np.broadcast_to(Bc, (Bt, L, N)).copy()), "C": _f32(np.broadcast_to(Cc, (Bt, L, N)).copy()),
        "A": _f32(A), "D": _f32(Dk), "delta_bias": _f32(bias), "h0": None,
    }
    y, _ = oracle.scan(x, lib_path=lib)
    # kernel from the stored (fp32) values, in float64
    A64, b64, D64 = _np(x["A"]), _np(x["delta_bias"]), _np(x["D"])
    B64, C64, u64 = _np(x["B"])[0, 0], _np(x["C"])[0, 0], _np(x["u"])[0]
    dr64 = _np(x["delta_raw"])[0, 0]
    for d in range(Dm):
        delta = float(_softplus_ref(dr64[d] + b64[d]))
        ab = np.exp(delta * A64[d])
        k = np.arange(L)
        K = (C64[None, :] * (ab[None, :] ** k[:, None]) * delta * B64[None, :]).sum(axis=1)
        direct = np.convolve(u64[:, d], K)[:L] + D64[d] * u64[:, d]
        nfft = 2 * L
        via_fft = np.fft.irfft(np.fft.rfft(u64[:, d], nfft) * np.fft.rfft(K, nfft), nfft)[:L] + D64[d] * u64[:, d]
        scale = np.abs(direct).max()
        _close(y[0, :, d], direct, 1e-11, 1e-12 * scale, "LTI direct convolution")
        _close(y[0, :, d], via_fft, 1e-9, 1e-11 * scale, "LTI FFT convolution")


def pin_delta_to_zero(lib=None):
    x = random_scan_inputs(2, 31, 4, 6, in_dtype="f32", seed=31, with_h0=True)
    x["delta_raw"] = torch.full_like(x["delta_raw"], -80.0)
    x["delta_bias"] = torch.zeros_like(x["delta_bias"])
    y, h = oracle.scan(x, lib_path=lib)
    h0 = _np(x["h0"])
    _close(h, h0, 1e-25, 0.0, "delta->0 keeps h")
    C, u, z, Dk = _np(x["C"]), _np(x["u"]), _np(x["z"]), _np(x["D"])
    yref = (np.einsum("btn,bdn->btd", C, h0) + Dk[None, None, :] * u) * z * expit(z)
    _close(y, yref, 1e-12, 1e-14, "delta->0 output")


def pin_large_delta_overwrites(lib=None):
    x = random_scan_inputs(1, 19, 3, 5, in_dtype="f32", seed=41, with_h0=True)
    x["delta_raw"] = torch.full_like(x["delta_raw"], 60.0)
    x["delta_bias"] = torch.zeros_like(x["delta_bias"])
    y, h = oracle.scan(x, lib_path=lib)
    B, C, u, z, Dk = _np(x["B"]), _np(x["C"]), _np(x["u"]), _np(x["z"]), _np(x["D"])
    delta = 60.0 + math.log1p(math.exp(-60.0))
    hstep = delta * B[:, :, None, :] * u[:, :, :, None]      # [Bt, L, D, N]: state = this step's input only
    yref = (np.einsum("btn,btdn->btd", C, hstep) + Dk * u) * z * expit(z)
    _close(y, yref, 1e-12, 1e-12, "large delta output")
    _close(h, hstep[:, -1], 1e-12, 1e-12, "large delta h_last")


def pin_chunk_associativity(lib=None):
    rng = np.random.default_rng(51)
    x = random_scan_inputs(2, 70, 3, 7, in_dtype="f32", seed=51, with_h0=True)
    x["z"] = None
    y, h = oracle.scan(x, lib_path=lib)
    A = _np(x["A"])
    for m in sorted(set(rng.integers(1, 69, size=4).tolist())):
        first = {k: (v[:, :m].contiguous() if k in ("u", "delta_raw", "B", "C") and v is not None else v)
                 for k, v in x.items()}
        second = {k: (v[:, m:].contiguous() if k in ("u", "delta_raw", "B", "C") and v is not None else v)
                  for k, v in x.items()}
        second["h0"] = None
        y1, h1 = oracle.scan(first, lib_path=lib)           # carry into the split: h1 (float64)
        y2, h2 = oracle.scan(second, lib_path=lib)          # second chunk from a zero state
        # carry pair of the second chunk: P = exp(A * sum(delta)), S = h2 (local state)
        dr, bias = _np(second["delta_raw"]), _np(second["delta_bias"])
        delta = _softplus_ref(dr + bias[None, None, :])     # [Bt, L2, D]
        S = np.cumsum(delta, axis=1)                        # [Bt, L2, D]
        Pt = np.exp(S[..., None] * A[None, None])           # [Bt, L2, D, N]
        # combine: state_t = P_t * h1 + local_t; y_t = local y_t + C_t . (P_t * h1)
        C2 = _np(second["C"])
        yfix = y2 + np.einsum("btn,btdn->btd", C2, Pt * h1[:, None])
        hfix = Pt[:, -1] * h1 + h2
        _close(y1, y[:, :m], 1e-13, 1e-14, "first chunk")
        _close(yfix, y[:, m:], 1e-10, 1e-12, f"combined chunk at split {m}")
        _close(hfix, h, 1e-10, 1e-12, f"combined h_last at split {m}")


def pin_geometric_series(lib=None):
    L = 60
    dr, bias, Bv, Cv, uv, Av = 0.2, -1.0, 0.75, -1.25, 0.5, -0.8
    x = {"u": _f32(np.full((1, L, 1), uv)), "delta_raw": _f32(np.full((1, L, 1), dr)), "z": None,
         "B": _f32(np.full((1, L, 1), Bv)), "C": _f32(np.full((1, L, 1), Cv)),
         "A": _f32([[Av]]), "D": None, "delta_bias": _f32([bias]), "h0": None}
    y, h = oracle.scan(x, lib_path=lib)
    delta = math.log1p(math.exp(float(np.float32(dr)) + float(np.float32(bias))))
    ab = math.exp(delta * float(np.float32(Av)))
    t = np.arange(L)
    hs = delta * Bv * uv * (1 - ab ** (t + 1)) / (1 - ab)
    _close(y[0, :, 0], Cv * hs, 1e-12, 0, "geometric y")
    _close(h[0, 0, 0], hs[-1], 1e-12, 0, "geometric h")


def pin_single_step_by_hand(lib=None):
    # one token, two states, every term present; evaluated with scalar math
    vals = dict(dr=0.3, bias=-0.5, u=1.25, z=-0.75, A=(-1.0, -2.5), B=(0.5, -1.5), C=(2.0, 0.25),
                D=0.5, h0=(0.1, -0.2))
    x = {"u": _f32([[[vals["u"]]]]), "delta_raw": _f32([[[vals["dr"]]]]), "z": _f32([[[vals["z"]]]]),
         "B": _f32([[vals["B"]]]), "C": _f32([[vals["C"]]]), "A": _f32([vals["A"]]),
         "D": _f32([vals["D"]]), "delta_bias": _f32([vals["bias"]]), "h0": _f32([[vals["h0"]]])}
    y, h = oracle.scan(x, lib_path=lib)
    f = lambda v: float(np.float32(v))  # the stored fp32 value
    delta = math.log(1.0 + math.exp(f(vals["dr"]) + f(vals["bias"])))
    hs = [math.exp(delta * f(vals["A"][n])) * f(vals["h0"][n]) + delta * f(vals["B"][n]) * f(vals["u"])
          for n in range(2)]
    yy = sum(f(vals["C"][n]) * hs[n] for n in range(2)) + f(vals["D"]) * f(vals["u"])
    zz = f(vals["z"])
    yy = yy * zz / (1.0 + math.exp(-zz))
    _close(h[0, 0], hs, 1e-14, 0, "single step h")
    _close(y[0, 0, 0], yy, 1e-14, 0, "single step y")


def pin_softplus_values(lib=None):
    # N=1, B=C=u=1, A=0 (Abar=1), no D, no gate: y_0 = delta exactly.
    for xr, want in [(0.0, math.log(2.0)), (800.0, 800.0), (-30.0, math.log1p(math.exp(-30.0))),
                     (20.5, 20.5 + math.log1p(math.exp(-20.5)))]:
        x = {"u": _f32([[[1.0]]]), "delta_raw": _f32([[[xr]]]), "z": None, "B": _f32([[[1.0]]]),
             "C": _f32([[[1.0]]]), "A": _f32([[0.0]]), "D": None, "delta_bias": None, "h0": None}
        y, _ = oracle.scan(x, lib_path=lib)
        _close(y[0, 0, 0], want, 1e-15, 0, f"softplus({xr})")


def pin_zeros(lib=None):
    x = random_scan_inputs(2, 25, 3, 4, in_dtype="f32", seed=61)
    x0 = dict(x, u=torch.zeros_like(x["u"]))
    y, h = oracle.scan(x0, lib_path=lib)
    assert np.all(y == 0.0) and np.all(h == 0.0), "u = 0 must give y = 0 and h = 0"
    u, z, Dk = _np(x["u"]), _np(x["z"]), _np(x["D"])
    gated_skip = Dk * u * (z * expit(z))
    for key in ("B", "C"):
        xk = dict(x, **{key: torch.zeros_like(x[key])})
        y, h = oracle.scan(xk, lib_path=lib)
        _close(y, gated_skip, 1e-14, 1e-300, f"{key} = 0 output")
        if key == "B":
            assert np.all(h == 0.0), "B = 0 must give h = 0"


def pin_linearity_in_u(lib=None):
    rng = np.random.default_rng(71)
    x = random_scan_inputs(1, 40, 3, 5, in_dtype="f32", seed=71)
    x["z"] = None
    x["D"] = None
    u1 = rng.integers(-32, 33, size=x["u"].shape) / 8.0
    u2 = rng.integers(-32, 33, size=x["u"].shape) / 8.0
    y1, h1 = oracle.scan(dict(x, u=_f32(u1)), lib_path=lib)
    y2, h2 = oracle.scan(dict(x, u=_f32(u2)), lib_path=lib)
    y3, h3 = oracle.scan(dict(x, u=_f32(2 * u1 - 3 * u2)), lib_path=lib)  # exact in fp32
    sc = np.abs(y3).max()
    _close(y3, 2 * y1 - 3 * y2, 1e-10, 1e-13 * sc, "linearity y")
    _close(h3, 2 * h1 - 3 * h2, 1e-10, 1e-13 * np.abs(h3).max(), "linearity h")


def pin_independence(lib=None):
    x = random_scan_inputs(2, 30, 5, 4, in_dtype="f32", seed=81, with_h0=True)
    y, h = oracle.scan(x, lib_path=lib)
    # perturb channel (1, 2) only
    x2 = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    for key in ("u", "delta_raw", "z"):
        x2[key][1, :, 2] += 0.5
    y2, h2 = oracle.scan(x2, lib_path=lib)
    mask = np.ones(y.shape, bool)
    mask[1, :, 2] = False
    assert np.array_equal(y[mask], y2[mask]), "other channels changed"
    assert not np.array_equal(y[1, :, 2], y2[1, :, 2]), "perturbed channel unchanged"
    # permute channels together with their parameters
    perm = torch.tensor([3, 0, 4, 1, 2])
    xp = dict(x)
    for key in ("u", "delta_raw", "z"):
        xp[key] = x[key][:, :, perm].contiguous()
    xp["A"] = x["A"][perm].contiguous()
    xp["D"] = x["D"][perm].contiguous()
    xp["delta_bias"] = x["delta_bias"][perm].contiguous()
    xp["h0"] = x["h0"][:, perm].contiguous()
    yp, hp = oracle.scan(xp, lib_path=lib)
    assert np.array_equal(yp, y[:, :, perm.numpy()]), "channel permutation not equivariant"
    assert np.array_equal(hp, h[:, perm.numpy()]), "state permutation not equivariant"
    # swap batch elements
    xb = {k: (v.flip(0).contiguous() if k in ("u", "delta_raw", "z", "B", "C", "h0") and v is not None else v)
          for k, v in x.items()}
    yb, hb = oracle.scan(xb, lib_path=lib)
    assert np.array_equal(yb, y[::-1]) and np.array_equal(hb, h[::-1]), "batch not independent"


def pin_decode_equals_scan(lib=None):
    x = random_scan_inputs(3, 21, 4, 16, in_dtype="bf16", seed=91, with_h0=True)
    y, h = oracle.scan(x, lib_path=lib)
    hs = x["h0"].double().numpy().copy()
    for t in range(x["u"].shape[1]):
        step = {"u": x["u"][:, t].contiguous(), "delta_raw": x["delta_raw"][:, t].contiguous(),
                "z": x["z"][:, t].contiguous(), "B": x["B"][:, t].contiguous(), "C": x["C"][:, t].contiguous(),
                "A": x["A"], "D": x["D"], "delta_bias": x["delta_bias"]}
        yt = oracle.state_update(hs, step, lib_path=lib)
        _close(yt, y[:, t], 1e-14, 1e-300, f"decode step {t}")
    _close(hs, h, 1e-14, 1e-300, "decode final state")


def pin_sampled_channels(lib=None):
    x = random_scan_inputs(3, 33, 7, 16, in_dtype="bf16", seed=101, with_h0=True)
    y, h = oracle.scan(x, lib_path=lib)
    ch = np.array([[0, 6], [2, 0], [1, 3], [2, 6]])
    ys, hs = oracle.scan(x, channels=ch, lib_path=lib)
    for i, (b, d) in enumerate(ch):
        assert np.array_equal(ys[i], y[b, :, d]) and np.array_equal(hs[i], h[b, d]), "sampled != full"


def pin_bf16_widening(lib=None):
    x = random_scan_inputs(2, 27, 5, 16, in_dtype="bf16", seed=111, with_h0=True)
    xf = {k: (v.float() if isinstance(v, torch.Tensor) and v.dtype == torch.bfloat16 else v)
          for k, v in x.items()}
    y, h = oracle.scan(x, lib_path=lib)
    yf, hf = oracle.scan(xf, lib_path=lib)
    assert np.array_equal(y, yf) and np.array_equal(h, hf), "bf16 widening is not exact"


def pin_stability_bound(lib=None):
    # A < 0 gives |Abar| < 1, hence |h_t| <= |h_0| + sum_s |delta_s B_s u_s| per state
    x = random_scan_inputs(2, 64, 6, 16, in_dtype="f32", seed=121, with_h0=True, delta_raw_scale=2.0)
    _, h = oracle.scan(x, lib_path=lib)
    dr, bias = _np(x["delta_raw"]), _np(x["delta_bias"])
    delta = _softplus_ref(dr + bias[None, None, :])
    B, u, h0 = _np(x["B"]), _np(x["u"]), _np(x["h0"])
    bound = np.abs(h0) + np.einsum("btd,btn->bdn", np.abs(delta * u), np.abs(B))
    assert np.all(np.abs(h) <= bound * (1 + 1e-12)), "stability bound violated"


# ----------------------------------------------------------------- convolution front-end
# The block's causal depthwise convolution with SiLU (review page, method step
# 3; mlqm.cn tutorial section 7.1) and its decode state (the inference page's
# decode-state table): pinned against numpy's convolution, impulse responses,
# chunk continuity through the carried state, and decode-equals-forward.

def _conv_ref(x):
    """Per channel: numpy.convolve of (state, x) with the reversed taps ('valid'),
    plus bias, then SiLU by scipy's logistic function."""
    xx = x["x"].double().numpy()
    w = x["weight"].double().numpy()
    b = x["bias"].double().numpy() if x.get("bias") is not None else np.zeros(w.shape[0])
    Bt, L, Dm = xx.shape
    K = w.shape[1]
    st = x["state"].double().numpy() if x.get("state") is not None else np.zeros((Bt, Dm, K - 1))
    pre = np.zeros((Bt, L, Dm))
    for bb in range(Bt):
        for d in range(Dm):
            e = np.concatenate([st[bb, d], xx[bb, :, d]])
            pre[bb, :, d] = np.convolve(e, w[d][::-1], mode="valid") + b[d]
    tail = np.concatenate([st, xx.transpose(0, 2, 1)], axis=2)[:, :, -(K - 1):] if K > 1 else np.zeros((Bt, Dm, 0))
    return pre, tail


def pin_conv_numpy(lib=None):
    from workloads.gen import random_conv_inputs
    path = lib
    for (Bt, L, Dm, K, dt, st) in [(2, 17, 5, 4, "f32", True), (1, 9, 3, 2, "bf16", False), (2, 2, 4, 4, "f32", True),
                                   (1, 12, 2, 3, "bf16", True)]:
        x = random_conv_inputs(Bt, L, Dm, K, dt, seed=Bt * 100 + L + K, with_state=st)
        pre, tail = _conv_ref(x)
        y, so = oracle.conv1d(x, silu=False, lib_path=path)
        np.testing.assert_allclose(y, pre, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(so, tail, rtol=0, atol=0)
        ys, _ = oracle.conv1d(x, silu=True, lib_path=path)
        np.testing.assert_allclose(ys, pre * expit(pre), rtol=1e-12, atol=1e-13)


def pin_conv_impulse(lib=None):
    # a unit impulse at t0 (no state) gives bias + w[d, K-1-j] at t0 + j, bias elsewhere
    path = lib
    Dm, K, L, t0 = 3, 4, 12, 5
    w = torch.tensor([[1.0, 2.0, 3.0, 4.0], [0.5, -1.0, 0.25, 2.0], [-3.0, 0.0, 1.5, 1.0]])
    bias = torch.tensor([0.1, -0.2, 0.0])
    xx = torch.zeros(1, L, Dm)
    xx[0, t0, :] = 1.0
    y, so = oracle.conv1d({"x": xx, "weight": w, "bias": bias, "state": None}, silu=False, lib_path=path)
    for d in range(Dm):
        expect = np.full(L, float(bias[d]))
        for j in range(K):
            expect[t0 + j] += float(w[d, K - 1 - j])
        np.testing.assert_allclose(y[0, :, d], expect, rtol=0, atol=1e-15)
    assert np.all(so == 0.0)


def pin_conv_chunk_continuity(lib=None):
    # running two halves, the second from the first's final state, equals one pass
    from workloads.gen import random_conv_inputs
    path = lib
    for K in (2, 3, 4):
        x = random_conv_inputs(2, 23, 6, K, "f32", seed=K, with_state=True)
        y, so = oracle.conv1d(x, lib_path=path)
        for m in (1, 2, 10):
            a = dict(x, x=x["x"][:, :m].contiguous())
            ya, sa = oracle.conv1d(a, lib_path=path)
            bpart = dict(x, x=x["x"][:, m:].contiguous(), state=torch.tensor(sa, dtype=torch.float32))
            yb, sb = oracle.conv1d(bpart, lib_path=path)
            np.testing.assert_allclose(np.concatenate([ya, yb], axis=1), y, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(sb, so, rtol=0, atol=0)


def pin_conv_decode_equals_forward(lib=None):
    from workloads.gen import random_conv_inputs
    path = lib
    x = random_conv_inputs(3, 11, 7, 4, "bf16", seed=5, with_state=True)
    y, so = oracle.conv1d(x, lib_path=path)
    st = x["state"].double().numpy().copy()
    for t in range(11):
        yt = oracle.conv1d_update(st, x["x"][:, t].contiguous(), x["weight"], x["bias"], lib_path=path)
        np.testing.assert_allclose(yt, y[:, t], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(st, so, rtol=0, atol=0)


# ----------------------------------------------------------------- gradients
# The backward pass the pages' training recomputes (review page, method step 2
# (3)), pinned against central finite differences of the forward oracle: with
# loss = sum(w_y * y) + sum(w_h * h_last), dy = w_y and dh_last = w_h; each
# sampled input entry is moved by +-2^-10 (exact in float32).

def _fd_loss(x, wy, wh, path):
    y, h = oracle.scan(x, lib_path=path)
    return float(np.sum(wy * y) + np.sum(wh * h))


def pin_backward_finite_differences(lib=None):
    path = lib
    rng = np.random.default_rng(5)
    for (Bt, L, Dm, N, seed, hz, with_h0) in [(2, 9, 3, 4, 1, True, True), (1, 6, 2, 3, 2, False, False)]:
        x = random_scan_inputs(Bt, L, Dm, N, in_dtype="f32", seed=seed, with_h0=with_h0, has_z=hz,
                               a_log_jitter=0.3, delta_raw_scale=1.0)
        if with_h0:
            x["h0"] = (0.5 * x["h0"]).contiguous()
        wy = rng.normal(size=(Bt, L, Dm))
        wh = rng.normal(size=(Bt, Dm, N))
        g = oracle.scan_bwd(x, torch.tensor(wy, dtype=torch.float32),
                            torch.tensor(wh, dtype=torch.float32), lib_path=path)
        # the loss weights as stored in float32 (what the backward saw)
        wy = torch.tensor(wy, dtype=torch.float32).double().numpy()
        wh = torch.tensor(wh, dtype=torch.float32).double().numpy()
        hstep = 2.0 ** -10
        checks = [("u", "du"), ("delta_raw", "ddelta_raw"), ("B", "dB"), ("C", "dC"), ("A", "dA"), ("D", "dD"),
                  ("delta_bias", "ddelta_bias")] + ([("z", "dz")] if hz else []) + ([("h0", "dh0")] if with_h0 else [])
        for name, gname in checks:
            t = x[name]
            flat = t.view(-1)
            for idx in rng.choice(flat.numel(), size=min(6, flat.numel()), replace=False):
                old = float(flat[idx])
                flat[idx] = old + hstep
                lp = _fd_loss(x, wy, wh, path)
                flat[idx] = old - hstep
                lm = _fd_loss(x, wy, wh, path)
                flat[idx] = old
                fd = (lp - lm) / (2 * hstep)
                an = g[gname].reshape(-1)[idx]
                assert abs(fd - an) <= 1e-5 * max(1.0, abs(fd)), (name, int(idx), fd, an)
        if not hz:
            assert np.all(g["dz"] == 0.0)


def pin_backward_bf16_widening(lib=None):
    # bf16 inputs give the gradients of the same values held as float32
    x = random_scan_inputs(2, 11, 3, 4, in_dtype="bf16", seed=8, with_h0=True)
    xf = {k: (v.float() if isinstance(v, torch.Tensor) and v.dtype == torch.bfloat16 else v) for k, v in x.items()}
    dy = torch.randn(2, 11, 3, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    g1 = oracle.scan_bwd(x, dy, lib_path=lib)
    g2 = oracle.scan_bwd(xf, dy.float(), lib_path=lib)
    for k in g1:
        np.testing.assert_allclose(g1[k], g2[k], rtol=0, atol=0)


# ------------------------------------------------- generalised scan (any N, groups, ZOH)

def _slice_group(x, g, G):
    """Channels of group g with that group's B and C as a shared (G = 1) problem."""
    Dm = x["u"].shape[2]
    lo, hi = g * (Dm // G), (g + 1) * (Dm // G)
    out = {}
    for k in ("u", "delta_raw", "z"):
        out[k] = x[k][:, :, lo:hi].contiguous() if x.get(k) is not None else None
    out["B"] = x["B"][:, :, g, :].contiguous()
    out["C"] = x["C"][:, :, g, :].contiguous()
    out["A"] = x["A"][lo:hi].contiguous()
    for k in ("D", "delta_bias"):
        out[k] = x[k][lo:hi].contiguous() if x.get(k) is not None else None
    out["h0"] = x["h0"][:, lo:hi].contiguous() if x.get("h0") is not None else None
    return out, lo, hi


def pin_general_zoh_scipy(lib=None):
    # LTI problem (delta, B, C constant over time): the zero-order-hold scan is
    # the discrete system scipy builds from (A, B, C, D) and the step delta
    from scipy.signal import cont2discrete, dlsim
    rng = np.random.default_rng(31)
    for N in (3, 64):
        Bt, L, Dm = 1, 40, 3
        dr_c = rng.normal(size=Dm)
        Bc, Cc = rng.normal(size=N), rng.normal(size=N)
        x = {"u": _f32(rng.normal(size=(Bt, L, Dm))),
             "delta_raw": _f32(np.broadcast_to(dr_c, (Bt, L, Dm))),
             "z": None,
             "B": _f32(np.broadcast_to(Bc, (Bt, L, 1, N))), "C": _f32(np.broadcast_to(Cc, (Bt, L, 1, N))),
             "A": _f32(-np.exp(rng.normal(size=(Dm, N)) * 0.7)),
             "D": _f32(rng.normal(size=Dm)), "delta_bias": _f32(rng.normal(size=Dm) * 0.3),
             "h0": _f32(rng.normal(size=(Bt, Dm, N)))}
        y, h = oracle.scan_general(x, 1, "zoh", lib_path=lib)
        u, A, Dk, h0 = _np(x["u"]), _np(x["A"]), _np(x["D"]), _np(x["h0"])
        Bv, Cv = _np(x["B"])[0, 0, 0], _np(x["C"])[0, 0, 0]
        for d in range(Dm):
            delta = float(_softplus_ref(_np(x["delta_raw"])[0, 0, d] + _np(x["delta_bias"])[d]))
            Ad, Bd, Cd, Dd, _ = cont2discrete((np.diag(A[d]), Bv[:, None], Cv[None, :], np.array([[Dk[d]]])),
                                              delta, method="zoh")
            # dlsim's state before input k; this scan's state after input t is dlsim's x[t + 1]
            _, _, xs = dlsim((Ad, Bd, Cd, Dd, delta), np.append(u[0, :, d], 0.0), x0=h0[0, d])
            ref = xs[1:] @ Cv + Dk[d] * u[0, :, d]
            _close(y[0, :, d], ref, 1e-9, 1e-11, f"zoh scipy y N={N}")
            _close(h[0, d], xs[L], 1e-9, 1e-11, f"zoh scipy h_last N={N}")


def pin_general_first_order_brute_force(lib=None):
    # the first-order generalised scan at state sizes 16 and 64 is the brute-force sum
    for N, seed, dtype in ((16, 41, "f32"), (64, 42, "bf16")):
        x = random_general_inputs(2, 11, 3, N, 1, in_dtype=dtype, seed=seed, with_h0=True, a_log_jitter=0.3)
        y, h = oracle.scan_general(x, 1, "euler", lib_path=lib)
        xb = dict(x, B=x["B"][:, :, 0, :], C=x["C"][:, :, 0, :])
        yb, hb = brute_force(xb)
        _close(y, yb, 1e-11, 1e-13, f"general euler y N={N}")
        _close(h, hb, 1e-11, 1e-13, f"general euler h_last N={N}")


def pin_general_groups(lib=None):
    # G groups: each group's channels give what a shared-B/C problem of that
    # group's channels and rows gives; first order checked against brute force
    G = 4
    x = random_general_inputs(2, 13, 8, 32, G, in_dtype="f32", seed=43, with_h0=True, a_log_jitter=0.3)
    for disc in ("euler", "zoh"):
        y, h = oracle.scan_general(x, G, disc, lib_path=lib)
        for g in range(G):
            xs, lo, hi = _slice_group(x, g, G)
            ys, hs = oracle.scan_general(xs, 1, disc, lib_path=lib)
            _close(y[:, :, lo:hi], ys, 0.0, 0.0, f"group {g} y {disc}")
            _close(h[:, lo:hi], hs, 0.0, 0.0, f"group {g} h {disc}")
            if disc == "euler":
                yb, hb = brute_force(xs)
                _close(ys, yb, 1e-11, 1e-13, f"group {g} brute force")
    # one B/C per channel (G = dim)
    x = random_general_inputs(1, 9, 6, 16, 6, in_dtype="f32", seed=44, with_h0=False)
    y, _ = oracle.scan_general(x, 6, "euler", lib_path=lib)
    for g in range(6):
        xs, lo, hi = _slice_group(x, g, 6)
        yb, _ = brute_force(xs)
        _close(y[:, :, lo:hi], yb, 1e-11, 1e-13, f"per-channel B/C, channel {g}")


def pin_general_zoh_small_step(lib=None):
    # for delta*A -> 0 the zero-order hold tends to the first-order form: the
    # difference of Bbar is delta B (e^{delta A} - 1 - delta A) / (delta A), of order delta^2 A B / 2
    x = random_general_inputs(1, 20, 4, 16, 1, in_dtype="f32", seed=45, with_h0=False)
    x["delta_raw"] = torch.full_like(x["delta_raw"], -12.0)
    x["delta_bias"] = None
    ye, _ = oracle.scan_general(x, 1, "euler", lib_path=lib)
    yz, _ = oracle.scan_general(x, 1, "zoh", lib_path=lib)
    delta = float(_softplus_ref(-12.0))
    amax = float(np.abs(_np(x["A"])).max())
    assert np.all(np.abs(yz - ye) <= 0.6 * delta * amax * np.abs(ye).max() + 1e-300), "zoh small step"
    assert np.any(yz != ye), "zoh identical to first order"


# ------------------------------------------------- state-space-dual (Mamba-2) layer

def ssd_dense(x, G):
    """y = M x with the dense semiseparable matrix per (batch, head), plus the
    initial state's decayed readout; h_last from the same weights."""
    X, dt, B, C = _np(x["x"]), _np(x["dt"]), _np(x["B"]), _np(x["C"])
    A, Dk, bias, h0 = _np(x["A"]), _np(x.get("D")), _np(x.get("dt_bias")), _np(x.get("h0"))
    Bt, L, H, P = X.shape
    N = B.shape[-1]
    y = np.zeros((Bt, L, H, P))
    hl = np.zeros((Bt, H, P, N))
    for b in range(Bt):
        for hd in range(H):
            g = hd // (H // G)
            delta = _softplus_ref(dt[b, :, hd] + (bias[hd] if bias is not None else 0.0))   # [L]
            cum = np.concatenate([[0.0], np.cumsum(delta * A[hd])])                         # cum[t+1] = sum_{k<=t}
            seg = cum[1:, None] - cum[None, 1:]                                             # sum_{s<k<=t}
            M = np.where(np.tri(L, dtype=bool), (C[b, :, g] @ B[b, :, g].T) * delta[None, :] * np.exp(
                np.where(np.tri(L, dtype=bool), seg, 0.0)), 0.0)
            y[b, :, hd] = M @ X[b, :, hd]
            w = np.exp(cum[L] - cum[1:]) * delta                                            # weight of step s in h_last
            hl[b, hd] = (X[b, :, hd] * w[:, None]).T @ B[b, :, g]
            if h0 is not None:
                y[b, :, hd] += np.exp(cum[1:])[:, None] * (C[b, :, g] @ h0[b, hd].T)
                hl[b, hd] += np.exp(cum[L]) * h0[b, hd]
            if Dk is not None:
                y[b, :, hd] += Dk[hd] * X[b, :, hd]
    return y, hl


def pin_ssd_semiseparable(lib=None):
    for (Bt, L, H, P, N, G, dtype, with_h0, seed) in [(2, 21, 4, 3, 5, 2, "f32", True, 51),
                                                       (1, 33, 2, 4, 16, 1, "bf16", False, 52)]:
        x = random_ssd_inputs(Bt, L, H, P, N, G, in_dtype=dtype, seed=seed, with_h0=with_h0)
        y, h = oracle.ssd(x, G, lib_path=lib)
        yd, hd = ssd_dense(x, G)
        _close(y, yd, 1e-10, 1e-12, "ssd y vs semiseparable matrix")
        _close(h, hd, 1e-10, 1e-12, "ssd h_last vs semiseparable matrix")


ALL_PINS = [pin_ssd_semiseparable, pin_general_zoh_scipy, pin_general_first_order_brute_force, pin_general_groups,
            pin_general_zoh_small_step, pin_backward_finite_differences, pin_backward_bf16_widening, pin_conv_numpy, pin_conv_impulse, pin_conv_chunk_continuity, pin_conv_decode_equals_forward,
            pin_brute_force, pin_lti_convolution, pin_delta_to_zero, pin_large_delta_overwrites,
            pin_chunk_associativity, pin_geometric_series, pin_single_step_by_hand, pin_softplus_values,
            pin_zeros, pin_linearity_in_u, pin_independence, pin_decode_equals_scan,
            pin_sampled_channels, pin_bf16_widening, pin_stability_bound]
