"""Float64 CPU oracle for the selective scan (S6) — TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this package. The product path (the CUDA library and its binding)
never imports, links or runs it.

The arithmetic lives in `ss_oracle.c` (plain sequential float64 loops, see its
header for the definition and the passages it follows); this module only
marshals host tensors into that library. Inputs are the exact stored values
(fp32, or bf16 bit patterns widened exactly to float64 inside the C code).

Every function here is pinned by the `-m "not gpu"` tests in
tests/test_oracle_pins.py (brute-force unrolled sum, LTI convolution checked
directly and by FFT, delta->0, large delta, chunk associativity, geometric
closed form, hand-computed L=1, zero/linearity/independence properties,
decode-equals-scan; for the gradients: central finite differences of the
forward oracle; for the convolution front-end: numpy's convolution,
impulse responses, chunk continuity through the state, decode-equals-forward;
for the generalised scan: scipy's zero-order-hold discretisation and
simulation, the scan on its special case, per-group slices, a split of the
states; for the state-space-dual layer: its dense semiseparable-matrix form,
computed in numpy).
"""

import ctypes
import os

import numpy as np
import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBS = {}

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


def load(path: str = None) -> ctypes.CDLL:
    """Load (building if needed) the oracle library; `path` selects another build."""
    path = path or _build.build()
    if path not in _LIBS:
        lib = ctypes.CDLL(path)
        lib.ss_oracle_scan.restype = ctypes.c_int
        lib.ss_oracle_scan.argtypes = [_I64, _I64, _I64, _I64, ctypes.c_int,
                                       _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _I64, _P, _P, ctypes.c_int]
        lib.ss_oracle_state_update.restype = ctypes.c_int
        lib.ss_oracle_state_update.argtypes = [_I64, _I64, _I64, ctypes.c_int, _P,
                                               _P, _P, _P, _P, _P, _P, _P, _P,
                                               _P, _I64, _P]
        lib.ss_oracle_scan_bwd.restype = ctypes.c_int
        lib.ss_oracle_scan_bwd.argtypes = [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int] + [_P] * 20
        lib.ss_oracle_scan_general.restype = ctypes.c_int
        lib.ss_oracle_scan_general.argtypes = [_I64, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                               _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, ctypes.c_int]
        lib.ss_oracle_conv1d.restype = ctypes.c_int
        lib.ss_oracle_conv1d.argtypes = [_I64, _I64, _I64, _I64, ctypes.c_int, _P, _P, _P, _P,
                                         ctypes.c_int, _P, _P]
        lib.ss_oracle_conv1d_update.restype = ctypes.c_int
        lib.ss_oracle_conv1d_update.argtypes = [_I64, _I64, _I64, ctypes.c_int, _P, _P, _P, _P,
                                                ctypes.c_int, _P]
        _LIBS[path] = lib
    return _LIBS[path]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"oracle inputs must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return t.data_ptr()


def _f32(t):
    if t is None:
        return None
    assert t.dtype == torch.float32
    return t.contiguous()


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def scan(x: dict, channels=None, nthreads: int = None, lib_path: str = None):
    """Selective scan in float64 on the host.

    x: dict of CPU tensors u, delta_raw, z (or None) [Bt, L, D]; B, C [Bt, L, N]
       (all float32 or all bfloat16); A [D, N], D [D] or None, delta_bias [D] or
       None, h0 [Bt, D, N] or None (float32).
    channels: None for every (b, d), or an int array [n, 2] of (b, d) pairs.
    Returns (y, h_last) as float64 numpy arrays: y [Bt, L, D] and h [Bt, D, N]
    for the full problem, else y [n, L] and h [n, N] for the listed channels.
    """
    lib = load(lib_path)
    u, dr, z, B, C = x["u"], x["delta_raw"], x.get("z"), x["B"], x["C"]
    Bt, L, Dm = u.shape
    N = B.shape[-1]
    code = _dtype_code(u)
    for t in (dr, z, B, C):
        if t is not None and _dtype_code(t) != code:
            raise TypeError("u, delta_raw, z, B, C must share one dtype")
    A = _f32(x["A"])
    Dk = _f32(x.get("D"))
    bias = _f32(x.get("delta_bias"))
    h0 = _f32(x.get("h0"))
    full = channels is None
    if full:
        bb, dd = np.meshgrid(np.arange(Bt), np.arange(Dm), indexing="ij")
        chans = np.stack([bb.ravel(), dd.ravel()], axis=1).astype(np.int64)
    else:
        chans = np.ascontiguousarray(np.asarray(channels, dtype=np.int64).reshape(-1, 2))
    n = chans.shape[0]
    y = np.zeros((n, L), dtype=np.float64)
    h = np.zeros((n, N), dtype=np.float64)
    rc = lib.ss_oracle_scan(Bt, L, Dm, N, code, _ptr(u), _ptr(dr), _ptr(z), _ptr(B), _ptr(C),
                            _ptr(A), _ptr(Dk), _ptr(bias), _ptr(h0),
                            chans.ctypes.data, n, y.ctypes.data, h.ctypes.data,
                            nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle scan rejected its arguments")
    if full:
        return y.reshape(Bt, Dm, L).transpose(0, 2, 1).copy(), h.reshape(Bt, Dm, N)
    return y, h


DISC = {"euler": 0, "zoh": 1}


def scan_general(x: dict, ngroups: int = 1, disc: str = "euler", channels=None, nthreads: int = None,
                 lib_path: str = None):
    """Generalised selective scan in float64: state size N = A.shape[1], B and C
    [Bt, L, G, N] (or [Bt, L, N] when G = 1) shared by the dim / G consecutive
    channels of each group, Bbar first order ("euler") or zero-order hold
    ("zoh"). Other inputs and the return value as for scan()."""
    lib = load(lib_path)
    u, dr, z, B, C = x["u"], x["delta_raw"], x.get("z"), x["B"], x["C"]
    Bt, L, Dm = u.shape
    A = _f32(x["A"])
    N = A.shape[1]
    code = _dtype_code(u)
    for t in (dr, z, B, C):
        if t is not None and _dtype_code(t) != code:
            raise TypeError("u, delta_raw, z, B, C must share one dtype")
    if B.dim() == 3:
        B, C = B.unsqueeze(2), C.unsqueeze(2)
    assert B.shape == (Bt, L, ngroups, N) and C.shape == (Bt, L, ngroups, N), (B.shape, ngroups, N)
    B, C = B.contiguous(), C.contiguous()
    full = channels is None
    if full:
        bb, dd = np.meshgrid(np.arange(Bt), np.arange(Dm), indexing="ij")
        chans = np.stack([bb.ravel(), dd.ravel()], axis=1).astype(np.int64)
    else:
        chans = np.ascontiguousarray(np.asarray(channels, dtype=np.int64).reshape(-1, 2))
    n = chans.shape[0]
    y = np.zeros((n, L), dtype=np.float64)
    h = np.zeros((n, N), dtype=np.float64)
    rc = lib.ss_oracle_scan_general(Bt, L, Dm, N, ngroups, DISC[disc], code, _ptr(u), _ptr(dr), _ptr(z), _ptr(B),
                                    _ptr(C), _ptr(A), _ptr(_f32(x.get("D"))), _ptr(_f32(x.get("delta_bias"))),
                                    _ptr(_f32(x.get("h0"))), chans.ctypes.data, n, y.ctypes.data, h.ctypes.data,
                                    nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle scan_general rejected its arguments")
    if full:
        return y.reshape(Bt, Dm, L).transpose(0, 2, 1).copy(), h.reshape(Bt, Dm, N)
    return y, h


def ssd(x: dict, ngroups: int = 1, channels=None, nthreads: int = None, lib_path: str = None):
    """State-space-dual (Mamba-2) layer in float64: per head h a scalar decay,
    h_t = exp(delta_t A_h) h_{t-1} + delta_t x_t B_t^T ([P, N] per head),
    y_t = h_t C_t + D_h x_t, delta = softplus(dt + dt_bias). That is the
    selective scan with channels (h, p), A[(h, p), n] = A_h for every n, and
    the group of head h (B, C shared by H / G consecutive heads), so it runs
    as scan_general on those expanded inputs.

    x: dict of CPU tensors x [Bt, L, H, P], dt [Bt, L, H], B, C [Bt, L, G, N]
    (one dtype), A [H], D [H] or None, dt_bias [H] or None, h0 [Bt, H, P, N] or
    None (float32). Returns float64 (y [Bt, L, H, P], h_last [Bt, H, P, N]);
    with channels, an int array [n, 3] of (b, h, p), y [n, L] and h_last [n, N].
    """
    xx, dt = x["x"], x["dt"]
    Bt, L, H, P = xx.shape
    N = x["B"].shape[-1]
    exp = {
        "u": xx.reshape(Bt, L, H * P).contiguous(),
        "delta_raw": dt.repeat_interleave(P, dim=2).contiguous(),
        "z": None,
        "B": x["B"], "C": x["C"],
        "A": _f32(x["A"]).repeat_interleave(P).view(H * P, 1).expand(H * P, N).contiguous(),
        "D": _f32(x["D"]).repeat_interleave(P).contiguous() if x.get("D") is not None else None,
        "delta_bias": _f32(x["dt_bias"]).repeat_interleave(P).contiguous() if x.get("dt_bias") is not None else None,
        "h0": _f32(x["h0"]).reshape(Bt, H * P, N).contiguous() if x.get("h0") is not None else None,
    }
    if channels is not None:
        ch = np.asarray(channels, dtype=np.int64).reshape(-1, 3)
        pairs = np.stack([ch[:, 0], ch[:, 1] * P + ch[:, 2]], axis=1)
        return scan_general(exp, ngroups, "euler", channels=pairs, nthreads=nthreads, lib_path=lib_path)
    y, h = scan_general(exp, ngroups, "euler", nthreads=nthreads, lib_path=lib_path)
    return y.reshape(Bt, L, H, P), h.reshape(Bt, H, P, N)


def state_update(h: np.ndarray, x: dict, channels=None, lib_path: str = None):
    """One decode step in float64, state updated in place.

    h: float64 numpy array [S, D, N] (modified); x: dict of CPU tensors u,
    delta_raw, z (or None) [S, D]; B, C [S, N]; A [D, N], D, delta_bias [D].
    Returns y as float64 [S, D] (full) or [n] for listed (b, d) channels.
    """
    lib = load(lib_path)
    u, dr, z, B, C = x["u"], x["delta_raw"], x.get("z"), x["B"], x["C"]
    S, Dm = u.shape
    N = B.shape[-1]
    code = _dtype_code(u)
    assert h.dtype == np.float64 and h.flags.c_contiguous and h.shape == (S, Dm, N)
    full = channels is None
    if full:
        bb, dd = np.meshgrid(np.arange(S), np.arange(Dm), indexing="ij")
        chans = np.stack([bb.ravel(), dd.ravel()], axis=1).astype(np.int64)
    else:
        chans = np.ascontiguousarray(np.asarray(channels, dtype=np.int64).reshape(-1, 2))
    n = chans.shape[0]
    y = np.zeros(n, dtype=np.float64)
    rc = lib.ss_oracle_state_update(S, Dm, N, code, h.ctypes.data, _ptr(u), _ptr(dr), _ptr(z),
                                    _ptr(B), _ptr(C), _ptr(_f32(x["A"])), _ptr(_f32(x.get("D"))),
                                    _ptr(_f32(x.get("delta_bias"))), chans.ctypes.data, n,
                                    y.ctypes.data)
    if rc != 0:
        raise ValueError("oracle state_update rejected its arguments")
    return y.reshape(S, Dm) if full else y


def conv1d(x: dict, silu: bool = True, lib_path: str = None):
    """Causal depthwise convolution front-end in float64 on the host.

    x: dict of CPU tensors x [Bt, L, D] (float32 or bfloat16), weight [D, K] and
    bias [D] or None (float32), state [Bt, D, K-1] or None (same dtype as x).
    Returns (y [Bt, L, D], state_out [Bt, D, K-1]) as float64 numpy arrays.
    """
    lib = load(lib_path)
    xx, w, bias, st = x["x"], _f32(x["weight"]), _f32(x.get("bias")), x.get("state")
    Bt, L, Dm = xx.shape
    K = w.shape[1]
    code = _dtype_code(xx)
    if st is not None and _dtype_code(st) != code:
        raise TypeError("x and state must share one dtype")
    y = np.zeros((Bt, L, Dm), dtype=np.float64)
    so = np.zeros((Bt, Dm, max(K - 1, 0)), dtype=np.float64)
    rc = lib.ss_oracle_conv1d(Bt, L, Dm, K, code, _ptr(xx), _ptr(w), _ptr(bias), _ptr(st), int(silu),
                              y.ctypes.data, so.ctypes.data)
    if rc != 0:
        raise ValueError("oracle conv1d rejected its arguments")
    return y, so


def conv1d_update(state: np.ndarray, x, weight, bias=None, silu: bool = True, lib_path: str = None):
    """One decode step of the convolution in float64, state [Bt, D, K-1]
    (float64 numpy, modified in place); x [Bt, D] CPU tensor. Returns y [Bt, D]."""
    lib = load(lib_path)
    Bt, Dm = x.shape
    w = _f32(weight)
    K = w.shape[1]
    assert state.dtype == np.float64 and state.flags.c_contiguous and state.shape == (Bt, Dm, K - 1)
    y = np.zeros((Bt, Dm), dtype=np.float64)
    rc = lib.ss_oracle_conv1d_update(Bt, Dm, K, _dtype_code(x), state.ctypes.data, _ptr(x.contiguous()), _ptr(w),
                                     _ptr(_f32(bias)), int(silu), y.ctypes.data)
    if rc != 0:
        raise ValueError("oracle conv1d_update rejected its arguments")
    return y


def scan_bwd(x: dict, dy, dh_last=None, lib_path: str = None) -> dict:
    """Gradients of the selective scan in float64 (reverse sweep of the adjoint).

    x: the forward inputs as for scan(); dy [Bt, L, D] CPU tensor (float32 or
    bfloat16): the gradient of y; dh_last [Bt, D, N] float32 or None: of h_last.
    Returns float64 numpy arrays du, ddelta_raw, dz [Bt, L, D]; dA [D, N];
    dB, dC [Bt, L, N]; dD, ddelta_bias [D]; dh0 [Bt, D, N].
    """
    lib = load(lib_path)
    u, dr, z, B, C = x["u"], x["delta_raw"], x.get("z"), x["B"], x["C"]
    Bt, L, Dm = u.shape
    N = B.shape[-1]
    out = {k: np.zeros(sh) for k, sh in [("du", (Bt, L, Dm)), ("ddelta_raw", (Bt, L, Dm)), ("dz", (Bt, L, Dm)),
                                         ("dA", (Dm, N)), ("dB", (Bt, L, N)), ("dC", (Bt, L, N)), ("dD", (Dm,)),
                                         ("ddelta_bias", (Dm,)), ("dh0", (Bt, Dm, N))]}
    rc = lib.ss_oracle_scan_bwd(Bt, L, Dm, N, _dtype_code(u), _dtype_code(dy), _ptr(u), _ptr(dr), _ptr(z), _ptr(B),
                                _ptr(C), _ptr(_f32(x["A"])), _ptr(_f32(x.get("D"))), _ptr(_f32(x.get("delta_bias"))),
                                _ptr(_f32(x.get("h0"))), _ptr(dy.contiguous()), _ptr(_f32(dh_last)),
                                *[out[k].ctypes.data for k in ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dD",
                                                               "ddelta_bias", "dh0")])
    if rc != 0:
        raise ValueError("oracle scan_bwd rejected its arguments")
    return out

