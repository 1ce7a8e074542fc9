"""ctypes binding of libssscan.so.

Argument marshalling only: every step of the scan and the decode step runs in
the library's sm_103a kernels. PyTorch provides device memory and streams.
The binding refuses to work without the compiled library (no fallback).
"""

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libssscan.so")

SS_OK, SS_ERR_INVALID_ARG, SS_ERR_UNSUPPORTED, SS_ERR_CUDA, SS_ERR_TIMEOUT = range(5)
SS_F32, SS_BF16 = 0, 1
SS_DISC_FIRST_ORDER, SS_DISC_ZOH = 0, 1
DISC = {"first_order": SS_DISC_FIRST_ORDER, "euler": SS_DISC_FIRST_ORDER, "zoh": SS_DISC_ZOH}
# bytes of the fixed scratch array behind ss_scan_fwd_noalloc (SS_SCAN_NOALLOC_SCRATCH_BYTES in the header)
SS_SCAN_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
STATUS_NAMES = {0: "SS_OK", 1: "SS_ERR_INVALID_ARG", 2: "SS_ERR_UNSUPPORTED", 3: "SS_ERR_CUDA",
                4: "SS_ERR_TIMEOUT"}

# Every function the C header declares, with its ctypes signature.
_I64, _P, _SZ = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
SIGNATURES = {
    "ss_version": (ctypes.c_int, []),
    "ss_last_error": (ctypes.c_char_p, []),
    "ss_scan_fwd_workspace_size": (_SZ, [_I64, _I64, _I64, _I64]),
    "ss_scan_fwd": (ctypes.c_int, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                   _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "ss_state_update": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                       _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ss_scan_fwd_noalloc": (ctypes.c_int, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                           _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "ss_conv1d_fwd": (ctypes.c_int, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                     _P, _P, _P, _P, ctypes.c_int, _P, _P, _P]),
    "ss_conv1d_update": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                        _P, _P, _P, _P, ctypes.c_int, _P, _P]),
    "ss_scan_bwd_workspace_size": (_SZ, [_I64, _I64, _I64, _I64]),
    "ss_scan_bwd": (ctypes.c_int, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int] + [_P] * 21 + [_SZ, _P]),
    "ss_scan_fwd_general": (ctypes.c_int, [_I64, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
                            + [_P] * 12 + [ctypes.c_size_t, _P]),
    "ss_scan_fwd_general_workspace_size": (ctypes.c_size_t, [_I64] * 5 + [ctypes.c_int, ctypes.c_int]),
    "ss_ssd_fwd": (ctypes.c_int, [_I64] * 6 + [ctypes.c_int, ctypes.c_int] + [_P] * 11 + [ctypes.c_size_t, _P]),
    "ss_ssd_fwd_workspace_size": (ctypes.c_size_t, [_I64] * 4),
    "ss_scan_set_tuning": (None, [ctypes.c_int, _I64, ctypes.c_int]),
    "ss_scan_set_wait_limit": (None, [ctypes.c_uint64, _I64]),
    "ss_scan_status": (ctypes.c_int, [_P, _P]),
}


class SSError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib(path: str = None) -> ctypes.CDLL:
    """The loaded library (built by selective_state_space_130_b300/build.py)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libssscan.so not found at {p}; build it with "
                          "`python selective_state_space_130_b300/build.py` (nvcc, sm_103a)")
    L = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = L
    return L


def _check(status):
    if status != SS_OK:
        raise SSError(status, lib().ss_last_error().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SS_F32
    if t.dtype == torch.bfloat16:
        return SS_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _tdt(code: int):
    return torch.bfloat16 if code == SS_BF16 else torch.float32


def _out_code(in_code, out_dtype, y):
    """Output dtype code: out_dtype if given, else that of a given y, else the
    input dtype. A given y must have the output dtype."""
    if out_dtype is not None:
        code = _dt(torch.empty(0, dtype=out_dtype))
    elif y is not None:
        code = _dt(y)
    else:
        code = in_code
    if y is not None and _dt(y) != code:
        raise TypeError(f"y has dtype {y.dtype}, the output dtype is {_tdt(code)}")
    return code


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def ss_version() -> int:
    return lib().ss_version()


def ss_last_error() -> str:
    return lib().ss_last_error().decode()


def ss_scan_set_tuning(threads_per_channel: int = 0, chunk_len: int = 0, max_workers: int = 0):
    lib().ss_scan_set_tuning(int(threads_per_channel), int(chunk_len), int(max_workers))


def ss_scan_set_wait_limit(wait_ns: int = 0, withhold_item: int = -1):
    lib().ss_scan_set_wait_limit(int(wait_ns), int(withhold_item))


def ss_scan_fwd_workspace_size(batch, seqlen, dim, dstate=16) -> int:
    return int(lib().ss_scan_fwd_workspace_size(batch, seqlen, dim, dstate))


def ss_scan_fwd(u, delta_raw, A, B, C, D=None, z=None, delta_bias=None, h0=None, *, out_dtype=None,
                y=None, h_last=None, workspace=None, return_h_last=True, stream=None):
    """Selective scan forward on device tensors.

    u, delta_raw, z: [Bt, L, D]; B, C: [Bt, L, N] (float32 or bfloat16, one dtype);
    A: [D, N], D, delta_bias: [D], h0: [Bt, D, N] float32. Returns (y, h_last);
    outputs and workspace are allocated with torch when not given.
    """
    Bt, L, Dm = u.shape
    N = B.shape[-1]
    code = _dt(u)
    out_code = _out_code(code, out_dtype, y)
    dev = u.device
    if y is None:
        y = torch.empty((Bt, L, Dm), dtype=_tdt(out_code), device=dev)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
    ws_bytes = ss_scan_fwd_workspace_size(Bt, L, Dm, N)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().ss_scan_fwd(Bt, L, Dm, N, code, out_code, _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(y), _ptr(h_last),
                             ws_ptr, ws_len, _stream(stream)))
    return y, h_last


def ss_scan_bwd_workspace_size(batch, seqlen, dim, dstate=16) -> int:
    return int(lib().ss_scan_bwd_workspace_size(batch, seqlen, dim, dstate))


def ss_scan_bwd(u, delta_raw, A, B, C, dy, D=None, z=None, delta_bias=None, h0=None, dh_last=None, *,
                out=None, workspace=None, stream=None) -> dict:
    """Gradients of the selective scan on device tensors.

    Inputs as for ss_scan_fwd, plus dy [Bt, L, D] (float32 or bfloat16) and
    dh_last [Bt, D, N] float32 or None. Returns a dict: du, ddelta_raw, dz (None
    without z) in the input dtype; dA [D, N], dB, dC [Bt, L, N], dD,
    ddelta_bias [D], dh0 [Bt, D, N] in float32. Tensors missing from `out` (and
    the workspace) are allocated with torch.
    """
    Bt, L, Dm = u.shape
    N = B.shape[-1]
    code = _dt(u)
    dev = u.device
    o = dict(out or {})
    shapes = {"du": ((Bt, L, Dm), u.dtype), "ddelta_raw": ((Bt, L, Dm), u.dtype), "dA": ((Dm, N), torch.float32),
              "dB": ((Bt, L, N), torch.float32), "dC": ((Bt, L, N), torch.float32), "dD": ((Dm,), torch.float32),
              "ddelta_bias": ((Dm,), torch.float32), "dh0": ((Bt, Dm, N), torch.float32)}
    if z is not None:
        shapes["dz"] = ((Bt, L, Dm), u.dtype)
    for k, (sh, dt) in shapes.items():
        if k not in o:
            o[k] = torch.empty(sh, dtype=dt, device=dev)
    o.setdefault("dz", None)
    ws_bytes = ss_scan_bwd_workspace_size(Bt, L, Dm, N)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().ss_scan_bwd(Bt, L, Dm, N, code, _dt(dy), _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(dy), _ptr(dh_last),
                             *[_ptr(o[k]) for k in ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dD", "ddelta_bias",
                                                    "dh0")],
                             ws_ptr, ws_len, _stream(stream)))
    return o


def ss_scan_fwd_general_workspace_size(batch, seqlen, dim, dstate, ngroups=1, disc="first_order",
                                       in_dtype=torch.bfloat16):
    code = SS_BF16 if in_dtype == torch.bfloat16 else SS_F32
    return int(lib().ss_scan_fwd_general_workspace_size(batch, seqlen, dim, dstate, ngroups, DISC[disc], code))


def ss_scan_fwd_general(u, delta_raw, A, B, C, D=None, z=None, delta_bias=None, h0=None, *, disc="first_order",
                        out_dtype=None, y=None, h_last=None, workspace=None, return_h_last=True, stream=None):
    """Generalised selective scan on device tensors: dstate = A.shape[1] (16, 32,
    64 or 128); B, C [Bt, L, G, N] (or [Bt, L, N] for G = 1); disc
    "first_order" (Bbar = delta B) or "zoh". Returns (y, h_last). The workspace
    (uint8) is allocated with torch when the problem can use one and none is
    given; workspace=False runs without one."""
    Bt, L, Dm = u.shape
    N = A.shape[1]
    G = 1 if B.dim() == 3 else B.shape[2]
    code = _dt(u)
    out_code = _out_code(code, out_dtype, y)
    dev = u.device
    if y is None:
        y = torch.empty((Bt, L, Dm), dtype=_tdt(out_code), device=dev)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
    if workspace is None:
        ws_bytes = ss_scan_fwd_general_workspace_size(Bt, L, Dm, N, G, disc, u.dtype)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else False
    ws_ptr = _ptr(workspace) if workspace is not False else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not False else 0
    _check(lib().ss_scan_fwd_general(Bt, L, Dm, N, G, DISC[disc], code, out_code, _ptr(u), _ptr(delta_raw), _ptr(A),
                                     _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(y),
                                     _ptr(h_last), ws_ptr, ws_len, _stream(stream)))
    return y, h_last


def ss_ssd_fwd_workspace_size(batch, seqlen, nheads, dstate):
    return int(lib().ss_ssd_fwd_workspace_size(batch, seqlen, nheads, dstate))


def ss_ssd_fwd(x, dt, A, B, C, D=None, dt_bias=None, h0=None, *, out_dtype=None, y=None, h_last=None,
               workspace=None, return_h_last=True, stream=None):
    """State-space-dual (Mamba-2) layer on device tensors: x [Bt, L, H, 64], dt
    [Bt, L, H], B, C [Bt, L, G, N] (bf16); A, D, dt_bias [H]; h0 [Bt, H, 64, N]
    float32. Returns (y, h_last). The workspace (uint8) is allocated with torch
    when the problem can use one and none is given; workspace=False runs
    without one."""
    Bt, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    code = _dt(x)
    out_code = _out_code(code, out_dtype, y)
    dev = x.device
    if y is None:
        y = torch.empty((Bt, L, H, P), dtype=_tdt(out_code), device=dev)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bt, H, P, N), dtype=torch.float32, device=dev)
    if workspace is None:
        ws_bytes = ss_ssd_fwd_workspace_size(Bt, L, H, N)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else False
    ws_ptr = _ptr(workspace) if workspace is not False else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not False else 0
    _check(lib().ss_ssd_fwd(Bt, L, H, P, N, G, code, out_code, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                            _ptr(dt_bias), _ptr(h0), _ptr(y), _ptr(h_last), ws_ptr, ws_len, _stream(stream)))
    return y, h_last


def ss_state_update(h, u, delta_raw, A, B, C, D=None, z=None, delta_bias=None, *, out_dtype=None, y=None,
                    stream=None):
    """One decode step on device tensors; h [S, D, N] float32 is updated in place.
    u, delta_raw, z: [S, D]; B, C: [S, N]. Returns y [S, D]."""
    S, Dm = u.shape
    N = B.shape[-1]
    code = _dt(u)
    out_code = _out_code(code, out_dtype, y)
    if y is None:
        y = torch.empty((S, Dm), dtype=_tdt(out_code), device=u.device)
    _check(lib().ss_state_update(S, Dm, N, code, out_code, _ptr(h), _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(B),
                                 _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(y), _stream(stream)))
    return y


def ss_scan_status(workspace=None, stream=None):
    """Raise SSError if a device-side wait of an earlier scan gave up."""
    _check(lib().ss_scan_status(_ptr(workspace) if workspace is not None else None, _stream(stream)))


def ss_scan_fwd_noalloc(u, delta_raw, A, B, C, D=None, z=None, delta_bias=None, h0=None, *, out_dtype=None,
                        y=None, h_last=None, return_h_last=True, stream=None):
    """Selective scan forward through the entry point that allocates nothing on
    the library side: its cross-block scratch is a fixed array inside the
    library (SS_SCAN_NOALLOC_SCRATCH_BYTES per device). Same arguments and
    results as ss_scan_fwd, without a workspace; outputs are allocated with
    torch here only when not given. Calls that overlap on the GPU race on the
    shared scratch."""
    Bt, L, Dm = u.shape
    N = B.shape[-1]
    code = _dt(u)
    out_code = _out_code(code, out_dtype, y)
    dev = u.device
    if y is None:
        y = torch.empty((Bt, L, Dm), dtype=_tdt(out_code), device=dev)
    if h_last is None and return_h_last:
        h_last = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
    _check(lib().ss_scan_fwd_noalloc(Bt, L, Dm, N, code, out_code, _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(B),
                                     _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(y), _ptr(h_last),
                                     _stream(stream)))
    return y, h_last


def ss_conv1d_fwd(x, weight, bias=None, state=None, *, silu=True, out_dtype=None, y=None, state_out=None,
                  return_state=True, stream=None):
    """Causal depthwise convolution front-end on device tensors.
    x: [Bt, L, D] (float32 or bfloat16); weight: [D, K] float32; bias: [D] float32;
    state: [Bt, D, K-1] in x's dtype (the inputs before t = 0) or None.
    Returns (y [Bt, L, D], state_out [Bt, D, K-1]); outputs are allocated with torch when not given."""
    Bt, L, Dm = x.shape
    K = weight.shape[1]
    code = _dt(x)
    out_code = _out_code(code, out_dtype, y)
    if y is None:
        y = torch.empty((Bt, L, Dm), dtype=_tdt(out_code), device=x.device)
    if state_out is None and return_state:
        state_out = torch.empty((Bt, Dm, K - 1), dtype=x.dtype, device=x.device)
    _check(lib().ss_conv1d_fwd(Bt, L, Dm, K, code, out_code, _ptr(x), _ptr(weight), _ptr(bias), _ptr(state),
                               int(bool(silu)), _ptr(y), _ptr(state_out), _stream(stream)))
    return y, state_out


def ss_conv1d_update(state, x, weight, bias=None, *, silu=True, out_dtype=None, y=None, stream=None):
    """One decode step of the convolution; state [S, D, K-1] (x's dtype) is updated
    in place with x [S, D]. Returns y [S, D]."""
    S, Dm = x.shape
    K = weight.shape[1]
    code = _dt(x)
    out_code = _out_code(code, out_dtype, y)
    if y is None:
        y = torch.empty((S, Dm), dtype=_tdt(out_code), device=x.device)
    _check(lib().ss_conv1d_update(S, Dm, K, code, out_code, _ptr(state), _ptr(x), _ptr(weight), _ptr(bias),
                                  int(bool(silu)), _ptr(y), _stream(stream)))
    return y

