"""Seeded generation of host (CPU) input tensors.

Every tensor is drawn from torch's CPU generator in fixed-size blocks; block k
of stream s under seed `seed` uses its own generator seeded from (seed, s, k),
so the values do not depend on the thread count and any block can be drawn on
its own. Values are drawn in float64/float32 and rounded once to the storage
dtype (bf16 by round-to-nearest-even via torch). Both the oracle and the GPU
path receive exactly these stored values.
"""

import math
import os
from concurrent.futures import ThreadPoolExecutor

import torch

from .configs import ScanWorkload, DecodeWorkload

BLOCK = 1 << 22

# stream ids (one per drawn tensor)
S_DT, S_ALOG, S_U, S_DRAW, S_Z, S_B, S_C, S_SYM, S_EMB = range(9)
S_CX, S_CW, S_CB, S_CS = range(9, 13)  # convolution front-end: input, weights, bias, state
S_DY, S_DH = range(13, 15)  # backward pass: gradients of y and of h_last


def _block_seed(seed: int, stream: int, block: int) -> int:
    return (seed * 1_000_003 + stream * 10_007 + block * 7_919 + 12_345) % (1 << 62)


def randn_blocks(numel: int, seed: int, stream: int, threads: int = 0) -> torch.Tensor:
    """numel standard-normal float32 values, drawn block by block."""
    out = torch.empty(numel, dtype=torch.float32)
    nblk = (numel + BLOCK - 1) // BLOCK

    def fill(k):
        g = torch.Generator().manual_seed(_block_seed(seed, stream, k))
        lo, hi = k * BLOCK, min(numel, (k + 1) * BLOCK)
        out[lo:hi] = torch.randn(hi - lo, generator=g, dtype=torch.float32)

    if nblk <= 1:
        for k in range(nblk):
            fill(k)
    else:
        n = threads or min(32, os.cpu_count() or 1)
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def _store(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x.to(torch.float32)
    raise ValueError(dtype)


def make_params(w: ScanWorkload):
    """Per-layer fp32 parameters A [D,N], D_skip [D], delta_bias [D].

    dt_d is log-uniform in [dt_min, dt_max]; delta_bias = softplus^{-1}(dt_d)
    = log(expm1(dt_d)); A_log[d, n] = log(n+1) (+ jitter); A = -exp(A_log),
    rounded once to fp32.
    """
    D, N = w.dim, w.dstate
    g = torch.Generator().manual_seed(_block_seed(w.seed, S_DT, 0))
    r = torch.rand(D, generator=g, dtype=torch.float64)
    dt = torch.exp(math.log(w.dt_min) + r * (math.log(w.dt_max) - math.log(w.dt_min)))
    bias = torch.log(torch.expm1(dt)).to(torch.float32)
    a_log = torch.log(torch.arange(1, N + 1, dtype=torch.float64)).expand(D, N).clone()
    if w.a_log_jitter:
        g2 = torch.Generator().manual_seed(_block_seed(w.seed, S_ALOG, 0))
        a_log += w.a_log_jitter * torch.randn(D, N, generator=g2, dtype=torch.float64)
    A = (-torch.exp(a_log)).to(torch.float32).contiguous()
    Dskip = torch.ones(D, dtype=torch.float32)
    return A, Dskip, bias


def make_scan_inputs(w: ScanWorkload, seed: int = None) -> dict:
    """Host tensors for one ss_scan_fwd call (contiguous, row-major):
    u, delta_raw, z: [Bt, L, D]; B, C: [Bt, L, N] in w.in_dtype;
    A: [D, N], D: [D], delta_bias: [D] float32."""
    s = w.seed if seed is None else seed
    Bt, L, D, N = w.batch, w.seqlen, w.dim, w.dstate
    A, Dskip, bias = make_params(w)
    n_td = Bt * L * D
    if w.u_kind == "normal":
        u = randn_blocks(n_td, s, S_U).view(Bt, L, D)
    elif w.u_kind == "alphabet4":
        g = torch.Generator().manual_seed(_block_seed(s, S_EMB, 0))
        emb = torch.randn(4, D, generator=g, dtype=torch.float32)
        g2 = torch.Generator().manual_seed(_block_seed(s, S_SYM, 0))
        sym = torch.randint(0, 4, (Bt, L), generator=g2)
        u = emb[sym]  # [Bt, L, D]
    else:
        raise ValueError(w.u_kind)
    out = {
        "u": _store(u, w.in_dtype).contiguous(),
        "delta_raw": _store(w.delta_raw_scale * randn_blocks(n_td, s, S_DRAW).view(Bt, L, D),
                            w.in_dtype).contiguous(),
        "z": _store(randn_blocks(n_td, s, S_Z).view(Bt, L, D), w.in_dtype).contiguous() if w.has_z else None,
        "B": _store(randn_blocks(Bt * L * N, s, S_B).view(Bt, L, N), w.in_dtype).contiguous(),
        "C": _store(randn_blocks(Bt * L * N, s, S_C).view(Bt, L, N), w.in_dtype).contiguous(),
        "A": A,
        "D": Dskip if w.has_d else None,
        "delta_bias": bias,
    }
    return out


def make_decode_steps(w: DecodeWorkload, first: int, count: int, threads: int = 0) -> dict:
    """Inputs of decode steps [first, first+count): u, delta_raw, z [count, S, D],
    B, C [count, S, N] in w.in_dtype. Step k draws from its own streams, so any
    range of steps can be generated alone."""
    S, D, N = w.streams, w.dim, w.dstate
    td = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    out = {
        "u": torch.empty(count, S, D, dtype=td), "delta_raw": torch.empty(count, S, D, dtype=td),
        "z": torch.empty(count, S, D, dtype=td), "B": torch.empty(count, S, N, dtype=td),
        "C": torch.empty(count, S, N, dtype=td),
    }

    def fill(i):
        sk = w.seed * 100_003 + first + i
        out["u"][i] = _store(randn_blocks(S * D, sk, S_U, threads=1).view(S, D), w.in_dtype)
        out["delta_raw"][i] = _store(w.delta_raw_scale * randn_blocks(S * D, sk, S_DRAW, threads=1).view(S, D),
                                     w.in_dtype)
        out["z"][i] = _store(randn_blocks(S * D, sk, S_Z, threads=1).view(S, D), w.in_dtype)
        out["B"][i] = _store(randn_blocks(S * N, sk, S_B, threads=1).view(S, N), w.in_dtype)
        out["C"][i] = _store(randn_blocks(S * N, sk, S_C, threads=1).view(S, N), w.in_dtype)

    n = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(n) as ex:
        list(ex.map(fill, range(count)))
    return out


def random_scan_inputs(batch, seqlen, dim, dstate, in_dtype="f32", seed=0, delta_raw_scale=0.5,
                       a_log_jitter=0.0, has_z=True, has_d=True, with_h0=False, dt_min=1e-3, dt_max=1e-1):
    """Small ad-hoc problems (edge shapes for tests) with the c0 recipe."""
    w = ScanWorkload("adhoc", batch, seqlen, dim, dstate, in_dtype, seed, delta_raw_scale,
                     a_log_jitter, has_z=has_z, has_d=has_d, dt_min=dt_min, dt_max=dt_max)
    x = make_scan_inputs(w)
    if with_h0:
        x["h0"] = randn_blocks(batch * dim * dstate, seed, 99).view(batch, dim, dstate).contiguous()
    else:
        x["h0"] = None
    return x


S_SYMTAB = 15  # symbol-table inputs: stream S_SYMTAB + 2 i (table) and + 2 i + 1 (symbols) for tensor i


def symbol_tensor(index_shape, row_shape, seed, slot, nsym=16, dtype="bf16", scale=1.0):
    """A tensor too large to draw value by value, as a table and its symbols:
    table [nsym, *row_shape] ~ scale * N(0,1) in `dtype`, symbols [*index_shape]
    uniform over {0 .. nsym-1}; the tensor is gather_symbols(table, symbols)
    [*index_shape, *row_shape]. `slot` picks the tensor's pair of streams."""
    rows = 1
    for r in row_shape:
        rows *= r
    table = _store(scale * randn_blocks(nsym * rows, seed, S_SYMTAB + 2 * slot).view(nsym, *row_shape), dtype)
    g = torch.Generator().manual_seed(_block_seed(seed, S_SYMTAB + 2 * slot + 1, 0))
    symbols = torch.randint(0, nsym, tuple(index_shape), generator=g)
    return table.contiguous(), symbols


def symbol_scan_inputs(batch, seqlen, dim, dstate=16, nsym=16, seed=5):
    """Inputs too large to draw value by value (more than 2^32 elements per
    [batch, seqlen, dim] tensor), in the style of the DNA workload's alphabet:
    u, delta_raw and z are each a table of `nsym` rows ~ N(0,1) over the
    channels, bf16, indexed by a symbol per (b, t) (symbol_tensor). B and C
    [batch, seqlen, dstate] ~ N(0,1) bf16 are drawn in full. A, D and
    delta_bias follow the layer recipe (A_log = log(n + 1), dt log-uniform in
    [1e-3, 1e-1]). Returns {"tables": {k: [nsym, dim]}, "symbols": {k: [batch,
    seqlen] int64} for k in u, delta_raw, z; "B", "C", "A", "D", "delta_bias"}."""
    w = ScanWorkload("symbols", batch, seqlen, dim, dstate, "bf16", seed, 1.0, 0.0)
    A, Dskip, bias = make_params(w)
    tables, symbols = {}, {}
    for i, k in enumerate(("u", "delta_raw", "z")):
        tables[k], symbols[k] = symbol_tensor((batch, seqlen), (dim,), seed, i, nsym)
    n = batch * seqlen * dstate
    return {
        "tables": tables,
        "symbols": symbols,
        "B": _store(randn_blocks(n, seed, S_B).view(batch, seqlen, dstate), "bf16").contiguous(),
        "C": _store(randn_blocks(n, seed, S_C).view(batch, seqlen, dstate), "bf16").contiguous(),
        "A": A,
        "D": Dskip,
        "delta_bias": bias,
    }


def gather_symbols(table: torch.Tensor, symbols: torch.Tensor) -> torch.Tensor:
    """table[symbols]: [*symbols.shape, table.shape[1]], contiguous, on the
    tensors' device (a plain index copy, no arithmetic on the values)."""
    return table[symbols].contiguous()


def random_conv_inputs(batch, seqlen, dim, width, in_dtype="bf16", seed=0, with_state=False, has_bias=True):
    """Inputs of the causal depthwise convolution front-end:
    x [batch, seqlen, dim] ~ N(0,1) in `in_dtype`; weight [dim, width] ~
    0.5 N(0,1) and bias [dim] ~ 0.1 N(0,1) in fp32; state [batch, dim, width-1]
    ~ N(0,1) in `in_dtype` (the inputs before t = 0) or None."""
    out = {
        "x": _store(randn_blocks(batch * seqlen * dim, seed, S_CX).view(batch, seqlen, dim), in_dtype).contiguous(),
        "weight": (0.5 * randn_blocks(dim * width, seed, S_CW)).view(dim, width).contiguous(),
        "bias": (0.1 * randn_blocks(dim, seed, S_CB)).contiguous() if has_bias else None,
        "state": None,
    }
    if with_state and width > 1:
        out["state"] = _store(randn_blocks(batch * dim * (width - 1), seed, S_CS).view(batch, dim, width - 1),
                              in_dtype).contiguous()
    return out



def random_output_grads(batch, seqlen, dim, dstate, dy_dtype="f32", seed=0, with_dh_last=True, channels=None,
                        threads: int = 0):
    """Gradients arriving at the scan's outputs, for the backward pass: dy
    [batch, seqlen, dim] in dy_dtype and dh_last [batch, dim, dstate] float32
    (None unless with_dh_last), standard normal. `channels`, a list of channel
    indices, keeps only those channels nonzero (the rest exactly 0)."""
    dy = randn_blocks(batch * seqlen * dim, seed, S_DY, threads).view(batch, seqlen, dim)
    dh = randn_blocks(batch * dim * dstate, seed, S_DH, threads).view(batch, dim, dstate) if with_dh_last else None
    if channels is not None:
        keep = torch.zeros(dim, dtype=torch.bool)
        keep[torch.as_tensor(channels, dtype=torch.long)] = True
        dy = dy * keep.to(dy.dtype)
        if dh is not None:
            dh = dh * keep.to(dh.dtype)[:, None]
    return _store(dy, dy_dtype).contiguous(), (dh.contiguous() if dh is not None else None)


def random_general_inputs(batch, seqlen, dim, dstate, ngroups=1, in_dtype="f32", seed=0, with_h0=False,
                          threads: int = 0, **kw):
    """Inputs of the generalised scan: as random_scan_inputs (A_log = log(n+1)
    for n < dstate), with B and C [batch, seqlen, ngroups, dstate] (standard
    normal, the same streams as B and C of the shared case)."""
    x = random_scan_inputs(batch, seqlen, dim, dstate, in_dtype=in_dtype, seed=seed, with_h0=with_h0, **kw)
    n = batch * seqlen * ngroups * dstate
    x["B"] = _store(randn_blocks(n, seed, S_B, threads).view(batch, seqlen, ngroups, dstate), in_dtype).contiguous()
    x["C"] = _store(randn_blocks(n, seed, S_C, threads).view(batch, seqlen, ngroups, dstate), in_dtype).contiguous()
    return x


def random_ssd_inputs(batch, seqlen, nheads, headdim, dstate, ngroups=1, in_dtype="bf16", seed=0, with_h0=False,
                      threads: int = 0):
    """Inputs of the state-space-dual (Mamba-2) layer: x [batch, L, H, P], dt
    [batch, L, H] (0.5 N(0,1)), B, C [batch, L, G, N] (N(0,1)) in in_dtype; A [H]
    = -U(1, 16) per head, D [H] = 1, dt_bias [H] = log(expm1(dt0)) with dt0 =
    exp(U(log 1e-3, log 0.1)) (float32); h0 [batch, H, P, N] or None."""
    n = batch * seqlen * nheads * headdim
    x = randn_blocks(n, seed, S_U, threads).view(batch, seqlen, nheads, headdim)
    dt = 0.5 * randn_blocks(batch * seqlen * nheads, seed, S_DRAW, threads).view(batch, seqlen, nheads)
    nb = batch * seqlen * ngroups * dstate
    B = randn_blocks(nb, seed, S_B, threads).view(batch, seqlen, ngroups, dstate)
    C = randn_blocks(nb, seed, S_C, threads).view(batch, seqlen, ngroups, dstate)
    g = torch.Generator().manual_seed(_block_seed(seed, S_ALOG, 0))
    A = -(1.0 + 15.0 * torch.rand(nheads, generator=g, dtype=torch.float64)).float()
    g = torch.Generator().manual_seed(_block_seed(seed, S_DT, 0))
    dt0 = torch.exp(math.log(1e-3) + (math.log(0.1) - math.log(1e-3)) * torch.rand(nheads, generator=g,
                                                                                   dtype=torch.float64))
    out = {"x": _store(x, in_dtype).contiguous(), "dt": _store(dt, in_dtype).contiguous(),
           "B": _store(B, in_dtype).contiguous(), "C": _store(C, in_dtype).contiguous(),
           "A": A.contiguous(), "D": torch.ones(nheads, dtype=torch.float32),
           "dt_bias": torch.log(torch.expm1(dt0)).float().contiguous()}
    out["h0"] = (randn_blocks(batch * nheads * headdim * dstate, seed, 99, threads)
                 .view(batch, nheads, headdim, dstate).contiguous() if with_h0 else None)
    return out
