"""GPU parity of the causal depthwise convolution front-end (ss_conv1d_fwd) and
its decode step (ss_conv1d_update) against the float64 oracle, through the C
ABI: every output compared, ragged shapes on both the vector and the scalar
path, widths 2-4, carried state in and out."""

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_130_b300 as ss
from parity import assert_close
from workloads import gen

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def _dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _run(x, out_dtype, silu=True):
    d = _dev(x)
    y, so = ss.ss_conv1d_fwd(d["x"], d["weight"], d.get("bias"), d.get("state"), silu=silu, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y, so


# (in_dtype, batch, L, D): D*elem a multiple of 16 bytes takes the vector path
SHAPES = [("bf16", 2, 17, 40), ("f32", 2, 17, 40), ("bf16", 1, 33, 5), ("f32", 3, 100, 7), ("bf16", 3, 100, 264),
          ("bf16", 2, 2, 16), ("f32", 1, 1, 4), ("bf16", 1, 64, 24)]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}-b{s[1]}-L{s[2]}-D{s[3]}" for s in SHAPES])
@pytest.mark.parametrize("width", [2, 3, 4])
@pytest.mark.parametrize("state", [False, True])
def test_conv1d_matches_oracle(shape, width, state):
    dt, Bt, L, Dm = shape
    in_dt = BF16 if dt == "bf16" else F32
    x = gen.random_conv_inputs(Bt, L, Dm, width, dt, seed=L * 7 + Dm + width, with_state=state, has_bias=(L % 2 == 1))
    for silu in (True, False):
        yr, sr = oracle.conv1d(x, silu=silu)
        for out in (F32, BF16):
            y, so = _run(x, out, silu)
            assert_close(y.double().cpu().numpy(), yr, in_dt, out_bf16=(out == BF16), what=f"conv y silu={silu}")
            # the carried state is a copy of stored inputs: exact
            assert np.array_equal(so.double().cpu().numpy(), sr), "conv state_out"


def test_conv1d_chunk_continuity_on_gpu():
    # two calls chained through the carried state give the one-call result bit for bit
    x = gen.random_conv_inputs(2, 300, 96, 4, "bf16", seed=3, with_state=True)
    y, so = _run(x, F32)
    for m in (1, 16, 17, 150):
        a = dict(x, x=x["x"][:, :m].contiguous())
        ya, sa = _run(a, F32)
        b = dict(x, x=x["x"][:, m:].contiguous(), state=sa.cpu())
        yb, sb = _run(b, F32)
        assert torch.equal(torch.cat([ya, yb], dim=1), y)
        assert torch.equal(sb, so)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("width", [2, 4])
def test_conv1d_update_matches_oracle_and_forward(dt, width):
    Bt, L, Dm = 3, 20, 45
    in_dt = BF16 if dt == "bf16" else F32
    x = gen.random_conv_inputs(Bt, L, Dm, width, dt, seed=9, with_state=True)
    yf, sf = _run(x, F32)
    st_ref = x["state"].double().numpy().copy()
    d = _dev(x)
    st = d["state"].clone()
    for t in range(L):
        xt = d["x"][:, t].contiguous()
        yt = ss.ss_conv1d_update(st, xt, d["weight"], d["bias"], out_dtype=F32)
        yr = oracle.conv1d_update(st_ref, x["x"][:, t].contiguous(), x["weight"], x["bias"])
        assert_close(yt.double().cpu().numpy(), yr, in_dt, what=f"conv decode y step {t}")
        assert torch.allclose(yt, yf[:, t], rtol=0, atol=1e-6 * float(yf.abs().max()))
    torch.cuda.synchronize()
    assert np.array_equal(st.double().cpu().numpy(), st_ref)
    assert torch.equal(st, sf)


def test_conv1d_full_layer_shape():
    # the Mamba-2.8B-shaped layer (4 x 2048 x 5120, bf16 in and out, width 4), every output
    x = gen.random_conv_inputs(4, 2048, 5120, 4, "bf16", seed=2, with_state=False)
    yr, sr = oracle.conv1d(x)
    y, so = _run(x, BF16)
    assert_close(y.double().cpu().numpy(), yr, BF16, out_bf16=True, what="layer conv y")
    assert np.array_equal(so.double().cpu().numpy(), sr)


@pytest.mark.parametrize("dt,width", [("bf16", 4), ("f32", 3)])
def test_conv1d_ranges_cross_blocks(dt, width):
    # 3 x 4000 x 1288: 63 tiles of 64 steps (the last 32 rows), 11 or 21
    # channel blocks (the last partial), so each CTA's range of about five
    # units crosses batch elements and channel blocks; carried state in and
    # out, y in x's type (staged in shared memory, one bulk store per tile)
    # and in the other type (stored from registers)
    in_dt = BF16 if dt == "bf16" else F32
    x = gen.random_conv_inputs(3, 4000, 1288, width, dt, seed=11, with_state=True)
    yr, sr = oracle.conv1d(x)
    for out in (in_dt, F32 if in_dt == BF16 else BF16):
        y, so = _run(x, out)
        assert_close(y.double().cpu().numpy(), yr, in_dt, out_bf16=(out == BF16), what=f"conv y out={out}")
        assert np.array_equal(so.double().cpu().numpy(), sr)


def test_conv1d_empty_and_errors():
    x = gen.random_conv_inputs(2, 3, 16, 4, "bf16", seed=1, with_state=True)
    d = _dev(x)
    so = torch.full((2, 16, 3), 7.0, dtype=BF16, device="cuda")
    ss.ss_conv1d_fwd(d["x"][:, :0].contiguous(), d["weight"], d["bias"], d["state"], y=torch.empty(2, 0, 16, device="cuda",
                     dtype=BF16), state_out=so)
    torch.cuda.synchronize()
    assert torch.equal(so, d["state"])  # L = 0: the state passes through
    with pytest.raises(ss.SSError) as ei:
        ss.ss_conv1d_fwd(d["x"], d["weight"], d["bias"], d["state"], state_out=d["state"])
    assert ei.value.status == ss._lib.SS_ERR_INVALID_ARG
    w5 = torch.zeros(16, 5, device="cuda")
    with pytest.raises(ss.SSError) as ei:
        ss.ss_conv1d_fwd(d["x"], w5)
    assert ei.value.status == ss._lib.SS_ERR_UNSUPPORTED
