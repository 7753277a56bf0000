"""Kernel-level parity: each C-ABI call against the oracle on seeded inputs.

Shapes span several tiles / vectors plus ragged tails and the degenerate cases (one row, empty
input).  Inputs come from ``workloads.random_tensor``; nothing the oracle reads comes from the
CUDA path.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import block as ob
from oracle import numerics as nx
from parity import (ACC_REL, Guarded, assert_e4m3_codes, assert_elementwise_close,
                    assert_gemm_close, assert_reduction_close, codes, np64, rms)
from steps import check_norm_dx, check_norm_params
from workloads import random_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"
TDT = {"bf16": torch.bfloat16, "f32": torch.float32}


def rt(shape, std=1.0, seed=0, dtype="bf16", mean=0.0):
    return random_tensor(shape, std=std, device=DEV, seed=seed, dtype=dtype, mean=mean)


# ------------------------------------------------------------------ quantize ---------------


@pytest.mark.parametrize("M,N", [(1, 8), (37, 264), (1024, 4096)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["delayed", "current"])
def test_quantize_bit_exact(M, N, dtype, mode):
    x = rt((M, N), std=3.0, seed=M + N, dtype=dtype)
    q = te.Quantizer(scale=17.0, mode=mode)
    gout = Guarded((M, N), torch.uint8)
    out = gout.t
    te.te_quantize(x, q, out)
    gout.check("quantize")
    xv = np64(x)
    amax = nx.amax_of(xv)
    assert q.amax.item() == amax  # order-free max: bit-exact
    scale = np.float32(17.0) if mode == "delayed" else nx.compute_scale(amax)[0]
    assert q.scale.item() == scale
    assert q.scale_inv.item() == np.float32(1.0) / scale
    assert_e4m3_codes(out, nx.quantize(xv, scale), what="quantize")


def test_quantize_saturates_and_keeps_sign():
    x = torch.tensor([[1000.0, -1000.0, 0.0, -0.0, 448.0, 464.0, 1e-3, -1e-3]], device=DEV)
    q = te.Quantizer(scale=1.0)
    out = torch.empty(1, 8, dtype=torch.uint8, device=DEV)
    te.te_quantize(x, q, out)
    assert_e4m3_codes(out, nx.quantize(np64(x), np.float32(1.0)), what="saturate")


def _nan_code(c):
    return (np.asarray(c) & 0x7F) == 0x7F


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["delayed", "current"])
def test_quantize_nan_inf(dtype, mode):
    """NaN encodes as an E4M3 NaN code (either sign) and is ignored by the amax; +-inf
    saturates to +-448 and makes the amax infinite, which current scaling turns into scale 1."""
    vals = [float("nan"), float("inf"), float("-inf"), 0.0, -0.0, 1.5, -3.25, 1000.0,
            -1000.0, 2.0 ** -10, float("nan"), 7.0, -0.5, 0.25, 448.0, -464.0]
    x = torch.tensor([vals], dtype=TDT[dtype], device=DEV)
    q = te.Quantizer(scale=2.0, mode=mode)
    out = torch.empty(1, 16, dtype=torch.uint8, device=DEV)
    te.te_quantize(x, q, out)
    torch.cuda.synchronize()
    xv = np64(x)
    assert q.amax.item() == float("inf")
    scale = np.float32(2.0) if mode == "delayed" else np.float32(1.0)
    assert q.scale.item() == scale and q.scale_inv.item() == 1.0 / scale
    got, want = codes(out), nx.quantize(xv, scale).astype(np.int64)
    nan = np.isnan(xv)
    assert _nan_code(got[nan]).all()
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0, 1] == 0x7E and got[0, 2] == 0xFE  # +-inf -> +-448


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_nan_and_zero_amax_current_scaling(dtype):
    """Current scaling: NaN does not enter the amax (scale from the finite values); an all-zero
    tensor has amax 0, which gives scale 1 and all-zero codes."""
    x = rt((8, 64), std=3.0, seed=41, dtype=dtype)
    x[3, 5] = float("nan")
    q = te.Quantizer(mode="current")
    out = torch.empty(8, 64, dtype=torch.uint8, device=DEV)
    te.te_quantize(x, q, out)
    torch.cuda.synchronize()
    xv = np64(x)
    amax = nx.amax_of(xv)
    assert np.isfinite(amax) and q.amax.item() == amax
    scale = nx.compute_scale(amax)[0]
    assert q.scale.item() == scale
    got, want = codes(out), nx.quantize(xv, scale).astype(np.int64)
    assert _nan_code(got[3, 5])
    got[3, 5] = want[3, 5] = 0
    assert np.array_equal(got, want)
    z = torch.zeros(8, 64, dtype=TDT[dtype], device=DEV)
    qz = te.Quantizer(scale=5.0, mode="current")
    te.te_quantize(z, qz, out)
    torch.cuda.synchronize()
    assert qz.amax.item() == 0.0 and qz.scale.item() == 1.0 and qz.scale_inv.item() == 1.0
    assert int(out.count_nonzero().item()) == 0


def test_norm_e4m3_zero_rows_and_all_zero_current_scaling():
    """RMSNorm of all-zero rows is zero; a tensor of only such rows has amax 0 -> scale 1 under
    current scaling.  LayerNorm of a constant row is beta exactly."""
    M, H = 70, 1024
    x = torch.zeros(M, H, dtype=torch.bfloat16, device=DEV)
    gamma = rt((H,), 0.1, 42, mean=1.0)
    q = te.Quantizer(scale=3.0, mode="current")
    out = torch.full((M, H), 0x55, dtype=torch.uint8, device=DEV)
    te.te_norm_fwd(x, gamma, None, "rmsnorm", False, 1e-6, out, q=q)
    torch.cuda.synchronize()
    assert q.amax.item() == 0.0 and q.scale.item() == 1.0
    assert int(out.count_nonzero().item()) == 0
    x[5].fill_(3.0)  # a constant LayerNorm row: y = beta
    beta = rt((H,), 0.1, 43)
    q2 = te.Quantizer(scale=64.0)
    te.te_norm_fwd(x, gamma, beta, "layernorm", False, 1e-6, out, q=q2)
    torch.cuda.synchronize()
    want = nx.quantize(np64(beta)[None, :].repeat(M, 0), np.float32(64.0))
    assert_e4m3_codes(out, want, what="constant rows")
    assert q2.amax.item() == nx.amax_of(np64(beta))


def test_dact_dbias_nan_zero_current_scaling():
    """dact + dbias + E4M3 in current scaling: an all-zero dy gives dx codes 0, dbias 0 and
    scale 1; a NaN in dy becomes a NaN code, a NaN in its dbias column, and stays out of the
    amax."""
    M, N = 300, 528
    h = rt((M, N), std=2.0, seed=44)
    dy = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    dx = torch.full((M, N), 0x55, dtype=torch.uint8, device=DEV)
    db = torch.full((N,), 1.0, dtype=torch.float32, device=DEV)
    q = te.Quantizer(scale=9.0, mode="current")
    te.te_dact_dbias_quantize(dy, h, "gelu", dx, dbias=db, q=q)
    torch.cuda.synchronize()
    assert q.amax.item() == 0.0 and q.scale.item() == 1.0
    # 0 * act'(h) is a signed zero (code 0x00 or 0x80, with the derivative's sign), nothing else
    assert int((dx & 0x7F).count_nonzero().item()) == 0 and int(db.count_nonzero().item()) == 0
    dy = rt((M, N), seed=45)
    dy[7, 11] = float("nan")
    te.te_dact_dbias_quantize(dy, h, "gelu", dx, dbias=db, q=q)
    torch.cuda.synchronize()
    pre = nx.to_f32(ob.act_bwd(np64(dy), np64(h), "gelu"))
    amax = nx.amax_of(pre)
    assert np.isfinite(q.amax.item()) and abs(q.amax.item() - amax) <= 1e-6 * amax
    got = codes(dx)
    assert _nan_code(got[7, 11])
    dbv = np64(db)
    assert np.isnan(dbv[11]) and np.isfinite(np.delete(dbv, 11)).all()


# ------------------------------------------------------------------ activation -------------


@pytest.mark.parametrize("act", ["relu", "gelu", "silu", "swiglu", "geglu", "reglu"])
@pytest.mark.parametrize("M,N", [(1, 16), (300, 1040)])
def test_act_lu_bf16(act, M, N):
    x = rt((M, N), std=2.0, seed=3)
    n_out = N // 2 if ob.GATED[act] else N
    gout = Guarded((M, n_out), torch.bfloat16)
    out = gout.t
    te.te_act_lu(x, act, out)
    gout.check(act)
    ref = ob.act_fwd(np64(x), act)
    assert_elementwise_close(out, nx.bf16_round(nx.to_f32(ref)), what=act)
    if act in ("relu", "reglu"):  # exact arithmetic (one rounding): bit-exact
        assert np.array_equal(np64(out), nx.bf16_round(ref))


@pytest.mark.parametrize("act", ["gelu", "swiglu", "geglu"])
@pytest.mark.parametrize("mode", ["delayed", "current"])
def test_act_lu_e4m3_and_dequantized(act, mode):
    M, N = 257, 2048
    x = rt((M, N), std=2.0, seed=4)
    n_out = N // 2 if ob.GATED[act] else N
    q = te.Quantizer(scale=64.0, mode=mode)
    out = torch.empty(M, n_out, dtype=torch.uint8, device=DEV)
    te.te_act_lu(x, act, out, q=q)
    torch.cuda.synchronize()
    pre = nx.to_f32(ob.act_fwd(np64(x), act))
    amax = q.amax.item()
    assert abs(amax - nx.amax_of(pre)) <= 1e-6 * amax
    if mode == "current":  # the GPU derived its scale from its own amax, in fp32
        assert q.scale.item() == nx.compute_scale(np.float32(amax))[0]
    scale = np.float32(64.0) if mode == "delayed" else nx.compute_scale(nx.amax_of(pre))[0]
    assert_e4m3_codes(out, nx.quantize(pre, scale), pre32=pre, scale=scale, rel=1e-5,
                      abs_tol=1e-6 * rms(pre), what="act e4m3")
    # dequantized output (the pages' activation() result) in bf16
    deq = torch.empty(M, n_out, dtype=torch.bfloat16, device=DEV)
    q2 = te.Quantizer(scale=64.0, mode=mode)
    te.te_act_lu(x, act, deq, q=q2)
    want = nx.bf16_round(nx.dequantize(codes(out), np.float32(1.0) / np.float32(q.scale.item())))
    got = np64(deq)
    mism = got != want
    assert mism.mean() <= 1e-3  # only where the code itself flipped


# ------------------------------------------------------------------ dact + dbias -----------


@pytest.mark.parametrize("act", ["gelu", "relu", "silu", "swiglu", "geglu", "reglu", "identity"])
@pytest.mark.parametrize("M,N_in", [(1, 16), (300, 528), (1000, 4096)])
def test_dact_dbias_bf16(act, M, N_in):
    n_out = N_in // 2 if ob.GATED.get(act, False) else N_in
    dy = rt((M, n_out), seed=5)
    h = rt((M, N_in), std=2.0, seed=6)
    gdx, gdb = Guarded((M, N_in), torch.bfloat16), Guarded((N_in,), torch.float32)
    dx, db = gdx.t, gdb.t
    te.te_dact_dbias_quantize(dy, h, act, dx, dbias=db)
    gdx.check("dx")
    gdb.check("dbias")
    ref = np64(dy) if act == "identity" else ob.act_bwd(np64(dy), np64(h), act)
    assert_elementwise_close(dx, nx.bf16_round(nx.to_f32(ref)), what=f"d{act}")
    assert_reduction_close(db, ob.colsum(nx.to_f32(ref)), what=f"dbias {act}")


@pytest.mark.parametrize("mode", ["delayed", "current"])
def test_dact_dbias_e4m3(mode):
    M, N = 1000, 2048
    dy = rt((M, N), seed=7)
    h = rt((M, N), std=2.0, seed=8)
    q = te.Quantizer(scale=32.0, mode=mode)
    dx = torch.empty(M, N, dtype=torch.uint8, device=DEV)
    db = torch.empty(N, dtype=torch.float32, device=DEV)
    te.te_dact_dbias_quantize(dy, h, "gelu", dx, dbias=db, q=q)
    torch.cuda.synchronize()
    pre = nx.to_f32(ob.act_bwd(np64(dy), np64(h), "gelu"))
    if mode == "current":
        assert q.scale.item() == nx.compute_scale(np.float32(q.amax.item()))[0]
    scale = np.float32(32.0) if mode == "delayed" else nx.compute_scale(nx.amax_of(pre))[0]
    assert_e4m3_codes(dx, nx.quantize(pre, scale), pre32=pre, scale=scale, rel=1e-5,
                      abs_tol=1e-6 * rms(pre), what="dact e4m3")
    assert_reduction_close(db, ob.colsum(pre), what="dbias")
    assert abs(q.amax.item() - nx.amax_of(pre)) <= 1e-6 * nx.amax_of(pre)


def test_dbias_deterministic():
    M, N = 4096, 1024
    dy, h = rt((M, N), seed=9), rt((M, N), seed=10)
    outs = []
    for _ in range(3):
        dx = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        db = torch.empty(N, dtype=torch.float32, device=DEV)
        te.te_dact_dbias_quantize(dy, h, "gelu", dx, dbias=db)
        outs.append(db.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ------------------------------------------------------------------ norm -------------------


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("M,H,dtype", [(1, 128, "f32"), (129, 136, "bf16"), (1000, 4096, "bf16"),
                                       (70, 8192, "bf16"), (64, 128, "f32"), (70, 4096, "f32"),
                                       (9000, 1024, "bf16"), (301, 2048, "bf16"),
                                       (257, 2048, "f32"), (33, 512, "f32")])
@pytest.mark.parametrize("zc", [False, True])
def test_norm_fwd(norm, M, H, dtype, zc):
    """Widths of 4, 8 or 16 vectors per lane of a warp (1024 / 2048 / 4096 bf16, 512 / 1024 /
    2048 fp32) take one row per warp; bf16 rows of 8192 the eight warps of a CTA with a ring of
    staged rows; the others a CTA of four warps per row."""
    x = rt((M, H), std=2.0, seed=11, dtype=dtype, mean=0.5)
    gamma = rt((H,), std=0.1, seed=12, dtype=dtype, mean=0.0 if zc else 1.0)
    beta = rt((H,), std=0.1, seed=13, dtype=dtype)
    gout = Guarded((M, H), TDT[dtype])
    gmu, grs = Guarded((M,), torch.float32), Guarded((M,), torch.float32)
    out, mu, rs = gout.t, gmu.t, grs.t
    q = te.Quantizer()
    te.te_norm_fwd(x, gamma, beta, norm, zc, 1e-5, out, q=q, mu=mu, rsigma=rs)
    for gb, name in ((gout, "y"), (gmu, "mu"), (grs, "rsigma")):
        gb.check(name)
    y, m_ref, r_ref = ob.norm_fwd(np64(x), np64(gamma), np64(beta), norm, zc, 1e-5)
    want = nx.to_f32(y) if dtype == "f32" else nx.bf16_round(nx.to_f32(y))
    assert_elementwise_close(out, want, what=f"{norm} y")
    assert_reduction_close(rs, r_ref, what="rsigma")
    if norm == "layernorm":
        assert_reduction_close(mu, m_ref, what="mu")
    torch.cuda.synchronize()
    assert abs(q.amax.item() - nx.amax_of(nx.to_f32(y))) <= 1e-5 * nx.amax_of(nx.to_f32(y))


@pytest.mark.parametrize("M,H,dtype", [(1000, 4096, "bf16"), (300, 1024, "f32"), (70, 8192, "bf16"),
                                       (129, 136, "bf16"), (65, 4096, "f32")])
def test_layernorm_fwd_without_beta(M, H, dtype):
    """A NULL beta is a zero beta, in every kernel form (one row per warp: 4096 bf16 and 1024
    fp32; the eight-warp row-sharing kernel: 8192 bf16; the four-warp row kernel: 136 bf16 and
    4096 fp32)."""
    x = rt((M, H), std=1.5, seed=61, dtype=dtype, mean=-0.5)
    gamma = rt((H,), std=0.1, seed=62, dtype=dtype, mean=1.0)
    gout = Guarded((M, H), TDT[dtype])
    te.te_norm_fwd(x, gamma, None, "layernorm", False, 1e-5, gout.t)
    gout.check("y")
    y, _, _ = ob.norm_fwd(np64(x), np64(gamma), np.zeros(H), "layernorm", False, 1e-5)
    want = nx.to_f32(y) if dtype == "f32" else nx.bf16_round(nx.to_f32(y))
    assert_elementwise_close(gout.t, want, what="layernorm y without beta")


@pytest.mark.parametrize("norm,zc", [("layernorm", False), ("rmsnorm", True)])
@pytest.mark.parametrize("H,dtype", [(4096, "bf16"), (2048, "f32"), (8192, "bf16"), (4096, "f32")])
@pytest.mark.parametrize("out_kind", ["same", "e4m3"])
def test_norm_fwd_long_runs(norm, zc, H, dtype, out_kind):
    """Long runs (12000 rows, a ragged number of rows per warp or CTA): rows of 16 vectors per
    lane (one row per warp, each warp working through about ten rows with the next one in
    flight), bf16 rows of 8192 (a ring per CTA, which wraps six times) and fp32 rows of 4096 (the
    four-warp row kernel): y (or its E4M3 codes), mu, rsigma and amax, with guard bands."""
    M = 12000
    x = rt((M, H), std=1.5, seed=51, dtype=dtype, mean=0.25)
    gamma = rt((H,), std=0.1, seed=52, dtype=dtype, mean=0.0 if zc else 1.0)
    beta = rt((H,), std=0.1, seed=53, dtype=dtype)
    odt = torch.uint8 if out_kind == "e4m3" else TDT[dtype]
    gout, gmu, grs = Guarded((M, H), odt), Guarded((M,), torch.float32), Guarded((M,), torch.float32)
    q = te.Quantizer(scale=16.0)
    te.te_norm_fwd(x, gamma, beta, norm, zc, 1e-5, gout.t, q=q, mu=gmu.t, rsigma=grs.t)
    for gb, name in ((gout, "y"), (gmu, "mu"), (grs, "rsigma")):
        gb.check(name)
    y, m_ref, r_ref = ob.norm_fwd(np64(x), np64(gamma), np64(beta), norm, zc, 1e-5)
    pre = nx.to_f32(y)
    if out_kind == "e4m3":
        assert_e4m3_codes(gout.t, nx.quantize(pre, np.float32(16.0)), pre32=pre,
                          scale=np.float32(16.0), rel=1e-5, abs_tol=1e-5 * rms(pre),
                          what="norm e4m3")
    else:
        want = pre if dtype == "f32" else nx.bf16_round(pre)
        assert_elementwise_close(gout.t, want, what=f"{norm} y")
    assert_reduction_close(grs.t, r_ref, what="rsigma")
    if norm == "layernorm":
        assert_reduction_close(gmu.t, m_ref, what="mu")
    assert abs(q.amax.item() - nx.amax_of(pre)) <= 1e-5 * nx.amax_of(pre)


@pytest.mark.parametrize("M", [70, 300, 457])
def test_norm_fwd_e4m3_8192_partial_steps(M):
    """8192-wide bf16 rows with E4M3 output: the row-sharing kernel then works on four rows per
    barrier, and these row counts leave CTAs with fewer rows than one step (and a partial last
    step): codes, mu, rsigma and amax, with guard bands."""
    H = 8192
    x = rt((M, H), std=1.5, seed=71, mean=0.25)
    gamma = rt((H,), std=0.1, seed=72, mean=1.0)
    beta = rt((H,), std=0.1, seed=73)
    gout, gmu, grs = Guarded((M, H), torch.uint8), Guarded((M,), torch.float32), Guarded((M,), torch.float32)
    q = te.Quantizer(scale=16.0)
    te.te_norm_fwd(x, gamma, beta, "layernorm", False, 1e-5, gout.t, q=q, mu=gmu.t, rsigma=grs.t)
    for gb, name in ((gout, "y"), (gmu, "mu"), (grs, "rsigma")):
        gb.check(name)
    y, m_ref, r_ref = ob.norm_fwd(np64(x), np64(gamma), np64(beta), "layernorm", False, 1e-5)
    pre = nx.to_f32(y)
    assert_e4m3_codes(gout.t, nx.quantize(pre, np.float32(16.0)), pre32=pre,
                      scale=np.float32(16.0), rel=1e-5, abs_tol=1e-5 * rms(pre),
                      what="norm e4m3 8192")
    assert_reduction_close(grs.t, r_ref, what="rsigma")
    assert_reduction_close(gmu.t, m_ref, what="mu")
    assert abs(q.amax.item() - nx.amax_of(pre)) <= 1e-5 * nx.amax_of(pre)


@pytest.mark.parametrize("mode", ["delayed", "current"])
def test_norm_fwd_e4m3(mode):
    M, H = 1000, 4096
    x = rt((M, H), seed=14)
    gamma, beta = rt((H,), 0.1, 15, mean=1.0), rt((H,), 0.1, 16)
    gout = Guarded((M, H), torch.uint8)
    out = gout.t
    q = te.Quantizer(scale=64.0, mode=mode)
    te.te_norm_fwd(x, gamma, beta, "layernorm", False, 1e-5, out, q=q)
    gout.check("norm e4m3")
    y, _, _ = ob.norm_fwd(np64(x), np64(gamma), np64(beta), "layernorm", False, 1e-5)
    pre = nx.to_f32(y)
    gpu_scale = np.float32(q.scale.item())
    if mode == "current":
        assert gpu_scale == nx.compute_scale(np.float32(q.amax.item()))[0]
        assert abs(q.amax.item() - nx.amax_of(pre)) <= 1e-5 * nx.amax_of(pre)
    assert q.scale_inv.item() == np.float32(1.0) / gpu_scale
    scale = np.float32(64.0) if mode == "delayed" else nx.compute_scale(nx.amax_of(pre))[0]
    assert_e4m3_codes(out, nx.quantize(pre, scale), pre32=pre, scale=scale, rel=1e-5,
                      abs_tol=1e-5 * rms(pre), what="norm e4m3")


def test_norm_scale_identity_outlier_rows():
    """LN(8x; eps) == LN(x; eps/64): rows scaled by 8 normalize to the unscaled rows' output."""
    M, H = 64, 1024
    x = rt((M, H), seed=17, dtype="f32")
    x8 = x * 8.0
    g, b = rt((H,), 0.1, 18, "f32", 1.0), rt((H,), 0.1, 19, "f32")
    o1 = torch.empty(M, H, device=DEV)
    o2 = torch.empty(M, H, device=DEV)
    te.te_norm_fwd(x8, g, b, "layernorm", False, 1e-5, o1)
    te.te_norm_fwd(x, g, b, "layernorm", False, 1e-5 / 64, o2)
    assert torch.allclose(o1, o2, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("M,H,dtype", [(1, 128, "bf16"), (300, 1032, "bf16"), (2000, 4096, "bf16"),
                                       (5000, 2048, "bf16"), (64, 8192, "bf16"),
                                       (300, 1032, "f32"), (70, 4096, "f32")])
def test_norm_bwd(norm, M, H, dtype):
    """Rows are dealt to CTAs round-robin and streamed through a ring of shared-memory slots;
    the (5000, 2048) case passes through every slot of the ring more than twice."""
    x = rt((M, H), std=2.0, seed=20, dtype=dtype)
    gamma = rt((H,), 0.1, 21, mean=1.0, dtype=dtype)
    dz = rt((M, H), seed=22, dtype=dtype)
    _, mu, rs = ob.norm_fwd(np64(x), np64(gamma), None if norm == "rmsnorm" else np.zeros(H),
                            norm, False, 1e-5)
    mu_t = torch.tensor(mu, dtype=torch.float32, device=DEV)
    rs_t = torch.tensor(rs, dtype=torch.float32, device=DEV)
    dx = torch.empty(M, H, dtype=TDT[dtype], device=DEV)
    dg = torch.empty(H, dtype=torch.float32, device=DEV)
    db = torch.empty(H, dtype=torch.float32, device=DEV)
    te.te_norm_bwd(dz, x, mu_t, rs_t, gamma, norm, False, dx, dg, db)
    # identical inputs: dx within the fp32 window of the norm backward's arithmetic, the column
    # sums to the 1e-4 reduction rule plus that window
    args = (np64(x), np64(mu_t), np64(rs_t))
    check_norm_dx(dx, np64(dz), 0.0, *args, np64(gamma), norm, False, stored=dtype,
                  dln_dtype=dtype)
    check_norm_params(dg, db if norm == "layernorm" else None, np64(dz), 0.0, *args, norm,
                      dln_dtype=dtype)


def test_norm_bwd_large_mean():
    """LayerNorm rows whose mean is 64 standard deviations from zero: the kernel forms xhat as
    x * rs - mu * rs, so the rounding of mu * rs must stay below the tolerances."""
    M, H = 600, 4096
    x = rt((M, H), std=1.0, seed=23, mean=64.0)
    gamma = rt((H,), 0.1, 24, mean=1.0)
    dz = rt((M, H), seed=25)
    _, mu, rs = ob.norm_fwd(np64(x), np64(gamma), np.zeros(H), "layernorm", False, 1e-5)
    mu_t = torch.tensor(mu, dtype=torch.float32, device=DEV)
    rs_t = torch.tensor(rs, dtype=torch.float32, device=DEV)
    dx = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
    dg = torch.empty(H, dtype=torch.float32, device=DEV)
    db = torch.empty(H, dtype=torch.float32, device=DEV)
    te.te_norm_bwd(dz, x, mu_t, rs_t, gamma, "layernorm", False, dx, dg, db)
    args = (np64(x), np64(mu_t), np64(rs_t))
    check_norm_dx(dx, np64(dz), 0.0, *args, np64(gamma), "layernorm", False, dln_dtype="bf16")
    check_norm_params(dg, db, np64(dz), 0.0, *args, "layernorm", dln_dtype="bf16")


# ------------------------------------------------------------------ GEMM -------------------


@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (False, True), (True, False),
                                             (True, True)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 272, 96), (520, 784, 1040)])
def test_gemm_bf16_layouts(a_trans, b_trans, M, N, K):
    if a_trans and M % 16:
        M += 16 - M % 16
    A = rt((K, M) if a_trans else (M, K), seed=23)
    B = rt((N, K) if b_trans else (K, N), seed=24)
    bias = rt((N,), 0.5, 25)
    gout = Guarded((M, N), torch.bfloat16)
    out = gout.t
    te.te_gemm(A, B, out, a_trans=a_trans, b_trans=b_trans, bias=bias)
    gout.check("gemm")
    a = np64(A).T if a_trans else np64(A)
    b = np64(B).T if b_trans else np64(B)
    ref = ob.gemm(a, b, np64(bias))
    assert_gemm_close(out, ref, K, rms(a), rms(b), what=f"gemm bf16 {a_trans}{b_trans}")


@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (False, True), (True, False),
                                             (True, True)])
def test_gemm_e4m3(a_trans, b_trans):
    M, N, K = 384, 528, 640
    Af = rt((K, M) if a_trans else (M, K), std=50.0, seed=26, dtype="f32")
    Bf = rt((N, K) if b_trans else (K, N), std=50.0, seed=27, dtype="f32")
    A = Af.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    B = Bf.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    sa = torch.tensor([1 / 64.0], device=DEV)
    sb = torch.tensor([1 / 128.0], device=DEV)
    out = torch.empty(M, N, dtype=torch.float32, device=DEV)
    te.te_gemm(A, B, out, a_trans=a_trans, b_trans=b_trans, a_scale_inv=sa, b_scale_inv=sb)
    a = nx.e4m3_decode(codes(A))
    b = nx.e4m3_decode(codes(B))
    a = a.T if a_trans else a
    b = b.T if b_trans else b
    ref = ob.gemm(a, b, None, alpha=ob.gemm_alpha(1 / 64.0, 1 / 128.0))
    # fp8 products are exact in fp32 accumulation up to summation order
    assert_gemm_close(out, ref, K, rms(a) / 64, rms(b) / 128, what="gemm e4m3")
    err = np.abs(np64(out) - ref).max()
    assert err <= 1e-4 * np.abs(ref).max() + 1e-6


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (False, True), (True, False)])
@pytest.mark.parametrize("M,N,K", [(300, 528, 16400), (1040, 272, 16384), (256, 256, 16384)])
def test_gemm_split_k(kind, a_trans, b_trans, M, N, K):
    """Tiles split along K (fewer tiles than SM pairs, long K; a ragged last k-block at
    K = 16400, ragged M and N): against the oracle, against the unsplit GEMM within the fp32
    accumulation window, bit-identical on repeated calls (the partial sums are added in chunk
    order), and nothing written outside the output or the workspace."""
    if a_trans and M % 16:
        M += 16 - M % 16
    A = rt((K, M) if a_trans else (M, K), std=1.0, seed=M + 31, dtype="f32")
    B = rt((N, K) if b_trans else (K, N), std=1.0, seed=N + 32, dtype="f32")
    bias = rt((N,), 0.5, 33)
    if kind == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
        a, b = np64(A), np64(B)
        sa = sb = None
        alpha = 1.0
        ab = te.binding.TE_BF16
    else:
        A = (A * 64).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        B = (B * 64).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        a, b = nx.e4m3_decode(codes(A)), nx.e4m3_decode(codes(B))
        sa = torch.tensor([1 / 64.0], device=DEV)
        sb = torch.tensor([1 / 64.0], device=DEV)
        alpha = ob.gemm_alpha(1 / 64.0, 1 / 64.0)
        ab = te.binding.TE_E4M3
    nws = te.workspace_size(te.binding.TE_OP_GEMM, M, K, N, ab)
    assert nws > 0, "these shapes leave SM pairs idle: the library should split them"
    ws = Guarded((nws,), torch.uint8)
    outs = []
    for split in (True, True, False):
        g = Guarded((M, N), torch.float32)
        te.te_gemm(A, B, g.t, a_trans=a_trans, b_trans=b_trans, a_scale_inv=sa, b_scale_inv=sb,
                   bias=bias, workspace=ws.t if split else None, split_k=split)
        g.check("split-K gemm out")
        outs.append(np64(g.t))
    ws.check("split-K workspace")
    assert np.array_equal(outs[0], outs[1]), "split-K result differs between two calls"
    a = a.T if a_trans else a
    b = b.T if b_trans else b
    ref = ob.gemm(a, b, np64(bias), alpha)
    absdot = np.abs(a) @ np.abs(b) * abs(alpha)
    for got, what in ((outs[0], "split"), (outs[2], "unsplit")):
        ratio = float((np.abs(got - ref) / absdot).max())
        assert ratio <= ACC_REL, f"{what}: {ratio:.3e} > ACC_REL {ACC_REL:.3e}"


@pytest.mark.parametrize("kind,M,N,K", [("bf16", 100, 528, 16384), ("tf32", 200, 256, 8192)])
def test_gemm_split_k_single_cta_tiles(kind, M, N, K):
    """The split along K with single-CTA tiles (128 x 256: M <= 128, and the tf32 path, which
    always runs them): against the oracle within the accumulation window, repeatable to the
    bit, and nothing written outside the output or the workspace."""
    if kind == "bf16":
        A = rt((M, K), seed=61)
        B = rt((N, K), seed=62)
        ab = te.binding.TE_BF16
    else:
        A = rt((M, K), seed=61, dtype="f32")
        B = rt((N, K), seed=62, dtype="f32")
        ab = te.binding.TE_F32
    nws = te.workspace_size(te.binding.TE_OP_GEMM, M, K, N, ab)
    assert nws > 0, "these shapes leave SM pairs idle: the library should split them"
    ws = Guarded((nws,), torch.uint8)
    outs = []
    for _ in range(2):
        g = Guarded((M, N), torch.float32)
        te.te_gemm(A, B, g.t, b_trans=True, workspace=ws.t)
        g.check("split-K gemm out")
        outs.append(np64(g.t))
    ws.check("split-K workspace")
    assert np.array_equal(outs[0], outs[1])
    a, b = np64(A), np64(B).T
    ref = ob.gemm(a, b, None)
    absdot = np.abs(a) @ np.abs(b)
    if kind == "bf16":
        ratio = float((np.abs(outs[0] - ref) / absdot).max())
        assert ratio <= ACC_REL, f"{ratio:.3e} > ACC_REL {ACC_REL:.3e}"
    else:  # tf32 operands: held to the bf16 rule of the fp32 workload
        assert_gemm_close(outs[0], ref, K, rms(a), rms(b), what="split-K tf32", stored="f32")


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
@pytest.mark.parametrize("a_trans,b_trans", [(False, False), (False, True), (True, False)])
@pytest.mark.parametrize("K", [512, 4096, 16384])
def test_gemm_accumulation_window(kind, a_trans, b_trans, K):
    """The fp32 accumulation error of the tensor-core GEMMs against the exact (float64) sum,
    relative to sum_k |a_k b_k|, stays within parity.ACC_REL: the window the step-by-step
    backward checks allow a bf16 GEMM output to round across a midpoint.  Output in fp32, so
    nothing but the accumulation is measured."""
    M, N = 256, 272
    A = rt((K, M) if a_trans else (M, K), std=1.0, seed=K + 1, dtype="f32")
    B = rt((N, K) if b_trans else (K, N), std=1.0, seed=K + 2, dtype="f32")
    if kind == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
        a, b = np64(A), np64(B)
        sa = sb = None
        alpha = 1.0
    else:
        A = (A * 64).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        B = (B * 64).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        a, b = nx.e4m3_decode(codes(A)), nx.e4m3_decode(codes(B))
        sa = torch.tensor([1 / 64.0], device=DEV)
        sb = torch.tensor([1 / 64.0], device=DEV)
        alpha = ob.gemm_alpha(1 / 64.0, 1 / 64.0)
    out = torch.empty(M, N, dtype=torch.float32, device=DEV)
    te.te_gemm(A, B, out, a_trans=a_trans, b_trans=b_trans, a_scale_inv=sa, b_scale_inv=sb)
    a = a.T if a_trans else a
    b = b.T if b_trans else b
    ref = ob.gemm(a, b, None, alpha)
    absdot = np.abs(a) @ np.abs(b) * abs(alpha)
    ratio = float((np.abs(np64(out) - ref) / absdot).max())
    print(f"accumulation error / sum|ab|: {ratio:.3e} ({kind}, K={K})")
    assert ratio <= ACC_REL, f"{ratio:.3e} > ACC_REL {ACC_REL:.3e}"


def test_gemm_tf32_k_major():
    M, N, K = 200, 288, 160
    A = rt((M, K), seed=28, dtype="f32")
    B = rt((N, K), seed=29, dtype="f32")
    bias = rt((N,), 0.1, 30, dtype="f32")
    out = torch.empty(M, N, dtype=torch.float32, device=DEV)
    te.te_gemm(A, B, out, b_trans=True, bias=bias)
    ref = ob.gemm(np64(A), np64(B).T, np64(bias))
    assert_gemm_close(out, ref, K, rms(np64(A)), rms(np64(B)), what="gemm tf32")


def test_gemm_tf32_rejects_mn_major():
    A = rt((64, 32), dtype="f32")
    B = rt((32, 64), dtype="f32")
    out = torch.empty(64, 64, dtype=torch.float32, device=DEV)
    with pytest.raises(te.TEError) as e:
        te.te_gemm(A, B, out)  # fp32 operands must be K-major (B stored [N, K])
    assert e.value.status == te.binding.TE_ERR_UNSUPPORTED


def test_gemm_rejects_bad_shapes():
    A = torch.zeros(16, 24, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(24, 16, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(16, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(te.TEError) as e:
        te.te_gemm(A, B, out)  # K = 24 is not a multiple of 16
    assert e.value.status == te.binding.TE_ERR_UNSUPPORTED


def test_no_device_timeouts_recorded():
    torch.cuda.synchronize()
    assert te.get_device_status() == 0
