"""Block-level parity: te_layernorm_dense_fwd and te_layernorm_mlp_fwd against the oracle.

Small cases run every workload's recipe at shapes that span several 128 x 256 tiles with ragged
tails, and are compared element by element.  Full-size cases run the exact benchmark
configurations and compare a seeded sample of whole output rows (the block is row-local, so the
oracle computes just those rows), plus properties that hold at any size.
FP8 cases use fixed (delayed) power-of-two scales so both sides quantize with the same scale.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import block as ob
from oracle import numerics as nx
from parity import (Guarded, assert_e4m3_codes, assert_gemm_close, assert_in_window,
                    assert_reduction_close, codes, decode, np64, quantize_fast, rms)
from steps import gemm_ref
from workloads import make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"

MLP_SCALES = dict(x=32.0, w1=2048.0, act=16.0, w2=2048.0)


def _qset(scales, mode="delayed"):
    return te.QuantizerSet(x=te.Quantizer(scales["x"], mode), kernel1=te.Quantizer(scales["w1"]),
                           act=te.Quantizer(scales["act"], mode),
                           kernel2=te.Quantizer(scales["w2"]))


def _fp8_oracle_scales(scales):
    """fp32 scales for the oracle; None (current scaling: the tensor's own amax) stays None."""
    return {k: None if v is None else np.float32(v) for k, v in scales.items()}


def run_mlp(inp, fp8=False, scales=MLP_SCALES, mode="delayed", rows=None):
    M, H, F = inp["M"], inp["H"], inp["F"]
    gated = ob.GATED[inp["act"]]
    dt = inp["x"].dtype
    guards = dict(out=Guarded((M, H), dt), h=Guarded((M, 2 * F if gated else F), dt),
                  ln=Guarded((M, H), torch.uint8 if fp8 else dt),
                  act=Guarded((M, F), torch.uint8 if fp8 else dt))
    out, saved_h, ln, act = (guards[k].t for k in ("out", "h", "ln", "act"))
    mu = torch.empty(M, dtype=torch.float32, device=DEV)
    rs = torch.empty(M, dtype=torch.float32, device=DEV)
    qs = _qset(scales, mode) if fp8 else None
    te.te_layernorm_mlp_fwd(inp["x"], inp["gamma"], inp["beta"], inp["w1"], inp["w2"],
                            inp.get("b1"), inp.get("b2"), out, norm_type=inp["norm"],
                            zero_centered_gamma=inp["zero_centered_gamma"], epsilon=inp["eps"],
                            activation_type=inp["act"], quantizer_set=qs, saved_h=saved_h,
                            saved_act=act, saved_ln_out=ln, mu=mu, rsigma=rs)
    for k, gb in guards.items():
        gb.check(k)
    return dict(out=out, h=saved_h, act=act, ln=ln, mu=mu, rsigma=rs, qs=qs)


def check_act(inp, got, fp8, rows=None, scale=None):
    """GEMM1's epilogue output against the oracle's activation of the GPU's own saved h (the
    activation input, identical on both sides): E4M3 codes under the one-step-flip rule with the
    fp32 activation error bound of the standalone activation test, the activation amax to 1e-6
    relative (an order-free max over values that differ from the oracle's by that fp32 error);
    bf16 outputs within one bf16 ulp, on at most 0.1% of elements."""
    sel = slice(None) if rows is None else rows
    pre = nx.to_f32(ob.act_fwd(np64(got["h"])[sel], inp["act"]))
    if fp8:
        scale = np.float32(got["qs"].act.scale.item()) if scale is None else np.float32(scale)
        assert_e4m3_codes(codes(got["act"])[sel], nx.quantize(pre, scale), pre32=pre,
                          scale=scale, rel=1e-5, abs_tol=1e-6 * rms(pre), what="act e4m3")
        if rows is None:
            amax = got["qs"].act.amax.item()
            assert abs(amax - nx.amax_of(pre)) <= 1e-6 * nx.amax_of(pre), "act amax"
    elif inp["dtype"] == "bf16":
        g, want = np64(got["act"])[sel], nx.bf16_round(pre)
        diff = g != want
        far = np.abs(g - want) > 2.0 ** -7 * np.abs(want)
        if far.any():
            h = np64(got["h"])[sel]
            i = np.argwhere(far)[0]
            raise AssertionError(f"act: {int(far.sum())} beyond one bf16 ulp; first at {tuple(i)}: "
                                 f"got {g[tuple(i)]!r} want {want[tuple(i)]!r} pre "
                                 f"{pre[tuple(i)]!r}")
        assert diff.mean() <= 1e-3, f"act: {int(diff.sum())} of {diff.size} one ulp apart"


def oracle_mlp(inp, fp8=False, scales=MLP_SCALES, rows=None):
    sel = slice(None) if rows is None else rows
    x = np64(inp["x"])[sel]
    return ob.layernorm_mlp_fwd(x, np64(inp["gamma"]), np64(inp["beta"]), np64(inp["w1"]),
                                np64(inp["w2"]), None if inp.get("b1") is None else np64(inp["b1"]),
                                None if inp.get("b2") is None else np64(inp["b2"]), inp["norm"],
                                inp["zero_centered_gamma"], inp["eps"], inp["act"],
                                "f32" if inp["dtype"] == "f32" else "bf16",
                                fp8=_fp8_oracle_scales(scales) if fp8 else None)


def check_mlp(inp, got, ref, fp8, rows=None):
    sel = slice(None) if rows is None else rows
    H = inp["H"]
    F = inp["F"]
    ln_ref = ref["ln"]
    # normalized operand
    if fp8:
        assert_e4m3_codes(codes(got["ln"])[sel], ln_ref.codes, pre32=ln_ref.pre,
                          scale=ln_ref.scale, rel=1e-5, abs_tol=1e-5 * rms(ln_ref.pre),
                          what="ln e4m3")
    else:
        np.testing.assert_allclose(np64(got["ln"])[sel], ln_ref.value, rtol=2e-2,
                                   atol=1e-3 * rms(ln_ref.value))
    assert_reduction_close(np64(got["rsigma"])[sel], ref["rsigma"], what="rsigma")
    # GEMM1 output (+ bias, rounded): contraction over H
    a1 = ln_ref.value * ln_ref.inv()
    w1 = ref["w1"].value * ref["w1"].inv()
    stored = "f32" if inp["dtype"] == "f32" else "bf16"
    assert_gemm_close(np64(got["h"])[sel], ref["h"].value, H, rms(a1), rms(w1), what="h",
                      stored=stored)
    # block output: contraction over F
    a2 = ref["a"].value * ref["a"].inv()
    w2 = ref["w2"].value * ref["w2"].inv()
    assert_gemm_close(np64(got["out"])[sel], ref["out"].value, F, rms(a2), rms(w2), what="out",
                      stored=stored)
    check_act(inp, got, fp8, rows=rows)


# -------------------------------------------------------------- small, element by element --

SMALL = [
    ("tiny_ln_mlp", {}),
    ("gpt_ln_mlp", dict(M=300, H=512, F=784)),
    ("llama_rms_mlp", dict(M=300, H=512, F=784)),
]


@pytest.mark.parametrize("name,shape", SMALL)
def test_mlp_small(name, shape):
    inp = make_inputs(name, device=DEV, **shape)
    got = run_mlp(inp)
    ref = oracle_mlp(inp)
    check_mlp(inp, got, ref, fp8=False)


@pytest.mark.parametrize("act", ["geglu", "reglu"])
@pytest.mark.parametrize("fp8", [False, True])
def test_mlp_small_other_gated(act, fp8):
    """("gelu", "linear") and ("relu", "linear") through GEMM1's gated epilogue, on the Llama
    workload's tensors (W1 holds [gate | linear] columns)."""
    inp = make_inputs("llama_rms_mlp", device=DEV, M=300, H=512, F=784)
    inp["act"] = act
    got = run_mlp(inp, fp8=fp8)
    ref = oracle_mlp(inp, fp8=fp8)
    check_mlp(inp, got, ref, fp8=fp8)


@pytest.mark.parametrize("shape", [dict(M=300, H=8192, F=784), dict(M=300, H=512, F=16384)])
@pytest.mark.parametrize("fp8", [False, True])
def test_mlp_split_k(shape, fp8):
    """Few tiles and a long contraction, so the library splits GEMM1 (the gated SwiGLU epilogue,
    K = H = 8192; bf16 only: E4M3 k-blocks are twice as deep, too few to split) or GEMM2 (K = F =
    16384) along K: element by element against the oracle, and bit-identical on a second call."""
    inp = make_inputs("llama_rms_mlp", device=DEV, **shape)
    got = run_mlp(inp, fp8=fp8)
    again = run_mlp(inp, fp8=fp8)
    for k in ("out", "h", "act"):
        assert torch.equal(got[k], again[k]), k
    ref = oracle_mlp(inp, fp8=fp8)
    check_mlp(inp, got, ref, fp8=fp8)


def test_mlp_workspace_without_split_room():
    """A workspace that stops short of the split scratch at its end is accepted: the call
    splits fewer or no tiles along K and gives the same result within the GEMM windows."""
    inp = make_inputs("llama_rms_mlp", device=DEV, M=300, H=512, F=16384)
    M, H, F = inp["M"], inp["H"], inp["F"]
    b = te.binding
    full = te.workspace_size(b.TE_OP_LAYERNORM_MLP_FWD, M, H, F, b.TE_BF16, False, b.TE_BF16,
                             b.TE_SWIGLU)
    outs = []
    for nbytes in (full, full - 16):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        out = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
        te.te_layernorm_mlp_fwd(inp["x"], inp["gamma"], inp["beta"], inp["w1"], inp["w2"], None,
                                None, out, norm_type=inp["norm"],
                                zero_centered_gamma=inp["zero_centered_gamma"],
                                epsilon=inp["eps"], activation_type=inp["act"], workspace=ws)
        outs.append(out)
    ref = oracle_mlp(inp)
    a2 = ref["a"].value * ref["a"].inv()
    w2 = ref["w2"].value * ref["w2"].inv()
    for out in outs:
        assert_gemm_close(np64(out), ref["out"].value, F, rms(a2), rms(w2), what="out",
                          stored="bf16")


def test_mlp_fp8_act_amax_sharing_storage_with_x():
    """The activation's amax is zeroed before the norm only when it has storage of its own; a
    quantizer set whose x and act amax share one scalar still ends with the activation's amax
    (the value an unshared act quantizer reports), the norm's amax having been overwritten."""
    inp = make_inputs("llama_rms_mlp", device=DEV, M=300, H=512, F=784)
    plain = run_mlp(inp, fp8=True)
    shared = torch.zeros(1, dtype=torch.float32, device=DEV)
    qx = te.Quantizer(MLP_SCALES["x"])
    qa = te.Quantizer(MLP_SCALES["act"])
    qs = te.QuantizerSet(
        x=te.Quantizer.from_tensors(qx.scale, qx.scale_inv, shared),
        kernel1=te.Quantizer(MLP_SCALES["w1"]),
        act=te.Quantizer.from_tensors(qa.scale, qa.scale_inv, shared),
        kernel2=te.Quantizer(MLP_SCALES["w2"]))
    out = torch.empty(inp["M"], inp["H"], dtype=torch.bfloat16, device=DEV)
    te.te_layernorm_mlp_fwd(inp["x"], inp["gamma"], inp["beta"], inp["w1"], inp["w2"], None, None,
                            out, norm_type=inp["norm"],
                            zero_centered_gamma=inp["zero_centered_gamma"], epsilon=inp["eps"],
                            activation_type=inp["act"], quantizer_set=qs)
    torch.cuda.synchronize()
    assert torch.equal(out, plain["out"])
    assert shared.item() == plain["qs"].act.amax.item()


@pytest.mark.parametrize("name,shape", SMALL[1:])
def test_mlp_small_fp8(name, shape):
    inp = make_inputs(name, device=DEV, **shape)
    got = run_mlp(inp, fp8=True)
    ref = oracle_mlp(inp, fp8=True)
    check_mlp(inp, got, ref, fp8=True)
    qs = got["qs"]
    # amax of the normalized output (the activation amax is held in check_act)
    assert abs(qs.x.amax.item() - float(ref["ln"].amax)) <= 1e-5 * float(ref["ln"].amax)
    assert qs.act.scale_inv.item() == np.float32(1.0) / np.float32(MLP_SCALES["act"])


@pytest.mark.parametrize("name,shape", SMALL[1:])
def test_mlp_small_fp8_current_scaling(name, shape):
    inp = make_inputs(name, device=DEV, **shape)
    got = run_mlp(inp, fp8=True, mode="current")
    qs = got["qs"]
    ref = oracle_mlp(inp, fp8=True, scales=dict(MLP_SCALES, x=None, act=None))
    # the scale is derived from this call's amax, in fp32, exactly as the recipe states
    for q in (qs.x, qs.act):
        amax = np.float32(q.amax.item())
        assert q.scale.item() == nx.compute_scale(amax)[0]
    # the normalized output's amax from identical inputs; the activation's from the GPU's own h
    assert abs(qs.x.amax.item() - float(ref["ln"].amax)) <= 1e-5 * float(ref["ln"].amax)
    check_act(inp, got, fp8=True)
    a2 = ref["a"].value * ref["a"].inv()
    w2 = ref["w2"].value * ref["w2"].inv()
    assert_gemm_close(got["out"], ref["out"].value, inp["F"], rms(a2), rms(w2), what="out")


@pytest.mark.parametrize("fp8", [False, True])
def test_ln_dense_small(fp8):
    inp = make_inputs("qkv_ln_dense", device=DEV, M=300, H=512, N=784)
    M, H, N = inp["M"], inp["H"], inp["N"]
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    ln = torch.empty(M, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)
    scales = dict(x=64.0, kernel=4096.0)
    qs = te.QuantizerSet(x=te.Quantizer(scales["x"]), kernel1=te.Quantizer(scales["kernel"])) if fp8 else None
    te.te_layernorm_dense_fwd(inp["x"], inp["kernel"], inp["gamma"], inp["beta"], inp["bias"],
                              out, epsilon=inp["eps"], quantizer_set=qs, saved_ln_out=ln)
    torch.cuda.synchronize()
    ref = ob.layernorm_dense_fwd(np64(inp["x"]), np64(inp["kernel"]), np64(inp["gamma"]),
                                 np64(inp["beta"]), np64(inp["bias"]), "layernorm", False,
                                 inp["eps"], "bf16",
                                 fp8={k: np.float32(v) for k, v in scales.items()} if fp8 else None)
    if fp8:
        assert_e4m3_codes(ln, ref["ln"].codes, pre32=ref["ln"].pre, scale=ref["ln"].scale,
                          rel=1e-5, abs_tol=1e-5 * rms(ref["ln"].pre), what="ln e4m3")
    a = ref["ln"].value * ref["ln"].inv()
    w = ref["kernel"].value * ref["kernel"].inv()
    assert_gemm_close(out, ref["out"].value, H, rms(a), rms(w), what="ln-dense out")


def test_ln_dense_prequantized_kernel_matches_per_call_cast():
    inp = make_inputs("qkv_ln_dense", device=DEV, M=256, H=256, N=512)
    M, H, N = inp["M"], inp["H"], inp["N"]
    qk = te.Quantizer(4096.0)
    kq = torch.empty(H, N, dtype=torch.uint8, device=DEV)
    te.te_quantize(inp["kernel"], qk, kq)
    outs = []
    for kernel in (inp["kernel"], kq):
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        qs = te.QuantizerSet(x=te.Quantizer(64.0), kernel1=te.Quantizer(4096.0))
        te.te_layernorm_dense_fwd(inp["x"], kernel, inp["gamma"], inp["beta"], inp["bias"], out,
                                  epsilon=inp["eps"], quantizer_set=qs)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_mlp_degenerate_inputs():
    # one row, and an empty batch
    for M in (1, 0):
        inp = make_inputs("gpt_ln_mlp", device=DEV, M=max(M, 1), H=256, F=512)
        x = inp["x"][:M]
        out = torch.empty(M, 256, dtype=torch.bfloat16, device=DEV)
        te.te_layernorm_mlp_fwd(x, inp["gamma"], inp["beta"], inp["w1"], inp["w2"], inp["b1"],
                                inp["b2"], out, activation_type="gelu", epsilon=1e-6)
        if M:
            ref = ob.layernorm_mlp_fwd(np64(x), np64(inp["gamma"]), np64(inp["beta"]),
                                       np64(inp["w1"]), np64(inp["w2"]), np64(inp["b1"]),
                                       np64(inp["b2"]), "layernorm", False, 1e-6, "gelu", "bf16")
            assert_gemm_close(out, ref["out"].value, 512, rms(ref["a"].value), rms(np64(inp["w2"])))


# -------------------------------------------------------------- full size, sampled rows ----

FULL = ["gpt_ln_mlp", "llama_rms_mlp"]


@pytest.mark.parametrize("name", FULL)
@pytest.mark.parametrize("fp8", [False, True])
def test_mlp_full_size_sampled(name, fp8):
    inp = make_inputs(name, device=DEV)
    got = run_mlp(inp, fp8=fp8)
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(inp["M"], size=48, replace=False))
    rows[-1] = inp["M"] - 1  # include the last (tail) row
    ref = oracle_mlp(inp, fp8=fp8, rows=rows)
    check_mlp(inp, got, ref, fp8=fp8, rows=rows)
    # properties over all rows: finite output, amax consistent with the stored codes
    assert torch.isfinite(got["out"].float()).all()
    if fp8:
        qs = got["qs"]
        deq_max = np.abs(nx.e4m3_decode(np.unique(codes(got["ln"])))).max() / MLP_SCALES["x"]
        assert abs(deq_max - qs.x.amax.item()) <= qs.x.amax.item() / 16


@pytest.mark.parametrize("fp8", [False, True])
def test_ln_dense_full_size_sampled(fp8):
    """The full QKV shape (16384 x 8192 -> 24576, 1% of rows x8), bf16 and FP8 (delayed
    scaling), in the launch configuration the benchmark times.  Sampled rows: the normalized
    operand (E4M3 codes under the one-step-flip rule), and the output both from the oracle's own
    chain (GEMM rule) and from the GPU's saved operand (the GEMM step given identical inputs,
    within its fp32 accumulation window).  The normalized output's amax over every row, in
    FP8 mode, to 1e-5."""
    inp = make_inputs("qkv_ln_dense", device=DEV)
    M, H, N = inp["M"], inp["H"], inp["N"]
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    ln = torch.empty(M, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)
    scales = dict(x=32.0, kernel=4096.0)
    qs = te.QuantizerSet(x=te.Quantizer(scales["x"]),
                         kernel1=te.Quantizer(scales["kernel"])) if fp8 else None
    te.te_layernorm_dense_fwd(inp["x"], inp["kernel"], inp["gamma"], inp["beta"], inp["bias"],
                              out, epsilon=inp["eps"], quantizer_set=qs, saved_ln_out=ln)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    rows = np.array([0, 1, 100, 5000, 8200, 12345, M - 1])  # rows 0 and 100 are the x8 rows
    x64 = np64(inp["x"])
    kern, gamma, beta, bias = (np64(inp[k]) for k in ("kernel", "gamma", "beta", "bias"))
    sc = {k: np.float32(v) for k, v in scales.items()} if fp8 else None
    # the oracle's forward on the sampled rows, step by step (the kernel's codes through the
    # pinned fast cast: the kernel is 201 M elements)
    y, _, _ = ob.norm_fwd(x64[rows], gamma, beta, "layernorm", False, inp["eps"])
    pre = nx.to_f32(y)
    got_ln = codes(ln)[rows] if fp8 else np64(ln)[rows]
    if fp8:
        ln_codes = nx.quantize(pre, sc["x"])
        assert_e4m3_codes(got_ln, ln_codes, pre32=pre, scale=sc["x"], rel=1e-5,
                          abs_tol=1e-5 * rms(pre), what="ln e4m3")
        alpha = ob.gemm_alpha(np.float32(1) / sc["x"], np.float32(1) / sc["kernel"])
        kv = decode(quantize_fast(kern, sc["kernel"]))
        a_ref = decode(ln_codes)
        a, w = a_ref * float(np.float32(1) / sc["x"]), kv * float(np.float32(1) / sc["kernel"])
        lv = decode(got_ln)
    else:
        alpha, kv = 1.0, kern  # kern holds bf16 values already
        a_ref = nx.bf16_round(pre)
        a, w = a_ref, kv
        lv = got_ln
    out_ref = nx.bf16_round(nx.to_f32(ob.gemm(a_ref, kv, bias, alpha)))
    assert_gemm_close(np64(out)[rows], out_ref, H, rms(a), rms(w), what="qkv out", stored="bf16")
    # the GEMM step from the GPU's own normalized operand
    v, wnd = gemm_ref(lv, kv, alpha)
    assert_in_window(np64(out)[rows], v + bias[None, :],
                     wnd + 2.0 ** -23 * (np.abs(v) + np.abs(bias)[None, :]),
                     "qkv out from the saved operand", stored="bf16")
    if fp8:
        amax = max(float(nx.amax_of(nx.to_f32(ob.norm_fwd(x64[r0:r0 + 2048], gamma, beta,
                                                          "layernorm", False, inp["eps"])[0])))
                   for r0 in range(0, M, 2048))
        assert abs(qs.x.amax.item() - amax) <= 1e-5 * amax
