"""te_layernorm_mlp_fwd_host: the LayerNorm MLP forward from pinned host buffers, its row slices'
copies overlapped with the compute of the others.

Each row's result does not depend on how the rows are cut, so with no GEMM tile split along K
(TE_GEMM_SPLIT_K=0) the output must equal, bit for bit, te_layernorm_mlp_fwd on device buffers
-- for every slice count, including ragged last slices -- and the small case is also held to the
oracle.  With splitting (the default) a slice's GEMMs have their own tile counts, so other tiles
are split than in the whole-batch call and the fp32 sums round differently: the full-size run
then holds sampled rows, the slice edges among them, to the oracle.
"""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from oracle import block as ob
from parity import assert_gemm_close, np64, rms
from workloads import make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def device_forward(inp):
    out = torch.empty(inp["M"], inp["H"], dtype=inp["x"].dtype, device=DEV)
    te.te_layernorm_mlp_fwd(inp["x"], inp["gamma"], inp["beta"], inp["w1"], inp["w2"],
                            inp.get("b1"), inp.get("b2"), out, norm_type=inp["norm"],
                            zero_centered_gamma=inp["zero_centered_gamma"], epsilon=inp["eps"],
                            activation_type=inp["act"])
    return out


def host_forward(inp, chunks):
    x_host = inp["x"].cpu().pin_memory()
    out_host = torch.full((inp["M"], inp["H"]), float("nan"), dtype=inp["x"].dtype).pin_memory()
    te.te_layernorm_mlp_fwd_host(x_host, inp["gamma"], inp["beta"], inp["w1"], inp["w2"],
                                 inp.get("b1"), inp.get("b2"), out_host, norm_type=inp["norm"],
                                 zero_centered_gamma=inp["zero_centered_gamma"],
                                 epsilon=inp["eps"], activation_type=inp["act"], chunks=chunks)
    torch.cuda.synchronize()
    return out_host


@pytest.mark.parametrize("name,shape", [("gpt_ln_mlp", dict(M=300, H=512, F=784)),
                                        ("llama_rms_mlp", dict(M=300, H=512, F=784)),
                                        ("tiny_ln_mlp", {})])
@pytest.mark.parametrize("chunks", [1, 3, 16])
def test_host_forward_equals_device_forward(name, shape, chunks, monkeypatch):
    monkeypatch.setenv("TE_GEMM_SPLIT_K", "0")
    inp = make_inputs(name, device=DEV, **shape)
    want = device_forward(inp).cpu()
    got = host_forward(inp, chunks)
    assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got,
                       want.view(torch.int16) if want.dtype == torch.bfloat16 else want)
    if name == "llama_rms_mlp" and chunks == 3:
        ref = ob.layernorm_mlp_fwd(np64(inp["x"]), np64(inp["gamma"]), None, np64(inp["w1"]),
                                   np64(inp["w2"]), None, None, "rmsnorm", True, inp["eps"],
                                   "swiglu", "bf16")
        a2 = ref["a"].value
        assert_gemm_close(got, ref["out"].value, inp["F"], rms(a2), rms(np64(inp["w2"])),
                          what="out")


def test_host_forward_full_size(monkeypatch):
    """The Llama benchmark shape (8192 tokens): bit-equal to the device-buffer forward without
    K splits; with them, sampled rows (the first and last of every slice among them) against
    the oracle."""
    inp = make_inputs("llama_rms_mlp", device=DEV)
    monkeypatch.setenv("TE_GEMM_SPLIT_K", "0")
    want = device_forward(inp).cpu()
    got = host_forward(inp, 4)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    monkeypatch.delenv("TE_GEMM_SPLIT_K")
    got = host_forward(inp, 4)
    M = inp["M"]
    edges = [0, 511, 512, 4095, 4096, 7679, 7680, M - 1]  # slices of 512, 3584, 3584, 512 rows
    rows = np.unique(np.concatenate([edges, np.random.default_rng(7).choice(M, 8, replace=False)]))
    ref = ob.layernorm_mlp_fwd(np64(inp["x"])[rows], np64(inp["gamma"]), None, np64(inp["w1"]),
                               np64(inp["w2"]), None, None, "rmsnorm", True, inp["eps"], "swiglu",
                               "bf16")
    assert_gemm_close(np64(got)[rows], ref["out"].value, inp["F"], rms(ref["a"].value),
                      rms(np64(inp["w2"])), what="host forward out, split K", stored="bf16")
