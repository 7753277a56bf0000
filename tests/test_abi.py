"""The C-ABI library builds for sm_103a, loads, and exports every function include/*.h declares.

CPU-only: no function that launches work is called.
"""

import glob
import os
import re

import fp8_transformer_gb300 as te

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+(te_[a-z0-9_]+)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("te_norm_fwd", "te_act_lu", "te_dact_dbias_quantize", "te_layernorm_dense_fwd",
               "te_layernorm_mlp_fwd"):
        assert fn in names


def test_library_exports_every_declared_symbol():
    lib = te.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(te.EXPORTED) <= declared_functions()


def test_host_only_calls():
    assert te.version() == 200
    assert te.status_string(0) == "TE_OK"
    assert "timed out" in te.status_string(4)
    b = te.binding
    ws = te.workspace_size(b.TE_OP_LAYERNORM_MLP_FWD, 8192, 4096, 14336, b.TE_BF16, True,
                           b.TE_BF16, b.TE_SWIGLU)
    # ln (E4M3) + act (E4M3) + act staging (fp32) + E4M3 copies of both kernels
    expect = 8192 * 4096 + 8192 * 14336 + 8192 * 14336 * 4 + 4096 * 28672 + 14336 * 4096
    assert expect <= ws <= expect + 5 * 256
    assert te.workspace_size(b.TE_OP_LAYERNORM_MLP_FWD, 8192, 4096, 14336, b.TE_BF16, True,
                             b.TE_E4M3, b.TE_SWIGLU) < ws


def test_invalid_arguments_rejected_before_launch():
    lib = te.lib()
    b = te.binding
    # NULL x with M > 0, and a bad enum: both refused on the host, nothing launched
    assert lib.te_norm_fwd(None, b.TE_BF16, 4, 128, None, None, 0, 0, 1e-5, None, None,
                           b.TE_BF16, None, None, None) == b.TE_ERR_INVALID_ARG
    assert lib.te_act_lu(None, b.TE_BF16, 0, 16, 99, None, None, b.TE_BF16,
                         None) == b.TE_ERR_INVALID_ARG
    # misaligned pointers and row lengths that are not whole 16-byte vectors
    assert lib.te_quantize(8, b.TE_BF16, 1, 12, None, 16, None) == b.TE_ERR_INVALID_ARG
    assert lib.te_gemm(16, 0, 32, 0, b.TE_BF16, 16, 24, 16, None, None, None, b.TE_F32, 64,
                       b.TE_BF16, None, 0, None) == b.TE_ERR_UNSUPPORTED
    assert lib.te_gemm(18, 0, 32, 0, b.TE_BF16, 16, 32, 16, None, None, None, b.TE_F32, 64,
                       b.TE_BF16, None, 0, None) == b.TE_ERR_UNSUPPORTED
    # the streaming reference: bad ratio, misaligned pointer, byte count not a multiple of 16
    assert lib.te_stream_probe(16, 32, 64, 0, 0, None) == b.TE_ERR_INVALID_ARG
    assert lib.te_stream_probe(16, 40, 64, 2, 0, None) == b.TE_ERR_INVALID_ARG
    assert lib.te_stream_probe(16, 32, 0, 1, 24, None) == b.TE_ERR_INVALID_ARG
    # a misaligned split-K workspace
    assert lib.te_gemm(16, 0, 32, 0, b.TE_BF16, 16, 32, 16, None, None, None, b.TE_F32, 64,
                       b.TE_BF16, 72, 4096, None) == b.TE_ERR_UNSUPPORTED


def test_selftest_limit_checked_on_the_host():
    lib = te.lib()
    b = te.binding
    for bad in (0, -5, 1000001):
        assert lib.te_selftest_wait_timeout(bad, None) == b.TE_ERR_INVALID_ARG


def test_backward_and_host_forward_arguments_checked_on_the_host():
    """The whole-block entry points refuse bad arguments before any CUDA call (fake, aligned,
    never dereferenced addresses stand in for device buffers)."""
    lib = te.lib()
    b = te.binding
    P = 4096  # a 16-byte aligned stand-in address; nothing reads it

    def mlp_bwd(dtype=b.TE_BF16, act=b.TE_GELU, H=512, F=784, gamma=P, saved_dh=None):
        return lib.te_layernorm_mlp_bwd(P, P, gamma, P, P, dtype, P, P, P, P, b.TE_LAYERNORM, 0,
                                        act, None, 64, H, F, dtype, P, P, P, P, P, P, P, P,
                                        saved_dh, 1 << 20, None)
    assert mlp_bwd(dtype=b.TE_F32) == b.TE_ERR_UNSUPPORTED       # bf16 only
    assert mlp_bwd(act=b.TE_IDENTITY) == b.TE_ERR_INVALID_ARG    # the MLP needs an activation
    assert mlp_bwd(gamma=None) == b.TE_ERR_INVALID_ARG
    assert mlp_bwd(H=520) == b.TE_ERR_UNSUPPORTED                # H not a multiple of 16
    assert mlp_bwd(saved_dh=P + 8) == b.TE_ERR_UNSUPPORTED       # optional output misaligned

    def mlp_fwd(saved_act=None, act=b.TE_SWIGLU):
        return lib.te_layernorm_mlp_fwd(P, P, P, P, P, b.TE_BF16, None, None, b.TE_RMSNORM, 1,
                                        1e-6, act, None, 64, 512, 784, b.TE_BF16, P, None,
                                        saved_act, None, None, None, P, 1 << 30, None)
    assert mlp_fwd(saved_act=P + 8) == b.TE_ERR_UNSUPPORTED
    assert mlp_fwd(act=b.TE_IDENTITY) == b.TE_ERR_INVALID_ARG

    def dense_bwd(dtype=b.TE_BF16, N=784, gamma=P):
        return lib.te_layernorm_dense_bwd(P, P, gamma, P, dtype, P, P, P, b.TE_LAYERNORM, 0, None,
                                          64, 512, N, dtype, P, P, P, P, P, P, 1 << 20, None)
    assert dense_bwd(dtype=b.TE_F32) == b.TE_ERR_UNSUPPORTED
    assert dense_bwd(gamma=None) == b.TE_ERR_INVALID_ARG
    assert dense_bwd(N=792) == b.TE_ERR_UNSUPPORTED              # N not a multiple of 16

    def host_fwd(M=64, chunks=4, dtype=b.TE_BF16):
        return lib.te_layernorm_mlp_fwd_host(P, P, P, P, P, None, None, b.TE_RMSNORM, 1, 1e-6,
                                             b.TE_SWIGLU, M, 512, 784, dtype, P, chunks, P,
                                             1 << 20, None)
    assert host_fwd(chunks=0) == b.TE_ERR_INVALID_ARG
    assert host_fwd(chunks=17) == b.TE_ERR_INVALID_ARG           # at most 16 row slices
    assert host_fwd(dtype=b.TE_E4M3) == b.TE_ERR_INVALID_ARG     # activations bf16 or fp32
    assert host_fwd(M=0) == b.TE_OK                              # no rows: nothing to do
