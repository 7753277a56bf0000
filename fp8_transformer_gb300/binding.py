"""ctypes binding of libte_gb300.so (the C ABI declared in include/te_gb300.h).

Argument marshalling only: each function takes torch tensors, checks their dtype/shape against
the C signature, and passes raw device pointers and sizes.  Every step of the computation runs
in the library's CUDA kernels; there is no fallback.  A missing or unbuildable library raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

(TE_OK, TE_ERR_INVALID_ARG, TE_ERR_UNSUPPORTED, TE_ERR_CUDA, TE_ERR_TIMEOUT, TE_ERR_WORKSPACE,
 TE_ERR_TOO_LARGE) = range(7)
TE_F32, TE_BF16, TE_E4M3 = 0, 1, 2
TE_LAYERNORM, TE_RMSNORM = 0, 1
TE_IDENTITY, TE_RELU, TE_GELU, TE_SILU, TE_SWIGLU, TE_GEGLU, TE_REGLU = range(7)
TE_SCALING_DELAYED, TE_SCALING_CURRENT = 0, 1
(TE_OP_NORM_FWD, TE_OP_ACT_LU, TE_OP_DACT_DBIAS, TE_OP_LAYERNORM_DENSE_FWD,
 TE_OP_LAYERNORM_MLP_FWD, TE_OP_NORM_BWD, TE_OP_LAYERNORM_MLP_BWD,
 TE_OP_LAYERNORM_DENSE_BWD, TE_OP_LAYERNORM_MLP_FWD_HOST, TE_OP_GEMM) = range(10)

NORM_TYPES = {"layernorm": TE_LAYERNORM, "rmsnorm": TE_RMSNORM}
ACT_TYPES = {"identity": TE_IDENTITY, "relu": TE_RELU, "gelu": TE_GELU, "silu": TE_SILU,
             "swiglu": TE_SWIGLU, "geglu": TE_GEGLU, "reglu": TE_REGLU}
# the pages' activation_type tuples
ACT_TUPLES = {("relu",): "relu", ("gelu",): "gelu", ("silu",): "silu",
              ("silu", "linear"): "swiglu", ("gelu", "linear"): "geglu",
              ("relu", "linear"): "reglu"}

_DTYPE = {torch.float32: TE_F32, torch.bfloat16: TE_BF16, torch.uint8: TE_E4M3,
          torch.float8_e4m3fn: TE_E4M3}

EXPORTED = ["te_status_string", "te_version", "te_get_device_status", "te_workspace_size",
            "te_norm_fwd", "te_act_lu", "te_dact_dbias_quantize", "te_quantize", "te_gemm",
            "te_layernorm_dense_fwd", "te_layernorm_mlp_fwd", "te_norm_bwd",
            "te_profile_begin", "te_profile_end", "te_layernorm_mlp_bwd",
            "te_layernorm_dense_bwd",
            "te_dact_dbias_quantize_noalloc",
            "te_dact_dbias_noalloc_capacity", "te_selftest_wait_timeout",
            "te_layernorm_mlp_fwd_host", "te_update_scales", "te_stream_probe"]
KERNEL_KINDS = ["norm_fwd", "quantize", "act_lu", "dact_dbias", "gemm", "gemm_act", "norm_bwd",
                "transpose"]


class TEError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {msg}")
        self.status = status


class _Quantizer(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_void_p), ("scale_inv", ctypes.c_void_p),
                ("amax", ctypes.c_void_p), ("mode", ctypes.c_int32)]


class _QuantizerSet(ctypes.Structure):
    _fields_ = [("x", _Quantizer), ("kernel1", _Quantizer), ("act", _Quantizer),
                ("kernel2", _Quantizer), ("grad", _Quantizer)]


_lib = None
_lock = threading.Lock()

_vp, _i64, _f, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int32, ctypes.c_size_t
_QP = ctypes.POINTER(_Quantizer)
_QSP = ctypes.POINTER(_QuantizerSet)

_SIGS = {
    "te_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "te_version": (ctypes.c_int, []),
    "te_get_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32)]),
    "te_workspace_size": (_sz, [ctypes.c_int, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int]),
    "te_norm_fwd": (ctypes.c_int, [_vp, ctypes.c_int, _i64, _i64, _vp, _vp, ctypes.c_int,
                                   ctypes.c_int, _f, _QP, _vp, ctypes.c_int, _vp, _vp, _vp]),
    "te_act_lu": (ctypes.c_int, [_vp, ctypes.c_int, _i64, _i64, ctypes.c_int, _QP, _vp,
                                 ctypes.c_int, _vp]),
    "te_dact_dbias_quantize": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _i64, _i64, ctypes.c_int,
                                              _QP, _vp, ctypes.c_int, _vp, _vp, _sz, _vp]),
    "te_quantize": (ctypes.c_int, [_vp, ctypes.c_int, _i64, _i64, _QP, _vp, _vp]),
    "te_gemm": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int, _i64, _i64,
                               _i64, _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _sz,
                               _vp]),
    "te_layernorm_dense_fwd": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _vp, _vp, _vp,
                                              ctypes.c_int, ctypes.c_int, _f, _QSP, _i64, _i64,
                                              _i64, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _sz,
                                              _vp]),
    "te_layernorm_mlp_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp,
                                            ctypes.c_int, ctypes.c_int, _f, ctypes.c_int, _QSP,
                                            _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp,
                                            _vp, _vp, _vp, _sz, _vp]),
    "te_norm_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _i64, _i64,
                                   ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp, _sz, _vp]),
    "te_profile_begin": (ctypes.c_int, [ctypes.c_int32]),
    "te_layernorm_mlp_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp,
                                            _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _QSP,
                                            _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp, _vp,
                                            _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "te_selftest_wait_timeout": (ctypes.c_int, [_i64, _vp]),
    "te_layernorm_mlp_fwd_host": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_float, ctypes.c_int, _i64,
                                                 _i64, _i64, ctypes.c_int, _vp, ctypes.c_int, _vp,
                                                 _sz, _vp]),
    "te_layernorm_dense_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp,
                                              ctypes.c_int, ctypes.c_int, _QSP, _i64, _i64, _i64,
                                              ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                              _vp]),
    "te_dact_dbias_quantize_noalloc": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _i64, _i64,
                                                      ctypes.c_int, _QP, _vp, ctypes.c_int, _vp,
                                                      _vp]),
    "te_dact_dbias_noalloc_capacity": (_sz, []),
    "te_profile_end": (ctypes.c_int, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int32)]),
    "te_update_scales": (ctypes.c_int, [_QP, ctypes.c_int, _vp]),
    "te_stream_probe": (ctypes.c_int, [_vp, _vp, _sz, ctypes.c_int, _sz, _vp]),
}


def lib_path() -> str:
    return _build.LIB_PATH


def lib(build_if_stale: bool = True) -> ctypes.CDLL:
    """The loaded library; compiles it first when it is missing or older than its sources."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_stale and not _build.up_to_date():
                _build.build()
            if not os.path.exists(_build.LIB_PATH):
                raise ImportError(f"{_build.LIB_PATH} is missing: build it with "
                                  "fp8_transformer_gb300.build.build()")
            h = ctypes.CDLL(_build.LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def _check(fn: str, status: int):
    if status != TE_OK:
        msg = lib().te_status_string(status).decode()
        raise TEError(fn, status, msg)


def _host_ptr(t):
    """Host tensor for the host-buffer entry points (pinned memory lets the copies overlap)."""
    if t.is_cuda:
        raise ValueError("this argument is a host buffer")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the CUDA library must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _dt(t) -> int:
    return _DTYPE[t.dtype]


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class Quantizer:
    """Device scalars of one FP8 quantizer (scale, scale_inv, amax) and its scaling mode."""

    def __init__(self, scale=1.0, mode="delayed", device="cuda"):
        self.scale = torch.tensor([float(scale)], dtype=torch.float32, device=device)
        self.scale_inv = torch.tensor([1.0 / float(scale)], dtype=torch.float32, device=device)
        self.amax = torch.zeros(1, dtype=torch.float32, device=device)
        self.mode = TE_SCALING_CURRENT if mode == "current" else TE_SCALING_DELAYED

    @classmethod
    def from_tensors(cls, scale, scale_inv, amax, mode="delayed"):
        """A quantizer over caller-owned one-element fp32 tensors (e.g. views into a bank)."""
        q = cls.__new__(cls)
        q.scale, q.scale_inv, q.amax = scale, scale_inv, amax
        q.mode = TE_SCALING_CURRENT if mode == "current" else TE_SCALING_DELAYED
        return q

    def c(self) -> _Quantizer:
        return _Quantizer(self.scale.data_ptr(), self.scale_inv.data_ptr(), self.amax.data_ptr(),
                          self.mode)


class QuantizerSet:
    """The pages' QuantizerSet: quantizers for x, kernel1, act, kernel2 and grad."""

    def __init__(self, x=None, kernel1=None, act=None, kernel2=None, grad=None):
        self.x, self.kernel1, self.act, self.kernel2, self.grad = x, kernel1, act, kernel2, grad

    def c(self) -> _QuantizerSet:
        z = _Quantizer(None, None, None, 0)
        return _QuantizerSet(*(q.c() if q is not None else z
                               for q in (self.x, self.kernel1, self.act, self.kernel2, self.grad)))


def _qp(q):
    return ctypes.byref(q.c()) if q is not None else None


def status_string(status: int) -> str:
    return lib().te_status_string(status).decode()


def version() -> int:
    return lib().te_version()


def get_device_status() -> int:
    v = ctypes.c_int32(0)
    _check("te_get_device_status", lib().te_get_device_status(ctypes.byref(v)))
    return v.value


def selftest_wait_timeout(limit_us: int = 20000, stream=None):
    """Launch the library's bounded-wait self-test: a wait that nothing completes gives up after
    limit_us and records TE_ERR_TIMEOUT, which get_device_status() then returns."""
    _check("te_selftest_wait_timeout", lib().te_selftest_wait_timeout(int(limit_us), _stream(stream)))


def workspace_size(op, M, H, F_or_N, dtype=TE_BF16, quantized=False, kernel_dtype=None,
                   act=TE_IDENTITY) -> int:
    kd = dtype if kernel_dtype is None else kernel_dtype
    return int(lib().te_workspace_size(op, M, H, F_or_N, dtype, int(bool(quantized)), kd, act))


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def _act_id(act) -> int:
    if isinstance(act, tuple):
        act = ACT_TUPLES[act]
    return ACT_TYPES[act] if isinstance(act, str) else int(act)


def _norm_id(norm) -> int:
    return NORM_TYPES[norm] if isinstance(norm, str) else int(norm)


# -------------------------------------------------------------------------- entry points ---


def te_norm_fwd(x, gamma, beta, norm_type, zero_centered_gamma, epsilon, out, q=None, mu=None,
                rsigma=None, stream=None):
    M, H = x.shape
    st = lib().te_norm_fwd(_ptr(x), _dt(x), M, H, _ptr(gamma), _ptr(beta), _norm_id(norm_type),
                           int(bool(zero_centered_gamma)), float(epsilon), _qp(q), _ptr(out),
                           _dt(out), _ptr(mu), _ptr(rsigma), _stream(stream))
    _check("te_norm_fwd", st)
    return out


def te_act_lu(x, act, out, q=None, stream=None):
    M, N_in = x.shape
    st = lib().te_act_lu(_ptr(x), _dt(x), M, N_in, _act_id(act), _qp(q), _ptr(out), _dt(out),
                         _stream(stream))
    _check("te_act_lu", st)
    return out


def te_dact_dbias_quantize(dy, x_preact, act, dx, dbias=None, q=None, workspace=None,
                           stream=None):
    M, N_in = dx.shape
    a = _act_id(act)
    if dbias is not None and workspace is None:
        workspace = _ws(workspace_size(TE_OP_DACT_DBIAS, M, 0, N_in), dx.device)
    st = lib().te_dact_dbias_quantize(_ptr(dy), _ptr(x_preact), _dt(dy), M, N_in, a, _qp(q),
                                      _ptr(dx), _dt(dx), _ptr(dbias), _ptr(workspace),
                                      0 if workspace is None else workspace.numel(),
                                      _stream(stream))
    _check("te_dact_dbias_quantize", st)
    return dx


def te_quantize(x, q, out, stream=None):
    M, N = x.shape if x.dim() == 2 else (1, x.numel())
    st = lib().te_quantize(_ptr(x), _dt(x), M, N, _qp(q), _ptr(out), _stream(stream))
    _check("te_quantize", st)
    return out


def te_gemm(A, B, out, a_trans=False, b_trans=False, a_scale_inv=None, b_scale_inv=None,
            bias=None, workspace=None, split_k=True, stream=None):
    """split_k=False passes no workspace: no tile is split along K."""
    M = A.shape[1] if a_trans else A.shape[0]
    K = A.shape[0] if a_trans else A.shape[1]
    N = B.shape[0] if b_trans else B.shape[1]
    if workspace is None and split_k:
        n = workspace_size(TE_OP_GEMM, M, K, N, _dt(A))
        workspace = _ws(n, A.device) if n > 0 else None
    st = lib().te_gemm(_ptr(A), int(bool(a_trans)), _ptr(B), int(bool(b_trans)), _dt(A), M, N, K,
                       _ptr(a_scale_inv), _ptr(b_scale_inv), _ptr(bias),
                       _dt(bias) if bias is not None else TE_F32, _ptr(out), _dt(out),
                       _ptr(workspace), 0 if workspace is None else workspace.numel(),
                       _stream(stream))
    _check("te_gemm", st)
    return out


def te_layernorm_dense_fwd(x, kernel, gamma, beta, bias, out, norm_type="layernorm",
                           zero_centered_gamma=False, epsilon=1e-6, quantizer_set=None,
                           saved_ln_out=None, mu=None, rsigma=None, workspace=None, stream=None):
    M, H = x.shape
    N = kernel.shape[1]
    dt = _dt(x)
    kd = _dt(kernel)
    if workspace is None:
        workspace = _ws(workspace_size(TE_OP_LAYERNORM_DENSE_FWD, M, H, N, dt,
                                       quantizer_set is not None, kd), x.device)
    qs = quantizer_set.c() if quantizer_set is not None else None
    st = lib().te_layernorm_dense_fwd(_ptr(x), _ptr(kernel), kd, _ptr(gamma), _ptr(beta),
                                      _ptr(bias), _norm_id(norm_type), int(bool(zero_centered_gamma)),
                                      float(epsilon), ctypes.byref(qs) if qs is not None else None,
                                      M, H, N, dt, _ptr(out), _ptr(saved_ln_out), _ptr(mu),
                                      _ptr(rsigma), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
    _check("te_layernorm_dense_fwd", st)
    return out


def te_layernorm_mlp_fwd(x, gamma, beta, kernel1, kernel2, bias1, bias2, out,
                         norm_type="layernorm", zero_centered_gamma=False, epsilon=1e-6,
                         activation_type=("relu",), quantizer_set=None, saved_h=None,
                         saved_ln_out=None, mu=None, rsigma=None, workspace=None, stream=None,
                         saved_act=None):
    M, H = x.shape
    F = kernel2.shape[0]
    act = _act_id(activation_type)
    dt = _dt(x)
    kd = _dt(kernel1)
    if workspace is None:
        workspace = _ws(workspace_size(TE_OP_LAYERNORM_MLP_FWD, M, H, F, dt,
                                       quantizer_set is not None, kd, act), x.device)
    qs = quantizer_set.c() if quantizer_set is not None else None
    st = lib().te_layernorm_mlp_fwd(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(kernel1),
                                    _ptr(kernel2), kd, _ptr(bias1), _ptr(bias2),
                                    _norm_id(norm_type), int(bool(zero_centered_gamma)),
                                    float(epsilon), act,
                                    ctypes.byref(qs) if qs is not None else None, M, H, F, dt,
                                    _ptr(out), _ptr(saved_h), _ptr(saved_act),
                                    _ptr(saved_ln_out), _ptr(mu), _ptr(rsigma), _ptr(workspace),
                                    workspace.numel(), _stream(stream))
    _check("te_layernorm_mlp_fwd", st)
    return out


def te_layernorm_mlp_fwd_host(x_host, gamma, beta, kernel1, kernel2, bias1, bias2, out_host,
                              norm_type="layernorm", zero_centered_gamma=False, epsilon=1e-6,
                              activation_type=("relu",), chunks=4, workspace=None, stream=None):
    """te_layernorm_mlp_fwd with x and out in (pinned) host memory, copies overlapped with the
    compute of other row slices; the weights are device tensors."""
    M, H = x_host.shape
    F = kernel2.shape[0]
    act = _act_id(activation_type)
    dt = _dt(x_host)
    if workspace is None:
        workspace = _ws(workspace_size(TE_OP_LAYERNORM_MLP_FWD_HOST, M, H, F, dt, False, dt, act),
                        kernel1.device)
    st = lib().te_layernorm_mlp_fwd_host(_host_ptr(x_host), _ptr(gamma), _ptr(beta), _ptr(kernel1),
                                         _ptr(kernel2), _ptr(bias1), _ptr(bias2),
                                         _norm_id(norm_type), int(bool(zero_centered_gamma)),
                                         float(epsilon), act, M, H, F, dt, _host_ptr(out_host),
                                         int(chunks), _ptr(workspace), workspace.numel(),
                                         _stream(stream))
    _check("te_layernorm_mlp_fwd_host", st)
    return out_host


def te_layernorm_mlp_bwd(dy, x, gamma, kernel1, kernel2, saved_h, saved_ln_out, mu, rsigma,
                         dx, dgamma, dkernel1, dkernel2, dbeta=None, dbias1=None, dbias2=None,
                         norm_type="layernorm", zero_centered_gamma=False,
                         activation_type=("relu",), quantizer_set=None, workspace=None,
                         stream=None, saved_dh=None):
    M, H = x.shape
    F = kernel2.shape[0]
    act = _act_id(activation_type)
    dt = _dt(x)
    kd = _dt(kernel1)
    if workspace is None:
        workspace = _ws(workspace_size(TE_OP_LAYERNORM_MLP_BWD, M, H, F, dt,
                                       quantizer_set is not None, kd, act), x.device)
    qs = quantizer_set.c() if quantizer_set is not None else None
    st = lib().te_layernorm_mlp_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(kernel1), _ptr(kernel2),
                                    kd, _ptr(saved_h), _ptr(saved_ln_out), _ptr(mu), _ptr(rsigma),
                                    _norm_id(norm_type), int(bool(zero_centered_gamma)), act,
                                    ctypes.byref(qs) if qs is not None else None, M, H, F, dt,
                                    _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(dkernel1),
                                    _ptr(dkernel2), _ptr(dbias1), _ptr(dbias2), _ptr(saved_dh),
                                    _ptr(workspace), workspace.numel(), _stream(stream))
    _check("te_layernorm_mlp_bwd", st)
    return dx


def te_layernorm_dense_bwd(dy, x, gamma, kernel, saved_ln_out, mu, rsigma, dx, dgamma, dkernel,
                           dbeta=None, dbias=None, norm_type="layernorm", zero_centered_gamma=False,
                           quantizer_set=None, workspace=None, stream=None):
    M, H = x.shape
    N = kernel.shape[1]
    dt = _dt(x)
    kd = _dt(kernel)
    if workspace is None:
        workspace = _ws(workspace_size(TE_OP_LAYERNORM_DENSE_BWD, M, H, N, dt,
                                       quantizer_set is not None, kd), x.device)
    qs = quantizer_set.c() if quantizer_set is not None else None
    st = lib().te_layernorm_dense_bwd(_ptr(dy), _ptr(x), _ptr(gamma), _ptr(kernel), kd,
                                      _ptr(saved_ln_out), _ptr(mu), _ptr(rsigma),
                                      _norm_id(norm_type), int(bool(zero_centered_gamma)),
                                      ctypes.byref(qs) if qs is not None else None, M, H, N, dt,
                                      _ptr(dx), _ptr(dgamma), _ptr(dbeta), _ptr(dkernel),
                                      _ptr(dbias), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
    _check("te_layernorm_dense_bwd", st)
    return dx


def te_norm_bwd(dz, x, mu, rsigma, gamma, norm_type, zero_centered_gamma, dx, dgamma,
                dbeta=None, workspace=None, stream=None):
    M, H = x.shape
    if workspace is None:
        workspace = _ws(workspace_size(TE_OP_NORM_BWD, M, H, 0), x.device)
    st = lib().te_norm_bwd(_ptr(dz), _ptr(x), _ptr(mu), _ptr(rsigma), _ptr(gamma), _dt(x), M, H,
                           _norm_id(norm_type), int(bool(zero_centered_gamma)), _ptr(dx),
                           _ptr(dgamma), _ptr(dbeta), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _check("te_norm_bwd", st)
    return dx


def profile_begin(max_records: int = 4096):
    """Start timing every library kernel launch with CUDA events on its launching stream."""
    _check("te_profile_begin", lib().te_profile_begin(int(max_records)))


def stream_probe(src, dst=None, write_bytes=0, ratio=1, read_only_bytes=0, stream=None):
    """One launch of the library's streaming reference kernel (te_stream_probe)."""
    _check("te_stream_probe", lib().te_stream_probe(_ptr(src), _ptr(dst), int(write_bytes),
                                                     int(ratio), int(read_only_bytes),
                                                     _stream(stream)))


def profile_end() -> dict:
    """Stop timing; returns {kind: (total_ms, launches)} for the kernels launched since begin."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    _check("te_profile_end", lib().te_profile_end(ms, cnt))
    return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(KERNEL_KINDS)}


def te_update_scales(quantizers, stream=None):
    """scale = 448 / amax and scale_inv = 1 / scale on the device for every given quantizer
    (the delayed-scaling update between calls, e.g. after an amax all-reduce)."""
    qs = [q for q in quantizers if q is not None]
    arr = (_Quantizer * max(len(qs), 1))(*(q.c() for q in qs))
    _check("te_update_scales", lib().te_update_scales(arr, len(qs), _stream(stream)))


def te_dact_dbias_quantize_noalloc(dy, x_preact, act, dx, dbias=None, q=None, stream=None):
    """te_dact_dbias_quantize without a workspace: the bias reduction uses the library's fixed
    device scratch (see include/te_gb300.h for its capacity and sharing rules)."""
    M, N_in = dx.shape
    st = lib().te_dact_dbias_quantize_noalloc(_ptr(dy), _ptr(x_preact), _dt(dy), M, N_in,
                                              _act_id(act), _qp(q), _ptr(dx), _dt(dx),
                                              _ptr(dbias), _stream(stream))
    _check("te_dact_dbias_quantize_noalloc", st)
    return dx


def dact_dbias_noalloc_capacity() -> int:
    """Floats of fixed device scratch behind te_dact_dbias_quantize_noalloc."""
    return int(lib().te_dact_dbias_noalloc_capacity())
