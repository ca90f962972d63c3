"""Python binding of libgf's C ABI (``include/gf.h``).

Argument marshalling only: each function checks that its tensors are CUDA,
float32 and contiguous (the pages' host wrappers check the same), takes their
device pointers and the current torch stream, sizes the workspace with the
matching ``*_workspace_size`` query and calls the C entry point of the same
name.  All arithmetic runs in the library's CUDA kernels; if ``libgf.so`` is
missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgf.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "gf.h")

GF_MODE_FP32_3XTF32 = 0
GF_MODE_BF16 = 1
GF_MODE_FP32_3XBF16 = 2
GF_FLAG_GELU_TANH = 0x100  # OR'd into the Conv1d chain's mode: tanh-approximate GELU
GF_FLAG_FUSED_PRODUCER = 0x200  # OR'd into the Conv1d chain's mode: LayerNorm + GELU inside the GEMM
GF_CHAIN_GROUPNORM, GF_CHAIN_LSE, GF_CHAIN_LINEAR = 0, 1, 2  # gf_linear_tile_width's chains

_lib = None
_lock = threading.Lock()

_P, _I64, _I32, _F, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t

_SIGS = {
    "gf_abi_version": (_I32, []),
    "gf_status_string": (ctypes.c_char_p, [_I32]),
    "gf_device_status": (_I32, [ctypes.POINTER(ctypes.c_int32)]),
    "gf_profile_begin": (_I32, [_I32]),
    "gf_profile_end": (_I32, [ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_float)]),
    "gf_measure_tensor_rate": (_I32, [_I32, _I32, _I32, ctypes.POINTER(ctypes.c_double)]),
    "gf_linear_tile_width": (_I32, [_I32, _I64, _I64, _I32, _I32, _I32]),
    "gf_testing_host_pipeline_trace": (_I32, [_I64, _I32, ctypes.c_char_p, _SZ]),
    "gf_linear_workspace_size": (_SZ, [_I64, _I64, _I64, _I32]),
    "gf_linear": (_I32, [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _SZ, _P]),
    "gf_linear_swish_bias_groupnorm_workspace_size": (_SZ, [_I64, _I64, _I64, _I32, _I32]),
    "gf_linear_swish_bias_groupnorm": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _F, _I32,
                                              _P, _SZ, _P]),
    "gf_linear_swish_bias_groupnorm_planes": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _F,
                                                     _P]),
    "gf_tf32_split": (_I32, [_P, _P, _I64, _P]),
    "gf_linear_swish_bias_groupnorm_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I32, _I32, _I64]),
    "gf_linear_swish_bias_groupnorm_host": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _F, _I32,
                                                   _I64, _P, _SZ, _P]),
    "gf_linear_lse_act_workspace_size": (_SZ, [_I64, _I64, _I64, _I32]),
    "gf_linear_lse_act": (_I32, [_P, _P, _P, _P, _I64, _I64, _I64, _F, _I32, _P, _SZ, _P]),
    "gf_ln_gelu_dconv1d_res_workspace_size": (_SZ, [_I64, _I64, _I64, _I32, _I32, _I32]),
    "gf_ln_gelu_dconv1d_res": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I32, _I32, _F, _I32,
                                      _P, _SZ, _P]),
    "gf_convt3d_swish_gn_hswish_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I64, _I32, _I32, _I32,
                                                        _I32]),
    "gf_convt3d_swish_gn_hswish": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I32,
                                          _I32, _I32, _I32, _F, _P, _SZ, _P]),
    "gf_ln_gelu_dconv1d_res_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I32, _I32, _I32, _I64]),
    "gf_ln_gelu_dconv1d_res_host": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I32, _I32, _F, _I32,
                                           _I64, _P, _SZ, _P]),
    "gf_convt3d_swish_gn_hswish_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I64, _I32, _I32,
                                                             _I32, _I32, _I64]),
    "gf_convt3d_swish_gn_hswish_host": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I32,
                                               _I32, _I32, _I32, _F, _I64, _P, _SZ, _P]),
    "gf_convt3d_noalloc_scratch_limit": (_SZ, []),
    "gf_convt3d_swish_gn_hswish_noalloc_scratch_size": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I64, _I32, _I32,
                                                              _I32, _I32]),
    "gf_convt3d_swish_gn_hswish_noalloc": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                                  _I32, _I32, _I32, _I32, _F, _P]),
}


class GFError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


def lib() -> ctypes.CDLL:
    """Load libgf.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libgf.so is not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions that include/gf.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gf_[a-z0-9_]+)\s*\(", text)))


def linear_tile_width(chain: int, M: int, N: int, groups: int, mode: int, sm_count: int) -> int:
    """The GEMM tile width the Linear chains' dispatch picks (host arithmetic
    only; 0 for invalid arguments)."""
    return lib().gf_linear_tile_width(chain, M, N, groups, mode, sm_count)


def measure_tensor_rate(kind: str, iters: int = 4096, repeats: int = 5) -> float:
    """The tensor pipe's measured dense rate in TFLOP/s for kind "tf32" or
    "bf16" (gf_measure_tensor_rate; synchronises)."""
    out = ctypes.c_double(0.0)
    st = lib().gf_measure_tensor_rate({"tf32": 0, "bf16": 1}[kind], iters, repeats, ctypes.byref(out))
    if st != 0:
        raise GFError(st, "gf_measure_tensor_rate")
    return out.value


def host_pipeline_trace(nchunks: int, fail_at: int = -1) -> tuple[int, str]:
    """(status, steps) of the host-buffer pipeline's schedule run against a
    recorder that fails at step fail_at (-1: none).  No device is touched."""
    buf = ctypes.create_string_buffer(64 * (3 * nchunks + 4))
    st = lib().gf_testing_host_pipeline_trace(nchunks, fail_at, buf, len(buf))
    return st, buf.value.decode()


def status_string(status: int) -> str:
    try:
        return lib().gf_status_string(status).decode()
    except Exception:  # pragma: no cover
        return "?"


def gf_device_status() -> int:
    """Synchronise and return (and clear) the device status bits."""
    bits = ctypes.c_int32(0)
    st = lib().gf_device_status(ctypes.byref(bits))
    if st not in (0, -8):
        raise GFError(st, "gf_device_status")
    return bits.value


class profile:
    """Context manager: time the dominant kernel of every library call made
    inside it (CUDA events recorded by the library on the call's stream).
    After exit, ``.calls`` and ``.total_ms`` hold the count and summed time."""

    def __init__(self, max_calls=100000):
        self.max_calls = max_calls
        self.calls = 0
        self.total_ms = 0.0

    def __enter__(self):
        st = lib().gf_profile_begin(self.max_calls)
        if st != 0:
            raise GFError(st, "gf_profile_begin")
        return self

    def __exit__(self, *exc):
        c, t = ctypes.c_int32(0), ctypes.c_float(0.0)
        st = lib().gf_profile_end(ctypes.byref(c), ctypes.byref(t))
        self.calls, self.total_ms = c.value, t.value
        if st != 0 and exc[0] is None:
            raise GFError(st, "gf_profile_end")
        return False

    @property
    def mean_ms(self):
        return self.total_ms / self.calls if self.calls else float("nan")


# --------------------------------------------------------------- plumbing
_ws_cache: dict = {}


def _workspace(device: torch.device, nbytes: int, stream=None):
    """Cached scratch buffer per (device, stream), grown on demand.  Calls on
    one stream are ordered, so they can share one buffer; calls on different
    streams get different buffers.  A buffer made for a stream other than
    the current one is recorded on that stream, so that the allocator does
    not hand its memory out again (after it is replaced) before the work
    queued there is done."""
    if nbytes == 0:
        return None
    index = device.index if device.index is not None else torch.cuda.current_device()
    s = stream if stream is not None else torch.cuda.current_stream(index)
    key = (index, s.cuda_stream)
    with _lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
            if s.cuda_stream != torch.cuda.current_stream(index).cuda_stream:
                buf.record_stream(s)
            _ws_cache[key] = buf
    return buf


def release_workspaces() -> int:
    """Drop the cached workspace buffers (all devices and streams) and return
    how many there were.  Safe while work that uses them is still queued:
    each buffer was allocated on, or recorded on, the stream it serves, so
    torch's allocator does not reuse its memory before that work is done."""
    with _lock:
        n = len(_ws_cache)
        _ws_cache.clear()
    return n


def _check(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
        if t.dtype != torch.float32:
            raise ValueError("tensors must be float32")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("tensors must be on one device")
    return dev


def _shape(t, shape, name):
    """Raise unless t (if given) has exactly this shape: the sizes passed to
    the library come from the leading operands, so every other tensor must
    agree with them or the kernels would read or write past its end."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _numel(t, n, name):
    """Raise unless t (if given) holds exactly n elements (any shape)."""
    if t is not None and t.numel() != n:
        raise ValueError(f"{name} holds {t.numel()} elements, expected {n}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise GFError(st, name)


def _gn_vectors(N, b_lin, bias, gamma, beta):
    for t, name in ((b_lin, "b_lin"), (bias, "bias"), (gamma, "gamma"), (beta, "beta")):
        _numel(t, N, name)


def _ws_args(device, nbytes, workspace, stream=None):
    if workspace is None:
        workspace = _workspace(device, nbytes, stream)
    elif workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace too small")
    return (None if workspace is None else workspace.data_ptr()), nbytes


# -------------------------------------------------------------- the ABI
def gf_linear(x, W, b=None, mode=GF_MODE_FP32_3XTF32, out=None, workspace=None, stream=None):
    """out[M, N] = x @ W.T + b (the contraction step alone)."""
    M, K = x.shape
    N = W.shape[0]
    _shape(W, (N, K), "W")
    _numel(b, N, "b")
    _shape(out, (M, N), "out")
    dev = _check(x, W, b, out)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        nbytes = lib().gf_linear_workspace_size(M, K, N, mode)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_linear", _ptr(x), _ptr(W), _ptr(b), _ptr(out), M, K, N, mode, wp, nb, _stream_ptr(stream))
    return out


def gf_linear_swish_bias_groupnorm(x, W, b_lin, bias, gamma, beta, groups, eps=1e-5,
                                   mode=GF_MODE_FP32_3XTF32, out=None, workspace=None, stream=None):
    """out[M, N] = GroupNorm(groups)(swish(x @ W.T + b_lin) + bias) * gamma + beta."""
    M, K = x.shape
    N = W.shape[0]
    _shape(W, (N, K), "W")
    _gn_vectors(N, b_lin, bias, gamma, beta)
    _shape(out, (M, N), "out")
    dev = _check(x, W, b_lin, bias, gamma, beta, out)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        nbytes = lib().gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, groups, mode)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_linear_swish_bias_groupnorm", _ptr(x), _ptr(W), _ptr(b_lin), _ptr(bias), _ptr(gamma),
              _ptr(beta), _ptr(out), M, K, N, groups, eps, mode, wp, nb, _stream_ptr(stream))
    return out


def gf_tf32_split(src, planes=None, stream=None):
    """planes[0] = src with the 13 low mantissa bits cleared, planes[1] = src - planes[0]."""
    _shape(planes, (2,) + tuple(src.shape), "planes")
    dev = _check(src, planes)
    if planes is None:
        planes = torch.empty((2,) + tuple(src.shape), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _call("gf_tf32_split", _ptr(src), _ptr(planes), src.numel(), _stream_ptr(stream))
    return planes


def gf_linear_swish_bias_groupnorm_planes(x_planes, W_planes, b_lin, bias, gamma, beta, groups, eps=1e-5, out=None,
                                          stream=None):
    """gf_linear_swish_bias_groupnorm on pre-split operands (x_planes [2,M,K], W_planes [2,N,K])."""
    _, M, K = x_planes.shape
    N = W_planes.shape[1]
    _shape(x_planes, (2, M, K), "x_planes")
    _shape(W_planes, (2, N, K), "W_planes")
    _gn_vectors(N, b_lin, bias, gamma, beta)
    _shape(out, (M, N), "out")
    dev = _check(x_planes, W_planes, b_lin, bias, gamma, beta, out)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _call("gf_linear_swish_bias_groupnorm_planes", _ptr(x_planes), _ptr(W_planes), _ptr(b_lin), _ptr(bias),
              _ptr(gamma), _ptr(beta), _ptr(out), M, K, N, groups, eps, _stream_ptr(stream))
    return out


def gf_linear_swish_bias_groupnorm_host(x_host, W, b_lin, bias, gamma, beta, groups, eps=1e-5,
                                        mode=GF_MODE_FP32_3XTF32, out_host=None, chunk_rows=0, workspace=None,
                                        stream=None):
    """gf_linear_swish_bias_groupnorm on host tensors: x_host (CPU, float32,
    ideally pinned) in, out_host (CPU) out; the weights are CUDA tensors.
    Chunks of rows are copied in, computed and copied out in an overlapped
    pipeline.  Enqueues and returns; synchronise the stream before reading
    out_host."""
    M, K = x_host.shape
    N = W.shape[0]
    _shape(W, (N, K), "W")
    _gn_vectors(N, b_lin, bias, gamma, beta)
    _shape(out_host, (M, N), "out_host")
    dev = _check(W, b_lin, bias, gamma, beta)
    for t in (x_host, out_host):
        if t is not None and (t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError("host tensors must be contiguous float32 CPU tensors")
    if out_host is None:
        out_host = torch.empty((M, N), dtype=torch.float32, pin_memory=x_host.is_pinned())
    with torch.cuda.device(dev):
        nbytes = lib().gf_linear_swish_bias_groupnorm_host_workspace_size(M, K, N, groups, mode, chunk_rows)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_linear_swish_bias_groupnorm_host", x_host.data_ptr(), _ptr(W), _ptr(b_lin), _ptr(bias),
              _ptr(gamma), _ptr(beta), out_host.data_ptr(), M, K, N, groups, eps, mode, chunk_rows, wp, nb,
              _stream_ptr(stream))
    return out_host


def gf_linear_lse_act(x, W, b, negative_slope=0.01, mode=GF_MODE_FP32_3XTF32, out=None, workspace=None,
                      stream=None):
    """out[M, 1] = gelu(gelu(lrelu(lrelu(logsumexp(x @ W.T + b, dim=1)))))."""
    M, K = x.shape
    N = W.shape[0]
    _shape(W, (N, K), "W")
    _numel(b, N, "b")
    _numel(out, M, "out")
    dev = _check(x, W, b, out)
    if out is None:
        out = torch.empty((M, 1), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        nbytes = lib().gf_linear_lse_act_workspace_size(M, K, N, mode)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_linear_lse_act", _ptr(x), _ptr(W), _ptr(b), _ptr(out), M, K, N, negative_slope, mode, wp, nb,
              _stream_ptr(stream))
    return out


def gf_ln_gelu_dconv1d_res(x, ln_gamma, ln_beta, conv_w, conv_b, dilation, padding, eps=1e-5,
                           mode=GF_MODE_FP32_3XTF32, out=None, workspace=None, stream=None, gelu="erf",
                           fused_producer=False):
    """out = conv1d(gelu(layer_norm(x, [C, L])), dilation, padding) + x.
    gelu: "erf" (exact) or "tanh" (the tanh approximation).  fused_producer:
    LayerNorm + GELU inside the GEMM (no activation planes in the
    workspace; slower)."""
    if gelu not in ("erf", "tanh"):
        raise ValueError("gelu must be 'erf' or 'tanh'")
    if gelu == "tanh":
        mode |= GF_FLAG_GELU_TANH
    if fused_producer:
        mode |= GF_FLAG_FUSED_PRODUCER
    B, C, L = x.shape
    ksize = conv_w.shape[2]
    _shape(conv_w, (C, C, ksize), "conv_w")
    _numel(ln_gamma, C * L, "ln_gamma")
    _numel(ln_beta, C * L, "ln_beta")
    _numel(conv_b, C, "conv_b")
    _shape(out, (B, C, L), "out")
    dev = _check(x, ln_gamma, ln_beta, conv_w, conv_b, out)
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(dev):
        nbytes = lib().gf_ln_gelu_dconv1d_res_workspace_size(B, C, L, ksize, dilation, mode)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_ln_gelu_dconv1d_res", _ptr(x), _ptr(ln_gamma), _ptr(ln_beta), _ptr(conv_w), _ptr(conv_b),
              _ptr(out), B, C, L, ksize, dilation, padding, eps, mode, wp, nb, _stream_ptr(stream))
    return out


def _host_tensors(*ts):
    for t in ts:
        if t is not None and (t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError("host tensors must be contiguous float32 CPU tensors")


def gf_ln_gelu_dconv1d_res_host(x_host, ln_gamma, ln_beta, conv_w, conv_b, dilation, padding, eps=1e-5,
                                mode=GF_MODE_FP32_3XTF32, out_host=None, chunk_samples=0, workspace=None, stream=None,
                                gelu="erf"):
    """gf_ln_gelu_dconv1d_res on host tensors: x_host (CPU, float32, ideally
    pinned) in, out_host (CPU) out; the parameters are CUDA tensors.  Chunks
    of whole samples are copied in, computed and copied out in an overlapped
    pipeline.  Enqueues and returns; synchronise the stream before reading
    out_host."""
    if gelu not in ("erf", "tanh"):
        raise ValueError("gelu must be 'erf' or 'tanh'")
    if gelu == "tanh":
        mode |= GF_FLAG_GELU_TANH
    B, C, L = x_host.shape
    ksize = conv_w.shape[2]
    _shape(conv_w, (C, C, ksize), "conv_w")
    _numel(ln_gamma, C * L, "ln_gamma")
    _numel(ln_beta, C * L, "ln_beta")
    _numel(conv_b, C, "conv_b")
    _shape(out_host, (B, C, L), "out_host")
    dev = _check(ln_gamma, ln_beta, conv_w, conv_b)
    _host_tensors(x_host, out_host)
    if out_host is None:
        out_host = torch.empty((B, C, L), dtype=torch.float32, pin_memory=x_host.is_pinned())
    with torch.cuda.device(dev):
        nbytes = lib().gf_ln_gelu_dconv1d_res_host_workspace_size(B, C, L, ksize, dilation, mode, chunk_samples)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_ln_gelu_dconv1d_res_host", x_host.data_ptr(), _ptr(ln_gamma), _ptr(ln_beta), _ptr(conv_w),
              _ptr(conv_b), out_host.data_ptr(), B, C, L, ksize, dilation, padding, eps, mode, chunk_samples, wp, nb,
              _stream_ptr(stream))
    return out_host


def convt3d_out_shape(x_shape, Cout, k, stride, pad):
    N, _, D, H, W = x_shape
    f = lambda i: (i - 1) * stride - 2 * pad + k  # noqa: E731
    return (N, Cout, f(D), f(H), f(W))


def _convt3d_shapes(x, w, b, gamma, beta, out, stride, pad):
    Cin, Cout, k = x.shape[1], w.shape[1], w.shape[2]
    _shape(w, (Cin, Cout, k, k, k), "w")
    _numel(b, Cout, "b")
    _numel(gamma, Cout, "gamma")
    _numel(beta, Cout, "beta")
    _shape(out, convt3d_out_shape(x.shape, Cout, k, stride, pad), "out")


def gf_convt3d_swish_gn_hswish(x, w, b, gamma, beta, stride, pad, groups, eps=1e-5, out=None, workspace=None,
                               stream=None):
    """out = hardswish(GroupNorm(groups)(swish(conv_transpose3d(x, w, b, stride, pad))))."""
    N, Cin, D, H, W = x.shape
    Cout, k = w.shape[1], w.shape[2]
    _convt3d_shapes(x, w, b, gamma, beta, out, stride, pad)
    dev = _check(x, w, b, gamma, beta, out)
    if out is None:
        out = torch.empty(convt3d_out_shape(x.shape, Cout, k, stride, pad), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        nbytes = lib().gf_convt3d_swish_gn_hswish_workspace_size(N, Cin, Cout, D, H, W, k, stride, pad, groups)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_convt3d_swish_gn_hswish", _ptr(x), _ptr(w), _ptr(b), _ptr(gamma), _ptr(beta), _ptr(out),
              N, Cin, Cout, D, H, W, k, stride, pad, groups, eps, wp, nb, _stream_ptr(stream))
    return out


def gf_convt3d_swish_gn_hswish_host(x_host, w, b, gamma, beta, stride, pad, groups, eps=1e-5, out_host=None,
                                    chunk_samples=0, workspace=None, stream=None):
    """gf_convt3d_swish_gn_hswish on host tensors: x_host (CPU, float32,
    ideally pinned) in, out_host (CPU) out; the parameters are CUDA tensors.
    Chunks of whole samples are copied in, computed and copied out in an
    overlapped pipeline.  Enqueues and returns; synchronise the stream before
    reading out_host."""
    N, Cin, D, H, W = x_host.shape
    Cout, k = w.shape[1], w.shape[2]
    _shape(w, (Cin, Cout, k, k, k), "w")
    _numel(b, Cout, "b")
    _numel(gamma, Cout, "gamma")
    _numel(beta, Cout, "beta")
    oshape = convt3d_out_shape(x_host.shape, Cout, k, stride, pad)
    _shape(out_host, oshape, "out_host")
    dev = _check(w, b, gamma, beta)
    _host_tensors(x_host, out_host)
    if out_host is None:
        out_host = torch.empty(oshape, dtype=torch.float32, pin_memory=x_host.is_pinned())
    with torch.cuda.device(dev):
        nbytes = lib().gf_convt3d_swish_gn_hswish_host_workspace_size(N, Cin, Cout, D, H, W, k, stride, pad, groups,
                                                                     chunk_samples)
        wp, nb = _ws_args(dev, nbytes, workspace, stream)
        _call("gf_convt3d_swish_gn_hswish_host", x_host.data_ptr(), _ptr(w), _ptr(b), _ptr(gamma), _ptr(beta),
              out_host.data_ptr(), N, Cin, Cout, D, H, W, k, stride, pad, groups, eps, chunk_samples, wp, nb,
              _stream_ptr(stream))
    return out_host


def gf_convt3d_swish_gn_hswish_noalloc(x, w, b, gamma, beta, stride, pad, groups, eps=1e-5, out=None, stream=None):
    """gf_convt3d_swish_gn_hswish without a workspace: for callers that cannot
    give the library device scratch memory; the library's own fixed scratch
    (gf_convt3d_noalloc_scratch_limit() bytes per device) is used instead.
    Calls that overlap on the GPU race on that scratch."""
    N, Cin, D, H, W = x.shape
    Cout, k = w.shape[1], w.shape[2]
    _convt3d_shapes(x, w, b, gamma, beta, out, stride, pad)
    dev = _check(x, w, b, gamma, beta, out)
    if out is None:
        out = torch.empty(convt3d_out_shape(x.shape, Cout, k, stride, pad), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _call("gf_convt3d_swish_gn_hswish_noalloc", _ptr(x), _ptr(w), _ptr(b), _ptr(gamma), _ptr(beta), _ptr(out),
              N, Cin, Cout, D, H, W, k, stride, pad, groups, eps, _stream_ptr(stream))
    return out
