"""Host-buffer entry points of the per-sample chains.

gf_ln_gelu_dconv1d_res_host and gf_convt3d_swish_gn_hswish_host copy chunks
of whole samples in, compute each chunk with the device entry point and copy
it out, overlapped on internal streams.  Both chains normalise within a
sample and tile within a sample, so a chunk's kernels do exactly what the
whole batch's do for those samples: the host call must reproduce the device
call bit for bit (ragged last chunks, the default chunk size, pageable
buffers, every mode, each ConvTranspose3d kernel family), and one case per
chain is also held against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_normalization_gb300 import binding as gf
from conv_activation_normalization_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 1e-4
RTOL = 1e-4


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("B,C,L,chunk,mode,pinned", [
    (5, 64, 256, 2, gf.GF_MODE_FP32_3XTF32, True),   # ragged last chunk
    (9, 32, 130, 0, gf.GF_MODE_FP32_3XTF32, True),   # default chunk (2 samples: 5 chunks), L % 4 != 0
    (4, 64, 256, 4, gf.GF_MODE_BF16, True),          # one chunk
    (3, 48, 200, 1, gf.GF_MODE_FP32_3XBF16, False),  # pageable host buffers
])
def test_dconv1d_host_matches_device_call(B, C, L, chunk, mode, pinned):
    s = synth.DConv1dShape(B=B, C=C, L=L)
    d = synth.dconv1d_inputs(s, 700 + B, affine="perturbed")
    dev = {k: T(d[k]) for k in ("ln_gamma", "ln_beta", "conv_w", "conv_b")}
    ref = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), dev["ln_gamma"], dev["ln_beta"], dev["conv_w"], dev["conv_b"],
                                    s.dilation, s.padding, s.eps, mode=mode).cpu()
    xh = _host(d["x"], pinned)
    oh = torch.full((B, C, L), float("nan"), dtype=torch.float32, pin_memory=pinned)
    gf.gf_ln_gelu_dconv1d_res_host(xh, dev["ln_gamma"], dev["ln_beta"], dev["conv_w"], dev["conv_b"], s.dilation,
                                   s.padding, s.eps, mode=mode, out_host=oh, chunk_samples=chunk)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh, ref)
    if mode == gf.GF_MODE_FP32_3XTF32:
        want = oracle.ln_gelu_dconv1d_res(d["x"], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"],
                                          s.dilation, s.padding, s.eps)
        np.testing.assert_allclose(oh.numpy(), want, atol=ATOL, rtol=RTOL)


@pytest.mark.parametrize("shape,chunk,pinned", [
    # the pages' configuration, Cin = 3: the single cooperative tensor-core kernel
    (dict(N=5, Cin=3, Cout=16, D=4, H=8, W=8, k=3, stride=2, pad=1, groups=4), 2, True),
    # samples of 12 x ceil(48 * 48 / 128) = 216 tiles, more than the SMs + 1:
    # the two-pass tensor-core kernels
    (dict(N=3, Cin=3, Cout=16, D=12, H=48, W=48, k=3, stride=2, pad=1, groups=4), 2, True),
    # the same with Cin = 6: the CUDA-core kernels for 5..8 input channels
    (dict(N=4, Cin=6, Cout=16, D=3, H=6, W=5, k=3, stride=2, pad=1, groups=4), 3, True),
    # another configuration: the general two-pass kernels; default chunk
    (dict(N=3, Cin=2, Cout=6, D=3, H=5, W=4, k=2, stride=1, pad=0, groups=3), 0, False),
])
def test_convt3d_host_matches_device_call(shape, chunk, pinned):
    s = synth.ConvT3dShape(**shape)
    d = synth.convt3d_inputs(s, 900 + s.N)
    dev = {k: T(d[k]) for k in ("w", "b", "gamma", "beta")}
    ref = gf.gf_convt3d_swish_gn_hswish(T(d["x"]), dev["w"], dev["b"], dev["gamma"], dev["beta"], s.stride, s.pad,
                                        s.groups, s.eps).cpu()
    xh = _host(d["x"], pinned)
    oh = torch.full(tuple(ref.shape), float("nan"), dtype=torch.float32, pin_memory=pinned)
    gf.gf_convt3d_swish_gn_hswish_host(xh, dev["w"], dev["b"], dev["gamma"], dev["beta"], s.stride, s.pad,
                                       s.groups, s.eps, out_host=oh, chunk_samples=chunk)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh, ref)
    if s.Cin == 3:
        want = oracle.convt3d_swish_gn_hswish(d["x"], d["w"], d["b"], d["gamma"], d["beta"], s.stride, s.pad,
                                              s.groups, s.eps)
        np.testing.assert_allclose(oh.numpy(), want, atol=ATOL, rtol=RTOL)


def test_dconv1d_host_tanh_gelu():
    s = synth.DConv1dShape(B=4, C=32, L=128)
    d = synth.dconv1d_inputs(s, 808, affine="perturbed")
    dev = {k: T(d[k]) for k in ("ln_gamma", "ln_beta", "conv_w", "conv_b")}
    ref = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), dev["ln_gamma"], dev["ln_beta"], dev["conv_w"], dev["conv_b"],
                                    s.dilation, s.padding, s.eps, gelu="tanh").cpu()
    xh = _host(d["x"], True)
    oh = gf.gf_ln_gelu_dconv1d_res_host(xh, dev["ln_gamma"], dev["ln_beta"], dev["conv_w"], dev["conv_b"],
                                        s.dilation, s.padding, s.eps, chunk_samples=3, gelu="tanh")
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh, ref)


def test_host_calls_report_the_device_calls_checks():
    # a device pointer that is not 16-byte aligned fails the device call's
    # own check on the first chunk; the host call returns that status after
    # draining what it had queued
    s = synth.DConv1dShape(B=2, C=32, L=64)
    d = synth.dconv1d_inputs(s, 77)
    dev = {k: T(d[k]) for k in ("ln_gamma", "ln_beta", "conv_w", "conv_b")}
    bad = torch.empty(s.C + 1, dtype=torch.float32, device="cuda")[1:]
    bad.copy_(dev["conv_b"])
    xh = torch.from_numpy(d["x"]).pin_memory()
    with pytest.raises(gf.GFError) as e:
        gf.gf_ln_gelu_dconv1d_res_host(xh, dev["ln_gamma"], dev["ln_beta"], dev["conv_w"], bad, s.dilation,
                                       s.padding, s.eps, chunk_samples=1)
    assert e.value.status == -3  # GF_ERR_ALIGN
    torch.cuda.synchronize()
