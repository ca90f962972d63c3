"""The workspace-free ConvTranspose3d entry point.

Some callers cannot give the library device scratch memory: a process that
owns the whole device memory budget through its own pool and forbids any
further cudaMalloc after start-up, or a plugin interface that hands a kernel
only its inputs and outputs.  gf_convt3d_swish_gn_hswish_noalloc serves them
from a fixed scratch array inside the library.  This test calls it through the
C ABI twice in a row (different inputs, so stale scratch contents from the
first call would show) and checks each result against the workspace entry
point gf_convt3d_swish_gn_hswish on the same inputs, within the parity
tolerance used everywhere else (1e-4 abs + 1e-4 rel).  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from conv_activation_normalization_gb300 import binding as gf
from conv_activation_normalization_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 1e-4
RTOL = 1e-4


@pytest.fixture(scope="module")
def L():
    from conv_activation_normalization_gb300 import build
    build.build()
    return gf.lib()


def _noalloc(L, t, s, out):
    return L.gf_convt3d_swish_gn_hswish_noalloc(
        t["x"].data_ptr(), t["w"].data_ptr(), t["b"].data_ptr(), t["gamma"].data_ptr(), t["beta"].data_ptr(),
        out.data_ptr(), s.N, s.Cin, s.Cout, s.D, s.H, s.W, s.k, s.stride, s.pad, s.groups, s.eps,
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_two_calls(L):
    shapes = [synth.ConvT3dShape(N=5, D=6, H=13, W=40), synth.ConvT3dShape(N=3, D=9, H=20, W=17)]
    for call, (s, seed) in enumerate(zip(shapes, (901, 902))):
        d = synth.convt3d_inputs(s, seed)
        t = {k: torch.from_numpy(v).cuda() for k, v in d.items()}
        ref = gf.gf_convt3d_swish_gn_hswish(t["x"], t["w"], t["b"], t["gamma"], t["beta"], s.stride, s.pad,
                                            s.groups, s.eps)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(L, t, s, out) == 0, f"call {call}"
        torch.cuda.synchronize()
        got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        err = np.abs(got - want)
        assert np.all(err <= ATOL + RTOL * np.abs(want)), f"call {call}: max err {np.nanmax(err):.3g}"
    assert gf.gf_device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(L):
    limit = L.gf_convt3d_noalloc_scratch_limit()
    assert limit == 4 << 20
    s = synth.ConvT3dShape(N=4000)
    need = L.gf_convt3d_swish_gn_hswish_workspace_size(s.N, s.Cin, s.Cout, s.D, s.H, s.W, 3, 2, 1, 4)
    assert need > limit
    # validation fails before any pointer is touched, so placeholders suffice
    p = [0x7F0000000000 + i * (1 << 36) for i in range(6)]
    st = L.gf_convt3d_swish_gn_hswish_noalloc(*p, s.N, s.Cin, s.Cout, s.D, s.H, s.W, 3, 2, 1, 4, 1e-5, None)
    assert st == -5  # GF_ERR_WORKSPACE
