"""Oracle parity of every GEMM kernel variant the Linear chains' dispatch can
launch (tests/dispatch_cases.py: each tile width x contraction mode x
epilogue), through the C ABI.  Tolerance: 1e-4 abs + 1e-4 rel in the
three-product modes, 3e-2 in the BF16 mode.  The plain Linear cases are
checked bit for bit on integer-valued operands (exact in every mode)."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from conv_activation_normalization_gb300 import binding as gf
from conv_activation_normalization_gb300 import synth

from . import dispatch_cases as dc

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 3e-2, 2: 1e-4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conv_activation_normalization_gb300 import build
    build.build()
    gf.lib()
    yield
    assert gf.gf_device_status() == 0


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    bad = ~(err <= tol + tol * np.abs(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} outside {tol}; max err {np.nanmax(err):.3g}"


@pytest.mark.parametrize("case", dc.cases(), ids=lambda c: c.name)
def test_dispatch_variant_matches_oracle(case):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    bn = gf.linear_tile_width(case.chain, case.M, case.N, case.groups, case.mode, sm)
    assert bn == case.bn, f"{case.name}: this GPU's {sm} SMs give tile width {bn}, the case targets {case.bn}"
    seed = 7000 + zlib.crc32(case.name.encode()) % 1000
    if case.chain == dc.GN:
        s = synth.LinearGNShape(M=case.M, K=case.K, N=case.N, groups=case.groups)
        d = synth.linear_gn_inputs(s, seed)
        got = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                                T(d["beta"]), s.groups, s.eps, mode=case.mode).cpu().numpy()
        ref = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                                 s.groups, s.eps)
        assert_close(got, ref, TOL[case.mode], case.name)
    elif case.chain == dc.LSE:
        s = synth.LinearLSEShape(M=case.M, K=case.K, N=case.N)
        d = synth.linear_lse_inputs(s, seed)
        got = gf.gf_linear_lse_act(T(d["x"]), T(d["W"]), T(d["b"]), s.negative_slope, mode=case.mode).cpu().numpy()
        ref = oracle.linear_lse_act(d["x"], d["W"], d["b"], s.negative_slope)
        assert_close(got, ref, TOL[case.mode], case.name)
    else:
        r = np.random.default_rng(seed)
        x = r.integers(-15, 16, size=(case.M, case.K)).astype(np.float32)
        W = r.integers(-15, 16, size=(case.N, case.K)).astype(np.float32)
        b = r.integers(-50, 51, size=case.N).astype(np.float32)
        got = gf.gf_linear(T(x), T(W), T(b), mode=case.mode).cpu().numpy()
        exact = x.astype(np.int64) @ W.astype(np.int64).T + b.astype(np.int64)
        assert np.array_equal(got.astype(np.int64), exact), case.name
        # and the oracle's contraction agrees
        assert np.array_equal(oracle.linear(x, W, b), exact.astype(np.float64))


def test_bf16_mode_full_size_linear_gn_sampled():
    # the BF16 mode at the 256-column tile width on the full workload (the
    # kernel the benchmark reports as the BF16 mode), sampled rows
    s, seed = synth.WORKLOADS["linear_gn_m32768"]
    d = synth.linear_gn_inputs(s, seed)
    assert gf.linear_tile_width(dc.GN, s.M, s.N, s.groups, 1, torch.cuda.get_device_properties(0).multi_processor_count) == 256
    out = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                            T(d["beta"]), s.groups, s.eps, mode=1).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, 200), np.random.default_rng(2).integers(0, s.M, 800),
                                     np.arange(s.M - 200, s.M)]))
    ref = oracle.linear_swish_bias_groupnorm(d["x"][rows], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                             s.groups, s.eps)
    assert_close(out[rows], ref, 3e-2, "linear_gn bf16 M=32768")
