"""Parity of the BF16 (one product) and 3xBF16 (three products of a bf16
hi/lo split) contraction modes with the fp64 oracle.

Tolerances: BF16 mode 3e-2 abs + 3e-2 rel (operands rounded to 8-bit
significands); 3xBF16 mode the fp32-mode bar, 1e-4 abs + 1e-4 rel.  The
contraction alone is checked bit for bit on small integers, which bf16
represents exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_normalization_gb300 import binding as gf
from conv_activation_normalization_gb300 import synth

pytestmark = pytest.mark.gpu

BF16, X3BF16 = 1, 2
TOL = {BF16: 3e-2, X3BF16: 1e-4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conv_activation_normalization_gb300 import build
    build.build()
    gf.lib()
    yield
    assert gf.gf_device_status() == 0


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    bad = ~(err <= tol + tol * np.abs(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} outside {tol}; max err {np.nanmax(err):.3g}"


@pytest.mark.parametrize("mode", [BF16, X3BF16])
@pytest.mark.parametrize("M,K,N", [(128, 64, 256), (300, 104, 520), (257, 1024, 4096), (70, 37, 130), (9, 5, 3)])
def test_linear_integer_exact(mode, M, K, N):
    r = np.random.default_rng(M + K + mode)
    x = r.integers(-15, 16, size=(M, K)).astype(np.float32)
    W = r.integers(-15, 16, size=(N, K)).astype(np.float32)
    got = gf.gf_linear(T(x), T(W), mode=mode).cpu().numpy()
    assert np.array_equal(got.astype(np.int64), x.astype(np.int64) @ W.astype(np.int64).T)


def test_linear_3xbf16_accuracy():
    # relative to sqrt(sum (x w)^2): one bf16 product errs by ~4e-3, the
    # three-product split (exact accumulation, CPU emulation) by <= 1.8e-5.
    r = np.random.default_rng(5)
    M, K, N = 256, 1024, 512
    x = r.standard_normal((M, K)).astype(np.float32)
    W = r.uniform(-1, 1, (N, K)).astype(np.float32)
    got = gf.gf_linear(T(x), T(W), mode=X3BF16).cpu().numpy().astype(np.float64)
    ref = oracle.linear(x, W)
    scale = np.sqrt((x.astype(np.float64) ** 2) @ (W.astype(np.float64) ** 2).T)
    err = np.abs(got - ref) / scale
    assert err.max() < 1e-4 and err.mean() < 2e-5, (err.max(), err.mean())


@pytest.mark.parametrize("mode", [BF16, X3BF16])
@pytest.mark.parametrize("M,K,N", [(256, 1024, 4096), (130, 40, 320)])
def test_linear_gn_modes(mode, M, K, N):
    s = synth.LinearGNShape(M=M, K=K, N=N, groups=N // 64)
    d = synth.linear_gn_inputs(s, 500 + M)
    out = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                            T(d["beta"]), s.groups, s.eps, mode=mode).cpu().numpy()
    ref = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"], s.groups,
                                             s.eps)
    assert_close(out, ref, TOL[mode], f"linear_gn mode {mode}")


@pytest.mark.parametrize("mode", [BF16, X3BF16])
@pytest.mark.parametrize("M,K,N,gw", [(130, 40, 320, 16), (200, 64, 512, 128), (150, 64, 768, 256)])
def test_linear_gn_modes_group_widths(mode, M, K, N, gw):
    s = synth.LinearGNShape(M=M, K=K, N=N, groups=N // gw)
    d = synth.linear_gn_inputs(s, 600 + gw)
    out = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                            T(d["beta"]), s.groups, s.eps, mode=mode).cpu().numpy()
    ref = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"], s.groups,
                                             s.eps)
    assert_close(out, ref, TOL[mode], f"linear_gn mode {mode} groups of {gw}")


# The BF16 mode writes the GroupNorm output as 32-row x 16-column boxes staged
# in shared memory and sent by TMA stores: ragged rows (the store clips them)
# and a last column tile that only partly exists, at each tile width the
# dispatch picks (shapes checked against gf_linear_tile_width), including 16-
# and 32-column groups whose last 64-column block has one or two quarters.
# The 256-column tiles run in two-CTA clusters over pairs of m-blocks: with an
# odd count the last pair's second tile lies past M (computed, not stored).
@pytest.mark.parametrize("M,K,N,gw,bn", [
    (777, 72, 2080, 32, 64),     # 7 x 17 tiles of 128 columns < 152 SMs: 64-column tiles; last block 2 quarters
    (1100, 96, 3088, 16, 128),   # 9 x 13 tiles of 256 < 152 <= 9 x 25 of 128; last 64-column block 1 quarter
    (2500, 128, 4160, 64, 256),  # 20 x 17 tiles of 256: the last tile has 64 of its 256 columns
    (2600, 136, 4160, 64, 256),  # 21 m-blocks (odd), 40 rows in the last
    (100, 64, 1024, 128, 256),   # one m-block: each pair's second tile lies past M
])
def test_bf16_box_stores_ragged(M, K, N, gw, bn):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert gf.linear_tile_width(gf.GF_CHAIN_GROUPNORM, M, N, N // gw, BF16, sm) == bn
    s = synth.LinearGNShape(M=M, K=K, N=N, groups=N // gw)
    d = synth.linear_gn_inputs(s, 700 + gw)
    out = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                            T(d["beta"]), s.groups, s.eps, mode=BF16).cpu().numpy()
    ref = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"], s.groups,
                                             s.eps)
    assert_close(out, ref, TOL[BF16], f"bf16 boxes M={M} N={N} gw={gw}")


def test_linear_gn_3xbf16_workload_m32768_sampled():
    s, seed = synth.WORKLOADS["linear_gn_m32768"]
    d = synth.linear_gn_inputs(s, seed)
    out = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                            T(d["beta"]), s.groups, s.eps, mode=X3BF16).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, 200), np.random.default_rng(1).integers(0, s.M, 800),
                                     np.arange(s.M - 200, s.M)]))
    ref = oracle.linear_swish_bias_groupnorm(d["x"][rows], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                             s.groups, s.eps)
    assert_close(out[rows], ref, 1e-4, "linear_gn 3xbf16 M=32768")


@pytest.mark.parametrize("mode", [BF16, X3BF16])
def test_linear_lse_modes(mode):
    s = synth.LinearLSEShape(M=200, K=512, N=1000)
    d = synth.linear_lse_inputs(s, 77)
    out = gf.gf_linear_lse_act(T(d["x"]), T(d["W"]), T(d["b"]), s.negative_slope, mode=mode).cpu().numpy()
    ref = oracle.linear_lse_act(d["x"], d["W"], d["b"], s.negative_slope)
    assert_close(out, ref, TOL[mode], f"lse mode {mode}")


def test_linear_lse_3xbf16_workload_sampled():
    s, seed = synth.WORKLOADS["linear_lse_m1024"]
    d = synth.linear_lse_inputs(s, seed)
    out = gf.gf_linear_lse_act(T(d["x"]), T(d["W"]), T(d["b"]), s.negative_slope, mode=X3BF16).cpu().numpy()
    rows = np.arange(0, s.M, 8)
    ref = oracle.linear_lse_act(d["x"][rows], d["W"], d["b"], s.negative_slope)
    assert_close(out[rows], ref, 1e-4, "lse 3xbf16 full workload")


@pytest.mark.parametrize("mode", [BF16, X3BF16])
@pytest.mark.parametrize("B,C,L,dil", [(2, 64, 300, 4), (2, 256, 520, 2), (1, 96, 200, 2), (2, 40, 128, 1)])
def test_dconv1d_modes(mode, B, C, L, dil):
    s = synth.DConv1dShape(B=B, C=C, L=L, dilation=dil, padding=dil)
    d = synth.dconv1d_inputs(s, 600 + L, affine="perturbed")
    out = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps, mode=mode).cpu().numpy()
    ref = oracle.ln_gelu_dconv1d_res(d["x"], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps)
    assert_close(out, ref, TOL[mode], f"dconv1d mode {mode}")


@pytest.mark.parametrize("mode", [BF16, X3BF16])
def test_dconv1d_modes_tanh_gelu(mode):
    s = synth.DConv1dShape(B=2, C=128, L=260, dilation=3, padding=3)
    d = synth.dconv1d_inputs(s, 650, affine="perturbed")
    out = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps, mode=mode, gelu="tanh").cpu().numpy()
    ref = oracle.ln_gelu_dconv1d_res(d["x"], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps, gelu="tanh")
    assert_close(out, ref, TOL[mode], f"dconv1d mode {mode} tanh GELU")


def test_dconv1d_3xbf16_workload_sampled():
    s, seed = synth.WORKLOADS["ln_dconv1d_b32"]
    d = synth.dconv1d_inputs(s, seed)
    out = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps, mode=X3BF16).cpu().numpy()
    idx = np.array([0, 31])
    ref = oracle.ln_gelu_dconv1d_res(d["x"][idx], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps)
    assert_close(out[idx], ref, 1e-4, "dconv1d 3xbf16 full workload")
