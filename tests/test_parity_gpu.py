"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bar: |gpu - oracle| <= 1e-4 + 1e-4 |oracle| element by element (the fp32-mode
tolerance), on seeded synthetic inputs: small shapes that span several tiles
and a ragged tail, degenerate cases, and the full-size workloads on samples
the oracle can compute one by one (rows, or whole samples for the
per-sample normalisations).  The contraction alone is checked bit for bit on
integer-valued inputs.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from conv_activation_normalization_gb300 import build
    build.build()
    gf.lib()
    yield
    assert gf.gf_device_status() == 0


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    lim = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; max err {np.nanmax(err):.3g}; "
                             f"first {idx.tolist()}")


# ------------------------------------------------------------ contraction
@pytest.mark.parametrize("M,K,N", [(128, 32, 256), (300, 100, 520), (1, 4, 1), (257, 1024, 4096), (70, 37, 130),
                                   (5, 1, 7)])
def test_linear_integer_exact(M, K, N):
    r = np.random.default_rng(M * 7 + K)
    x = r.integers(-15, 16, size=(M, K)).astype(np.float32)
    W = r.integers(-15, 16, size=(N, K)).astype(np.float32)
    b = r.integers(-50, 51, size=N).astype(np.float32)
    got = gf.gf_linear(T(x), T(W), T(b)).cpu().numpy()
    exact = x.astype(np.int64) @ W.astype(np.int64).T + b.astype(np.int64)
    assert np.array_equal(got.astype(np.int64), exact)
    assert np.array_equal(got, exact.astype(np.float32))


def test_linear_3xtf32_accuracy():
    # Values with all 24 mantissa bits in use.  Relative to the scale
    # sqrt(sum_k (x w)^2), a single TF32 product (emulated exactly on the CPU
    # for these inputs) is off by up to 3.5e-3 (mean 5.8e-4); the hi/lo split
    # with exact accumulation by up to 1.6e-6.  The tensor core accumulates in
    # fp32 with its own rounding over K/8 * 3 chained MMA steps, which adds up
    # to ~2^-17 |y| (4.5e-5 of the scale here); the bounds sit well below
    # what a single TF32 product gives.
    r = np.random.default_rng(5)
    M, K, N = 256, 1024, 512
    x = r.standard_normal((M, K)).astype(np.float32)
    W = r.uniform(-1, 1, (N, K)).astype(np.float32)
    got = gf.gf_linear(T(x), T(W)).cpu().numpy().astype(np.float64)
    ref = oracle.linear(x, W)
    scale = np.sqrt((x.astype(np.float64) ** 2) @ (W.astype(np.float64) ** 2).T)
    err = np.abs(got - ref)
    assert np.max(err / scale) < 1e-4
    assert np.mean(err / scale) < 2e-5


# ------------------------------------------------ Linear->Swish->bias->GN
def _lgn_case(M, K, N, groups, seed):
    s = synth.LinearGNShape(M=M, K=K, N=N, groups=groups)
    d = synth.linear_gn_inputs(s, seed)
    return s, d


def _lgn_run(s, d, rows=None):
    out = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                            T(d["beta"]), s.groups, s.eps).cpu().numpy()
    xr = d["x"] if rows is None else d["x"][rows]
    ref = oracle.linear_swish_bias_groupnorm(xr, d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"], s.groups,
                                             s.eps)
    return (out if rows is None else out[rows]), ref


def test_linear_gn_workload_m256():
    s, seed = synth.WORKLOADS["linear_gn_m256"]
    got, ref = _lgn_run(s, synth.linear_gn_inputs(s, seed))
    assert_close(got, ref, "linear_gn M=256")


@pytest.mark.parametrize("M,K,N", [(1, 4, 64), (130, 36, 320), (383, 260, 4096), (129, 1024, 192)])
def test_linear_gn_ragged(M, K, N):
    s, d = _lgn_case(M, K, N, N // 64, 100 + M)
    got, ref = _lgn_run(s, d)
    assert_close(got, ref, f"linear_gn {M}x{K}x{N}")


# GroupNorm groups of 16, 32 and 128 columns (64 is the workloads' width):
# ragged rows and columns, a 128-column group in the partial last tile, and a
# single row
@pytest.mark.parametrize("M,K,N,gw", [(130, 36, 320, 16), (383, 260, 4096, 32), (1, 4, 48, 16), (257, 64, 96, 32),
                                      (300, 64, 384, 128), (129, 100, 512, 128), (1, 4, 128, 128),
                                      (200, 1024, 4096, 128)])
def test_linear_gn_group_widths(M, K, N, gw):
    s, d = _lgn_case(M, K, N, N // gw, 300 + gw + M)
    got, ref = _lgn_run(s, d)
    assert_close(got, ref, f"linear_gn {M}x{K}x{N} groups of {gw}")


# other group widths: t stored by the GEMM epilogue, rows normalised by a
# second kernel (any width dividing N, including one group per row)
@pytest.mark.parametrize("M,K,N,groups", [(130, 36, 512, 2), (200, 64, 4096, 16), (64, 32, 384, 4), (97, 40, 96, 12),
                                          (33, 16, 1000, 5), (1, 4, 4096, 1), (129, 1024, 4096, 8)])
def test_linear_gn_other_group_widths(M, K, N, groups):
    s, d = _lgn_case(M, K, N, groups, 800 + N // groups)
    got, ref = _lgn_run(s, d)
    assert_close(got, ref, f"linear_gn {M}x{K}x{N} in {groups} groups of {N // groups}")


def test_linear_gn_group_width_128_halves_differ():
    # a 128-column group whose halves have very different means: the merge of
    # the halves' (mean, M2) must carry the between-halves term
    s, d = _lgn_case(96, 32, 256, 2, 11)
    d["bias"][:64] += 3.0
    d["bias"][128:192] -= 2.0
    got, ref = _lgn_run(s, d)
    assert_close(got, ref, "linear_gn groups of 128, shifted halves")


@pytest.mark.parametrize("M,K,N", [(130, 37, 256), (64, 1, 128), (200, 1023, 512)])
def test_linear_gn_unaligned_k(M, K, N):
    # K not a whole number of 16-byte rows: the pre-pass pads every plane
    s, d = _lgn_case(M, K, N, N // 64, 850 + K)
    got, ref = _lgn_run(s, d)
    assert_close(got, ref, f"linear_gn {M}x{K}x{N}")


def test_linear_gn_no_linear_bias_and_constant_group():
    s, d = _lgn_case(64, 64, 256, 4, 7)
    d["W"][:64] = 0.0      # group 0: t = swish(0) + bias = bias, varies per channel
    d["bias"][64:128] = 0.5
    d["W"][64:128] = 0.0   # group 1: constant t -> output beta
    out = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), None, T(d["bias"]), T(d["gamma"]), T(d["beta"]),
                                            s.groups, s.eps).cpu().numpy()
    ref = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], None, d["bias"], d["gamma"], d["beta"], s.groups, s.eps)
    assert_close(out, ref, "no b_lin")
    np.testing.assert_array_equal(out[:, 64:128], np.broadcast_to(d["beta"][64:128], (64, 64)))


def test_linear_gn_workload_m32768_sampled():
    s, seed = synth.WORKLOADS["linear_gn_m32768"]
    d = synth.linear_gn_inputs(s, seed)
    r = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 130), r.integers(0, s.M, 600), np.arange(s.M - 130, s.M)]))
    got, ref = _lgn_run(s, d, rows)
    assert_close(got, ref, "linear_gn M=32768 (sampled rows)")


@pytest.mark.parametrize("w_dist", ["default", "normal"])
def test_linear_gn_uniform01_inputs(w_dist):
    # x ~ U[0,1) (torch.rand inputs), with the module's default weights or
    # W ~ N(0,1): page Kimi-K2.6__l2_p37, turn 1, reasons about both
    s = synth.LinearGNShape(M=130, K=1024, N=4096)
    d = synth.linear_gn_inputs(s, 13, x_dist="uniform01", w_dist=w_dist)
    got, ref = _lgn_run(s, d)
    assert_close(got, ref, f"linear_gn U[0,1) x, {w_dist} W")


def test_linear_gn_all_uniform_inputs():
    # x and W ~ U[0,1) (page Kimi-K2.6__l2_p64's all-uniform case): every y is
    # about 256 = K/4, and the tensor core's truncating fp32 accumulation
    # biases it by about -5e-3 (a few 1e-4 apart between channels).  GroupNorm
    # cancels the common part; the rest, over a group spread of about 5,
    # stays within 1e-4 in the 3xBF16 mode (half the accumulation steps) and
    # within 2e-4 in the 3xTF32 mode, whose 256-column tiles leave no TMEM for
    # the chunked accumulation the logsumexp chain uses
    s = synth.LinearGNShape(M=130, K=1024, N=4096)
    d = synth.linear_gn_inputs(s, 13, x_dist="uniform01", w_dist="uniform01")
    ref = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"], s.groups,
                                             s.eps)
    for mode, tol in ((2, 1e-4), (0, 2e-4)):
        got = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                                T(d["beta"]), s.groups, s.eps, mode=mode).cpu().numpy()
        err = np.abs(got.astype(np.float64) - ref)
        assert np.all(err <= tol + tol * np.abs(ref)), (mode, float(err.max()))


def test_linear_gn_deterministic():
    s, d = _lgn_case(512, 256, 1024, 16, 3)
    a = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                          T(d["beta"]), s.groups).cpu().numpy()
    b = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                          T(d["beta"]), s.groups).cpu().numpy()
    assert np.array_equal(a, b)


# ------------------------------------------------- Linear->LSE->act chain
def _lse_run(s, d, rows=None):
    out = gf.gf_linear_lse_act(T(d["x"]), T(d["W"]), T(d["b"]), s.negative_slope).cpu().numpy()
    xr = d["x"] if rows is None else d["x"][rows]
    ref = oracle.linear_lse_act(xr, d["W"], d["b"], s.negative_slope)
    return (out if rows is None else out[rows]), ref


@pytest.mark.parametrize("M,K,N", [(1, 4, 1), (200, 512, 1000), (129, 260, 8192), (384, 2048, 300)])
def test_linear_lse_small(M, K, N):
    s = synth.LinearLSEShape(M=M, K=K, N=N)
    got, ref = _lse_run(s, synth.linear_lse_inputs(s, 200 + M))
    assert_close(got, ref, f"lse {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(100, 3, 300), (129, 1001, 2048)])
def test_linear_lse_unaligned_k(M, K, N):
    s = synth.LinearLSEShape(M=M, K=K, N=N)
    got, ref = _lse_run(s, synth.linear_lse_inputs(s, 860 + K))
    assert_close(got, ref, f"lse {M}x{K}x{N}")


def test_linear_lse_negative_branch():
    s = synth.LinearLSEShape(M=64, K=256, N=8192)
    d = synth.linear_lse_inputs(s, 11, bias_shift=-30.0)
    got, ref = _lse_run(s, d)
    assert np.all(ref < 0)
    assert_close(got, ref, "lse negative branch")


def test_linear_lse_uniform01_inputs():
    # x, W, b ~ U[0,1): every logit is a sum of 8192 products of mean 1/4,
    # so logsumexp is about 2100 and the tiles' maxima differ by tens; the
    # (max, sum exp) merge rescales across them (page Kimi-K2.6__l2_p64,
    # turn 1, reasons about exactly this input)
    s = synth.LinearLSEShape(M=160, K=8192, N=8192)
    d = synth.linear_lse_inputs(s, 12, dist="uniform01")
    got, ref = _lse_run(s, d)
    assert ref.min() > 1500
    assert_close(got, ref, "lse U[0,1) inputs")
    # the same in the 3xBF16 mode (chunked accumulation too)
    got = gf.gf_linear_lse_act(T(d["x"]), T(d["W"]), T(d["b"]), s.negative_slope, mode=2).cpu().numpy()
    assert_close(got, ref, "lse U[0,1) inputs, 3xbf16")


def test_linear_lse_workload_sampled():
    s, seed = synth.WORKLOADS["linear_lse_m1024"]
    d = synth.linear_lse_inputs(s, seed)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(500, 530), np.arange(s.M - 64, s.M)]))
    got, ref = _lse_run(s, d, rows)
    assert_close(got, ref, "lse full workload (sampled rows)")


# --------------------------------------------- LN->GELU->dilated conv->+x
def _dc_run(s, d, samples=None):
    out = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps).cpu().numpy()
    xs = d["x"] if samples is None else d["x"][samples]
    ref = oracle.ln_gelu_dconv1d_res(xs, d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation, s.padding,
                                     s.eps)
    return (out if samples is None else out[samples]), ref


@pytest.mark.parametrize("B,C,L,dil", [(2, 64, 300, 4), (1, 32, 4, 4), (3, 256, 520, 2), (2, 96, 1024, 1)])
def test_dconv1d_small(B, C, L, dil):
    s = synth.DConv1dShape(B=B, C=C, L=L, dilation=dil, padding=dil)
    got, ref = _dc_run(s, synth.dconv1d_inputs(s, 300 + L, affine="perturbed"))
    assert_close(got, ref, f"dconv1d {B}x{C}x{L} d{dil}")


@pytest.mark.parametrize("B,C,L,dil", [(2, 64, 300, 4), (3, 256, 520, 2)])
def test_dconv1d_tanh_gelu(B, C, L, dil):
    # the tanh-approximate GELU variant (flag GF_FLAG_GELU_TANH)
    s = synth.DConv1dShape(B=B, C=C, L=L, dilation=dil, padding=dil)
    d = synth.dconv1d_inputs(s, 700 + L, affine="perturbed")
    got = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps, gelu="tanh").cpu().numpy()
    ref = oracle.ln_gelu_dconv1d_res(d["x"], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps, gelu="tanh")
    assert_close(got, ref, f"dconv1d tanh GELU {B}x{C}x{L}")
    erf = oracle.ln_gelu_dconv1d_res(d["x"], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps)
    assert np.abs(got - erf).max() > 1e-4  # the variant is really the other GELU


@pytest.mark.parametrize("B,C,L,dil", [(2, 384, 260, 2), (1, 512, 200, 4), (1, 1024, 64, 1)])
def test_dconv1d_wide(B, C, L, dil):
    # more than 256 channels: the output channels span several 256-column tiles
    s = synth.DConv1dShape(B=B, C=C, L=L, dilation=dil, padding=dil)
    got, ref = _dc_run(s, synth.dconv1d_inputs(s, 950 + C, affine="perturbed"))
    assert_close(got, ref, f"dconv1d {B}x{C}x{L} d{dil}")


@pytest.mark.parametrize("B,C,L,dil", [(2, 48, 300, 4), (1, 100, 128, 2), (3, 1, 64, 1), (2, 33, 520, 3)])
def test_dconv1d_unaligned_channels(B, C, L, dil):
    # channel counts that are not whole k-blocks: zero-padded operand planes
    s = synth.DConv1dShape(B=B, C=C, L=L, dilation=dil, padding=dil)
    got, ref = _dc_run(s, synth.dconv1d_inputs(s, 970 + C, affine="perturbed"))
    assert_close(got, ref, f"dconv1d {B}x{C}x{L} d{dil}")


@pytest.mark.parametrize("B,C,L,dil", [(2, 64, 301, 4), (1, 40, 7, 1), (3, 32, 1, 2), (1, 256, 4093, 4)])
def test_dconv1d_any_length(B, C, L, dil):
    # lengths that are not multiples of 4: scalar loads in the LayerNorm passes
    s = synth.DConv1dShape(B=B, C=C, L=L, dilation=dil, padding=dil)
    got, ref = _dc_run(s, synth.dconv1d_inputs(s, 990 + L, affine="perturbed"))
    assert_close(got, ref, f"dconv1d {B}x{C}x{L} d{dil}")


@pytest.mark.parametrize("B,C,L,k,dil,gelu", [(2, 64, 300, 3, 46, "erf"), (2, 64, 300, 3, 4, "erf"),
                                              (1, 32, 4, 3, 4, "erf"), (3, 256, 520, 3, 2, "tanh"),
                                              (2, 40, 262, 5, 23, "erf"), (1, 300, 200, 3, 46, "erf"),
                                              (3, 20, 131, 3, 1, "tanh"), (2, 33, 301, 3, 3, "erf"),
                                              (1, 1024, 64, 3, 1, "erf")])
def test_dconv1d_fused_producer(B, C, L, k, dil, gelu):
    # GF_FLAG_FUSED_PRODUCER: LayerNorm + GELU inside the GEMM's operand
    # build; taps spanning up to 92 positions ((k - 1) dil = 92 is the widest
    # window), any channel count and length (scalar loads when L % 4 != 0)
    s = synth.DConv1dShape(B=B, C=C, L=L, ksize=k, dilation=dil, padding=dil * (k - 1) // 2)
    d = synth.dconv1d_inputs(s, 1100 + dil + C, affine="perturbed")
    got = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps, gelu=gelu, fused_producer=True).cpu().numpy()
    ref = oracle.ln_gelu_dconv1d_res(d["x"], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps, gelu=gelu)
    assert_close(got, ref, f"dconv1d fused producer {B}x{C}x{L} k{k} d{dil} {gelu}")


def test_dconv1d_fused_producer_workload_sampled():
    s, seed = synth.WORKLOADS["ln_dconv1d_b32"]
    d = synth.dconv1d_inputs(s, seed)
    got = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps, fused_producer=True).cpu().numpy()
    idx = np.array([0, 31])
    ref = oracle.ln_gelu_dconv1d_res(d["x"][idx], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps)
    assert_close(got[idx], ref, "dconv1d fused producer, full workload (samples 0, 31)")


def test_dconv1d_fused_producer_rejects_wide_taps_and_other_modes():
    s = synth.DConv1dShape(B=1, C=32, L=300, ksize=3, dilation=47, padding=47)
    d = synth.dconv1d_inputs(s, 5)
    args = [T(d[k]) for k in ("x", "ln_gamma", "ln_beta", "conv_w", "conv_b")]
    with pytest.raises(gf.GFError) as e:
        gf.gf_ln_gelu_dconv1d_res(*args, s.dilation, s.padding, s.eps, fused_producer=True)
    assert e.value.status == -2  # GF_ERR_SHAPE: (k - 1) dilation = 94 > 92
    with pytest.raises(gf.GFError) as e:
        gf.gf_ln_gelu_dconv1d_res(*args, 4, 4, s.eps, mode=1, fused_producer=True)
    assert e.value.status == -6  # GF_ERR_MODE: the 3xTF32 mode only


def test_dconv1d_kernel_size_5():
    s = synth.DConv1dShape(B=2, C=64, L=256, ksize=5, dilation=3, padding=6)
    got, ref = _dc_run(s, synth.dconv1d_inputs(s, 5, affine="perturbed"))
    assert_close(got, ref, "dconv1d k5")


def test_dconv1d_tap_offsets_delta_weights():
    # one nonzero weight per output channel on one tap: shows the tap offset,
    # the zero padding at both ends and the residual.
    s = synth.DConv1dShape(B=1, C=32, L=256)
    d = synth.dconv1d_inputs(s, 9, affine="perturbed")
    w = np.zeros_like(d["conv_w"])
    for co in range(s.C):
        w[co, (co * 7) % s.C, co % 3] = 1.0
    d["conv_w"] = w
    got, ref = _dc_run(s, d)
    assert_close(got, ref, "dconv1d delta taps")


def test_dconv1d_workload_sampled():
    s, seed = synth.WORKLOADS["ln_dconv1d_b32"]
    d = synth.dconv1d_inputs(s, seed)
    got, ref = _dc_run(s, d, samples=np.array([0, 17, 31]))
    assert_close(got, ref, "dconv1d full workload (samples 0, 17, 31)")


# -------------------------------------- ConvT3d->Swish->GN->HardSwish
def _ct_run(s, d, samples=None):
    out = gf.gf_convt3d_swish_gn_hswish(T(d["x"]), T(d["w"]), T(d["b"]), T(d["gamma"]), T(d["beta"]), s.stride,
                                        s.pad, s.groups, s.eps)
    out = out.cpu().numpy()
    xs = d["x"] if samples is None else d["x"][samples]
    ref = oracle.convt3d_swish_gn_hswish(xs, d["w"], d["b"], d["gamma"], d["beta"], s.stride, s.pad, s.groups, s.eps)
    return (out if samples is None else out[samples]), ref


# Cin <= 4 runs the single-kernel tensor-core path while a sample has at most
# (CTAs + 1) tiles of 128 cells: (9, 3, 8, 24, 24) spans three rounds of tiles
# with samples straddling rounds; (1, 3, 40, 40, 40) and (1, 4, 40, 40, 40)
# have 520 tiles in their one sample and take the two-pass tensor-core kernels
# (Cin = 4 fills K = 32, so the conv bias is added in the epilogue instead of
# riding in the K padding); Cin > 4 the SIMT kernels.
@pytest.mark.parametrize("N,Cin,D,H,W", [(2, 3, 5, 7, 9), (1, 1, 1, 1, 1), (3, 3, 4, 33, 40), (1, 8, 3, 8, 64),
                                         (2, 4, 3, 6, 10), (1, 2, 2, 5, 130), (2, 5, 3, 4, 9), (9, 3, 8, 24, 24),
                                         (1, 3, 40, 40, 40), (1, 4, 40, 40, 40)])
def test_convt3d_small(N, Cin, D, H, W):
    s = synth.ConvT3dShape(N=N, Cin=Cin, D=D, H=H, W=W)
    got, ref = _ct_run(s, synth.convt3d_inputs(s, 400 + W))
    assert_close(got, ref, f"convt3d {N}x{Cin}x{D}x{H}x{W}")


# Shapes outside the pages' configuration (other kernel sizes, strides,
# paddings, channel counts and groups; Cin > 8): the general CUDA-core kernels
@pytest.mark.parametrize("N,Cin,Cout,G,k,st,pd,D,H,W", [
    (2, 12, 16, 4, 3, 2, 1, 3, 5, 6), (2, 3, 8, 2, 3, 2, 1, 4, 6, 7), (1, 3, 32, 8, 4, 2, 1, 3, 4, 5),
    (2, 2, 6, 3, 5, 3, 2, 3, 4, 4), (2, 4, 16, 4, 2, 2, 0, 5, 5, 6), (1, 3, 16, 4, 3, 1, 1, 6, 7, 8),
    (3, 1, 4, 1, 1, 1, 0, 3, 3, 3), (1, 3, 16, 16, 3, 2, 0, 3, 4, 5), (1, 5, 12, 3, 8, 4, 3, 2, 3, 3),
    (40, 2, 9, 3, 3, 2, 2, 2, 3, 4)])
def test_convt3d_general(N, Cin, Cout, G, k, st, pd, D, H, W):
    s = synth.ConvT3dShape(N=N, Cin=Cin, Cout=Cout, D=D, H=H, W=W, k=k, stride=st, pad=pd, groups=G)
    got, ref = _ct_run(s, synth.convt3d_inputs(s, 900 + 10 * k + st + Cout))
    assert_close(got, ref, f"convt3d general Cin {Cin} Cout {Cout}/{G} k{k} s{st} p{pd}")


def test_convt3d_general_noalloc_matches_workspace_call():
    s = synth.ConvT3dShape(N=2, Cin=3, Cout=8, D=4, H=5, W=6, k=4, stride=2, pad=1, groups=2)
    d = synth.convt3d_inputs(s, 31)
    args = (T(d["x"]), T(d["w"]), T(d["b"]), T(d["gamma"]), T(d["beta"]), s.stride, s.pad, s.groups, s.eps)
    a = gf.gf_convt3d_swish_gn_hswish(*args).cpu()
    b = gf.gf_convt3d_swish_gn_hswish_noalloc(*args).cpu()
    assert torch.equal(a, b)


def test_convt3d_uniform_inputs():
    s = synth.ConvT3dShape(N=2, D=6, H=12, W=12)
    got, ref = _ct_run(s, synth.convt3d_inputs(s, 77, x_dist="uniform01"))
    assert_close(got, ref, "convt3d U[0,1) inputs")


def test_convt3d_workload_sampled():
    s, seed = synth.WORKLOADS["convt3d_n128"]
    d = synth.convt3d_inputs(s, seed)
    got, ref = _ct_run(s, d, samples=np.array([0, 63, 127]))
    assert got.shape == (3, 16, 31, 63, 63)
    assert_close(got, ref, "convt3d full workload (samples 0, 63, 127)")


# The 3xTF32 lo planes come from a pre-pass at 256-column tiles and are
# computed in the SM at 64-column tiles (few rows).  lo = x - trunc(x) is the
# same value either way and every output element takes the same products in
# the same K order, so rows computed at M = 256 equal the same rows computed
# inside a call whose tile width is 256, bit for bit, for each fused group
# width.
@pytest.mark.parametrize("gw", [16, 32, 64, 128])
def test_linear_gn_lo_in_sm_matches_pre_pass(gw):
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    K, N = 1024, 4096
    big, small = 2432, 256
    assert gf.linear_tile_width(gf.GF_CHAIN_GROUPNORM, big, N, N // gw, 0, sm) == 256
    assert gw == 128 or gf.linear_tile_width(gf.GF_CHAIN_GROUPNORM, small, N, N // gw, 0, sm) == 64
    s, d = _lgn_case(big, K, N, N // gw, 4600 + gw)
    dev = {k: T(d[k]) for k in ("W", "b_lin", "bias", "gamma", "beta")}
    x = T(d["x"])
    whole = gf.gf_linear_swish_bias_groupnorm(x, dev["W"], dev["b_lin"], dev["bias"], dev["gamma"], dev["beta"],
                                              s.groups, s.eps)
    part = gf.gf_linear_swish_bias_groupnorm(x[:small].contiguous(), dev["W"], dev["b_lin"], dev["bias"],
                                             dev["gamma"], dev["beta"], s.groups, s.eps)
    assert torch.equal(part, whole[:small])


# ------------------------------------------------- host-buffer pipeline
@pytest.mark.parametrize("pinned,chunk,groups", [(True, 0, 8), (True, 200, 8), (False, 384, 8), (True, 200, 4),
                                                 (True, 0, 16), (True, 200, 2)])
def test_linear_gn_host_pipeline_matches_device_call(pinned, chunk, groups):
    # Rows are independent and each chunk runs the same kernels, so the
    # pipelined host-buffer call must reproduce the device call bit for bit.
    s, d = _lgn_case(1000, 256, 512, groups, 4242)
    dev = {k: T(d[k]) for k in ("W", "b_lin", "bias", "gamma", "beta")}
    ref = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), dev["W"], dev["b_lin"], dev["bias"], dev["gamma"],
                                            dev["beta"], s.groups, s.eps).cpu()
    xh = torch.from_numpy(d["x"])
    if pinned:
        xh = xh.pin_memory()
    oh = torch.full((s.M, s.N), float("nan"), dtype=torch.float32, pin_memory=pinned)
    gf.gf_linear_swish_bias_groupnorm_host(xh, dev["W"], dev["b_lin"], dev["bias"], dev["gamma"], dev["beta"],
                                           s.groups, s.eps, out_host=oh, chunk_rows=chunk)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh, ref)
    ref64 = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                               s.groups, s.eps)
    assert_close(oh.numpy(), ref64, "host pipeline")


def test_linear_gn_host_pipeline_unaligned_k_and_row_kernel():
    # a K that is not a whole number of 16-byte rows (padded planes per
    # chunk) and a group width that takes the second row kernel
    s, d = _lgn_case(700, 37, 768, 3, 4343)
    dev = {k: T(d[k]) for k in ("W", "b_lin", "bias", "gamma", "beta")}
    ref = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), dev["W"], dev["b_lin"], dev["bias"], dev["gamma"],
                                            dev["beta"], s.groups, s.eps).cpu()
    xh = torch.from_numpy(d["x"]).pin_memory()
    oh = torch.full((s.M, s.N), float("nan"), dtype=torch.float32, pin_memory=True)
    gf.gf_linear_swish_bias_groupnorm_host(xh, dev["W"], dev["b_lin"], dev["bias"], dev["gamma"], dev["beta"],
                                           s.groups, s.eps, out_host=oh, chunk_rows=256)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh, ref)
    ref64 = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                               s.groups, s.eps)
    assert_close(oh.numpy(), ref64, "host pipeline, K = 37, groups of 256")


@pytest.mark.gpu
def test_dconv1d_offset_input_statistics():
    # mean 100, std 0.01: the LayerNorm statistics must not lose the variance
    # to cancellation.
    s = synth.DConv1dShape(B=2, C=64, L=512)
    d = synth.dconv1d_inputs(s, 31, affine="perturbed")
    d["x"] = (d["x"] * np.float32(0.01) + np.float32(100.0)).astype(np.float32)
    got, ref = _dc_run(s, d)
    assert_close(got, ref, "dconv1d offset input")


# ------------------------------------------------- CUDA graph capture
def test_calls_replay_from_a_cuda_graph():
    # every device entry point is stream-ordered and allocates nothing, so a
    # captured call replays to the eager result bit for bit (the workspace
    # comes from the binding's cache, filled by the eager calls)
    s1, d1 = _lgn_case(300, 64, 256, 4, 5)
    s2 = synth.LinearLSEShape(M=100, K=64, N=500)
    d2 = synth.linear_lse_inputs(s2, 6)
    s3 = synth.DConv1dShape(B=2, C=64, L=128, dilation=2, padding=2)
    d3 = synth.dconv1d_inputs(s3, 7)
    s4 = synth.ConvT3dShape(N=2, D=4, H=8, W=8)   # the single cooperative kernel
    d4 = synth.convt3d_inputs(s4, 8)
    s5 = synth.ConvT3dShape(N=2, Cout=8, groups=2, D=3, H=4, W=4, k=4)  # the general kernels
    d5 = synth.convt3d_inputs(s5, 9)
    # device inputs first: a capture may contain no host-to-device copy
    g1 = [T(d1[k]) for k in ("x", "W", "b_lin", "bias", "gamma", "beta")]
    g2 = [T(d2[k]) for k in ("x", "W", "b")]
    g3 = [T(d3[k]) for k in ("x", "ln_gamma", "ln_beta", "conv_w", "conv_b")]
    g4 = [T(d4[k]) for k in ("x", "w", "b", "gamma", "beta")]
    g5 = [T(d5[k]) for k in ("x", "w", "b", "gamma", "beta")]
    calls = [
        lambda: gf.gf_linear_swish_bias_groupnorm(*g1, s1.groups, s1.eps),
        lambda: gf.gf_linear_lse_act(*g2, s2.negative_slope),
        lambda: gf.gf_ln_gelu_dconv1d_res(*g3, s3.dilation, s3.padding, s3.eps),
        lambda: gf.gf_convt3d_swish_gn_hswish(*g4, s4.stride, s4.pad, s4.groups, s4.eps),
        lambda: gf.gf_convt3d_swish_gn_hswish(*g5, s5.stride, s5.pad, s5.groups, s5.eps),
    ]
    for i, call in enumerate(calls):
        ref = call().clone()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            out = call()
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {i}"


def test_calls_on_two_streams_use_separate_default_workspaces():
    # the lo planes of x and W live in the workspace: two concurrent calls
    # with different inputs would corrupt each other through a shared one
    s, d = _lgn_case(2048, 512, 2048, 32, 21)
    x2 = d["x"][::-1].copy()
    rest = [T(d[k]) for k in ("W", "b_lin", "bias", "gamma", "beta")]
    xa, xb = T(d["x"]), T(x2)
    ref_a = gf.gf_linear_swish_bias_groupnorm(xa, *rest, s.groups, s.eps).clone()
    ref_b = gf.gf_linear_swish_bias_groupnorm(xb, *rest, s.groups, s.eps).clone()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        with torch.cuda.stream(sa):
            oa = gf.gf_linear_swish_bias_groupnorm(xa, *rest, s.groups, s.eps, stream=sa)
        with torch.cuda.stream(sb):
            ob = gf.gf_linear_swish_bias_groupnorm(xb, *rest, s.groups, s.eps, stream=sb)
        torch.cuda.synchronize()
        assert torch.equal(oa, ref_a) and torch.equal(ob, ref_b)
