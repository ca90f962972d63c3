"""Plant plausible mistakes in the oracle (on the CPU) and check that at least
one pin fails for each: evidence that the pins can see a dropped term, a wrong
sign or index, or a transposed operand."""
import numpy as np
import pytest

import oracle
import oracle.ops as ops
import tests.test_oracle_pins as P


_ORIG = {n: getattr(ops, n) for n in ("group_norm_rows", "dilated_conv1d", "conv_transpose3d_zero_insert",
                                      "conv_transpose3d_scatter", "layer_norm_sample", "group_norm_nc",
                                      "ln_gelu_dconv1d_res", "linear_lse_act")}


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(ops, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _gn_unbiased(t, groups, gamma=None, beta=None, eps=1e-5):
    t = np.asarray(t, np.float64)
    M, C = t.shape
    tg = t.reshape(M, groups, C // groups)
    mu = tg.mean(axis=2, keepdims=True)
    var = ((tg - mu) ** 2).sum(axis=2, keepdims=True) / (C // groups - 1)
    o = ((tg - mu) / np.sqrt(var + eps)).reshape(M, C)
    return o * (1 if gamma is None else gamma) + (0 if beta is None else beta)


def _gn_no_eps(t, groups, gamma=None, beta=None, eps=1e-5):
    return _ORIG["group_norm_rows"](t, groups, gamma, beta, 0.0)


def _lsbg_bias_first(x, W, b_lin, bias, gamma, beta, groups, eps=1e-5):
    y = ops.linear(x, W, b_lin) + np.asarray(bias, np.float64)[None, :]
    return ops.group_norm_rows(ops.silu(y), groups, gamma, beta, eps)


def _conv_flipped_taps(a, w, b, dilation, padding):
    return _ORIG["dilated_conv1d"](a, np.asarray(w)[:, :, ::-1], b, dilation, padding)


def _zero_insert_no_flip(x, w, b, stride, pad):
    return _ORIG["conv_transpose3d_zero_insert"](x, np.asarray(w)[:, :, ::-1, ::-1, ::-1], b, stride, pad)


def _lse_no_max_log(y):
    y = np.asarray(y, np.float64)
    return np.exp(y).sum(axis=1)


def _ln_no_eps(x, gamma=None, beta=None, eps=1e-5):
    return _ORIG["layer_norm_sample"](x, gamma, beta, 0.0)


def _gelu_tanh(v):
    v = np.asarray(v, np.float64)
    return 0.5 * v * (1 + np.tanh(np.sqrt(2 / np.pi) * (v + 0.044715 * v ** 3)))


def _gelu_tanh_wrong_cubic(v):
    v = np.asarray(v, np.float64)
    return 0.5 * v * (1 + np.tanh(np.sqrt(2 / np.pi) * (v + 0.0447 * v ** 2)))


def _gelu_tanh_is_erf(v):
    return oracle.gelu_erf(v)


def _silu_is_sigmoid(v):
    v = np.asarray(v, np.float64)
    return 1.0 / (1.0 + np.exp(-v))


def _lrelu_wrong_slope(v, negative_slope=0.01):
    v = np.asarray(v, np.float64)
    return np.where(v > 0, v, 0.1 * v)


def _linear_transposed_w(x, W, b=None):
    # reads W as [in, out] instead of [out, in] (only defined when in == out)
    W = np.asarray(W, np.float64)
    x = np.asarray(x, np.float64)
    Wt = W.reshape(W.shape[1], W.shape[0])
    y = x @ Wt
    return y if b is None else y + np.asarray(b, np.float64)[None, :]


def _hswish_no_sixth(v):
    v = np.asarray(v, np.float64)
    return v * np.clip(v + 3, 0, 6)


def _hswish_no_factor(v):
    v = np.asarray(v, np.float64)
    return np.clip(v + 3, 0, 6) / 6


def _gn_nc_per_channel(t, groups, gamma=None, beta=None, eps=1e-5):
    # statistics per channel (instance norm) instead of per group of channels
    return _ORIG["group_norm_nc"](t, np.shape(t)[1], gamma, beta, eps)


def _gn_nc_pooled_batch(t, groups, gamma=None, beta=None, eps=1e-5):
    # statistics pooled over the batch instead of per sample
    t = np.asarray(t, np.float64)
    N, C = t.shape[:2]
    tg = np.moveaxis(t, 0, 1).reshape(groups, -1)
    mu = tg.mean(axis=1, keepdims=True)
    var = ((tg - mu) ** 2).mean(axis=1, keepdims=True)
    o = np.moveaxis(((tg - mu) / np.sqrt(var + eps)).reshape((C, N) + t.shape[2:]), 0, 1)
    bshape = (1, C) + (1,) * (t.ndim - 2)
    if gamma is not None:
        o = o * np.asarray(gamma, np.float64).reshape(bshape)
    if beta is not None:
        o = o + np.asarray(beta, np.float64).reshape(bshape)
    return o


def _gn_rows_interleaved(t, groups, gamma=None, beta=None, eps=1e-5):
    # channel n in group n % groups instead of n // (N / groups)
    t = np.asarray(t, np.float64)
    M, C = t.shape
    cg = C // groups
    perm = np.arange(C).reshape(cg, groups).T.ravel()  # the channels of each strided group, adjacent
    o = np.empty_like(t)
    o[:, perm] = _ORIG["group_norm_rows"](t[:, perm], groups)
    return o * (1 if gamma is None else np.asarray(gamma)) + (0 if beta is None else np.asarray(beta))


def _scatter_flipped(x, w, b, stride, pad):
    return _ORIG["conv_transpose3d_scatter"](x, np.asarray(w)[:, :, ::-1, ::-1, ::-1], b, stride, pad)


def _scatter_no_bias(x, w, b, stride, pad):
    return _ORIG["conv_transpose3d_scatter"](x, w, None, stride, pad)


def _convt_chain_gn_before_swish(x, w, b, gamma, beta, stride, pad, groups, eps=1e-5):
    y = ops.conv_transpose3d_scatter(x, w, b, stride, pad)
    return ops.hardswish(ops.silu(ops.group_norm_nc(y, groups, gamma, beta, eps)))


def _dconv_no_residual(x, ln_gamma, ln_beta, conv_w, conv_b, dilation, padding, eps=1e-5, gelu="erf"):
    return _ORIG["ln_gelu_dconv1d_res"](x, ln_gamma, ln_beta, conv_w, conv_b, dilation, padding, eps, gelu) - \
        np.asarray(x, np.float64)


def _conv_shifted_taps(a, w, b, dilation, padding):
    # taps at j + k d instead of j - p + k d (all the padding put on the right)
    a, w = np.asarray(a, np.float64), np.asarray(w, np.float64)
    B, C, L = a.shape
    ap = np.concatenate([a, np.zeros((B, C, 2 * padding))], axis=2)
    out = sum(np.matmul(w[:, :, k], ap[:, :, k * dilation:k * dilation + L]) for k in range(w.shape[2]))
    return out + (0 if b is None else np.asarray(b, np.float64)[None, :, None])


def _ln_per_channel(x, gamma=None, beta=None, eps=1e-5):
    x = np.asarray(x, np.float64)
    mu = x.mean(axis=2, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=2, keepdims=True)
    o = (x - mu) / np.sqrt(var + eps)
    if gamma is not None:
        o = o * np.asarray(gamma, np.float64)[None]
    if beta is not None:
        o = o + np.asarray(beta, np.float64)[None]
    return o


def _lse_chain_one_lrelu(x, W, b, negative_slope=0.01):
    lse = ops.logsumexp_rows(ops.linear(x, W, b))[:, None]
    return ops.gelu_erf(ops.gelu_erf(ops.leaky_relu(lse, negative_slope)))


def _lse_chain_one_gelu(x, W, b, negative_slope=0.01):
    lse = ops.logsumexp_rows(ops.linear(x, W, b))[:, None]
    return ops.gelu_erf(ops.leaky_relu(ops.leaky_relu(lse, negative_slope), negative_slope))


MUTATIONS = [
    ("group_norm_rows", _gn_unbiased, [P.test_o1_gn_invariants_mean0_var_ratio, P.test_o1_torch_float64_cross_check]),
    ("group_norm_rows", _gn_no_eps, [P.test_o1_gn_invariants_mean0_var_ratio]),
    ("linear_swish_bias_groupnorm", _lsbg_bias_first, [P.test_o1_brute_force_tiny]),
    ("silu", _silu_is_sigmoid, [P.test_silu_extremes]),
    ("dilated_conv1d", _conv_flipped_taps, [P.test_o3_tap_offsets_delta_weights]),
    ("conv_transpose3d_zero_insert", _zero_insert_no_flip, [P.test_o4_scatter_equals_zero_insert_with_flip]),
    ("logsumexp_rows", _lse_no_max_log, [P.test_o2_constant_row_closed_form]),
    ("layer_norm_sample", _ln_no_eps, [P.test_o3_ln_invariant]),
    ("gelu_erf", _gelu_tanh, [P.test_gelu_is_erf_not_tanh]),
    ("gelu_tanh", _gelu_tanh_wrong_cubic, [P.test_gelu_tanh_form, P.test_o3_tanh_gelu_variant]),
    ("gelu_tanh", _gelu_tanh_is_erf, [P.test_gelu_tanh_form, P.test_o3_tanh_gelu_variant]),
    ("leaky_relu", _lrelu_wrong_slope, [P.test_o2_negative_branch]),
    ("linear", _linear_transposed_w, [P.test_o2_brute_force_tiny]),
    ("hardswish", _hswish_no_sixth, [P.test_hardswish_knots]),
    ("hardswish", _hswish_no_factor, [P.test_hardswish_knots]),
    ("group_norm_nc", _gn_nc_per_channel, [P.test_o4_gn_invariants, P.test_o4_brute_force_tiny]),
    ("group_norm_nc", _gn_nc_pooled_batch, [P.test_o4_gn_invariants, P.test_o4_torch_float64_cross_check]),
    ("group_norm_rows", _gn_rows_interleaved, [P.test_o1_brute_force_tiny, P.test_o1_torch_float64_cross_check]),
    ("conv_transpose3d_scatter", _scatter_flipped, [P.test_o4_scatter_equals_zero_insert_with_flip,
                                                    P.test_o4_torch_float64_cross_check]),
    ("conv_transpose3d_scatter", _scatter_no_bias, [P.test_o4_brute_force_tiny]),
    ("convt3d_swish_gn_hswish", _convt_chain_gn_before_swish, [P.test_o4_brute_force_tiny,
                                                               P.test_o4_torch_float64_cross_check]),
    ("ln_gelu_dconv1d_res", _dconv_no_residual, [P.test_o3_torch_float64_cross_check]),
    ("dilated_conv1d", _conv_shifted_taps, [P.test_o3_tap_offsets_delta_weights]),
    ("layer_norm_sample", _ln_per_channel, [P.test_o3_ln_invariant, P.test_o3_torch_float64_cross_check]),
    ("linear_lse_act", _lse_chain_one_lrelu, [P.test_o2_negative_branch, P.test_o2_torch_float64_cross_check]),
    ("linear_lse_act", _lse_chain_one_gelu, [P.test_o2_brute_force_tiny, P.test_o2_torch_float64_cross_check]),
]


@pytest.mark.parametrize("name,mutant,pins", MUTATIONS, ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_pin_catches_planted_mistake(monkeypatch, name, mutant, pins):
    _patch(monkeypatch, name, mutant)
    failures = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught mutant {mutant.__name__} of {name}"
