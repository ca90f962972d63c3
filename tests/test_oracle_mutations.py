"""Plant plausible mistakes in the oracle (on the CPU) and check that at least
one pin fails for each: evidence that the pins can see a dropped term, a wrong
sign or index, or a transposed operand."""
import numpy as np
import pytest

import oracle
import oracle.ops as ops
import tests.test_oracle_pins as P


_ORIG = {n: getattr(ops, n) for n in ("group_norm_rows", "dilated_conv1d",
                                      "conv_transpose3d_zero_insert", "layer_norm_sample")}


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
