"""The Python binding rejects tensors whose shapes disagree with the sizes it
derives from the leading operands, before any device or library call: the C
entry points take only sizes and pointers, so a short bias or a W with the
wrong K would otherwise be read past its end.  CPU tensors suffice: the shape
checks come first, and tensors of the right shapes then fail the CUDA check.
Also: the cached default workspaces are dropped on request."""
import pytest
import torch

from conv_activation_normalization_gb300 import binding as gf


def z(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def _raises(match, fn, *a, **k):
    with pytest.raises(ValueError, match=match):
        fn(*a, **k)


def test_linear_shapes():
    M, K, N = 8, 12, 16
    _raises("W has shape", gf.gf_linear, z(M, K), z(N, K + 1))
    _raises("b holds", gf.gf_linear, z(M, K), z(N, K), z(N - 1))
    _raises("out has shape", gf.gf_linear, z(M, K), z(N, K), None, out=z(N, M))
    _raises("CUDA", gf.gf_linear, z(M, K), z(N, K), z(N), out=z(M, N))


def test_linear_groupnorm_shapes():
    M, K, N, G = 8, 12, 16, 4
    ok = dict(x=z(M, K), W=z(N, K), b_lin=z(N), bias=z(N), gamma=z(N), beta=z(N), groups=G)
    for name, bad, msg in (("W", z(N, K - 1), "W has shape"), ("b_lin", z(N + 1), "b_lin holds"),
                           ("bias", z(1), "bias holds"), ("gamma", z(2, N), "gamma holds"),
                           ("beta", z(N - 4), "beta holds")):
        _raises(msg, gf.gf_linear_swish_bias_groupnorm, **{**ok, name: bad})
    _raises("out has shape", gf.gf_linear_swish_bias_groupnorm, **ok, out=z(M, N + 1))
    _raises("CUDA", gf.gf_linear_swish_bias_groupnorm, **ok)
    # the pre-split and host-buffer forms check the same
    _raises("W_planes has shape", gf.gf_linear_swish_bias_groupnorm_planes, z(2, M, K), z(2, N, K + 4), z(N), z(N),
            z(N), z(N), G)
    _raises("x_planes has shape", gf.gf_linear_swish_bias_groupnorm_planes, z(3, M, K), z(2, N, K), z(N), z(N),
            z(N), z(N), G)
    _raises("gamma holds", gf.gf_linear_swish_bias_groupnorm_host, z(M, K), z(N, K), z(N), z(N), z(N + 1), z(N), G)
    _raises("out_host has shape", gf.gf_linear_swish_bias_groupnorm_host, z(M, K), z(N, K), z(N), z(N), z(N), z(N),
            G, out_host=z(M + 1, N))
    _raises("planes has shape", gf.gf_tf32_split, z(M, K), z(2, M, K + 1))


def test_linear_lse_shapes():
    M, K, N = 8, 12, 40
    _raises("W has shape", gf.gf_linear_lse_act, z(M, K), z(K, N), z(N))
    _raises("b holds", gf.gf_linear_lse_act, z(M, K), z(N, K), z(K))
    _raises("out holds", gf.gf_linear_lse_act, z(M, K), z(N, K), z(N), out=z(M + 1, 1))
    _raises("CUDA", gf.gf_linear_lse_act, z(M, K), z(N, K), z(N), out=z(M))  # [M] and [M, 1] both hold M


def test_dconv1d_shapes():
    B, C, L, k = 2, 6, 20, 3
    ok = dict(x=z(B, C, L), ln_gamma=z(C, L), ln_beta=z(C, L), conv_w=z(C, C, k), conv_b=z(C), dilation=2, padding=2)
    for name, bad, msg in (("ln_gamma", z(C, L - 1), "ln_gamma holds"), ("ln_beta", z(L), "ln_beta holds"),
                           ("conv_w", z(C + 1, C, k), "conv_w has shape"), ("conv_w", z(C, C - 1, k), "conv_w has shape"),
                           ("conv_b", z(C + 2), "conv_b holds")):
        _raises(msg, gf.gf_ln_gelu_dconv1d_res, **{**ok, name: bad})
    _raises("out has shape", gf.gf_ln_gelu_dconv1d_res, **ok, out=z(B, C, L + 1))
    _raises("CUDA", gf.gf_ln_gelu_dconv1d_res, **{**ok, "conv_b": None})


@pytest.mark.parametrize("fn", [gf.gf_convt3d_swish_gn_hswish, gf.gf_convt3d_swish_gn_hswish_noalloc])
def test_convt3d_shapes(fn):
    N, Cin, Cout, k = 2, 3, 8, 3
    x = z(N, Cin, 4, 5, 6)
    ok = dict(x=x, w=z(Cin, Cout, k, k, k), b=z(Cout), gamma=z(Cout), beta=z(Cout), stride=2, pad=1, groups=2)
    for name, bad, msg in (("w", z(Cin + 1, Cout, k, k, k), "w has shape"), ("w", z(Cin, Cout, k, k, k - 1),
                                                                             "w has shape"),
                           ("b", z(Cout - 1), "b holds"), ("gamma", z(2 * Cout), "gamma holds"),
                           ("beta", z(1), "beta holds")):
        _raises(msg, fn, **{**ok, name: bad})
    # out [N, Cout, (I-1)*2 - 2 + 3 ...] = [2, 8, 7, 9, 11]
    assert gf.convt3d_out_shape(x.shape, Cout, k, 2, 1) == (2, 8, 7, 9, 11)
    _raises("out has shape", fn, **ok, out=z(2, 8, 8, 9, 11))
    _raises("CUDA", fn, **{**ok, "b": None}, out=z(2, 8, 7, 9, 11))


def test_release_workspaces_empties_the_cache():
    gf.release_workspaces()
    gf._ws_cache[(0, 0)] = z(4)  # stands in for a cached buffer (no device needed)
    gf._ws_cache[(0, 1)] = z(4)
    assert gf.release_workspaces() == 2
    assert gf._ws_cache == {} and gf.release_workspaces() == 0
