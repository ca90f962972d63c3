"""Plain float64 definitions of the four operator chains.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Nothing here is tuned:
every step is the textbook definition, written so that it can be checked
against the source pages by eye.

Source pages (POPCORNBENCH level-2 agent transcripts; "turn n" is the n-th
agent turn on that page):
  * Kimi-K2.6__l2_p37  Linear -> Swish -> +bias -> GroupNorm
  * Kimi-K2.6__l2_p64  Linear -> logsumexp -> LeakyReLU x2 -> GELU x2
  * Kimi-K2.6__l2_p5   LayerNorm -> GELU -> dilated Conv1d -> +x
  * Kimi-K2.6__l2_p60  ConvTranspose3d -> Swish -> GroupNorm -> HardSwish
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf as _erf


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- activations
def silu(v):
    """Swish / SiLU: ``v * sigmoid(v)`` with ``sigmoid(v) = 1 / (1 + e^-v)``.

    Page Kimi-K2.6__l2_p37, turn 1 (the model multiplies its input by its sigmoid);
    page Kimi-K2.6__l2_p60, turn 1 (swish before the GroupNorm).
    For v below about -709, e^-v overflows to inf and the quotient is the
    correct limit -0.
    """
    v = _f64(v)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def gelu_erf(v):
    """Exact GELU ``v * Phi(v) = 0.5 v (1 + erf(v / sqrt 2))``.

    Page Kimi-K2.6__l2_p64, turn 1 (PyTorch's ``approximate='none'`` default,
    the erf form).  The tanh form that page Kimi-K2.6__l2_p5 turn 2 claims is
    the default is not used (it is not PyTorch's default).
    """
    v = _f64(v)
    return 0.5 * v * (1.0 + _erf(v / np.sqrt(2.0)))


def gelu_tanh(v):
    """The tanh approximation of GELU,
    ``0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))``: the form page
    Kimi-K2.6__l2_p5 turn 2 takes for the module's GELU (an opt-in variant
    here; the erf form stays the default)."""
    v = _f64(v)
    return 0.5 * v * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (v + 0.044715 * v ** 3)))


def hardswish(v):
    """HardSwish ``v * clamp(v + 3, 0, 6) / 6`` (page Kimi-K2.6__l2_p60, turn 1)."""
    v = _f64(v)
    return v * np.clip(v + 3.0, 0.0, 6.0) / 6.0


def leaky_relu(v, negative_slope=0.01):
    """``v if v > 0 else negative_slope * v`` (page Kimi-K2.6__l2_p64, turn 1)."""
    v = _f64(v)
    return np.where(v > 0.0, v, negative_slope * v)


# ------------------------------------------------- O1: Linear->Swish->bias->GN
def linear(x, W, b=None):
    """``y[m, n] = sum_k x[m, k] W[n, k] + b[n]`` with W stored [out, in]
    (nn.Linear / addmm; page Kimi-K2.6__l2_p37, turn 1)."""
    y = _f64(x) @ _f64(W).T
    if b is not None:
        y = y + _f64(b)[None, :]
    return y


def group_norm_rows(t, groups, gamma=None, beta=None, eps=1e-5):
    """GroupNorm of a [M, C] tensor: per row, per group of C/groups contiguous
    channels, subtract the mean and divide by sqrt(biased variance + eps), then
    the per-channel affine.

    Page Kimi-K2.6__l2_p37, turn 1: statistics per sample and per group of 64
    contiguous channels, population (biased) variance, eps 1e-5, affine gamma
    and beta per channel.
    """
    t = _f64(t)
    M, C = t.shape
    if C % groups:
        raise ValueError("channels not divisible by groups")
    tg = t.reshape(M, groups, C // groups)
    mu = tg.mean(axis=2, keepdims=True)
    var = ((tg - mu) ** 2).mean(axis=2, keepdims=True)
    o = ((tg - mu) / np.sqrt(var + eps)).reshape(M, C)
    if gamma is not None:
        o = o * _f64(gamma)[None, :]
    if beta is not None:
        o = o + _f64(beta)[None, :]
    return o


def linear_swish_bias_groupnorm(x, W, b_lin, bias, gamma, beta, groups, eps=1e-5):
    """O1.  ``GN(swish(x W^T + b_lin) + bias)``.

    Order fixed by page Kimi-K2.6__l2_p37, turn 1: the linear (with its own
    bias), then Swish, then the extra per-channel bias, then GroupNorm.
    """
    y = linear(x, W, b_lin)
    t = silu(y) + _f64(bias)[None, :]
    return group_norm_rows(t, groups, gamma, beta, eps)


# ---------------------------------------------- O2: Linear->LSE->LReLU2->GELU2
def logsumexp_rows(y):
    """Stable row-wise logsumexp ``m + ln sum_j e^(y_j - m)``, ``m = max_j y_j``
    (page Kimi-K2.6__l2_p64, turn 1)."""
    y = _f64(y)
    m = y.max(axis=1)
    return m + np.log(np.exp(y - m[:, None]).sum(axis=1))


def linear_lse_act(x, W, b, negative_slope=0.01):
    """O2.  out[M, 1] = GELU(GELU(LReLU(LReLU(logsumexp_n(x W^T + b))))).

    Page Kimi-K2.6__l2_p64, turn 1: logsumexp over dim 1 with keepdim, then
    leaky_relu(0.01) twice, then GELU twice (exact erf form).
    """
    lse = logsumexp_rows(linear(x, W, b))[:, None]
    a = leaky_relu(leaky_relu(lse, negative_slope), negative_slope)
    return gelu_erf(gelu_erf(a))


# ------------------------------------------- O3: LN->GELU->dilated Conv1d->+x
def layer_norm_sample(x, gamma=None, beta=None, eps=1e-5):
    """LayerNorm over all of [C, L] for each sample of x[B, C, L]: biased
    variance, eps 1e-5, elementwise affine of shape [C, L].

    Page Kimi-K2.6__l2_p5, turn 1 (normalized_shape = [channels, seq_len]) and
    turn 2 (population variance).
    """
    x = _f64(x)
    mu = x.mean(axis=(1, 2), keepdims=True)
    var = ((x - mu) ** 2).mean(axis=(1, 2), keepdims=True)
    o = (x - mu) / np.sqrt(var + eps)
    if gamma is not None:
        o = o * _f64(gamma)[None]
    if beta is not None:
        o = o + _f64(beta)[None]
    return o


def conv1d_out_len(L, ksize, dilation, padding, stride=1):
    """``floor((L + 2p - d (k - 1) - 1) / s) + 1`` (page Kimi-K2.6__l2_p5, turn 1)."""
    return (L + 2 * padding - dilation * (ksize - 1) - 1) // stride + 1


def dilated_conv1d(a, w, b, dilation, padding):
    """Stride-1 Conv1d as cross-correlation (no kernel flip) with zero padding:
    ``out[b, co, j] = bias[co] + sum_{ci, k} w[co, ci, k] a[b, ci, j - p + k d]``,
    where ``a`` is zero outside [0, L).

    Page Kimi-K2.6__l2_p5, turn 1 (taps at j-4, j, j+4 for k=3, d=4, p=4) and
    turn 2 (cross-correlation; padding zeros apply to the activation).
    """
    a = _f64(a)
    w = _f64(w)
    B, Cin, L = a.shape
    Cout, Cin2, K = w.shape
    assert Cin == Cin2
    Lout = conv1d_out_len(L, K, dilation, padding)
    apad = np.zeros((B, Cin, L + 2 * padding), dtype=np.float64)
    apad[:, :, padding:padding + L] = a
    out = np.zeros((B, Cout, Lout), dtype=np.float64)
    for k in range(K):
        # a_pad index j + k d  <->  a index j - p + k d
        out += np.matmul(w[:, :, k], apad[:, :, k * dilation:k * dilation + Lout])
    if b is not None:
        out += _f64(b)[None, :, None]
    return out


def ln_gelu_dconv1d_res(x, ln_gamma, ln_beta, conv_w, conv_b, dilation, padding, eps=1e-5, gelu="erf"):
    """O3.  ``out = Conv1d(GELU(LayerNorm(x))) + x`` (page Kimi-K2.6__l2_p5,
    turns 1-2).  The residual requires the length-preserving padding.
    ``gelu="tanh"`` takes the tanh approximation (the page's turn-2 reading)."""
    if gelu not in ("erf", "tanh"):
        raise ValueError("gelu must be 'erf' or 'tanh'")
    act = gelu_erf if gelu == "erf" else gelu_tanh
    a = act(layer_norm_sample(x, ln_gamma, ln_beta, eps))
    y = dilated_conv1d(a, conv_w, conv_b, dilation, padding)
    if y.shape != np.shape(x):
        raise ValueError("residual needs L_out == L")
    return y + _f64(x)


# ------------------------------------- O4: ConvT3d->Swish->GroupNorm->HardSwish
def convt3d_out_size(I, k, stride, pad, output_padding=0):
    """``(I - 1) s - 2 p + k + output_padding`` (page Kimi-K2.6__l2_p60, turn 1:
    31 x 63 x 63 for 16 x 32 x 32, k 3, s 2, p 1)."""
    return (I - 1) * stride - 2 * pad + k + output_padding


def _scatter_range(I, O, k, stride, pad):
    """Input indices i with 0 <= s i - p + k < O, and the first output index."""
    i0 = max(0, -((k - pad) // stride))          # ceil((p - k) / s)
    i1 = min(I - 1, (O - 1 + pad - k) // stride)  # floor((O - 1 + p - k) / s)
    return i0, i1, stride * i0 - pad + k


def conv_transpose3d_scatter(x, w, b, stride, pad):
    """ConvTranspose3d by its scatter definition (the authoritative form):
    every input voxel i of channel ci adds ``x[n, ci, i] w[ci, co, k]`` to the
    output voxel ``o = s i - p + k`` (per dimension), for every tap k.
    Weight layout [C_in, C_out, kD, kH, kW] (nn.ConvTranspose3d; page
    Kimi-K2.6__l2_p60, turn 1).
    """
    x = _f64(x)
    w = _f64(w)
    N, Cin, D, H, W = x.shape
    Cin2, Cout, kD, kH, kW = w.shape
    assert Cin == Cin2
    OD = convt3d_out_size(D, kD, stride, pad)
    OH = convt3d_out_size(H, kH, stride, pad)
    OW = convt3d_out_size(W, kW, stride, pad)
    y = np.zeros((N, Cout, OD, OH, OW), dtype=np.float64)
    for kd in range(kD):
        d0, d1, od0 = _scatter_range(D, OD, kd, stride, pad)
        for kh in range(kH):
            h0, h1, oh0 = _scatter_range(H, OH, kh, stride, pad)
            for kw in range(kW):
                w0, w1, ow0 = _scatter_range(W, OW, kw, stride, pad)
                if d1 < d0 or h1 < h0 or w1 < w0:
                    continue
                xs = x[:, :, d0:d1 + 1, h0:h1 + 1, w0:w1 + 1]
                contrib = np.einsum("ncdhw,co->nodhw", xs, w[:, :, kd, kh, kw])
                nd, nh, nw = xs.shape[2:]
                y[:, :,
                  od0:od0 + stride * nd:stride,
                  oh0:oh0 + stride * nh:stride,
                  ow0:ow0 + stride * nw:stride] += contrib
    if b is not None:
        y += _f64(b)[None, :, None, None, None]
    return y


def conv_transpose3d_zero_insert(x, w, b, stride, pad):
    """ConvTranspose3d as the stride-1 convolution of the zero-inserted input
    (page Kimi-K2.6__l2_p60, turn 1): insert s-1 zeros between inputs, pad by
    k-1-p on each side, and cross-correlate with the weight permuted to
    [C_out, C_in, ...] and flipped in every spatial dimension.  The page leaves
    the flip open; it is the reading that agrees with the scatter definition.
    """
    x = _f64(x)
    w = _f64(w)
    N, Cin, D, H, W = x.shape
    _, Cout, kD, kH, kW = w.shape
    assert kD == kH == kW
    k = kD
    q = k - 1 - pad
    if q < 0:
        raise ValueError("zero-insertion form needs pad <= k - 1")
    Z = lambda I: stride * (I - 1) + 1  # noqa: E731
    z = np.zeros((N, Cin, Z(D) + 2 * q, Z(H) + 2 * q, Z(W) + 2 * q), dtype=np.float64)
    z[:, :, q:q + Z(D):stride, q:q + Z(H):stride, q:q + Z(W):stride] = x
    wf = np.transpose(w, (1, 0, 2, 3, 4))[:, :, ::-1, ::-1, ::-1]  # [Cout, Cin, k, k, k]
    OD, OH, OW = (convt3d_out_size(I, k, stride, pad) for I in (D, H, W))
    y = np.zeros((N, Cout, OD, OH, OW), dtype=np.float64)
    for a in range(k):
        for bb in range(k):
            for c in range(k):
                win = z[:, :, a:a + OD, bb:bb + OH, c:c + OW]
                y += np.einsum("ncdhw,oc->nodhw", win, wf[:, :, a, bb, c])
    if b is not None:
        y += _f64(b)[None, :, None, None, None]
    return y


def group_norm_nc(t, groups, gamma=None, beta=None, eps=1e-5):
    """GroupNorm of t[N, C, *spatial]: per sample and group of C/groups
    contiguous channels times all spatial positions; biased variance; per-channel
    affine (page Kimi-K2.6__l2_p60, turn 1: each group is a run of adjacent
    channels, 4 of the 16 here)."""
    t = _f64(t)
    N, C = t.shape[:2]
    if C % groups:
        raise ValueError("channels not divisible by groups")
    tg = t.reshape(N, groups, -1)
    mu = tg.mean(axis=2, keepdims=True)
    var = ((tg - mu) ** 2).mean(axis=2, keepdims=True)
    o = ((tg - mu) / np.sqrt(var + eps)).reshape(t.shape)
    bshape = (1, C) + (1,) * (t.ndim - 2)
    if gamma is not None:
        o = o * _f64(gamma).reshape(bshape)
    if beta is not None:
        o = o + _f64(beta).reshape(bshape)
    return o


def convt3d_swish_gn_hswish(x, w, b, gamma, beta, stride, pad, groups, eps=1e-5):
    """O4.  ``hardswish(GN(swish(ConvTranspose3d(x))))`` (page
    Kimi-K2.6__l2_p60, turn 1)."""
    y = conv_transpose3d_scatter(x, w, b, stride, pad)
    return hardswish(group_norm_nc(silu(y), groups, gamma, beta, eps))
