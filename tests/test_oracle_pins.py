"""Pins for the fp64 oracle, independent of the oracle itself.

Each test checks an oracle function against something the pages or the
mathematics fix: values the pages print (tests/golden/page_facts.json), closed
forms, invariants, special cases that reduce to a library routine (torch CPU
float64), and brute force written as plain Python loops on tiny inputs.
No GPU is used.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def rng(seed):
    return np.random.default_rng(seed)


def _t(a):
    return torch.tensor(np.asarray(a, dtype=np.float64))


# ============================================================ O1 pins
def _bf_linear_swish_bias_gn(x, W, b_lin, bias, gamma, beta, G, eps):
    """Plain-loop brute force: one scalar at a time."""
    M, K = len(x), len(x[0])
    N = len(W)
    cg = N // G
    out = [[0.0] * N for _ in range(M)]
    for m in range(M):
        t = []
        for n in range(N):
            y = b_lin[n]
            for k in range(K):
                y += x[m][k] * W[n][k]
            s = y * (1.0 / (1.0 + math.exp(-y)))
            t.append(s + bias[n])
        for g in range(G):
            vals = t[g * cg:(g + 1) * cg]
            mu = sum(vals) / cg
            var = sum((v - mu) ** 2 for v in vals) / cg
            for i, v in enumerate(vals):
                n = g * cg + i
                out[m][n] = (v - mu) / math.sqrt(var + eps) * gamma[n] + beta[n]
    return np.array(out)


def test_o1_brute_force_tiny():
    r = rng(1)
    M, K, N, G = 3, 5, 8, 2
    x, W = r.normal(size=(M, K)), r.normal(size=(N, K)) * 0.5
    b_lin, bias = r.normal(size=N), r.normal(size=N)
    gamma, beta = r.uniform(0.5, 1.5, N), r.normal(size=N) * 0.1
    ref = _bf_linear_swish_bias_gn(x.tolist(), W.tolist(), b_lin, bias, gamma, beta, G, 1e-5)
    got = oracle.linear_swish_bias_groupnorm(x, W, b_lin, bias, gamma, beta, G, 1e-5)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_o1_gn_invariants_mean0_var_ratio():
    # gamma = 1, beta = 0: every (row, group) has mean 0 and mean square
    # v/(v+eps), where v is the group's biased variance -- not exactly 1.
    r = rng(2)
    M, N, G, eps = 4, 64, 4, 1e-2
    t = r.normal(size=(M, N)) * r.uniform(0.05, 2.0, size=(M, 1))
    o = oracle.group_norm_rows(t, G, np.ones(N), np.zeros(N), eps)
    tg = t.reshape(M, G, -1)
    v = tg.var(axis=2)  # numpy biased variance
    og = o.reshape(M, G, -1)
    np.testing.assert_allclose(og.mean(axis=2), 0.0, atol=1e-12)
    np.testing.assert_allclose((og ** 2).mean(axis=2), v / (v + eps), rtol=1e-12)


def test_o1_permutation_within_group():
    r = rng(3)
    M, K, N, G = 5, 7, 16, 2
    x, W = r.normal(size=(M, K)), r.normal(size=(N, K))
    b_lin, bias = r.normal(size=N), r.normal(size=N)
    gamma, beta = r.uniform(0.5, 1.5, N), r.normal(size=N)
    perm = np.concatenate([r.permutation(8), 8 + r.permutation(8)])
    a = oracle.linear_swish_bias_groupnorm(x, W, b_lin, bias, gamma, beta, G)
    b = oracle.linear_swish_bias_groupnorm(x, W[perm], b_lin[perm], bias[perm], gamma[perm], beta[perm], G)
    np.testing.assert_allclose(b, a[:, perm], rtol=1e-13, atol=1e-13)


def test_o1_integer_contraction_exact():
    r = rng(4)
    x = r.integers(-15, 16, size=(6, 33))
    W = r.integers(-15, 16, size=(10, 33))
    exact = [[sum(int(x[m, k]) * int(W[n, k]) for k in range(33)) for n in range(10)] for m in range(6)]
    assert np.array_equal(oracle.linear(x, W), np.array(exact, dtype=np.float64))


def test_o1_single_channel_groups_give_beta():
    # groups == channels: t - mu == 0 in every group, so the output is beta.
    r = rng(5)
    M, K, N = 3, 4, 8
    beta = r.normal(size=N)
    o = oracle.linear_swish_bias_groupnorm(r.normal(size=(M, K)), r.normal(size=(N, K)), r.normal(size=N),
                                           r.normal(size=N), r.uniform(0.5, 1.5, N), beta, groups=N)
    np.testing.assert_array_equal(o, np.broadcast_to(beta, (M, N)))


def test_o1_torch_float64_cross_check():
    r = rng(6)
    M, K, N, G = 16, 40, 128, 2
    x, W = r.normal(size=(M, K)), r.uniform(-0.2, 0.2, (N, K))
    b_lin, bias = r.uniform(-0.2, 0.2, N), r.normal(size=N)
    gamma, beta = r.uniform(0.5, 1.5, N), r.normal(size=N) * 0.1
    ref = F.group_norm(F.silu(F.linear(_t(x), _t(W), _t(b_lin))) + _t(bias), G, _t(gamma), _t(beta), 1e-5)
    got = oracle.linear_swish_bias_groupnorm(x, W, b_lin, bias, gamma, beta, G, 1e-5)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_o1_page_group_width():
    f = GOLDEN["gn_channels_per_group"]
    assert f["N"] // f["groups"] == f["channels_per_group"] == 64


def test_silu_extremes():
    v = np.array([-1000.0, -50.0, 0.0, 50.0, 1000.0])
    s = oracle.silu(v)
    assert s[0] == 0.0 and s[2] == 0.0 and s[4] == 1000.0
    assert abs(s[1] - (-50.0 * math.exp(-50.0) / (1 + math.exp(-50.0)))) < 1e-30
    np.testing.assert_allclose(s, F.silu(_t(v)).numpy(), rtol=1e-15, atol=0)


# ============================================================ O2 pins
def test_o2_constant_row_closed_form():
    f = GOLDEN["lse_closed_form"]
    N = f["N"]
    c = 0.37
    y = np.full((2, N), c)
    lse = oracle.logsumexp_rows(y)
    np.testing.assert_allclose(lse, c + f["ln_N"], rtol=0, atol=1e-12)
    assert abs(f["ln_N"] - math.log(N)) < 1e-15


def test_o2_shift_invariance_and_large_values():
    r = rng(7)
    y = r.normal(size=(3, 50))
    base = oracle.logsumexp_rows(y)
    np.testing.assert_allclose(oracle.logsumexp_rows(y + 1000.0), base + 1000.0, rtol=0, atol=1e-10)
    np.testing.assert_allclose(oracle.logsumexp_rows(y - 1000.0), base - 1000.0, rtol=0, atol=1e-10)
    assert np.all(np.isfinite(oracle.logsumexp_rows(y * 1e3)))


def test_o2_zero_weight_gives_lse_of_bias():
    r = rng(8)
    M, K, N = 3, 6, 9
    b = r.normal(size=N)
    lse = oracle.logsumexp_rows(oracle.linear(r.normal(size=(M, K)), np.zeros((N, K)), b))
    exact = math.log(sum(math.exp(v) for v in b))
    np.testing.assert_allclose(lse, exact, rtol=1e-14)


def test_o2_negative_branch():
    # b = -30 everywhere and W = 0: lse = -30 + ln 8192; both LeakyReLUs take
    # the 0.01 branch; GELU acts near zero.
    N = 8192
    out = oracle.linear_lse_act(np.ones((1, 4)), np.zeros((N, 4)), np.full(N, -30.0), 0.01)
    lse = -30.0 + math.log(N)
    a = lse * 0.01 * 0.01
    g = F.gelu(F.gelu(torch.tensor([a], dtype=torch.float64))).item()
    assert a < 0
    np.testing.assert_allclose(out[0, 0], g, rtol=1e-14)


def test_o2_brute_force_tiny():
    r = rng(9)
    M, K, N = 2, 3, 5
    x, W, b = r.normal(size=(M, K)), r.normal(size=(N, K)), r.normal(size=N) * 3
    got = oracle.linear_lse_act(x, W, b, 0.01)
    for m in range(M):
        ys = [b[n] + sum(x[m, k] * W[n, k] for k in range(K)) for n in range(N)]
        s = math.log(sum(math.exp(v) for v in ys))
        for _ in range(2):
            s = s if s > 0 else 0.01 * s
        for _ in range(2):
            s = 0.5 * s * (1.0 + math.erf(s / math.sqrt(2.0)))
        np.testing.assert_allclose(got[m, 0], s, rtol=1e-13)


def test_o2_torch_float64_cross_check():
    r = rng(10)
    M, K, N = 8, 64, 300
    x, W, b = r.normal(size=(M, K)), r.uniform(-0.3, 0.3, (N, K)), r.uniform(-0.3, 0.3, N)
    y = F.linear(_t(x), _t(W), _t(b))
    ref = F.gelu(F.gelu(F.leaky_relu(F.leaky_relu(torch.logsumexp(y, 1, keepdim=True), 0.01), 0.01),
                        approximate="none"), approximate="none")
    got = oracle.linear_lse_act(x, W, b, 0.01)
    assert got.shape == (M, 1)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-13, atol=1e-13)


def test_gelu_is_erf_not_tanh():
    v = np.linspace(-4, 4, 33)
    np.testing.assert_allclose(oracle.gelu_erf(v), F.gelu(_t(v), approximate="none").numpy(), rtol=1e-14, atol=1e-15)
    assert np.abs(oracle.gelu_erf(v) - F.gelu(_t(v), approximate="tanh").numpy()).max() > 1e-5


def test_gelu_tanh_form():
    # against torch's independent tanh-approximate GELU, the odd-part identity
    # g(v) - g(-v) = v shared by both forms (0.5 (1 + h) with h odd), the
    # limits, and the known gap to the erf form (largest near |v| = 2, a few
    # 1e-4, never above 1e-3)
    v = np.linspace(-6, 6, 97)
    np.testing.assert_allclose(oracle.gelu_tanh(v), F.gelu(_t(v), approximate="tanh").numpy(), rtol=1e-14,
                               atol=1e-15)
    np.testing.assert_allclose(oracle.gelu_tanh(v) - oracle.gelu_tanh(-v), v, rtol=0, atol=1e-14)
    assert oracle.gelu_tanh(0.0) == 0.0
    assert abs(oracle.gelu_tanh(30.0) - 30.0) < 1e-12 and abs(oracle.gelu_tanh(-30.0)) < 1e-12
    gap = np.abs(oracle.gelu_tanh(v) - oracle.gelu_erf(v))
    assert 1e-4 < gap.max() < 1e-3


def test_o3_tanh_gelu_variant():
    r = rng(17)
    B, C, L = 2, 8, 40
    x = r.normal(size=(B, C, L))
    g, be = r.uniform(0.5, 1.5, (C, L)), r.normal(size=(C, L)) * 0.1
    w, cb = r.uniform(-0.2, 0.2, (C, C, 3)), r.uniform(-0.2, 0.2, C)
    a = F.gelu(F.layer_norm(_t(x), (C, L), _t(g), _t(be), 1e-5), approximate="tanh")
    ref = F.conv1d(a, _t(w), _t(cb), padding=2, dilation=2) + _t(x)
    got = oracle.ln_gelu_dconv1d_res(x, g, be, w, cb, 2, 2, gelu="tanh")
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.abs(got - oracle.ln_gelu_dconv1d_res(x, g, be, w, cb, 2, 2)).max() > 1e-6
    with pytest.raises(ValueError):
        oracle.ln_gelu_dconv1d_res(x, g, be, w, cb, 2, 2, gelu="sigmoid")


def test_o2_page_flop_counts():
    for key in ("linear_gn_gflop", "linear_lse_gflop"):
        f = GOLDEN[key]
        assert round(2 * f["M"] * f["N"] * f["K"] / 1e9, 1) == f["gflop"]


# ============================================================ O3 pins
def test_o3_out_len_and_gemm_shape():
    f = GOLDEN["conv1d_out_len"]
    assert oracle.conv1d_out_len(f["L"], f["k"], f["dilation"], f["padding"]) == f["out"]
    g = GOLDEN["conv1d_gemm_shape"]
    assert (32 * 4096, 256, 256 * 3) == (g["M"], g["N"], g["K"])


def test_o3_tap_offsets_delta_weights():
    # A weight that is 1 on one (co, ci, k) and 0 elsewhere reads a[j + off_k].
    offs = GOLDEN["conv1d_tap_offsets"]["offsets"]
    r = rng(11)
    B, C, L = 1, 2, 16
    a = r.normal(size=(B, C, L))
    for k, off in enumerate(offs):
        w = np.zeros((C, C, 3))
        w[1, 0, k] = 1.0
        out = oracle.dilated_conv1d(a, w, None, dilation=4, padding=4)
        exp = np.zeros(L)
        for j in range(L):
            if 0 <= j + off < L:
                exp[j] = a[0, 0, j + off]
        np.testing.assert_array_equal(out[0, 1], exp)
        np.testing.assert_array_equal(out[0, 0], 0.0)


def test_o3_center_tap_identity_block():
    # W[co, ci, 1] = delta(co, ci): out = GELU(LN(x)) + conv_b + x.
    r = rng(12)
    B, C, L = 2, 4, 24
    x = r.normal(size=(B, C, L)) * 2 + 0.5
    g, be = r.uniform(0.5, 1.5, (C, L)), r.normal(size=(C, L)) * 0.1
    cb = r.normal(size=C)
    w = np.zeros((C, C, 3))
    w[np.arange(C), np.arange(C), 1] = 1.0
    out = oracle.ln_gelu_dconv1d_res(x, g, be, w, cb, 4, 4)
    ln = F.layer_norm(_t(x), (C, L), _t(g), _t(be), 1e-5)
    exp = F.gelu(ln) + _t(cb)[None, :, None] + _t(x)
    np.testing.assert_allclose(out, exp.numpy(), rtol=1e-12, atol=1e-12)


def test_o3_ln_invariant():
    r = rng(13)
    x = r.normal(size=(3, 5, 7)) * r.uniform(0.01, 3, (3, 1, 1)) + 4.0
    eps = 1e-3
    o = oracle.layer_norm_sample(x, eps=eps)
    v = x.reshape(3, -1).var(axis=1)
    np.testing.assert_allclose(o.reshape(3, -1).mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((o.reshape(3, -1) ** 2).mean(axis=1), v / (v + eps), rtol=1e-12)


@pytest.mark.parametrize("dil", [2, 4])
def test_o3_brute_force_tiny(dil):
    r = rng(14 + dil)
    B, C, L, K = 2, 4, 16, 3
    x = r.normal(size=(B, C, L))
    g, be = r.uniform(0.5, 1.5, (C, L)), r.normal(size=(C, L)) * 0.1
    w, cb = r.normal(size=(C, C, K)), r.normal(size=C)
    pad = dil
    got = oracle.ln_gelu_dconv1d_res(x, g, be, w, cb, dil, pad)
    for b in range(B):
        vals = [x[b, c, l] for c in range(C) for l in range(L)]
        mu = sum(vals) / len(vals)
        var = sum((v - mu) ** 2 for v in vals) / len(vals)
        a = [[0.0] * L for _ in range(C)]
        for c in range(C):
            for l in range(L):
                h = (x[b, c, l] - mu) / math.sqrt(var + 1e-5) * g[c, l] + be[c, l]
                a[c][l] = 0.5 * h * (1 + math.erf(h / math.sqrt(2)))
        for co in range(C):
            for j in range(L):
                acc = cb[co] + x[b, co, j]
                for ci in range(C):
                    for k in range(K):
                        p = j - pad + k * dil
                        if 0 <= p < L:
                            acc += w[co, ci, k] * a[ci][p]
                assert abs(got[b, co, j] - acc) < 1e-12


def test_o3_torch_float64_cross_check():
    r = rng(16)
    B, C, L = 2, 8, 64
    x = r.normal(size=(B, C, L))
    g, be = r.uniform(0.5, 1.5, (C, L)), r.normal(size=(C, L)) * 0.1
    w, cb = r.uniform(-0.2, 0.2, (C, C, 3)), r.uniform(-0.2, 0.2, C)
    a = F.gelu(F.layer_norm(_t(x), (C, L), _t(g), _t(be), 1e-5))
    ref = F.conv1d(a, _t(w), _t(cb), padding=4, dilation=4) + _t(x)
    got = oracle.ln_gelu_dconv1d_res(x, g, be, w, cb, 4, 4)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


# ============================================================ O4 pins
def test_o4_out_size_page_value():
    f = GOLDEN["convt3d_out_size"]
    got = [oracle.convt3d_out_size(i, f["k"], f["stride"], f["pad"]) for i in f["input_dhw"]]
    assert got == f["out_dhw"]
    z = GOLDEN["convt1d_zero_insert_len"]
    for L in (1, 5, 16):
        assert oracle.convt3d_out_size(L, z["k"], z["stride"], z["pad"]) == 2 * L - 1
        zl = z["stride"] * (L - 1) + 1 + 2 * z["zero_insert_pad"]
        assert zl - z["k"] + 1 == 2 * L - 1


def test_o4_errata_counts():
    e = GOLDEN["errata"]
    OD, OH, OW = GOLDEN["convt3d_out_size"]["out_dhw"]
    assert 4 * OD * OH * OW == e["convt_group_elems"]["correct"] != e["convt_group_elems"]["page_value"]
    assert 128 * 16 * OD * OH * OW == e["convt_total_elems"]["correct"] != e["convt_total_elems"]["page_value"]


def _valid_taps_1d(I, O, k, s, p):
    """Per output index, the list of (i, tap) pairs with o = s i - p + tap."""
    taps = [[] for _ in range(O)]
    for i in range(I):
        for t in range(k):
            o = s * i - p + t
            if 0 <= o < O:
                taps[o].append((i, t))
    return taps


def test_o4_taps_per_dim_and_total_count():
    per_dim = set(GOLDEN["convt_taps_per_dim"]["values"])
    tot = 1
    for I in (16, 32, 32):
        O = oracle.convt3d_out_size(I, 3, 2, 1)
        taps = _valid_taps_1d(I, O, 3, 2, 1)
        assert {len(t) for t in taps} == per_dim
        tot *= sum(len(t) for t in taps)
    assert tot == GOLDEN["errata"]["convt_avg_taps"]["correct_valid_triples_per_pair"]


def test_o4_delta_footprint():
    # x = delta at (id, ih, iw), all-ones w, no bias: outputs 2i-1..2i+1 are 1
    # in each dimension (clipped), everything else 0.
    D, H, W = 3, 4, 5
    for (i0, i1, i2) in [(0, 0, 0), (1, 2, 3), (2, 3, 4)]:
        x = np.zeros((1, 1, D, H, W))
        x[0, 0, i0, i1, i2] = 1.0
        y = oracle.conv_transpose3d_scatter(x, np.ones((1, 2, 3, 3, 3)), None, 2, 1)
        exp = np.zeros(y.shape[2:])
        exp[max(0, 2 * i0 - 1):2 * i0 + 2, max(0, 2 * i1 - 1):2 * i1 + 2, max(0, 2 * i2 - 1):2 * i2 + 2] = 1.0
        np.testing.assert_array_equal(y[0, 0], exp)
        np.testing.assert_array_equal(y[0, 1], exp)


def test_o4_scatter_equals_zero_insert_with_flip():
    r = rng(17)
    x = r.normal(size=(2, 3, 3, 4, 5))
    w = r.normal(size=(3, 4, 3, 3, 3))
    b = r.normal(size=4)
    a = oracle.conv_transpose3d_scatter(x, w, b, 2, 1)
    z = oracle.conv_transpose3d_zero_insert(x, w, b, 2, 1)
    np.testing.assert_allclose(a, z, rtol=1e-12, atol=1e-12)


def test_o4_brute_force_tiny():
    r = rng(18)
    N, Cin, Cout, D, H, W, G = 1, 2, 4, 3, 3, 2, 2
    x = r.normal(size=(N, Cin, D, H, W))
    w = r.normal(size=(Cin, Cout, 3, 3, 3)) * 0.3
    b = r.normal(size=Cout) * 0.1
    gamma, beta = r.uniform(0.5, 1.5, Cout), r.normal(size=Cout) * 0.1
    got = oracle.convt3d_swish_gn_hswish(x, w, b, gamma, beta, 2, 1, G)
    OD, OH, OW = (oracle.convt3d_out_size(i, 3, 2, 1) for i in (D, H, W))
    td, th, tw = (_valid_taps_1d(I, O, 3, 2, 1) for I, O in ((D, OD), (H, OH), (W, OW)))
    s = np.zeros((Cout, OD, OH, OW))
    for co in range(Cout):
        for od in range(OD):
            for oh in range(OH):
                for ow in range(OW):
                    y = b[co]
                    for ci in range(Cin):
                        for (id_, kd) in td[od]:
                            for (ih, kh) in th[oh]:
                                for (iw, kw) in tw[ow]:
                                    y += x[0, ci, id_, ih, iw] * w[ci, co, kd, kh, kw]
                    s[co, od, oh, ow] = y / (1 + math.exp(-y))
    cg = Cout // G
    for g in range(G):
        vals = s[g * cg:(g + 1) * cg].ravel()
        mu = vals.sum() / vals.size
        var = ((vals - mu) ** 2).sum() / vals.size
        for c in range(g * cg, (g + 1) * cg):
            h = (s[c] - mu) / math.sqrt(var + 1e-5) * gamma[c] + beta[c]
            hs = h * np.clip(h + 3, 0, 6) / 6
            np.testing.assert_allclose(got[0, c], hs, rtol=1e-12, atol=1e-12)


def test_o4_torch_float64_cross_check():
    r = rng(19)
    x = r.normal(size=(2, 3, 4, 6, 5))
    w = r.uniform(-0.05, 0.05, (3, 16, 3, 3, 3))
    b = r.uniform(-0.05, 0.05, 16)
    gamma, beta = r.uniform(0.5, 1.5, 16), r.normal(size=16) * 0.1
    y = F.conv_transpose3d(_t(x), _t(w), _t(b), stride=2, padding=1)
    ref = F.hardswish(F.group_norm(F.silu(y), 4, _t(gamma), _t(beta), 1e-5))
    got = oracle.convt3d_swish_gn_hswish(x, w, b, gamma, beta, 2, 1, 4)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


# Other kernel sizes, strides, paddings, channel counts and groups (the
# module's constructor arguments on page Kimi-K2.6__l2_p60, turn 1)
GENERAL_CT = [(3, 1, 1), (4, 2, 1), (5, 3, 2), (2, 2, 0), (3, 2, 0), (1, 1, 0), (4, 3, 3)]


@pytest.mark.parametrize("k,s,p", GENERAL_CT)
def test_o4_general_scatter_equals_zero_insert_and_torch(k, s, p):
    r = rng(20 + 7 * k + s + p)
    x = r.normal(size=(2, 3, 3, 4, 5))
    w = r.normal(size=(3, 6, k, k, k))
    b = r.normal(size=6)
    a = oracle.conv_transpose3d_scatter(x, w, b, s, p)
    assert a.shape[2:] == tuple(oracle.convt3d_out_size(i, k, s, p) for i in (3, 4, 5))
    np.testing.assert_allclose(a, oracle.conv_transpose3d_zero_insert(x, w, b, s, p), rtol=1e-12, atol=1e-12)
    ref = F.conv_transpose3d(_t(x), _t(w), _t(b), stride=s, padding=p)
    np.testing.assert_allclose(a, ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("k,s,p,Cout,G", [(4, 2, 1, 6, 3), (2, 3, 0, 4, 1), (3, 1, 1, 8, 8)])
def test_o4_general_brute_force_tiny(k, s, p, Cout, G):
    r = rng(30 + k + s + p + Cout)
    N, Cin, D, H, W = 1, 2, 3, 2, 3
    x = r.normal(size=(N, Cin, D, H, W))
    w = r.normal(size=(Cin, Cout, k, k, k)) * 0.3
    b = r.normal(size=Cout) * 0.1
    gamma, beta = r.uniform(0.5, 1.5, Cout), r.normal(size=Cout) * 0.1
    got = oracle.convt3d_swish_gn_hswish(x, w, b, gamma, beta, s, p, G)
    OD, OH, OW = (oracle.convt3d_out_size(i, k, s, p) for i in (D, H, W))
    assert min(OD, OH, OW) >= 1
    td, th, tw = (_valid_taps_1d(I, O, k, s, p) for I, O in ((D, OD), (H, OH), (W, OW)))
    sw = np.zeros((Cout, OD, OH, OW))
    for co in range(Cout):
        for od in range(OD):
            for oh in range(OH):
                for ow in range(OW):
                    y = b[co]
                    for ci in range(Cin):
                        for (id_, kd) in td[od]:
                            for (ih, kh) in th[oh]:
                                for (iw, kw) in tw[ow]:
                                    y += x[0, ci, id_, ih, iw] * w[ci, co, kd, kh, kw]
                    sw[co, od, oh, ow] = y / (1 + math.exp(-y))
    cg = Cout // G
    for g in range(G):
        vals = sw[g * cg:(g + 1) * cg].ravel()
        mu = vals.sum() / vals.size
        var = ((vals - mu) ** 2).sum() / vals.size
        for c in range(g * cg, (g + 1) * cg):
            h = (sw[c] - mu) / math.sqrt(var + 1e-5) * gamma[c] + beta[c]
            np.testing.assert_allclose(got[0, c], h * np.clip(h + 3, 0, 6) / 6, rtol=1e-12, atol=1e-12)


def test_o4_gn_invariants():
    r = rng(20)
    t = r.normal(size=(2, 8, 3, 4, 5)) * 0.05 + 0.02
    eps = 1e-5
    o = oracle.group_norm_nc(t, 2, eps=eps)
    tg = t.reshape(2, 2, -1)
    v = tg.var(axis=2)
    og = o.reshape(2, 2, -1)
    np.testing.assert_allclose(og.mean(axis=2), 0, atol=1e-12)
    np.testing.assert_allclose((og ** 2).mean(axis=2), v / (v + eps), rtol=1e-12)


def test_hardswish_knots():
    v = np.array([-4.0, -3.0, -1.5, 0.0, 1.5, 3.0, 4.0])
    np.testing.assert_array_equal(oracle.hardswish(v), [0.0, 0.0, -0.375, 0.0, 1.125, 3.0, 4.0])
    np.testing.assert_allclose(oracle.hardswish(v), F.hardswish(_t(v)).numpy(), rtol=0, atol=0)
