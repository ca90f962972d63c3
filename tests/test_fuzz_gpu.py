"""Seeded random shapes for every chain, through the C ABI, against the fp64
oracle: sizes, ragged tails, precision modes, group widths, GELU forms and
ConvTranspose3d configurations drawn from a fixed generator (the same cases
on every run), so that combinations the hand-picked parity cases miss are
covered too.

Tolerances as in the other parity tests: 1e-4 abs + 1e-4 rel in the fp32
modes (3xTF32, 3xBF16), 3e-2 in the BF16 mode.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_activation_normalization_gb300 import binding as gf
from conv_activation_normalization_gb300 import synth

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
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = ~(err <= tol + tol * np.abs(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} outside {tol}; max err {np.nanmax(err):.3g}"


def _cases(seed, n, draw):
    r = np.random.default_rng(seed)
    return [draw(r) for _ in range(n)]


def _lgn_case(r):
    mode = int(r.integers(0, 3))
    gw = int(r.choice([16, 32, 64, 128, 8, 48, 256, 320]))
    return dict(M=int(r.integers(1, 400)), K=int(r.integers(1, 512)), gw=gw, groups=int(r.integers(1, 12)),
                mode=mode, seed=int(r.integers(1 << 30)))


@pytest.mark.parametrize("c", _cases(101, 12, _lgn_case), ids=lambda c: f"M{c['M']}K{c['K']}gw{c['gw']}m{c['mode']}")
def test_fuzz_linear_gn(c):
    s = synth.LinearGNShape(M=c["M"], K=c["K"], N=c["gw"] * c["groups"], groups=c["groups"])
    d = synth.linear_gn_inputs(s, c["seed"])
    got = gf.gf_linear_swish_bias_groupnorm(T(d["x"]), T(d["W"]), T(d["b_lin"]), T(d["bias"]), T(d["gamma"]),
                                            T(d["beta"]), s.groups, s.eps, mode=c["mode"]).cpu().numpy()
    ref = oracle.linear_swish_bias_groupnorm(d["x"], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"], s.groups,
                                             s.eps)
    assert_close(got, ref, TOL[c["mode"]], f"linear_gn {c}")


def _lse_case(r):
    mode = int(r.integers(0, 3))
    return dict(M=int(r.integers(1, 300)), K=int(r.integers(1, 512)), N=int(r.integers(1, 1500)), mode=mode,
                seed=int(r.integers(1 << 30)))


@pytest.mark.parametrize("c", _cases(202, 10, _lse_case), ids=lambda c: f"M{c['M']}K{c['K']}N{c['N']}m{c['mode']}")
def test_fuzz_linear_lse(c):
    s = synth.LinearLSEShape(M=c["M"], K=c["K"], N=c["N"])
    d = synth.linear_lse_inputs(s, c["seed"])
    got = gf.gf_linear_lse_act(T(d["x"]), T(d["W"]), T(d["b"]), s.negative_slope, mode=c["mode"]).cpu().numpy()
    ref = oracle.linear_lse_act(d["x"], d["W"], d["b"], s.negative_slope)
    assert_close(got, ref, TOL[c["mode"]], f"lse {c}")


def _dc_case(r):
    mode = int(r.integers(0, 3))
    ksize = int(r.choice([1, 2, 3, 4, 5, 7]))
    dil = int(r.integers(1, 6))
    if (ksize - 1) * dil % 2:
        dil += 1  # length-preserving padding needs an even span
    return dict(B=int(r.integers(1, 4)), C=int(r.integers(1, 513)), L=int(r.integers(1, 600)),
                ksize=ksize, dil=dil, mode=mode, gelu=str(r.choice(["erf", "tanh"])), seed=int(r.integers(1 << 30)))


@pytest.mark.parametrize("c", _cases(303, 10, _dc_case),
                         ids=lambda c: f"B{c['B']}C{c['C']}L{c['L']}k{c['ksize']}d{c['dil']}m{c['mode']}{c['gelu']}")
def test_fuzz_dconv1d(c):
    pad = (c["ksize"] - 1) * c["dil"] // 2
    s = synth.DConv1dShape(B=c["B"], C=c["C"], L=c["L"], ksize=c["ksize"], dilation=c["dil"], padding=pad)
    d = synth.dconv1d_inputs(s, c["seed"], affine="perturbed")
    got = gf.gf_ln_gelu_dconv1d_res(T(d["x"]), T(d["ln_gamma"]), T(d["ln_beta"]), T(d["conv_w"]), T(d["conv_b"]),
                                    s.dilation, s.padding, s.eps, mode=c["mode"], gelu=c["gelu"]).cpu().numpy()
    ref = oracle.ln_gelu_dconv1d_res(d["x"], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                     s.padding, s.eps, gelu=c["gelu"])
    assert_close(got, ref, TOL[c["mode"]], f"dconv1d {c}")


def _ct_case(r):
    if r.random() < 0.4:  # the pages' configuration with random sizes (specialized kernels)
        return dict(N=int(r.integers(1, 4)), Cin=int(r.integers(1, 9)), Cout=16, G=4, k=3, st=2, pd=1,
                    D=int(r.integers(1, 9)), H=int(r.integers(1, 13)), W=int(r.integers(1, 13)),
                    seed=int(r.integers(1 << 30)))
    while True:
        k = int(r.integers(1, 6))
        st = int(r.integers(1, 4))
        pd = int(r.integers(0, k))
        D, H, W = (int(v) for v in r.integers(1, 7, 3))
        if min((i - 1) * st - 2 * pd + k for i in (D, H, W)) >= 1:
            break
    Cout = int(r.choice([4, 8, 12, 16, 24]))
    G = int(r.choice([g for g in (1, 2, 3, 4, 8) if Cout % g == 0]))
    return dict(N=int(r.integers(1, 4)), Cin=int(r.integers(1, 11)), Cout=Cout, G=G, k=k, st=st, pd=pd, D=D, H=H, W=W,
                seed=int(r.integers(1 << 30)))


@pytest.mark.parametrize("c", _cases(404, 14, _ct_case),
                         ids=lambda c: f"N{c['N']}Ci{c['Cin']}Co{c['Cout']}G{c['G']}k{c['k']}s{c['st']}p{c['pd']}")
def test_fuzz_convt3d(c):
    s = synth.ConvT3dShape(N=c["N"], Cin=c["Cin"], Cout=c["Cout"], D=c["D"], H=c["H"], W=c["W"], k=c["k"],
                           stride=c["st"], pad=c["pd"], groups=c["G"])
    d = synth.convt3d_inputs(s, c["seed"])
    got = gf.gf_convt3d_swish_gn_hswish(T(d["x"]), T(d["w"]), T(d["b"]), T(d["gamma"]), T(d["beta"]), s.stride, s.pad,
                                        s.groups, s.eps).cpu().numpy()
    ref = oracle.convt3d_swish_gn_hswish(d["x"], d["w"], d["b"], d["gamma"], d["beta"], s.stride, s.pad, s.groups,
                                         s.eps)
    assert_close(got, ref, 1e-4, f"convt3d {c}")
