"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments with the documented status codes
before touching the device (all pointers here are fake and never
dereferenced)."""
import ctypes

import pytest

from conv_activation_normalization_gb300 import binding


@pytest.fixture(scope="module")
def L():
    from conv_activation_normalization_gb300 import build
    build.build()
    return binding.lib()


GF_OK, GF_ERR_NULL, GF_ERR_SHAPE, GF_ERR_ALIGN, GF_ERR_ALIAS, GF_ERR_WORKSPACE, GF_ERR_MODE = 0, -1, -2, -3, -4, -5, -6
GF_ERR_CUDA = -7

# Fake, 256-byte aligned, far-apart "device addresses" (never dereferenced:
# every call below fails validation first).
BASE = 0x7f0000000000
P = [BASE + i * (1 << 36) for i in range(16)]


def test_exports_every_header_symbol(L):
    names = binding.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
        assert n in binding._SIGS, f"binding lacks a signature for {n}"
    assert L.gf_abi_version() == 2


def test_status_strings(L):
    for code in range(-9, 1):
        s = L.gf_status_string(code)
        assert s and len(s) > 1
    assert L.gf_status_string(12345) == b"unknown status"


def _lgn(L, x=P[0], W=P[1], bl=P[2], bias=P[3], g=P[4], b=P[5], out=P[6], M=256, K=1024, N=4096, groups=64,
         eps=1e-5, mode=0, ws=P[7], wsb=None):
    if wsb is None:
        wsb = L.gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, groups, mode)
    return L.gf_linear_swish_bias_groupnorm(x, W, bl, bias, g, b, out, M, K, N, groups, eps, mode, ws, wsb, None)


def test_linear_gn_validation(L):
    assert _lgn(L, x=None) == GF_ERR_NULL
    assert _lgn(L, out=None) == GF_ERR_NULL
    assert _lgn(L, mode=3) == GF_ERR_MODE
    assert _lgn(L, mode=-1) == GF_ERR_MODE
    assert _lgn(L, mode=0x100) == GF_ERR_MODE     # the GELU flag belongs to the Conv1d chain
    assert _lgn(L, groups=3) == GF_ERR_SHAPE       # groups must divide N
    assert _lgn(L, groups=8192) == GF_ERR_SHAPE
    assert _lgn(L, groups=0) == GF_ERR_SHAPE
    assert _lgn(L, K=0) == GF_ERR_SHAPE
    assert _lgn(L, M=-1) == GF_ERR_SHAPE
    assert _lgn(L, eps=float("nan")) == GF_ERR_SHAPE
    assert _lgn(L, eps=-1.0) == GF_ERR_SHAPE
    assert _lgn(L, x=P[0] + 4) == GF_ERR_ALIGN
    assert _lgn(L, out=P[6] + 8) == GF_ERR_ALIGN
    assert _lgn(L, wsb=100) == GF_ERR_WORKSPACE
    assert _lgn(L, ws=None) == GF_ERR_NULL
    assert _lgn(L, out=P[0]) == GF_ERR_ALIAS        # out == x
    assert _lgn(L, out=P[7] + 1024) == GF_ERR_ALIAS  # out inside the workspace
    assert _lgn(L, out=P[1] - 256) == GF_ERR_ALIAS  # out runs into W


def test_workspace_sizes(L):
    M, K, N = 32768, 1024, 4096
    ws = L.gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, 64, 0)
    assert ws == 4 * (M * K + N * K)                # fp32 lo planes (the raw operands serve as hi)
    assert L.gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, 64, 1) == 2 * (M * K + N * K)  # bf16 hi
    assert L.gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, 64, 2) == 4 * (M * K + N * K)  # bf16 hi+lo
    assert L.gf_linear_swish_bias_groupnorm_workspace_size(M, K, N, 64, 3) == 0
    assert L.gf_linear_workspace_size(M, K, N, 0) == ws
    M, K, N = 1024, 8192, 8192
    # one (max, sum) float2 per row and column half of each n-block, sized
    # for the narrowest (160-column) tile width
    assert L.gf_linear_lse_act_workspace_size(M, K, N, 0) == 4 * (M * K + N * K) + M * (-(-N // 160) * 2) * 8
    # the default keeps the activations' raw fp32 plane (4 B per activation
    # in the 3xTF32 mode: the GEMM computes the lo plane itself) and the
    # weight planes; GF_FLAG_FUSED_PRODUCER (3xTF32, taps within 92
    # positions) only the LayerNorm partials, statistics and weight planes
    FUSED = 0x200
    planes = L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 4, 0)
    assert 4 * 32 * 256 * 4096 < planes < 4 * 32 * 256 * 4096 + (4 << 20)
    fused = L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 4, FUSED)
    assert 2 * 4 * 256 * 256 * 3 <= fused < 4 << 20
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 46, FUSED) == fused
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 47, FUSED) == 0  # taps span 94 > 92
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 4, FUSED | 1) == 0  # 3xTF32 only
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 4, 2) > 2 * 2 * 32 * 256 * 4096
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 0, 0) == 0  # dilation >= 1
    GELU_TANH = 0x100
    for mode in (0, 1, 2):  # the GELU flag changes no buffer
        for dil in (4, 64):
            assert (L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, dil, mode | GELU_TANH) ==
                    L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, dil, mode))
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 4, 0x400) == 0
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 4, 0x800) == 0
    assert L.gf_linear_workspace_size(M, K, N, GELU_TANH) == 0  # other calls take no flag
    assert L.gf_convt3d_swish_gn_hswish_workspace_size(128, 3, 16, 16, 32, 32, 3, 2, 1, 4) > 0
    # other strides, kernel sizes, channel counts and groups take the general
    # kernels: per (sample, channel, block) fp64 sums and per-channel
    # coefficients
    ws = L.gf_convt3d_swish_gn_hswish_workspace_size(128, 3, 16, 16, 32, 32, 3, 1, 1, 4)
    assert ws >= 128 * 16 * 2 * 8 + 128 * 16 * 8
    assert L.gf_convt3d_swish_gn_hswish_workspace_size(2, 12, 32, 4, 5, 6, 4, 3, 2, 8) > 0
    assert L.gf_convt3d_swish_gn_hswish_workspace_size(2, 3, 16, 1, 1, 1, 1, 1, 1, 4) == 0  # empty output


def test_lse_validation(L):
    def call(**kw):
        a = dict(x=P[0], W=P[1], b=P[2], out=P[3], M=1024, K=8192, N=8192, slope=0.01, mode=0, ws=P[4], wsb=None)
        a.update(kw)
        if a["wsb"] is None:
            a["wsb"] = L.gf_linear_lse_act_workspace_size(a["M"], a["K"], a["N"], a["mode"])
        return L.gf_linear_lse_act(a["x"], a["W"], a["b"], a["out"], a["M"], a["K"], a["N"], a["slope"], a["mode"],
                                   a["ws"], a["wsb"], None)
    assert call(W=None) == GF_ERR_NULL
    assert call(K=0) == GF_ERR_SHAPE
    assert call(N=0) == GF_ERR_SHAPE
    assert call(slope=float("inf")) == GF_ERR_SHAPE
    assert call(b=P[2] + 4) == GF_ERR_ALIGN
    assert call(wsb=1) == GF_ERR_WORKSPACE
    assert call(out=P[2] + 16) == GF_ERR_ALIAS


def test_dconv1d_validation(L):
    def call(**kw):
        a = dict(x=P[0], g=P[1], b=P[2], w=P[3], cb=P[4], out=P[5], B=32, C=256, L=4096, k=3, d=4, p=4, eps=1e-5,
                 mode=0, ws=P[6], wsb=None)
        a.update(kw)
        if a["wsb"] is None:
            a["wsb"] = L.gf_ln_gelu_dconv1d_res_workspace_size(a["B"], a["C"], a["L"], a["k"], max(a["d"], 1),
                                                               a["mode"])
        return L.gf_ln_gelu_dconv1d_res(a["x"], a["g"], a["b"], a["w"], a["cb"], a["out"], a["B"], a["C"], a["L"],
                                        a["k"], a["d"], a["p"], a["eps"], a["mode"], a["ws"], a["wsb"], None)
    assert call(g=None) == GF_ERR_NULL
    assert call(p=3) == GF_ERR_SHAPE               # not length-preserving
    assert call(C=0) == GF_ERR_SHAPE
    assert call(C=1056) == GF_ERR_SHAPE            # at most 1024 channels
    assert call(L=0) == GF_ERR_SHAPE
    assert call(mode=5) == GF_ERR_MODE
    assert call(mode=0x400) == GF_ERR_MODE         # unknown flag bit
    assert call(mode=0x201) == GF_ERR_MODE         # the fused producer is 3xTF32 only
    assert call(mode=0x200, d=47, p=47) == GF_ERR_SHAPE  # taps span 94 > 92
    assert call(mode=0x103) == GF_ERR_MODE         # tanh flag on an unknown precision mode
    assert call(mode=0x100, L=0) == GF_ERR_SHAPE   # the flag passes; the shape does not
    assert call(w=P[3] + 4) == GF_ERR_ALIGN
    assert call(wsb=5) == GF_ERR_WORKSPACE
    assert call(out=P[0]) == GF_ERR_ALIAS          # in-place residual is rejected


def test_convt3d_validation(L):
    def call(**kw):
        a = dict(x=P[0], w=P[1], b=P[2], g=P[3], be=P[4], out=P[5], N=128, Cin=3, Cout=16, D=16, H=32, W=32, k=3, s=2,
                 p=1, G=4, eps=1e-5, ws=P[6], wsb=None)
        a.update(kw)
        if a["wsb"] is None:
            a["wsb"] = L.gf_convt3d_swish_gn_hswish_workspace_size(a["N"], a["Cin"], a["Cout"], a["D"], a["H"], a["W"],
                                                                   a["k"], a["s"], a["p"], a["G"])
        return L.gf_convt3d_swish_gn_hswish(a["x"], a["w"], a["b"], a["g"], a["be"], a["out"], a["N"], a["Cin"],
                                            a["Cout"], a["D"], a["H"], a["W"], a["k"], a["s"], a["p"], a["G"], a["eps"],
                                            a["ws"], a["wsb"], None)
    assert call(x=None) == GF_ERR_NULL
    assert call(G=3) == GF_ERR_SHAPE               # 16 channels in 3 groups
    assert call(G=0) == GF_ERR_SHAPE
    assert call(Cin=2000) == GF_ERR_SHAPE
    assert call(k=9) == GF_ERR_SHAPE               # kernel sizes 1..8
    assert call(s=0) == GF_ERR_SHAPE
    assert call(p=-1) == GF_ERR_SHAPE
    assert call(D=1, k=1, s=1, p=1) == GF_ERR_SHAPE  # output extent (1-1)*1 - 2 + 1 < 1
    assert call(N=70000, k=4) == GF_ERR_SHAPE       # general kernels: N <= 65535
    assert call(k=4, wsb=8) == GF_ERR_WORKSPACE     # general kernels: the same checks
    assert call(k=4, out=P[6]) == GF_ERR_ALIAS
    assert call(k=4, w=P[1] + 8) == GF_ERR_ALIGN
    assert call(be=None) == GF_ERR_NULL
    assert call(g=P[3] + 4) == GF_ERR_ALIGN
    assert call(wsb=8) == GF_ERR_WORKSPACE
    assert call(out=P[6]) == GF_ERR_ALIAS


def test_device_status_signature(L):
    # the argument is optional; the call itself needs a device, so only the
    # ctypes signature is checked here
    assert L.gf_device_status.argtypes == [ctypes.POINTER(ctypes.c_int32)]


def _header_text():
    import re
    return re.sub(r"/\*.*?\*/", "", open(binding.HEADER_PATH).read(), flags=re.S)


def test_binding_constants_match_the_header():
    import re
    defs = {m.group(1): int(m.group(2), 0) for m in
            re.finditer(r"#define\s+(GF_[A-Z0-9_]+)\s+(-?(?:0x[0-9a-fA-F]+|\d+))\b", _header_text())}
    for name in ("GF_MODE_FP32_3XTF32", "GF_MODE_BF16", "GF_MODE_FP32_3XBF16", "GF_FLAG_GELU_TANH",
                 "GF_FLAG_FUSED_PRODUCER", "GF_CHAIN_GROUPNORM", "GF_CHAIN_LSE", "GF_CHAIN_LINEAR"):
        assert getattr(binding, name) == defs[name], name
    for name, v in (("GF_OK", GF_OK), ("GF_ERR_NULL", GF_ERR_NULL), ("GF_ERR_SHAPE", GF_ERR_SHAPE),
                    ("GF_ERR_ALIGN", GF_ERR_ALIGN), ("GF_ERR_ALIAS", GF_ERR_ALIAS),
                    ("GF_ERR_WORKSPACE", GF_ERR_WORKSPACE), ("GF_ERR_MODE", GF_ERR_MODE)):
        assert defs[name] == v, name


def test_binding_signatures_match_the_header_prototypes():
    """Each ctypes signature has the prototype's parameter count, and each
    parameter the ctypes type of its C type (pointers as pointers, int64_t,
    int32_t/gf_status, float, size_t), as has the return type."""
    import re
    protos = {}
    for m in re.finditer(r"([A-Za-z_][\w \*]*?)\b(gf_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", _header_text()):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        ps = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        protos[name] = (ret, ps)
    assert set(protos) == set(binding.header_functions())

    def kind(c):
        c = " ".join(c.split())
        if "*" in c:
            return "ptr"
        base = c.replace("const ", "").split()[0]
        return {"int64_t": "i64", "int32_t": "i32", "gf_status": "i32", "float": "f32", "size_t": "size"}[base]

    def ckind(t):
        if t in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
            return "ptr"
        return {ctypes.c_int64: "i64", ctypes.c_int32: "i32", ctypes.c_float: "f32", ctypes.c_size_t: "size"}[t]

    for name, (ret, ps) in protos.items():
        res, args = binding._SIGS[name]
        assert len(args) == len(ps), (name, len(args), len(ps))
        for i, (p, a) in enumerate(zip(ps, args)):
            assert kind(p) == ckind(a), (name, i, p, a)
        assert kind(ret) == ckind(res), (name, ret, res)


# ------------------------------------------------------------ empty batches
def test_empty_batches_launch_nothing(L):
    # M / B / N = 0 is an empty batch: GF_OK before any device call (so it
    # passes here, without a GPU), NULL x and out allowed, workspace query 0;
    # the other arguments are still checked
    assert L.gf_linear_swish_bias_groupnorm_workspace_size(0, 1024, 4096, 64, 0) == 0
    assert _lgn(L, M=0, x=None, out=None, ws=None, wsb=0) == GF_OK
    assert _lgn(L, M=0, groups=3, ws=None, wsb=0) == GF_ERR_SHAPE
    assert _lgn(L, M=0, W=None, ws=None, wsb=0) == GF_ERR_NULL
    assert _lgn(L, M=0, mode=7, ws=None, wsb=0) == GF_ERR_MODE
    assert L.gf_linear(None, P[1], None, None, 0, 64, 128, 0, None, 0, None) == GF_OK
    assert L.gf_linear_workspace_size(0, 64, 128, 0) == 0
    assert L.gf_linear_lse_act(None, P[1], P[2], None, 0, 64, 128, 0.01, 0, None, 0, None) == GF_OK
    assert L.gf_linear_lse_act(None, P[1], P[2], None, 0, 64, 0, 0.01, 0, None, 0, None) == GF_ERR_SHAPE
    assert L.gf_linear_lse_act_workspace_size(0, 64, 128, 0) == 0
    assert L.gf_linear_swish_bias_groupnorm_planes(None, P[1], P[2], P[3], P[4], P[5], None, 0, 64, 256, 4, 1e-5,
                                                   None) == GF_OK
    assert L.gf_linear_swish_bias_groupnorm_host(None, P[1], P[2], P[3], P[4], P[5], None, 0, 64, 256, 4, 1e-5, 0, 0,
                                                 None, 0, None) == GF_OK
    assert L.gf_linear_swish_bias_groupnorm_host_workspace_size(0, 64, 256, 4, 0, 0) == 0
    assert L.gf_ln_gelu_dconv1d_res_workspace_size(0, 256, 4096, 3, 4, 0) == 0
    assert L.gf_ln_gelu_dconv1d_res(None, P[1], P[2], P[3], P[4], None, 0, 256, 4096, 3, 4, 4, 1e-5, 0, None, 0,
                                    None) == GF_OK
    assert L.gf_ln_gelu_dconv1d_res(None, P[1], P[2], P[3], P[4], None, 0, 256, 4096, 3, 4, 3, 1e-5, 0, None, 0,
                                    None) == GF_ERR_SHAPE
    for k, s, p, G in ((3, 2, 1, 4), (4, 3, 2, 8)):
        assert L.gf_convt3d_swish_gn_hswish_workspace_size(0, 3, 16, 16, 32, 32, k, s, p, G) == 0
        assert L.gf_convt3d_swish_gn_hswish(None, P[1], P[2], P[3], P[4], None, 0, 3, 16, 16, 32, 32, k, s, p, G,
                                            1e-5, None, 0, None) == GF_OK
        assert L.gf_convt3d_swish_gn_hswish_noalloc(None, P[1], P[2], P[3], P[4], None, 0, 3, 16, 16, 32, 32, k, s,
                                                    p, G, 1e-5, None) == GF_OK
    assert L.gf_convt3d_swish_gn_hswish(None, P[1], P[2], P[3], P[4], None, 0, 3, 16, 16, 32, 32, 3, 2, 1, 3,
                                        1e-5, None, 0, None) == GF_ERR_SHAPE  # 16 channels in 3 groups
    assert L.gf_convt3d_swish_gn_hswish(None, P[1], P[2], P[3], P[4], None, -1, 3, 16, 16, 32, 32, 3, 2, 1, 4,
                                        1e-5, None, 0, None) != GF_OK


# ------------------------------------------------- dispatch tile widths
def test_tile_width_rule(L):
    GN, LSE, LIN = binding.GF_CHAIN_GROUPNORM, binding.GF_CHAIN_LSE, binding.GF_CHAIN_LINEAR
    tw = L.gf_linear_tile_width
    # 256 columns once every SM gets a tile; else 128; else 64 (152 SMs)
    assert tw(GN, 32768, 4096, 64, 0, 152) == 256
    assert tw(GN, 2432, 2048, 32, 0, 152) == 256       # 19 m-blocks x 8 = 152 tiles
    assert tw(GN, 2304, 2048, 32, 0, 152) == 128       # 18 x 8 = 144 < 152
    assert tw(GN, 1024, 4096, 64, 1, 152) == 128
    assert tw(GN, 256, 4096, 64, 0, 152) == 64
    assert tw(GN, 256, 4096, 32, 2, 152) == 256        # groups of 128: always 256-column tiles
    assert tw(GN, 256, 4096, 2, 0, 152) == 64          # groups of 2048: the row kernel's width rule
    assert tw(GN, 256, 4096, 3, 0, 152) == 0           # 3 does not divide 4096
    assert tw(LIN, 256, 4096, 0, 0, 152) == 64
    # logsumexp: 160 columns in the three-product modes (three smem stages,
    # room in TMEM for the chunked accumulation's totals); the BF16 mode 224
    # or 256, whichever needs fewer waves
    assert tw(LSE, 1024, 8192, 0, 0, 152) == 160
    assert tw(LSE, 1024, 8192, 0, 2, 152) == 160
    assert tw(LSE, 128, 30000, 0, 0, 152) == 160
    assert tw(LSE, 1024, 8192, 0, 1, 152) == 224
    assert tw(LSE, 512, 8960, 0, 1, 152) == 256
    assert tw(GN, 256, 4096, 64, 9, 152) == 0          # unknown mode
    assert tw(7, 256, 4096, 64, 0, 152) == 0           # unknown chain
    assert tw(GN, 256, 4096, 64, 0, 0) == 0


# -------------------------------------- host pipeline schedule and errors
def test_host_pipeline_schedule(L):
    st, tr = binding.host_pipeline_trace(3)
    assert st == GF_OK
    assert tr == "setup in0 compute0 out0 in1 compute1 out1 in2 compute2 out2 join"
    st, tr = binding.host_pipeline_trace(0)
    assert st == GF_OK and tr == "setup join"


@pytest.mark.parametrize("fail_at", range(0, 11))
def test_host_pipeline_error_path_drains(L, fail_at):
    # a failing step stops the schedule at once and the call waits for the
    # copies already queued (drain) before it returns GF_ERR_CUDA, so none of
    # them can touch the caller's host buffers after the return
    st, tr = binding.host_pipeline_trace(3, fail_at)
    steps = tr.split()
    assert st == GF_ERR_CUDA
    assert steps[-1] == "drain"
    assert len(steps) == fail_at + 2          # the steps up to the failing one, then drain
    assert "join" not in steps[:-1] or fail_at == 10


# ------------------------------------------------ no-workspace scratch
def test_noalloc_scratch_query_agrees_with_accept_reject(L):
    """The no-workspace call accepts a shape exactly when
    gf_convt3d_swish_gn_hswish_noalloc_scratch_size() is within the limit
    (accepted calls get past validation and then fail here only for want of
    a device)."""
    limit = L.gf_convt3d_noalloc_scratch_limit()
    shapes = [(128, 3, 16, 16, 32, 32, 3, 2, 1, 4),    # the pages' workload: its own kernels' scratch is small
              (1, 3, 16, 4, 5, 6, 3, 2, 1, 4), (4000, 3, 16, 16, 32, 32, 3, 2, 1, 4), (2000, 3, 16, 16, 32, 32, 3, 2, 1, 4),
              (3, 6, 16, 16, 32, 32, 3, 2, 1, 4), (2, 3, 8, 4, 5, 6, 4, 2, 1, 2), (3000, 3, 8, 4, 5, 6, 4, 2, 1, 2),
              (64, 2, 32, 30, 30, 30, 3, 1, 1, 8)]
    seen = set()
    for sh in shapes:
        need = L.gf_convt3d_swish_gn_hswish_noalloc_scratch_size(*sh)
        assert need > 0, sh
        st = L.gf_convt3d_swish_gn_hswish_noalloc(P[0], P[1], P[2], P[3], P[4], P[5], *sh, 1e-5, None)
        assert (st == GF_ERR_WORKSPACE) == (need > limit), (sh, need, st)
        seen.add(need > limit)
    assert seen == {True, False}
    # the headline workload needs far less than the workspace entry point's
    # query reports (that one sizes the tensor-core kernels)
    need = L.gf_convt3d_swish_gn_hswish_noalloc_scratch_size(*shapes[0])
    assert need <= limit < L.gf_convt3d_swish_gn_hswish_workspace_size(*shapes[0])
    assert L.gf_convt3d_swish_gn_hswish_noalloc_scratch_size(0, 3, 16, 16, 32, 32, 3, 2, 1, 4) == 0
    assert L.gf_convt3d_swish_gn_hswish_noalloc_scratch_size(1, 3, 16, 16, 32, 32, 3, 2, 1, 3) == 0


# ------------------------------------------- per-sample host-buffer calls
def _sample_ws(chunk, in_item, out_item, inner):
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    return 2 * up(chunk * in_item) + 2 * up(chunk * out_item) + up(inner)


def test_sample_host_workspace_sizes(L):
    # two input and two output staging buffers of a chunk, then the device
    # call's workspace for a chunk; chunk 0 = B/8 rounded up
    B, C, Lq, k, dil = 32, 256, 4096, 3, 4
    for chunk, eff in ((0, 4), (5, 5), (100, 32)):
        inner = L.gf_ln_gelu_dconv1d_res_workspace_size(eff, C, Lq, k, dil, 0)
        assert inner > 0
        assert L.gf_ln_gelu_dconv1d_res_host_workspace_size(B, C, Lq, k, dil, 0, chunk) == \
            _sample_ws(eff, C * Lq * 4, C * Lq * 4, inner)
    assert L.gf_ln_gelu_dconv1d_res_host_workspace_size(3, 64, 100, 3, 4, 0, 0) == \
        _sample_ws(1, 64 * 100 * 4, 64 * 100 * 4, L.gf_ln_gelu_dconv1d_res_workspace_size(1, 64, 100, 3, 4, 0))
    assert L.gf_ln_gelu_dconv1d_res_host_workspace_size(0, C, Lq, k, dil, 0, 0) == 0
    assert L.gf_ln_gelu_dconv1d_res_host_workspace_size(B, 0, Lq, k, dil, 0, 0) == 0
    assert L.gf_ln_gelu_dconv1d_res_host_workspace_size(B, C, Lq, k, dil, 0, -1) == 0
    N, Cin, Cout, D, H, W = 128, 3, 16, 16, 32, 32
    inner = L.gf_convt3d_swish_gn_hswish_workspace_size(16, Cin, Cout, D, H, W, 3, 2, 1, 4)
    assert inner > 0
    assert L.gf_convt3d_swish_gn_hswish_host_workspace_size(N, Cin, Cout, D, H, W, 3, 2, 1, 4, 0) == \
        _sample_ws(16, Cin * D * H * W * 4, Cout * 31 * 63 * 63 * 4, inner)
    assert L.gf_convt3d_swish_gn_hswish_host_workspace_size(N, Cin, Cout, D, H, W, 3, 2, 1, 5, 0) == 0  # 16 % 5
    assert L.gf_convt3d_swish_gn_hswish_host_workspace_size(0, Cin, Cout, D, H, W, 3, 2, 1, 4, 0) == 0


def test_sample_host_calls_check_arguments_first(L):
    # every case returns before any CUDA call (nothing is dereferenced)
    import ctypes
    host = (ctypes.c_float * 16)()
    h = ctypes.addressof(host)
    dc = lambda x, o, B, C, chunk, ws, nb: L.gf_ln_gelu_dconv1d_res_host(  # noqa: E731
        x, P[1], P[2], P[3], P[4], o, B, C, 256, 3, 4, 4, 1e-5, 0, chunk, ws, nb, None)
    need = L.gf_ln_gelu_dconv1d_res_host_workspace_size(4, 64, 256, 3, 4, 0, 2)
    assert dc(None, None, 0, 64, 0, None, 0) == GF_OK  # empty batch
    assert dc(None, h, 4, 64, 2, P[5], need) == GF_ERR_NULL
    assert dc(h, None, 4, 64, 2, P[5], need) == GF_ERR_NULL
    assert dc(h, h, 4, 64, 2, None, need) == GF_ERR_NULL
    assert dc(h, h, 4, 64, -1, P[5], need) == GF_ERR_SHAPE
    assert dc(h, h, 4, 0, 2, P[5], need) == GF_ERR_SHAPE
    assert dc(h, h, 4, 64, 2, P[5] + 4, need) == GF_ERR_ALIGN
    assert dc(h, h, 4, 64, 2, P[5], need - 1) == GF_ERR_WORKSPACE
    ct = lambda x, o, N, groups, ws, nb: L.gf_convt3d_swish_gn_hswish_host(  # noqa: E731
        x, P[1], P[2], P[3], P[4], o, N, 3, 16, 4, 8, 8, 3, 2, 1, groups, 1e-5, 0, ws, nb, None)
    need = L.gf_convt3d_swish_gn_hswish_host_workspace_size(4, 3, 16, 4, 8, 8, 3, 2, 1, 4, 0)
    assert ct(None, None, 0, 4, None, 0) == GF_OK
    assert ct(None, h, 4, 4, P[5], need) == GF_ERR_NULL
    assert ct(h, h, 4, 5, P[5], need) == GF_ERR_SHAPE
    assert ct(h, h, 4, 4, P[5] + 8, need) == GF_ERR_ALIGN
    assert ct(h, h, 4, 4, P[5], need - 1) == GF_ERR_WORKSPACE
