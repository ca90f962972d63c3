"""Every GEMM kernel variant the Linear chains' dispatch can launch has a
named parity case (tests/dispatch_cases.py), run against the oracle by
test_dispatch_parity_gpu.py.  Host arithmetic only: the library's tile-width
rule (gf_linear_tile_width) is swept over a grid of shapes to find the
reachable variants."""
import pytest

from conv_activation_normalization_gb300 import binding

from . import dispatch_cases as dc


@pytest.fixture(scope="module")
def L():
    from conv_activation_normalization_gb300 import build
    build.build()
    return binding.lib()


def _epilogue(chain, N, groups):
    return dc.Case("", chain, 0, 1, 1, N, groups, 0).epilogue


def test_cases_declare_the_width_the_dispatch_picks(L):
    for c in dc.cases():
        got = L.gf_linear_tile_width(c.chain, c.M, c.N, c.groups, c.mode, dc.SM_COUNT)
        assert got == c.bn, (c.name, got)


def test_every_reachable_variant_has_a_case(L):
    reachable = set()
    Ms = [1, 127, 128, 256, 300, 512, 1024, 2048, 2432, 4096, 8192, 32768, 100000]
    Ns = [16, 64, 96, 128, 256, 512, 1000, 2048, 4096, 8192, 8960, 16384, 30000, 36000, 50000, 100000]
    for mode in dc.MODES:
        for M in Ms:
            for N in Ns:
                for chain in (dc.GN, dc.LSE, dc.LIN):
                    group_opts = [0] if chain != dc.GN else [g for g in (1, 2, 3, 4, 8, 16, 32, 64, 128, 256, 512)
                                                            if N % g == 0]
                    for g in group_opts:
                        bn = L.gf_linear_tile_width(chain, M, N, g, mode, dc.SM_COUNT)
                        assert bn > 0, (chain, M, N, g, mode)
                        reachable.add((_epilogue(chain, N, g), bn, mode))
    covered = {(c.epilogue, c.bn, c.mode) for c in dc.cases()}
    missing = reachable - covered
    assert not missing, sorted(missing)
    # and the expected variant count: GroupNorm epilogues 16/32/64/row kernel
    # at 3 widths, 128-column groups at 256 only, plain Linear at 3 widths, in
    # 3 modes; logsumexp at 160 (three-product modes) and 224/256 (BF16)
    assert len(reachable) == 3 * (4 * 3 + 1 + 3) + 2 + 2
