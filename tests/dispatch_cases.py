"""Named parity cases that together reach every GEMM kernel variant the
Linear chains' dispatch can launch: (chain, epilogue, tile width, mode).

The tile width comes from the library's own rule (gf_linear_tile_width, the
function the dispatch calls), for a GPU with SM_COUNT SMs.  The CPU test
test_dispatch_coverage_cpu.py checks that these cases cover every variant the
rule can produce; test_dispatch_parity_gpu.py runs each case through the C ABI
and compares it with the fp64 oracle.  K is kept small so that the oracle
finishes quickly; the tile width does not depend on K.
"""
from __future__ import annotations

import dataclasses

SM_COUNT = 152  # GB300

MODES = {0: "3xtf32", 1: "bf16", 2: "3xbf16"}
GN, LSE, LIN = 0, 1, 2  # the chains of gf_linear_tile_width

# shapes whose GroupNorm / Linear tile width is 256, 128 and 64 columns on
# 152 SMs: 19 m-blocks x 8 n-blocks of 256 = 152 tiles; 8 x 16 = 128 < 152
# but 8 x 32 n-blocks of 128 = 256 >= 152; 2 x 32 = 64 < 152.
GN_SHAPES = {256: (2432, 2048), 128: (1024, 4096), 64: (256, 4096)}
# GroupNorm group widths: 16, 32, 64 and 128 run in the GEMM epilogue, any
# other width (256 here) stores t for the row kernel
GN_WIDTHS = (16, 32, 64, 128, 256)
# logsumexp tile widths by (mode, width): (M, N).  The three-product modes
# always take 160 columns (chunked accumulation); the BF16 mode 224 or 256,
# whichever needs fewer waves (4 m-blocks x 40 n-blocks of 224 = 160 tiles,
# two waves; x 35 of 256 = 140, one wave).
LSE_SHAPES = {
    (0, 160): (1024, 8192), (2, 160): (1024, 8192),
    (1, 224): (1024, 8192), (1, 256): (512, 8960),
}


@dataclasses.dataclass(frozen=True)
class Case:
    name: str
    chain: int
    mode: int
    M: int
    K: int
    N: int
    groups: int   # GroupNorm groups (GN chain), else 0
    bn: int       # the tile width the dispatch picks for it (on SM_COUNT SMs)

    @property
    def epilogue(self):
        if self.chain == LSE:
            return "lse"
        if self.chain == LIN:
            return "store"
        gw = self.N // self.groups
        return f"gn{gw}" if gw in (16, 32, 64, 128) else "gn_rows"


def cases():
    out = []
    for mode in MODES:
        for gw in GN_WIDTHS:
            for bn, (M, N) in GN_SHAPES.items():
                if gw == 128 and bn != 256:
                    continue  # 128-column groups always take 256-column tiles
                out.append(Case(f"gn_{MODES[mode]}_gw{gw}_bn{bn}", GN, mode, M, 96, N, N // gw, bn))
        # a 128-column group on the shapes that would otherwise take 128/64
        out.append(Case(f"gn_{MODES[mode]}_gw128_m256", GN, mode, 256, 96, 4096, 32, 256))
        for bn, (M, N) in GN_SHAPES.items():
            out.append(Case(f"linear_{MODES[mode]}_bn{bn}", LIN, mode, M, 96, N, 0, bn))
    for (mode, bn), (M, N) in LSE_SHAPES.items():
        out.append(Case(f"lse_{MODES[mode]}_bn{bn}", LSE, mode, M, 64, N, 0, bn))
    return out
