"""fp64 CPU oracle for the fused contraction + activation/normalisation path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
package; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import or run it.  It shares no code with the CUDA path.

Every function takes float arrays (any float dtype), upcasts them to float64
and computes the plain definition of the operator chain named on the source
pages (POPCORNBENCH level-2 transcripts, pages ``Kimi-K2.6__l2_p37``,
``Kimi-K2.6__l2_p64``, ``Kimi-K2.6__l2_p5`` and ``Kimi-K2.6__l2_p60``).
A library matmul (numpy) and ``scipy.special.erf`` serve as steps; there is
no blocking, fusion or reordering beyond the definitions.

Parity status: every public function here is pinned by ``tests/test_oracle_*``
(brute force on tiny shapes, closed forms, invariants, the zero-insertion
equivalence and float64 torch library cross-checks).  No function is
"parity unpinned".
"""
from .ops import (  # noqa: F401
    silu,
    gelu_erf,
    gelu_tanh,
    hardswish,
    leaky_relu,
    group_norm_rows,
    linear,
    linear_swish_bias_groupnorm,
    logsumexp_rows,
    linear_lse_act,
    layer_norm_sample,
    dilated_conv1d,
    ln_gelu_dconv1d_res,
    convt3d_out_size,
    conv_transpose3d_scatter,
    conv_transpose3d_zero_insert,
    conv1d_out_len,
    group_norm_nc,
    convt3d_swish_gn_hswish,
)
