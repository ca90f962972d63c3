// ConvTranspose3d -> Swish -> GroupNorm -> HardSwish for any kernel size,
// stride, padding, channel counts and groups (page Kimi-K2.6__l2_p60, turn 1:
// the module's constructor arguments), on the CUDA cores.  The tensor-core
// kernels cover the pages' configuration (k 3, stride 2, pad 1, 16 output
// channels in 4 groups); everything else the entry point sends here.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gf.h"

namespace gf {

struct CtGenShape {
  int64_t N, Cin, Cout, D, H, W;
  int K, S, Pd, G;         // kernel size, stride, padding, groups
  int64_t OD, OH, OW;      // (I - 1) S - 2 Pd + K per dimension
  int P;                   // blocks per sample
  size_t part, coef, total;  // workspace layout (bytes)
};

// GF_OK and the filled shape when the general kernels take these arguments:
// 1 <= k <= 8, 1 <= stride <= 8, 0 <= pad, every output extent >= 1,
// 1 <= Cin, Cout <= 1024, Cout % groups == 0, N <= 65535, fewer than 2^30
// output voxels and 2^31 input elements per sample.
gf_status ct_general_shape(int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H, int64_t W, int32_t k,
                           int32_t stride, int32_t pad, int32_t groups, CtGenShape* s);

// Two passes over the output (statistics, then output), a finalize kernel
// between them; `workspace` holds s.total bytes.
gf_status launch_ct_general(const CtGenShape& s, const float* x, const float* w, const float* b, const float* gamma,
                            const float* beta, float* out, float eps, void* workspace, cudaStream_t stream);

}  // namespace gf
