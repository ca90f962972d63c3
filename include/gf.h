/*
 * gf.h -- C ABI of libgf: a dense contraction (Linear GEMM, or a convolution
 * lowered to implicit GEMM) fused with its elementwise and normalisation
 * epilogue, for one GB300 (sm_103a).
 *
 * The operator chains are the four problems of the POPCORNBENCH level-2
 * transcripts this library follows:
 *   gf_linear_swish_bias_groupnorm  page "Kimi-K2.6__l2_p37", turn 1
 *   gf_linear_lse_act               page "Kimi-K2.6__l2_p64", turns 1-2
 *   gf_ln_gelu_dconv1d_res          page "Kimi-K2.6__l2_p5",  turns 1-2
 *   gf_convt3d_swish_gn_hswish      page "Kimi-K2.6__l2_p60", turn 1
 *
 * Conventions shared by every compute entry point:
 *   - Every tensor pointer is a DEVICE pointer to fp32, contiguous and
 *     row-major in PyTorch's layout, 16-byte aligned.  The caller owns every
 *     buffer; the library never allocates device memory and keeps no pointer
 *     after the call returns.
 *   - `workspace` is caller-owned device scratch of at least the size the
 *     matching *_workspace_size() query returns (256-byte aligned).  It may be
 *     NULL only when that size is 0.  Its contents on entry do not matter.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued on it and the call returns without synchronising.  The device
 *     entry points make only stream-ordered CUDA calls (kernel launches,
 *     including cooperative ones, and async memsets), so a call can be
 *     captured into a CUDA graph and replayed with the same arguments
 *     (the host-buffer entry point, which waits on copies, cannot).
 *   - Arguments are validated before anything is launched; a rejected call
 *     launches nothing and returns a negative gf_status.  No C++ exception
 *     crosses this boundary.
 *   - An empty batch (M = 0 for the Linear chains, B = 0 for the Conv1d
 *     chain, N = 0 for the ConvTranspose3d chain) is valid: the other sizes
 *     are still checked, the batch-sized pointers (x and out) may then be
 *     NULL, the workspace queries return 0, and the call launches nothing
 *     and returns GF_OK, as the pages' PyTorch modules return an empty
 *     output for an empty batch.
 *   - `out` must not overlap any input or the workspace (GF_ERR_ALIAS).
 *   - Device-side errors (a bounded wait inside a kernel that ran out) are
 *     recorded in a device status word; gf_device_status() reads it.
 *   - mode selects how the contraction runs on the tensor cores; every mode
 *     accumulates in fp32 and runs the epilogue in fp32:
 *       GF_MODE_FP32_3XTF32  three TF32 products (hi*hi + hi*lo + lo*hi of a
 *                            hi/lo split of both operands); matches an fp64
 *                            evaluation within 1e-4 abs + 1e-4 rel on the
 *                            pages' workloads.  The default.
 *       GF_MODE_BF16         one BF16 product (operands rounded to bf16);
 *                            within 3e-2 abs + 3e-2 rel.
 *       GF_MODE_FP32_3XBF16  three BF16 products of a bf16 hi/lo split, at
 *                            twice the TF32 tensor rate; within 1e-4 abs +
 *                            1e-4 rel on the pages' workloads.
 *     K must be a multiple of 8 (C a multiple of 64) in the BF16 modes.
 */
#ifndef GF_H_
#define GF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t gf_status;

#define GF_OK                    0
#define GF_ERR_NULL             -1  /* a required pointer is NULL              */
#define GF_ERR_SHAPE            -2  /* a size is out of range or unsupported   */
#define GF_ERR_ALIGN            -3  /* a pointer is not 16-byte aligned        */
#define GF_ERR_ALIAS            -4  /* out overlaps an input or the workspace  */
#define GF_ERR_WORKSPACE        -5  /* workspace smaller than the query says   */
#define GF_ERR_MODE             -6  /* unknown or unsupported mode             */
#define GF_ERR_CUDA             -7  /* a CUDA runtime/driver call failed       */
#define GF_ERR_DEVICE_CHECK     -8  /* a kernel recorded a device-side error   */
#define GF_ERR_UNSUPPORTED_ARCH -9  /* current device is not sm_103            */

#define GF_MODE_FP32_3XTF32 0
#define GF_MODE_BF16        1
#define GF_MODE_FP32_3XBF16 2

/* Flag OR'd into the mode of gf_ln_gelu_dconv1d_res (and its workspace
 * query): GELU in its tanh approximation,
 * 0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3))), the form page
 * Kimi-K2.6__l2_p5 turn 2 reads the module's GELU as, instead of the exact
 * erf form.  Other calls reject it (GF_ERR_MODE). */
#define GF_FLAG_GELU_TANH 0x100

/* Flag OR'd into the mode of gf_ln_gelu_dconv1d_res (and its workspace
 * query), 3xTF32 mode only: LayerNorm and GELU are applied inside the conv
 * GEMM while it builds its operand tiles (page Kimi-K2.6__l2_p5 turn 2 fuses
 * them into the loading step), so the workspace holds no activation planes:
 * about 2 MB instead of 8 B per activation (270 MB for x[32,256,4096]).  It is
 * slower than the default (about 0.46 against 0.32 ms per call on that
 * workload) and needs (ksize - 1) * dilation <= 92 (else GF_ERR_SHAPE; other
 * modes: GF_ERR_MODE).  Results equal the default path's up to rounding. */
#define GF_FLAG_FUSED_PRODUCER 0x200

/* Chains whose GEMM tile width gf_linear_tile_width reports. */
#define GF_CHAIN_GROUPNORM 0  /* gf_linear_swish_bias_groupnorm (and _planes, _host) */
#define GF_CHAIN_LSE       1  /* gf_linear_lse_act                                    */
#define GF_CHAIN_LINEAR    2  /* gf_linear                                            */

/* Version of this ABI (bumped on any signature change). */
int32_t gf_abi_version(void);

/* Static, NUL-terminated description of a status code.  Never NULL. */
const char* gf_status_string(gf_status status);

/* Synchronises the current device, then writes the device status word
 * accumulated by every kernel of this library since the last call into
 * *device_bits (0 = no device-side error) and clears it.  Returns GF_OK, or
 * GF_ERR_DEVICE_CHECK when the word was non-zero, or GF_ERR_CUDA.
 * device_bits may be NULL. */
gf_status gf_device_status(int32_t* device_bits);

/* Profiling.  Between gf_profile_begin(max_calls) and gf_profile_end(), each
 * compute entry point records a pair of CUDA events on its stream around its
 * dominant kernel (the fused GEMM; for the ConvTranspose3d chain, the pass that
 * writes the output), for up to max_calls calls.  gf_profile_end() waits for
 * the recorded events, returns the number of calls recorded and the sum of
 * their kernel times in milliseconds, and releases the events.  The recorder
 * is process-wide: profile one stream at a time.  Returns GF_ERR_SHAPE when
 * begin is called twice or end without begin. */
gf_status gf_profile_begin(int32_t max_calls);
gf_status gf_profile_end(int32_t* calls, float* total_ms);

/* Measures the tensor pipe's dense rate on this GPU: one CTA per SM issues
 * tcgen05.mma instructions back to back (128 x 256 fp32 accumulator in TMEM,
 * operands already in shared memory, nothing loaded or stored) for `iters`
 * rounds of four K-steps, kind 0 = kind::tf32, 1 = kind::f16 with BF16
 * operands.  Launches once to warm up, then `repeats` times on an internal
 * stream, waits for them, and writes the best rate in TFLOP/s (2 M N K per
 * instruction) into *tflops.  A measurement utility (it synchronises), not
 * part of any operator.  Supported: 1 <= iters <= 65536, 1 <= repeats <= 100. */
gf_status gf_measure_tensor_rate(int32_t kind, int32_t iters, int32_t repeats, double* tflops);

/* ------------------------------------------------------------------------
 * Linear alone: out[m,n] = sum_k x[m,k] * W[n,k] + b[n]
 *
 * The contraction step shared by the two Linear chains (nn.Linear / addmm,
 * page Kimi-K2.6__l2_p37 turn 1 and page Kimi-K2.6__l2_p64 turn 1), exposed
 * so that it can be checked on its own.  x [M,K], W [N,K], b [N] (may be
 * NULL), out [M,N].  Supported: M >= 0, K, N >= 1 (a K that is not a multiple of
 * 4 fp32 / 8 bf16 elements is zero-padded in the workspace's operand planes).
 * With integer-valued x and W (|v| <= 2^11) and |out| < 2^24 the result is
 * exact.
 * ---------------------------------------------------------------------- */
size_t gf_linear_workspace_size(int64_t M, int64_t K, int64_t N, int32_t mode);
gf_status gf_linear(const float* x, const float* W, const float* b, float* out, int64_t M, int64_t K,
                    int64_t N, int32_t mode, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Linear -> Swish -> +bias -> GroupNorm            (page Kimi-K2.6__l2_p37)
 *
 *   y[m,n]   = sum_k x[m,k] * W[n,k] + b_lin[n]
 *   t[m,n]   = y * sigmoid(y) + bias[n]
 *   out[m,n] = (t - mu[m,g]) / sqrt(var[m,g] + eps) * gamma[n] + beta[n]
 * with g = n / (N/groups), mu and var the mean and biased variance of t over
 * the N/groups contiguous channels of group g in row m.
 *
 *   x [M,K], W [N,K] (nn.Linear layout), b_lin/bias/gamma/beta [N], out [M,N].
 *   b_lin may be NULL (no linear bias).
 *   Supported: M >= 0, K >= 1 (K padded as for gf_linear),
 *   groups >= 1 with N % groups == 0.  Group widths N/groups of 16, 32, 64
 *   and 128 run inside the GEMM epilogue (groups of 128 on 256-column
 *   tiles); any other width stores t and normalises the rows in a second
 *   kernel (one more pass over out).
 * ---------------------------------------------------------------------- */
size_t gf_linear_swish_bias_groupnorm_workspace_size(int64_t M, int64_t K, int64_t N,
                                                     int32_t groups, int32_t mode);
gf_status gf_linear_swish_bias_groupnorm(const float* x, const float* W, const float* b_lin,
                                         const float* bias, const float* gamma, const float* beta,
                                         float* out, int64_t M, int64_t K, int64_t N,
                                         int32_t groups, float eps, int32_t mode,
                                         void* workspace, size_t workspace_bytes, void* stream);

/* The same operator on operands already split for the tensor cores (see
 * gf_tf32_split): x_planes [2][M][K], W_planes [2][N][K].  It launches the
 * fused GEMM kernel alone, so a caller can split a weight once and reuse it.
 * Same checks and result as gf_linear_swish_bias_groupnorm; K must be a
 * multiple of 4 (the planes' rows are read as they are). */
gf_status gf_linear_swish_bias_groupnorm_planes(const float* x_planes, const float* W_planes,
                                                const float* b_lin, const float* bias,
                                                const float* gamma, const float* beta, float* out,
                                                int64_t M, int64_t K, int64_t N, int32_t groups,
                                                float eps, void* stream);

/* The same operator on HOST buffers: x_host [M,K] in, out_host [M,N] out
 * (page-locked host memory lets the copies overlap the compute; pageable
 * memory works but serialises them).  W, b_lin, bias, gamma and beta are
 * device pointers as above.  Rows are processed in chunks of chunk_rows
 * (0 = a size that fills whole waves of tiles, at least 2048 rows): chunk i
 * is copied in on an internal stream while chunk i-1 is computed on `stream`
 * and chunk i-2 is copied out on a second internal stream, through two device
 * staging buffers in the workspace.  Returns once everything is enqueued;
 * out_host is complete when `stream` reaches that point (synchronise it
 * before reading).  Workspace: the matching *_host_workspace_size() query.
 * The internal streams and events are created and released by each call.
 * If a CUDA call fails after work was enqueued, the call stops enqueuing,
 * blocks until the copies already queued on its internal streams have
 * finished (and the computes they wait on), then returns GF_ERR_CUDA: no copy
 * of this call reads x_host or writes out_host after it returns, and rows
 * whose chunks were not reached are left as they were. */
size_t gf_linear_swish_bias_groupnorm_host_workspace_size(int64_t M, int64_t K, int64_t N,
                                                          int32_t groups, int32_t mode,
                                                          int64_t chunk_rows);
gf_status gf_linear_swish_bias_groupnorm_host(const float* x_host, const float* W, const float* b_lin,
                                              const float* bias, const float* gamma, const float* beta,
                                              float* out_host, int64_t M, int64_t K, int64_t N,
                                              int32_t groups, float eps, int32_t mode,
                                              int64_t chunk_rows, void* workspace,
                                              size_t workspace_bytes, void* stream);

/* The GEMM tile width (output columns per CTA tile: 64, 128 or 256, or
 * 160, 224 or 256 for GF_CHAIN_LSE) that the chain's dispatch picks for a
 * call of M rows and N output columns in `mode` (for GF_CHAIN_GROUPNORM with
 * `groups` groups; ignored otherwise) on a GPU with sm_count SMs.  Pure host
 * arithmetic (no device call), the same function the dispatch uses; 0 for
 * invalid arguments.  Lets tests check that every kernel variant the dispatch
 * can reach is exercised. */
int32_t gf_linear_tile_width(int32_t chain, int64_t M, int64_t N, int32_t groups, int32_t mode,
                             int32_t sm_count);

/* Testing hook of the host-buffer pipeline's schedule: runs the schedule of
 * gf_linear_swish_bias_groupnorm_host for nchunks chunks with the CUDA calls
 * replaced by a recorder, making step number fail_at (counted from 0; -1:
 * none) fail as a failed CUDA call would.  Writes the steps taken, separated
 * by spaces ("setup in0 compute0 out0 ... join", "drain" after a failure),
 * into trace (NUL-terminated, truncated to trace_bytes) and returns the
 * status the real call would return.  Touches no device. */
gf_status gf_testing_host_pipeline_trace(int64_t nchunks, int32_t fail_at, char* trace,
                                         size_t trace_bytes);

/* Splits n fp32 values (n % 4 == 0) into the two planes the 3xTF32
 * contraction reads: planes[0][i] = src[i] with its 13 low mantissa bits
 * cleared (a TF32 value) and planes[1][i] = src[i] - planes[0][i] (exact).
 * planes holds 2*n floats and must not overlap src. */
gf_status gf_tf32_split(const float* src, float* planes, int64_t n, void* stream);

/* ------------------------------------------------------------------------
 * Linear -> logsumexp(dim 1) -> LeakyReLU x2 -> GELU(erf) x2
 *                                                   (page Kimi-K2.6__l2_p64)
 *
 *   y[m,n]  = sum_k x[m,k] * W[n,k] + b[n]
 *   l[m]    = max_n y + ln sum_n exp(y - max_n y)
 *   a       = lrelu(lrelu(l)),  lrelu(v) = v > 0 ? v : negative_slope * v
 *   out[m]  = gelu(gelu(a)),    gelu(v) = v * Phi(v)   (exact, erf form)
 *
 *   x [M,K], W [N,K], b [N] (may be NULL), out [M,1].
 *   Supported: M >= 0, K, N >= 1 (K padded as for gf_linear).
 * ---------------------------------------------------------------------- */
size_t gf_linear_lse_act_workspace_size(int64_t M, int64_t K, int64_t N, int32_t mode);
gf_status gf_linear_lse_act(const float* x, const float* W, const float* b, float* out,
                            int64_t M, int64_t K, int64_t N, float negative_slope, int32_t mode,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * LayerNorm([C,L]) -> GELU(erf) -> dilated Conv1d -> +x
 *                                                    (page Kimi-K2.6__l2_p5)
 *
 *   h[b,c,l]   = (x - mu_b) / sqrt(var_b + eps) * ln_gamma[c,l] + ln_beta[c,l]
 *                (mu_b, var_b: mean and biased variance of x[b] over all C*L)
 *   a          = gelu(h), and a = 0 outside 0 <= l < L (the conv's padding);
 *                gelu is 0.5 h (1 + erf(h / sqrt 2)), or its tanh
 *                approximation when mode carries GF_FLAG_GELU_TANH
 *   out[b,o,j] = conv_b[o] + sum_{c,t} conv_w[o,c,t] * a[b,c, j - padding + t*dilation]
 *                + x[b,o,j]
 *
 *   x, out [B,C,L]; ln_gamma, ln_beta [C,L]; conv_w [C,C,ksize] (nn.Conv1d
 *   layout, cross-correlation); conv_b [C] (may be NULL).
 *   Supported: 1 <= C <= 1024 (input channels padded to whole k-blocks of
 *   32, or 64 in the BF16 modes, inside the workspace; output channels in
 *   tiles of 256),
 *   L >= 1, 1 <= ksize <= 16, dilation >= 1,
 *   2*padding == dilation*(ksize-1) (length-preserving, as the residual needs).
 *   The workspace query takes the dilation and the mode with its flags: the
 *   size depends on whether GF_FLAG_FUSED_PRODUCER is given.
 * ---------------------------------------------------------------------- */
size_t gf_ln_gelu_dconv1d_res_workspace_size(int64_t B, int64_t C, int64_t L, int32_t ksize,
                                             int32_t dilation, int32_t mode);
gf_status gf_ln_gelu_dconv1d_res(const float* x, const float* ln_gamma, const float* ln_beta,
                                 const float* conv_w, const float* conv_b, float* out,
                                 int64_t B, int64_t C, int64_t L, int32_t ksize, int32_t dilation,
                                 int32_t padding, float eps, int32_t mode,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* The same operator on HOST buffers: x_host [B,C,L] in, out_host [B,C,L] out
 * (page-locked host memory lets the copies overlap the compute; pageable
 * memory works but serialises them).  ln_gamma, ln_beta, conv_w and conv_b
 * are device pointers as above.  The batch is processed in chunks of
 * chunk_samples whole samples (0 = B/8 rounded up, so at most eight chunks):
 * chunk i is copied in on an internal stream while chunk i-1 is computed on
 * `stream` by gf_ln_gelu_dconv1d_res and chunk i-2 is copied out on a second
 * internal stream, through two device staging buffers each way in the
 * workspace.  Each sample is normalised on its own, so the result equals one
 * gf_ln_gelu_dconv1d_res call over the batch.  Returns once everything is
 * enqueued; out_host is complete when `stream` reaches that point.
 * Workspace: gf_ln_gelu_dconv1d_res_host_workspace_size() bytes with the
 * same chunk_samples (0 for an invalid shape or mode).  Errors: the device
 * call's own checks (shape, mode, alignment of the device pointers, which run
 * on the first chunk); GF_ERR_NULL for a NULL host buffer or workspace; on a
 * failed CUDA call after work was enqueued, the call stops enqueuing, blocks
 * until the copies already queued on its internal streams have finished,
 * then returns: no copy of this call touches x_host or out_host after it
 * returns, and samples whose chunks were not reached are left as they were.
 * B = 0 returns GF_OK. */
size_t gf_ln_gelu_dconv1d_res_host_workspace_size(int64_t B, int64_t C, int64_t L, int32_t ksize,
                                                  int32_t dilation, int32_t mode,
                                                  int64_t chunk_samples);
gf_status gf_ln_gelu_dconv1d_res_host(const float* x_host, const float* ln_gamma,
                                      const float* ln_beta, const float* conv_w,
                                      const float* conv_b, float* out_host, int64_t B, int64_t C,
                                      int64_t L, int32_t ksize, int32_t dilation, int32_t padding,
                                      float eps, int32_t mode, int64_t chunk_samples,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * ConvTranspose3d -> Swish -> GroupNorm -> HardSwish
 *                                                   (page Kimi-K2.6__l2_p60)
 *
 *   y[n,o,od,oh,ow] = b[o] + sum x[n,c,id,ih,iw] * w[c,o,kd,kh,kw]
 *                     over od = s*id - p + kd (and likewise for h, w)
 *   s_ = y * sigmoid(y)
 *   h  = GroupNorm(groups, eps, affine gamma/beta)(s_)   (per sample, per
 *        group of Cout/groups contiguous channels x all voxels, biased var)
 *   out = h * clamp(h + 3, 0, 6) / 6
 *
 *   x [N,Cin,D,H,W]; w [Cin,Cout,k,k,k] (nn.ConvTranspose3d layout);
 *   b [Cout] (may be NULL); gamma, beta [Cout];
 *   out [N,Cout,(D-1)s-2p+k, (H-1)s-2p+k, (W-1)s-2p+k].
 *   Supported: 1 <= k <= 8, 1 <= stride <= 8, 0 <= pad <= 64 with every
 *   output extent >= 1, 1 <= Cin, Cout <= 1024, Cout % groups == 0,
 *   N <= 65535, fewer than 2^30 output voxels per sample; output_padding
 *   is 0.
 *
 *   The pages' configuration (k == 3, stride == 2, pad == 1, Cout == 16,
 *   groups == 4) with Cin <= 8 runs on specialized kernels (the tensor
 *   cores for Cin <= 4, described next; the CUDA cores for 5..8); every
 *   other shape on general CUDA-core kernels (gather form of the transposed
 *   convolution, two passes, statistics in fp64).
 *
 *   With Cin <= 4 and at most (number of SMs + 1) tiles of 128 (h, w) cells
 *   per sample the call is one cooperative kernel (one CTA per SM, every CTA
 *   resident) that exchanges the GroupNorm statistics through the workspace;
 *   the workspace's counters are zeroed by a memset on `stream` first, so two
 *   calls that run at the same time must not share a workspace.  Otherwise
 *   the call runs two passes (statistics, then output).  Results are the same
 *   either way up to rounding.
 * ---------------------------------------------------------------------- */
size_t gf_convt3d_swish_gn_hswish_workspace_size(int64_t N, int64_t Cin, int64_t Cout,
                                                 int64_t D, int64_t H, int64_t W, int32_t k,
                                                 int32_t stride, int32_t pad, int32_t groups);
gf_status gf_convt3d_swish_gn_hswish(const float* x, const float* w, const float* b,
                                     const float* gamma, const float* beta, float* out,
                                     int64_t N, int64_t Cin, int64_t Cout, int64_t D, int64_t H,
                                     int64_t W, int32_t k, int32_t stride, int32_t pad,
                                     int32_t groups, float eps,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* The same operator on HOST buffers: x_host [N,Cin,D,H,W] in, out_host (the
 * output shape above) out, page-locked for overlapped copies; w, b, gamma
 * and beta are device pointers.  Chunks of chunk_samples whole samples (0 =
 * N/8 rounded up) are copied in, computed by gf_convt3d_swish_gn_hswish on
 * `stream` and copied out in the overlapped schedule of
 * gf_ln_gelu_dconv1d_res_host, with the same workspace query (with
 * chunk_samples), completion and error behaviour.  GroupNorm normalises
 * within a sample, so the result equals one gf_convt3d_swish_gn_hswish call
 * over the batch.  N = 0 returns GF_OK. */
size_t gf_convt3d_swish_gn_hswish_host_workspace_size(int64_t N, int64_t Cin, int64_t Cout,
                                                      int64_t D, int64_t H, int64_t W, int32_t k,
                                                      int32_t stride, int32_t pad, int32_t groups,
                                                      int64_t chunk_samples);
gf_status gf_convt3d_swish_gn_hswish_host(const float* x_host, const float* w, const float* b,
                                          const float* gamma, const float* beta, float* out_host,
                                          int64_t N, int64_t Cin, int64_t Cout, int64_t D,
                                          int64_t H, int64_t W, int32_t k, int32_t stride,
                                          int32_t pad, int32_t groups, float eps,
                                          int64_t chunk_samples, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * ConvTranspose3d -> Swish -> GroupNorm -> HardSwish without any workspace
 *
 * The source pages have no counterpart of this entry point; it exists for
 * callers that cannot hand the library device scratch memory.  Typical ones:
 * a host process that owns the whole device memory budget through its own
 * pool and forbids any further cudaMalloc once it has started, or a plugin
 * interface that passes a kernel only its input and output buffers.  Such a
 * caller cannot call gf_convt3d_swish_gn_hswish, whose statistics need a
 * workspace.
 *
 * Same operator, arguments (minus workspace), supported shapes and result as
 * gf_convt3d_swish_gn_hswish (up to rounding: the pages' configuration runs
 * on the CUDA-core two-pass kernels here, not on the tensor-core kernels the
 * workspace entry point uses for Cin <= 4).  The caller still owns and passes
 * x, w, b, gamma, beta and out.  The scratch (the per-block GroupNorm sums and
 * the per-channel affine coefficients) lives in a fixed array inside the
 * library, 4 MiB (gf_convt3d_noalloc_scratch_limit()) on every GPU that loads
 * the library, held until the process exits.  The bytes a shape needs are
 * what gf_convt3d_swish_gn_hswish_noalloc_scratch_size() returns (NOT the
 * workspace entry point's query, whose kernels differ); shapes that need more
 * than the limit return GF_ERR_WORKSPACE before anything is launched.  No call
 * allocates: the entry point calls no cudaMalloc, cudaFree or allocating
 * library routine.
 *
 * The first call on a device looks up the array's device address (once per
 * device and CUDA context, with that device current); make that first call
 * before any stream capture.  Every call on a device uses the same array and
 * leaves its contents behind; the kernels overwrite all of it that they read,
 * so nothing needs clearing between calls.  Two calls whose kernels overlap
 * on the GPU (different streams, no ordering between them) race on the
 * array: order them, e.g. by issuing them on one stream.
 * ---------------------------------------------------------------------- */
size_t gf_convt3d_noalloc_scratch_limit(void);
size_t gf_convt3d_swish_gn_hswish_noalloc_scratch_size(int64_t N, int64_t Cin, int64_t Cout,
                                                       int64_t D, int64_t H, int64_t W, int32_t k,
                                                       int32_t stride, int32_t pad, int32_t groups);
gf_status gf_convt3d_swish_gn_hswish_noalloc(const float* x, const float* w, const float* b,
                                             const float* gamma, const float* beta, float* out,
                                             int64_t N, int64_t Cin, int64_t Cout, int64_t D,
                                             int64_t H, int64_t W, int32_t k, int32_t stride,
                                             int32_t pad, int32_t groups, float eps, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GF_H_ */
