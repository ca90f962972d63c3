// Library-wide entry points (version, status strings, device status word) and
// the host helpers declared in host_common.h.
#include <cstring>
#include <mutex>
#include <new>

#include "host_common.h"

namespace gf {

// Bits recorded by kernels (see status.cuh).  One word per device.
__device__ uint32_t g_device_status = 0;

gf_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GF_OK : GF_ERR_CUDA; }

gf_status check_no_alias(Span out, const Span* ins, int n) {
  for (int i = 0; i < n; ++i)
    if (overlaps(out, ins[i])) return GF_ERR_ALIAS;
  return GF_OK;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_info_ok[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
uint32_t* g_status_ptr[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
unsigned long long g_status_ctx[kMaxDevices];

template <class F>
bool driver_entry(const char* name, F* fn) {
  if (*fn) return true;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p)
    return false;
  *fn = reinterpret_cast<F>(p);
  return true;
}
}  // namespace

gf_status current_context_id(unsigned long long* id) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!driver_entry("cuCtxGetCurrent", &g_ctx_current) || !driver_entry("cuCtxGetId", &g_ctx_id))
      return GF_ERR_CUDA;
  }
  // make the current device's primary context current on this thread (the
  // runtime creates contexts lazily; cudaSetDevice initialises it)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return GF_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return GF_ERR_CUDA;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS ? GF_OK : GF_ERR_CUDA;
}

gf_status current_device(DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GF_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GF_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_info_ok[dev]) {
    DeviceInfo d{};
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return GF_ERR_CUDA;
    g_info[dev] = d;
    g_info_ok[dev] = true;
  }
  *info = g_info[dev];
  if (info->cc_major != 10 || info->cc_minor != 3) return GF_ERR_UNSUPPORTED_ARCH;
  return GF_OK;
}

uint32_t* device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned long long ctx = 0;
  if (current_context_id(&ctx) != GF_OK) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev] || g_status_ctx[dev] != ctx) {  // looked up again in a new context
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
    g_status_ctx[dev] = ctx;
  }
  return g_status_ptr[dev];
}

gf_status make_tmap(CUtensorMap* map, const void* base, int elem_bytes, int rank, const uint64_t* dims,
                    const uint32_t* box, int swizzle_bytes) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return GF_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  if (rank < 1 || rank > 5 || (elem_bytes != 4 && elem_bytes != 2) || (swizzle_bytes != 128 && swizzle_bytes != 64) ||
      box[0] * uint32_t(elem_bytes) != uint32_t(swizzle_bytes))
    return GF_ERR_SHAPE;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t bdim[5], estride[5];
  uint64_t stride = uint64_t(elem_bytes);
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = g_encode(map, dt, cuuint32_t(rank), const_cast<void*>(base),
                              gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GF_OK : GF_ERR_CUDA;
}

namespace {
struct Profile {
  bool active = false;
  int capacity = 0, used = 0;
  bool open = false;
  cudaEvent_t* ev = nullptr;  // 2 * capacity
};
Profile g_prof;
std::mutex g_prof_mu;
}  // namespace

void profile_mark_begin(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof.active || g_prof.used >= g_prof.capacity) return;
  cudaEventRecord(g_prof.ev[2 * g_prof.used], s);
  g_prof.open = true;
}

void profile_mark_end(cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof.active || !g_prof.open) return;
  cudaEventRecord(g_prof.ev[2 * g_prof.used + 1], s);
  g_prof.open = false;
  ++g_prof.used;
}

}  // namespace gf

extern "C" {

gf_status gf_profile_begin(int32_t max_calls) {
  using namespace gf;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (g_prof.active || max_calls < 1 || max_calls > (1 << 20)) return GF_ERR_SHAPE;
  g_prof.ev = new (std::nothrow) cudaEvent_t[2 * size_t(max_calls)];
  if (!g_prof.ev) return GF_ERR_CUDA;
  for (int i = 0; i < 2 * max_calls; ++i) {
    if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
      delete[] g_prof.ev;
      g_prof.ev = nullptr;
      return GF_ERR_CUDA;
    }
  }
  g_prof.capacity = max_calls;
  g_prof.used = 0;
  g_prof.open = false;
  g_prof.active = true;
  return GF_OK;
}

gf_status gf_profile_end(int32_t* calls, float* total_ms) {
  using namespace gf;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof.active) return GF_ERR_SHAPE;
  gf_status st = GF_OK;
  float total = 0.f;
  for (int i = 0; i < g_prof.used; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) {
      st = GF_ERR_CUDA;
      break;
    }
    total += ms;
  }
  for (int i = 0; i < 2 * g_prof.capacity; ++i) cudaEventDestroy(g_prof.ev[i]);
  delete[] g_prof.ev;
  if (calls) *calls = g_prof.used;
  if (total_ms) *total_ms = total;
  g_prof = Profile{};
  return st;
}


int32_t gf_abi_version(void) { return 2; }

const char* gf_status_string(gf_status s) {
  switch (s) {
    case GF_OK: return "ok";
    case GF_ERR_NULL: return "a required pointer is NULL";
    case GF_ERR_SHAPE: return "unsupported or out-of-range size";
    case GF_ERR_ALIGN: return "pointer not 16-byte aligned";
    case GF_ERR_ALIAS: return "output overlaps an input or the workspace";
    case GF_ERR_WORKSPACE: return "workspace smaller than required";
    case GF_ERR_MODE: return "unknown or unsupported mode";
    case GF_ERR_CUDA: return "CUDA runtime or driver call failed";
    case GF_ERR_DEVICE_CHECK: return "a kernel recorded a device-side error";
    case GF_ERR_UNSUPPORTED_ARCH: return "current device is not sm_103 (GB300)";
    default: return "unknown status";
  }
}

gf_status gf_device_status(int32_t* device_bits) {
  uint32_t* p = gf::device_status_word();
  if (!p) return GF_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return GF_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return GF_ERR_CUDA;
  const uint32_t zero = 0;
  if (v && cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GF_ERR_CUDA;
  if (device_bits) *device_bits = int32_t(v);
  return v ? GF_ERR_DEVICE_CHECK : GF_OK;
}

}  // extern "C"
