// Host-side runtime of the library: device status word, tensor-map encoding
// through the driver entry point (no link against libcuda), per-device
// caches, status strings.
#include <mutex>

#include "common.cuh"

namespace mxq {
// One status word per device context; kernels receive its address.
__device__ int g_status = 0;
}  // namespace mxq

namespace mxq_host {

std::mutex g_mu;
namespace {
constexpr int kMaxDev = 64;
int g_sms[kMaxDev] = {};
int g_ok[kMaxDev] = {};          // 0 unknown, 1 ok, -1 not sm_103
int* g_status_ptr[kMaxDev] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cur_dev() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return (d >= 0 && d < kMaxDev) ? d : -1;
}
}  // namespace

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  const int d = cur_dev();
  if (d < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

bool device_ok() {
  const int d = cur_dev();
  if (d < 0) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ok[d]) {
    int maj = 0, mnr = 0;
    cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&mnr, cudaDevAttrComputeCapabilityMinor, d);
    g_ok[d] = (maj == 10 && mnr == 3) ? 1 : -1;
  }
  return g_ok[d] == 1;
}

int* status_ptr() {
  const int d = cur_dev();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, mxq::g_status) != cudaSuccess) return nullptr;
    g_status_ptr[d] = static_cast<int*>(p);
  }
  return g_status_ptr[d];
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA; }

int g_test_stall = 0;

bool take_test_stall(int which) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_test_stall != which) return false;
  g_test_stall = 0;
  return true;
}

}  // namespace mxq_host

extern "C" int mxq_last_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MXQ_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, mxq::g_status, sizeof(int)) != cudaSuccess) return MXQ_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(mxq::g_status, &zero, sizeof(int)) != cudaSuccess) return MXQ_ERR_CUDA;
  }
  return v;
}

extern "C" const char* mxq_strerror(int s) {
  switch (s) {
    case MXQ_OK: return "ok";
    case MXQ_ERR_BAD_ARG: return "bad argument (NULL pointer, unknown enum value or bad ring index)";
    case MXQ_ERR_BAD_SHAPE: return "bad shape (size not a multiple of the block or tile)";
    case MXQ_ERR_MISALIGNED: return "misaligned pointer or leading dimension (16 bytes required)";
    case MXQ_ERR_UNSUPPORTED: return "unsupported format/orientation combination or device (needs sm_103)";
    case MXQ_ERR_CUDA: return "CUDA launch or driver error";
    case MXQ_ERR_TIMEOUT: return "a bounded device wait expired";
    default: return "unknown status";
  }
}

extern "C" int mxq_test_stall_next_launch(int which) {
  if (which != 0 && which != 1 && which != 2) return MXQ_ERR_BAD_ARG;
  std::lock_guard<std::mutex> lk(mxq_host::g_mu);
  mxq_host::g_test_stall = which;
  return MXQ_OK;
}

extern "C" int mxq_version(void) { return 200; }
