// L2 read-bandwidth probe (measurement helper, see include/icpnn_probe.h).
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "icpnn_internal.h"
#include "icpnn_probe.h"

namespace icpnn {
namespace {

__global__ void __launch_bounds__(256) l2_read_kernel(const uint4* __restrict__ buf, int64_t n16, int repeats,
                                                      uint32_t* __restrict__ sink) {
  uint32_t acc = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int r = 0; r < repeats; ++r) {
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
      const uint4 a = __ldcg(&buf[i]);
      const uint4 b = __ldcg(&buf[i + stride]);
      const uint4 c = __ldcg(&buf[i + 2 * stride]);
      const uint4 d = __ldcg(&buf[i + 3 * stride]);
      acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
      const uint4 a = __ldcg(&buf[i]);
      acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
  }
  if (acc == 0x9e3779b9u) *sink = acc;  // never true for a buffer of ones; keeps the loads
}

}  // namespace
}  // namespace icpnn

extern "C" int icpnn_probe_l2_read(const void* buf, int64_t bytes, int32_t repeats, uint32_t* sink, void* stream) {
  using namespace icpnn;
  clear_error();
  if (buf == nullptr || sink == nullptr || bytes < 16 || bytes % 16 != 0 || repeats < 1 ||
      (reinterpret_cast<uintptr_t>(buf) & 15u) != 0)
    return fail(ICPNN_ERR_INVALID_ARG, "probe_l2_read: bad buffer, size or repeats");
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  l2_read_kernel<<<8 * sms, 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(buf), bytes / 16,
                                                                          repeats, sink);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ICPNN_ERR_CUDA, std::string("probe_l2_read: ") + cudaGetErrorString(e));
  return ICPNN_OK;
}
