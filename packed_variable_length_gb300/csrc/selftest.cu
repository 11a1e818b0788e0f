// pvl_selftest_wait_timeout: exercises the bounded-wait path every kernel of
// the library uses, without a fault.  One CTA of two warps: warp 0 waits on
// an mbarrier that nothing arrives on, with a short limit, and records a
// timeout; warp 1 waits on a second such barrier with a long limit and must
// leave through the CTA's abort flag that warp 0's timeout raised.  Both
// waits return false and the kernel ends; the host then finds the timeout
// (site kSiteSelftest) in the device error record.
#include <cuda_runtime.h>

#include "pvl_device.cuh"

namespace pvl {
namespace {

constexpr uint32_t kSiteSelftestShort = 91;
constexpr uint32_t kSiteSelftestLong = 92;

__device__ int g_selftest_out[2];

__global__ void __launch_bounds__(64) wait_timeout_kernel(DeviceError* err, uint64_t short_ns, uint64_t long_ns) {
  __shared__ uint64_t bar_a, bar_b;
  __shared__ int abort_s;
  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bar_a, 1);
    mbar_init(&bar_b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const KernelCtl ctl{err, &abort_s, warp == 0 ? short_ns : long_ns};
  const bool ok = __all_sync(0xffffffffu, mbar_wait(warp == 0 ? &bar_a : &bar_b, 0, ctl,
                                                     warp == 0 ? kSiteSelftestShort : kSiteSelftestLong));
  if ((threadIdx.x & 31) == 0) g_selftest_out[warp] = ok ? 1 : 0;
  __syncthreads();
}

}  // namespace
}  // namespace pvl

using namespace pvl;

extern "C" pvl_status pvl_selftest_wait_timeout(uint64_t short_ns, uint64_t long_ns, int32_t* out,
                                                pvl_stream_t stream) {
  if (!out) return fail(PVL_ERR_INVALID_ARG, "pvl_selftest_wait_timeout: out is null");
  if (short_ns == 0 || short_ns > 10000000000ull || long_ns < short_ns || long_ns > 60000000000ull)
    return fail(PVL_ERR_INVALID_ARG, "pvl_selftest_wait_timeout: need 0 < short_ns <= long_ns, short <= 10 s, long <= 60 s");
  DeviceError* err = device_error_record();
  if (!err) return fail(PVL_ERR_CUDA, "pvl_selftest_wait_timeout: no usable CUDA device");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  wait_timeout_kernel<<<1, 64, 0, s>>>(err, short_ns, long_ns);
  pvl_status st = check_cuda(cudaGetLastError(), "pvl_selftest_wait_timeout launch");
  if (st != PVL_OK) return st;
  int host[2] = {-1, -1};
  st = check_cuda(cudaMemcpyFromSymbolAsync(host, g_selftest_out, sizeof(host), 0, cudaMemcpyDeviceToHost, s),
                  "pvl_selftest_wait_timeout copy");
  if (st == PVL_OK) st = check_cuda(cudaStreamSynchronize(s), "pvl_selftest_wait_timeout sync");
  out[0] = host[0];
  out[1] = host[1];
  return st;
}
