// Host runtime pieces shared by all entry points: status messages, the
// per-device error record, SM counts and TMA tensor-map creation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <unordered_map>

#include "pvl_internal.h"

namespace pvl {

__device__ DeviceError g_device_error;

// Work-item counters of the forward, one per (device, stream) in use.
constexpr int kSchedSlots = 256;
__device__ unsigned int g_fwd_sched[kSchedSlots];

namespace {
thread_local char t_message[512] = "ok";
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceError* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

std::atomic<uint64_t> g_attn_wait_ns{kDefaultTimeoutNs};
unsigned int* g_sched_base[kMaxDevices] = {};
std::unordered_map<uintptr_t, int> g_sched_slot[kMaxDevices];
thread_local void* t_mark_before = nullptr;
thread_local void* t_mark_after = nullptr;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
}  // namespace

pvl_status fail(pvl_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_message, sizeof(t_message), fmt, ap);
  va_end(ap);
  return s;
}

pvl_status check_cuda(int err, const char* what) {
  if (err == cudaSuccess) return PVL_OK;
  return fail(PVL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
}

DeviceError* device_error_record() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<DeviceError*>(p);
  }
  return g_err_ptr[dev];
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

uint64_t attn_wait_timeout_ns() { return g_attn_wait_ns.load(std::memory_order_relaxed); }

unsigned int* fwd_sched_counter(void* stream) {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  uintptr_t key = reinterpret_cast<uintptr_t>(stream);
  // the per-thread default stream is one handle for a different stream in
  // every host thread
  if (stream == reinterpret_cast<void*>(cudaStreamPerThread))
    key ^= std::hash<std::thread::id>{}(std::this_thread::get_id()) << 4;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sched_base[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_sched) != cudaSuccess) return nullptr;
    g_sched_base[dev] = static_cast<unsigned int*>(p);
  }
  auto& slots = g_sched_slot[dev];
  const auto found = slots.find(key);
  if (found != slots.end()) return g_sched_base[dev] + found->second;
  if (static_cast<int>(slots.size()) >= kSchedSlots) return nullptr;
  const int slot = static_cast<int>(slots.size());
  slots.emplace(key, slot);
  return g_sched_base[dev] + slot;
}

void take_bwd_main_marks(void** before, void** after) {
  *before = t_mark_before;
  *after = t_mark_after;
  t_mark_before = t_mark_after = nullptr;
}

pvl_status validate_attn(const char* who, const void* const* ptrs, int nptrs, int B, int L, int H, int D,
                         float scale) {
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i]) return fail(PVL_ERR_INVALID_ARG, "%s: pointer argument %d is null", who, i);
  if (B < 1 || L < 1 || H < 1) return fail(PVL_ERR_INVALID_ARG, "%s: B, L and H must be >= 1", who);
  if (!(scale > 0.0f) || !(scale < 1e30f)) return fail(PVL_ERR_INVALID_ARG, "%s: scale must be positive and finite", who);
  if (D != 64 && D != 128) return fail(PVL_ERR_UNSUPPORTED, "%s: D = %d (supported: 64, 128)", who, D);
  if (L > PVL_MAX_L) return fail(PVL_ERR_UNSUPPORTED, "%s: L = %d exceeds %d", who, L, PVL_MAX_L);
  if (static_cast<long long>(B) * L * H * D >= (1ll << 40))
    return fail(PVL_ERR_UNSUPPORTED, "%s: tensor of %lld elements is too large", who,
                static_cast<long long>(B) * L * H * D);
  if (static_cast<long long>(B) * ((L + 127) / 128) * H >= (1ll << 31))
    return fail(PVL_ERR_UNSUPPORTED, "%s: too many work items", who);
  for (int i = 0; i < nptrs; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0)
      return fail(PVL_ERR_UNSUPPORTED, "%s: pointer argument %d is not 16-byte aligned", who, i);
  return PVL_OK;
}

pvl_status validate_attn_qk(const char* who, const void* const* ptrs, int nptrs, int B, int Lq, int Lk, int H, int D,
                            float scale) {
  if (Lk < 1) return fail(PVL_ERR_INVALID_ARG, "%s: Lk must be >= 1", who);
  if (Lk > PVL_MAX_L) return fail(PVL_ERR_UNSUPPORTED, "%s: Lk = %d exceeds %d", who, Lk, PVL_MAX_L);
  if (static_cast<long long>(B) * Lk * H * D >= (1ll << 40))
    return fail(PVL_ERR_UNSUPPORTED, "%s: key tensor of %lld elements is too large", who,
                static_cast<long long>(B) * Lk * H * D);
  if (static_cast<long long>(B) * ((Lk + 127) / 128) * H >= (1ll << 31))
    return fail(PVL_ERR_UNSUPPORTED, "%s: too many work items", who);
  return validate_attn(who, ptrs, nptrs, B, Lq, H, D, scale);
}

namespace {
pvl_status encode_bhld(void* map_out, const void* base, CUtensorMapDataType type, int esize, int B, int L, int H,
                       int D, const cuuint32_t box[4], CUtensorMapSwizzle swizzle);
}  // namespace

pvl_status make_bhld_tensor_map(void* map_out, const void* base, int B, int L, int H, int D) {
  const cuuint32_t box[4] = {64, 1, 128, 1};
  return encode_bhld(map_out, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, L, H, D, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

pvl_status make_bhld_f32_tensor_map(void* map_out, const void* base, int B, int L, int H, int D, int box_d,
                                    int box_rows) {
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_d), 1, static_cast<cuuint32_t>(box_rows), 1};
  // a 128-byte box row takes the 128-byte swizzle, so that a warp writing one
  // row per lane stages it without shared-memory bank conflicts
  const CUtensorMapSwizzle sw = box_d * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  return encode_bhld(map_out, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B, L, H, D, box, sw);
}

namespace {
pvl_status encode_bhld(void* map_out, const void* base, CUtensorMapDataType type, int esize, int B, int L, int H,
                       int D, const cuuint32_t box[4], CUtensorMapSwizzle swizzle) {
  // cuTensorMapEncodeTiled is a driver call and needs a current context on
  // this thread.  A thread that has made no runtime call yet (for example a
  // torch autograd worker) has none; setting the current device binds the
  // device's primary context.
  {
    int dev = 0;
    pvl_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st == PVL_OK) st = check_cuda(cudaSetDevice(dev), "cudaSetDevice");
    if (st != PVL_OK) return st;
  }
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      const cudaError_t e =
          cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(PVL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(B)};
  const cuuint64_t es = static_cast<cuuint64_t>(esize);
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * es, static_cast<cuuint64_t>(H) * D * es,
                                 static_cast<cuuint64_t>(L) * H * D * es};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map_out), type, 4, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PVL_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  return PVL_OK;
}
}  // namespace

}  // namespace pvl

using namespace pvl;

extern "C" pvl_status pvl_device_error_detail(pvl_stream_t stream, int32_t* info) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  pvl_status st = check_cuda(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  if (st != PVL_OK) return st;
  DeviceError* rec = device_error_record();
  if (!rec) return fail(PVL_ERR_CUDA, "device error record is not available");
  DeviceError h{};
  st = check_cuda(cudaMemcpy(&h, rec, sizeof(h), cudaMemcpyDeviceToHost), "reading the device error record");
  if (st != PVL_OK) return st;
  if (h.code != 0) {
    const DeviceError zero{};
    st = check_cuda(cudaMemcpy(rec, &zero, sizeof(zero), cudaMemcpyHostToDevice), "clearing the device error record");
    if (st != PVL_OK) return st;
  }
  if (info) {
    info[0] = static_cast<int32_t>(h.code);
    info[1] = static_cast<int32_t>(h.where);
    info[2] = static_cast<int32_t>(h.block);
    info[3] = static_cast<int32_t>(h.thread);
  }
  if (h.code == kDevErrTimeout)
    return fail(PVL_ERR_TIMEOUT, "device wait timed out (site %u, block %u, thread %u)", h.where, h.block, h.thread);
  if (h.code == kDevErrTileMap)
    return fail(PVL_ERR_INVALID_ARG, "tile map was built for another shape or block size");
  if (h.code != 0) return fail(PVL_ERR_CUDA, "unknown device error code %u", h.code);
  return PVL_OK;
}

extern "C" pvl_status pvl_device_error(pvl_stream_t stream) { return pvl_device_error_detail(stream, nullptr); }

extern "C" pvl_status pvl_set_attn_wait_timeout_ns(uint64_t ns) {
  if (ns > 60000000000ull) return fail(PVL_ERR_INVALID_ARG, "pvl_set_attn_wait_timeout_ns: %llu ns exceeds 60 s",
                                       static_cast<unsigned long long>(ns));
  g_attn_wait_ns.store(ns == 0 ? kDefaultTimeoutNs : ns, std::memory_order_relaxed);
  return PVL_OK;
}

extern "C" pvl_status pvl_mark_next_bwd_main(void* before, void* after) {
  t_mark_before = before;
  t_mark_after = after;
  return PVL_OK;
}

extern "C" const char* pvl_last_error_message(void) { return t_message; }

extern "C" int pvl_version(void) { return 0x000100; }
