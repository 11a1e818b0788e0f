// pack_build_seq_ids: per-token episode id from a segment table.
//
// "lingbot_va_packing" §2.1: tokens of latent frames at or past
// valid_frames[b] get seq_id -1 so FlexAttention drops them on both sides;
// "lingbot_va_attn_profiling" (packing proposal): concatenated episodes carry
// a per-token document id.  Row b holds K segments laid end to end; segment k
// covers seg_frames[b,k] frames, the first seg_valid[b,k] of them real.
#include <cuda_runtime.h>

#include "pvl_internal.h"

namespace pvl {
namespace {

struct SegmentTable {
  int32_t frames[PVL_MAX_SEGMENTS];
  int32_t valid[PVL_MAX_SEGMENTS];
};

constexpr int kThreads = 256;

// grid (ceil(L / 256), B).  The block first turns row b's segment lengths
// into token start offsets (one scan by thread 0: K is small), then every
// thread labels one position by binary search over the starts.
__global__ void __launch_bounds__(kThreads) seq_ids_kernel(const __grid_constant__ SegmentTable tab, int K,
                                                           int T, int L, int32_t* __restrict__ seq_id) {
  extern __shared__ int32_t starts[];  // K + 1 entries
  const int b = blockIdx.y;
  if (threadIdx.x == 0) {
    int32_t pos = 0;
    for (int k = 0; k < K; ++k) {
      starts[k] = pos;
      pos += tab.frames[b * K + k] * T;
    }
    starts[K] = pos;
  }
  __syncthreads();
  const int p = blockIdx.x * kThreads + threadIdx.x;
  if (p >= L) return;
  int32_t id = -1;
  if (p < starts[K]) {
    // last segment whose start is <= p; a zero-frame segment shares its start
    // with the next one, so "last" lands on the segment that holds p
    int lo = 0, hi = K - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (starts[mid] <= p) lo = mid; else hi = mid - 1;
    }
    const int frame = (p - starts[lo]) / T;
    if (frame < tab.valid[b * K + lo]) id = b * K + lo;
  }
  seq_id[static_cast<size_t>(b) * L + p] = id;
}

}  // namespace
}  // namespace pvl

using namespace pvl;

extern "C" pvl_status pack_build_seq_ids(const int32_t* seg_frames, const int32_t* seg_valid, int B, int K,
                                         int tokens_per_frame, int L, int32_t* seq_id, pvl_stream_t stream) {
  if (!seg_frames || !seg_valid || !seq_id) return fail(PVL_ERR_INVALID_ARG, "pack_build_seq_ids: null pointer");
  if (B < 1 || K < 1 || L < 1 || tokens_per_frame < 1)
    return fail(PVL_ERR_INVALID_ARG, "pack_build_seq_ids: B, K, L and tokens_per_frame must be >= 1");
  if (static_cast<long long>(B) * K > PVL_MAX_SEGMENTS)
    return fail(PVL_ERR_UNSUPPORTED, "pack_build_seq_ids: B*K = %lld exceeds %d", static_cast<long long>(B) * K,
                PVL_MAX_SEGMENTS);
  if (L > PVL_MAX_L) return fail(PVL_ERR_UNSUPPORTED, "pack_build_seq_ids: L = %d exceeds %d", L, PVL_MAX_L);
  SegmentTable tab;
  for (int b = 0; b < B; ++b) {
    long long tokens = 0;
    for (int k = 0; k < K; ++k) {
      const int f = seg_frames[b * K + k], v = seg_valid[b * K + k];
      if (f < 0 || v < 0 || v > f)
        return fail(PVL_ERR_INVALID_ARG, "pack_build_seq_ids: row %d segment %d needs 0 <= valid (%d) <= frames (%d)",
                    b, k, v, f);
      tokens += static_cast<long long>(f) * tokens_per_frame;
      tab.frames[b * K + k] = f;
      tab.valid[b * K + k] = v;
    }
    if (tokens > L)
      return fail(PVL_ERR_INVALID_ARG, "pack_build_seq_ids: row %d needs %lld tokens > L = %d", b, tokens, L);
  }
  dim3 grid((L + kThreads - 1) / kThreads, B);
  seq_ids_kernel<<<grid, kThreads, (K + 1) * sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)>>>(
      tab, K, tokens_per_frame, L, seq_id);
  return check_cuda(cudaGetLastError(), "pack_build_seq_ids launch");
}
