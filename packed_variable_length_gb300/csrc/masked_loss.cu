// masked_mse_loss / masked_mse_loss_bwd: the squared-error loss averaged
// over the valid frames only, and its gradient, for sm_103a.
//
// What it computes ("lingbot_va_packing" §2.1, compute_loss: frame_valid =
// f < valid_frames[b], latent and action losses averaged over valid frames;
// "furniture_packing_variable_length", the loss paragraph): per stream of
// tokens [B, L] with C values each and the token mask seq_id >= 0 (the mask
// the attention uses; on pad-collated rows it is frame_valid spread over
// the frame's tokens),
//   loss  = sum_{valid tokens} sum_c (pred - target)^2 / (C n_valid),
//   dpred = dloss 2 (pred - target) / (C n_valid) on valid tokens, else 0,
// with loss = 0 and dpred = 0 when no token is valid.
//
// Design.  The loss sits right after the model's output projection and is
// HBM bound: 2 bytes of pred and 2 of target read per valid element, 2 of
// gradient written per element.  One cooperative launch (every CTA resident,
// so the CTAs may wait on one another), after a 64-byte clear of the
// workspace counters:
//   - each CTA counts the valid tokens of its share of seq_id while its
//     first block of data is in flight and adds (one arrival | its count) to
//     one 64-bit word in one integer atomic (exact in any order);
//   - with the gradient, a grid barrier on that word (a bounded wait: on
//     expiry the kernel records a timeout and returns): a CTA that sees every
//     arrival in the word sees the whole count too, so no fence is needed.
//     The loss alone needs no barrier;
//   - every CTA streams its grid-stride share of 16-byte vectors: the
//     token's id decides whether pred and target are read at all (padding
//     tokens cost no reads), the squared error goes into a per-thread fp32
//     sum and the gradient is written in the same pass, the next block's ids
//     fetched while the current block's data is in flight;
//   - the CTA's sum (its warps' fp32 sums added as a pair hi + lo of fp32
//     values) lands in a slot; the last CTA to finish adds the slots in CTA
//     order, also as a pair, and divides once: the loss is deterministic for
//     a given grid, and no step uses fp64, which GB300 runs at a small
//     fraction of its fp32 rate.
#include <cuda_runtime.h>

#include "pvl_device.cuh"

namespace pvl {
namespace {

constexpr int kLossThreads = 512;
constexpr int kMaxLossCtas = 2048;
constexpr int kUnroll = 2;
constexpr uint32_t kSiteGridBarrier = 61;

// workspace layout (bytes); the first 64 are cleared before every launch
constexpr size_t kWsCount = 0;   // uint64: CTAs arrived (high 32 bits) | valid tokens counted (low 32 bits)
constexpr size_t kWsDone = 8;    // uint32: CTAs finished
constexpr size_t kWsClear = 64;
constexpr size_t kWsParts = 64;  // per CTA its squared-error sum as a pair (hi, lo) of fp32 values
constexpr size_t kWsBytes = kWsParts + 8 * kMaxLossCtas;

struct LossParams {
  const __nv_bfloat16* pred;
  const __nv_bfloat16* target;
  const int32_t* seq_id;
  float* loss;              // null: gradient only
  __nv_bfloat16* grad;      // null: loss only
  const float* dloss;       // device upstream gradient, or null for grad_scale
  float grad_scale;
  uint8_t* ws;
  DeviceError* err;
  long long n_ids;          // B * L
  long long n_vec;          // B * L * C / 8
  int vec_per_tok;          // C / 8
  int C;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// (hi, lo) += (bh, bl) for unevaluated pairs hi + lo of fp32 values: the
// exact error of hi + bh (Knuth's two-sum) plus the low parts, renormalised
// (Dekker's fast two-sum).  Commutative, so both lanes of a butterfly step
// get the same pair.
__device__ __forceinline__ void pair_add(float& hi, float& lo, float bh, float bl) {
  const float s = __fadd_rn(hi, bh);
  const float bb = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(bh, bb)), __fadd_rn(lo, bl));
  hi = __fadd_rn(s, e);
  lo = __fsub_rn(e, __fsub_rn(hi, s));
}

// (hi + lo) / den for an integer den < 2^48 (here C n_valid < 2^40): den
// split into dh + dl (dl exact), the quotient hi / dh corrected by its
// remainder, which the fused multiply-add gives exactly; within about one
// fp32 ulp.
__device__ __forceinline__ float pair_div(float hi, float lo, unsigned long long den) {
  const float dh = static_cast<float>(den);
  const float dl = static_cast<float>(static_cast<long long>(den) - static_cast<long long>(dh));
  const float q0 = __fdiv_rn(hi, dh);
  const float r = __fadd_rn(__fsub_rn(fmaf(-q0, dh, hi), __fmul_rn(q0, dl)), lo);
  return __fadd_rn(q0, __fdiv_rn(r, dh));
}

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <bool kLoss, bool kGrad>
__global__ void __launch_bounds__(kLossThreads, 2) loss_kernel(const LossParams p) {
  __shared__ uint32_t warp_n[kLossThreads / 32];
  __shared__ float warp_s[kLossThreads / 32];
  __shared__ int flag_s;
  __shared__ uint32_t n_valid_s;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;

  // This thread's vectors: v0, v0 + stride, ..., taken kUnroll at a time;
  // the ids of the next block are fetched while the current block's data is
  // in flight.  Token and position in the token advance without a division
  // per vector.
  const long long stride = static_cast<long long>(gridDim.x) * kLossThreads;
  const long long v0 = static_cast<long long>(blockIdx.x) * kLossThreads + t;
  const long long stride_tok = stride / p.vec_per_tok;
  const int stride_rem = static_cast<int>(stride % p.vec_per_tok);
  long long tok = v0 / p.vec_per_tok;  // token of the next vector whose id is fetched
  int rem = static_cast<int>(v0 % p.vec_per_tok);
  auto fetch_ids = [&](long long vbase, int (&ids)[kUnroll]) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      ids[u] = vbase + u * stride < p.n_vec ? __ldg(p.seq_id + tok) : -1;
      tok += stride_tok;
      rem += stride_rem;
      if (rem >= p.vec_per_tok) {
        rem -= p.vec_per_tok;
        ++tok;
      }
    }
  };
  auto load_data = [&](long long vbase, const int (&ids)[kUnroll], uint4 (&a)[kUnroll], uint4 (&b)[kUnroll]) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (ids[u] >= 0) {
        a[u] = ld_stream(p.pred + (vbase + u * stride) * 8);
        b[u] = ld_stream(p.target + (vbase + u * stride) * 8);
      } else {
        a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  int ids[kUnroll], ids_next[kUnroll];
  uint4 a[kUnroll], b[kUnroll];
  fetch_ids(v0, ids);
  load_data(v0, ids, a, b);  // the first block is in flight across the count and the barrier

  // Valid tokens of this CTA's share of the ids (16 bytes at a time; CTA 0
  // takes the ragged tail).
  {
    uint32_t n = 0;
    const long long n4 = p.n_ids / 4;
    for (long long i = static_cast<long long>(blockIdx.x) * kLossThreads + t; i < n4; i += stride) {
      const int4 q = __ldg(reinterpret_cast<const int4*>(p.seq_id) + i);
      n += (q.x >= 0) + (q.y >= 0) + (q.z >= 0) + (q.w >= 0);
    }
    if (blockIdx.x == 0 && t < 4 && n4 * 4 + t < p.n_ids) n += p.seq_id[n4 * 4 + t] >= 0;
    n = __reduce_add_sync(0xffffffffu, n);
    if (lane == 0) warp_n[w] = n;
  }
  __syncthreads();
  // Arrival and count go into one word in one atomic: a CTA that sees every
  // arrival in it sees the whole count too, with no fence.
  uint64_t* count_word = reinterpret_cast<uint64_t*>(p.ws + kWsCount);
  if (t == 0) {
    uint32_t cta_n = 0;
    for (int i = 0; i < kLossThreads / 32; ++i) cta_n += warp_n[i];
    atomicAdd(reinterpret_cast<unsigned long long*>(count_word), (1ull << 32) | cta_n);
  }

  float norm = 0.0f;
  if constexpr (kGrad) {
    // The gradient needs n_valid: a grid barrier on the count word.  Every
    // CTA is resident (cooperative launch), so the wait ends unless something
    // is broken; it is bounded all the same.
    if (t == 0) {
      int ok = 1;
      const uint64_t t0 = global_timer_ns();
      uint64_t c = ld_relaxed(count_word);
      while ((c >> 32) < gridDim.x) {
        __nanosleep(100);
        if (global_timer_ns() - t0 > p.timeout_ns) {
          if (atomicCAS(&p.err->code, 0u, kDevErrTimeout) == 0u) {
            p.err->where = kSiteGridBarrier;
            p.err->block = blockIdx.x;
            p.err->thread = 0;
          }
          ok = 0;
          break;
        }
        c = ld_relaxed(count_word);
      }
      n_valid_s = static_cast<uint32_t>(c);
      flag_s = ok;
    }
    __syncthreads();
    if (!flag_s) return;
    const uint32_t n_valid = n_valid_s;
    if (n_valid > 0)
      norm = 2.0f * (p.dloss ? *p.dloss : p.grad_scale) / (static_cast<float>(p.C) * static_cast<float>(n_valid));
  }

  float sse = 0.0f;
  for (long long v = v0; v < p.n_vec; v += kUnroll * stride) {
    fetch_ids(v + kUnroll * stride, ids_next);  // the next block's ids, while this block's data is in flight
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long vv = v + u * stride;
      if (vv >= p.n_vec) continue;
      const uint32_t wa[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
      const uint32_t wb[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
      uint32_t og[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 pa = make_float2(__uint_as_float(wa[e] << 16), __uint_as_float(wa[e] & 0xFFFF0000u));
        const float2 pb = make_float2(__uint_as_float(wb[e] << 16), __uint_as_float(wb[e] & 0xFFFF0000u));
        const float2 d = make_float2(pa.x - pb.x, pa.y - pb.y);
        if (kLoss) sse = fmaf(d.x, d.x, fmaf(d.y, d.y, sse));
        if (kGrad) og[e] = pack_bf16x2(d.x * norm, d.y * norm);
      }
      if (kGrad) st_stream(p.grad + vv * 8, make_uint4(og[0], og[1], og[2], og[3]));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) ids[u] = ids_next[u];
    load_data(v + kUnroll * stride, ids, a, b);
  }

  if constexpr (kLoss) {
    // The CTA's sum (fp32 inside each warp, then the warp sums as a pair
    // hi + lo of fp32 values, about 48 significant bits) goes to its slot;
    // the last CTA to finish adds the slots in a fixed order, so the loss is
    // deterministic for a given grid, and needs no fp64 unit.  Every CTA added
    // its count before it counted itself done (release), so the last one
    // (acquire) reads the whole count.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sse += __shfl_xor_sync(0xffffffffu, sse, o);
    if (lane == 0) warp_s[w] = sse;
    __syncthreads();
    if (w != 0) return;
    float hi = lane < kLossThreads / 32 ? warp_s[lane] : 0.0f, lo = 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
    float2* parts = reinterpret_cast<float2*>(p.ws + kWsParts);
    uint32_t last = 0;
    if (lane == 0) {
      parts[blockIdx.x] = make_float2(hi, lo);
      last = atom_add_acq_rel(reinterpret_cast<uint32_t*>(p.ws + kWsDone), 1u) == gridDim.x - 1;
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __syncwarp();     // the other lanes read after lane 0's acquire
    fence_acq_rel();
    hi = lo = 0.0f;
    for (int i = lane; i < static_cast<int>(gridDim.x); i += 32) {
      const float2 q = __ldcg(parts + i);
      pair_add(hi, lo, q.x, q.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
    if (lane == 0) {
      const uint32_t n_valid = static_cast<uint32_t>(ld_relaxed(count_word));
      *p.loss = n_valid > 0 ? pair_div(hi, lo, static_cast<unsigned long long>(p.C) * n_valid) : 0.0f;
    }
  }
}

pvl_status validate(const char* who, const void* const* ptrs, int nptrs, int B, int L, int C) {
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i]) return fail(PVL_ERR_INVALID_ARG, "%s: pointer argument %d is null", who, i);
  if (B < 1 || L < 1 || C < 1) return fail(PVL_ERR_INVALID_ARG, "%s: B, L and C must be >= 1", who);
  if (C % 8 != 0) return fail(PVL_ERR_UNSUPPORTED, "%s: C = %d (supported: multiples of 8)", who, C);
  const long long tokens = static_cast<long long>(B) * L;
  if (tokens >= (1ll << 31) || tokens * C >= (1ll << 40)) return fail(PVL_ERR_UNSUPPORTED, "%s: tensor too large", who);
  for (int i = 0; i < nptrs; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0)
      return fail(PVL_ERR_UNSUPPORTED, "%s: pointer argument %d is not 16-byte aligned", who, i);
  return PVL_OK;
}

template <bool kLoss, bool kGrad>
pvl_status launch_loss(LossParams& p, long long needed, int sms, cudaStream_t s, const char* who) {
  int occ = 0;
  pvl_status st = check_cuda(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, loss_kernel<kLoss, kGrad>,
                                                                           kLossThreads, 0), who);
  if (st != PVL_OK) return st;
  if (occ < 1) return fail(PVL_ERR_CUDA, "%s: the kernel does not fit on an SM", who);
  long long grid = needed;
  if (grid > static_cast<long long>(occ) * sms) grid = static_cast<long long>(occ) * sms;  // all resident
  if (grid > kMaxLossCtas) grid = kMaxLossCtas;
  void* args[] = {&p};
  return check_cuda(cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(loss_kernel<kLoss, kGrad>),
                                                dim3(static_cast<unsigned>(grid)), dim3(kLossThreads), args, 0, s),
                    who);
}

pvl_status launch(LossParams p, int B, int L, int C, size_t ws_bytes, cudaStream_t s, const char* who) {
  if (ws_bytes < kWsBytes) return fail(PVL_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed", who, ws_bytes, kWsBytes);
  p.err = device_error_record();
  if (!p.err) return fail(PVL_ERR_CUDA, "%s: no usable CUDA device", who);
  const int sms = sm_count();
  if (sms <= 0) return fail(PVL_ERR_CUDA, "%s: no usable CUDA device", who);
  p.n_ids = static_cast<long long>(B) * L;
  p.C = C;
  p.vec_per_tok = C / 8;
  p.n_vec = p.n_ids * (C / 8);
  p.timeout_ns = kDefaultTimeoutNs;
  long long needed = (p.n_vec + static_cast<long long>(kLossThreads) * kUnroll - 1) /
                     (static_cast<long long>(kLossThreads) * kUnroll);
  if (needed < 1) needed = 1;
  const pvl_status st = check_cuda(cudaMemsetAsync(p.ws, 0, kWsClear, s), who);
  if (st != PVL_OK) return st;
  if (p.loss && p.grad) return launch_loss<true, true>(p, needed, sms, s, who);
  if (p.loss) return launch_loss<true, false>(p, needed, sms, s, who);
  return launch_loss<false, true>(p, needed, sms, s, who);
}

}  // namespace
}  // namespace pvl

using namespace pvl;

extern "C" size_t masked_mse_ws_bytes(int B, int L, int C) {
  if (B < 1 || L < 1 || C < 1) return 0;
  return kWsBytes;
}

extern "C" pvl_status masked_mse_loss(const pvl_bf16* pred, const pvl_bf16* target, const int32_t* seq_id, int B,
                                      int L, int C, float* loss, pvl_bf16* grad, float grad_scale, void* ws,
                                      size_t ws_bytes, pvl_stream_t stream) {
  const void* ptrs[] = {pred, target, seq_id, ws};
  pvl_status st = validate("masked_mse_loss", ptrs, 4, B, L, C);
  if (st != PVL_OK) return st;
  if (!loss) return fail(PVL_ERR_INVALID_ARG, "masked_mse_loss: loss is null");
  if (reinterpret_cast<uintptr_t>(loss) % 4 || (grad && reinterpret_cast<uintptr_t>(grad) % 16))
    return fail(PVL_ERR_UNSUPPORTED, "masked_mse_loss: loss must be 4-byte and grad 16-byte aligned");
  if (!(grad_scale == grad_scale) || grad_scale > 3.0e38f || grad_scale < -3.0e38f)
    return fail(PVL_ERR_INVALID_ARG, "masked_mse_loss: grad_scale must be finite");
  LossParams p{};
  p.pred = reinterpret_cast<const __nv_bfloat16*>(pred);
  p.target = reinterpret_cast<const __nv_bfloat16*>(target);
  p.seq_id = seq_id;
  p.loss = loss;
  p.grad = reinterpret_cast<__nv_bfloat16*>(grad);
  p.grad_scale = grad_scale;
  p.ws = static_cast<uint8_t*>(ws);
  return launch(p, B, L, C, ws_bytes, reinterpret_cast<cudaStream_t>(stream), "masked_mse_loss");
}

extern "C" pvl_status masked_mse_loss_bwd(const pvl_bf16* pred, const pvl_bf16* target, const int32_t* seq_id,
                                          int B, int L, int C, const float* dloss, pvl_bf16* grad, void* ws,
                                          size_t ws_bytes, pvl_stream_t stream) {
  const void* ptrs[] = {pred, target, seq_id, grad, ws};
  pvl_status st = validate("masked_mse_loss_bwd", ptrs, 5, B, L, C);
  if (st != PVL_OK) return st;
  if (!dloss) return fail(PVL_ERR_INVALID_ARG, "masked_mse_loss_bwd: dloss is null");
  if (reinterpret_cast<uintptr_t>(dloss) % 4)
    return fail(PVL_ERR_UNSUPPORTED, "masked_mse_loss_bwd: dloss must be 4-byte aligned");
  LossParams p{};
  p.pred = reinterpret_cast<const __nv_bfloat16*>(pred);
  p.target = reinterpret_cast<const __nv_bfloat16*>(target);
  p.seq_id = seq_id;
  p.grad = reinterpret_cast<__nv_bfloat16*>(grad);
  p.dloss = dloss;
  p.grad_scale = 1.0f;
  p.ws = static_cast<uint8_t*>(ws);
  return launch(p, B, L, C, ws_bytes, reinterpret_cast<cudaStream_t>(stream), "masked_mse_loss_bwd");
}
