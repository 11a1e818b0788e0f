// adaln_fwd / adaln_bwd: layer norm over the feature dimension followed by
// the AdaLN modulation, fused, for sm_103a.
//
// What it computes ("AdaptiveLoad" §2.B, the fused LayerNorm-Modulate
// kernel of a DiT / MMDiT block): per batch row b and token n,
//   mu = mean_d x,  r = 1 / sqrt(mean_d (x - mu)^2 + eps),  xh = (x - mu) r,
//   y  = xh (1 + scale_b) + shift_b;
// backward, with g = dy (1 + scale_b):
//   dx = r (g - mean_d g - xh mean_d(g xh)),
//   dshift_b = sum_n dy,  dscale_b = sum_n dy xh.
//
// Design.  The path is HBM bound (2 bytes read and 2 written per element
// forward, 4 read and 2 written backward), so everything is about keeping
// bytes in flight and touching each element once:
//   - one persistent CTA of 256 threads per SM walks rows; thread 0 streams
//     the rows (x, and dy backward) into a ring of shared-memory stages with
//     bulk asynchronous copies, so several rows are in flight without
//     holding them in registers;
//   - the CTA works on one row at a time: each thread owns the same 8-wide
//     feature groups of every row; row sums go through a warp shuffle and a
//     block reduction (two-level, as the page describes), and the statistics
//     never leave the chip; the modulation is applied on the way out;
//   - backward, the rows of a work item (one batch row, a tile of
//     kRowsPerTile tokens) accumulate dshift / dscale in the registers of
//     the threads that own each feature: the sequence-direction reduction of
//     the page's D-tile scheme, with coalesced reads along the features.
//     Each item writes its partial sums once; a small kernel adds the tiles'
//     partials per batch row, in a fixed order (deterministic).
// Every wait is bounded; on expiry the CTA records the failure, waits for
// its copies in flight and returns.
#include <cuda_runtime.h>

#include "pvl_device.cuh"

namespace pvl {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerTile = 64;  // backward work item: tokens of one batch row
constexpr int kMaxD = 8192;

enum AdalnSite : uint32_t { kSiteRowFull = 41 };

// Stage bytes of one row of D bf16, rounded up to 128 bytes.
__host__ __device__ constexpr int row_bytes(int D) { return ((D * 2 + 127) / 128) * 128; }

__device__ __forceinline__ float2 warp_sum2(float2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  return v;
}

// Sum over the CTA through `red` (kWarps slots, not reused before the next
// __syncthreads of the caller).
__device__ __forceinline__ float2 block_sum2(float2 v, float2* red) {
  v = warp_sum2(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float2 t = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    t.x += red[w].x;
    t.y += red[w].y;
  }
  return t;
}

// 8 fp32 values as 4 pairs from global memory through the read-only cache
__device__ __forceinline__ void load_scale(const float* p8, float2 (&v)[4]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p8));
  const float4 c = __ldg(reinterpret_cast<const float4*>(p8) + 1);
  v[0] = make_float2(a.x, a.y);
  v[1] = make_float2(a.z, a.w);
  v[2] = make_float2(c.x, c.y);
  v[3] = make_float2(c.z, c.w);
}

// 8 bf16 values (one 16-byte vector) as 4 fp32 pairs, in order
__device__ __forceinline__ void unpack8x2(const uint4 u, float2 (&f)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
}

struct AdalnParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* dy;  // backward only
  const float* shift;       // forward only
  const float* scale;
  __nv_bfloat16* out;       // y forward, dx backward
  float* mean;              // forward, optional
  float* rstd;              // forward, optional
  float* part;              // backward: [2][B * n_tiles][D] tile partials
  DeviceError* err;
  int B, N, D, n_tiles;
  long long items;          // forward: rows; backward: B * n_tiles
  float eps;
  uint64_t timeout_ns;
};

// CTAs per SM: two, except the widest backward rows (registers).
template <int kV, bool kBwd>
constexpr int ctas_per_sm() {
  return (kBwd && kV == 4) ? 1 : 2;
}

template <int kV, bool kBwd, int kStages>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<kV, kBwd>()) adaln_kernel(const AdalnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kStages];
  __shared__ float2 red_m[kWarps];  // row statistics
  __shared__ float2 red[kWarps];    // backward: sums of g and g xh
  __shared__ int abort_s;
  constexpr int kTensors = kBwd ? 2 : 1;
  const int D = p.D;
  const int RB = row_bytes(D);
  const int nvec = D / 8;
  const int t = threadIdx.x;
  const KernelCtl ctl{p.err, &abort_s, p.timeout_ns};

  if (t == 0) {
    abort_s = 0;
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // The rows this CTA handles, in order: forward rows blockIdx.x,
  // blockIdx.x + gridDim.x, ...; backward whole items, kRowsPerTile tokens
  // each (fewer in the last tile of a batch row).
  auto item_rows = [&](long long item) -> int {
    if (!kBwd) return 1;
    const int tile = static_cast<int>(item % p.n_tiles);
    const int n0 = tile * kRowsPerTile;
    return min(kRowsPerTile, p.N - n0);
  };
  auto row_index = [&](long long item, int k) -> long long {  // global row b * N + n
    if (!kBwd) return item;
    const long long b = item / p.n_tiles;
    const int tile = static_cast<int>(item % p.n_tiles);
    return b * p.N + static_cast<long long>(tile) * kRowsPerTile + k;
  };
  // Producer state (thread 0): next (item, k) to load.
  long long ld_item = blockIdx.x;
  int ld_k = 0;
  uint32_t ld_n = 0;  // rows issued
  auto issue_next = [&]() {
    if (ld_item >= p.items) return;
    const int st = ld_n % kStages;
    const long long r = row_index(ld_item, ld_k);
    uint8_t* dst = smem + static_cast<size_t>(st) * kTensors * RB;
    mbar_arrive_expect_tx(&full[st], kTensors * D * 2);
    bulk_load(dst, p.x + r * D, D * 2, &full[st]);
    if (kBwd) bulk_load(dst + RB, p.dy + r * D, D * 2, &full[st]);
    ++ld_n;
    if (++ld_k == item_rows(ld_item)) {
      ld_k = 0;
      ld_item += gridDim.x;
    }
  };
  if (t == 0)
    for (int s = 0; s < kStages; ++s) issue_next();

  uint32_t use_n = 0;  // rows consumed
  bool alive = true;
  // per-thread modulation of the owned feature groups, reloaded when the
  // batch row changes
  float2 mod[kV][4];  // 1 + scale (forward)
  float2 sh[kV][4];   // shift (forward)
  int cur_b = -1;
  for (long long item = blockIdx.x; item < p.items && alive; item += gridDim.x) {
    const int nrows = item_rows(item);
    const int b = static_cast<int>(row_index(item, 0) / p.N);
    float2 acc_s[kBwd ? kV : 1][4], acc_c[kBwd ? kV : 1][4];  // dshift, dscale partials
    const bool reload = !kBwd && b != cur_b;
    cur_b = b;
#pragma unroll
    for (int i = 0; i < kV; ++i) {
      if (kBwd) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_s[i][e] = acc_c[i][e] = make_float2(0.f, 0.f);
      }
      if (!reload) continue;
      const int v = t + i * kThreads;
      if (v < nvec) {
        float2 sc[4], sf[4];
        load_scale(p.scale + static_cast<size_t>(b) * D + v * 8, sc);
        load_scale(p.shift + static_cast<size_t>(b) * D + v * 8, sf);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          mod[i][e] = make_float2(1.0f + sc[e].x, 1.0f + sc[e].y);
          sh[i][e] = sf[e];
        }
      }
    }
    for (int k = 0; k < nrows; ++k, ++use_n) {
      const int st = use_n % kStages;
      if (!__syncthreads_and(mbar_wait(&full[st], (use_n / kStages) & 1, ctl, kSiteRowFull))) {
        alive = false;
        break;
      }
      const uint8_t* src = smem + static_cast<size_t>(st) * kTensors * RB;
      const long long r = row_index(item, k);
      // Row statistics in one reduction of shifted sums: with K the row's
      // first element, S1 = sum (x - K), S2 = sum (x - K)^2, mean = K + S1/D
      // and var = S2/D - (S1/D)^2.  K is a sample of the row, so (mean - K)^2
      // stays within a factor ~D of the variance even for an outlier K: the
      // cancellation costs at most ~D * 2^-24 relative, far below bf16's 2^-9.
      const float K = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(src)) << 16);
      const float2 nk = make_float2(-K, -K);
      float2 xv[kV][4];
      float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = t + i * kThreads;
        if (v < nvec) {
          unpack8x2(reinterpret_cast<const uint4*>(src)[v], xv[i]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 d = fadd2(xv[i][e], nk);
            s1 = fadd2(s1, d);
            s2 = ffma2(d, d, s2);
          }
        }
      }
      const float2 sums = block_sum2(make_float2(s1.x + s1.y, s2.x + s2.y), red_m);
      const float m1 = sums.x / D;
      const float mu = K + m1;
      const float rs = rsqrtf(fmaxf(fmaf(-m1, m1, sums.y / D), 0.0f) + p.eps);
      const float2 rs2 = make_float2(rs, rs);
      const float2 nmu = make_float2(-mu, -mu);  // (x - mu) r: exactly 0 where x equals the mean
      if (!kBwd) {
#pragma unroll
        for (int i = 0; i < kV; ++i) {
          const int v = t + i * kThreads;
          if (v < nvec) {
            uint4 o;
            uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 xh = fmul2(fadd2(xv[i][e], nmu), rs2);
              const float2 yy = ffma2(xh, mod[i][e], sh[i][e]);
              w[e] = pack_bf16x2(yy.x, yy.y);
            }
            reinterpret_cast<uint4*>(p.out + r * D)[v] = o;
          }
        }
        if (t == 0) {
          if (p.mean) p.mean[r] = mu;
          if (p.rstd) p.rstd[r] = rs;
        }
      } else {
        const float* scale_row = p.scale + static_cast<size_t>(b) * D;
        float2 sg = make_float2(0.f, 0.f), sgx = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kV; ++i) {
          const int v = t + i * kThreads;
          if (v < nvec) {
            float2 dv[4], sc[4];
            unpack8x2(reinterpret_cast<const uint4*>(src + RB)[v], dv);
            load_scale(scale_row + v * 8, sc);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 xh = fmul2(fadd2(xv[i][e], nmu), rs2);
              xv[i][e] = xh;
              const float2 gg = ffma2(dv[e], sc[e], dv[e]);  // dy (1 + scale)
              sg = fadd2(sg, gg);
              sgx = ffma2(gg, xh, sgx);
              acc_s[i][e] = fadd2(acc_s[i][e], dv[e]);
              acc_c[i][e] = ffma2(dv[e], xh, acc_c[i][e]);
            }
          }
        }
        const float2 m = block_sum2(make_float2(sg.x + sg.y, sgx.x + sgx.y), red);
        const float2 nmg = make_float2(-m.x / D, -m.x / D), nmgx = make_float2(-m.y / D, -m.y / D);
#pragma unroll
        for (int i = 0; i < kV; ++i) {
          const int v = t + i * kThreads;
          if (v < nvec) {
            float2 dv[4], sc[4];  // dy again from shared memory: g = dy (1 + scale)
            unpack8x2(reinterpret_cast<const uint4*>(src + RB)[v], dv);
            load_scale(scale_row + v * 8, sc);
            uint4 o;
            uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 gg = ffma2(dv[e], sc[e], dv[e]);
              const float2 dd = fmul2(fadd2(ffma2(xv[i][e], nmgx, gg), nmg), rs2);
              w[e] = pack_bf16x2(dd.x, dd.y);
            }
            reinterpret_cast<uint4*>(p.out + r * D)[v] = o;
          }
        }
      }
      // every thread is done with this stage and with the reduction slots
      __syncthreads();
      if (t == 0) issue_next();
    }
    if (!alive) break;
    if (kBwd) {
      // this item's partial modulation gradients, coalesced along the features
      float* ps = p.part + static_cast<size_t>(item) * D;
      float* pc = p.part + (static_cast<size_t>(p.items) + item) * D;
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = t + i * kThreads;
        if (v < nvec) {
          reinterpret_cast<float4*>(ps + v * 8)[0] = make_float4(acc_s[i][0].x, acc_s[i][0].y, acc_s[i][1].x, acc_s[i][1].y);
          reinterpret_cast<float4*>(ps + v * 8)[1] = make_float4(acc_s[i][2].x, acc_s[i][2].y, acc_s[i][3].x, acc_s[i][3].y);
          reinterpret_cast<float4*>(pc + v * 8)[0] = make_float4(acc_c[i][0].x, acc_c[i][0].y, acc_c[i][1].x, acc_c[i][1].y);
          reinterpret_cast<float4*>(pc + v * 8)[1] = make_float4(acc_c[i][2].x, acc_c[i][2].y, acc_c[i][3].x, acc_c[i][3].y);
        }
      }
    }
  }
  // copies still in flight land before the CTA leaves
  if (t == 0)
    for (uint32_t n = use_n; n < ld_n; ++n) mbar_drain(&full[n % kStages], (n / kStages) & 1, 100000000ull);
  __syncthreads();
}

// dshift[b, d] / dscale[b, d] = sum over the batch row's tiles, in tile order.
__global__ void __launch_bounds__(256) adaln_bwd_finalize(const float* __restrict__ part, int B, int D, int n_tiles,
                                                          float* __restrict__ dshift, float* __restrict__ dscale) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long bd = static_cast<long long>(B) * D;
  if (i >= 2 * bd) return;
  const bool is_scale = i >= bd;
  const long long j = is_scale ? i - bd : i;
  const int b = static_cast<int>(j / D), d = static_cast<int>(j % D);
  const float* src = part + (is_scale ? static_cast<size_t>(B) * n_tiles * D : 0) + static_cast<size_t>(b) * n_tiles * D + d;
  float s = 0.0f;
  for (int tl = 0; tl < n_tiles; ++tl) s += src[static_cast<size_t>(tl) * D];
  (is_scale ? dscale : dshift)[j] = s;
}

// stages per CTA: at most ~96 KB of shared memory with two CTAs per SM,
// ~192 KB with one
template <bool kBwd>
constexpr int stages_for(int kV) {
  return kBwd ? (kV <= 2 ? 6 : (kV == 3 ? 4 : 6)) : (kV <= 3 ? 6 : 5);
}

template <int kV, bool kBwd>
pvl_status launch_rows(const AdalnParams& p, cudaStream_t s, const char* who) {
  constexpr int kStages = stages_for<kBwd>(kV);
  const int smem = kStages * (kBwd ? 2 : 1) * row_bytes(p.D);
  pvl_status st = check_cuda(
      cudaFuncSetAttribute(adaln_kernel<kV, kBwd, kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem), who);
  if (st != PVL_OK) return st;
  const int sms = sm_count();
  if (sms <= 0) return fail(PVL_ERR_CUDA, "%s: no usable CUDA device", who);
  const long long cap = static_cast<long long>(ctas_per_sm<kV, kBwd>()) * sms;
  const long long grid = p.items < cap ? p.items : cap;
  adaln_kernel<kV, kBwd, kStages><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p);
  return check_cuda(cudaGetLastError(), who);
}

template <bool kBwd>
pvl_status dispatch(const AdalnParams& p, cudaStream_t s, const char* who) {
  const int vec_per_thread = (p.D / 8 + kThreads - 1) / kThreads;
  if (vec_per_thread <= 1) return launch_rows<1, kBwd>(p, s, who);
  if (vec_per_thread <= 2) return launch_rows<2, kBwd>(p, s, who);
  if (vec_per_thread <= 3) return launch_rows<3, kBwd>(p, s, who);
  return launch_rows<4, kBwd>(p, s, who);
}

pvl_status validate(const char* who, const void* const* ptrs, int nptrs, int B, int N, int D, float eps) {
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i]) return fail(PVL_ERR_INVALID_ARG, "%s: pointer argument %d is null", who, i);
  if (B < 1 || N < 1 || D < 1) return fail(PVL_ERR_INVALID_ARG, "%s: B, N and D must be >= 1", who);
  if (!(eps >= 0.0f) || !(eps < 1e30f)) return fail(PVL_ERR_INVALID_ARG, "%s: eps must be >= 0 and finite", who);
  if (D % 8 != 0 || D > kMaxD)
    return fail(PVL_ERR_UNSUPPORTED, "%s: D = %d (supported: multiples of 8 up to %d)", who, D, kMaxD);
  if (static_cast<long long>(B) * N * D >= (1ll << 40)) return fail(PVL_ERR_UNSUPPORTED, "%s: tensor too large", who);
  for (int i = 0; i < nptrs; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0)
      return fail(PVL_ERR_UNSUPPORTED, "%s: pointer argument %d is not 16-byte aligned", who, i);
  return PVL_OK;
}

int n_tiles_of(int N) { return (N + kRowsPerTile - 1) / kRowsPerTile; }

}  // namespace
}  // namespace pvl

using namespace pvl;

extern "C" pvl_status adaln_fwd(const pvl_bf16* x, const float* shift, const float* scale, int B, int N, int D,
                                float eps, pvl_bf16* y, float* mean, float* rstd, pvl_stream_t stream) {
  const void* ptrs[] = {x, shift, scale, y};
  pvl_status st = validate("adaln_fwd", ptrs, 4, B, N, D, eps);
  if (st != PVL_OK) return st;
  if ((mean && reinterpret_cast<uintptr_t>(mean) % 4) || (rstd && reinterpret_cast<uintptr_t>(rstd) % 4))
    return fail(PVL_ERR_UNSUPPORTED, "adaln_fwd: mean / rstd must be 4-byte aligned");
  DeviceError* err = device_error_record();
  if (!err) return fail(PVL_ERR_CUDA, "adaln_fwd: no usable CUDA device");
  AdalnParams p{};
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.shift = shift;
  p.scale = scale;
  p.out = reinterpret_cast<__nv_bfloat16*>(y);
  p.mean = mean;
  p.rstd = rstd;
  p.err = err;
  p.B = B;
  p.N = N;
  p.D = D;
  p.items = static_cast<long long>(B) * N;
  p.eps = eps;
  p.timeout_ns = kDefaultTimeoutNs;
  return dispatch<false>(p, reinterpret_cast<cudaStream_t>(stream), "adaln_fwd launch");
}

extern "C" size_t adaln_bwd_ws_bytes(int B, int N, int D) {
  if (B < 1 || N < 1 || D < 1) return 0;
  return 2ull * B * n_tiles_of(N) * D * sizeof(float);
}

extern "C" pvl_status adaln_bwd(const pvl_bf16* x, const float* scale, const pvl_bf16* dy, int B, int N, int D,
                                float eps, pvl_bf16* dx, float* dshift, float* dscale, void* ws, size_t ws_bytes,
                                pvl_stream_t stream) {
  const void* ptrs[] = {x, scale, dy, dx, dshift, dscale, ws};
  pvl_status st = validate("adaln_bwd", ptrs, 7, B, N, D, eps);
  if (st != PVL_OK) return st;
  if (ws_bytes < adaln_bwd_ws_bytes(B, N, D))
    return fail(PVL_ERR_INVALID_ARG, "adaln_bwd: workspace %zu bytes < %zu needed", ws_bytes,
                adaln_bwd_ws_bytes(B, N, D));
  DeviceError* err = device_error_record();
  if (!err) return fail(PVL_ERR_CUDA, "adaln_bwd: no usable CUDA device");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  AdalnParams p{};
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.dy = reinterpret_cast<const __nv_bfloat16*>(dy);
  p.scale = scale;
  p.out = reinterpret_cast<__nv_bfloat16*>(dx);
  p.part = static_cast<float*>(ws);
  p.err = err;
  p.B = B;
  p.N = N;
  p.D = D;
  p.n_tiles = n_tiles_of(N);
  p.items = static_cast<long long>(B) * p.n_tiles;
  p.eps = eps;
  p.timeout_ns = kDefaultTimeoutNs;
  st = dispatch<true>(p, s, "adaln_bwd launch");
  if (st != PVL_OK) return st;
  const long long n = 2ll * B * D;
  adaln_bwd_finalize<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(p.part, B, D, p.n_tiles, dshift, dscale);
  return check_cuda(cudaGetLastError(), "adaln_bwd finalize launch");
}
