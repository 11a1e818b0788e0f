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
//   - persistent CTAs walk rows, each sized to the row: its threads own the
//     row's 8-wide feature groups evenly (one or two per thread, 320
//     threads at D = 5120), as many CTAs per SM as registers allow; thread 0
//     streams the rows (x, and dy backward) into a ring of shared-memory
//     stages with bulk asynchronous copies, so several rows are in flight
//     without holding them in registers;
//   - the CTA works on one row at a time: each thread owns the same feature
//     groups of every row; row sums go through a warp shuffle and a block
//     reduction (two-level, as the page describes), and the statistics never
//     leave the chip; the modulation is applied on the way out.  The barrier
//     that opens a row also frees the previous row's stage;
//   - the rows are split evenly among the CTAs in contiguous ranges;
//     backward, each CTA accumulates dshift / dscale over its rows of one
//     batch row in the registers of the threads that own each feature (the
//     sequence-direction reduction of the page's D-tile scheme, with
//     coalesced reads along the features) and writes one partial sum per
//     batch row it meets; a small kernel adds the partials per batch row in
//     a fixed order (deterministic).
// Every wait is bounded; on expiry the CTA records the failure, waits for
// its copies in flight and returns.
#include <cuda_runtime.h>

#include "pvl_device.cuh"

namespace pvl {
namespace {

constexpr int kMaxThreads = 512;
constexpr int kMaxWarps = kMaxThreads / 32;
constexpr int kMaxStages = 8;
constexpr int kMaxCtas = 2048;    // CTAs per launch at most (bounds the partial-sum slots)
constexpr int kMaxD = 8192;

enum AdalnSite : uint32_t { kSiteRowFull = 41 };

// Stage bytes of one row of D bf16, rounded up to 128 bytes.
__host__ __device__ constexpr int row_bytes(int D) { return ((D * 2 + 127) / 128) * 128; }

// CTA-wide sums of kN values (2 or 4), the same in every thread.  Inside a
// warp the values are reduce-scattered (each halving step sends half of the
// remaining values), so lane group q = lane / (32 / kN) ends with value q;
// one lane per group stores it in red[warp * kN + q].  After the barrier
// each warp reads the table with one lane per entry and sums over the warps
// with xor shuffles.  `red` holds kMaxWarps * kN floats and is not written
// again before every thread has passed the caller's next __syncthreads.
// Every thread returns the same bits (the order of the additions is fixed).
template <int kN>
__device__ __forceinline__ void block_sum(float (&a)[kN], float* red, int nwarps) {
  static_assert(kN == 2 || kN == 4, "2 or 4 values");
  const int lane = threadIdx.x & 31;
  float kept;
  if (kN == 4) {
    const bool hi = lane & 16;
    float k0 = hi ? a[2] : a[0], k1 = hi ? a[3] : a[1];
    const float s0 = hi ? a[0] : a[2], s1 = hi ? a[1] : a[3];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    const bool h8 = lane & 8;
    kept = h8 ? k1 : k0;
    kept += __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
  } else {
    const bool hi = lane & 16;
    kept = hi ? a[1] : a[0];
    kept += __shfl_xor_sync(0xffffffffu, hi ? a[0] : a[1], 16);
    kept += __shfl_xor_sync(0xffffffffu, kept, 8);
  }
  kept += __shfl_xor_sync(0xffffffffu, kept, 4);
  kept += __shfl_xor_sync(0xffffffffu, kept, 2);
  kept += __shfl_xor_sync(0xffffffffu, kept, 1);
  constexpr int kGroup = 32 / kN;
  if ((lane & (kGroup - 1)) == 0) red[(threadIdx.x >> 5) * kN + lane / kGroup] = kept;
  __syncthreads();
  // entry lane (and lane + 32) of the table: warp lane / kN, value lane % kN
  const int n = nwarps * kN;
  float t = lane < n ? red[lane] : 0.0f;
  if (n > 32 && lane + 32 < n) t += red[lane + 32];
#pragma unroll
  for (int o = kN; o < 32; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
#pragma unroll
  for (int q = 0; q < kN; ++q) a[q] = __shfl_sync(0xffffffffu, t, q);
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
  float* part;              // backward: [2][n_slots][D] partial sums
  DeviceError* err;
  int B, N, D;
  long long rows;           // B * N
  long long rows_per_cta;   // CTA c takes rows [c R, (c + 1) R) of the B * N
  int n_slots;              // partial-sum slots: kMaxCtas (at most B * N) + B - 1
  int stages;               // shared-memory row stages, 2..kMaxStages
  float eps;
  uint64_t timeout_ns;
};

// Backward rows keep their values in registers between the two passes at
// one or two feature groups per thread and re-read them from shared memory
// at more (where the per-feature accumulators take the registers).
template <int kV>
__host__ __device__ constexpr bool holds_row() {
  return kV <= 2;
}

// Register budget per thread for kV feature groups per thread.
template <int kV, bool kBwd>
constexpr int max_regs() {
  return kBwd ? (kV == 1 ? 64 : (kV == 2 ? 96 : 128)) : (kV == 1 ? 48 : (kV == 2 ? 64 : (kV == 3 ? 96 : 128)));
}

// CTA c takes the rows [c R, (c + 1) R) of the B * N (the last CTA fewer):
// every CTA gets the same number of rows to within one.  Its rows split into
// segments at batch-row boundaries; every thread owns the feature groups
// t, t + blockDim.x, ... (kV of them at most) of every row.  Backward, a
// segment's dshift / dscale sums go to partial-sum slot c + b (b its batch
// row; no two (CTA, batch row) pairs that meet share a slot).
template <int kV, bool kBwd>
__global__ void __maxnreg__((max_regs<kV, kBwd>())) adaln_kernel(const AdalnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ float red[kMaxWarps * 4];
  __shared__ int abort_s;
  constexpr int kTensors = kBwd ? 2 : 1;
  constexpr bool kHold = !kBwd || holds_row<kV>();
  const int D = p.D;
  const int RB = row_bytes(D);
  const int nvec = D / 8;
  const int t = threadIdx.x;
  const int nthr = blockDim.x;
  const int nwarps = nthr / 32;
  const int S = p.stages;
  const float inv_d = 1.0f / static_cast<float>(D);
  const KernelCtl ctl{p.err, &abort_s, p.timeout_ns};
  const long long r_begin = static_cast<long long>(blockIdx.x) * p.rows_per_cta;
  const long long r_end = min(r_begin + p.rows_per_cta, p.rows);

  if (t == 0) {
    abort_s = 0;
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // Producer (thread 0): the CTA's rows in order, x and dy of a row into one
  // stage.
  long long ld_r = r_begin;
  uint32_t ld_n = 0;  // rows issued
  int ld_st = 0;
  auto issue_next = [&]() {
    if (ld_r >= r_end) return;
    uint8_t* dst = smem + static_cast<size_t>(ld_st) * kTensors * RB;
    mbar_arrive_expect_tx(&full[ld_st], kTensors * D * 2);
    bulk_load(dst, p.x + ld_r * D, D * 2, &full[ld_st]);
    if (kBwd) bulk_load(dst + RB, p.dy + ld_r * D, D * 2, &full[ld_st]);
    ++ld_r;
    ++ld_n;
    if (++ld_st == S) ld_st = 0;
  };
  if (t == 0)
    for (int s = 0; s < S; ++s) issue_next();

  uint32_t use_n = 0;  // rows consumed
  int use_st = 0;
  uint32_t use_ph = 0;
  bool alive = true;
  // per-thread modulation of the owned feature groups (forward), loaded per
  // segment
  float2 mod[kBwd ? 1 : kV][4];  // 1 + scale
  float2 sh[kBwd ? 1 : kV][4];   // shift
  int b = r_begin < r_end ? static_cast<int>(r_begin / p.N) : p.B;
  for (long long r = r_begin; r < r_end && alive; ++b) {
    const long long seg_end = min(r_end, static_cast<long long>(b + 1) * p.N);
    float2 acc_s[kBwd ? kV : 1][4], acc_c[kBwd ? kV : 1][4];  // dshift, dscale partials
#pragma unroll
    for (int i = 0; i < kV; ++i) {
      if (kBwd) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_s[i][e] = acc_c[i][e] = make_float2(0.f, 0.f);
      } else {
        const int v = t + i * nthr;
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
    }
    const float* scale_row = p.scale + static_cast<size_t>(b) * D;
    for (; r < seg_end; ++r) {
      if (!__syncthreads_and(mbar_wait(&full[use_st], use_ph, ctl, kSiteRowFull))) {
        alive = false;
        break;
      }
      // Every thread is past the previous row: its stage and the reduction
      // table are free, so the stage is refilled now.
      if (t == 0 && use_n > 0) issue_next();
      const uint8_t* src = smem + static_cast<size_t>(use_st) * kTensors * RB;
      // Row statistics from shifted sums: with K the row's first element and
      // d = x - K, S1 = sum d, S2 = sum d^2, m1 = S1/D, mean = K + m1,
      // var = S2/D - m1^2 and xh = (d - m1) r.  K is a sample of the row, so
      // m1^2 stays within a factor ~D of the variance even for an outlier K:
      // the cancellation costs at most ~D * 2^-24 relative, far below bf16's
      // 2^-9.  d is exact (two bf16 values), so xh = 0 exactly where x equals
      // the mean.  Backward, the same pass sums g = dy (1 + scale) and g d:
      // sum g xh = r (sum g d - m1 sum g), one reduction per row.
      const float K = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(src)) << 16);
      const float2 nk = make_float2(-K, -K);
      float2 xv[kHold ? kV : 1][4];  // d
      float2 dv[kBwd && kHold ? kV : 1][4];
      float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
      float2 sg = make_float2(0.f, 0.f), sgd = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = t + i * nthr;
        if (v < nvec) {
          float2 xr[4], dr[4], sc[4];
          unpack8x2(reinterpret_cast<const uint4*>(src)[v], xr);
          if (kBwd) {
            unpack8x2(reinterpret_cast<const uint4*>(src + RB)[v], dr);
            load_scale(scale_row + v * 8, sc);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 d = fadd2(xr[e], nk);
            s1 = fadd2(s1, d);
            s2 = ffma2(d, d, s2);
            if (kHold) xv[kHold ? i : 0][e] = d;
            if (kBwd) {
              const float2 g = ffma2(dr[e], sc[e], dr[e]);
              sg = fadd2(sg, g);
              sgd = ffma2(g, d, sgd);
              acc_s[kBwd ? i : 0][e] = fadd2(acc_s[kBwd ? i : 0][e], dr[e]);
              if (kHold) dv[kBwd && kHold ? i : 0][e] = dr[e];
            }
          }
        }
      }
      float m1, rs;
      float a = 0.f, c = 0.f;  // backward: dx = g r + xh a + c
      if (!kBwd) {
        float sums[2] = {s1.x + s1.y, s2.x + s2.y};
        block_sum<2>(sums, red, nwarps);
        m1 = sums[0] * inv_d;
        rs = rsqrtf(fmaxf(fmaf(-m1, m1, sums[1] * inv_d), 0.0f) + p.eps);
      } else {
        float sums[4] = {s1.x + s1.y, s2.x + s2.y, sg.x + sg.y, sgd.x + sgd.y};
        block_sum<4>(sums, red, nwarps);
        m1 = sums[0] * inv_d;
        rs = rsqrtf(fmaxf(fmaf(-m1, m1, sums[1] * inv_d), 0.0f) + p.eps);
        const float mean_g = sums[2] * inv_d;
        const float mean_gxh = rs * fmaf(-m1, sums[2], sums[3]) * inv_d;
        a = -rs * mean_gxh;
        c = -rs * mean_g;
      }
      const float2 rs2 = make_float2(rs, rs);
      const float2 nm1 = make_float2(-m1, -m1);
      const float2 a2 = make_float2(a, a), c2 = make_float2(c, c);
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = t + i * nthr;
        if (v < nvec) {
          float2 d[4], dr[4];
          if (kHold) {
#pragma unroll
            for (int e = 0; e < 4; ++e) d[e] = xv[kHold ? i : 0][e];
          } else {
            unpack8x2(reinterpret_cast<const uint4*>(src)[v], d);
#pragma unroll
            for (int e = 0; e < 4; ++e) d[e] = fadd2(d[e], nk);
          }
          if (kBwd) {
            if (kHold) {
#pragma unroll
              for (int e = 0; e < 4; ++e) dr[e] = dv[kBwd && kHold ? i : 0][e];
            } else {
              unpack8x2(reinterpret_cast<const uint4*>(src + RB)[v], dr);
            }
          }
          float2 sc[4];
          if (kBwd) load_scale(scale_row + v * 8, sc);
          uint4 o;
          uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 xh = fmul2(fadd2(d[e], nm1), rs2);
            float2 out;
            if (!kBwd) {
              out = ffma2(xh, mod[kBwd ? 0 : i][e], sh[kBwd ? 0 : i][e]);
            } else {
              const float2 g = ffma2(dr[e], sc[e], dr[e]);
              out = ffma2(g, rs2, ffma2(xh, a2, c2));
              acc_c[kBwd ? i : 0][e] = ffma2(dr[e], xh, acc_c[kBwd ? i : 0][e]);
            }
            w[e] = pack_bf16x2(out.x, out.y);
          }
          reinterpret_cast<uint4*>(p.out + r * D)[v] = o;
        }
      }
      if (!kBwd && t == 0) {
        if (p.mean) p.mean[r] = K + m1;
        if (p.rstd) p.rstd[r] = rs;
      }
      ++use_n;
      if (++use_st == S) {
        use_st = 0;
        use_ph ^= 1u;
      }
    }
    if (!alive) break;
    if (kBwd) {
      // the segment's partial modulation gradients, coalesced along the features
      const size_t slot = static_cast<size_t>(blockIdx.x) + b;
      float* ps = p.part + slot * D;
      float* pc = p.part + (static_cast<size_t>(p.n_slots) + slot) * D;
#pragma unroll
      for (int i = 0; i < kV; ++i) {
        const int v = t + i * nthr;
        if (v < nvec) {
          const int j = kBwd ? i : 0;
          reinterpret_cast<float4*>(ps + v * 8)[0] = make_float4(acc_s[j][0].x, acc_s[j][0].y, acc_s[j][1].x, acc_s[j][1].y);
          reinterpret_cast<float4*>(ps + v * 8)[1] = make_float4(acc_s[j][2].x, acc_s[j][2].y, acc_s[j][3].x, acc_s[j][3].y);
          reinterpret_cast<float4*>(pc + v * 8)[0] = make_float4(acc_c[j][0].x, acc_c[j][0].y, acc_c[j][1].x, acc_c[j][1].y);
          reinterpret_cast<float4*>(pc + v * 8)[1] = make_float4(acc_c[j][2].x, acc_c[j][2].y, acc_c[j][3].x, acc_c[j][3].y);
        }
      }
    }
  }
  // copies still in flight land before the CTA leaves
  __syncthreads();
  if (t == 0)
    for (uint32_t n = use_n; n < ld_n; ++n) mbar_drain(&full[n % S], (n / S) & 1, 100000000ull);
  __syncthreads();
}

// dshift[b, d] / dscale[b, d] = sum of the slots c + b of the CTAs c that
// met batch row b, in CTA order.  A CTA (blockIdx.x: batch row, then dshift
// / dscale; blockIdx.y: 128-feature block) has lane l of warp w add the
// float4 at features 4l.. of CTAs c0 + w, c0 + w + 8, ... (four loads in
// flight), then warp 0 adds the eight warps' sums in warp order.  The order
// of every addition is fixed: the result is deterministic.
constexpr int kFinThreads = 256;
__global__ void __launch_bounds__(kFinThreads) adaln_bwd_finalize(const float* __restrict__ part, int B, int N, int D,
                                                                  long long rows_per_cta, int n_slots,
                                                                  float* __restrict__ dshift,
                                                                  float* __restrict__ dscale) {
  __shared__ float4 acc[kFinThreads / 32][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int d = blockIdx.y * 128 + lane * 4;
  const int b = static_cast<int>(blockIdx.x % B);
  const bool is_scale = static_cast<int>(blockIdx.x) >= B;
  const int c0 = static_cast<int>(static_cast<long long>(b) * N / rows_per_cta);
  const int c1 = static_cast<int>((static_cast<long long>(b + 1) * N - 1) / rows_per_cta);  // inclusive
  const int n = c1 - c0 + 1;
  const float* src = part + (is_scale ? static_cast<size_t>(n_slots) * D : 0) + (static_cast<size_t>(c0) + b) * D + d;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (d < D) {
    constexpr int kW = kFinThreads / 32;
    int i = w;
    for (; i + 3 * kW < n; i += 4 * kW) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(i + u * kW) * D));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        s.x += v[u].x;
        s.y += v[u].y;
        s.z += v[u].z;
        s.w += v[u].w;
      }
    }
    for (; i < n; i += kW) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(i) * D));
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
  }
  acc[w][lane] = s;
  __syncthreads();
  if (w == 0 && d < D) {
    float4 t = acc[0][lane];
#pragma unroll
    for (int i = 1; i < kFinThreads / 32; ++i) {
      const float4 v = acc[i][lane];
      t.x += v.x;
      t.y += v.y;
      t.z += v.z;
      t.w += v.w;
    }
    float* dst = (is_scale ? dscale : dshift) + static_cast<size_t>(b) * D + d;
    *reinterpret_cast<float4*>(dst) = t;
  }
}

// Launch shape: the CTA's threads cover the row's 8-wide feature groups
// evenly (kV groups per thread, rounded to whole warps); as many CTAs per SM
// as registers allow; the shared memory of the SM split among them as row
// stages (2 to kMaxStages).
template <int kV, bool kBwd>
pvl_status launch_rows(AdalnParams p, cudaStream_t s, const char* who, long long* rows_per_cta) {
  const int nvec = p.D / 8;
  const int threads = ((nvec + kV - 1) / kV + 31) / 32 * 32;
  const int stage_bytes = (kBwd ? 2 : 1) * row_bytes(p.D);
  int dev = 0, sms = 0, smem_sm = 0;
  pvl_status st = check_cuda(cudaGetDevice(&dev), who);
  if (st == PVL_OK) st = check_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), who);
  if (st == PVL_OK)
    st = check_cuda(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev), who);
  int occ = 0;
  if (st == PVL_OK)
    st = check_cuda(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, adaln_kernel<kV, kBwd>, threads, 0), who);
  if (st != PVL_OK) return st;
  if (sms <= 0 || occ <= 0) return fail(PVL_ERR_CUDA, "%s: no usable CUDA device", who);
  constexpr int kReserve = 2048;  // per CTA: the system's share and the static shared memory
  int stages = 0;
  for (; occ >= 1; --occ) {
    stages = (smem_sm / occ - kReserve) / stage_bytes;
    if (stages >= 2) break;
  }
  if (occ < 1) return fail(PVL_ERR_UNSUPPORTED, "%s: D = %d does not fit in shared memory", who, p.D);
  p.stages = stages < kMaxStages ? stages : kMaxStages;
  const int smem = p.stages * stage_bytes;
  st = check_cuda(cudaFuncSetAttribute(adaln_kernel<kV, kBwd>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem), who);
  if (st != PVL_OK) return st;
  long long grid = static_cast<long long>(occ) * sms;
  if (grid > kMaxCtas) grid = kMaxCtas;
  if (grid > p.rows) grid = p.rows;
  p.rows_per_cta = (p.rows + grid - 1) / grid;
  grid = (p.rows + p.rows_per_cta - 1) / p.rows_per_cta;
  *rows_per_cta = p.rows_per_cta;
  adaln_kernel<kV, kBwd><<<static_cast<unsigned>(grid), threads, smem, s>>>(p);
  return check_cuda(cudaGetLastError(), who);
}

// Four feature groups per thread (a few warps per row: the per-row barrier
// and reduction are paid by fewer warps, and more CTAs share an SM); fewer
// only where that would leave less than one warp per row.
template <bool kBwd>
pvl_status dispatch(const AdalnParams& p, cudaStream_t s, const char* who, long long* rows_per_cta) {
  const int nvec = p.D / 8;
  if (nvec >= 4 * 32) return launch_rows<4, kBwd>(p, s, who, rows_per_cta);
  if (nvec >= 2 * 32) return launch_rows<2, kBwd>(p, s, who, rows_per_cta);
  return launch_rows<1, kBwd>(p, s, who, rows_per_cta);
}

pvl_status validate(const char* who, const void* const* ptrs, int nptrs, int B, int N, int D, float eps) {
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i]) return fail(PVL_ERR_INVALID_ARG, "%s: pointer argument %d is null", who, i);
  if (B < 1 || N < 1 || D < 1) return fail(PVL_ERR_INVALID_ARG, "%s: B, N and D must be >= 1", who);
  if (!(eps >= 0.0f) || !(eps < 1e30f)) return fail(PVL_ERR_INVALID_ARG, "%s: eps must be >= 0 and finite", who);
  if (D % 8 != 0 || D > kMaxD)
    return fail(PVL_ERR_UNSUPPORTED, "%s: D = %d (supported: multiples of 8 up to %d)", who, D, kMaxD);
  if (static_cast<long long>(B) * N * D >= (1ll << 40) || N > (1 << 30) || B > (1 << 30))
    return fail(PVL_ERR_UNSUPPORTED, "%s: tensor too large", who);
  for (int i = 0; i < nptrs; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0)
      return fail(PVL_ERR_UNSUPPORTED, "%s: pointer argument %d is not 16-byte aligned", who, i);
  return PVL_OK;
}

// partial-sum slots of the backward: one per (CTA, batch row) pair that meets
int slots_of(int B, int N) {
  const long long rows = static_cast<long long>(B) * N;
  return static_cast<int>((rows < kMaxCtas ? rows : kMaxCtas) + B - 1);
}

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
  p.rows = static_cast<long long>(B) * N;
  p.eps = eps;
  p.timeout_ns = kDefaultTimeoutNs;
  long long rows_per_cta = 0;
  return dispatch<false>(p, reinterpret_cast<cudaStream_t>(stream), "adaln_fwd launch", &rows_per_cta);
}

extern "C" size_t adaln_bwd_ws_bytes(int B, int N, int D) {
  if (B < 1 || N < 1 || D < 1) return 0;
  return 2ull * slots_of(B, N) * D * sizeof(float);
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
  p.rows = static_cast<long long>(B) * N;
  p.n_slots = slots_of(B, N);
  p.eps = eps;
  p.timeout_ns = kDefaultTimeoutNs;
  long long rows_per_cta = 0;
  st = dispatch<true>(p, s, "adaln_bwd launch", &rows_per_cta);
  if (st != PVL_OK) return st;
  const dim3 fin_grid(2 * B, (D + 127) / 128);
  adaln_bwd_finalize<<<fin_grid, kFinThreads, 0, s>>>(p.part, B, N, D, rows_per_cta, p.n_slots, dshift, dscale);
  return check_cuda(cudaGetLastError(), "adaln_bwd finalize launch");
}
