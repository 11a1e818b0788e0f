// masked_attn_fwd: seq_id-masked softmax attention, forward, for sm_103a.
//
// What it computes ("furniture_packing_variable_length", attention masking;
// "lingbot_va_attn_profiling", doc_id[q] == doc_id[k] mask): for every batch
// row b, head h and query i with s_i >= 0,
//   O_i = sum_{j: s_j = s_i} softmax_j(scale * <q_i, k_j>) v_j,
//   LSE_i = log sum_{j: s_j = s_i} exp(scale * <q_i, k_j>);
// rows with s_i = -1 get O_i = 0 and LSE_i = -inf.
//
// Design.  One persistent CTA per SM walks work items (b, query tile, head) in
// the tile map's longest-first order, round-robin over CTAs.  Per item only
// the key tiles the tile map lists as non-empty are touched, FULL ones first
// (no per-element mask), then PARTIAL ones (mask from the key seq_ids).
//   warp 4      TMA producer: Q tile once per item, K/V tiles into a 2-stage
//               ring; for PARTIAL tiles it also stages the key seq_ids.
//   warp 5      owns TMEM (512 columns) and issues tcgen05.mma from one
//               thread: S = Q K^T into one of two TMEM S buffers (so S_{j+1}
//               runs while the softmax works on S_j), then O += P V.
//   warps 0-3   softmax: thread t owns query row t (TMEM lane t), loads its S
//               row, applies the mask on PARTIAL tiles, keeps a running max
//               and sum, writes P (bf16) to shared memory in the 128-byte
//               swizzled layout the MMA reads, and rescales O in TMEM only
//               when its running max grows by more than 2^8 (the stale max
//               bounds every P by 256, and the final division uses the same
//               max, so the result is unchanged).  The epilogue divides by
//               the row sum and writes O (bf16) and LSE (fp32).
// Every wait is bounded; on expiry the CTA records the failure, drains its
// outstanding copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pvl_device.cuh"

namespace pvl {
namespace {

constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;   // O accumulator columns [256, 256 + D)
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum FwdSite : uint32_t {
  kSiteQEmpty = 1, kSiteKvEmpty, kSiteQFull, kSiteKFull, kSiteSFree, kSitePFull, kSiteVFull, kSiteOFree,
  kSiteSFull, kSitePvDone, kSiteKseq, kSiteFinal
};

template <int D>
struct FwdSmem {
  static constexpr int kTile = 128 * D * 2;  // one 128 x D bf16 tile (D / 64 swizzled 16 KB blocks)
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kP = kV + kStages * kTile;  // 128 x 128 bf16 probabilities
  static constexpr int kEnd = kP + 128 * 128 * 2;
  // 1 KB alignment slack; never below 120 KB so two CTAs can not share an SM
  // (each CTA allocates all 512 TMEM columns).
  static constexpr int kBytes = (kEnd + 1024) > 120 * 1024 ? (kEnd + 1024) : 120 * 1024;
};

struct FwdParams {
  const int32_t* seq_id;
  const int32_t* header;
  const int32_t* row_count;
  const int32_t* row_full;
  const int32_t* row_list;
  const int32_t* q_order;
  __nv_bfloat16* o;
  float* lse;
  DeviceError* err;
  int B, L, H, nT;
  long long total_items;
  float scale_log2;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_base, int kk) {
  // K-major operand with 64-element (128 B) swizzled rows: 16-element K steps
  // advance 32 B inside a block, blocks of 64 are 128 rows * 128 B apart.
  return sdesc_sw128(tile_base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}

__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile_base, int kk) {
  // MN-major operand stored as K rows of 64 MN elements: a 16-row K step is
  // 2 KB; the second 64-wide MN block sits 16 KB further (LBO).
  return sdesc_sw128(tile_base + kk * 2048, 16384, 1024);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  using S = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q_full, bar_q_empty, bar_p_full, bar_pv_done, bar_o_free, bar_final;
  __shared__ uint64_t bar_k_full[kStages], bar_v_full[kStages], bar_kv_empty[kStages];
  __shared__ uint64_t bar_s_full[2], bar_s_free[2];
  __shared__ int32_t kseq_s[kStages][128];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nT = p.nT;

  // The tile map must describe this call; otherwise do nothing.
  {
    const int32_t* hd = p.header;
    const bool ok = hd[0] == kTileMapMagic && hd[1] == kTileMapVersion && hd[2] == p.B && hd[3] == p.L &&
                    hd[4] == 128 && hd[5] == 128;
    if (!ok) {
      if (threadIdx.x == 0 && atomicCAS(&p.err->code, 0u, kDevErrTileMap) == 0u) p.err->block = blockIdx.x;
      return;
    }
  }

  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 1);
    mbar_init(&bar_p_full, 128);
    mbar_init(&bar_pv_done, 1);
    mbar_init(&bar_o_free, 128);
    mbar_init(&bar_final, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_s_free[s], 128);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_s, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = tmem_base_s;
  const KernelCtl ctl{p.err, &abort_s, p.timeout_ns};
  const uint32_t sQ = smem_u32(smem + S::kQ);
  const uint32_t sK0 = smem_u32(smem + S::kK);
  const uint32_t sV0 = smem_u32(smem + S::kV);
  const uint32_t sP = smem_u32(smem + S::kP);
  constexpr uint32_t kTileBytes = S::kTile;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    uint32_t kv_it = 0, q_it = 0;
    bool alive = true;
    for (long long w = blockIdx.x; w < p.total_items && alive; w += gridDim.x) {
      const int tile = p.q_order[w / p.H];
      const int h = static_cast<int>(w % p.H);
      const int b = tile / nT, qt = tile % nT;
      const int n = p.row_count[tile];
      if (n == 0) continue;
      const int nfull = p.row_full[tile];
      const int32_t* list = p.row_list + static_cast<size_t>(tile) * nT;
      bool ok = lane == 0 ? mbar_wait(&bar_q_empty, (q_it & 1) ^ 1, ctl, kSiteQEmpty) : true;
      if (!__shfl_sync(0xffffffffu, ok, 0)) { alive = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_q_full, kTileBytes);
#pragma unroll
        for (int s = 0; s < D / 64; ++s) tma_load_4d(smem + S::kQ + s * 16384, &tmap_q, &bar_q_full, s * 64, h, qt * 128, b);
      }
      ++q_it;
      for (int j = 0; j < n; ++j, ++kv_it) {
        const int kt = list[j];
        const int st = kv_it % kStages;
        ok = lane == 0 ? mbar_wait(&bar_kv_empty[st], ((kv_it / kStages) & 1) ^ 1, ctl, kSiteKvEmpty) : true;
        if (!__shfl_sync(0xffffffffu, ok, 0)) { alive = false; break; }
        if (j >= nfull) {  // PARTIAL: stage the key seq_ids for the mask
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int c = lane * 4 + r;
            const int kpos = kt * 128 + c;
            kseq_s[st][c] = kpos < p.L ? p.seq_id[static_cast<size_t>(b) * p.L + kpos] : -1;
          }
        }
        __syncwarp();
        if (lane == 0) {
          uint8_t* kdst = smem + S::kK + st * kTileBytes;
          uint8_t* vdst = smem + S::kV + st * kTileBytes;
          mbar_arrive_expect_tx(&bar_k_full[st], kTileBytes);
#pragma unroll
          for (int s = 0; s < D / 64; ++s) tma_load_4d(kdst + s * 16384, &tmap_k, &bar_k_full[st], s * 64, h, kt * 128, b);
          mbar_arrive_expect_tx(&bar_v_full[st], kTileBytes);
#pragma unroll
          for (int s = 0; s < D / 64; ++s) tma_load_4d(vdst + s * 16384, &tmap_v, &bar_v_full[st], s * 64, h, kt * 128, b);
        }
        __syncwarp();
      }
    }
    if (abort_s && lane == 0) {
      // let copies still in flight land before the CTA leaves
      if (q_it > 0) mbar_drain(&bar_q_full, (q_it - 1) & 1, 100000000ull);
      for (uint32_t it = kv_it > kStages ? kv_it - kStages : 0; it < kv_it; ++it) {
        mbar_drain(&bar_k_full[it % kStages], (it / kStages) & 1, 100000000ull);
        mbar_drain(&bar_v_full[it % kStages], (it / kStages) & 1, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
    uint32_t kv_it = 0, q_it = 0, s_it = 0, p_it = 0, o_it = 0;
    bool alive = true;
    auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      bool ok = lane == 0 ? mbar_wait(bar, parity, ctl, site) : true;
      return __shfl_sync(0xffffffffu, ok, 0);
    };
    for (long long w = blockIdx.x; w < p.total_items && alive; w += gridDim.x) {
      const int tile = p.q_order[w / p.H];
      const int n = p.row_count[tile];
      if (n == 0) continue;
      if (!wait1(&bar_q_full, q_it & 1, kSiteQFull)) { alive = false; break; }
      ++q_it;
      const uint32_t kv_base = kv_it;
      // S_j = Q K_j^T into S buffer (s_it & 1)
      auto issue_s = [&](int j) -> bool {
        const uint32_t idx = kv_base + j;
        const int st = idx % kStages;
        if (!wait1(&bar_k_full[st], (idx / kStages) & 1, kSiteKFull)) return false;
        const uint32_t sb = s_it & 1;
        if (!wait1(&bar_s_free[sb], ((s_it >> 1) & 1) ^ 1, kSiteSFree)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kbase = sK0 + st * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + sb * 128, kmajor_desc(sQ, kk), kmajor_desc(kbase, kk), idesc_s, kk > 0 ? 1u : 0u);
          umma_commit(&bar_s_full[sb]);
        }
        __syncwarp();
        ++s_it;
        return true;
      };
      if (!issue_s(0)) { alive = false; break; }
      for (int j = 0; j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) { alive = false; break; }
        const uint32_t idx = kv_base + j;
        const int st = idx % kStages;
        if (!wait1(&bar_p_full, p_it & 1, kSitePFull)) { alive = false; break; }
        ++p_it;
        if (!wait1(&bar_v_full[st], (idx / kStages) & 1, kSiteVFull)) { alive = false; break; }
        if (j == 0) {
          if (!wait1(&bar_o_free, (o_it & 1) ^ 1, kSiteOFree)) { alive = false; break; }
          ++o_it;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vbase = sV0 + st * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss(tmem + kTmemO, kmajor_desc(sP, kk), mnmajor_desc(vbase, kk), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bar_pv_done);
          umma_commit(&bar_kv_empty[st]);
        }
        __syncwarp();
      }
      kv_it = kv_base + n;
      if (!alive) break;
      if (lane == 0) umma_commit(&bar_q_empty);
      __syncwarp();
    }
    // every MMA issued by this thread has finished before TMEM is released
    if (lane == 0) {
      umma_commit(&bar_final);
      mbar_drain(&bar_final, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int row = threadIdx.x;  // query row inside the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t s_it = 0, pv_it = 0, kv_it = 0;
    bool alive = true;
    auto waitw = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, site));
    };
    for (long long w = blockIdx.x; w < p.total_items && alive; w += gridDim.x) {
      const int tile = p.q_order[w / p.H];
      const int h = static_cast<int>(w % p.H);
      const int b = tile / nT, qt = tile % nT;
      const int n = p.row_count[tile];
      const int qpos = qt * 128 + row;
      const bool in_range = qpos < p.L;
      __nv_bfloat16* orow = p.o + ((static_cast<size_t>(b) * p.L + qpos) * p.H + h) * D;
      float* lse_out = p.lse + (static_cast<size_t>(b) * p.H + h) * p.L + qpos;
      if (n == 0) {  // no valid query in this tile
        if (in_range) {
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
          *lse_out = -INFINITY;
        }
        continue;
      }
      const int nfull = p.row_full[tile];
      const int my_seq = in_range ? p.seq_id[static_cast<size_t>(b) * p.L + qpos] : -1;
      float m_ref = -INFINITY;  // running max of scale*log2(e)*s
      float l = 0.0f;           // running sum of 2^(...) w.r.t. m_ref
      for (int j = 0; j < n; ++j, ++kv_it) {
        const uint32_t sb = s_it & 1;
        if (!waitw(&bar_s_full[sb], (s_it >> 1) & 1, kSiteSFull)) { alive = false; break; }
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + sb * 128 + c * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(&bar_s_free[sb]);
        ++s_it;
        if (j >= nfull) {  // PARTIAL tile: per-element seq_id mask
          const int st = kv_it % kStages;
          if (!waitw(&bar_k_full[st], (kv_it / kStages) & 1, kSiteKseq)) { alive = false; break; }
          const int32_t* ks = kseq_s[st];
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (my_seq < 0 || ks[c] != my_seq) s[c] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; ++c) mx = fmaxf(mx, s[c]);
        const float mx2 = mx * p.scale_log2;
        const bool grow = mx2 > m_ref + kRescaleThreshold;
        const float m_new = grow ? mx2 : m_ref;
        const float alpha = grow ? ex2(m_ref - m_new) : 1.0f;
        l *= alpha;
        if (j > 0) {  // PV_{j-1} done: O is stable and the P buffer is free
          if (!waitw(&bar_pv_done, pv_it & 1, kSitePvDone)) { alive = false; break; }
          ++pv_it;
          tc_fence_after();
          const bool rescale = grow && m_ref != -INFINITY;
          if (__any_sync(0xffffffffu, rescale)) {
            const float f = rescale ? alpha : 1.0f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + kTmemO + c * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
              tmem_st32(tmem + lane_base + kTmemO + c * 32, r);
            }
            tmem_wait_st();
          }
        }
        m_ref = m_new;
        const float neg_m = m_ref == -INFINITY ? 0.0f : -m_ref;
        const bool any = m_ref != -INFINITY;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = half * 64 + ch * 8 + e * 2;
              const float p0 = any ? ex2(fmaf(s[c], p.scale_log2, neg_m)) : 0.0f;
              const float p1 = any ? ex2(fmaf(s[c + 1], p.scale_log2, neg_m)) : 0.0f;
              l += p0 + p1;
              pk[e] = pack_bf16x2(p0, p1);
            }
            st_shared_v4(sP + half * 16384 + sw128_offset(row, ch), pk[0], pk[1], pk[2], pk[3]);
          }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_p_full);
      }
      if (!alive) break;
      // epilogue: the last PV has finished
      if (!waitw(&bar_pv_done, pv_it & 1, kSitePvDone)) { alive = false; break; }
      ++pv_it;
      tc_fence_after();
      const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kTmemO + c * 32, r);
        tmem_wait_ld();
        if (in_range) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 out;
            out.x = pack_bf16x2(__uint_as_float(r[v * 8 + 0]) * inv_l, __uint_as_float(r[v * 8 + 1]) * inv_l);
            out.y = pack_bf16x2(__uint_as_float(r[v * 8 + 2]) * inv_l, __uint_as_float(r[v * 8 + 3]) * inv_l);
            out.z = pack_bf16x2(__uint_as_float(r[v * 8 + 4]) * inv_l, __uint_as_float(r[v * 8 + 5]) * inv_l);
            out.w = pack_bf16x2(__uint_as_float(r[v * 8 + 6]) * inv_l, __uint_as_float(r[v * 8 + 7]) * inv_l);
            reinterpret_cast<uint4*>(orow)[c * 4 + v] = out;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_o_free);
      if (in_range) *lse_out = l > 0.0f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
pvl_status launch_fwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const int32_t* seq_id,
                      const void* tile_ws, int B, int L, int H, float scale, pvl_bf16* o, float* lse,
                      cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  pvl_status st = make_bhld_tensor_map(&tq, q, B, L, H, D);
  if (st == PVL_OK) st = make_bhld_tensor_map(&tk, k, B, L, H, D);
  if (st == PVL_OK) st = make_bhld_tensor_map(&tv, v, B, L, H, D);
  if (st != PVL_OK) return st;
  DeviceError* err = device_error_record();
  const int sms = sm_count();
  if (!err || sms <= 0) return fail(PVL_ERR_CUDA, "masked_attn_fwd: no usable CUDA device");
  const TileMapView tm = tile_map_view(tile_ws, B, L, 128, 128);
  FwdParams prm;
  prm.seq_id = seq_id;
  prm.header = tm.header;
  prm.row_count = tm.row_count;
  prm.row_full = tm.row_full;
  prm.row_list = tm.row_list;
  prm.q_order = tm.q_order;
  prm.o = reinterpret_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.err = err;
  prm.B = B;
  prm.L = L;
  prm.H = H;
  prm.nT = tm.nTq;
  prm.total_items = static_cast<long long>(B) * tm.nTq * H;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.timeout_ns = kDefaultTimeoutNs;
  const int smem = FwdSmem<D>::kBytes;
  st = check_cuda(cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                  "masked_attn_fwd smem attribute");
  if (st != PVL_OK) return st;
  const long long grid = prm.total_items < sms ? prm.total_items : sms;
  fwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tq, tk, tv, prm);
  return check_cuda(cudaGetLastError(), "masked_attn_fwd launch");
}

}  // namespace
}  // namespace pvl

using namespace pvl;

extern "C" pvl_status masked_attn_fwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const int32_t* seq_id,
                                      const void* tile_ws, int B, int L, int H, int D, float scale, pvl_bf16* o,
                                      float* lse, pvl_stream_t stream) {
  const void* ptrs[] = {q, k, v, seq_id, tile_ws, o, lse};
  const pvl_status st = validate_attn("masked_attn_fwd", ptrs, 7, B, L, H, D, scale);
  if (st != PVL_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 64) return launch_fwd<64>(q, k, v, seq_id, tile_ws, B, L, H, scale, o, lse, s);
  return launch_fwd<128>(q, k, v, seq_id, tile_ws, B, L, H, scale, o, lse, s);
}
