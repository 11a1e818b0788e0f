// masked_attn_bwd: gradients of seq_id-masked softmax attention, sm_103a.
//
// What it computes (the backward of the masked attention the pages run as a
// FlexAttention template, "lingbot_va_attn_profiling" kernel table), with
// P_ij = M_ij exp(scale <q_i, k_j> - LSE_i) recomputed from the saved LSE:
//   Delta_i = <dO_i, O_i>,  dS = P * (dO V^T - Delta),
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
// Keys with seq_id -1 get dK = dV = 0 and queries with seq_id -1 get dQ = 0.
// Cross attention ("lingbot_va_packing" §2.1): queries [B, Lq] and keys
// [B, Lk] carry their own ids; a key (query) whose id no query (key) carries
// also gets zero gradients.
//
// Three launches on the caller's stream:
//   bwd_pre      Delta and LSE * log2(e) per query (fp32, padded to whole
//                128-row tiles), the padded query seq_ids, a zeroed fp32
//                dQ accumulator and a zeroed work-item counter;
//   bwd_main     one persistent CTA per SM over work items (b, key tile, head)
//                in the tile map's longest-first key order, head-major (the
//                CTAs working at one time add into one head's dQ rows, which
//                stay in L2).  Items are handed out at run time from a
//                counter in the workspace, so a CTA that finishes early takes
//                the next one (items differ in length; a fixed round-robin
//                share left the CTAs 5-20 % apart).  Per item the K/V
//                tile stays in shared memory while the non-empty query tiles
//                stream through (FULL first, PARTIAL last), Q in a 2-stage
//                ring, dO with the tile's LSE / Delta / seq_id rows in one:
//                  warp 8     TMA producer (K/V per item, Q_i, dO_i and the
//                             row arrays per tile);
//                  warp 9     TMEM owner and MMA issuer:
//                             S^T = K Q_i^T, dP^T = V dO_i^T, then
//                             dV += P^T dO_i (frees dO), dQ_i = dS K,
//                             dK += dS^T Q_i;
//                  warps 0-7  two warpgroups over the same 128 key rows
//                             (thread row = TMEM lane), each owning half of
//                             the query columns and half of the feature
//                             columns: P^T = exp2(S^T scale log2e - LSE log2e)
//                             and dS^T = P^T (dP^T - Delta) (mask on PARTIAL
//                             tiles only); P^T goes back into TMEM over S^T
//                             (the dV MMA reads it from there), dS^T into
//                             swizzled shared memory (the dQ and dK MMAs read
//                             it); then each warp stages its 32 rows of
//                             dQ_i in shared memory and adds them to the fp32
//                             accumulator with TMA bulk reductions; at the
//                             end each writes half of dK (times scale) and dV.
//   bwd_convert  dQ = bf16(scale * accumulator).
// The score matrix never reaches global memory.  Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pvl_device.cuh"

namespace pvl {
namespace {

constexpr int kThreads = 320;  // warps 0-7 compute, 8 TMA, 9 MMA
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kComputeThreads = 256;
constexpr int kStages = 2;        // Q ring
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S^T            [0, 128); P^T packed over [64 g, 64 g + 32)
constexpr uint32_t kColDP = 128;  // dP^T, then dQ  [128, 256)
constexpr uint32_t kColDV = 256;  // dV             [256, 256 + D)
// dK at [256 + D, 256 + 2 D)

enum BwdSite : uint32_t {
  kSiteKvEmpty = 21, kSiteQdoEmpty, kSiteKvFull, kSiteQdoFull, kSiteDqFree, kSitePsFull, kSiteAccFree,
  kSiteSFull, kSiteDpFull, kSiteMmaDone, kSiteDqReady, kSiteDoEmpty, kSiteDoFull, kSiteDoFullC, kSiteItemEmpty,
  kSiteItemFull
};

// Work items are handed out at run time: the producer thread takes the next
// item index from a global counter (atomicAdd) and passes it to the MMA and
// compute warps through a ring of this many shared-memory slots.
constexpr int kItemSlots = 2;

template <int D>
struct BwdSmem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;             // kStages tiles
  static constexpr int kDO = kQ + kStages * kTile;  // one tile
  static constexpr int kDST = kDO + kTile;          // dS^T bf16 [128 keys][128 queries]
  static constexpr int kStage = kDST + 128 * 256;   // dQ staging: 8 warps x (32 rows x 32 fp32)
  static constexpr int kEnd = kStage + 8 * 4096;
  static constexpr int kBytes = (kEnd + 1024) > 120 * 1024 ? (kEnd + 1024) : 120 * 1024;
};

struct BwdParams {
  const int32_t* header;
  const int32_t* col_count;
  const int32_t* col_full;
  const int32_t* col_list;
  const int32_t* k_order;
  const int32_t* k_seq;   // [B, Lk]    key seq_ids
  const float* delta;     // [B, H, Lp]
  const float* lse2;      // [B, H, Lp] LSE * log2(e)
  const int32_t* qseq;    // [B, Lp]    query seq_ids, -1 past Lq
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  DeviceError* err;
  unsigned int* sched;  // work-item counter, zero at launch
  int B, Lq, Lk, Lp, H;
  int nT;   // key tiles per row (items)
  int nTq;  // query tiles per row: the length of each key tile's query list
  // Lp: Lq rounded up to whole 128-row tiles
  long long total_items;  // n_kt * H, head-major
  int n_kt;               // B * nT: entries of the longest-first key-tile order
  float scale_log2;
  float scale;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_base, int kk) {
  return sdesc_sw128(tile_base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile_base, int kk) {
  return sdesc_sw128(tile_base + kk * 2048, 16384, 1024);
}

// ------------------------------------------------------------- preprocess
// One group of D/8 lanes per (b, l, h) row: Delta = <dO, O> in fp32,
// LSE * log2(e), the row's query seq_id (h = 0), and the row's dQ accumulator
// set to zero unless the query is padding (seq_id -1: its accumulator row
// only ever receives zeros, and the conversion writes its dQ = 0 without
// reading it).  Then the padding positions L <= l < Lp of the padded arrays.
// Row groups per thread and loop iteration of the preprocess (their loads
// issued together; four measured no faster than two).
constexpr int kPreUnroll = 2;
// Idx: the index type, 32-bit whenever B * L * H * D / 8 fits (the
// divisions by H and L are then short).
template <int D, typename Idx>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      const float* __restrict__ lse, const int32_t* __restrict__ seq_id,
                                                      float* __restrict__ delta, float* __restrict__ lse2,
                                                      int32_t* __restrict__ qseq, float* __restrict__ dq_acc,
                                                      unsigned int* __restrict__ sched, int B, int L, int Lp, int H) {
  constexpr int G = D / 8;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0u;  // the main kernel's work-item counter
  const Idx uH = static_cast<Idx>(H), uL = static_cast<Idx>(L);
  const Idx rows = static_cast<Idx>(B) * uL * uH;
  const Idx total = rows * G;
  const Idx stride = static_cast<Idx>(gridDim.x) * blockDim.x;  // a multiple of 32
  // warp-aligned loop: every lane of a warp runs the same iterations, so the
  // shuffles below always see the whole warp.  kPreUnroll groups of rows per
  // iteration, their loads issued together (more bytes in flight per thread).
  for (Idx base = static_cast<Idx>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
       base += kPreUnroll * stride) {
    Idx t[kPreUnroll], row[kPreUnroll], bl[kPreUnroll];
    bool act[kPreUnroll];
    int part[kPreUnroll], my_id[kPreUnroll];
    uint4 a[kPreUnroll], c[kPreUnroll];
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      t[u] = base + u * stride + lane;
      act[u] = t[u] < total;
      row[u] = act[u] ? t[u] / G : 0;
      part[u] = static_cast<int>(t[u] % G);
      bl[u] = row[u] / uH;
      my_id[u] = act[u] ? seq_id[bl[u]] : -1;
      if (act[u]) {
        a[u] = reinterpret_cast<const uint4*>(o + static_cast<size_t>(row[u]) * D)[part[u]];
        c[u] = reinterpret_cast<const uint4*>(dO + static_cast<size_t>(row[u]) * D)[part[u]];
      }
    }
#pragma unroll
    for (int u = 0; u < kPreUnroll; ++u) {
      float s = 0.0f;
      if (act[u]) {
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
        const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c[u]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 x = __bfloat1622float2(a2[i]);
          const float2 y = __bfloat1622float2(c2[i]);
          s = fmaf(x.x, y.x, s);
          s = fmaf(x.y, y.y, s);
        }
      }
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (act[u]) {
        if (my_id[u] >= 0) {
          float4* acc = reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(row[u]) * D + part[u] * 8);
          acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (part[u] == 0) {
          const size_t h = row[u] - bl[u] * uH;
          const size_t b = bl[u] / uL;
          const size_t l = bl[u] - b * uL;
          delta[(b * H + h) * Lp + l] = s;
          lse2[(b * H + h) * Lp + l] = lse[(b * H + h) * L + l] * 1.4426950408889634f;
          if (h == 0) qseq[b * Lp + l] = my_id[u];
        }
      }
    }
  }
  const long long pad = static_cast<long long>(B) * H * (Lp - L);
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < pad;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long bh = t / (Lp - L);
    const long long l = L + t % (Lp - L);
    delta[bh * Lp + l] = 0.0f;
    lse2[bh * Lp + l] = 0.0f;
    if (bh % H == 0) qseq[(bh / H) * Lp + l] = -1;
  }
}

// ------------------------------------------------------------------ convert
// dQ = bf16(scale * accumulator) per group of 8 features; padding queries
// (seq_id -1, whose accumulator rows were not zeroed) get exact zeros
// without a read of the accumulator.
template <typename Idx>
__global__ void __launch_bounds__(256) bwd_convert_kernel(const float* __restrict__ dq_acc,
                                                          const int32_t* __restrict__ seq_id,
                                                          __nv_bfloat16* __restrict__ dq, float scale, long long n8_,
                                                          int groups_per_pos) {
  const Idx n8 = static_cast<Idx>(n8_), gpp = static_cast<Idx>(groups_per_pos);
  const Idx gid = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x;
  const Idx stride = static_cast<Idx>(gridDim.x) * blockDim.x;
  for (Idx i = gid; i < n8; i += stride) {
    if (seq_id[i / gpp] < 0) {  // (b, l) of this group: H * D / 8 groups per position
      reinterpret_cast<uint4*>(dq)[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
    uint4 out;
    out.x = pack_bf16x2(a.x * scale, a.y * scale);
    out.y = pack_bf16x2(a.z * scale, a.w * scale);
    out.z = pack_bf16x2(b.x * scale, b.y * scale);
    out.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = out;
  }
}

// P^T and dS^T for the 64 query columns of group g of one key row: reads
// S^T and dP^T from TMEM, LSE*log2e / Delta / seq_id from shared memory,
// writes P^T (packed bf16) back over S^T columns this group has read and
// dS^T (bf16) into the swizzled shared tile.  kMasked: PARTIAL tile.  Four
// chunks of 16 queries: the next chunk's S^T and dP^T are read from TMEM
// while the current one is computed (1.8 % off the main kernel against two
// chunks of 32 read one after the other).
template <bool kMasked>
__device__ __forceinline__ void pds_chunks(uint32_t tmem_lane, int g, int row, uint32_t sDST, const float* lse2_s,
                                           const float* delta_s, const int32_t* qseq_s, int my_seq, float scale_log2) {
  const float2 c2 = make_float2(scale_log2, scale_log2);
  uint32_t rs[2][16], rd[2][16];
  tmem_ld16(tmem_lane + kColS + 64 * g, rs[0]);
  tmem_ld16(tmem_lane + kColDP + 64 * g, rd[0]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int cur = c & 1;
    tmem_wait_ld_regs(rs[cur], rd[cur]);
    if (c + 1 < 4) {
      tmem_ld16(tmem_lane + kColS + 64 * g + 16 * (c + 1), rs[cur ^ 1]);
      tmem_ld16(tmem_lane + kColDP + 64 * g + 16 * (c + 1), rd[cur ^ 1]);
    }
    uint32_t pp[8], dd[8];
#pragma unroll
    for (int e4 = 0; e4 < 16; e4 += 4) {
      const int q = 64 * g + 16 * c + e4;
      const float4 l4 = *reinterpret_cast<const float4*>(lse2_s + q);
      const float4 d4 = *reinterpret_cast<const float4*>(delta_s + q);
#pragma unroll
      for (int u = 0; u < 4; u += 2) {
        const float2 lv = u == 0 ? make_float2(-l4.x, -l4.y) : make_float2(-l4.z, -l4.w);
        const float2 dv = u == 0 ? make_float2(-d4.x, -d4.y) : make_float2(-d4.z, -d4.w);
        const float2 x = ffma2(make_float2(__uint_as_float(rs[cur][e4 + u]), __uint_as_float(rs[cur][e4 + u + 1])),
                               c2, lv);
        float2 pv = make_float2(ex2(x.x), ex2(x.y));
        if (kMasked) {
          const int4 s4 = *reinterpret_cast<const int4*>(qseq_s + q);
          const int sa = u == 0 ? s4.x : s4.z, sb = u == 0 ? s4.y : s4.w;
          if (my_seq < 0 || sa != my_seq) pv.x = 0.0f;
          if (my_seq < 0 || sb != my_seq) pv.y = 0.0f;
        }
        const float2 ds =
            fmul2(pv, fadd2(make_float2(__uint_as_float(rd[cur][e4 + u]), __uint_as_float(rd[cur][e4 + u + 1])), dv));
        pp[(e4 + u) / 2] = pack_bf16x2(pv.x, pv.y);
        dd[(e4 + u) / 2] = pack_bf16x2(ds.x, ds.y);
      }
    }
    // packed P^T of these 16 queries goes to columns [8 c, 8 c + 8) of the
    // group's S^T, whose values chunk c / 2 <= c has already read (the load
    // in flight reads columns 16 (c + 1) and up)
    tmem_st8(tmem_lane + kColS + 64 * g + 8 * c, pp);
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const uint32_t off = static_cast<uint32_t>(g) * 16384 + sw128_offset(row, c * 2 + v);
      st_shared_v4(sDST + off, dd[4 * v], dd[4 * v + 1], dd[4 * v + 2], dd[4 * v + 3]);
    }
  }
}

// --------------------------------------------------------------------- main
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_do,
                    const __grid_constant__ CUtensorMap tmap_dq, const BwdParams p) {
  using S = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_kv_full, bar_kv_empty, bar_q_full[kStages], bar_q_empty[kStages], bar_do_full, bar_do_empty;
  __shared__ uint64_t bar_s_full, bar_dp_full, bar_ps_full, bar_mma_done, bar_dq_ready, bar_dq_free, bar_acc_free,
      bar_final;
  // LSE * log2(e), Delta and seq_id of the current query tile (loaded with dO)
  __shared__ __align__(16) float lse2_s[128];
  __shared__ __align__(16) float delta_s[128];
  __shared__ __align__(16) int32_t qseq_s[128];
  __shared__ int item_s[kItemSlots];
  __shared__ uint64_t bar_item_full[kItemSlots], bar_item_empty[kItemSlots];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nT = p.nT;
  constexpr uint32_t kColDK = kColDV + D;

  {
    const int32_t* hd = p.header;
    const bool ok = hd[0] == kTileMapMagic && hd[1] == kTileMapVersion && hd[2] == p.B && hd[3] == p.Lq && hd[8] == p.Lk &&
                    hd[4] == 128 && hd[5] == 128;
    if (!ok) {
      if (threadIdx.x == 0 && atomicCAS(&p.err->code, 0u, kDevErrTileMap) == 0u) p.err->block = blockIdx.x;
      return;
    }
  }

  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bar_kv_full, 1);
    mbar_init(&bar_kv_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_q_full[s], 1);
      mbar_init(&bar_q_empty[s], 1 + kComputeThreads / 32);  // dK MMA done + each compute warp's dQ reads
    }
    mbar_init(&bar_do_full, 1);
    mbar_init(&bar_do_empty, 1);
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_ps_full, kComputeThreads);
    mbar_init(&bar_mma_done, 1);
    mbar_init(&bar_dq_ready, 1);
    mbar_init(&bar_dq_free, kComputeThreads);
    mbar_init(&bar_acc_free, kComputeThreads);
    mbar_init(&bar_final, 1);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&bar_item_full[s], 1);                        // the producer thread
      mbar_init(&bar_item_empty[s], 1 + kComputeThreads / 32);  // the MMA warp and each compute warp
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
    tma_prefetch_desc(&tmap_do);
    tma_prefetch_desc(&tmap_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = tmem_base_s;
  const KernelCtl ctl{p.err, &abort_s, p.timeout_ns};
  const uint32_t sK = smem_u32(smem + S::kK);
  const uint32_t sV = smem_u32(smem + S::kV);
  const uint32_t sQ0 = smem_u32(smem + S::kQ);
  const uint32_t sDO = smem_u32(smem + S::kDO);
  const uint32_t sDST = smem_u32(smem + S::kDST);
  constexpr uint32_t kTileBytes = S::kTile;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    uint32_t kv_it = 0, qi = 0;
    bool alive = true;
    auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      bool ok = lane == 0 ? mbar_wait(bar, parity, ctl, site) : true;
      return __shfl_sync(0xffffffffu, ok, 0);
    };
    for (uint32_t it = 0; alive; ++it) {
      // take the next work item and pass it on (-1: none left)
      const int slot = it % kItemSlots;
      if (!wait1(&bar_item_empty[slot], ((it / kItemSlots) & 1) ^ 1, kSiteItemEmpty)) { alive = false; break; }
      if (lane == 0) {
        const unsigned int t = atomicAdd(p.sched, 1u);
        item_s[slot] = t < static_cast<unsigned long long>(p.total_items) ? static_cast<int>(t) : -1;
        mbar_arrive(&bar_item_full[slot]);
      }
      __syncwarp();
      const long long w = item_s[slot];
      if (w < 0) break;
      const int tile = p.k_order[w % p.n_kt];
      const int h = static_cast<int>(w / p.n_kt);
      const int b = tile / nT, kt = tile % nT;
      const int n = p.col_count[tile];
      if (n == 0) continue;
      const int32_t* list = p.col_list + static_cast<size_t>(tile) * p.nTq;
      if (!wait1(&bar_kv_empty, (kv_it & 1) ^ 1, kSiteKvEmpty)) { alive = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_kv_full, 2 * kTileBytes);
#pragma unroll
        for (int s = 0; s < D / 64; ++s) {
          tma_load_4d(smem + S::kK + s * 16384, &tmap_k, &bar_kv_full, s * 64, h, kt * 128, b);
          tma_load_4d(smem + S::kV + s * 16384, &tmap_v, &bar_kv_full, s * 64, h, kt * 128, b);
        }
      }
      __syncwarp();
      ++kv_it;
      const size_t row_off = (static_cast<size_t>(b) * p.H + h) * p.Lp;
      for (int i = 0; i < n; ++i, ++qi) {
        const int qt = list[i];
        const int st = qi % kStages;
        if (!wait1(&bar_q_empty[st], ((qi / kStages) & 1) ^ 1, kSiteQdoEmpty)) { alive = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_q_full[st], kTileBytes);
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(smem + S::kQ + st * kTileBytes + s * 16384, &tmap_q, &bar_q_full[st], s * 64, h, qt * 128, b);
        }
        __syncwarp();
        if (!wait1(&bar_do_empty, (qi & 1) ^ 1, kSiteDoEmpty)) { alive = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_do_full, kTileBytes + 3 * 512);
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(smem + S::kDO + s * 16384, &tmap_do, &bar_do_full, s * 64, h, qt * 128, b);
          bulk_load(lse2_s, p.lse2 + row_off + qt * 128, 512, &bar_do_full);
          bulk_load(delta_s, p.delta + row_off + qt * 128, 512, &bar_do_full);
          bulk_load(qseq_s, p.qseq + static_cast<size_t>(b) * p.Lp + qt * 128, 512, &bar_do_full);
        }
        __syncwarp();
      }
    }
    if (abort_s && lane == 0) {
      if (kv_it > 0) mbar_drain(&bar_kv_full, (kv_it - 1) & 1, 100000000ull);
      for (uint32_t it = qi > kStages ? qi - kStages : 0; it <= qi; ++it)
        mbar_drain(&bar_q_full[it % kStages], (it / kStages) & 1, 100000000ull);
      if (qi > 0) mbar_drain(&bar_do_full, (qi - 1) & 1, 100000000ull);
      mbar_drain(&bar_do_full, qi & 1, 100000000ull);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_st = idesc_bf16(128, 128, false, false);  // S^T, dP^T
    constexpr uint32_t idesc_acc = idesc_bf16(128, D, false, true);    // dV, dK
    constexpr uint32_t idesc_dq = idesc_bf16(128, D, true, true);      // dQ
    uint32_t kv_it = 0, qi = 0, item_it = 0;
    bool alive = true;
    // All lanes wait (no divergence to rejoin); one lane issues.  Where two
    // barriers gate the next MMA, both are tested at once first.
    auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, site));
    };
    auto ready2 = [&](uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1) {
      return __all_sync(0xffffffffu, mbar_try_wait(b0, p0) & mbar_try_wait(b1, p1));
    };
    for (uint32_t it = 0; alive; ++it) {
      const int slot = it % kItemSlots;
      if (!wait1(&bar_item_full[slot], (it / kItemSlots) & 1, kSiteItemFull)) { alive = false; break; }
      const long long w = item_s[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_item_empty[slot]);
      if (w < 0) break;
      const int tile = p.k_order[w % p.n_kt];
      const int n = p.col_count[tile];
      if (n == 0) continue;
      if (!wait1(&bar_kv_full, kv_it & 1, kSiteKvFull)) { alive = false; break; }
      ++kv_it;
      for (int i = 0; i < n; ++i, ++qi) {
        const int st = qi % kStages;
        const uint32_t sQ = sQ0 + st * kTileBytes;
        if (!wait1(&bar_q_full[st], (qi / kStages) & 1, kSiteQdoFull)) { alive = false; break; }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + kColS, kmajor_desc(sK, kk), kmajor_desc(sQ, kk), idesc_st, kk > 0 ? 1u : 0u);
          umma_commit(&bar_s_full);
        }
        __syncwarp();
        // dP^T overwrites the columns dQ of the previous query tile used
        if (!ready2(&bar_dq_free, (qi & 1) ^ 1, &bar_do_full, qi & 1)) {
          if (!wait1(&bar_dq_free, (qi & 1) ^ 1, kSiteDqFree)) { alive = false; break; }
          if (!wait1(&bar_do_full, qi & 1, kSiteDoFull)) { alive = false; break; }
        }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + kColDP, kmajor_desc(sV, kk), kmajor_desc(sDO, kk), idesc_st, kk > 0 ? 1u : 0u);
          umma_commit(&bar_dp_full);
        }
        __syncwarp();
        if (!wait1(&bar_ps_full, qi & 1, kSitePsFull)) { alive = false; break; }
        if (i == 0 && !wait1(&bar_acc_free, (item_it & 1) ^ 1, kSiteAccFree)) { alive = false; break; }
        tc_fence_after();
        if (lane == 0) {
          // dV += P^T dO_i first (P^T in TMEM: query columns [0, 64) at TMEM
          // columns [0, 32), [64, 128) at [64, 96)), so dO can be reloaded
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + kColDV, tmem + kColS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8), mnmajor_desc(sDO, kk),
                    idesc_acc, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bar_do_empty);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss(tmem + kColDP, mnmajor_desc(sDST, kk), mnmajor_desc(sK, kk), idesc_dq, kk > 0 ? 1u : 0u);
          umma_commit(&bar_dq_ready);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss(tmem + kColDK, kmajor_desc(sDST, kk), mnmajor_desc(sQ, kk), idesc_acc, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bar_mma_done);
          umma_commit(&bar_q_empty[st]);
        }
        __syncwarp();
      }
      if (!alive) break;
      if (lane == 0) umma_commit(&bar_kv_empty);
      __syncwarp();
      ++item_it;
    }
    if (lane == 0) {
      umma_commit(&bar_final);
      mbar_drain(&bar_final, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- compute
    // Two warpgroups, g = 0 (warps 0-3) and g = 1 (warps 4-7).  Both cover the
    // 128 key rows (thread row = TMEM lane); group g owns query columns
    // [64 g, 64 g + 64) of S^T, dP^T, P^T, dS^T and feature columns
    // [g D/2, (g + 1) D/2) of dQ, dK and dV, so the groups never exchange data.
    constexpr int kHalfD = D / 2;
    constexpr int kHalfChunks = kHalfD / 32;
    const int g = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // per-warp dQ staging: one 32-row x 32-float buffer (slice 0)
    uint8_t* stage = smem + S::kStage + warp * 4096;
    uint32_t qi = 0, md_it = 0;
    int pend_q = -1;  // Q stage whose dQ staging reads are still to be released
    bool alive = true;
    auto waitw = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, site));
    };
    for (uint32_t it = 0; alive; ++it) {
      const int slot = it % kItemSlots;
      if (!waitw(&bar_item_full[slot], (it / kItemSlots) & 1, kSiteItemFull)) { alive = false; break; }
      const long long w = item_s[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_item_empty[slot]);
      if (w < 0) break;
      const int tile = p.k_order[w % p.n_kt];
      const int h = static_cast<int>(w / p.n_kt);
      const int b = tile / nT, kt = tile % nT;
      const int n = p.col_count[tile];
      const int kpos = kt * 128 + row;
      const bool k_in = kpos < p.Lk;
      const size_t krow = ((static_cast<size_t>(b) * p.Lk + kpos) * p.H + h) * D + g * kHalfD;
      if (n == 0) {  // no valid key in this tile: zero gradients
        if (k_in) {
#pragma unroll
          for (int c = 0; c < kHalfD / 8; ++c) {
            reinterpret_cast<uint4*>(p.dk + krow)[c] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(p.dv + krow)[c] = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      const int nfull = p.col_full[tile];
      const int32_t* list = p.col_list + static_cast<size_t>(tile) * p.nTq;
      const int my_seq = k_in ? p.k_seq[static_cast<size_t>(b) * p.Lk + kpos] : -1;
      for (int i = 0; i < n; ++i, ++qi) {
        const int qt = list[i];
        const bool partial = i >= nfull;
        if (!waitw(&bar_s_full, qi & 1, kSiteSFull)) { alive = false; break; }
        if (!waitw(&bar_dp_full, qi & 1, kSiteDpFull)) { alive = false; break; }
        // acquire this tile's LSE / Delta / seq_id rows (their phase can not
        // advance before the dV MMA, which waits for this group)
        if (!waitw(&bar_do_full, qi & 1, kSiteDoFullC)) { alive = false; break; }
        tc_fence_after();
        if (!partial)
          pds_chunks<false>(tmem + lane_base, g, row, sDST, lse2_s, delta_s, qseq_s, my_seq, p.scale_log2);
        else
          pds_chunks<true>(tmem + lane_base, g, row, sDST, lse2_s, delta_s, qseq_s, my_seq, p.scale_log2);
        tmem_wait_st();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_ps_full);
        // the previous tile's dQ reductions read this warp's staging buffer
        // and its part of that tile's Q stage: once they have, the stage goes
        // back to the producer (its next load is two tiles ahead)
        if (pend_q >= 0) {
          if (lane == 0) {
            bulk_wait_group_read<0>();
            mbar_arrive(&bar_q_empty[pend_q]);
          }
          __syncwarp();
          pend_q = -1;
        }
        if (!waitw(&bar_dq_ready, qi & 1, kSiteDqReady)) { alive = false; break; }
        tc_fence_after();
        uint32_t r[kHalfChunks][32];
#pragma unroll
        for (int c = 0; c < kHalfChunks; ++c) tmem_ld32(tmem + lane_base + kColDP + g * kHalfD + c * 32, r[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar_dq_free);
        // dQ_i rows of this warp (32 query rows x this group's D/2 columns) ->
        // fp32 accumulator with TMA reductions of 32 x 32 slices.  Slice 0 goes
        // through the warp's staging buffer, slice 1 (D = 128) through the
        // warp's 4 KB of this tile's Q stage once the dK MMA has read Q_i (the
        // stage is handed back to the producer after the reductions read it);
        // padding rows add exact zeros, boxes wholly past L are skipped.
        const int row0 = qt * 128 + (warp & 3) * 32;
        const int qst = static_cast<int>(qi % kStages);
        uint8_t* dst_slice = smem + S::kQ + qst * S::kTile + warp * 4096;
#pragma unroll
        for (int c = 0; c < kHalfChunks; ++c) {
          if (c == 1) {
            if (!waitw(&bar_mma_done, md_it & 1, kSiteMmaDone)) { alive = false; break; }
            ++md_it;
          }
          uint8_t* buf = c == 0 ? stage : dst_slice;
          // 128-byte swizzle (the map's): 16-byte chunk v of row `lane` sits at
          // chunk v ^ (lane & 7), so the eight lanes of a store phase hit
          // distinct banks
          const uint32_t dst = smem_u32(buf + lane * 128);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            st_shared_v4(dst + ((v ^ (lane & 7)) << 4), r[c][4 * v], r[c][4 * v + 1], r[c][4 * v + 2],
                         r[c][4 * v + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0 && row0 >= 0 && row0 < p.Lq) tma_reduce_add_4d(&tmap_dq, buf, g * kHalfD + 32 * c, h, row0, b);
        }
        if (!alive) break;
        if (kHalfChunks < 2) {  // D = 64: the dS^T slice was not used, but the MMAs must still be waited for
          if (!waitw(&bar_mma_done, md_it & 1, kSiteMmaDone)) { alive = false; break; }
          ++md_it;
        }
        if (lane == 0) bulk_commit_group();
        pend_q = qst;
      }
      if (!alive) break;
      // epilogue: the last tile's mma_done (waited above) covers every dV / dK
      // MMA of this item
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kHalfChunks; ++c) {
        uint32_t rv[32], rk[32];
        tmem_ld32(tmem + lane_base + kColDV + g * kHalfD + c * 32, rv);
        tmem_ld32(tmem + lane_base + kColDK + g * kHalfD + c * 32, rk);
        tmem_wait_ld();
        if (k_in) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 ov, ok;
            ov.x = pack_bf16x2(__uint_as_float(rv[8 * v + 0]), __uint_as_float(rv[8 * v + 1]));
            ov.y = pack_bf16x2(__uint_as_float(rv[8 * v + 2]), __uint_as_float(rv[8 * v + 3]));
            ov.z = pack_bf16x2(__uint_as_float(rv[8 * v + 4]), __uint_as_float(rv[8 * v + 5]));
            ov.w = pack_bf16x2(__uint_as_float(rv[8 * v + 6]), __uint_as_float(rv[8 * v + 7]));
            ok.x = pack_bf16x2(__uint_as_float(rk[8 * v + 0]) * p.scale, __uint_as_float(rk[8 * v + 1]) * p.scale);
            ok.y = pack_bf16x2(__uint_as_float(rk[8 * v + 2]) * p.scale, __uint_as_float(rk[8 * v + 3]) * p.scale);
            ok.z = pack_bf16x2(__uint_as_float(rk[8 * v + 4]) * p.scale, __uint_as_float(rk[8 * v + 5]) * p.scale);
            ok.w = pack_bf16x2(__uint_as_float(rk[8 * v + 6]) * p.scale, __uint_as_float(rk[8 * v + 7]) * p.scale);
            reinterpret_cast<uint4*>(p.dv + krow)[c * 4 + v] = ov;
            reinterpret_cast<uint4*>(p.dk + krow)[c * 4 + v] = ok;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_acc_free);
    }
    // every dQ reduction of this warp has completed before the CTA leaves
    // (after an abort the last reductions may not have been committed yet:
    // commit them, so that the wait covers them too)
    if (lane == 0) {
      bulk_commit_group();
      bulk_wait_group_all();
      if (pend_q >= 0) mbar_arrive(&bar_q_empty[pend_q]);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int grid_for(long long work, int threads) {
  const int sms = sm_count();
  long long g = (work + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 132) * 8;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

template <int D>
pvl_status launch_bwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const pvl_bf16* o,
                      const pvl_bf16* dO, const float* lse, const int32_t* q_seq, const int32_t* k_seq,
                      const void* tile_ws, int B, int L, int Lk, int H, float scale, pvl_bf16* dq, pvl_bf16* dk,
                      pvl_bf16* dv, void* ws, cudaStream_t stream) {
  // L: queries (Lq), Lk: keys
  void* mark_before = nullptr;  // measurement events of this call, if any
  void* mark_after = nullptr;
  take_bwd_main_marks(&mark_before, &mark_after);
  CUtensorMap tq, tk, tv, tdo, tdq;
  pvl_status st = make_bhld_tensor_map(&tq, q, B, L, H, D);
  if (st == PVL_OK) st = make_bhld_tensor_map(&tk, k, B, Lk, H, D);
  if (st == PVL_OK) st = make_bhld_tensor_map(&tv, v, B, Lk, H, D);
  if (st == PVL_OK) st = make_bhld_tensor_map(&tdo, dO, B, L, H, D);
  if (st != PVL_OK) return st;
  DeviceError* err = device_error_record();
  const int sms = sm_count();
  if (!err || sms <= 0) return fail(PVL_ERR_CUDA, "masked_attn_bwd: no usable CUDA device");
  st = make_bhld_f32_tensor_map(&tdq, ws, B, L, H, D, 32, 32);  // dQ accumulator at the start of ws
  if (st != PVL_OK) return st;

  const int Lp = bwd_lp(L);
  char* wsb = static_cast<char*>(ws);
  float* dq_acc = reinterpret_cast<float*>(wsb);
  float* delta = reinterpret_cast<float*>(wsb + bwd_ws_dq_bytes(B, L, H, D));
  float* lse2 = reinterpret_cast<float*>(wsb + bwd_ws_dq_bytes(B, L, H, D) + bwd_ws_rows_bytes(B, L, H));
  int32_t* qseq = reinterpret_cast<int32_t*>(wsb + bwd_ws_dq_bytes(B, L, H, D) + 2 * bwd_ws_rows_bytes(B, L, H));
  unsigned int* sched = reinterpret_cast<unsigned int*>(wsb + bwd_ws_sched_offset(B, L, H, D));
  const long long rows = static_cast<long long>(B) * L * H;

  // 32-bit indices when every index (and its grid-stride successor) fits
  const bool idx32 = rows * (D / 8) + static_cast<long long>(kPreUnroll) * sms * 8 * 256 < (1ll << 31);
  if (idx32)
    bwd_pre_kernel<D, uint32_t><<<grid_for(rows * (D / 8), 256), 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(o), reinterpret_cast<const __nv_bfloat16*>(dO), lse, q_seq, delta,
        lse2, qseq, dq_acc, sched, B, L, Lp, H);
  else
    bwd_pre_kernel<D, unsigned long long><<<grid_for(rows * (D / 8), 256), 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(o), reinterpret_cast<const __nv_bfloat16*>(dO), lse, q_seq, delta,
        lse2, qseq, dq_acc, sched, B, L, Lp, H);
  st = check_cuda(cudaGetLastError(), "masked_attn_bwd preprocess launch");
  if (st != PVL_OK) return st;

  const TileMapView tm = tile_map_view(tile_ws, B, L, Lk, 128, 128, 0);
  BwdParams prm;
  prm.header = tm.header;
  prm.col_count = tm.col_count;
  prm.col_full = tm.col_full;
  prm.col_list = tm.col_list;
  prm.k_order = tm.k_order;
  prm.k_seq = k_seq;
  prm.delta = delta;
  prm.lse2 = lse2;
  prm.qseq = qseq;
  prm.dq_acc = dq_acc;
  prm.dk = reinterpret_cast<__nv_bfloat16*>(dk);
  prm.dv = reinterpret_cast<__nv_bfloat16*>(dv);
  prm.err = err;
  prm.sched = sched;
  prm.B = B;
  prm.Lq = L;
  prm.Lk = Lk;
  prm.Lp = Lp;
  prm.H = H;
  prm.nT = tm.nTk;
  prm.nTq = tm.nTq;
  prm.n_kt = B * tm.nTk;
  prm.total_items = static_cast<long long>(prm.n_kt) * H;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.scale = scale;
  prm.timeout_ns = attn_wait_timeout_ns();
  const int smem = BwdSmem<D>::kBytes;
  st = check_cuda(cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                  "masked_attn_bwd smem attribute");
  if (st != PVL_OK) return st;
  const long long grid = prm.total_items < sms ? prm.total_items : sms;
  if (mark_before) {
    st = check_cuda(cudaEventRecord(static_cast<cudaEvent_t>(mark_before), stream), "masked_attn_bwd marker");
    if (st != PVL_OK) return st;
  }
  bwd_main_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tq, tk, tv, tdo, tdq, prm);
  st = check_cuda(cudaGetLastError(), "masked_attn_bwd main launch");
  if (st != PVL_OK) return st;
  if (mark_after) {
    st = check_cuda(cudaEventRecord(static_cast<cudaEvent_t>(mark_after), stream), "masked_attn_bwd marker");
    if (st != PVL_OK) return st;
  }

  const long long n8 = rows * D / 8;
  if (idx32)
    bwd_convert_kernel<uint32_t><<<grid_for(n8, 256), 256, 0, stream>>>(
        dq_acc, q_seq, reinterpret_cast<__nv_bfloat16*>(dq), scale, n8, H * D / 8);
  else
    bwd_convert_kernel<unsigned long long><<<grid_for(n8, 256), 256, 0, stream>>>(
        dq_acc, q_seq, reinterpret_cast<__nv_bfloat16*>(dq), scale, n8, H * D / 8);
  return check_cuda(cudaGetLastError(), "masked_attn_bwd convert launch");
}

}  // namespace
}  // namespace pvl

using namespace pvl;

extern "C" size_t masked_attn_bwd_ws_bytes_cross(int B, int Lq, int Lk, int H, int D) {
  if (B < 1 || Lq < 1 || Lk < 1 || H < 1 || D < 1) return 0;
  return bwd_ws_total_bytes(B, Lq, H, D);  // every scratch array is on the query side
}

extern "C" size_t masked_attn_bwd_ws_bytes(int B, int L, int H, int D) {
  return masked_attn_bwd_ws_bytes_cross(B, L, L, H, D);
}

extern "C" pvl_status masked_attn_bwd_cross(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v,
                                            const pvl_bf16* o, const pvl_bf16* dO, const float* lse,
                                            const int32_t* q_seq_id, const int32_t* k_seq_id, const void* tile_ws,
                                            int B, int Lq, int Lk, int H, int D, float scale, pvl_bf16* dq,
                                            pvl_bf16* dk, pvl_bf16* dv, void* ws, size_t ws_bytes,
                                            pvl_stream_t stream) {
  const void* ptrs[] = {q, k, v, o, dO, lse, q_seq_id, k_seq_id, tile_ws, dq, dk, dv, ws};
  if (ws && ws_bytes < masked_attn_bwd_ws_bytes_cross(B, Lq, Lk, H, D))
    return fail(PVL_ERR_INVALID_ARG, "masked_attn_bwd: workspace %zu bytes < %zu needed", ws_bytes,
                masked_attn_bwd_ws_bytes_cross(B, Lq, Lk, H, D));
  pvl_status st = validate_attn_qk("masked_attn_bwd", ptrs, 13, B, Lq, Lk, H, D, scale);
  if (st != PVL_OK) return st;
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return fail(PVL_ERR_INVALID_ARG, "masked_attn_bwd: workspace must be 256-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 64)
    return launch_bwd<64>(q, k, v, o, dO, lse, q_seq_id, k_seq_id, tile_ws, B, Lq, Lk, H, scale, dq, dk, dv, ws, s);
  return launch_bwd<128>(q, k, v, o, dO, lse, q_seq_id, k_seq_id, tile_ws, B, Lq, Lk, H, scale, dq, dk, dv, ws, s);
}

extern "C" pvl_status masked_attn_bwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const pvl_bf16* o,
                                      const pvl_bf16* dO, const float* lse, const int32_t* seq_id,
                                      const void* tile_ws, int B, int L, int H, int D, float scale, pvl_bf16* dq,
                                      pvl_bf16* dk, pvl_bf16* dv, void* ws, size_t ws_bytes, pvl_stream_t stream) {
  return masked_attn_bwd_cross(q, k, v, o, dO, lse, seq_id, seq_id, tile_ws, B, L, L, H, D, scale, dq, dk, dv, ws,
                               ws_bytes, stream);
}

// ------------------------------------------------------------------------
// masked_attn_bwd_no_alloc: the same backward for callers that cannot
// allocate device memory.  Its scratch (fp32 dQ accumulator and Delta) lives
// in this file-scope array instead of a caller-provided workspace.
namespace pvl {
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(PVL_NO_ALLOC_SCRATCH_BYTES);

// Held by every GPU that loads the library until the process exits.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

std::mutex g_no_alloc_mu;
void* g_no_alloc_ptr[64] = {};

// Device address of the scratch array on the current device.  Host code only
// sees a host-side stand-in under the array's name, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.  The kept
// address is that of the device's context when it was looked up (one primary
// context per device for the life of the process; cudaDeviceReset would make
// it stale).
pvl_status no_alloc_scratch(void** out) {
  int dev = -1;
  pvl_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != PVL_OK) return st;
  if (dev < 0 || dev >= 64) return fail(PVL_ERR_UNSUPPORTED, "masked_attn_bwd_no_alloc: device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_no_alloc_mu);
  if (!g_no_alloc_ptr[dev]) {
    void* p = nullptr;
    st = check_cuda(cudaGetSymbolAddress(&p, g_no_alloc_scratch), "cudaGetSymbolAddress(scratch)");
    if (st != PVL_OK) return st;
    g_no_alloc_ptr[dev] = p;
  }
  *out = g_no_alloc_ptr[dev];
  return PVL_OK;
}

}  // namespace
}  // namespace pvl

extern "C" pvl_status masked_attn_bwd_no_alloc(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v,
                                               const pvl_bf16* o, const pvl_bf16* dO, const float* lse,
                                               const int32_t* seq_id, const void* tile_ws, int B, int L, int H,
                                               int D, float scale, pvl_bf16* dq, pvl_bf16* dk, pvl_bf16* dv,
                                               pvl_stream_t stream) {
  const void* ptrs[] = {q, k, v, o, dO, lse, seq_id, tile_ws, dq, dk, dv};
  pvl_status st = validate_attn("masked_attn_bwd_no_alloc", ptrs, 11, B, L, H, D, scale);
  if (st != PVL_OK) return st;
  const size_t need = masked_attn_bwd_ws_bytes(B, L, H, D);
  if (need > kNoAllocScratchBytes)
    return fail(PVL_ERR_UNSUPPORTED,
                "masked_attn_bwd_no_alloc: this shape needs %zu bytes of scratch; the library's static scratch "
                "holds %zu bytes (about B*L*H*(D+2)*4 must fit); use masked_attn_bwd with a workspace instead",
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  st = no_alloc_scratch(&scratch);
  if (st != PVL_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 64)
    return launch_bwd<64>(q, k, v, o, dO, lse, seq_id, seq_id, tile_ws, B, L, L, H, scale, dq, dk, dv, scratch, s);
  return launch_bwd<128>(q, k, v, o, dO, lse, seq_id, seq_id, tile_ws, B, L, L, H, scale, dq, dk, dv, scratch, s);
}
