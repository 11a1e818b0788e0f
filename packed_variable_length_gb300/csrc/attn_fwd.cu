// masked_attn_fwd: seq_id-masked softmax attention, forward, for sm_103a.
//
// What it computes ("furniture_packing_variable_length", attention masking;
// "lingbot_va_attn_profiling", doc_id[q] == doc_id[k] mask): for every batch
// row b, head h and query i with s_i >= 0,
//   O_i = sum_{j: s_j = s_i} softmax_j(scale * <q_i, k_j>) v_j,
//   LSE_i = log sum_{j: s_j = s_i} exp(scale * <q_i, k_j>);
// rows with s_i = -1 get O_i = 0 and LSE_i = -inf.  For cross attention
// ("lingbot_va_packing" §2.1) the keys carry their own ids t_j and length Lk
// (j: t_j = s_i above); a query whose id no key carries also gets O_i = 0,
// LSE_i = -inf.
//
// Design.  One persistent CTA per SM walks work items (b, query-tile pair,
// head): two adjacent 128-row query tiles A and B that share one stream of
// key tiles, taken from level 1 of the tile map (256-row query tiles) in its
// longest-first order, head-major (the CTAs running together read one
// head's K and V, 34 MB at 64k tokens, which stay in L2).  Items are handed
// out at run time from a per-stream counter, so a CTA that finishes early
// takes the next one (a fixed round-robin share left the CTAs 5-16 % apart).  Only the key tiles the map
// lists as non-empty are touched, FULL ones first (no per-element mask),
// then PARTIAL ones (mask from the seq_ids).
//   warp 8      TMA producer: the Q pair once per item, K and V tiles into
//               separate 2-stage rings (a K stage frees as soon as both S
//               MMAs that read it are done).
//   warps 9, 10 issue tcgen05.mma from one thread each, warp 9 for tile A
//               (and owns TMEM: S_A, S_B, O_A, O_B, 512 columns), warp 10
//               for tile B, each bracket PV_x(j), S_x(j+1); a turn token
//               keeps the brackets in the order A, B, A, B, ..., so the
//               tensor core works on one query tile while the other tile's
//               softmax runs, and each issuer checks its gates while the
//               other one issues.  An issuer passes the turn before its
//               bracket's last MMA and commits (an MMA issue returns only
//               when the tensor core takes the instruction), so the other
//               bracket queues right behind.  PV reads P straight from TMEM.
//   warps 0-7   softmax, tile A then tile B of each key tile: warp w holds
//               query rows 32 (w % 4) .. + 31 (its TMEM lanes) and key half
//               w / 4 of them, so that the two warps on each SM
//               sub-partition share its exponential unit.  A half row of S
//               comes into registers with one TMEM wait (warpgroup 2 gives
//               up registers for this); in PARTIAL tiles inadmissible keys
//               are set to -inf.  The two halves swap their partial row
//               maxima (shared memory and an mbarrier per warp pair), then
//               P = exp2(scale*log2e*S - m) with its row sum, and P written
//               as packed bf16 over the first 64 columns of the same S
//               buffer.  O is rescaled in TMEM only when the running max
//               grows by more than 2^8 (the stale max bounds every P by 256
//               and the final division uses the same max).  The epilogue
//               adds the halves' row sums, divides and writes O and LSE.
// Every wait is bounded; on expiry the CTA records the failure, drains its
// outstanding copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pvl_device.cuh"

namespace pvl {
namespace {

// warps 0-7 softmax (two warpgroups, one per key half), 8 TMA, 9 and 10 MMA
// issuers (tiles A and B), 11 idle; warpgroup 2's registers go to the
// softmax groups
constexpr int kThreads = 384;
// registers per thread after reallocation: 256 x 208 + 128 x 88 = 384 x 168,
// the launch's own allotment (168 = 65536 / 384 rounded down to 8)
constexpr uint32_t kRegsSoftmax = 208;
constexpr uint32_t kRegsOther = 88;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;    // MMA issuer of query tile A; owns TMEM
constexpr int kMmaWarpB = 10;  // MMA issuer of query tile B
constexpr int kStages = 2;
// MMAs of a bracket issued after the turn has passed to the other issuer
constexpr int kTurnEarly = 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S_X at [128 X, 128 X + 128); P_X packed over its first 64 columns
constexpr uint32_t kColO = 256;  // O_X at [256 + X D, 256 + (X + 1) D)
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum FwdSite : uint32_t {
  kSiteQEmpty = 1, kSiteKEmpty, kSiteVEmpty, kSiteQFull, kSiteKFull, kSiteVFull, kSitePFull, kSiteOFree,
  kSiteSFull, kSitePvDone, kSiteTurn, kSiteItemEmpty, kSiteItemFull, kSiteXch
};

// Work items are handed out at run time: the producer thread takes the next
// item index from a counter (atomicAdd) and passes it to the MMA and softmax
// warps through a ring of this many shared-memory slots.
constexpr int kItemSlots = 2;

template <int D>
struct FwdSmem {
  static constexpr int kTile = 128 * D * 2;  // one 128 x D bf16 tile (D / 64 swizzled 16 KB blocks)
  static constexpr int kQ = 0;               // Q_A then Q_B
  static constexpr int kK = kQ + 2 * kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kEnd = kV + kStages * kTile;
  // 1 KB alignment slack; never below 120 KB so two CTAs can not share an SM
  // (each CTA allocates all 512 TMEM columns).
  static constexpr int kBytes = (kEnd + 1024) > 120 * 1024 ? (kEnd + 1024) : 120 * 1024;
};

struct FwdParams {
  const int32_t* q_seq;      // [B, Lq] query seq_ids
  const int32_t* k_seq;      // [B, Lk] key seq_ids (q_seq for self attention)
  const int32_t* header;     // level-1 map (256-row query tiles)
  const int32_t* row_count;
  const int32_t* row_full;
  const int32_t* row_list;
  const int32_t* q_order;
  __nv_bfloat16* o;
  float* lse;
  DeviceError* err;
  unsigned int* sched;       // work-item counter, zero at launch; null: fixed round-robin
  int B, Lq, Lk, H, nP, nK;  // query-tile pairs and key tiles per row
  long long total_items;  // n_pairs * H, head-major
  int n_pairs;            // B * nP: entries of the longest-first query-tile-pair order
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

// Admissibility of keys kt*128 + 32w .. +31 for a query with id my_seq, as a
// 32-bit mask (bit c = key kt*128 + 32w + c may be attended).
__device__ __forceinline__ uint32_t key_mask_word(const int32_t* __restrict__ seq_row, int L, int kt, int w,
                                                  int my_seq) {
  if (my_seq < 0) return 0u;
  const int k0 = kt * 128 + 32 * w;
  uint32_t bits = 0;
  if (k0 + 32 <= L && (reinterpret_cast<uintptr_t>(seq_row + k0) & 15u) == 0) {
    const int4* src = reinterpret_cast<const int4*>(seq_row + k0);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const int4 s4 = __ldg(src + v);
      bits |= (s4.x == my_seq ? 1u : 0u) << (4 * v);
      bits |= (s4.y == my_seq ? 1u : 0u) << (4 * v + 1);
      bits |= (s4.z == my_seq ? 1u : 0u) << (4 * v + 2);
      bits |= (s4.w == my_seq ? 1u : 0u) << (4 * v + 3);
    }
  } else {
    for (int c = 0; c < 32; ++c) {
      const int kpos = k0 + c;
      if (kpos < L && __ldg(seq_row + kpos) == my_seq) bits |= 1u << c;
    }
  }
  return bits;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Half hf of one query row of S (keys [64 hf, 64 hf + 64)) into registers
// with a single TMEM wait; in a PARTIAL tile the inadmissible keys are set to
// -inf, so that they drop out of the max and exponentiate to 0.  Returns the
// max over these 64 keys.
template <bool kMasked>
__device__ __forceinline__ float load_half_row(uint32_t s_col, int hf, uint32_t (&s)[2][32], const int32_t* seq_row,
                                               int L, int kt, int my_seq) {
#pragma unroll
  for (int c = 0; c < 2; ++c) tmem_ld32(s_col + 64 * hf + 32 * c, s[c]);
  uint32_t mk[2];
  if (kMasked) {
#pragma unroll
    for (int c = 0; c < 2; ++c) mk[c] = key_mask_word(seq_row, L, kt, 2 * hf + c, my_seq);
  }
  tmem_wait_ld();
  if (kMasked) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (!((mk[c] >> i) & 1u)) s[c][i] = __float_as_uint(-INFINITY);
  }
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int i = 0; i < 32; i += 8)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        m[u] = fmax3(m[u], __uint_as_float(s[c][i + 2 * u]), __uint_as_float(s[c][i + 2 * u + 1]));
  return fmax3(m[0], m[1], fmaxf(m[2], m[3]));
}

// P = 2^(scale_log2 * S + neg_m) for half hf of one row held in registers,
// written as packed bf16 over columns [32 hf, 32 hf + 32) of the same S
// buffer (P of keys 2c and 2c + 1 in column c); returns the sum of these 64
// values of P.  Masked keys hold -inf and give exactly 0.
__device__ __forceinline__ float exp_store_half(uint32_t s_col, int hf, const uint32_t (&s)[2][32], float scale_log2,
                                                float neg_m) {
  const float2 c2 = make_float2(scale_log2, scale_log2);
  const float2 m2 = make_float2(neg_m, neg_m);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float2 x = ffma2(make_float2(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), c2, m2);
      const float p0 = ex2(x.x), p1 = ex2(x.y);
      if ((e >> 1) & 1) acc1 = fadd2(acc1, make_float2(p0, p1));
      else acc0 = fadd2(acc0, make_float2(p0, p1));
      pk[e >> 1] = pack_bf16x2(p0, p1);
    }
    tmem_st16(s_col + 32 * hf + 16 * c, pk);
  }
  return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  using S = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q_full, bar_q_empty, bar_o_free[2], bar_final[2], bar_turn[2];
  __shared__ uint64_t bar_k_full[kStages], bar_k_empty[kStages], bar_v_full[kStages], bar_v_empty[kStages];
  __shared__ uint64_t bar_s_full[2], bar_p_full[2], bar_pv_done[2];
  // the two warps holding halves of the same 32 rows swap their partial row
  // maxima (per key tile) and row sums (per item) here: [tile][slot][half][row]
  __shared__ uint64_t bar_xch[2][4];
  __shared__ float xch_s[2][2][2][128];
  __shared__ int item_s[kItemSlots];
  __shared__ uint64_t bar_item_full[kItemSlots], bar_item_empty[kItemSlots];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nP = p.nP, nK = p.nK;

  // The tile map must describe this call; otherwise do nothing.
  {
    const int32_t* hd = p.header;
    const bool ok = hd[0] == kTileMapMagic && hd[1] == kTileMapVersion && hd[2] == p.B && hd[3] == p.Lq && hd[8] == p.Lk &&
                    hd[4] == 256 && hd[5] == 128;
    if (!ok) {
      if (threadIdx.x == 0 && atomicCAS(&p.err->code, 0u, kDevErrTileMap) == 0u) p.err->block = blockIdx.x;
      return;
    }
  }

  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, 2);  // both MMA issuers
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_k_empty[s], 2);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_v_empty[s], 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_o_free[x], 256);  // every softmax thread
      mbar_init(&bar_final[x], 1);
      mbar_init(&bar_turn[x], 1);
      mbar_init(&bar_s_full[x], 1);
      mbar_init(&bar_p_full[x], 256);
      for (int q = 0; q < 4; ++q) mbar_init(&bar_xch[x][q], 2);  // lane 0 of each warp of the pair
      mbar_init(&bar_pv_done[x], 1);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&bar_item_full[s], 1);      // the producer thread
      mbar_init(&bar_item_empty[s], 2 + 8);  // both MMA warps and each softmax warp
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
  constexpr uint32_t kTileBytes = S::kTile;

  // Register reallocation inside each role (a softmax thread holds a whole
  // 128-key row of S in registers).
  if (warp >= 8) {
    // warpgroup 2 hands registers to the softmax groups; warp 11 idles
    regs_dec<kRegsOther>();
    if (warp == kTmaWarp) {
      // ------------------------------------------------------------ producer
      uint32_t kv_it = 0, q_it = 0;
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
          const unsigned long long t = p.sched ? atomicAdd(p.sched, 1u)
                                               : blockIdx.x + static_cast<unsigned long long>(it) * gridDim.x;
          item_s[slot] = t < static_cast<unsigned long long>(p.total_items) ? static_cast<int>(t) : -1;
          mbar_arrive(&bar_item_full[slot]);
        }
        __syncwarp();
        const long long w = item_s[slot];
        if (w < 0) break;
        const int tile = p.q_order[w % p.n_pairs];
        const int h = static_cast<int>(w / p.n_pairs);
        const int b = tile / nP, pp = tile % nP;
        const int n = p.row_count[tile];
        if (n == 0) continue;
        const int32_t* list = p.row_list + static_cast<size_t>(tile) * nK;
        if (!wait1(&bar_q_empty, (q_it & 1) ^ 1, kSiteQEmpty)) { alive = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_q_full, 2 * kTileBytes);
  #pragma unroll
          for (int x = 0; x < 2; ++x)
  #pragma unroll
            for (int s = 0; s < D / 64; ++s)
              tma_load_4d(smem + S::kQ + x * kTileBytes + s * 16384, &tmap_q, &bar_q_full, s * 64, h,
                          pp * 256 + x * 128, b);
        }
        __syncwarp();
        ++q_it;
        for (int j = 0; j < n; ++j, ++kv_it) {
          const int kt = list[j];
          const int st = kv_it % kStages;
          const uint32_t ph = ((kv_it / kStages) & 1) ^ 1;
          if (!wait1(&bar_k_empty[st], ph, kSiteKEmpty)) { alive = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar_k_full[st], kTileBytes);
  #pragma unroll
            for (int s = 0; s < D / 64; ++s)
              tma_load_4d(smem + S::kK + st * kTileBytes + s * 16384, &tmap_k, &bar_k_full[st], s * 64, h, kt * 128, b);
          }
          __syncwarp();
          if (!wait1(&bar_v_empty[st], ph, kSiteVEmpty)) { alive = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar_v_full[st], kTileBytes);
  #pragma unroll
            for (int s = 0; s < D / 64; ++s)
              tma_load_4d(smem + S::kV + st * kTileBytes + s * 16384, &tmap_v, &bar_v_full[st], s * 64, h, kt * 128, b);
          }
          __syncwarp();
        }
      }
      if (abort_s && lane == 0) {
        // let copies still in flight land before the CTA leaves
        if (q_it > 0) mbar_drain(&bar_q_full, (q_it - 1) & 1, 100000000ull);
        for (uint32_t it = kv_it > kStages ? kv_it - kStages : 0; it <= kv_it; ++it) {
          mbar_drain(&bar_k_full[it % kStages], (it / kStages) & 1, 100000000ull);
          mbar_drain(&bar_v_full[it % kStages], (it / kStages) & 1, 100000000ull);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarpB) {
      // -------------------------------------------------------- MMA issuers
      // Warp 9 issues the brackets of query tile A (S_A of the item's first
      // key tile, then PV_A(j), S_A(j+1) for each j), warp 10 those of tile B.
      // A turn token makes them strictly alternate A, B, A, B, ..., so the
      // tensor core still runs one tile's MMAs while the other tile's softmax
      // runs; each issuer tests its own gates while the other one issues,
      // which takes the gate tests and barrier round trips off the tensor
      // core's path.  K and V stages and the Q pair are released by both
      // issuers (barrier counts of 2).
      const int x = warp == kMmaWarp ? 0 : 1;
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, D, false, true);
      uint32_t kv_it = 0, q_it = 0, p_it = 0, o_it = 0, turn_it = 0;
      bool alive = true;
      // All lanes wait (no divergence to rejoin); one lane issues.
      auto wait1 = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, site));
      };
      // this issuer's turn: tile A's k-th bracket follows tile B's (k-1)-th,
      // tile B's k-th follows tile A's k-th
      auto wait_turn = [&]() {
        const uint32_t parity = x == 0 ? (turn_it & 1) ^ 1 : (turn_it & 1);
        return wait1(&bar_turn[x], parity, kSiteTurn);
      };
      auto pass_turn = [&]() {
        ++turn_it;
        if (lane == 0) mbar_arrive(&bar_turn[x ^ 1]);
        __syncwarp();
      };
      const uint32_t qbase = sQ + x * kTileBytes;
      // The K steps [k0, k1) of S_x = Q_x K^T (K stage of key tile idx).
      auto issue_s = [&](uint32_t idx, int k0, int k1) {
        const uint32_t kbase = sK0 + (idx % kStages) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          if (kk >= k0 && kk < k1)
            umma_ss(tmem + kColS + x * 128, kmajor_desc(qbase, kk), kmajor_desc(kbase, kk), idesc_s, kk > 0 ? 1u : 0u);
      };
      auto commit_s = [&](uint32_t idx) {
        umma_commit(&bar_s_full[x]);
        umma_commit(&bar_k_empty[idx % kStages]);
      };
      // The K steps [k0, k1) of O_x += P_x V (P_x in TMEM).
      auto issue_pv = [&](uint32_t idx, bool accumulate, int k0, int k1) {
        const uint32_t vbase = sV0 + (idx % kStages) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk >= k0 && kk < k1)
            umma_ts(tmem + kColO + x * D, tmem + kColS + x * 128 + kk * 8, mnmajor_desc(vbase, kk), idesc_o,
                    (accumulate || kk > 0) ? 1u : 0u);
      };
      auto commit_pv = [&](uint32_t idx) {
        umma_commit(&bar_pv_done[x]);
        umma_commit(&bar_v_empty[idx % kStages]);
      };
      for (uint32_t it = 0; alive; ++it) {
        const int slot = it % kItemSlots;
        if (!wait1(&bar_item_full[slot], (it / kItemSlots) & 1, kSiteItemFull)) { alive = false; break; }
        const long long w = item_s[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_item_empty[slot]);
        if (w < 0) break;
        const int tile = p.q_order[w % p.n_pairs];
        const int n = p.row_count[tile];
        if (n == 0) continue;
        if (!wait1(&bar_q_full, q_it & 1, kSiteQFull)) { alive = false; break; }
        ++q_it;
        const uint32_t base = kv_it;
        if (!wait1(&bar_k_full[base % kStages], (base / kStages) & 1, kSiteKFull)) { alive = false; break; }
        if (!wait_turn()) { alive = false; break; }
        tc_fence_after();
        if (lane == 0) {
          issue_s(base, 0, D / 16);
          commit_s(base);
        }
        __syncwarp();
        pass_turn();
        for (int j = 0; j < n; ++j) {
          const uint32_t idx = base + j;
          const bool more = j + 1 < n;
          // Everything PV_x(j) and S_x(j+1) need: V(j), P_x(j), O_x free
          // (first key tile), K(j+1).  Usually all are there already: test
          // them at once and fall back to the waits one by one.
          const uint32_t pv = (idx / kStages) & 1, pk = ((idx + 1) / kStages) & 1;
          const bool ready = mbar_try_wait(&bar_v_full[idx % kStages], pv) & mbar_try_wait(&bar_p_full[x], p_it & 1) &
                             (j > 0 || mbar_try_wait(&bar_o_free[x], (o_it & 1) ^ 1)) &
                             (!more || mbar_try_wait(&bar_k_full[(idx + 1) % kStages], pk));
          if (!__all_sync(0xffffffffu, ready)) {
            if (!wait1(&bar_v_full[idx % kStages], pv, kSiteVFull)) { alive = false; break; }
            if (!wait1(&bar_p_full[x], p_it & 1, kSitePFull)) { alive = false; break; }
            if (j == 0 && !wait1(&bar_o_free[x], (o_it & 1) ^ 1, kSiteOFree)) { alive = false; break; }
            if (more && !wait1(&bar_k_full[(idx + 1) % kStages], pk, kSiteKFull)) { alive = false; break; }
          }
          if (j == 0) ++o_it;
          ++p_it;
          if (!wait_turn()) { alive = false; break; }
          tc_fence_after();
          // An MMA issue returns only once the tensor core has taken the
          // instruction, near the end of the work queued before it.  The turn
          // goes to the other issuer while the last kTurnEarly MMAs of this
          // bracket are still to be issued: they are queued well before the
          // other issuer wakes up, so its bracket follows without a gap.
          if (lane == 0) {
            if (more) {
              issue_pv(idx, j > 0, 0, 8);
              commit_pv(idx);
              issue_s(idx + 1, 0, D / 16 - kTurnEarly);
            } else {
              issue_pv(idx, j > 0, 0, 8 - kTurnEarly);
            }
          }
          __syncwarp();
          pass_turn();
          if (lane == 0) {
            if (more) {
              issue_s(idx + 1, D / 16 - kTurnEarly, D / 16);
              commit_s(idx + 1);
            } else {
              issue_pv(idx, j > 0, 8 - kTurnEarly, 8);
              commit_pv(idx);
            }
          }
          __syncwarp();
        }
        kv_it = base + n;
        if (!alive) break;
        if (lane == 0) umma_commit(&bar_q_empty);
        __syncwarp();
      }
      if (!alive && lane == 0) mbar_arrive(&bar_turn[x ^ 1]);  // let the other issuer notice the abort
      // every MMA issued by this thread has finished before TMEM is released
      if (lane == 0) {
        umma_commit(&bar_final[x]);
        mbar_drain(&bar_final[x], 0, 100000000ull);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------- softmax
    // Both warpgroups work on each query tile, tile A then tile B of each key
    // tile: warp w holds rows 32 (w % 4) .. + 31 (its TMEM lanes) and key
    // half hf = w / 4 of them, so that two warps share each SM sub-partition
    // and one's FMA work fills the other's waits for the exponential unit.
    // The two warps of a pair swap partial row maxima through shared memory
    // (an mbarrier pair wait, bounded) and agree on the running max.
    regs_inc<kRegsSoftmax>();
    const int hf = warp >> 2;            // key half: columns [64 hf, 64 hf + 64) of S
    const int q4 = warp & 3;             // lane quarter
    const int row = threadIdx.x & 127;   // query row inside the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    constexpr int kHalfD = D / 2;        // O columns of this half
    uint32_t s_it = 0, pv_it = 0;
    uint32_t xc_it[2] = {0u, 0u};        // exchanges per tile
    bool alive = true;
    auto waitw = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl, site));
    };
    // publish v for the partner warp and return the partner's value
    auto swap = [&](int x, float v, float& other) {
      const uint32_t slot = xc_it[x] & 1;
      xch_s[x][slot][hf][row] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_xch[x][q4]);
      if (!waitw(&bar_xch[x][q4], slot, kSiteXch)) return false;
      other = xch_s[x][slot][hf ^ 1][row];
      ++xc_it[x];
      return true;
    };
    for (uint32_t it = 0; alive; ++it) {
      const int slot = it % kItemSlots;
      if (!waitw(&bar_item_full[slot], (it / kItemSlots) & 1, kSiteItemFull)) { alive = false; break; }
      const long long w = item_s[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_item_empty[slot]);
      if (w < 0) break;
      const int tile = p.q_order[w % p.n_pairs];
      const int h = static_cast<int>(w / p.n_pairs);
      const int b = tile / nP, pp = tile % nP;
      const int n = p.row_count[tile];
      if (n == 0) {  // no valid query in this pair of tiles
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int qpos = pp * 256 + x * 128 + row;
          if (qpos < p.Lq) {
            __nv_bfloat16* orow = p.o + ((static_cast<size_t>(b) * p.Lq + qpos) * p.H + h) * D + hf * kHalfD;
#pragma unroll
            for (int c = 0; c < kHalfD / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
            if (hf == 0) p.lse[(static_cast<size_t>(b) * p.H + h) * p.Lq + qpos] = -INFINITY;
          }
        }
        continue;
      }
      const int nfull = p.row_full[tile];
      const int32_t* list = p.row_list + static_cast<size_t>(tile) * nK;
      const int32_t* seq_row = p.k_seq + static_cast<size_t>(b) * p.Lk;  // key ids of this row
      int my_seq[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int qpos = pp * 256 + x * 128 + row;
        my_seq[x] = qpos < p.Lq ? p.q_seq[static_cast<size_t>(b) * p.Lq + qpos] : -1;
      }
      float m_ref[2] = {-INFINITY, -INFINITY};  // running max of scale*log2(e)*s, per tile
      float l[2] = {0.0f, 0.0f};                // this half's running sum of 2^(...) relative to m_ref
      for (int j = 0; j < n && alive; ++j) {
        const bool partial = j >= nfull;
        const int kt = partial ? list[j] : 0;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const uint32_t s_col = tmem + lane_base + kColS + x * 128;
          if (!waitw(&bar_s_full[x], s_it & 1, kSiteSFull)) { alive = false; break; }
          tc_fence_after();
          // this half of the S row into registers (PARTIAL tiles: inadmissible keys -> -inf)
          uint32_t srow[2][32];
          float mh;
          if (!partial) mh = load_half_row<false>(s_col, hf, srow, seq_row, p.Lk, kt, my_seq[x]);
          else mh = load_half_row<true>(s_col, hf, srow, seq_row, p.Lk, kt, my_seq[x]);
          // the partner has loaded its half too once the swap completes, so
          // P may then be written over S columns [0, 64)
          float mo;
          if (!swap(x, mh, mo)) { alive = false; break; }
          const float mx2 = fmaxf(mh, mo) * p.scale_log2;
          const bool grow = mx2 > m_ref[x] + kRescaleThreshold;
          const float m_new = grow ? mx2 : m_ref[x];
          const float alpha = grow ? ex2(m_ref[x] - m_new) : 1.0f;
          const bool any = m_new != -INFINITY;
          const float neg_m = any ? -m_new : 0.0f;
          // P = 2^(scale*log2e*S - m), packed bf16 over S columns [32 hf, 32 hf + 32)
          const float lsum = exp_store_half(s_col, hf, srow, p.scale_log2, neg_m);
          l[x] = l[x] * alpha + lsum;
          // PV_x of the previous key tile has completed: S_x of this tile was
          // issued after it by the same thread, and the commit that completed
          // s_full tracks every earlier MMA of that thread, so its pv_done
          // phase needs no wait of its own (only the item's last one is waited
          // for, before the epilogue).  Rescale this half's O_x columns when
          // the max grew.
          if (j > 0) {
            const bool rescale = grow && m_ref[x] != -INFINITY;
            if (__any_sync(0xffffffffu, rescale)) {
              const float f = rescale ? alpha : 1.0f;
              const uint32_t o_col = tmem + lane_base + kColO + x * D + hf * kHalfD;
#pragma unroll
              for (int c = 0; c < kHalfD / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(o_col + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
                tmem_st32(o_col + c * 32, r);
              }
            }
          }
          m_ref[x] = m_new;
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar_p_full[x]);
        }
        if (!alive) break;
        ++s_it;
        if (j > 0) ++pv_it;
      }
      if (!alive) break;
      // epilogues: the last PV_x has finished
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (!waitw(&bar_pv_done[x], pv_it & 1, kSitePvDone)) { alive = false; break; }
        tc_fence_after();
        float lo;
        if (!swap(x, l[x], lo)) { alive = false; break; }
        const float lt = l[x] + lo;
        const float inv_l = lt > 0.0f ? 1.0f / lt : 0.0f;
        const int qpos = pp * 256 + x * 128 + row;
        const bool in_range = qpos < p.Lq;
        __nv_bfloat16* orow = p.o + ((static_cast<size_t>(b) * p.Lq + qpos) * p.H + h) * D + hf * kHalfD;
        const uint32_t o_col = tmem + lane_base + kColO + x * D + hf * kHalfD;
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(o_col + c * 32, r);
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
        mbar_arrive(&bar_o_free[x]);
        if (in_range && hf == 0)
          p.lse[(static_cast<size_t>(b) * p.H + h) * p.Lq + qpos] =
              lt > 0.0f ? (m_ref[x] + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
      }
      if (!alive) break;
      ++pv_it;
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
pvl_status launch_fwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const int32_t* q_seq,
                      const int32_t* k_seq, const void* tile_ws, int B, int Lq, int Lk, int H, float scale,
                      pvl_bf16* o, float* lse, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  pvl_status st = make_bhld_tensor_map(&tq, q, B, Lq, H, D);
  if (st == PVL_OK) st = make_bhld_tensor_map(&tk, k, B, Lk, H, D);
  if (st == PVL_OK) st = make_bhld_tensor_map(&tv, v, B, Lk, H, D);
  if (st != PVL_OK) return st;
  DeviceError* err = device_error_record();
  const int sms = sm_count();
  if (!err || sms <= 0) return fail(PVL_ERR_CUDA, "masked_attn_fwd: no usable CUDA device");
  const TileMapView tm = tile_map_view(tile_ws, B, Lq, Lk, 128, 128, 1);  // pairs of query tiles
  FwdParams prm;
  prm.q_seq = q_seq;
  prm.k_seq = k_seq;
  prm.header = tm.header;
  prm.row_count = tm.row_count;
  prm.row_full = tm.row_full;
  prm.row_list = tm.row_list;
  prm.q_order = tm.q_order;
  prm.o = reinterpret_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.err = err;
  prm.B = B;
  prm.Lq = Lq;
  prm.Lk = Lk;
  prm.H = H;
  prm.nP = tm.nTq;
  prm.nK = tm.nTk;
  prm.n_pairs = B * tm.nTq;
  prm.total_items = static_cast<long long>(prm.n_pairs) * H;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.timeout_ns = attn_wait_timeout_ns();
  prm.sched = fwd_sched_counter(stream);
  if (prm.sched) {
    st = check_cuda(cudaMemsetAsync(prm.sched, 0, sizeof(unsigned int), stream), "masked_attn_fwd counter reset");
    if (st != PVL_OK) return st;
  }
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

extern "C" pvl_status masked_attn_fwd_cross(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v,
                                            const int32_t* q_seq_id, const int32_t* k_seq_id, const void* tile_ws,
                                            int B, int Lq, int Lk, int H, int D, float scale, pvl_bf16* o,
                                            float* lse, pvl_stream_t stream) {
  const void* ptrs[] = {q, k, v, q_seq_id, k_seq_id, tile_ws, o, lse};
  const pvl_status st = validate_attn_qk("masked_attn_fwd", ptrs, 8, B, Lq, Lk, H, D, scale);
  if (st != PVL_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 64) return launch_fwd<64>(q, k, v, q_seq_id, k_seq_id, tile_ws, B, Lq, Lk, H, scale, o, lse, s);
  return launch_fwd<128>(q, k, v, q_seq_id, k_seq_id, tile_ws, B, Lq, Lk, H, scale, o, lse, s);
}

extern "C" pvl_status masked_attn_fwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const int32_t* seq_id,
                                      const void* tile_ws, int B, int L, int H, int D, float scale, pvl_bf16* o,
                                      float* lse, pvl_stream_t stream) {
  return masked_attn_fwd_cross(q, k, v, seq_id, seq_id, tile_ws, B, L, L, H, D, scale, o, lse, stream);
}
