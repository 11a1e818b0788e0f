// tile_map_build: classify every (query tile, key tile) pair of the seq_id
// mask as EMPTY / PARTIAL / FULL and compact the non-empty pairs into
// per-tile work lists plus a longest-first order of the tiles.
//
// "lingbot_va_packing" §2.1-§2.2: FlexAttention derives a block mask from the
// seq_ids and skips blocks with no admissible pair.  Here the map (both of
// its levels at once) is built by three small kernels on the caller's
// stream:
//   1. tile_stats:  per tile, count / min / max of the valid ids;
//   2. tile_lists:  one warp per query tile (and per key tile) classifies its
//                   pairs from the stats and compacts FULL then PARTIAL
//                   indices with ballots;
//   3. tile_order:  bitonic sort of (count desc, index asc): in registers with
//                   warp shuffles for partners less than 32 apart when every
//                   thread holds one key, else in shared memory.
#include <cuda_runtime.h>

#include <algorithm>

#include "pvl_internal.h"

namespace pvl {
namespace {

struct TileMapPtrs {
  int32_t* header;
  int32_t *q_nv, *q_lo, *q_hi, *k_nv, *k_lo, *k_hi;
  uint8_t* cls;
  int32_t *row_count, *row_full, *row_list, *col_count, *col_full, *col_list, *q_order, *k_order;
};

TileMapPtrs tile_map_ptrs(void* ws, const TileMapLayout& t) {
  char* p = static_cast<char*>(ws);
  auto i32 = [&](int f) { return reinterpret_cast<int32_t*>(p + t.off[f]); };
  TileMapPtrs r;
  r.header = i32(PVL_TM_HEADER);
  r.q_nv = i32(PVL_TM_Q_NV);
  r.q_lo = i32(PVL_TM_Q_LO);
  r.q_hi = i32(PVL_TM_Q_HI);
  r.k_nv = i32(PVL_TM_K_NV);
  r.k_lo = i32(PVL_TM_K_LO);
  r.k_hi = i32(PVL_TM_K_HI);
  r.cls = reinterpret_cast<uint8_t*>(p + t.off[PVL_TM_CLS]);
  r.row_count = i32(PVL_TM_ROW_COUNT);
  r.row_full = i32(PVL_TM_ROW_FULL);
  r.row_list = i32(PVL_TM_ROW_LIST);
  r.col_count = i32(PVL_TM_COL_COUNT);
  r.col_full = i32(PVL_TM_COL_FULL);
  r.col_list = i32(PVL_TM_COL_LIST);
  r.q_order = i32(PVL_TM_Q_ORDER);
  r.k_order = i32(PVL_TM_K_ORDER);
  return r;
}

constexpr int kStatThreads = 128;

// One level of the map: its arrays, tile sizes and tile counts.
struct TileLevel {
  TileMapPtrs m;
  int bm, nTq, nTk;
};
struct TileLevels {
  TileLevel lv[PVL_TM_LEVELS];
};

// grid (sum over levels of nTq + nTk, B), levels one after the other: in a
// level's range, blocks [0, nTq) summarise query tiles of bm positions over
// the query ids, the rest key tiles of bn positions over the key ids (the
// same array for self attention).
__global__ void __launch_bounds__(kStatThreads) tile_stats_kernel(const int32_t* __restrict__ q_seq,
                                                                  const int32_t* __restrict__ k_seq, int B, int Lq,
                                                                  int Lk, int bn, TileLevels levels) {
  int x = blockIdx.x, lvi = 0;
  while (lvi + 1 < PVL_TM_LEVELS && x >= levels.lv[lvi].nTq + levels.lv[lvi].nTk) {
    x -= levels.lv[lvi].nTq + levels.lv[lvi].nTk;
    ++lvi;
  }
  const TileMapPtrs& m = levels.lv[lvi].m;
  const int bm = levels.lv[lvi].bm, nTq = levels.lv[lvi].nTq, nTk = levels.lv[lvi].nTk;
  const int b = blockIdx.y;
  const bool is_q = x < nTq;
  const int t = is_q ? x : x - nTq;
  const int bs = is_q ? bm : bn;
  const int L = is_q ? Lq : Lk;
  const int32_t* seq_id = is_q ? q_seq : k_seq;
  int cnt = 0, lo = INT32_MAX, hi = INT32_MIN;
  for (int i = threadIdx.x; i < bs; i += kStatThreads) {
    const long long p = static_cast<long long>(t) * bs + i;
    if (p < L) {
      const int32_t s = seq_id[static_cast<size_t>(b) * L + p];
      if (s >= 0) {
        ++cnt;
        lo = min(lo, s);
        hi = max(hi, s);
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  __shared__ int s_cnt[kStatThreads / 32], s_lo[kStatThreads / 32], s_hi[kStatThreads / 32];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_cnt[w] = cnt;
    s_lo[w] = lo;
    s_hi[w] = hi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kStatThreads / 32; ++i) {
      cnt += s_cnt[i];
      lo = min(lo, s_lo[i]);
      hi = max(hi, s_hi[i]);
    }
    if (cnt == 0) lo = hi = 0;
    const int idx = b * (is_q ? nTq : nTk) + t;
    (is_q ? m.q_nv : m.k_nv)[idx] = cnt;
    (is_q ? m.q_lo : m.k_lo)[idx] = lo;
    (is_q ? m.q_hi : m.k_hi)[idx] = hi;
    if (x == 0 && b == 0) {
      m.header[0] = kTileMapMagic;
      m.header[1] = kTileMapVersion;
      m.header[2] = B;
      m.header[3] = Lq;
      m.header[4] = bm;
      m.header[5] = bn;
      m.header[6] = nTq;
      m.header[7] = nTk;
      m.header[8] = Lk;
      for (int i = 9; i < 16; ++i) m.header[i] = 0;
    }
  }
}

__device__ __forceinline__ uint8_t classify(int nvq, int loq, int hiq, int bm, int nvk, int lok, int hik, int bn) {
  if (nvq == 0 || nvk == 0 || hiq < lok || hik < loq) return kEmpty;
  if (loq == hiq && lok == hik && loq == lok && nvq == bm && nvk == bn) return kFull;
  return kPartial;
}

constexpr int kListWarps = 8;
constexpr int kGroup = 8;  // chunks of 32 classified per load round

// One warp per list, levels one after the other.  In a level's range, warps
// [0, B*nTq) own query tile rows (and write CLS), warps [B*nTq, B*nTq + B*nTk)
// own key tile columns.
__global__ void __launch_bounds__(kListWarps * 32) tile_lists_kernel(int B, int bn, TileLevels levels) {
  long long w = static_cast<long long>(blockIdx.x) * kListWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  int lvi = 0;
  while (lvi + 1 < PVL_TM_LEVELS &&
         w >= static_cast<long long>(B) * (levels.lv[lvi].nTq + levels.lv[lvi].nTk)) {
    w -= static_cast<long long>(B) * (levels.lv[lvi].nTq + levels.lv[lvi].nTk);
    ++lvi;
  }
  const TileMapPtrs& m = levels.lv[lvi].m;
  const int bm = levels.lv[lvi].bm, nTq = levels.lv[lvi].nTq, nTk = levels.lv[lvi].nTk;
  const long long nrows = static_cast<long long>(B) * nTq;
  const long long ncols = static_cast<long long>(B) * nTk;
  if (w >= nrows + ncols) return;
  const bool is_row = w < nrows;
  const int b = static_cast<int>(is_row ? w / nTq : (w - nrows) / nTk);
  const int t = static_cast<int>(is_row ? w % nTq : (w - nrows) % nTk);
  const int n_other = is_row ? nTk : nTq;
  // this tile's summary
  const int nv0 = is_row ? m.q_nv[b * nTq + t] : m.k_nv[b * nTk + t];
  const int lo0 = is_row ? m.q_lo[b * nTq + t] : m.k_lo[b * nTk + t];
  const int hi0 = is_row ? m.q_hi[b * nTq + t] : m.k_hi[b * nTk + t];
  int32_t* list = is_row ? m.row_list + (static_cast<size_t>(b) * nTq + t) * nTk
                         : m.col_list + (static_cast<size_t>(b) * nTk + t) * nTq;
  // the other side's summaries of this batch row
  const int32_t* o_nv = is_row ? m.k_nv + b * nTk : m.q_nv + b * nTq;
  const int32_t* o_lo = is_row ? m.k_lo + b * nTk : m.q_lo + b * nTq;
  const int32_t* o_hi = is_row ? m.k_hi + b * nTk : m.q_hi + b * nTq;
  int written = 0, nfull = 0;
  for (int pass = 0; pass < 2; ++pass) {
    const uint8_t want = pass == 0 ? kFull : kPartial;
    // kGroup chunks of 32 per step: their loads are issued together, so the
    // list pays one load latency per group instead of one per chunk
    for (int base0 = 0; base0 < n_other; base0 += 32 * kGroup) {
      int nv[kGroup], lo[kGroup], hi[kGroup];
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int o = base0 + 32 * u + lane;
        nv[u] = 0;
        lo[u] = hi[u] = 0;
        if (o < n_other) {
          nv[u] = __ldg(o_nv + o);
          lo[u] = __ldg(o_lo + o);
          hi[u] = __ldg(o_hi + o);
        }
      }
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const int o = base0 + 32 * u + lane;
        uint8_t c = kEmpty;
        if (o < n_other) {
          c = is_row ? classify(nv0, lo0, hi0, bm, nv[u], lo[u], hi[u], bn)
                     : classify(nv[u], lo[u], hi[u], bm, nv0, lo0, hi0, bn);
          if (is_row && pass == 0) m.cls[(static_cast<size_t>(b) * nTq + t) * nTk + o] = c;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, o < n_other && c == want);
        if (c == want && o < n_other) list[written + __popc(hit & ((1u << lane) - 1u))] = o;
        written += __popc(hit);
      }
    }
    if (pass == 0) nfull = written;
  }
  for (int o = written + lane; o < n_other; o += 32) list[o] = -1;
  if (lane == 0) {
    if (is_row) {
      m.row_count[b * nTq + t] = written;
      m.row_full[b * nTq + t] = nfull;
    } else {
      m.col_count[b * nTk + t] = written;
      m.col_full[b * nTk + t] = nfull;
    }
  }
}

constexpr int kOrderThreads = 1024;
constexpr int kIdxBits = 14;  // PVL_MAX_ORDER_TILES == 1 << 14

// Two blocks per level: block 2 lv sorts the level's query tiles, block
// 2 lv + 1 its key tiles.  Key = (PVL_MAX_ORDER_TILES - count) << 14 | index,
// ascending, so larger counts come first and ties keep ascending index;
// padding keys are 0xFFFFFFFF.
__global__ void __launch_bounds__(kOrderThreads) tile_order_kernel(int B, TileLevels levels) {
  extern __shared__ uint32_t keys[];
  const TileMapPtrs& m = levels.lv[blockIdx.x >> 1].m;
  const bool is_q = (blockIdx.x & 1) == 0;
  const int n = B * (is_q ? levels.lv[blockIdx.x >> 1].nTq : levels.lv[blockIdx.x >> 1].nTk);
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  const int32_t* cnt = is_q ? m.row_count : m.col_count;
  int32_t* out = is_q ? m.q_order : m.k_order;
  if (np2 <= kOrderThreads) {
    // one key per thread: partners less than 32 apart are in the same warp
    // (shuffles); only the wider stages go through shared memory
    const int i = threadIdx.x;
    uint32_t key = i < n ? (static_cast<uint32_t>(PVL_MAX_ORDER_TILES - cnt[i]) << kIdxBits) | static_cast<uint32_t>(i)
                         : 0xFFFFFFFFu;
    for (int k = 2; k <= np2; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        uint32_t other;
        if (j >= 32) {
          if (i < np2) keys[i] = key;
          __syncthreads();
          other = i < np2 ? keys[i ^ j] : 0xFFFFFFFFu;
          __syncthreads();
        } else {
          other = __shfl_xor_sync(0xffffffffu, key, j);
        }
        // the pair's lower index keeps the smaller key where the run ascends
        const bool ascending = (i & k) == 0;
        const bool lower = (i & j) == 0;
        key = (lower == ascending) ? min(key, other) : max(key, other);
      }
    }
    if (i < n) out[i] = static_cast<int32_t>(key & ((1u << kIdxBits) - 1u));
    return;
  }
  for (int i = threadIdx.x; i < np2; i += kOrderThreads)
    keys[i] = i < n ? (static_cast<uint32_t>(PVL_MAX_ORDER_TILES - cnt[i]) << kIdxBits) | static_cast<uint32_t>(i)
                    : 0xFFFFFFFFu;
  __syncthreads();
  for (int k = 2; k <= np2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < np2; i += kOrderThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint32_t a = keys[i], c = keys[ixj];
          const bool ascending = (i & k) == 0;
          if ((a > c) == ascending) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += kOrderThreads)
    out[i] = static_cast<int32_t>(keys[i] & ((1u << kIdxBits) - 1u));
}

int next_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

}  // namespace
}  // namespace pvl

using namespace pvl;

namespace pvl {
namespace {

pvl_status build_tile_map(const char* who, const int32_t* q_seq, const int32_t* k_seq, int B, int Lq, int Lk,
                          int block_m, int block_n, void* tile_ws, size_t ws_bytes, cudaStream_t s) {
  if (!q_seq || !k_seq || !tile_ws) return fail(PVL_ERR_INVALID_ARG, "%s: null pointer", who);
  if (B < 1 || Lq < 1 || Lk < 1) return fail(PVL_ERR_INVALID_ARG, "%s: B and the lengths must be >= 1", who);
  if (block_m < 1 || block_m > 1024 || block_n < 1 || block_n > 1024)
    return fail(PVL_ERR_UNSUPPORTED, "%s: block sizes must be in 1..1024", who);
  if (Lq > PVL_MAX_L || Lk > PVL_MAX_L)
    return fail(PVL_ERR_UNSUPPORTED, "%s: length %d exceeds %d", who, Lq > Lk ? Lq : Lk, PVL_MAX_L);
  if (reinterpret_cast<uintptr_t>(tile_ws) % 256 != 0)
    return fail(PVL_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  const TileMapLayouts all = tile_map_layouts(B, Lq, Lk, block_m, block_n);
  if (ws_bytes < all.total)
    return fail(PVL_ERR_INVALID_ARG, "%s: workspace %zu bytes < %zu needed", who, ws_bytes, all.total);
  const long long nq0 = static_cast<long long>(B) * all.level[0].nTq, nk0 = static_cast<long long>(B) * all.level[0].nTk;
  if (nq0 > PVL_MAX_ORDER_TILES || nk0 > PVL_MAX_ORDER_TILES)
    return fail(PVL_ERR_UNSUPPORTED, "%s: B * tiles = %lld exceeds %d", who, nq0 > nk0 ? nq0 : nk0,
                PVL_MAX_ORDER_TILES);
  TileLevels levels;
  int stat_blocks = 0;
  long long nwarps = 0, np2_max = 1;
  for (int lv = 0; lv < PVL_TM_LEVELS; ++lv) {
    const TileMapLayout& t = all.level[lv];
    levels.lv[lv].m = tile_map_ptrs(tile_ws, t);
    levels.lv[lv].bm = lv == 0 ? block_m : 2 * block_m;
    levels.lv[lv].nTq = t.nTq;
    levels.lv[lv].nTk = t.nTk;
    stat_blocks += t.nTq + t.nTk;
    nwarps += static_cast<long long>(B) * (t.nTq + t.nTk);
    np2_max = std::max<long long>(np2_max, next_pow2(B * std::max(t.nTq, t.nTk)));
  }
  tile_stats_kernel<<<dim3(stat_blocks, B), kStatThreads, 0, s>>>(q_seq, k_seq, B, Lq, Lk, block_n, levels);
  pvl_status st = check_cuda(cudaGetLastError(), "tile_stats launch");
  if (st != PVL_OK) return st;
  tile_lists_kernel<<<static_cast<unsigned>((nwarps + kListWarps - 1) / kListWarps), kListWarps * 32, 0, s>>>(
      B, block_n, levels);
  st = check_cuda(cudaGetLastError(), "tile_lists launch");
  if (st != PVL_OK) return st;
  const int smem = static_cast<int>(np2_max) * static_cast<int>(sizeof(uint32_t));
  if (smem > 48 * 1024) {
    st = check_cuda(cudaFuncSetAttribute(tile_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                    "tile_order smem attribute");
    if (st != PVL_OK) return st;
  }
  tile_order_kernel<<<2 * PVL_TM_LEVELS, kOrderThreads, smem, s>>>(B, levels);
  st = check_cuda(cudaGetLastError(), "tile_order launch");
  if (st != PVL_OK) return st;
  return PVL_OK;
}

pvl_status layout_offsets(const char* who, int B, int Lq, int Lk, int block_m, int block_n, size_t* offsets) {
  if (!offsets) return fail(PVL_ERR_INVALID_ARG, "%s: null offsets", who);
  if (B < 1 || Lq < 1 || Lk < 1 || block_m < 1 || block_n < 1)
    return fail(PVL_ERR_INVALID_ARG, "%s: sizes must be >= 1", who);
  const TileMapLayouts t = tile_map_layouts(B, Lq, Lk, block_m, block_n);
  for (int lv = 0; lv < PVL_TM_LEVELS; ++lv)
    for (int i = 0; i < PVL_TM_NFIELDS; ++i) offsets[lv * PVL_TM_NFIELDS + i] = t.level[lv].off[i];
  return PVL_OK;
}

}  // namespace
}  // namespace pvl

extern "C" size_t tile_map_ws_bytes(int B, int L, int block_m, int block_n) {
  return tile_map_ws_bytes_cross(B, L, L, block_m, block_n);
}

extern "C" size_t tile_map_ws_bytes_cross(int B, int Lq, int Lk, int block_m, int block_n) {
  if (B < 1 || Lq < 1 || Lk < 1 || block_m < 1 || block_n < 1) return 0;
  return tile_map_layouts(B, Lq, Lk, block_m, block_n).total;
}

extern "C" pvl_status tile_map_layout(int B, int L, int block_m, int block_n, size_t* offsets) {
  return layout_offsets("tile_map_layout", B, L, L, block_m, block_n, offsets);
}

extern "C" pvl_status tile_map_layout_cross(int B, int Lq, int Lk, int block_m, int block_n, size_t* offsets) {
  return layout_offsets("tile_map_layout_cross", B, Lq, Lk, block_m, block_n, offsets);
}

extern "C" pvl_status tile_map_build(const int32_t* seq_id, int B, int L, int block_m, int block_n, void* tile_ws,
                                     size_t ws_bytes, pvl_stream_t stream) {
  return build_tile_map("tile_map_build", seq_id, seq_id, B, L, L, block_m, block_n, tile_ws, ws_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}

extern "C" pvl_status tile_map_build_cross(const int32_t* q_seq_id, const int32_t* k_seq_id, int B, int Lq, int Lk,
                                           int block_m, int block_n, void* tile_ws, size_t ws_bytes,
                                           pvl_stream_t stream) {
  return build_tile_map("tile_map_build_cross", q_seq_id, k_seq_id, B, Lq, Lk, block_m, block_n, tile_ws, ws_bytes,
                        reinterpret_cast<cudaStream_t>(stream));
}
