// Internal definitions shared by the host entry points and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "pvl.h"

#ifdef __CUDACC__
#define PVL_HD __host__ __device__
#else
#define PVL_HD
#endif

namespace pvl {

// ------------------------------------------------------------ device errors
constexpr uint32_t kDevErrTimeout = 1;  // a bounded wait ran out
constexpr uint32_t kDevErrTileMap = 2;  // tile map header does not match the call

struct DeviceError {
  unsigned int code;
  unsigned int where;
  unsigned int block;
  unsigned int thread;
};

// Default bound on any single device-side wait.
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

// --------------------------------------------------------- tile map layout
constexpr int32_t kTileMapMagic = 0x544C5650;  // "PVLT"
constexpr int32_t kTileMapVersion = 2;  // header: magic, version, B, Lq, bm, bn, nTq, nTk, Lk
constexpr uint8_t kEmpty = 0, kPartial = 1, kFull = 2;

PVL_HD inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct TileMapLayout {
  size_t off[PVL_TM_NFIELDS];  // absolute byte offsets inside the workspace
  size_t total;                // end of this level
  int nTq, nTk;
};

// One level of the map (block sizes bm x bn) of Lq queries against Lk keys,
// starting at byte `base`.
PVL_HD inline TileMapLayout tile_map_level_layout(int B, int Lq, int Lk, int bm, int bn, size_t base) {
  TileMapLayout t{};
  t.nTq = (Lq + bm - 1) / bm;
  t.nTk = (Lk + bn - 1) / bn;
  const size_t nq = static_cast<size_t>(B) * t.nTq;
  const size_t nk = static_cast<size_t>(B) * t.nTk;
  const size_t nqk = nq * t.nTk;
  size_t sizes[PVL_TM_NFIELDS];
  sizes[PVL_TM_HEADER] = 16 * 4;
  sizes[PVL_TM_Q_NV] = sizes[PVL_TM_Q_LO] = sizes[PVL_TM_Q_HI] = nq * 4;
  sizes[PVL_TM_K_NV] = sizes[PVL_TM_K_LO] = sizes[PVL_TM_K_HI] = nk * 4;
  sizes[PVL_TM_CLS] = nqk;
  sizes[PVL_TM_ROW_COUNT] = sizes[PVL_TM_ROW_FULL] = nq * 4;
  sizes[PVL_TM_ROW_LIST] = nqk * 4;
  sizes[PVL_TM_COL_COUNT] = sizes[PVL_TM_COL_FULL] = nk * 4;
  sizes[PVL_TM_COL_LIST] = nqk * 4;
  sizes[PVL_TM_Q_ORDER] = nq * 4;
  sizes[PVL_TM_K_ORDER] = nk * 4;
  size_t pos = base;
  for (int i = 0; i < PVL_TM_NFIELDS; ++i) {
    t.off[i] = pos;
    pos = align256(pos + sizes[i]);
  }
  t.total = pos;
  return t;
}

// The workspace holds PVL_TM_LEVELS maps: level 0 at (bm, bn), level 1 at
// (2 bm, bn) -- the query-tile pairs the forward kernel processes together.
struct TileMapLayouts {
  TileMapLayout level[PVL_TM_LEVELS];
  size_t total;
};

PVL_HD inline TileMapLayouts tile_map_layouts(int B, int Lq, int Lk, int bm, int bn) {
  TileMapLayouts r{};
  r.level[0] = tile_map_level_layout(B, Lq, Lk, bm, bn, 0);
  r.level[1] = tile_map_level_layout(B, Lq, Lk, 2 * bm, bn, r.level[0].total);
  r.total = r.level[1].total;
  return r;
}

// Read-only view of one level of a tile map.
struct TileMapView {
  const int32_t* header;
  const uint8_t* cls;
  const int32_t* row_count;
  const int32_t* row_full;
  const int32_t* row_list;
  const int32_t* col_count;
  const int32_t* col_full;
  const int32_t* col_list;
  const int32_t* q_order;
  const int32_t* k_order;
  int nTq, nTk;
};

inline TileMapView tile_map_view(const void* ws, int B, int Lq, int Lk, int bm, int bn, int level) {
  const TileMapLayout t = tile_map_layouts(B, Lq, Lk, bm, bn).level[level];
  const char* p = static_cast<const char*>(ws);
  TileMapView v;
  v.header = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_HEADER]);
  v.cls = reinterpret_cast<const uint8_t*>(p + t.off[PVL_TM_CLS]);
  v.row_count = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_ROW_COUNT]);
  v.row_full = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_ROW_FULL]);
  v.row_list = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_ROW_LIST]);
  v.col_count = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_COL_COUNT]);
  v.col_full = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_COL_FULL]);
  v.col_list = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_COL_LIST]);
  v.q_order = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_Q_ORDER]);
  v.k_order = reinterpret_cast<const int32_t*>(p + t.off[PVL_TM_K_ORDER]);
  v.nTq = t.nTq;
  v.nTk = t.nTk;
  return v;
}

// ------------------------------------------------------- host-side helpers
// Implemented in pvl_runtime.cu.
pvl_status fail(pvl_status s, const char* fmt, ...);
pvl_status check_cuda(int err, const char* what);  // err is a cudaError_t
DeviceError* device_error_record();                // current device, null on failure
int sm_count();                                    // current device, 0 on failure
// Bound on any single wait of the attention kernels launched now
// (kDefaultTimeoutNs unless pvl_set_attn_wait_timeout_ns changed it).
uint64_t attn_wait_timeout_ns();
// Device address of the forward's work-item counter for `stream` on the
// current device: one slot per (device, stream), so that calls on one stream
// (ordered) share it and calls on different streams do not.  The forward
// zeroes it on the stream before each launch.  Null when the slots are all
// taken (the forward then hands out its items in a fixed round-robin).
unsigned int* fwd_sched_counter(void* stream);
// Events (cudaEvent_t) to record just before and just after the main
// backward kernel of the calling thread's next backward call, set by
// pvl_mark_next_bwd_main; handing them out clears them.
void take_bwd_main_marks(void** before, void** after);

// Shared argument checks of the attention calls: null pointers and sizes
// (INVALID_ARG), D, alignment and limits (UNSUPPORTED).
pvl_status validate_attn(const char* who, const void* const* ptrs, int nptrs, int B, int L, int H, int D, float scale);
// The same for Lq queries against Lk keys (the query-side checks use Lq).
pvl_status validate_attn_qk(const char* who, const void* const* ptrs, int nptrs, int B, int Lq, int Lk, int H, int D,
                            float scale);

// Backward workspace, each part 256-byte aligned: the fp32 dQ accumulator
// [B, L, H, D]; then, over query positions padded to whole 128-row tiles
// (Lp), Delta and LSE * log2(e) as fp32 [B, H, Lp] and the query seq_ids as
// int32 [B, Lp] (padding positions hold 0, 0 and -1); then the main
// kernel's work-item counter (one uint32, zeroed by the preprocess).
inline int bwd_lp(int L) { return ((L + 127) / 128) * 128; }
inline size_t bwd_ws_dq_bytes(int B, int L, int H, int D) {
  return align256(static_cast<size_t>(B) * L * H * D * 4);
}
inline size_t bwd_ws_rows_bytes(int B, int L, int H) {
  return align256(static_cast<size_t>(B) * H * bwd_lp(L) * 4);
}
inline size_t bwd_ws_sched_offset(int B, int L, int H, int D) {
  return bwd_ws_dq_bytes(B, L, H, D) + 2 * bwd_ws_rows_bytes(B, L, H) +
         align256(static_cast<size_t>(B) * bwd_lp(L) * 4);
}
inline size_t bwd_ws_total_bytes(int B, int L, int H, int D) { return bwd_ws_sched_offset(B, L, H, D) + 256; }

// bf16 [B, L, H, D] tensor map with a (64 x 1 x 128 x 1) box and 128-byte
// swizzle: one box is 128 rows of 64 features (16 KB).
pvl_status make_bhld_tensor_map(void* map_out /* CUtensorMap* */, const void* base, int B, int L, int H,
                                int D);

// fp32 [B, L, H, D] tensor map with a (box_d x 1 x box_rows x 1) box, for TMA
// reductions.  A 128-byte box row (box_d = 32) takes the 128-byte swizzle; a
// narrower one none (rows of box_d floats, packed).
pvl_status make_bhld_f32_tensor_map(void* map_out /* CUtensorMap* */, const void* base, int B, int L, int H, int D,
                                    int box_d, int box_rows);

}  // namespace pvl
