// masked_attn_bwd (kernels to come).
#include <cuda_runtime.h>

#include "pvl_internal.h"

using namespace pvl;

extern "C" size_t masked_attn_bwd_ws_bytes(int B, int L, int H, int D) {
  if (B < 1 || L < 1 || H < 1 || D < 1) return 0;
  return bwd_ws_total_bytes(B, L, H, D);
}

extern "C" pvl_status masked_attn_bwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const pvl_bf16* o,
                                      const pvl_bf16* dO, const float* lse, const int32_t* seq_id,
                                      const void* tile_ws, int B, int L, int H, int D, float scale, pvl_bf16* dq,
                                      pvl_bf16* dk, pvl_bf16* dv, void* ws, size_t ws_bytes, pvl_stream_t stream) {
  const void* ptrs[] = {q, k, v, o, dO, lse, seq_id, tile_ws, dq, dk, dv, ws};
  if (ws && ws_bytes < masked_attn_bwd_ws_bytes(B, L, H, D))
    return fail(PVL_ERR_INVALID_ARG, "masked_attn_bwd: workspace %zu bytes < %zu needed", ws_bytes,
                masked_attn_bwd_ws_bytes(B, L, H, D));
  pvl_status st = validate_attn("masked_attn_bwd", ptrs, 12, B, L, H, D, scale);
  if (st != PVL_OK) return st;
  (void)stream;
  return fail(PVL_ERR_UNSUPPORTED, "masked_attn_bwd: not built yet");
}
