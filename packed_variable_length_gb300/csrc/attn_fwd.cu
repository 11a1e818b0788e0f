// masked_attn_fwd (kernel to come).
#include <cuda_runtime.h>

#include "pvl_internal.h"

using namespace pvl;

extern "C" pvl_status masked_attn_fwd(const pvl_bf16* q, const pvl_bf16* k, const pvl_bf16* v, const int32_t* seq_id,
                                      const void* tile_ws, int B, int L, int H, int D, float scale, pvl_bf16* o,
                                      float* lse, pvl_stream_t stream) {
  const void* ptrs[] = {q, k, v, seq_id, tile_ws, o, lse};
  pvl_status st = validate_attn("masked_attn_fwd", ptrs, 7, B, L, H, D, scale);
  if (st != PVL_OK) return st;
  (void)stream;
  return fail(PVL_ERR_UNSUPPORTED, "masked_attn_fwd: not built yet");
}
