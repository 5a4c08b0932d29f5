// Host-side entry points that launch nothing: workspace sizing and version.
#include <cuda_runtime.h>

#include "m3s_score_common.cuh"

namespace {
size_t round16(size_t n) { return (n + 15) & ~static_cast<size_t>(15); }
}  // namespace

extern "C" size_t m3s_workspace_bytes(int op, int32_t R, int32_t B, int32_t max_blocks, int32_t Hq,
                                      int32_t Hkv, int32_t Hi, int32_t topk, int32_t max_q) {
  (void)Hi;
  (void)Hq;
  (void)Hkv;
  if (R <= 0 || topk <= 0) return 0;
  // more tiles than the calls take: they return M3S_ERR_UNSUPPORTED before
  // they look at the workspace, so there is no size to give
  const bool index_tiles_ok = R <= m3s::kMaxTiles;   // index ops: a tile per row
  switch (op) {
    case M3S_OP_INDEX_CANDIDATES:   // always the streaming form
      return index_tiles_ok ? round16(m3s::topk_ws_bytes(R, 1, topk)) : 0;
    case M3S_OP_INDEX_ATTENTION:    // the scorer's candidate lists and each row's slot range
      return index_tiles_ok ? round16(m3s::index_attention_ws_bytes(R, topk)) : 0;
    case M3S_OP_INDEX_SCORE_TOPK:   // one tile per row
      return index_tiles_ok ? round16(m3s::score_topk_ws_bytes(R, 1, R, max_blocks, topk)) : 0;
    case M3S_OP_VERIFY_SCORE_TOPK: {   // tiles of up to 8 rows of one request
      const int cpr = max_q > 0 ? (max_q + 7) / 8 : 1;
      const long long nt = B > 0 ? static_cast<long long>(B) * cpr : 0;
      if (nt > m3s::kMaxTiles) return 0;
      return round16(m3s::score_topk_ws_bytes(nt, 8, R, max_blocks, topk));
    }
    case M3S_OP_VERIFY_INDEX_ATTENTION: {   // candidate lists, block-maximum scratch, row ranges
      const int cpr = max_q > 0 ? (max_q + 7) / 8 : 1;
      const long long nt = B > 0 ? static_cast<long long>(B) * cpr : 0;
      if (nt > m3s::kMaxTiles) return 0;
      return round16(m3s::verify_attention_ws_bytes(static_cast<int>(nt), R, topk, max_blocks));
    }
    case M3S_OP_SPARSE_ATTENTION:
      // split-K partials are combined inside a thread-block cluster: no workspace
      return 0;
    default:
      return 0;
  }
}

extern "C" const char* m3s_version(void) { return "m3s 0.2 (sm_103a; NVFP4 and MXFP4 planes, quantise-at-write)"; }
