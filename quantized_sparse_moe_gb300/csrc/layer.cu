// The whole layer in one call: router -> grouping -> expert FFNs and
// combine, over the tokens in chunks of at most `chunk` tokens.
//
// "Optimizing on-device inference for Apple Silicon", section "Qwen creates
// three distinct workload shapes" (a long prompt is processed in chunks) and
// section "Keeping expert routing on the GPU" (the chunk's grouping never
// leaves the device).  Each chunk is an independent layer call on its own
// rows of x, topk and y, so chunking changes no token's routing; the FFN of
// a token does not depend on the other tokens of its chunk except for the
// order of the fp32 reduce-adds of the prefill combine.  The workspace is
// sized for one chunk and reused, which bounds it for any prompt length.
#include "qsm_common.cuh"

namespace qsm {
namespace {

inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

struct LayerWs {
  size_t route, group, ffn;   // offsets
  size_t route_bytes, ffn_bytes, total;
  int max_tiles;
};

// Largest needs over the chunk sizes a T-token call uses: full chunks of
// `chunk` tokens and the tail.
bool layer_ws(const qsm_moe_layer* L, int T, int chunk, LayerWs* w) {
  const int full = T < chunk ? T : chunk;
  const int tail = T % chunk;
  const int sizes[2] = {full, tail};
  size_t rb = 0, fb = 0;
  int mt = 0;
  for (int s : sizes) {
    if (s <= 0) continue;
    const size_t r = moe_route_workspace_bytes(s, L->H, L->E);
    const size_t f = moe_ffn_workspace_bytes(L, s);
    if (f == 0) return false;  // unsupported layer or size
    rb = r > rb ? r : rb;
    fb = f > fb ? f : fb;
    const int m = moe_group_max_tiles(s, L->k, L->E, moe_ffn_tile_rows(s));
    mt = m > mt ? m : mt;
  }
  const size_t a = (size_t)full * L->k;  // assignments per chunk
  const size_t group_bytes =
      up256(L->E * 4) + up256((L->E + 1) * 4) + 2 * up256(a * 4) +
      up256((size_t)2 * (mt > 0 ? mt : 1) * 4) + 256;
  w->route = 0;
  w->route_bytes = up256(rb > 256 ? rb : 256);
  w->group = w->route + w->route_bytes;
  w->ffn = w->group + group_bytes;
  w->ffn_bytes = up256(fb);
  w->total = w->ffn + w->ffn_bytes;
  w->max_tiles = mt > 0 ? mt : 1;
  return true;
}

}  // namespace
}  // namespace qsm

extern "C" size_t moe_layer_workspace_bytes(const qsm_moe_layer* L, int32_t T,
                                            int32_t chunk) {
  qsm::LayerWs w;
  if (!L || T <= 0 || chunk <= 0 || !qsm::layer_ws(L, T, chunk, &w)) return 0;
  return w.total;
}

extern "C" qsm_status moe_layer_forward(const qsm_moe_layer* L, const uint16_t* x,
                                        int32_t T, int32_t chunk,
                                        const float* w_router,
                                        const float* logit_bias,
                                        int32_t renormalize, int32_t* topk_idx,
                                        float* topk_w, uint16_t* y, float* y_f32,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* dev_status, cudaStream_t stream) {
  using namespace qsm;
  if (!L || T < 0 || chunk <= 0) return QSM_ERR_INVALID_ARGUMENT;
  if (T == 0) return QSM_OK;
  if (!x || !w_router || !topk_idx || !topk_w || !y || !workspace || !dev_status)
    return QSM_ERR_INVALID_ARGUMENT;
  LayerWs w;
  if (!layer_ws(L, T, chunk, &w)) return QSM_ERR_UNSUPPORTED;
  if (workspace_bytes < w.total) return QSM_ERR_WORKSPACE_TOO_SMALL;
  char* ws = static_cast<char*>(workspace);
  const int E = L->E, k = L->k, H = L->H;
  const size_t a = (size_t)(T < chunk ? T : chunk) * k;
  char* gp = ws + w.group;
  qsm_grouping g;
  g.counts = reinterpret_cast<int32_t*>(gp);
  gp += up256(E * 4);
  g.offsets = reinterpret_cast<int32_t*>(gp);
  gp += up256((E + 1) * 4);
  g.perm = reinterpret_cast<int32_t*>(gp);
  gp += up256(a * 4);
  g.inv_perm = reinterpret_cast<int32_t*>(gp);
  gp += up256(a * 4);
  g.tile_map = reinterpret_cast<int32_t*>(gp);
  gp += up256((size_t)2 * w.max_tiles * 4);
  g.n_tiles = reinterpret_cast<int32_t*>(gp);
  g.max_tiles = w.max_tiles;
  for (int off = 0; off < T; off += chunk) {
    const int tc = T - off < chunk ? T - off : chunk;
    const uint16_t* xc = x + (size_t)off * H;
    int32_t* ic = topk_idx + (size_t)off * k;
    float* wc = topk_w + (size_t)off * k;
    qsm_status st = moe_route(xc, w_router, logit_bias, tc, H, E, k, renormalize, ic,
                              wc, ws + w.route, w.route_bytes, dev_status, stream);
    if (st != QSM_OK) return st;
    g.tile_rows = moe_ffn_tile_rows(tc);
    st = moe_group_tokens(ic, tc, k, E, &g, dev_status, stream);
    if (st != QSM_OK) return st;
    st = moe_ffn_forward(L, xc, tc, ic, wc, &g, y + (size_t)off * H,
                         y_f32 ? y_f32 + (size_t)off * H : nullptr, ws + w.ffn,
                         w.ffn_bytes, dev_status, stream);
    if (st != QSM_OK) return st;
  }
  return QSM_OK;
}
