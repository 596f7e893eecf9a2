// C ABI entry points of the FFN, argument validation and status strings.
#include <atomic>

#include "qsm_common.cuh"

namespace qsm {

qsm_status decode_ffn_launch(const qsm_moe_layer* L, const uint16_t* x, int T,
                             const float* topk_w, const qsm_grouping* g,
                             uint16_t* y, float* y32, void* ws,
                             int32_t* dev_status, cudaStream_t stream);
size_t decode_ffn_workspace_bytes(const qsm_moe_layer* L, int T);
bool prefill_supported(const qsm_moe_layer* L);
size_t prefill_ffn_workspace_bytes(const qsm_moe_layer* L, int T);
qsm_status prefill_ffn_launch(const qsm_moe_layer* L, const uint16_t* x, int T,
                              const float* topk_w, const qsm_grouping* g,
                              uint16_t* y, float* y32, void* ws,
                              int32_t* dev_status, cudaStream_t stream);

std::atomic<unsigned long long> g_launch_count{0};
float* g_gu_dump = nullptr;
size_t g_gu_dump_floats = 0;

namespace {

std::atomic<int> g_force_path{0};

constexpr int kDecodeTileRows = 8;
constexpr int kPrefillTileRows = 128;
constexpr int kDecodeMaxT = 128;   // d2 keeps a [T, 16] fp32 slab per warp
constexpr int kDecodeAutoMaxT = 64;

// Path for T tokens: the decode kernels for few tokens, the tensor-core
// grouped GEMMs for many (the test hook can force either where it applies).
bool use_decode(int T) {
  const int mode = g_force_path.load();
  if (mode == 1) return T <= kDecodeMaxT;
  if (mode == 2) return false;
  return T <= kDecodeAutoMaxT;
}

// Shape checks of one quantized tensor (the "same type, same group size,
// same bits and mode" eligibility of the oMLX gate/up fusion becomes: all
// four tensors of a layer share one qtype).
bool check_q(const qsm_qweights& w, int qtype, int experts, int rows, int cols) {
  if (w.qtype != qtype || w.experts != experts || w.rows != rows || w.cols != cols)
    return false;
  if (!w.codes || !w.scales || !aligned16(w.codes) || !aligned4(w.scales))
    return false;
  if (qtype == QSM_Q8_0) return w.biases == nullptr && cols % 64 == 0;
  if (qtype == QSM_AFFINE4_G64)
    return w.biases != nullptr && aligned4(w.biases) && cols % 64 == 0;
  return false;
}

qsm_status check_layer(const qsm_moe_layer* L) {
  if (!L) return QSM_ERR_INVALID_ARGUMENT;
  if (L->H < 64 || L->H % 64 || L->I < 64 || L->I % 64 || L->E < 1 ||
      L->E > 1024 || L->k < 1 || L->k > L->E || L->k > 32)
    return QSM_ERR_INVALID_ARGUMENT;
  const int qt = L->gate_up.qtype;
  if (qt != QSM_Q8_0 && qt != QSM_AFFINE4_G64) return QSM_ERR_UNSUPPORTED;
  if (!check_q(L->gate_up, qt, L->E, 2 * L->I, L->H) ||
      !check_q(L->down, qt, L->E, L->H, L->I) ||
      !check_q(L->shared_gate_up, qt, 1, 2 * L->I, L->H) ||
      !check_q(L->shared_down, qt, 1, L->H, L->I))
    return QSM_ERR_INVALID_ARGUMENT;
  if (L->shared_gate && !aligned16(L->shared_gate)) return QSM_ERR_INVALID_ARGUMENT;
  return QSM_OK;
}

}  // namespace
}  // namespace qsm

extern "C" int32_t moe_ffn_tile_rows(int32_t T) {
  return qsm::use_decode(T) ? qsm::kDecodeTileRows : qsm::kPrefillTileRows;
}

extern "C" size_t moe_ffn_workspace_bytes(const qsm_moe_layer* L, int32_t T) {
  if (!L || T < 0 || qsm::check_layer(L) != QSM_OK) return 0;
  if (qsm::use_decode(T)) return qsm::decode_ffn_workspace_bytes(L, T);
  if (!qsm::prefill_supported(L)) return 0;
  return qsm::prefill_ffn_workspace_bytes(L, T);
}

extern "C" qsm_status moe_ffn_forward(const qsm_moe_layer* L,
                                      const uint16_t* x, int32_t T,
                                      const int32_t* topk_idx,
                                      const float* topk_w,
                                      const qsm_grouping* g, uint16_t* y,
                                      float* y_f32, void* workspace,
                                      size_t workspace_bytes,
                                      int32_t* dev_status,
                                      cudaStream_t stream) {
  using namespace qsm;
  const qsm_status ls = check_layer(L);
  if (ls != QSM_OK) return ls;
  if (T < 0 || !g) return QSM_ERR_INVALID_ARGUMENT;
  if (T == 0) return QSM_OK;
  (void)topk_idx;  // the grouping carries the assignment -> expert map
  if (!x || !topk_w || !y || !workspace || !dev_status || !g->perm ||
      !g->offsets || !g->tile_map || !g->n_tiles)
    return QSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(y) || !aligned16(workspace) ||
      (y_f32 && !aligned16(y_f32)) || !aligned4(topk_w))
    return QSM_ERR_INVALID_ARGUMENT;
  if (g->tile_rows != moe_ffn_tile_rows(T) ||
      g->max_tiles < moe_group_max_tiles(T, L->k, L->E, g->tile_rows))
    return QSM_ERR_INVALID_ARGUMENT;
  const bool decode = use_decode(T);
  if (!decode && !prefill_supported(L)) return QSM_ERR_UNSUPPORTED;
  if (workspace_bytes < moe_ffn_workspace_bytes(L, T))
    return QSM_ERR_WORKSPACE_TOO_SMALL;
  if (decode)
    return decode_ffn_launch(L, x, T, topk_w, g, y, y_f32, workspace,
                             dev_status, stream);
  return prefill_ffn_launch(L, x, T, topk_w, g, y, y_f32, workspace,
                            dev_status, stream);
}

extern "C" const char* qsm_status_str(qsm_status s) {
  switch (s) {
    case QSM_OK: return "ok";
    case QSM_ERR_INVALID_ARGUMENT: return "invalid argument";
    case QSM_ERR_UNSUPPORTED: return "unsupported shape or type";
    case QSM_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case QSM_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

extern "C" int32_t qsm_abi_version(void) { return QSM_ABI_VERSION; }

extern "C" uint64_t qsm_launch_count(void) {
  return qsm::g_launch_count.load(std::memory_order_relaxed);
}

extern "C" qsm_status qsm_debug_force_path(int32_t mode) {
  if (mode < 0 || mode > 2) return QSM_ERR_INVALID_ARGUMENT;
  qsm::g_force_path.store(mode);
  return QSM_OK;
}

extern "C" qsm_status qsm_debug_gu_dump(float* buf, size_t n_floats) {
  if ((buf == nullptr) != (n_floats == 0)) return QSM_ERR_INVALID_ARGUMENT;
  if (buf && !qsm::aligned4(buf)) return QSM_ERR_INVALID_ARGUMENT;
  qsm::g_gu_dump = buf;
  qsm::g_gu_dump_floats = n_floats;
  return QSM_OK;
}
