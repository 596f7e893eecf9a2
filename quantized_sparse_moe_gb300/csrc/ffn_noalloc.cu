// moe_ffn_forward_noalloc: the expert FFN for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or hand us a workspace: a plugin that
// runs inside another runtime's memory pool, code on a latency-critical
// thread where an allocation (and the device synchronisation it can cause)
// is not allowed, or a host application that only owns the activations and
// the stream.  For them this entry point takes the FFN's scratch (the fp16
// SwiGLU output of every token-expert pair) from a fixed array that lives
// in the library itself, so the caller passes only inputs and outputs.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds its own copy (kNoAllocScratchBytes) until the process
// exits.  In host code its name is only a host-side stand-in, not a device
// address, so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and then passed to the
// kernels.  The lookup happens on the first call made on each device.
#include <mutex>

#include "qsm_common.cuh"

namespace {

// 1 MiB per device: enough for the decode path at T <= 64 tokens with
// k = 8 and I = 512 ((T*k + T) * I fp16 values = 576 KiB).
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kNoAllocMaxT = 64;

static __device__ __align__(256) unsigned char g_ffn_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of g_ffn_scratch (looked up once per
// device, on the first call made with that device current).  The address
// stays valid for the life of the device's primary context: after
// cudaDeviceReset the module is loaded again, possibly elsewhere, and calls
// are not supported.
qsm_status scratch_of_current_device(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return QSM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ffn_scratch) != cudaSuccess || p == nullptr)
      return QSM_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QSM_OK;
}

}  // namespace

extern "C" qsm_status moe_ffn_forward_noalloc(
    const qsm_moe_layer* L, const uint16_t* x, int32_t T,
    const int32_t* topk_idx, const float* topk_w, const qsm_grouping* g,
    uint16_t* y, float* y_f32, int32_t* dev_status, cudaStream_t stream) {
  if (T < 0) return QSM_ERR_INVALID_ARGUMENT;
  if (T > kNoAllocMaxT) return QSM_ERR_UNSUPPORTED;
  if (T == 0) return moe_ffn_forward(L, x, T, topk_idx, topk_w, g, y, y_f32, nullptr, 0,
                                     dev_status, stream);
  const size_t need = moe_ffn_workspace_bytes(L, T);
  if (need == 0) return QSM_ERR_INVALID_ARGUMENT;  // bad layer
  if (need > kNoAllocScratchBytes) return QSM_ERR_UNSUPPORTED;
  // The scratch belongs to the current device: a stream of another device
  // would hand that device's kernels this device's address.
  int dev = -1, sdev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return QSM_ERR_CUDA;
  if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return QSM_ERR_CUDA;
  if (sdev != dev) return QSM_ERR_INVALID_ARGUMENT;
  void* scratch = nullptr;
  const qsm_status s = scratch_of_current_device(dev, &scratch);
  if (s != QSM_OK) return s;
  // Nothing in the scratch has to start at zero: every value the FFN reads
  // back was written earlier in the same call.  The size check above and
  // the call below each consult the path in force; a test hook that switched
  // it in between could make the scratch too small, which is reported as
  // unsupported like any other size beyond it.
  const qsm_status r = moe_ffn_forward(L, x, T, topk_idx, topk_w, g, y, y_f32, scratch,
                                       kNoAllocScratchBytes, dev_status, stream);
  return r == QSM_ERR_WORKSPACE_TOO_SMALL ? QSM_ERR_UNSUPPORTED : r;
}
