// Shared device and host helpers for the qsmoe CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <unordered_set>
#include <utility>

#include "qsmoe.h"

#define QSM_CUDA_TRY(expr)                      \
  do {                                          \
    cudaError_t err_ = (expr);                  \
    if (err_ != cudaSuccess) return QSM_ERR_CUDA; \
  } while (0)

namespace qsm {

// ------------------------------------------------------------ host helpers

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}
inline bool aligned4(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 3u) == 0;
}

// Every kernel runs with the largest shared-memory carveout, so CTAs of
// consecutive (overlapping) launches can share an SM without waiting for it
// to drain and change its L1 / shared-memory split.  Set once per kernel.
inline void max_smem_carveout(const void* kernel) {
  static std::mutex mu;
  static std::unordered_set<const void*> done;
  std::lock_guard<std::mutex> lock(mu);
  if (done.insert(kernel).second)
    cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
}

// Number of kernel launches this library has issued (or recorded into a
// graph under capture), process-wide.  Read through qsm_launch_count().
extern std::atomic<unsigned long long> g_launch_count;

// Test hook (qsm_debug_gu_dump): when set, the kernels that compute the
// fused gate_up projection also write its fp32 gate and up values, before
// SwiGLU, to this device buffer of g_gu_dump_floats floats (layout per
// kernel family in include/qsmoe.h).
extern float* g_gu_dump;
extern size_t g_gu_dump_floats;

// Launch with programmatic dependent launch enabled: the kernel may start
// while its predecessor on the stream drains; it must execute
// pdl_wait() before touching anything the predecessor writes (or reads).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                              size_t smem, cudaStream_t stream,
                              Args&&... args) {
  max_smem_carveout(reinterpret_cast<const void*>(kernel));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// launch_pdl with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                      unsigned cluster_x, size_t smem,
                                      cudaStream_t stream, Args&&... args) {
  max_smem_carveout(reinterpret_cast<const void*>(kernel));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// ---------------------------------------------------------- device helpers

// Wait until the preceding grid on the stream has completed and its memory
// is visible (no-op when launched without programmatic serialization).
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next grid on the stream to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_status(int32_t* st, int32_t bits) {
  if (st) atomicOr(st, bits);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Top k of the values a warp holds, v[i] at index lane + 32 i (i < KPER,
// indices >= E ignored), in descending order with ties to the lower index.
// Lane j < k receives the j-th value and its index.  Non-finite values must
// be mapped to -inf by the caller.  Candidates are compared as (order-
// preserving key, inverted index) pairs, a strict total order.
//
// KPER == 8: each lane sorts its 8 candidates once (a 19-exchange network),
// then every round takes the best head over the warp with two warp
// reductions (the largest key, then among the lanes holding it the largest
// inverted index) and the winning lane drops its head.  Other KPER: each
// round takes every lane's best untaken candidate and a butterfly of 64-bit
// maxima.  Both give the same selection.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t kv) {
  return __uint_as_float((kv & 0x80000000u) ? (kv & 0x7fffffffu) : ~kv);
}
__device__ __forceinline__ void cas_desc(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

template <int KPER>
__device__ __forceinline__ void warp_topk(const float (&v)[KPER], int E, int k,
                                          float& out_v, int& out_e) {
  const int lane = threadIdx.x & 31;
  out_v = 0.f;
  out_e = 0;
  if constexpr (KPER == 8) {
    unsigned long long c[8];  // (key << 32 | ~index), 0 = no candidate
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      c[i] = e < E ? ((unsigned long long)order_key(v[i]) << 32) | (uint32_t)~e : 0ull;
    }
    // Batcher's odd-even merge sort of 8, descending
    cas_desc(c[0], c[1]); cas_desc(c[2], c[3]); cas_desc(c[4], c[5]); cas_desc(c[6], c[7]);
    cas_desc(c[0], c[2]); cas_desc(c[1], c[3]); cas_desc(c[4], c[6]); cas_desc(c[5], c[7]);
    cas_desc(c[1], c[2]); cas_desc(c[5], c[6]);
    cas_desc(c[0], c[4]); cas_desc(c[1], c[5]); cas_desc(c[2], c[6]); cas_desc(c[3], c[7]);
    cas_desc(c[2], c[4]); cas_desc(c[3], c[5]);
    cas_desc(c[1], c[2]); cas_desc(c[3], c[4]); cas_desc(c[5], c[6]);
    for (int j = 0; j < k; ++j) {
      const uint32_t hk = (uint32_t)(c[0] >> 32), hi = (uint32_t)c[0];
      const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
      const uint32_t mi = __reduce_max_sync(0xffffffffu, hk == mk ? hi : 0u);
      if (hk == mk && hi == mi) {  // this lane held the winner: drop it
#pragma unroll
        for (int i = 0; i < 7; ++i) c[i] = c[i + 1];
        c[7] = 0ull;
      }
      if (lane == j) {
        out_v = key_value(mk);
        out_e = (int)~mi;
      }
    }
  } else {
    uint32_t key[KPER];
#pragma unroll
    for (int i = 0; i < KPER; ++i) key[i] = order_key(v[i]);
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int i = 0; i < KPER; ++i) {
        const int e = lane + 32 * i;
        const unsigned long long c =
            ((unsigned long long)key[i] << 32) | (unsigned long long)(~(uint32_t)e);
        if (e < E && !((taken >> i) & 1u) && c > best) best = c;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      const uint32_t e = ~(uint32_t)best;
      const uint32_t kv = (uint32_t)(best >> 32);
      if ((e & 31u) == (uint32_t)lane) taken |= 1u << (e >> 5);
      if (lane == j) {
        out_v = key_value(kv);
        out_e = (int)e;
      }
    }
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) {
  return __uint_as_float(v << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t v) {
  return __uint_as_float(v & 0xffff0000u);
}

// Two bf16 (packed) -> two fp16 (packed), round to nearest even.  Exact for
// bf16 values whose magnitude lies in [2^-17, 65504].
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  __half2 h = __floats2half2_rn(bf16_lo(v), bf16_hi(v));
  return *reinterpret_cast<uint32_t*>(&h);
}

// Four signed int8 codes (one 32-bit word) -> two packed fp16 pairs holding
// the exact integers: lo = (b0, b1), hi = (b2, b3).  The byte is biased to
// unsigned (xor 0x80), placed under the fp16 exponent of 1024 (0x64xx =
// 1024 + byte), and 1152 = 1024 + 128 is subtracted.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo,
                                                uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col).  Not volatile: a
// pure function of its operands, so the compiler may interleave independent
// MMAs (their latency is what bounds a warp's tile loop).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];"
               : "=r"(r)
               : "l"(p));
  return r;
}

// silu(g) = g / (1 + e^-g) with an approximate reciprocal (a few ulp of
// fp32).  For g below about -88, e^-g overflows and the quotient is 0, the
// limit of silu; an IEEE division would take its slow path there.
__device__ __forceinline__ float silu(float g) {
  return __fdividef(g, 1.0f + __expf(-g));
}


// ------------------------------------------------- TMA bulk copies, mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}
// Distributed shared memory: the address of `p` (this CTA's shared memory)
// in the CTA of cluster rank `rank`, and a 32-bit store there.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// The same as dsmem_addr for a shared-memory address held as u32.
__device__ __forceinline__ uint32_t dsmem_addr_u32(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 dsmem_ld_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Every thread of every CTA of the cluster: stores before it are visible to
// loads after it in all of the cluster's CTAs.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Orders the computation of v before everything after this point: a
// consumer that releases a shared-memory slot puts the values computed from
// the slot here first, so that no load from the slot can still be in flight
// when the release is issued (the compiler may otherwise move the
// arithmetic, and with it the wait for the loads, past the release).
__device__ __forceinline__ void consumed(float v) { asm volatile("" ::"f"(v) : "memory"); }
__device__ __forceinline__ void consumed(const float (&v)[4]) {
  asm volatile("" ::"f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]) : "memory");
}

// Make an initialised mbarrier visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Raise the byte count phase `bar` waits for, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Global -> shared bulk copy (16-byte aligned, size a multiple of 16) that
// signals `bar` with its byte count on completion.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src,
                                         uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Bulk prefetch of global memory into L2 (no shared memory, no completion).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src,
                                                 uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` with an iteration limit (each try_wait
// may suspend for a while); false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar,
                                                  uint32_t parity,
                                                  uint32_t max_iter) {
  for (uint32_t i = 0; i < max_iter; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
constexpr uint32_t kWaitIters = 1u << 22;

}  // namespace qsm
