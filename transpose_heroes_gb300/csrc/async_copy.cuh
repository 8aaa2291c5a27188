// Asynchronous global -> shared copies on sm_103a: mbarriers with bounded waits, 1-D bulk copies and
// 2-D tensor (TMA) tile loads, plus the per-translation-unit device fault word the bounded waits
// report to.
#pragma once
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "hlo_internal.h"

namespace hlo {

constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz: far beyond any legitimate wait

// Fault bits recorded by this translation unit's kernels (internal linkage: every .cu file that
// includes this header has its own word, read through read_tu_faults()).
static __device__ unsigned int g_tu_faults;

__device__ __forceinline__ void record_fault(unsigned int bits) { atomicOr(&g_tu_faults, bits); }

// Host side: copies this unit's fault word out and optionally clears it (the caller has waited for the
// device). Every unit that includes this header registers it when the library is loaded, so
// hlo_device_faults reads the words of all of them.
static inline cudaError_t read_tu_faults(unsigned int* faults, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(faults, g_tu_faults, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tu_faults, &zero, sizeof zero);
}
static const int g_tu_fault_reader_index = register_fault_reader(&read_tu_faults);

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

// Makes mbarrier initialisation visible to the async proxy (the copy engine).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses before later async-proxy writes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Waits for phase `parity` of the mbarrier; returns false if `limit` clock cycles ran out first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit = kWaitCycles) {
  long long t0 = -1;
  while (true) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.u32 %0, 1, 0, P; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    const long long now = clock64();
    if (t0 < 0) t0 = now;
    else if (now - t0 > limit) return false;
  }
}

// One arrival that also announces `bytes` of copies completing on this barrier's current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) into shared memory.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// 2-D tensor tile load: the box of `map` whose first element has coordinates (x, y) (x innermost, in
// elements; x * element size must be a multiple of 16 bytes) lands in shared memory at dst (128-byte
// aligned), completing on `bar`. Elements outside the tensor are filled with zeros.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// The driver's tensor-map encoder, looked up once through the runtime (no link against libcuda).
static inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool looked = false;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!looked) {
    looked = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t pending = cudaPeekAtLastError();
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else if (pending == cudaSuccess)
      cudaGetLastError();  // the lookup's own error: the caller falls back to plain loads
  }
  return fn;
}

}  // namespace hlo
