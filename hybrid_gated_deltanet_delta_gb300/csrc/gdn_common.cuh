// Internal helpers shared by the library's translation units (not part of the
// C ABI).  Device code here is plain CUDA C++ with a few inline-PTX memory
// operations; nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// First device-side error wins; the caller zeroes the word before the call.
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// 16-byte global load through the read-only (non-coherent) path: only for
// data that no thread writes during the kernel.
__device__ __forceinline__ float4 ld_nc_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte global load cached in L2 only: used to read back data this thread
// wrote earlier in the same kernel (program order makes it visible).
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st_f4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

// Asynchronous global -> shared copies (cp.async): the copies are all in
// flight together; cp_async_wait_all() blocks until this thread's copies land.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation allowed (launch_pdl), so that the
// next kernel on the stream is set up while this one runs.  Each kernel
// starts with pdl_enter(): it waits until the previous kernel has completed
// and its memory operations are visible, before any global-memory access of
// its own, so stream order holds for every read and write; then it lets the
// next kernel begin launching.  The next kernel's blocks thus wait, resident,
// for this one to finish, and at most one kernel ahead is waiting (a trigger
// before the wait would let a whole queue of launches pile up on the SMs,
// which measured slower).  After an operation that is not such a kernel (a
// copy, an event, a kernel launched without the attribute) the wait returns
// at once.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, Args... args) {
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
  if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
    (void)cudaGetLastError();
    return GDN_ERR_CUDA;
  }
  return launch_status();
}

}  // namespace gdn
