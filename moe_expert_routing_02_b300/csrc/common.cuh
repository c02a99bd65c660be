// Internal helpers shared by the kernels of libmoe (device side).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

// Device error word, one per device (this library is built as one translation
// unit, so every kernel sees the same variable).
//   bit 0: a kernel met invalid device data (expert id out of range,
//          inconsistent group offsets, loads breaking the replication bound)
//   bit 1: a bounded wait ran out (tcgen05 pipeline)
#define MOE_DEVERR_DATA 1u
#define MOE_DEVERR_TIMEOUT 2u
__device__ unsigned int g_moe_dev_error = 0;

__device__ __forceinline__ void moe_flag_error(unsigned int bits) { atomicOr(&g_moe_dev_error, bits); }

// Programmatic dependent launch.  A kernel launched with launch_pdl may be
// started by the hardware once every block of the stream's previous kernel
// has exited, before that kernel's completion is processed; it calls
// pdl_wait() before its first access to memory that earlier work writes or
// reads, which waits for that completion and its memory operations.  Without
// a programmatic predecessor pdl_wait() returns at once.  One kernel releases
// its dependent early: the front's route kernel, for short token rows, lets
// the scatter/copy blocks start and ask L2 for their rows while it routes
// (parked blocks with nothing to do measured slower than the launch latency
// they hide); every other dependent starts only after its predecessor's
// blocks have exited, so it never shares the GPU with them.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// host option (moe_set_option(MOE_OPT_PDL, ...)); read once per launch
inline std::atomic<int> g_moe_pdl{1};

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_moe_pdl.load(std::memory_order_relaxed) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}
