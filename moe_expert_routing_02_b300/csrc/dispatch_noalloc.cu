// moe_dispatch_noalloc: moe_dispatch with library-owned scratch.
//
// The pages have no counterpart to this entry point.  It serves callers that
// cannot allocate device memory when they dispatch: a host framework that owns
// every byte of device memory and forbids plug-ins from allocating, code that
// enqueues work while a stream is being captured (allocation is not allowed
// there), or a latency-critical thread that must not call cudaMalloc because it
// can synchronise the device.  Such a caller still provides the inputs and
// outputs; only the scratch moves into the library.
//
// The scratch is one file-scope device array of a fixed size.  Every GPU that
// loads the library holds it until the process exits.  In host code the
// array's name is a host-side stand-in, not a device address, so the address
// handed to the kernels comes from cudaGetSymbolAddress, taken once per device
// (with that device current) on the first call there and kept for the life of
// the process.  A cudaDeviceReset destroys the context the address belongs to;
// the library does not detect that, so the header tells callers not to use
// this entry point on a device after resetting it.
//
// This file is compiled as part of the library's single translation unit (it
// is included at the end of moe_api.cu), so its kernels report through the
// same device error word that moe_check reads.

// Every word the dispatch kernels read from the scratch is written earlier in
// the same call (per-tile counts by the count kernel, per-expert totals by the
// scan kernel), so nothing in it has to be cleared between calls.
static __device__ __align__(256) unsigned char g_dispatch_noalloc_scratch[MOE_DISPATCH_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_scratch_ptr[kMaxDevices] = {};
}  // namespace

extern "C" moe_status moe_dispatch_noalloc(const uint16_t* x, const int32_t* idx, int T, int k, int H, int E,
                                           const int32_t* rep_base, int32_t* group_offsets, int32_t* perm,
                                           int32_t* inv_perm, uint16_t* xp, void* stream) {
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E)
    return fail(MOE_ERR_INVALID, "moe_dispatch_noalloc: need T>=0, 1<=E<=256, 1<=k<=min(E,8)");
  if ((long long)T * k >= (1LL << 31)) return fail(MOE_ERR_INVALID, "moe_dispatch_noalloc: T*k too large");
  const size_t need = dispatch::workspace_bytes((long long)T * k, E);
  if (T > 0 && need > (size_t)MOE_DISPATCH_NOALLOC_SCRATCH_BYTES)
    return fail(MOE_ERR_WORKSPACE,
                "moe_dispatch_noalloc: T*k=%lld assignments over E=%d experts need %zu bytes of scratch, more than "
                "the %zu bytes this library holds per device; call moe_dispatch with a workspace instead",
                (long long)T * k, E, need, (size_t)MOE_DISPATCH_NOALLOC_SCRATCH_BYTES);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "moe_dispatch_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "moe_dispatch_noalloc: device id %d", dev);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_dispatch_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr)
        return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                           "moe_dispatch_noalloc: cudaGetSymbolAddress of the scratch array");
      g_noalloc_scratch_ptr[dev] = p;
    }
    scratch = g_noalloc_scratch_ptr[dev];
  }
  return moe_dispatch(x, idx, T, k, H, E, rep_base, group_offsets, perm, inv_perm, xp, scratch,
                      (size_t)MOE_DISPATCH_NOALLOC_SCRATCH_BYTES, stream);
}
