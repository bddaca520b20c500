// Embedding backward for callers that cannot allocate device memory.
//
// nc_op_embed_bwd needs a scratch buffer from its caller (partial row sums
// and index lists).  Some callers cannot provide one: a host that hands this
// library only its input and output buffers under a device-memory budget fixed
// in advance, or a process whose allocator has reserved the device memory up
// front, so an extra cudaMalloc would fail or fragment its pool.  This file
// gives them nc_op_embed_bwd_noalloc, which runs the same kernels on a scratch
// area that lives in a file-scope device array instead.
//
// The array is NC_NOALLOC_SCRATCH_BYTES (64 MiB) and is held by every GPU
// that loads the library until the process exits.  All calls share it.
#include <mutex>

#include <cuda.h>

#include "nc_kernels.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[NC_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};   // the context the cached address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// A process-unique id of the current device's context (0 if it cannot be
// read).  cudaDeviceReset destroys the primary context; the next runtime call
// creates a new one with a new id, into which the module (and the array) is
// loaded afresh, possibly at another address.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    looked_up = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = (CtxGetCurrentFn)f;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = (CtxGetIdFn)f;
    cudaGetLastError();
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// The array's device address on the current device.  In host code the name
// g_noalloc_scratch stands for a host-side shadow, never a device address, so
// the address is looked up with the device current and cached per device,
// together with the id of the context it was found in.  The first call on a
// device therefore does this set-up; so does the first call after
// cudaDeviceReset, since the cached address then belongs to a destroyed context.
nc_status scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long ctx = current_ctx_id();   // 0 when there is no live context
  if (!g_dev_ptr[dev] || ctx == 0 || ctx != g_ctx_id[dev]) {
    void* p = nullptr;
    // a runtime call: it also re-creates a primary context that cudaDeviceReset destroyed
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return NC_ERR_CUDA;
    }
    g_dev_ptr[dev] = p;
    g_ctx_id[dev] = current_ctx_id();
  }
  *out = g_dev_ptr[dev];
  return NC_OK;
}

}  // namespace

extern "C" nc_status nc_op_embed_bwd_noalloc(int64_t n, int32_t C, int32_t V, const int32_t* tokens,
                                             const float* dx, float* dwte, void* stream) {
  if (!tokens || !dx || !dwte || n < 0 || C <= 0 || V <= 0) return NC_ERR_ARG;
  if (embed_bwd_scratch_bytes(n, C, V) > (size_t)NC_NOALLOC_SCRATCH_BYTES) return NC_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  NC_TRY(scratch_ptr(&scratch));
  // launch_embed_bwd zeroes the counters it needs (cudaMemsetAsync) and
  // overwrites every other scratch word before reading it, so the contents
  // left by the previous call do not matter.
  return launch_embed_bwd(n, C, V, tokens, dx, dwte, scratch, as_stream(stream));
}
