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

#include "nc_kernels.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[NC_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

// The array's device address on the current device.  In host code the name
// g_noalloc_scratch stands for a host-side shadow, never a device address, so
// the address is looked up once per device (with that device current) and
// cached.  The first call on a device therefore does this set-up.
nc_status scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return NC_ERR_CUDA;
    }
    g_dev_ptr[dev] = p;
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
