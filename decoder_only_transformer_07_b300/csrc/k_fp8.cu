// Per-tensor E4M3 quantisation for the 8-bit GEMM.  The woshipm nanochat
// analysis lists FP8 among nanochat's speed levers on Hopper-class tensor
// cores (§一.2 and §六.2, the precision strategy) but fixes no recipe; this
// is current per-tensor scaling:
//   amax  = max_i |x_i|                                   (exact)
//   scale = fl32(448 / amax) if finite and > 0, else 1    (448 = largest E4M3)
//   code  = E4M3 round-to-nearest-even, saturating, of fl32(x_i * scale)
//   scale_inv = fl32(1 / scale)                           (the GEMM's dequantisation factor)
// Two passes over x: the absolute maximum (grid-stride, one atomic per block,
// into stats[0] read as unsigned bits), then the cast (16-byte loads, 8 codes
// per thread).
#include <cuda_fp8.h>

#include "nc_kernels.cuh"

#define FP8_THREADS 256

__device__ __forceinline__ void load8(const float* x, int64_t i, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(x + i);
  const float4 b = *reinterpret_cast<const float4*>(x + i + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16* x, int64_t i, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(x + i);
  const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(h[e]);
}

// amax_bits: the absolute maximum's bit pattern (non-negative floats order as
// unsigned integers), zeroed by the caller.
template <typename T>
__global__ void __launch_bounds__(FP8_THREADS) k_fp8_amax(const T* __restrict__ x, int64_t n, unsigned* amax_bits) {
  __shared__ float sh[32];
  float m = 0.f;
  const int64_t n8 = n & ~(int64_t)7;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 8;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < n8; i += stride) {
    float f[8];
    load8(x, i, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
  }
  if (blockIdx.x == 0 && threadIdx.x < n - n8) m = fmaxf(m, fabsf(to_f32(x[n8 + threadIdx.x])));
  m = block_max(m, sh);
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(m));
}

// stats = {amax, scale, scale_inv}; stats[0] holds amax's bits on entry
__global__ void k_fp8_scale(float* stats) {
  const float amax = __uint_as_float(*reinterpret_cast<const unsigned*>(stats));
  float scale = 448.f / amax;
  if (!(scale > 0.f) || !isfinite(scale)) scale = 1.f;
  stats[0] = amax;
  stats[1] = scale;
  stats[2] = 1.f / scale;
}

__device__ __forceinline__ uint32_t e4m3(float v) {
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

template <typename T>
__global__ void __launch_bounds__(FP8_THREADS) k_fp8_cast(const T* __restrict__ x, int64_t n,
                                                          const float* __restrict__ stats, uint8_t* __restrict__ y) {
  const float s = stats[1];
  const int64_t n8 = n & ~(int64_t)7;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 8;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < n8; i += stride) {
    float f[8];
    load8(x, i, f);
    uint2 o;   // byte e of the 8 holds element i + e
    o.x = e4m3(f[0] * s) | (e4m3(f[1] * s) << 8) | (e4m3(f[2] * s) << 16) | (e4m3(f[3] * s) << 24);
    o.y = e4m3(f[4] * s) | (e4m3(f[5] * s) << 8) | (e4m3(f[6] * s) << 16) | (e4m3(f[7] * s) << 24);
    *reinterpret_cast<uint2*>(y + i) = o;
  }
  if (blockIdx.x == 0 && threadIdx.x < n - n8) {
    const float v = to_f32(x[n8 + threadIdx.x]) * s;
    y[n8 + threadIdx.x] = (uint8_t)e4m3(v);
  }
}

nc_status launch_quantize_fp8(int dtype, const void* x, int64_t n, uint8_t* y, float* stats, cudaStream_t st) {
  if (n < 0 || !stats || (n > 0 && (!x || !y))) return NC_ERR_ARG;
  if ((((uintptr_t)x) & 15) || (((uintptr_t)y) & 7) || (((uintptr_t)stats) & 3)) return NC_ERR_ARG;
  if (dtype != NC_FP32 && dtype != NC_BF16) return NC_ERR_ARG;
  if (!g_num_sms) {
    int dev = 0;
    NC_CUDA_TRY(cudaGetDevice(&dev));
    NC_CUDA_TRY(cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev));
  }
  unsigned* amax = (unsigned*)stats;
  NC_CUDA_TRY(cudaMemsetAsync(amax, 0, sizeof(unsigned), st));
  // whole waves of 8 resident blocks per SM, fewer for small inputs
  const long long want = std::max<long long>(1, (n / 8 + FP8_THREADS - 1) / FP8_THREADS);
  const unsigned grid = (unsigned)std::min<long long>(want, 8LL * g_num_sms);
  if (n > 0) {
    if (dtype == NC_BF16) k_fp8_amax<bf16><<<grid, FP8_THREADS, 0, st>>>((const bf16*)x, n, amax);
    else k_fp8_amax<float><<<grid, FP8_THREADS, 0, st>>>((const float*)x, n, amax);
    NC_CUDA_TRY(cudaGetLastError());
  }
  k_fp8_scale<<<1, 1, 0, st>>>(stats);
  NC_CUDA_TRY(cudaGetLastError());
  if (n > 0) {
    if (dtype == NC_BF16) k_fp8_cast<bf16><<<grid, FP8_THREADS, 0, st>>>((const bf16*)x, n, stats, y);
    else k_fp8_cast<float><<<grid, FP8_THREADS, 0, st>>>((const float*)x, n, stats, y);
    NC_CUDA_TRY(cudaGetLastError());
  }
  return NC_OK;
}
