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

// ---------------------------------------------------------------- the step's quantiser pieces
// The same rule as above in fewer launches: the amax pass leaves out the
// memset (the step zeroes every statistic slot of a step at once), and the
// cast pass forms the scale itself (the scale kernel's formula), so a
// quantisation is two launches, or one when the producer of x has already
// taken its maximum.

__device__ __forceinline__ float fp8_scale_of(float amax) {
  float scale = 448.f / amax;
  if (!(scale > 0.f) || !isfinite(scale)) scale = 1.f;
  return scale;
}

// The scaled cast of a [rows][cols] bf16 tensor written in both layouts: y
// [rows][cols] (codes as the standalone quantiser's cast writes them, the
// scale formed here from the maximum in stats[0]), and yt [cols][ldt] (ldt >= rows,
// a multiple of 16), its transpose: the K-major operand of a product that
// contracts over rows.  One block per 64 x 64 tile through shared memory; the
// tile's own rows and columns past the end are skipped.
__global__ void __launch_bounds__(256) k_fp8_cast_dual(const bf16* __restrict__ x, int rows, int cols,
                                                       float* __restrict__ stats, uint8_t* __restrict__ y,
                                                       uint8_t* __restrict__ yt, int64_t ldt) {
  __shared__ __align__(16) uint8_t tile[64][80];
  const float s = fp8_scale_of(__uint_as_float(*reinterpret_cast<const unsigned*>(stats)));
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    stats[1] = s;
    stats[2] = 1.f / s;
  }
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64, t = threadIdx.x;
  {   // thread t: row r0 + t / 4, columns c0 + 16 (t % 4) .. +16
    const int r = t >> 2, cc = (t & 3) * 16;
    const int gr = r0 + r, gc = c0 + cc;
    uint32_t q[4] = {0u, 0u, 0u, 0u};
    if (gr < rows) {
      const bf16* xr = x + (int64_t)gr * cols + gc;
      uint8_t* yr = y + (int64_t)gr * cols + gc;
      if (gc + 16 <= cols && (cols & 15) == 0) {
        const uint4 a = *reinterpret_cast<const uint4*>(xr), b = *reinterpret_cast<const uint4*>(xr + 8);
        const bf16* ha = reinterpret_cast<const bf16*>(&a);
        const bf16* hb = reinterpret_cast<const bf16*>(&b);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          q[e >> 2] |= e4m3(__bfloat162float(ha[e]) * s) << (8 * (e & 3));
          q[2 + (e >> 2)] |= e4m3(__bfloat162float(hb[e]) * s) << (8 * (e & 3));
        }
        *reinterpret_cast<uint4*>(yr) = make_uint4(q[0], q[1], q[2], q[3]);
      } else {
        for (int e = 0; e < 16 && gc + e < cols; ++e) {
          const uint32_t c = e4m3(__bfloat162float(xr[e]) * s);
          q[e >> 2] |= c << (8 * (e & 3));
          yr[e] = (uint8_t)c;
        }
      }
    }
    *reinterpret_cast<uint4*>(&tile[r][cc]) = make_uint4(q[0], q[1], q[2], q[3]);
  }
  __syncthreads();
  {   // thread t: transposed row c0 + t / 4 (a column of x), rows r0 + 16 (t % 4) .. +16
    const int c = t >> 2, rr = (t & 3) * 16;
    const int gc = c0 + c, gr = r0 + rr;
    if (gc < cols && gr < rows) {
      uint32_t q[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < 16; ++e) q[e >> 2] |= (uint32_t)tile[rr + e][c] << (8 * (e & 3));
      uint8_t* yo = yt + (int64_t)gc * ldt + gr;
      if (gr + 16 <= rows) {
        *reinterpret_cast<uint4*>(yo) = make_uint4(q[0], q[1], q[2], q[3]);
      } else {
        for (int e = 0; gr + e < rows; ++e) yo[e] = (uint8_t)(q[e >> 2] >> (8 * (e & 3)));
      }
    }
  }
}

nc_status launch_fp8_cast_dual(const void* x, int rows, int cols, float* stats, uint8_t* y, uint8_t* yt, int64_t ldt,
                               cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return NC_OK;
  if (!x || !stats || !y || !yt || ldt < rows || (ldt & 15) || (((uintptr_t)x) & 15) || (((uintptr_t)y) & 15) ||
      (((uintptr_t)yt) & 15) || rows > 65535 * 64)
    return NC_ERR_ARG;
  k_fp8_cast_dual<<<dim3((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64)), 256, 0, st>>>(
      (const bf16*)x, rows, cols, stats, y, yt, ldt);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// Multi-tensor form over fp32 tensors (the weight operands of one step): block
// b handles chunk b - chunk0[t] (OPT_CHUNK elements) of tensor t.
__device__ __forceinline__ int fp8_tensor_of(const OptTensors& tl, int blk) {
  int lo = 0, hi = tl.n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tl.chunk0[mid] <= blk) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(FP8_THREADS) k_fp8_amax_multi(const __grid_constant__ OptTensors tl,
                                                                const float* __restrict__ master,
                                                                float* __restrict__ stats) {
  __shared__ float sh[32];
  const int t = fp8_tensor_of(tl, blockIdx.x);
  const int64_t e0 = (int64_t)(blockIdx.x - tl.chunk0[t]) * OPT_CHUNK;
  const int64_t e1 = min(tl.len[t], e0 + OPT_CHUNK);
  const float* x = master + tl.off[t];
  float m = 0.f;
  for (int64_t e = e0 + threadIdx.x; e < e1; e += FP8_THREADS) m = fmaxf(m, fabsf(x[e]));
  m = block_max(m, sh);
  if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned*>(stats + 4 * t), __float_as_uint(m));
}

__global__ void __launch_bounds__(FP8_THREADS) k_fp8_cast_multi(const __grid_constant__ OptTensors tl,
                                                                const float* __restrict__ master,
                                                                float* __restrict__ stats, uint8_t* __restrict__ y) {
  const int t = fp8_tensor_of(tl, blockIdx.x);
  const int64_t e0 = (int64_t)(blockIdx.x - tl.chunk0[t]) * OPT_CHUNK;
  const int64_t e1 = min(tl.len[t], e0 + OPT_CHUNK);
  float* st = stats + 4 * t;
  const float s = fp8_scale_of(__uint_as_float(*reinterpret_cast<const unsigned*>(st)));
  if (e0 == 0 && threadIdx.x == 0) {
    st[1] = s;
    st[2] = 1.f / s;
  }
  const float* x = master + tl.off[t];
  uint8_t* out = y + tl.soff[t];
  for (int64_t e = e0 + threadIdx.x; e < e1; e += FP8_THREADS) out[e] = (uint8_t)e4m3(x[e] * s);
}

nc_status launch_fp8_quantize_multi(const OptTensors& tl, const float* master, float* stats, uint8_t* y,
                                    cudaStream_t st) {
  const int nb = tl.chunk0[tl.n];
  if (nb <= 0) return NC_OK;
  k_fp8_amax_multi<<<nb, FP8_THREADS, 0, st>>>(tl, master, stats);
  NC_CUDA_TRY(cudaGetLastError());
  k_fp8_cast_multi<<<nb, FP8_THREADS, 0, st>>>(tl, master, stats, y);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// Transposed copies of the weight codes, for the input-gradient products
// dX = dY W, whose B operand is W^T in the K-major layout the 8-bit GEMM
// reads: codes [rows][cols] of tensor t at src + tt.off[t] become
// [cols][rows] at dst + tt.off[t] (the same factor applies).  One block per
// 64 x 64 tile through shared memory: 16-byte loads of the tile's rows, then
// each thread gathers 16 bytes of one column and stores them as one piece;
// partial edge pieces go byte by byte.
__global__ void __launch_bounds__(256) k_fp8_transpose_multi(const __grid_constant__ Fp8Transposes tt,
                                                             const uint8_t* __restrict__ src, uint8_t* __restrict__ dst) {
  __shared__ __align__(16) uint8_t tile[64][80];
  int lo = 0, hi = tt.n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tt.tile0[mid] <= (int)blockIdx.x) lo = mid; else hi = mid;
  }
  const int t = lo;
  const int rows = tt.rows[t], cols = tt.cols[t];
  const int tc = (cols + 63) / 64;
  const int k = (int)blockIdx.x - tt.tile0[t];
  const int r0 = (k / tc) * 64, c0 = (k % tc) * 64;
  const uint8_t* s = src + tt.off[t];
  uint8_t* d = dst + tt.off[t];
  const int th = threadIdx.x;
  {   // row r0 + th / 4, columns c0 + 16 (th % 4) .. +16
    const int r = th >> 2, cc = (th & 3) * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < rows) {
      const uint8_t* sr = s + (int64_t)(r0 + r) * cols + c0 + cc;
      if (c0 + cc + 16 <= cols && (cols & 15) == 0) {
        v = *reinterpret_cast<const uint4*>(sr);
      } else {
        uint8_t* vb = reinterpret_cast<uint8_t*>(&v);
        for (int e = 0; e < 16 && c0 + cc + e < cols; ++e) vb[e] = sr[e];
      }
    }
    *reinterpret_cast<uint4*>(&tile[r][cc]) = v;
  }
  __syncthreads();
  {   // transposed row c0 + th / 4 (a column), rows r0 + 16 (th % 4) .. +16
    const int c = th >> 2, rr = (th & 3) * 16;
    if (c0 + c < cols && r0 + rr < rows) {
      uint32_t q[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < 16; ++e) q[e >> 2] |= (uint32_t)tile[rr + e][c] << (8 * (e & 3));
      uint8_t* o = d + (int64_t)(c0 + c) * rows + r0 + rr;
      if (r0 + rr + 16 <= rows && (rows & 15) == 0) {
        *reinterpret_cast<uint4*>(o) = make_uint4(q[0], q[1], q[2], q[3]);
      } else {
        for (int e = 0; r0 + rr + e < rows && e < 16; ++e) o[e] = (uint8_t)(q[e >> 2] >> (8 * (e & 3)));
      }
    }
  }
}

nc_status launch_fp8_transpose_multi(const Fp8Transposes& tt, const uint8_t* src, uint8_t* dst, cudaStream_t st) {
  const int nb = tt.tile0[tt.n];
  if (nb <= 0) return NC_OK;
  k_fp8_transpose_multi<<<nb, 256, 0, st>>>(tt, src, dst);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
