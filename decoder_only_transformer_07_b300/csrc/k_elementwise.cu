// Memory-bound kernels of the step: weight init and cast, RMSNorm forward and
// backward, fused RoPE + QK-norm forward and backward.
//
// RMSNorm without gain: cosmicrealm "noao-chat-0-项目总体介绍" §2.1 item 5.
// RoPE by half-split rotation, y1 = x1 cos + x2 sin, y2 = -x1 sin + x2 cos:
// §2.1 item 1 (and §5.3); q and k are normalised after the rotation: item 2.
#include "nc_kernels.cuh"

// ---------------------------------------------------------------- init
// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): output e of the stream
// starting at state0 is mix13(state0 + (e + 1) * gamma).  Box-Muller turns one
// 64-bit word into one normal: u1 from the top 24 bits, u2 from bits 16..39.
__device__ __forceinline__ uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void k_init_normal(float* __restrict__ out, int64_t count, uint64_t state0, float std) {
  const uint64_t gamma = 0x9E3779B97F4A7C15ull;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < count;
       e += (int64_t)gridDim.x * blockDim.x) {
    uint64_t w = sm64_mix(state0 + (uint64_t)(e + 1) * gamma);
    double u1 = ((double)(w >> 40) + 0.5) / 16777216.0;
    double u2 = ((double)((w >> 16) & 0xFFFFFFull) + 0.5) / 16777216.0;
    double z = sqrt(-2.0 * log(u1)) * cos(2.0 * 3.14159265358979323846 * u2);
    out[e] = (float)(z * (double)std);
  }
}

nc_status launch_init_normal(float* out, int64_t count, uint64_t seed, int tensor_index,
                             float std, cudaStream_t st) {
  const uint64_t gamma = 0x9E3779B97F4A7C15ull;
  uint64_t state0 = seed ^ ((uint64_t)(tensor_index + 1) * gamma);
  if (count <= 0) return NC_OK;
  unsigned grid = (unsigned)std::min<int64_t>((count + 255) / 256, 148 * 64);
  k_init_normal<<<grid, 256, 0, st>>>(out, count, state0, std);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// fp32 -> bf16, 8 elements per thread when aligned.
__global__ void k_cast_bf16(const float* __restrict__ src, bf16* __restrict__ dst, int64_t n) {
  int64_t n8 = n / 8;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += stride) {
    float4 a = reinterpret_cast<const float4*>(src)[2 * i];
    float4 b = reinterpret_cast<const float4*>(src)[2 * i + 1];
    __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t*>(&p0);
    o.y = *reinterpret_cast<uint32_t*>(&p1);
    o.z = *reinterpret_cast<uint32_t*>(&p2);
    o.w = *reinterpret_cast<uint32_t*>(&p3);
    reinterpret_cast<uint4*>(dst)[i] = o;
  }
  for (int64_t i = n8 * 8 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = __float2bfloat16_rn(src[i]);
}

nc_status launch_cast_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t st) {
  if (n <= 0) return NC_OK;
  if ((((uintptr_t)src) & 15) || (((uintptr_t)dst) & 15)) return NC_ERR_ARG;
  unsigned grid = (unsigned)std::min<int64_t>((n / 8 + 255) / 256 + 1, 148 * 16);
  k_cast_bf16<<<grid, 256, 0, st>>>(src, dst, n);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// ---------------------------------------------------------------- RoPE table
__global__ void k_rope_table(float* __restrict__ tab, int T, int hd, double base) {
  const int d = hd / 2;
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= T * d) return;
  int t = idx / d, i = idx % d;
  double omega = pow(base, -2.0 * (double)i / (double)hd);
  double th = (double)t * omega;
  tab[2 * idx] = (float)cos(th);
  tab[2 * idx + 1] = (float)sin(th);
}

nc_status launch_rope_table(int T, int hd, float base, float* tab, cudaStream_t st) {
  if (T <= 0 || hd <= 0 || (hd & 1) || !tab) return NC_ERR_ARG;
  int n = T * (hd / 2);
  k_rope_table<<<cdiv(n, 256), 256, 0, st>>>(tab, T, hd, (double)base);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// ---------------------------------------------------------------- RMSNorm
// One warp per row; C % 4 == 0.  y = x * rstd, rstd = 1/sqrt(mean(x^2) + eps).
template <typename T>
__global__ void k_rmsnorm_fwd(int64_t rows, int C, const float* __restrict__ x,
                              T* __restrict__ y, float* __restrict__ rstd, float eps) {
  int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + row * C);
  float ss = 0.f;
  for (int c = lane; c < C / 4; c += 32) {
    float4 v = xr[c];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  float r = rsqrtf(ss / (float)C + eps);
  if (lane == 0) rstd[row] = r;
  T* yr = y + row * C;
  for (int c = lane; c < C / 4; c += 32) {
    float4 v = xr[c];
    yr[4 * c + 0] = from_f32<T>(v.x * r);
    yr[4 * c + 1] = from_f32<T>(v.y * r);
    yr[4 * c + 2] = from_f32<T>(v.z * r);
    yr[4 * c + 3] = from_f32<T>(v.w * r);
  }
}

// dx += rstd * (dy - y * mean(dy * y)); dx_act = act(dx) if given.
template <typename T>
__global__ void k_rmsnorm_bwd(int64_t rows, int C, const float* __restrict__ dy,
                              const T* __restrict__ y, const float* __restrict__ rstd,
                              float* __restrict__ dx, T* __restrict__ dx_act) {
  int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* dyr = dy + row * C;
  const T* yr = y + row * C;
  float dot = 0.f;
  for (int c = lane; c < C; c += 32) dot += dyr[c] * to_f32(yr[c]);
  dot = warp_sum(dot) / (float)C;
  float r = rstd[row];
  float* dxr = dx + row * C;
  for (int c = lane; c < C; c += 32) {
    float v = dxr[c] + r * (dyr[c] - to_f32(yr[c]) * dot);
    dxr[c] = v;
    if (dx_act) dx_act[row * C + c] = from_f32<T>(v);
  }
}

template <typename T>
nc_status launch_rmsnorm_fwd_t(int64_t rows, int C, const float* x, T* y, float* rstd, float eps,
                               cudaStream_t st) {
  if (rows <= 0) return NC_OK;
  if (C % 4 || (((uintptr_t)x) & 15)) return NC_ERR_ARG;
  k_rmsnorm_fwd<T><<<cdiv(rows, 8), 256, 0, st>>>(rows, C, x, y, rstd, eps);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
template <typename T>
nc_status launch_rmsnorm_bwd_t(int64_t rows, int C, const float* dy, const T* y, const float* rstd,
                               float* dx, T* dx_act, cudaStream_t st) {
  if (rows <= 0) return NC_OK;
  k_rmsnorm_bwd<T><<<cdiv(rows, 8), 256, 0, st>>>(rows, C, dy, y, rstd, dx, dx_act);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_rmsnorm_fwd(int dtype, int64_t rows, int C, const float* x, void* y, float* rstd,
                             float eps, cudaStream_t st) {
  if (dtype == NC_BF16) return launch_rmsnorm_fwd_t<bf16>(rows, C, x, (bf16*)y, rstd, eps, st);
  return launch_rmsnorm_fwd_t<float>(rows, C, x, (float*)y, rstd, eps, st);
}
nc_status launch_rmsnorm_bwd(int dtype, int64_t rows, int C, const float* dy, const void* y,
                             const float* rstd, float* dx, void* dx_act, cudaStream_t st) {
  if (dtype == NC_BF16)
    return launch_rmsnorm_bwd_t<bf16>(rows, C, dy, (const bf16*)y, rstd, dx, (bf16*)dx_act, st);
  return launch_rmsnorm_bwd_t<float>(rows, C, dy, (const float*)y, rstd, dx, (float*)dx_act, st);
}

// ---------------------------------------------------------------- RoPE + QK-norm
// One warp per (token row, head j in [0, H + Hkv)): query heads occupy columns
// [0, H*hd) of qkv and key heads [H*hd, (H+Hkv)*hd), so head j starts at j*hd.
template <typename T>
__global__ void k_rope_qknorm_fwd(int64_t rows, int T_, int nh, int hd, int64_t ld,
                                  T* __restrict__ qkv, float* __restrict__ rstd,
                                  const float2* __restrict__ tab, float eps) {
  int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (w >= rows * nh) return;
  int64_t row = w / nh;
  int j = (int)(w % nh);
  int t = (int)(row % T_);
  const int d = hd / 2;
  T* p = qkv + row * ld + (int64_t)j * hd;
  const float2* cs = tab + (int64_t)t * d;
  float y1[4], y2[4];   // hd <= 256
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int i = lane + 32 * k;
    y1[k] = y2[k] = 0.f;
    if (i < d) {
      float x1 = to_f32(p[i]), x2 = to_f32(p[i + d]);
      float2 c = cs[i];
      y1[k] = x1 * c.x + x2 * c.y;
      y2[k] = -x1 * c.y + x2 * c.x;
      ss += y1[k] * y1[k] + y2[k] * y2[k];
    }
  }
  ss = warp_sum(ss);
  float r = rsqrtf(ss / (float)hd + eps);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int i = lane + 32 * k;
    if (i < d) {
      p[i] = from_f32<T>(y1[k] * r);
      p[i + d] = from_f32<T>(y2[k] * r);
    }
  }
  if (lane == 0) rstd[row * nh + j] = r;
}

template <typename T>
__global__ void k_rope_qknorm_bwd(int64_t rows, int T_, int nh, int hd, int64_t ld,
                                  T* __restrict__ dqkv, const T* __restrict__ qkv,
                                  const float* __restrict__ rstd, const float2* __restrict__ tab) {
  int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (w >= rows * nh) return;
  int64_t row = w / nh;
  int j = (int)(w % nh);
  int t = (int)(row % T_);
  const int d = hd / 2;
  T* g = dqkv + row * ld + (int64_t)j * hd;
  const T* y = qkv + row * ld + (int64_t)j * hd;
  const float2* cs = tab + (int64_t)t * d;
  float dy1[4], dy2[4], yy1[4], yy2[4];
  float dot = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int i = lane + 32 * k;
    dy1[k] = dy2[k] = yy1[k] = yy2[k] = 0.f;
    if (i < d) {
      dy1[k] = to_f32(g[i]); dy2[k] = to_f32(g[i + d]);
      yy1[k] = to_f32(y[i]); yy2[k] = to_f32(y[i + d]);
      dot += dy1[k] * yy1[k] + dy2[k] * yy2[k];
    }
  }
  dot = warp_sum(dot) / (float)hd;
  float r = rstd[row * nh + j];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    int i = lane + 32 * k;
    if (i < d) {
      float r1 = r * (dy1[k] - yy1[k] * dot);   // through the per-head RMSNorm
      float r2 = r * (dy2[k] - yy2[k] * dot);
      float2 c = cs[i];
      g[i] = from_f32<T>(r1 * c.x - r2 * c.y);   // transpose of the rotation
      g[i + d] = from_f32<T>(r1 * c.y + r2 * c.x);
    }
  }
}

nc_status launch_rope_qknorm_fwd(int dtype, int B, int T, int H, int Hkv, int hd, void* qkv,
                                 float* rstd, const float* tab, float eps, cudaStream_t st) {
  if (hd > 256 || (hd & 1)) return NC_ERR_ARG;
  int64_t rows = (int64_t)B * T;
  int nh = H + Hkv;
  int64_t ld = (int64_t)(H + 2 * Hkv) * hd;
  int64_t warps = rows * nh;
  if (warps == 0) return NC_OK;
  if (dtype == NC_BF16)
    k_rope_qknorm_fwd<bf16><<<cdiv(warps, 8), 256, 0, st>>>(rows, T, nh, hd, ld, (bf16*)qkv, rstd,
                                                             (const float2*)tab, eps);
  else
    k_rope_qknorm_fwd<float><<<cdiv(warps, 8), 256, 0, st>>>(rows, T, nh, hd, ld, (float*)qkv, rstd,
                                                              (const float2*)tab, eps);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_rope_qknorm_bwd(int dtype, int B, int T, int H, int Hkv, int hd, void* dqkv,
                                 const void* qkv, const float* rstd, const float* tab,
                                 cudaStream_t st) {
  if (hd > 256 || (hd & 1)) return NC_ERR_ARG;
  int64_t rows = (int64_t)B * T;
  int nh = H + Hkv;
  int64_t ld = (int64_t)(H + 2 * Hkv) * hd;
  int64_t warps = rows * nh;
  if (warps == 0) return NC_OK;
  if (dtype == NC_BF16)
    k_rope_qknorm_bwd<bf16><<<cdiv(warps, 8), 256, 0, st>>>(rows, T, nh, hd, ld, (bf16*)dqkv,
                                                             (const bf16*)qkv, rstd, (const float2*)tab);
  else
    k_rope_qknorm_bwd<float><<<cdiv(warps, 8), 256, 0, st>>>(rows, T, nh, hd, ld, (float*)dqkv,
                                                              (const float*)qkv, rstd, (const float2*)tab);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
