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
// cos / sin of t * base^(-2i/hd) in fp64, rounded to float.  `tab` is
// [T][hd/2][2]; `pairs` (optional, hd % 4 == 0) holds the same numbers
// pair-major, [hd/4][T][4] = (cos_i, sin_i, cos_i+1, sin_i+1) for even i, so
// that 32 threads handling 32 consecutive positions read 512 contiguous bytes.
__global__ void k_rope_table(float* __restrict__ tab, float* __restrict__ pairs, int T, int hd, double base) {
  const int d = hd / 2;
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= T * d) return;
  int t = idx / d, i = idx % d;
  double omega = pow(base, -2.0 * (double)i / (double)hd);
  double th = (double)t * omega;
  const float c = (float)cos(th), sn = (float)sin(th);
  if (tab) {
    tab[2 * idx] = c;
    tab[2 * idx + 1] = sn;
  }
  if (pairs) {
    float* q = pairs + ((size_t)(i >> 1) * T + t) * 4 + (i & 1) * 2;
    q[0] = c;
    q[1] = sn;
  }
}

nc_status launch_rope_table(int T, int hd, float base, float* tab, float* pairs, cudaStream_t st) {
  if (T <= 0 || hd <= 0 || (hd & 1) || (!tab && !pairs) || (pairs && (hd & 3))) return NC_ERR_ARG;
  int n = T * (hd / 2);
  k_rope_table<<<cdiv(n, 256), 256, 0, st>>>(tab, pairs, T, hd, (double)base);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// ---------------------------------------------------------------- RMSNorm
// Four consecutive activation-type values <-> float4.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const bf16* p) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x), b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// One warp per row; C % 4 == 0.  y = x * rstd, rstd = 1/sqrt(mean(x^2) + eps).
// amax_bits (optional): atomic maximum of |y| as stored (after rounding to T),
// as the bits of a non-negative float, for the 8-bit quantiser of y; one
// atomic per block.
template <typename T>
__global__ void k_rmsnorm_fwd(int64_t rows, int C, const float* __restrict__ x,
                              T* __restrict__ y, float* __restrict__ rstd, float eps, unsigned* __restrict__ amax_bits) {
  __shared__ float wmax[8];
  int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  float am = 0.f;
  if (row < rows) {
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
      const float4 o = make_float4(v.x * r, v.y * r, v.z * r, v.w * r);
      st4(yr + 4 * c, o);
      if (amax_bits)
        am = fmaxf(am, fmaxf(fmaxf(fabsf(round_act<T>(o.x)), fabsf(round_act<T>(o.y))),
                             fmaxf(fabsf(round_act<T>(o.z)), fabsf(round_act<T>(o.w)))));
    }
  }
  if (amax_bits) {   // uniform across the block: every thread reaches this point
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    if (lane == 0) wmax[threadIdx.x >> 5] = am;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = wmax[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
      atomicMax(amax_bits, __float_as_uint(m));
    }
  }
}

// dx += rstd * (dy - y * mean(dy * y)); dx_act = act(dx) if given.  One warp
// per row, four columns per lane per step (C % 4 == 0).
// amax_bits (optional, with dx_act): atomic maximum of |dx_act| as stored, as
// float bits, for the 8-bit quantiser of dx_act; one atomic per block.
template <typename T>
__global__ void k_rmsnorm_bwd(int64_t rows, int C, const float* __restrict__ dy,
                              const T* __restrict__ y, const float* __restrict__ rstd,
                              float* __restrict__ dx, T* __restrict__ dx_act, unsigned* __restrict__ amax_bits) {
  __shared__ float wmax[8];
  int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  float am = 0.f;
  if (row < rows) {
    const float* dyr = dy + row * C;
    const T* yr = y + row * C;
    float dot = 0.f;
    for (int c = lane * 4; c < C; c += 128) {
      float4 a = ld4(dyr + c), b = ld4(yr + c);
      dot += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
    }
    dot = warp_sum(dot) / (float)C;
    const float r = rstd[row];
    float* dxr = dx + row * C;
    for (int c = lane * 4; c < C; c += 128) {
      float4 a = ld4(dyr + c), b = ld4(yr + c), d = ld4(dxr + c);
      d.x += r * (a.x - b.x * dot);
      d.y += r * (a.y - b.y * dot);
      d.z += r * (a.z - b.z * dot);
      d.w += r * (a.w - b.w * dot);
      st4(dxr + c, d);
      if (dx_act) {
        st4(dx_act + row * C + c, d);
        if (amax_bits)
          am = fmaxf(am, fmaxf(fmaxf(fabsf(round_act<T>(d.x)), fabsf(round_act<T>(d.y))),
                               fmaxf(fabsf(round_act<T>(d.z)), fabsf(round_act<T>(d.w)))));
      }
    }
  }
  if (amax_bits) {   // uniform across the block: every thread reaches this point
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
    if (lane == 0) wmax[threadIdx.x >> 5] = am;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = wmax[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
      atomicMax(amax_bits, __float_as_uint(m));
    }
  }
}

template <typename T>
nc_status launch_rmsnorm_fwd_t(int64_t rows, int C, const float* x, T* y, float* rstd, float eps,
                               cudaStream_t st, unsigned* amax_bits = nullptr) {
  if (rows <= 0) return NC_OK;
  if (C % 4 || (((uintptr_t)x) & 15)) return NC_ERR_ARG;
  k_rmsnorm_fwd<T><<<cdiv(rows, 8), 256, 0, st>>>(rows, C, x, y, rstd, eps, amax_bits);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
template <typename T>
nc_status launch_rmsnorm_bwd_t(int64_t rows, int C, const float* dy, const T* y, const float* rstd,
                               float* dx, T* dx_act, cudaStream_t st, unsigned* amax_bits = nullptr) {
  if (rows <= 0) return NC_OK;
  if (C % 4 || (((uintptr_t)dy) & 15) || (((uintptr_t)dx) & 15) || (((uintptr_t)y) & 7)) return NC_ERR_ARG;
  k_rmsnorm_bwd<T><<<cdiv(rows, 8), 256, 0, st>>>(rows, C, dy, y, rstd, dx, dx_act, dx_act ? amax_bits : nullptr);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_rmsnorm_fwd(int dtype, int64_t rows, int C, const float* x, void* y, float* rstd,
                             float eps, cudaStream_t st, unsigned* amax_bits) {
  if (dtype == NC_BF16) return launch_rmsnorm_fwd_t<bf16>(rows, C, x, (bf16*)y, rstd, eps, st, amax_bits);
  return launch_rmsnorm_fwd_t<float>(rows, C, x, (float*)y, rstd, eps, st, amax_bits);
}
nc_status launch_rmsnorm_bwd(int dtype, int64_t rows, int C, const float* dy, const void* y,
                             const float* rstd, float* dx, void* dx_act, cudaStream_t st, unsigned* amax_bits) {
  if (dtype == NC_BF16)
    return launch_rmsnorm_bwd_t<bf16>(rows, C, dy, (const bf16*)y, rstd, dx, (bf16*)dx_act, st, amax_bits);
  return launch_rmsnorm_bwd_t<float>(rows, C, dy, (const float*)y, rstd, dx, (float*)dx_act, st, amax_bits);
}

// ---------------------------------------------------------------- RoPE + QK-norm
// One warp per (token row, head j in [0, H + Hkv)): query heads occupy columns
// [0, H*hd) of qkv and key heads [H*hd, (H+Hkv)*hd), so head j starts at j*hd.
// Each lane owns pairs (i, i+1) of the first half and (i+d, i+d+1) of the
// second, i = 2*lane + 64*k, so loads and stores are 2-element vectors.
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld2(const bf16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st2(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }
__device__ __forceinline__ void st2(bf16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

template <typename T>
__global__ void k_rope_qknorm_fwd(int64_t rows, int T_, int nh, int hd, int64_t ld,
                                  T* __restrict__ qkv, float* __restrict__ rstd,
                                  const float2* __restrict__ tab, float eps, const int32_t* __restrict__ pos0,
                                  T* __restrict__ kc, T* __restrict__ vc, int hq, int max_len) {
  // with a cache, Hkv more warps per row copy the v heads into it
  const int hkv = nh - hq;
  const int nw = kc ? nh + hkv : nh;
  int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (w >= rows * nw) return;
  int64_t row = w / nw;
  int j = (int)(w % nw);
  int t = (int)(row % T_) + (pos0 ? *pos0 : 0);
  const int64_t cache_row = kc ? ((row / T_) * hkv + (j - hq - (j >= nh ? hkv : 0))) * max_len + t : 0;
  if (j >= nh) {   // v head j - nh: copied as computed
    const T* src = qkv + row * ld + (int64_t)j * hd;
    T* dst = vc + cache_row * hd;
    for (int i = lane; i < hd; i += 32) dst[i] = src[i];
    return;
  }
  const int d = hd / 2;
  T* p = qkv + row * ld + (int64_t)j * hd;
  const float2* cs = tab + (int64_t)t * d;
  float y[2][4];   // [k][x1a, x1b, x2a, x2b] for hd <= 256
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = 2 * lane + 64 * k;
    y[k][0] = y[k][1] = y[k][2] = y[k][3] = 0.f;
    if (i < d) {
      float2 a = ld2(p + i), b = ld2(p + i + d);
      float4 c = *reinterpret_cast<const float4*>(cs + i);   // cos_i, sin_i, cos_i+1, sin_i+1
      y[k][0] = a.x * c.x + b.x * c.y;
      y[k][2] = -a.x * c.y + b.x * c.x;
      y[k][1] = a.y * c.z + b.y * c.w;
      y[k][3] = -a.y * c.w + b.y * c.z;
      ss += y[k][0] * y[k][0] + y[k][1] * y[k][1] + y[k][2] * y[k][2] + y[k][3] * y[k][3];
    }
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)hd + eps);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = 2 * lane + 64 * k;
    if (i < d) {
      st2(p + i, y[k][0] * r, y[k][1] * r);
      st2(p + i + d, y[k][2] * r, y[k][3] * r);
      if (kc && j >= hq) {   // k head j - hq: also into the cache
        T* q = kc + cache_row * hd;
        st2(q + i, y[k][0] * r, y[k][1] * r);
        st2(q + i + d, y[k][2] * r, y[k][3] * r);
      }
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
  float dy[2][4], yy[2][4];
  float dot = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = 2 * lane + 64 * k;
#pragma unroll
    for (int e = 0; e < 4; ++e) dy[k][e] = yy[k][e] = 0.f;
    if (i < d) {
      float2 g1 = ld2(g + i), g2 = ld2(g + i + d), y1 = ld2(y + i), y2 = ld2(y + i + d);
      dy[k][0] = g1.x; dy[k][1] = g1.y; dy[k][2] = g2.x; dy[k][3] = g2.y;
      yy[k][0] = y1.x; yy[k][1] = y1.y; yy[k][2] = y2.x; yy[k][3] = y2.y;
#pragma unroll
      for (int e = 0; e < 4; ++e) dot += dy[k][e] * yy[k][e];
    }
  }
  dot = warp_sum(dot) / (float)hd;
  const float r = rstd[row * nh + j];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = 2 * lane + 64 * k;
    if (i < d) {
      float q[4];   // through the per-head RMSNorm
#pragma unroll
      for (int e = 0; e < 4; ++e) q[e] = r * (dy[k][e] - yy[k][e] * dot);
      float4 c = *reinterpret_cast<const float4*>(cs + i);
      // transpose of the rotation: dx1 = dr1 cos - dr2 sin, dx2 = dr1 sin + dr2 cos
      st2(g + i, q[0] * c.x - q[2] * c.y, q[1] * c.z - q[3] * c.w);
      st2(g + i + d, q[0] * c.y + q[2] * c.x, q[1] * c.w + q[3] * c.z);
    }
  }
}

nc_status launch_rope_qknorm_fwd(int dtype, int B, int T, int H, int Hkv, int hd, void* qkv,
                                 float* rstd, const float* tab, float eps, cudaStream_t st, const int32_t* pos0,
                                 void* kc, void* vc, int max_len) {
  if (hd > 256 || (hd & 3) || (((uintptr_t)qkv) & 7) || (((uintptr_t)tab) & 15)) return NC_ERR_ARG;
  int64_t rows = (int64_t)B * T;
  int nh = H + Hkv;
  int64_t ld = (int64_t)(H + 2 * Hkv) * hd;
  if ((kc == nullptr) != (vc == nullptr) || (kc && max_len < 1)) return NC_ERR_ARG;
  int64_t warps = rows * (nh + (kc ? Hkv : 0));
  if (warps == 0) return NC_OK;
  if (dtype == NC_BF16)
    k_rope_qknorm_fwd<bf16><<<cdiv(warps, 8), 256, 0, st>>>(rows, T, nh, hd, ld, (bf16*)qkv, rstd,
                                                             (const float2*)tab, eps, pos0, (bf16*)kc, (bf16*)vc, H,
                                                             max_len);
  else
    k_rope_qknorm_fwd<float><<<cdiv(warps, 8), 256, 0, st>>>(rows, T, nh, hd, ld, (float*)qkv, rstd,
                                                              (const float2*)tab, eps, pos0, (float*)kc, (float*)vc,
                                                              H, max_len);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_rope_qknorm_bwd(int dtype, int B, int T, int H, int Hkv, int hd, void* dqkv,
                                 const void* qkv, const float* rstd, const float* tab,
                                 cudaStream_t st) {
  if (hd > 256 || (hd & 3) || (((uintptr_t)dqkv) & 7) || (((uintptr_t)tab) & 15)) return NC_ERR_ARG;
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
