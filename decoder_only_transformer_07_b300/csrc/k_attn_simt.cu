// Causal grouped-query attention, forward and backward, in fp32 arithmetic on
// CUDA cores.  This is the attention of the fp32 compute mode (and works for
// any head_dim that is a multiple of 16, up to 256).
//
// Scores s = q.k / sqrt(hd) with a causal mask, p = softmax(s), o = p v; query
// head h reads kv head h / (H / Hkv) (cosmicrealm "noao-chat-0-项目总体介绍"
// §2.1 item 6).  The forward keeps lse = log(sum exp s) per query row; the
// backward recomputes p from it.
//
// Work split: TPQ = hd/16 threads share one query (or key) row, each owning
// 16 consecutive dims; dot products finish with shuffles inside the group.
// The backward is two deterministic kernels: one over query tiles (dq), one
// over key tiles looping over the group's query heads (dk, dv), so no atomics.
#include "nc_kernels.cuh"

#define AT_DPT 16
#define AT_THREADS 256
#define AT_KT 32   // key rows staged in shared memory per step

struct AttnShape {
  int B, T, H, Hkv, hd;
  int64_t ld_qkv;   // row stride of qkv / dqkv
  int64_t ld_o;     // row stride of o / do
};

template <int TPQ>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = 1; o < TPQ; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T>
__device__ __forceinline__ void load16(const T* p, float* r) {
#pragma unroll
  for (int i = 0; i < AT_DPT; ++i) r[i] = to_f32(p[i]);
}

// Stage `rows` rows of hd values (row r at src + r*ld) into shared memory as floats.
template <typename T>
__device__ __forceinline__ void stage_rows(float* dst, const T* src, int64_t ld, int rows, int hd) {
  for (int idx = threadIdx.x; idx < rows * hd; idx += blockDim.x) {
    int r = idx / hd, c = idx % hd;
    dst[idx] = to_f32(src[(int64_t)r * ld + c]);
  }
}

template <typename T, int TPQ>
__global__ void __launch_bounds__(AT_THREADS) k_attn_fwd_simt(AttnShape sh, const T* __restrict__ qkv,
                                                              T* __restrict__ o, float* __restrict__ lse) {
  constexpr int R = AT_THREADS / TPQ;     // query rows per block
  extern __shared__ float smem[];
  const int hd = sh.hd;
  float* Ks = smem;
  float* Vs = smem + AT_KT * hd;
  const int bh = blockIdx.y, b = bh / sh.H, h = bh % sh.H;
  const int g = h / (sh.H / sh.Hkv);
  const int qi = blockIdx.x * R + threadIdx.x / TPQ;
  const int sub = threadIdx.x % TPQ;
  const bool active = qi < sh.T;
  const int64_t row0 = (int64_t)b * sh.T;
  const float scale = rsqrtf((float)hd);
  float q[AT_DPT], acc[AT_DPT];
  if (active) load16(qkv + (row0 + qi) * sh.ld_qkv + (int64_t)h * hd + sub * AT_DPT, q);
#pragma unroll
  for (int i = 0; i < AT_DPT; ++i) acc[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int q_last = min(sh.T - 1, (int)(blockIdx.x * R + R - 1));
  for (int k0 = 0; k0 <= q_last; k0 += AT_KT) {
    const int nk = min(AT_KT, sh.T - k0);
    __syncthreads();
    stage_rows(Ks, qkv + (row0 + k0) * sh.ld_qkv + (int64_t)(sh.H + g) * hd, sh.ld_qkv, nk, hd);
    stage_rows(Vs, qkv + (row0 + k0) * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * hd, sh.ld_qkv, nk, hd);
    __syncthreads();
    float s[AT_KT];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < AT_KT; ++j) {
      float part = 0.f;
      if (j < nk) {
        const float* kr = Ks + j * hd + sub * AT_DPT;
#pragma unroll
        for (int i = 0; i < AT_DPT; ++i) part = fmaf(q[i], kr[i], part);
      }
      part = group_sum<TPQ>(part) * scale;
      s[j] = (j < nk && k0 + j <= qi) ? part : -INFINITY;
      tmax = fmaxf(tmax, s[j]);
    }
    if (!active || tmax == -INFINITY) continue;
    const float mn = fmaxf(m, tmax);
    const float corr = expf(m - mn);
    l *= corr;
#pragma unroll
    for (int i = 0; i < AT_DPT; ++i) acc[i] *= corr;
#pragma unroll
    for (int j = 0; j < AT_KT; ++j) {
      if (s[j] == -INFINITY) continue;   // masked, or past the last key
      float p = expf(s[j] - mn);
      l += p;
      const float* vr = Vs + j * hd + sub * AT_DPT;
#pragma unroll
      for (int i = 0; i < AT_DPT; ++i) acc[i] = fmaf(p, vr[i], acc[i]);
    }
    m = mn;
  }
  if (!active) return;
  const float inv = 1.f / l;
  T* orow = o + (row0 + qi) * sh.ld_o + (int64_t)h * hd + sub * AT_DPT;
#pragma unroll
  for (int i = 0; i < AT_DPT; ++i) orow[i] = from_f32<T>(acc[i] * inv);
  if (sub == 0) lse[(int64_t)bh * sh.T + qi] = m + logf(l);
}

// D[b,h,t] = sum_d do[b,t,h,d] * o[b,t,h,d]; one warp per (row, head).
template <typename T>
__global__ void k_attn_rowdot(AttnShape sh, const T* __restrict__ o, const T* __restrict__ dout,
                              float* __restrict__ Dv) {
  int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  int64_t rows = (int64_t)sh.B * sh.T;
  if (w >= rows * sh.H) return;
  int64_t row = w / sh.H;
  int h = (int)(w % sh.H);
  const T* a = o + row * sh.ld_o + (int64_t)h * sh.hd;
  const T* c = dout + row * sh.ld_o + (int64_t)h * sh.hd;
  float s = 0.f;
  for (int i = lane; i < sh.hd; i += 32) s += to_f32(a[i]) * to_f32(c[i]);
  s = warp_sum(s);
  int b = (int)(row / sh.T), t = (int)(row % sh.T);
  if (lane == 0) Dv[((int64_t)b * sh.H + h) * sh.T + t] = s;
}

template <typename T, int TPQ>
__global__ void __launch_bounds__(AT_THREADS) k_attn_bwd_dq_simt(AttnShape sh, const T* __restrict__ qkv,
                                                                 const T* __restrict__ dout,
                                                                 const float* __restrict__ lse,
                                                                 const float* __restrict__ Dv,
                                                                 T* __restrict__ dqkv) {
  constexpr int R = AT_THREADS / TPQ;
  extern __shared__ float smem[];
  const int hd = sh.hd;
  float* Ks = smem;
  float* Vs = smem + AT_KT * hd;
  const int bh = blockIdx.y, b = bh / sh.H, h = bh % sh.H;
  const int g = h / (sh.H / sh.Hkv);
  const int qi = blockIdx.x * R + threadIdx.x / TPQ;
  const int sub = threadIdx.x % TPQ;
  const bool active = qi < sh.T;
  const int64_t row0 = (int64_t)b * sh.T;
  const float scale = rsqrtf((float)hd);
  float q[AT_DPT], dov[AT_DPT], dq[AT_DPT];
  float L = 0.f, Dq = 0.f;
  if (active) {
    load16(qkv + (row0 + qi) * sh.ld_qkv + (int64_t)h * hd + sub * AT_DPT, q);
    load16(dout + (row0 + qi) * sh.ld_o + (int64_t)h * hd + sub * AT_DPT, dov);
    L = lse[(int64_t)bh * sh.T + qi];
    Dq = Dv[(int64_t)bh * sh.T + qi];
  } else {
#pragma unroll
    for (int i = 0; i < AT_DPT; ++i) q[i] = dov[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < AT_DPT; ++i) dq[i] = 0.f;
  const int q_last = min(sh.T - 1, (int)(blockIdx.x * R + R - 1));
  for (int k0 = 0; k0 <= q_last; k0 += AT_KT) {
    const int nk = min(AT_KT, sh.T - k0);
    __syncthreads();
    stage_rows(Ks, qkv + (row0 + k0) * sh.ld_qkv + (int64_t)(sh.H + g) * hd, sh.ld_qkv, nk, hd);
    stage_rows(Vs, qkv + (row0 + k0) * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * hd, sh.ld_qkv, nk, hd);
    __syncthreads();
    for (int j = 0; j < nk; ++j) {
      const float* kr = Ks + j * hd + sub * AT_DPT;
      const float* vr = Vs + j * hd + sub * AT_DPT;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int i = 0; i < AT_DPT; ++i) { s = fmaf(q[i], kr[i], s); dp = fmaf(dov[i], vr[i], dp); }
      s = group_sum<TPQ>(s);
      dp = group_sum<TPQ>(dp);
      if (!active || k0 + j > qi) continue;
      float p = expf(s * scale - L);
      float ds = p * (dp - Dq) * scale;
#pragma unroll
      for (int i = 0; i < AT_DPT; ++i) dq[i] = fmaf(ds, kr[i], dq[i]);
    }
  }
  if (!active) return;
  T* dst = dqkv + (row0 + qi) * sh.ld_qkv + (int64_t)h * hd + sub * AT_DPT;
#pragma unroll
  for (int i = 0; i < AT_DPT; ++i) dst[i] = from_f32<T>(dq[i]);
}

template <typename T, int TPQ>
__global__ void __launch_bounds__(AT_THREADS) k_attn_bwd_dkv_simt(AttnShape sh, const T* __restrict__ qkv,
                                                                  const T* __restrict__ dout,
                                                                  const float* __restrict__ lse,
                                                                  const float* __restrict__ Dv,
                                                                  T* __restrict__ dqkv) {
  constexpr int R = AT_THREADS / TPQ;     // key rows per block
  extern __shared__ float smem[];
  const int hd = sh.hd;
  float* Qs = smem;                    // [AT_KT][hd]
  float* Ds = smem + AT_KT * hd;       // [AT_KT][hd] (dO rows)
  float* Ls = Ds + AT_KT * hd;         // [AT_KT]
  float* DDs = Ls + AT_KT;             // [AT_KT]
  const int bg = blockIdx.y, b = bg / sh.Hkv, g = bg % sh.Hkv;
  const int G = sh.H / sh.Hkv;
  const int kj = blockIdx.x * R + threadIdx.x / TPQ;
  const int sub = threadIdx.x % TPQ;
  const bool active = kj < sh.T;
  const int64_t row0 = (int64_t)b * sh.T;
  const float scale = rsqrtf((float)hd);
  float k[AT_DPT], v[AT_DPT], dk[AT_DPT], dv[AT_DPT];
  if (active) {
    load16(qkv + (row0 + kj) * sh.ld_qkv + (int64_t)(sh.H + g) * hd + sub * AT_DPT, k);
    load16(qkv + (row0 + kj) * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * hd + sub * AT_DPT, v);
  } else {
#pragma unroll
    for (int i = 0; i < AT_DPT; ++i) k[i] = v[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < AT_DPT; ++i) dk[i] = dv[i] = 0.f;
  const int k_first = blockIdx.x * R;
  for (int hh = 0; hh < G; ++hh) {
    const int h = g * G + hh;
    for (int q0 = (k_first / AT_KT) * AT_KT; q0 < sh.T; q0 += AT_KT) {
      const int nq = min(AT_KT, sh.T - q0);
      __syncthreads();
      stage_rows(Qs, qkv + (row0 + q0) * sh.ld_qkv + (int64_t)h * hd, sh.ld_qkv, nq, hd);
      stage_rows(Ds, dout + (row0 + q0) * sh.ld_o + (int64_t)h * hd, sh.ld_o, nq, hd);
      for (int i = threadIdx.x; i < nq; i += blockDim.x) {
        Ls[i] = lse[((int64_t)b * sh.H + h) * sh.T + q0 + i];
        DDs[i] = Dv[((int64_t)b * sh.H + h) * sh.T + q0 + i];
      }
      __syncthreads();
      for (int j = 0; j < nq; ++j) {
        const float* qr = Qs + j * hd + sub * AT_DPT;
        const float* dr = Ds + j * hd + sub * AT_DPT;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int i = 0; i < AT_DPT; ++i) { s = fmaf(k[i], qr[i], s); dp = fmaf(v[i], dr[i], dp); }
        s = group_sum<TPQ>(s);
        dp = group_sum<TPQ>(dp);
        if (!active || q0 + j < kj) continue;
        float p = expf(s * scale - Ls[j]);
        float ds = p * (dp - DDs[j]) * scale;
#pragma unroll
        for (int i = 0; i < AT_DPT; ++i) {
          dv[i] = fmaf(p, dr[i], dv[i]);
          dk[i] = fmaf(ds, qr[i], dk[i]);
        }
      }
    }
  }
  if (!active) return;
  T* dkp = dqkv + (row0 + kj) * sh.ld_qkv + (int64_t)(sh.H + g) * hd + sub * AT_DPT;
  T* dvp = dqkv + (row0 + kj) * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * hd + sub * AT_DPT;
#pragma unroll
  for (int i = 0; i < AT_DPT; ++i) {
    dkp[i] = from_f32<T>(dk[i]);
    dvp[i] = from_f32<T>(dv[i]);
  }
}

template <typename T, int TPQ>
static nc_status attn_fwd_t(AttnShape sh, const void* qkv, void* o, float* lse, cudaStream_t st) {
  constexpr int R = AT_THREADS / TPQ;
  size_t smem = 2 * AT_KT * sh.hd * sizeof(float);
  auto kern = k_attn_fwd_simt<T, TPQ>;
  NC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  dim3 grid(cdiv(sh.T, R), sh.B * sh.H);
  kern<<<grid, AT_THREADS, smem, st>>>(sh, (const T*)qkv, (T*)o, lse);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

template <typename T, int TPQ>
static nc_status attn_bwd_t(AttnShape sh, const void* qkv, const void* o, const float* lse,
                            const void* dout, void* dqkv, float* Dv, cudaStream_t st) {
  constexpr int R = AT_THREADS / TPQ;
  int64_t warps = (int64_t)sh.B * sh.T * sh.H;
  k_attn_rowdot<T><<<cdiv(warps, 8), 256, 0, st>>>(sh, (const T*)o, (const T*)dout, Dv);
  NC_CUDA_TRY(cudaGetLastError());
  size_t smem_q = 2 * AT_KT * sh.hd * sizeof(float);
  auto kq = k_attn_bwd_dq_simt<T, TPQ>;
  NC_CUDA_TRY(cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q));
  kq<<<dim3(cdiv(sh.T, R), sh.B * sh.H), AT_THREADS, smem_q, st>>>(sh, (const T*)qkv, (const T*)dout, lse, Dv,
                                                                   (T*)dqkv);
  NC_CUDA_TRY(cudaGetLastError());
  size_t smem_k = (2 * AT_KT * sh.hd + 2 * AT_KT) * sizeof(float);
  auto kk = k_attn_bwd_dkv_simt<T, TPQ>;
  NC_CUDA_TRY(cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_k));
  kk<<<dim3(cdiv(sh.T, R), sh.B * sh.Hkv), AT_THREADS, smem_k, st>>>(sh, (const T*)qkv, (const T*)dout, lse, Dv,
                                                                     (T*)dqkv);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

static bool attn_shape(int B, int T, int H, int Hkv, int hd, AttnShape* sh) {
  if (B <= 0 || T <= 0 || H <= 0 || Hkv <= 0 || H % Hkv || hd % 16 || hd > 256) return false;
  if ((int64_t)B * H > 65535 || (int64_t)B * Hkv > 65535) return false;
  sh->B = B; sh->T = T; sh->H = H; sh->Hkv = Hkv; sh->hd = hd;
  sh->ld_qkv = (int64_t)(H + 2 * Hkv) * hd;
  sh->ld_o = (int64_t)H * hd;
  return true;
}

#define AT_DISPATCH(T, FN, ...)                                              \
  switch (sh.hd / AT_DPT) {                                                  \
    case 1: return FN<T, 1>(__VA_ARGS__);                                    \
    case 2: return FN<T, 2>(__VA_ARGS__);                                    \
    case 4: return FN<T, 4>(__VA_ARGS__);                                    \
    case 8: return FN<T, 8>(__VA_ARGS__);                                    \
    case 16: return FN<T, 16>(__VA_ARGS__);                                  \
    default: return NC_ERR_UNSUPPORTED;                                      \
  }

nc_status launch_attn_fwd_simt(int dtype, int B, int T, int H, int Hkv, int hd, const void* qkv, void* o,
                               float* lse, cudaStream_t st) {
  AttnShape sh;
  if (!attn_shape(B, T, H, Hkv, hd, &sh)) return NC_ERR_ARG;
  if (dtype == NC_BF16) { AT_DISPATCH(bf16, attn_fwd_t, sh, qkv, o, lse, st) }
  AT_DISPATCH(float, attn_fwd_t, sh, qkv, o, lse, st)
}

nc_status launch_attn_bwd_simt(int dtype, int B, int T, int H, int Hkv, int hd, const void* qkv,
                               const void* o, const float* lse, const void* dout, void* dqkv, float* Dv,
                               cudaStream_t st) {
  AttnShape sh;
  if (!attn_shape(B, T, H, Hkv, hd, &sh)) return NC_ERR_ARG;
  if (dtype == NC_BF16) { AT_DISPATCH(bf16, attn_bwd_t, sh, qkv, o, lse, dout, dqkv, Dv, st) }
  AT_DISPATCH(float, attn_bwd_t, sh, qkv, o, lse, dout, dqkv, Dv, st)
}
