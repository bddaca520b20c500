// Incremental decoding with a key/value cache (woshipm nanochat analysis §三
// item 4: generation reuses the KV cache): the keys and values of every
// position already seen are kept per layer, so one new token per sequence
// costs one row of every projection plus one attention row over the cache.
//
// Cache layout, per layer: K and V as [B][Hkv][max_len][hd] in the compute
// dtype (one contiguous run of hd elements per position), so a key run of one
// (sequence, kv head) is contiguous and read once for the whole query group.
//
// Decode attention is split over the key positions (flash decoding): CTA
// (b, g, s) takes keys [256 s, 256 s + 256) of kv head g for every query head
// of its group, each warp an interleaved quarter of them with an online
// softmax, and leaves a partial (max, sum, unnormalised output) per head; a
// second kernel merges the partials of a row.  Scores are q.k / sqrt(hd) in
// fp32 (exp2 form), as in the training attention.
#include "nc_kernels.cuh"

namespace {

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_f(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_f(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// Row r of qkv[rows, ld] is (sequence r / T, position t0 + r % T): its k and v
// heads go to the cache at that position.  One thread per element.
template <typename E>
__global__ void k_kv_store(int64_t rows, int T, int t0, const int32_t* __restrict__ t0_dev, int H, int Hkv, int hd,
                           const E* __restrict__ qkv, int64_t ld, E* __restrict__ kc, E* __restrict__ vc,
                           int max_len) {
  const int64_t per_row = (int64_t)Hkv * hd;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * per_row) return;
  const int64_t r = i / per_row;
  const int rem = (int)(i % per_row);
  const int g = rem / hd, d = rem % hd;
  const int64_t b = r / T;
  const int t = (t0_dev ? *t0_dev : t0) + (int)(r % T);
  const int64_t dst = ((b * Hkv + g) * max_len + t) * hd + d;
  kc[dst] = qkv[r * ld + (int64_t)(H + g) * hd + d];
  vc[dst] = qkv[r * ld + (int64_t)(H + Hkv + g) * hd + d];
}

constexpr int DEC_CHUNK = 256;
constexpr int DEC_WARPS = 4;

// Partials: part[((b * H + h) * nsplit + s) * (HD + 2) + {0: max (log2 units), 1: sum, 2..: output}]
// len_dev (device, may be NULL): the key count is *len_dev + 1 (the position of
// the token just appended, plus one); chunks past it leave empty partials.
template <typename E, int HD, int G>
__global__ void __launch_bounds__(DEC_WARPS * 32)
    k_decode_attn(int H, int Hkv, int len, const int32_t* __restrict__ len_dev, int nsplit,
                  const E* __restrict__ qkv, int64_t ld, const E* __restrict__ kc, const E* __restrict__ vc,
                  int max_len, float scale_log2, float* __restrict__ part) {
  constexpr int DPL = HD / 32;
  if (len_dev) len = *len_dev + 1;
  const int bg = blockIdx.x, s = blockIdx.y;
  const int b = bg / Hkv, g = bg % Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = s * DEC_CHUNK, k1 = min(len, k0 + DEC_CHUNK);
  float q[G][DPL], mx[G], sm[G], o[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const E* qp = qkv + (int64_t)b * ld + (int64_t)(g * G + h) * HD + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      q[h][i] = ld_f(qp + i) * scale_log2;
      o[h][i] = 0.f;
    }
    mx[h] = -INFINITY;
    sm[h] = 0.f;
  }
  const E* kb = kc + ((int64_t)(b * Hkv + g) * max_len) * HD + lane * DPL;
  const E* vb = vc + ((int64_t)(b * Hkv + g) * max_len) * HD + lane * DPL;
  for (int t = k0 + warp; t < k1; t += DEC_WARPS) {
    float kv[DPL], vv[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      kv[i] = ld_f(kb + (int64_t)t * HD + i);
      vv[i] = ld_f(vb + (int64_t)t * HD + i);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float sc = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) sc = fmaf(q[h][i], kv[i], sc);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
      const float mn = fmaxf(mx[h], sc);
      const float alpha = exp2f(mx[h] - mn), p = exp2f(sc - mn);
      sm[h] = fmaf(sm[h], alpha, p);
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[h][i] = fmaf(o[h][i], alpha, p * vv[i]);
      mx[h] = mn;
    }
  }
  // merge the warps' partials through shared memory; warp 0 writes the CTA's
  __shared__ float sm_mx[DEC_WARPS][G], sm_sum[DEC_WARPS][G], sm_o[DEC_WARPS][G][HD];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) {
      sm_mx[warp][h] = mx[h];
      sm_sum[warp][h] = sm[h];
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) sm_o[warp][h][lane * DPL + i] = o[h][i];
  }
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, sm_mx[w][h]);
    float S = 0.f, acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < DEC_WARPS; ++w) {
        const float f = exp2f(sm_mx[w][h] - M);   // 0 for a warp that saw no key
        S = fmaf(sm_sum[w][h], f, S);
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = fmaf(sm_o[w][h][lane * DPL + i], f, acc[i]);
      }
    }
    float* pp = part + ((int64_t)(b * H + g * G + h) * nsplit + s) * (HD + 2);
    if (lane == 0) {
      pp[0] = M;
      pp[1] = S;
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) pp[2 + lane * DPL + i] = acc[i];
  }
}

// o[b, h*HD + d] = merged output of row (b, h); one warp per row.
template <typename E, int HD>
__global__ void k_decode_combine(int64_t rows, int nsplit, const float* __restrict__ part, E* __restrict__ out,
                                 int64_t ldo, int H) {
  constexpr int DPL = HD / 32;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float* pr = part + r * nsplit * (HD + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pr[s * (HD + 2)]);
  float S = 0.f, acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float* ps = pr + s * (HD + 2);
    if (ps[0] == -INFINITY) continue;
    const float f = exp2f(ps[0] - M);
    S = fmaf(ps[1], f, S);
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = fmaf(ps[2 + lane * DPL + i], f, acc[i]);
  }
  const float inv = S > 0.f ? 1.f / S : 0.f;
  const int64_t b = r / H;
  const int h = (int)(r % H);
  E* op = out + b * ldo + (int64_t)h * HD + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) st_f(op + i, acc[i] * inv);
}

template <typename E, int HD, int G>
nc_status decode_attn_t(int B, int H, int Hkv, int len, const int32_t* len_dev, const E* qkv, int64_t ld,
                        const E* kc, const E* vc, int max_len, float* part, E* o, int64_t ldo, cudaStream_t st) {
  // with the length on the device the grid covers the whole capacity
  const int nsplit = ((len_dev ? max_len : len) + DEC_CHUNK - 1) / DEC_CHUNK;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  k_decode_attn<E, HD, G><<<dim3((unsigned)(B * Hkv), (unsigned)nsplit), DEC_WARPS * 32, 0, st>>>(
      H, Hkv, len, len_dev, nsplit, qkv, ld, kc, vc, max_len, scale_log2, part);
  NC_CUDA_TRY(cudaGetLastError());
  const int64_t rows = (int64_t)B * H;
  k_decode_combine<E, HD><<<cdiv(rows, 8), 256, 0, st>>>(rows, nsplit, part, o, ldo, H);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

template <typename E, int HD>
nc_status decode_attn_g(int G, int B, int H, int Hkv, int len, const int32_t* len_dev, const E* qkv, int64_t ld,
                        const E* kc, const E* vc, int max_len, float* part, E* o, int64_t ldo, cudaStream_t st) {
  switch (G) {
    case 1: return decode_attn_t<E, HD, 1>(B, H, Hkv, len, len_dev, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 2: return decode_attn_t<E, HD, 2>(B, H, Hkv, len, len_dev, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 3: return decode_attn_t<E, HD, 3>(B, H, Hkv, len, len_dev, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 4: return decode_attn_t<E, HD, 4>(B, H, Hkv, len, len_dev, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 8: return decode_attn_t<E, HD, 8>(B, H, Hkv, len, len_dev, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    default: return NC_ERR_UNSUPPORTED;
  }
}

}  // namespace

size_t decode_part_floats(int B, int H, int hd, int max_len) {
  return (size_t)B * H * ((max_len + DEC_CHUNK - 1) / DEC_CHUNK) * (hd + 2);
}

nc_status launch_kv_store(int dtype, int64_t rows, int T, int t0, int H, int Hkv, int hd, const void* qkv, int64_t ld,
                          void* kc, void* vc, int max_len, cudaStream_t st, const int32_t* t0_dev) {
  const int64_t n = rows * Hkv * hd;
  if (n <= 0) return NC_OK;
  if (dtype == NC_BF16)
    k_kv_store<bf16><<<cdiv(n, 256), 256, 0, st>>>(rows, T, t0, t0_dev, H, Hkv, hd, (const bf16*)qkv, ld, (bf16*)kc,
                                                    (bf16*)vc, max_len);
  else
    k_kv_store<float><<<cdiv(n, 256), 256, 0, st>>>(rows, T, t0, t0_dev, H, Hkv, hd, (const float*)qkv, ld, (float*)kc,
                                                     (float*)vc, max_len);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_decode_attn(int dtype, int B, int H, int Hkv, int hd, int len, const void* qkv, int64_t ld,
                             const void* kc, const void* vc, int max_len, float* part, void* o, int64_t ldo,
                             cudaStream_t st, const int32_t* len_dev) {
  if (B <= 0 || (!len_dev && (len <= 0 || len > max_len)) || H % Hkv || (hd != 64 && hd != 128)) return NC_ERR_ARG;
  const int G = H / Hkv;
  if (dtype == NC_BF16)
    return hd == 128 ? decode_attn_g<bf16, 128>(G, B, H, Hkv, len, len_dev, (const bf16*)qkv, ld, (const bf16*)kc,
                                                (const bf16*)vc, max_len, part, (bf16*)o, ldo, st)
                     : decode_attn_g<bf16, 64>(G, B, H, Hkv, len, len_dev, (const bf16*)qkv, ld, (const bf16*)kc,
                                               (const bf16*)vc, max_len, part, (bf16*)o, ldo, st);
  return hd == 128 ? decode_attn_g<float, 128>(G, B, H, Hkv, len, len_dev, (const float*)qkv, ld, (const float*)kc,
                                               (const float*)vc, max_len, part, (float*)o, ldo, st)
                   : decode_attn_g<float, 64>(G, B, H, Hkv, len, len_dev, (const float*)qkv, ld, (const float*)kc,
                                              (const float*)vc, max_len, part, (float*)o, ldo, st);
}

namespace {
__global__ void k_set_i32(int32_t* p, int32_t v, int32_t add) { *p = add ? *p + v : v; }
}  // namespace

nc_status launch_set_i32(int32_t* p, int32_t v, bool add, cudaStream_t st) {
  k_set_i32<<<1, 1, 0, st>>>(p, v, add ? 1 : 0);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// ---------------------------------------------------------------- skinny GEMM
// D[m, n] (op)= sum_k A[m, k] W[n, k] for M <= 32 rows (the decode step's
// projections: one row per sequence).  With so few rows every weight is used
// M times at most, so the product is bound by reading W once; it runs on the
// CUDA cores with one warp per output column n streaming W's row n in 16-byte
// pieces, and A staged in shared memory in K chunks that all 8 warps of the
// CTA share.  Accumulation is fp32 in a fixed order.
namespace {

constexpr int SK_WARPS = 8;
// K chunk staged per round: 1024, or less so that the chunk of A stays within 32 KB
template <typename E, int MB>
__host__ __device__ constexpr int sk_kc() { return MB * (int)sizeof(E) * 1024 <= 32768 ? 1024 : 32768 / (MB * (int)sizeof(E)); }

__device__ __forceinline__ void ld8(const float* p, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void ld8(const bf16* p, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(h[e]);
}

// NORM: the rows come from the fp32 residual stream and are normalised on the
// way in, A = act(x * rstd(x)) with rstd = 1/sqrt(mean(x^2) + eps) formed as the
// RMSNorm kernel forms it (so the staged values are the ones it would write);
// M <= SK_WARPS then, one warp per row's statistics.
template <typename E, int MB, bool NORM>
__global__ void __launch_bounds__(SK_WARPS * 32)
    k_gemm_skinny(int M, int N, int K, const void* __restrict__ Ain, int64_t lda, const E* __restrict__ W,
                  int64_t ldw, int ep, void* __restrict__ D, int64_t ldd, float eps) {
  constexpr int SK_KC = sk_kc<E, MB>();
  __shared__ __align__(16) E xs[MB][SK_KC];
  __shared__ float rs[MB];
  const E* A = reinterpret_cast<const E*>(Ain);
  const float* X = reinterpret_cast<const float*>(Ain);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * SK_WARPS + warp;
  if (NORM && warp < M) {
    const float4* xr = reinterpret_cast<const float4*>(X + (int64_t)warp * lda);
    float ss = 0.f;
    for (int c = lane; c < K / 4; c += 32) {
      const float4 v = xr[c];
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) rs[warp] = rsqrtf(ss / (float)K + eps);
  }
  float acc[MB];
#pragma unroll
  for (int m = 0; m < MB; ++m) acc[m] = 0.f;
  for (int k0 = 0; k0 < K; k0 += SK_KC) {
    const int kc = min(SK_KC, K - k0);
    __syncthreads();
    for (int i = threadIdx.x * 8; i < MB * SK_KC; i += SK_WARPS * 32 * 8) {
      const int m = i / SK_KC, k = i % SK_KC;
      if (m < M && k < kc) {
        if (NORM) {
          const float r = rs[m];
#pragma unroll
          for (int e = 0; e < 8; ++e) st_f(&xs[m][k + e], X[(int64_t)m * lda + k0 + k + e] * r);
        } else {
          *reinterpret_cast<uint4*>(&xs[m][k]) = *reinterpret_cast<const uint4*>(A + (int64_t)m * lda + k0 + k);
          if (sizeof(E) == 4) *reinterpret_cast<uint4*>(&xs[m][k + 4]) =
              *reinterpret_cast<const uint4*>(A + (int64_t)m * lda + k0 + k + 4);
        }
      }
    }
    __syncthreads();
    if (n < N) {
      const E* wr = W + (int64_t)n * ldw + k0;
      // four 16-byte pieces of the row in flight per lane before any is used
      for (int kb = lane * 8; kb < kc; kb += 1024) {
        float w[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (kb + 256 * u < kc) ld8(wr + kb + 256 * u, w[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = kb + 256 * u;
          if (k >= kc) break;
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            if (m < M) {
              float x[8];
              ld8(&xs[m][k], x);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[m] = fmaf(x[e], w[u][e], acc[m]);
            }
          }
        }
      }
    }
  }
  if (n >= N) return;
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    float v = acc[m];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0 && m < M) {
      if (ep == NC_EP_STORE_F32) reinterpret_cast<float*>(D)[(int64_t)m * ldd + n] = v;
      else if (ep == NC_EP_ACCUM_F32) reinterpret_cast<float*>(D)[(int64_t)m * ldd + n] += v;
      else {
        if (ep == NC_EP_RELU2_SQ) { v = fmaxf(v, 0.f); v *= v; }
        st_f(reinterpret_cast<E*>(D) + (int64_t)m * ldd + n, v);
      }
    }
  }
}

template <typename E, int MB, bool NORM>
nc_status skinny_t(int M, int N, int K, const void* A, int64_t lda, const E* W, int64_t ldw, int ep, void* D,
                   int64_t ldd, float eps, cudaStream_t st) {
  k_gemm_skinny<E, MB, NORM><<<cdiv(N, SK_WARPS), SK_WARPS * 32, 0, st>>>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

template <typename E, bool NORM>
nc_status skinny_e(int M, int N, int K, const void* A, int64_t lda, const E* W, int64_t ldw, int ep, void* D,
                   int64_t ldd, float eps, cudaStream_t st) {
  if (M <= 1) return skinny_t<E, 1, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if (M <= 2) return skinny_t<E, 2, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if (M <= 4) return skinny_t<E, 4, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if (M <= 8 || NORM) return skinny_t<E, 8, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if (M <= 16) return skinny_t<E, 16, false>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  return skinny_t<E, 32, false>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
}

}  // namespace

nc_status launch_gemm_skinny(int dtype, int M, int N, int K, const void* A, int64_t lda, const void* W, int64_t ldw,
                             int ep, void* D, int64_t ldd, cudaStream_t st) {
  if (M < 1 || M > SKINNY_MAX_M || N < 1 || K < 8 || K % 8 || lda % 8 || ldw % 8 ||
      (ep != NC_EP_STORE && ep != NC_EP_STORE_F32 && ep != NC_EP_ACCUM_F32 && ep != NC_EP_RELU2_SQ))
    return NC_ERR_ARG;
  if ((((uintptr_t)A) & 15) || (((uintptr_t)W) & 15)) return NC_ERR_ARG;
  if (dtype == NC_BF16) return skinny_e<bf16, false>(M, N, K, A, lda, (const bf16*)W, ldw, ep, D, ldd, 0.f, st);
  return skinny_e<float, false>(M, N, K, A, lda, (const float*)W, ldw, ep, D, ldd, 0.f, st);
}

nc_status launch_gemm_skinny_norm(int dtype, int M, int N, int K, const float* x, int64_t ldx, const void* W,
                                  int64_t ldw, int ep, void* D, int64_t ldd, float eps, cudaStream_t st) {
  if (M < 1 || M > SK_WARPS || N < 1 || K < 8 || K % 8 || ldx % 4 || ldw % 8 ||
      (ep != NC_EP_STORE && ep != NC_EP_STORE_F32 && ep != NC_EP_ACCUM_F32 && ep != NC_EP_RELU2_SQ))
    return NC_ERR_ARG;
  if ((((uintptr_t)x) & 15) || (((uintptr_t)W) & 15)) return NC_ERR_ARG;
  if (dtype == NC_BF16) return skinny_e<bf16, true>(M, N, K, x, ldx, (const bf16*)W, ldw, ep, D, ldd, eps, st);
  return skinny_e<float, true>(M, N, K, x, ldx, (const float*)W, ldw, ep, D, ldd, eps, st);
}
