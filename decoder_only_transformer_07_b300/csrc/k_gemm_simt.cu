// Exact-fp32 GEMM for the fp32 compute mode: D[M,N] (op)= sum_k A(m,k) B(n,k),
// fp32 fused multiply-add only (no TF32), with the step's epilogues.
// A is [M][K] (K-major) or [K][M]; B is [N][K] or [K][N].
#include "nc_kernels.cuh"

#define SG_BM 64
#define SG_BN 64
#define SG_BK 16

template <typename T>
__device__ __forceinline__ void ep_apply(int ep, int64_t m, int64_t n, float acc, void* D,
                                         int64_t ldd, void* aux, int64_t ldaux) {
  switch (ep) {
    case NC_EP_STORE: ((T*)D)[m * ldd + n] = from_f32<T>(acc); break;
    case NC_EP_STORE_F32: ((float*)D)[m * ldd + n] = acc; break;
    case NC_EP_ACCUM_F32: ((float*)D)[m * ldd + n] += acc; break;
    case NC_EP_RELU2: {
      float r = fmaxf(acc, 0.f);
      ((T*)D)[m * ldd + n] = from_f32<T>(r);
      ((T*)aux)[m * ldaux + n] = from_f32<T>(r * r);
      break;
    }
    case NC_EP_RELU2_BWD: {
      float r = to_f32(((const T*)aux)[m * ldaux + n]);
      ((T*)D)[m * ldd + n] = from_f32<T>(acc * 2.f * r);
      break;
    }
    case NC_EP_RELU2_SQ: {
      float r = fmaxf(acc, 0.f);
      ((T*)D)[m * ldd + n] = from_f32<T>(r * r);
      break;
    }
    case NC_EP_RELU2_SQ_BWD: {
      float r = sqrtf(to_f32(((const T*)aux)[m * ldaux + n]));
      ((T*)D)[m * ldd + n] = from_f32<T>(acc * 2.f * r);
      break;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) k_gemm_simt(int M, int N, int K, const T* __restrict__ A, int64_t lda,
                                                   int a_kmajor, const T* __restrict__ B, int64_t ldb,
                                                   int b_kmajor, int ep, void* D, int64_t ldd, void* aux,
                                                   int64_t ldaux) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = (int64_t)blockIdx.y * SG_BM, n0 = (int64_t)blockIdx.x * SG_BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SG_BK) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      int idx = tid + 256 * r;
      int mm, kk;
      if (a_kmajor) { mm = idx / SG_BK; kk = idx % SG_BK; } else { mm = idx % SG_BM; kk = idx / SG_BM; }
      int64_t gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < M && gk < K) v = to_f32(a_kmajor ? A[gm * lda + gk] : A[gk * lda + gm]);
      As[kk][mm] = v;
      int nn;
      if (b_kmajor) { nn = idx / SG_BK; kk = idx % SG_BK; } else { nn = idx % SG_BN; kk = idx / SG_BN; }
      int64_t gn = n0 + nn;
      gk = k0 + kk;
      v = 0.f;
      if (gn < N && gk < K) v = to_f32(b_kmajor ? B[gn * ldb + gk] : B[gk * ldb + gn]);
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int64_t m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
      if (m < M && n < N) ep_apply<T>(ep, m, n, acc[i][j], D, ldd, aux, ldaux);
    }
}

nc_status launch_gemm_simt(int dtype, int M, int N, int K, const void* A, int64_t lda, int a_kmajor,
                           const void* B, int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd,
                           void* aux, int64_t ldaux, cudaStream_t st) {
  if (M <= 0 || N <= 0) return NC_OK;
  dim3 grid(cdiv(N, SG_BN), cdiv(M, SG_BM));
  if (grid.y > 65535) return NC_ERR_UNSUPPORTED;
  if (dtype == NC_BF16)
    k_gemm_simt<bf16><<<grid, 256, 0, st>>>(M, N, K, (const bf16*)A, lda, a_kmajor, (const bf16*)B, ldb,
                                            b_kmajor, ep, D, ldd, aux, ldaux);
  else
    k_gemm_simt<float><<<grid, 256, 0, st>>>(M, N, K, (const float*)A, lda, a_kmajor, (const float*)B, ldb,
                                             b_kmajor, ep, D, ldd, aux, ldaux);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
