// The optimizer step that follows the gradients (cosmicrealm
// "noao-chat-0-项目总体介绍" §2.2 and §4.2; woshipm nanochat analysis §六.1):
// Muon for the weight matrices, AdamW for the embedding and the output head.
//
// Muon (the published method: Jordan et al., 2024) per matrix W[rows, cols]:
//   M <- mu M + G;  U = G + mu M (Nesterov) or M;
//   X = U / (||U||_F + 1e-7), then `steps` times  X <- (a I + b A + c A^2) X
//   with A = X X^T (wide) — for a tall matrix the same map is X (a I + b A + c A^2)
//   with A = X^T X, so no transpose is ever formed; (a, b, c) = (3.4445,
//   -4.7750, 2.0315);  W <- W - lr sqrt(max(1, rows / cols)) X.
// AdamW (bias-corrected, decoupled weight decay) per element of wte / lm_head.
//
// The memory-bound parts are one launch each over every matrix of the model:
// each block owns a chunk of one tensor (found by binary search in the tensor
// list, which travels as a kernel parameter), so per-tensor sums of squares are
// block partials summed afterwards in a fixed order (bitwise reproducible).
// The products of the iteration run on the step's GEMM kernels (tcgen05 in
// bf16 mode, exact fp32 otherwise).
#include <algorithm>

#include "nc_kernels.cuh"

namespace {

constexpr int OPT_THREADS = 256;

__device__ __forceinline__ int opt_tensor_of(const OptTensors& tl, int blk) {
  int lo = 0, hi = tl.n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tl.chunk0[mid] <= blk) lo = mid; else hi = mid;
  }
  return lo;
}

template <typename T> __device__ __forceinline__ T to_act(float v);
template <> __device__ __forceinline__ float to_act<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 to_act<bf16>(float v) { return __float2bfloat16_rn(v); }
__device__ __forceinline__ float act_f(float v) { return v; }
__device__ __forceinline__ float act_f(bf16 v) { return __bfloat162float(v); }

// M <- mu M + G;  U = nesterov ? G + mu M : M;  partial[block] = sum of U^2 over the block's chunk.
__global__ void __launch_bounds__(OPT_THREADS) k_muon_momentum(const __grid_constant__ OptTensors tl,
                                                               const float* __restrict__ G, float* __restrict__ Mb,
                                                               float* __restrict__ U, float mu, int nesterov,
                                                               float* __restrict__ partial) {
  const int t = opt_tensor_of(tl, blockIdx.x);
  const int64_t e0 = (int64_t)(blockIdx.x - tl.chunk0[t]) * OPT_CHUNK;
  const int64_t e1 = min(tl.len[t], e0 + OPT_CHUNK);
  const float* g = G + tl.off[t];
  float* mb = Mb + tl.soff[t];
  float* u = U + tl.soff[t];
  float ss = 0.f;
  for (int64_t e = e0 + threadIdx.x; e < e1; e += OPT_THREADS) {
    const float gv = g[e];
    const float m = fmaf(mu, mb[e], gv);
    mb[e] = m;
    const float uv = nesterov ? fmaf(mu, m, gv) : m;
    u[e] = uv;
    ss = fmaf(uv, uv, ss);
  }
  __shared__ float red[OPT_THREADS / 32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < OPT_THREADS / 32; ++w) s += red[w];
    partial[blockIdx.x] = s;
  }
}

// norm[t] = sqrt(sum of tensor t's partials), summed in chunk order; one warp per tensor.
__global__ void k_norm_finalize(const __grid_constant__ OptTensors tl, const float* __restrict__ partial,
                                float* __restrict__ norm) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= tl.n) return;
  double s = 0.0;
  for (int c = tl.chunk0[t] + lane; c < tl.chunk0[t + 1]; c += 32) s += (double)partial[c];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) norm[t] = (float)sqrt(s);
}

// X = U / (norm + eps) in the compute dtype.
template <typename T>
__global__ void __launch_bounds__(OPT_THREADS) k_ns_init(const __grid_constant__ OptTensors tl,
                                                         const float* __restrict__ U, const float* __restrict__ norm,
                                                         float eps, T* __restrict__ X) {
  const int t = opt_tensor_of(tl, blockIdx.x);
  const int64_t e0 = (int64_t)(blockIdx.x - tl.chunk0[t]) * OPT_CHUNK;
  const int64_t e1 = min(tl.len[t], e0 + OPT_CHUNK);
  const float inv = 1.f / (norm[t] + eps);
  const float* u = U + tl.soff[t];
  T* x = X + tl.soff[t];
  for (int64_t e = e0 + threadIdx.x; e < e1; e += OPT_THREADS) x[e] = to_act<T>(u[e] * inv);
}

// B = c A2 + b A + a I (n x n, written over A2), for `gridDim.y` matrices whose
// rows start nr rows apart (padding rows after each are left alone).  One
// block per row: eight elements per thread and step in 16-byte pieces when
// the rows allow, else one at a time.
template <typename T>
__global__ void __launch_bounds__(256) k_ns_poly(int n, int64_t nr, const T* __restrict__ A, T* __restrict__ A2,
                                                 float a, float b, float c) {
  const int r = blockIdx.x;
  const int64_t base = ((int64_t)blockIdx.y * nr + r) * n;
  const T* ar = A + base;
  T* br = A2 + base;
  constexpr int V = 16 / sizeof(T);   // elements per 16-byte piece
  if (n % V == 0) {
    for (int c0 = threadIdx.x * V; c0 < n; c0 += blockDim.x * V) {
      uint4 ua = *reinterpret_cast<const uint4*>(ar + c0);
      uint4 ub = *reinterpret_cast<const uint4*>(br + c0);
      const T* ea = reinterpret_cast<const T*>(&ua);
      T* eb = reinterpret_cast<T*>(&ub);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        float v = fmaf(c, act_f(eb[e]), b * act_f(ea[e]));
        if (c0 + e == r) v += a;
        eb[e] = to_act<T>(v);
      }
      *reinterpret_cast<uint4*>(br + c0) = ub;
    }
  } else {
    for (int col = threadIdx.x; col < n; col += blockDim.x) {
      float v = fmaf(c, act_f(br[col]), b * act_f(ar[col]));
      if (col == r) v += a;
      br[col] = to_act<T>(v);
    }
  }
}

// W <- W - lr X for every tensor t of tl: W at master + tl.off[t], X (compute
// dtype) at X + tl.soff[t], tl.len[t] elements; one block per chunk.
template <typename T>
__global__ void __launch_bounds__(OPT_THREADS) k_muon_apply_multi(const __grid_constant__ OptTensors tl,
                                                                  float* __restrict__ W, const T* __restrict__ X,
                                                                  float lr) {
  const int t = opt_tensor_of(tl, blockIdx.x);
  const int64_t e0 = (int64_t)(blockIdx.x - tl.chunk0[t]) * OPT_CHUNK;
  const int64_t e1 = min(tl.len[t], e0 + OPT_CHUNK);
  float* w = W + tl.off[t];
  const T* x = X + tl.soff[t];
  for (int64_t e = e0 + threadIdx.x; e < e1; e += OPT_THREADS) w[e] = fmaf(-lr, act_f(x[e]), w[e]);
}

// W <- W - lr X over one tensor.
template <typename T>
__global__ void k_muon_apply(int64_t n, float* __restrict__ W, const T* __restrict__ X, float lr) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    W[i] = fmaf(-lr, act_f(X[i]), W[i]);
}

template <typename T>
__global__ void k_cast_out(int64_t n, const T* __restrict__ X, float* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = act_f(X[i]);
}

__global__ void k_adamw(int64_t n, float* __restrict__ W, const float* __restrict__ G, float* __restrict__ m,
                        float* __restrict__ v, float lr, float b1, float b2, float eps, float wd, float inv_bc1,
                        float inv_bc2) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float g = G[i];
    const float mi = fmaf(b1, m[i], (1.f - b1) * g);
    const float vi = fmaf(b2, v[i], (1.f - b2) * g * g);
    m[i] = mi;
    v[i] = vi;
    const float w = W[i];
    W[i] = w - lr * (mi * inv_bc1 / (sqrtf(vi * inv_bc2) + eps) + wd * w);
  }
}

int grid_for(int64_t n) {
  const int64_t cap = (int64_t)(g_num_sms > 0 ? g_num_sms : 148) * 16;
  return (int)std::min<int64_t>((n + 255) / 256, cap);
}

}  // namespace

nc_status launch_muon_momentum(const OptTensors& tl, const float* G, float* M, float* U, float mu, int nesterov,
                               float* partial, cudaStream_t st) {
  const int nb = tl.chunk0[tl.n];
  if (nb <= 0) return NC_OK;
  k_muon_momentum<<<nb, OPT_THREADS, 0, st>>>(tl, G, M, U, mu, nesterov, partial);
  NC_CUDA_TRY(cudaGetLastError());
  k_norm_finalize<<<(tl.n + 7) / 8, 256, 0, st>>>(tl, partial, tl.norm);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_ns_init(int dtype, const OptTensors& tl, const float* U, float eps, void* X, cudaStream_t st) {
  const int nb = tl.chunk0[tl.n];
  if (nb <= 0) return NC_OK;
  if (dtype == NC_BF16) k_ns_init<bf16><<<nb, OPT_THREADS, 0, st>>>(tl, U, tl.norm, eps, (bf16*)X);
  else k_ns_init<float><<<nb, OPT_THREADS, 0, st>>>(tl, U, tl.norm, eps, (float*)X);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// `steps` iterations on X[rows, cols] (compute dtype); X0 is read from `x0` and
// the result left in one of ping[0], ping[1] (returned through *out).  A and A2
// hold min(rows, cols)^2 elements each.
nc_status newton_schulz_run(int dtype, int rows, int cols, int steps, const void* x0, void* ping0, void* ping1,
                            void* A, void* A2, const void** out, int32_t* err, void* gemm_ws, size_t gemm_ws_bytes,
                            cudaStream_t st) {
  const float ca = 3.4445f, cb = -4.7750f, cc = 2.0315f;
  const bool tall = rows > cols;
  const int n = tall ? cols : rows;          // A is n x n
  const void* cur = x0;
  void* ping[2] = {ping0, ping1};
  auto gemm = [&](int M, int N, int K, const void* a, int64_t lda, int akm, const void* b, int64_t ldb, int bkm,
                  void* d, int64_t ldd) -> nc_status {
    if (dtype == NC_BF16)
      return launch_gemm_tc(M, N, K, (const bf16*)a, lda, akm, (const bf16*)b, ldb, bkm, NC_EP_STORE, d, ldd, nullptr,
                            0, err, gemm_ws, gemm_ws_bytes, st);
    return launch_gemm_simt(NC_FP32, M, N, K, a, lda, akm, b, ldb, bkm, NC_EP_STORE, d, ldd, nullptr, 0, st);
  };
  for (int it = 0; it < steps; ++it) {
    void* nxt = ping[it & 1];
    if (!tall) {
      // A = X X^T (K = cols), A2 = A A, B = c A2 + b A + a I, X <- B X
      NC_TRY(gemm(n, n, cols, cur, cols, 1, cur, cols, 1, A, n));
      NC_TRY(gemm(n, n, n, A, n, 1, A, n, 1, A2, n));
    } else {
      // A = X^T X (K = rows; both operands are X read MN-major), X <- X B
      NC_TRY(gemm(n, n, rows, cur, cols, 0, cur, cols, 0, A, n));
      NC_TRY(gemm(n, n, n, A, n, 1, A, n, 1, A2, n));
    }
    if (dtype == NC_BF16) k_ns_poly<bf16><<<dim3(n, 1), 256, 0, st>>>(n, n, (const bf16*)A, (bf16*)A2, ca, cb, cc);
    else k_ns_poly<float><<<dim3(n, 1), 256, 0, st>>>(n, n, (const float*)A, (float*)A2, ca, cb, cc);
    NC_CUDA_TRY(cudaGetLastError());
    if (!tall) NC_TRY(gemm(rows, cols, rows, A2, n, 1, cur, cols, 0, nxt, cols));
    else NC_TRY(gemm(rows, cols, cols, cur, cols, 1, A2, n, 1, nxt, cols));
    cur = nxt;
  }
  *out = cur;
  return NC_OK;
}

// The iteration above on `batch` bf16 matrices X_b [rows, cols] at once (the
// same products, one batched launch each, so that a step of many small
// matrices fills the GPU).  X_b starts b * xr rows into ping0 (xr >= rows
// rounded up to 256; the padding rows take the tiles' spill), A and A2 hold
// the n x n products with row stride nr (>= n rounded up to 256).  rows must
// be a multiple of 128 (an MN-major operand's K).  The result is left in
// ping0 or ping1 (returned through *out).
nc_status newton_schulz_batched(int batch, int rows, int cols, int steps, void* ping0, void* ping1, int64_t xr,
                                void* A, void* A2, int64_t nr, const void** out, int32_t* err, cudaStream_t st) {
  const float ca = 3.4445f, cb = -4.7750f, cc = 2.0315f;
  const bool tall = rows > cols;
  const int n = tall ? cols : rows;
  if (rows % 128 || xr < (rows + 255) / 256 * 256 || nr < (n + 255) / 256 * 256) return NC_ERR_ARG;
  bf16* ping[2] = {(bf16*)ping0, (bf16*)ping1};
  bf16 *a = (bf16*)A, *a2 = (bf16*)A2;
  for (int it = 0; it < steps; ++it) {
    const bf16* cur = ping[it & 1];
    bf16* nxt = ping[(it + 1) & 1];
    if (!tall) {
      // A = X X^T, A2 = A A (A symmetric), B = c A2 + b A + a I, X <- B X (X read MN-major)
      NC_TRY(launch_gemm_tc_batched(batch, n, n, cols, cur, cols, 1, xr, cur, cols, 1, xr, a, n, nr, err, st));
      NC_TRY(launch_gemm_tc_batched(batch, n, n, n, a, n, 1, nr, a, n, 1, nr, a2, n, nr, err, st));
    } else {
      // A = X^T X (both operands X read MN-major), X <- X B
      NC_TRY(launch_gemm_tc_batched(batch, n, n, rows, cur, cols, 0, xr, cur, cols, 0, xr, a, n, nr, err, st));
      NC_TRY(launch_gemm_tc_batched(batch, n, n, n, a, n, 1, nr, a, n, 1, nr, a2, n, nr, err, st));
    }
    k_ns_poly<bf16><<<dim3(n, batch), 256, 0, st>>>(n, nr, a, a2, ca, cb, cc);
    NC_CUDA_TRY(cudaGetLastError());
    if (!tall)
      NC_TRY(launch_gemm_tc_batched(batch, rows, cols, rows, a2, n, 1, nr, cur, cols, 0, xr, nxt, cols, xr, err, st));
    else
      NC_TRY(launch_gemm_tc_batched(batch, rows, cols, cols, cur, cols, 1, xr, a2, n, 1, nr, nxt, cols, xr, err, st));
  }
  *out = ping[steps & 1];
  return NC_OK;
}

nc_status launch_muon_apply(int dtype, int64_t n, float* W, const void* X, float lr, cudaStream_t st) {
  if (n <= 0) return NC_OK;
  if (dtype == NC_BF16) k_muon_apply<bf16><<<grid_for(n), 256, 0, st>>>(n, W, (const bf16*)X, lr);
  else k_muon_apply<float><<<grid_for(n), 256, 0, st>>>(n, W, (const float*)X, lr);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_muon_apply_multi(int dtype, const OptTensors& tl, float* W, const void* X, float lr, cudaStream_t st) {
  const int nb = tl.chunk0[tl.n];
  if (nb <= 0) return NC_OK;
  if (dtype == NC_BF16) k_muon_apply_multi<bf16><<<nb, OPT_THREADS, 0, st>>>(tl, W, (const bf16*)X, lr);
  else k_muon_apply_multi<float><<<nb, OPT_THREADS, 0, st>>>(tl, W, (const float*)X, lr);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_cast_out(int dtype, int64_t n, const void* X, float* out, cudaStream_t st) {
  if (n <= 0) return NC_OK;
  if (dtype == NC_BF16) k_cast_out<bf16><<<grid_for(n), 256, 0, st>>>(n, (const bf16*)X, out);
  else k_cast_out<float><<<grid_for(n), 256, 0, st>>>(n, (const float*)X, out);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_adamw(int64_t n, float* W, const float* G, float* m, float* v, float lr, float b1, float b2,
                       float eps, float wd, int64_t t, cudaStream_t st) {
  if (n <= 0) return NC_OK;
  const float inv_bc1 = (float)(1.0 / (1.0 - pow((double)b1, (double)t)));
  const float inv_bc2 = (float)(1.0 / (1.0 - pow((double)b2, (double)t)));
  k_adamw<<<grid_for(n), 256, 0, st>>>(n, W, G, m, v, lr, b1, b2, eps, wd, inv_bc1, inv_bc2);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
