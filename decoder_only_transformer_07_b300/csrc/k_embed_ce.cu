// Token embedding gather and its deterministic scatter-add backward, and the
// next-token cross-entropy with its gradient.
//
// The embedding `wte` is a separate (untied) table read by token id
// (cosmicrealm "noao-chat-0-项目总体介绍" §2.1 item 3); the loss is next-token
// cross-entropy (devpress "用不到100美元，亲手训练一个属于你的GPT-2" §2.2 item 2).
#include <algorithm>

#include "nc_kernels.cuh"
#include "nc_ptx.cuh"

// ---------------------------------------------------------------- gather
// One warp per token row: x[i] = float(round_act(wte[tokens[i]])).  An id
// outside [0, V) sets the token error bit and writes a zero row.  With NORM
// (the variant with a norm after the embedding) the row is then RMS-normalised
// in fp32, x[i] = e * rstd with rstd = 1/sqrt(mean(e^2) + eps) saved per row,
// the arithmetic of the step's RMSNorm kernel.
template <typename T, bool NORM>
__global__ void k_embed_fwd(int64_t n, int C, int V, const int32_t* __restrict__ tokens,
                            const float* __restrict__ wte, float* __restrict__ x,
                            int32_t* __restrict__ err, float* __restrict__ rstd, float eps) {
  int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (i >= n) return;
  int tok = tokens[i];
  bool ok = tok >= 0 && tok < V;
  if (!ok && lane == 0 && err) atomicOr(err, NC_DEVERR_TOKEN);
  const float4* src = reinterpret_cast<const float4*>(wte + (int64_t)(ok ? tok : 0) * C);
  float4* dst = reinterpret_cast<float4*>(x + i * C);
  float r = 1.f;
  if (NORM) {
    float ss = 0.f;
    for (int c = lane; c < C / 4; c += 32) {
      float4 v = ok ? src[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      v.x = round_act<T>(v.x); v.y = round_act<T>(v.y);
      v.z = round_act<T>(v.z); v.w = round_act<T>(v.w);
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = warp_sum(ss);
    r = rsqrtf(ss / (float)C + eps);
    if (lane == 0) rstd[i] = r;
  }
  for (int c = lane; c < C / 4; c += 32) {
    float4 v = ok ? src[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    v.x = round_act<T>(v.x); v.y = round_act<T>(v.y);
    v.z = round_act<T>(v.z); v.w = round_act<T>(v.w);
    if (NORM) { v.x *= r; v.y *= r; v.z *= r; v.w *= r; }
    dst[c] = v;
  }
}

nc_status launch_embed_fwd(int dtype, int64_t n, int C, int V, const int32_t* tokens,
                           const float* wte, float* x, int32_t* err, cudaStream_t st, float* rstd, float eps) {
  if (n <= 0) return NC_OK;
  if (C % 4 || (((uintptr_t)wte) & 15) || (((uintptr_t)x) & 15)) return NC_ERR_ARG;
  const unsigned g = (unsigned)cdiv(n, 8);
  if (rstd) {
    if (dtype == NC_BF16) k_embed_fwd<bf16, true><<<g, 256, 0, st>>>(n, C, V, tokens, wte, x, err, rstd, eps);
    else k_embed_fwd<float, true><<<g, 256, 0, st>>>(n, C, V, tokens, wte, x, err, rstd, eps);
  } else {
    if (dtype == NC_BF16) k_embed_fwd<bf16, false><<<g, 256, 0, st>>>(n, C, V, tokens, wte, x, err, nullptr, 0.f);
    else k_embed_fwd<float, false><<<g, 256, 0, st>>>(n, C, V, tokens, wte, x, err, nullptr, 0.f);
  }
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// Backward of the norm after the embedding, in place on dx (float [n, C]):
// dx <- rstd * (dx - y * mean(dx * y)) with y = round_act(wte[tok]) * rstd
// recomputed from the table (one warp per row).  Rows of out-of-range ids
// (reported by the forward) are left as they are.
template <typename T>
__global__ void k_embed_norm_bwd(int64_t n, int C, int V, const int32_t* __restrict__ tokens,
                                 const float* __restrict__ wte, const float* __restrict__ rstd,
                                 float* __restrict__ dx) {
  int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (i >= n) return;
  const int tok = tokens[i];
  if (tok < 0 || tok >= V) return;
  const float4* src = reinterpret_cast<const float4*>(wte + (int64_t)tok * C);
  float4* d = reinterpret_cast<float4*>(dx + i * C);
  const float r = rstd[i];
  float dot = 0.f;
  for (int c = lane; c < C / 4; c += 32) {
    const float4 e = src[c], g = d[c];
    dot += g.x * (round_act<T>(e.x) * r) + g.y * (round_act<T>(e.y) * r) + g.z * (round_act<T>(e.z) * r) +
           g.w * (round_act<T>(e.w) * r);
  }
  dot = warp_sum(dot) / (float)C;
  for (int c = lane; c < C / 4; c += 32) {
    const float4 e = src[c];
    float4 g = d[c];
    g.x = r * (g.x - round_act<T>(e.x) * r * dot);
    g.y = r * (g.y - round_act<T>(e.y) * r * dot);
    g.z = r * (g.z - round_act<T>(e.z) * r * dot);
    g.w = r * (g.w - round_act<T>(e.w) * r * dot);
    d[c] = g;
  }
}

nc_status launch_embed_norm_bwd(int dtype, int64_t n, int C, int V, const int32_t* tokens, const float* wte,
                                const float* rstd, float* dx, cudaStream_t st) {
  if (n <= 0) return NC_OK;
  if (C % 4 || (((uintptr_t)wte) & 15) || (((uintptr_t)dx) & 15)) return NC_ERR_ARG;
  if (dtype == NC_BF16) k_embed_norm_bwd<bf16><<<(unsigned)cdiv(n, 8), 256, 0, st>>>(n, C, V, tokens, wte, rstd, dx);
  else k_embed_norm_bwd<float><<<(unsigned)cdiv(n, 8), 256, 0, st>>>(n, C, V, tokens, wte, rstd, dx);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// ---------------------------------------------------------------- scatter
// dwte[v] = sum of dx[i] over i with tokens[i] == v, in increasing i.
//  1. chunks of EMB_CH positions: sort (token, position) in shared memory,
//     sum each run of equal tokens in position order into one partial row;
//  2. count partial rows per token, exclusive scan -> offsets;
//  3. list each token's partial rows (slot order arbitrary);
//  4. per token row: sort its partial slots (= chunk order), add them in that
//     order; ids that never occur get +0.0.
// Every floating-point sum has a fixed order, so the result is bitwise
// reproducible.
#define EMB_CH 256
#define EMB_MAXV4 8          // C <= 4 * 8 * EMB_CH = 8192
#define EMB_MAX_CHUNKS 4096  // n <= 2^20

struct EmbScratch {
  float* partial;   // [n, C]
  int* run_tok;     // [n]
  int* nruns;       // [nchunks]
  int* count;       // [V]
  int* offs;        // [V]
  int* cursor;      // [V]
  int* list;        // [n]
};

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

static EmbScratch emb_carve(void* base, int64_t n, int C, int V) {
  EmbScratch s;
  char* p = (char*)base;
  int64_t nchunks = (n + EMB_CH - 1) / EMB_CH;
  s.partial = (float*)p; p += align256((size_t)n * C * sizeof(float));
  s.run_tok = (int*)p; p += align256((size_t)n * sizeof(int));
  s.nruns = (int*)p; p += align256((size_t)nchunks * sizeof(int));
  s.count = (int*)p; p += align256((size_t)V * sizeof(int));
  s.offs = (int*)p; p += align256((size_t)V * sizeof(int));
  s.cursor = (int*)p; p += align256((size_t)V * sizeof(int));
  s.list = (int*)p; p += align256((size_t)n * sizeof(int));
  return s;
}

size_t embed_bwd_scratch_bytes(int64_t n, int C, int V) {
  int64_t nchunks = (n + EMB_CH - 1) / EMB_CH;
  return align256((size_t)n * C * sizeof(float)) + 2 * align256((size_t)n * sizeof(int)) +
         align256((size_t)nchunks * sizeof(int)) + 3 * align256((size_t)V * sizeof(int));
}

// Bitonic sort of `len` (power of two, <= blockDim.x * k) keys in shared memory.
template <typename K>
__device__ void block_bitonic_sort(K* keys, int len) {
  for (int size = 2; size <= len; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < len; i += blockDim.x) {
        int j = i ^ stride;
        if (j > i) {
          bool up = ((i & size) == 0);
          K a = keys[i], b = keys[j];
          if ((a > b) == up) { keys[i] = b; keys[j] = a; }
        }
      }
    }
  }
  __syncthreads();
}

// A position whose id lies outside [0, V) sets the token error bit and takes
// part in no run: its key is the sentinel ~0 (which sorts last and which no
// valid id can produce, since V < 2^31), so no count, offset or list slot is
// ever formed from it.
__global__ void __launch_bounds__(EMB_CH) k_emb_bwd_runs(int64_t n, int C, int V, const int32_t* __restrict__ tokens,
                                                          const float* __restrict__ dx, EmbScratch s,
                                                          int32_t* __restrict__ err) {
  __shared__ unsigned long long keys[EMB_CH];
  __shared__ int run_of[EMB_CH];
  const int64_t base = (int64_t)blockIdx.x * EMB_CH;
  const int tid = threadIdx.x;
  int64_t i = base + tid;
  bool in_range = false;
  unsigned long long key = ~0ull;
  if (i < n) {
    const int tok = tokens[i];
    in_range = (unsigned)tok < (unsigned)V;
    if (in_range) key = ((unsigned long long)(unsigned)tok << 32) | (unsigned)tid;
    else if (err) atomicOr(err, NC_DEVERR_TOKEN);
  }
  keys[tid] = key;
  // the in-range positions, which the sort places first
  const int valid = __syncthreads_count(in_range);
  block_bitonic_sort(keys, EMB_CH);
  // run index of each sorted position (inclusive scan of run starts; EMB_CH is small)
  if (tid == 0) {
    int r = -1;
    for (int k = 0; k < valid; ++k) {
      if (k == 0 || (keys[k] >> 32) != (keys[k - 1] >> 32)) {
        ++r;
        int v = (int)(keys[k] >> 32);
        s.run_tok[base + r] = v;
        atomicAdd(&s.count[v], 1);
      }
      run_of[k] = r;
    }
    s.nruns[blockIdx.x] = r + 1;
  }
  __syncthreads();
  const int C4 = C / 4;
  float4 acc[EMB_MAXV4];
#pragma unroll
  for (int k = 0; k < EMB_MAXV4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < valid; ++k) {
    const float4* row = reinterpret_cast<const float4*>(dx + (base + (int)(keys[k] & 0xffffffffu)) * C);
#pragma unroll
    for (int q = 0; q < EMB_MAXV4; ++q) {
      int c = tid + q * EMB_CH;
      if (c < C4) {
        float4 v = row[c];
        acc[q].x += v.x; acc[q].y += v.y; acc[q].z += v.z; acc[q].w += v.w;
      }
    }
    if (k == valid - 1 || run_of[k + 1] != run_of[k]) {
      float4* dst = reinterpret_cast<float4*>(s.partial + (base + run_of[k]) * C);
#pragma unroll
      for (int q = 0; q < EMB_MAXV4; ++q) {
        int c = tid + q * EMB_CH;
        if (c < C4) dst[c] = acc[q];
        acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// Exclusive scan of count[V] into offs[V]; one block of 1024 threads.
__global__ void __launch_bounds__(1024) k_emb_bwd_scan(int V, const int* __restrict__ count, int* __restrict__ offs) {
  __shared__ int part[1024];
  const int per = (V + 1023) / 1024;
  const int a = threadIdx.x * per, b = min(V, a + per);
  int sum = 0;
  for (int v = a; v < b; ++v) sum += count[v];
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    int t = (threadIdx.x >= off) ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += t;
    __syncthreads();
  }
  int run = part[threadIdx.x] - sum;
  for (int v = a; v < b; ++v) { offs[v] = run; run += count[v]; }
}

__global__ void k_emb_bwd_list(EmbScratch s) {
  const int64_t base = (int64_t)blockIdx.x * EMB_CH;
  int r = threadIdx.x;
  if (r >= s.nruns[blockIdx.x]) return;
  int v = s.run_tok[base + r];
  int pos = atomicAdd(&s.cursor[v], 1);
  s.list[s.offs[v] + pos] = (int)(base + r);
}

__global__ void __launch_bounds__(256) k_emb_bwd_rows(int V, int C, EmbScratch s, float* __restrict__ dwte,
                                                      int accumulate) {
  __shared__ int slots[EMB_MAX_CHUNKS];
  const int v = blockIdx.x;
  const int cnt = s.count[v];
  float4* dst = reinterpret_cast<float4*>(dwte + (int64_t)v * C);
  const int C4 = C / 4;
  if (cnt == 0) {
    if (!accumulate)
      for (int c = threadIdx.x; c < C4; c += blockDim.x) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  auto put = [&](int c, float4 v4) {
    if (accumulate) {
      const float4 d = dst[c];
      v4.x += d.x; v4.y += d.y; v4.z += d.z; v4.w += d.w;
    }
    dst[c] = v4;
  };
  const int o = s.offs[v];
  if (cnt == 1) {
    const float4* src = reinterpret_cast<const float4*>(s.partial + (int64_t)s.list[o] * C);
    for (int c = threadIdx.x; c < C4; c += blockDim.x) put(c, src[c]);
    return;
  }
  int len = 1;
  while (len < cnt) len <<= 1;
  for (int k = threadIdx.x; k < len; k += blockDim.x) slots[k] = (k < cnt) ? s.list[o + k] : 0x7fffffff;
  block_bitonic_sort(slots, len);
  for (int c = threadIdx.x; c < C4; c += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < cnt; ++k) {
      float4 p = reinterpret_cast<const float4*>(s.partial + (int64_t)slots[k] * C)[c];
      acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
    }
    put(c, acc);
  }
}

nc_status launch_embed_bwd(int64_t n, int C, int V, const int32_t* tokens, const float* dx,
                           float* dwte, void* scratch, cudaStream_t st, int accumulate, int32_t* err) {
  if (C % 4 || C > 4 * EMB_MAXV4 * EMB_CH || V <= 0) return NC_ERR_ARG;
  int64_t nchunks = (n + EMB_CH - 1) / EMB_CH;
  if (nchunks > EMB_MAX_CHUNKS) return NC_ERR_UNSUPPORTED;
  if (!scratch || (((uintptr_t)scratch) & 255)) return NC_ERR_ARG;
  EmbScratch s = emb_carve(scratch, n, C, V);
  NC_CUDA_TRY(cudaMemsetAsync(s.count, 0, sizeof(int) * (size_t)V, st));
  NC_CUDA_TRY(cudaMemsetAsync(s.cursor, 0, sizeof(int) * (size_t)V, st));
  if (nchunks > 0) {
    k_emb_bwd_runs<<<(unsigned)nchunks, EMB_CH, 0, st>>>(n, C, V, tokens, dx, s, err);
    NC_CUDA_TRY(cudaGetLastError());
  }
  k_emb_bwd_scan<<<1, 1024, 0, st>>>(V, s.count, s.offs);
  NC_CUDA_TRY(cudaGetLastError());
  if (nchunks > 0) {
    k_emb_bwd_list<<<(unsigned)nchunks, EMB_CH, 0, st>>>(s);
    NC_CUDA_TRY(cudaGetLastError());
  }
  k_emb_bwd_rows<<<V, 256, 0, st>>>(V, C, s, dwte, accumulate);
  NC_CUDA_TRY(cudaGetLastError());
  return NC_OK;
}

// ---------------------------------------------------------------- cross-entropy
// One block per row.  row_loss = logsumexp(z) - z[target];
// z <- (softmax(z) - onehot(target)) * scale, in place.
//
// CAP (the logit soft-cap variant, cap = c > 0): every logit enters as
// zc = c tanh(z / c), and the gradient written is the one with respect to the
// raw z, (softmax(zc) - onehot) * (1 - tanh(z / c)^2) * scale.  The fp32
// kernel evaluates tanhf; the bf16 kernels take tanh and its derivative from
// one SFU exponential (tanh_sech2).
template <typename T, bool CAP>
__global__ void __launch_bounds__(512) k_cross_entropy(int V, T* __restrict__ z, int64_t ldz,
                                                       const int32_t* __restrict__ targets,
                                                       float* __restrict__ row_loss, float scale,
                                                       int32_t* __restrict__ err, float cap) {
  __shared__ float sh[32];
  const int64_t row = blockIdx.x;
  T* zr = z + row * ldz;
  const float icap = CAP ? 1.f / cap : 0.f;
  auto capped = [&](float v) { return CAP ? cap * tanhf(v * icap) : v; };
  float m = -INFINITY;
  for (int v = threadIdx.x; v < V; v += blockDim.x) m = fmaxf(m, capped(to_f32(zr[v])));
  m = block_max(m, sh);
  float s = 0.f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(capped(to_f32(zr[v])) - m);
  s = block_sum(s, sh);
  const float lse = m + logf(s);
  const int tgt = targets[row];
  const bool ok = tgt >= 0 && tgt < V;
  if (threadIdx.x == 0) {
    if (!ok && err) atomicOr(err, NC_DEVERR_TOKEN);
    row_loss[row] = ok ? lse - capped(to_f32(zr[tgt])) : 0.f;
  }
  __syncthreads();   // z[tgt] is read above before any thread overwrites it
  const float inv = 1.f / s;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float zv = to_f32(zr[v]);
    const float t = CAP ? tanhf(zv * icap) : 0.f;
    float p = expf((CAP ? cap * t : zv) - m) * inv;
    if (v == tgt) p -= 1.f;
    if (CAP) p *= 1.f - t * t;
    zr[v] = from_f32<T>(p * scale);
  }
}

__device__ __forceinline__ uint4 pack8_bf16_rn(const float* p) {
  uint4 o;
  __nv_bfloat162 q0 = __floats2bfloat162_rn(p[0], p[1]), q1 = __floats2bfloat162_rn(p[2], p[3]);
  __nv_bfloat162 q2 = __floats2bfloat162_rn(p[4], p[5]), q3 = __floats2bfloat162_rn(p[6], p[7]);
  o.x = *reinterpret_cast<uint32_t*>(&q0);
  o.y = *reinterpret_cast<uint32_t*>(&q1);
  o.z = *reinterpret_cast<uint32_t*>(&q2);
  o.w = *reinterpret_cast<uint32_t*>(&q3);
  return o;
}

// bf16 rows with V % 8 == 0 and V <= 8 * CE_THREADS * CE_VEC: the row is read once
// into registers (16-byte loads), reduced, and dz written from registers.
#define CE_THREADS 1024
#define CE_VEC 8
template <bool CAP>
__global__ void __launch_bounds__(CE_THREADS) k_cross_entropy_bf16(int V, bf16* __restrict__ z, int64_t ldz,
                                                                   const int32_t* __restrict__ targets,
                                                                   float* __restrict__ row_loss, float scale,
                                                                   int32_t* __restrict__ err, float cap) {
  __shared__ float sh[32];
  __shared__ float ztgt;
  const int64_t row = blockIdx.x;
  bf16* zr = z + row * ldz;
  const int nv = V / 8;
  const float icap = CAP ? 1.f / cap : 0.f;
  auto capped = [&](float v) {
    float d;
    return CAP ? cap * tanh_sech2(v * icap, &d) : v;
  };
  uint4 v[CE_VEC];
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < CE_VEC; ++k) {
    const int i = threadIdx.x + k * CE_THREADS;
    if (i < nv) {
      v[k] = reinterpret_cast<const uint4*>(zr)[i];
      const bf16* e = reinterpret_cast<const bf16*>(&v[k]);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, capped(__bfloat162float(e[j])));
    }
  }
  const int tgt = targets[row];
  const bool ok = tgt >= 0 && tgt < V;
  if (threadIdx.x == 0) ztgt = ok ? capped(__bfloat162float(zr[tgt])) : 0.f;
  m = block_max(m, sh);
  const float L2E = 1.4426950408889634f;
  const float mb = m * L2E;
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < CE_VEC; ++k) {
    const int i = threadIdx.x + k * CE_THREADS;
    if (i < nv) {
      const bf16* e = reinterpret_cast<const bf16*>(&v[k]);
#pragma unroll
      for (int j = 0; j < 8; ++j) sum += ex2_approx(fmaf(capped(__bfloat162float(e[j])), L2E, -mb));
    }
  }
  sum = block_sum(sum, sh);
  const float lse = m + logf(sum);
  if (threadIdx.x == 0) {
    if (!ok && err) atomicOr(err, NC_DEVERR_TOKEN);
    row_loss[row] = ok ? lse - ztgt : 0.f;
  }
  const float inv = scale / sum;
#pragma unroll
  for (int k = 0; k < CE_VEC; ++k) {
    const int i = threadIdx.x + k * CE_THREADS;
    if (i < nv) {
      const bf16* e = reinterpret_cast<const bf16*>(&v[k]);
      float p[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float zv = __bfloat162float(e[j]);
        float d = 1.f;
        const float t = CAP ? tanh_sech2(zv * icap, &d) : 0.f;
        p[j] = ex2_approx(fmaf(CAP ? cap * t : zv, L2E, -mb)) * inv;
        if (i * 8 + j == tgt) p[j] -= scale;
        if (CAP) p[j] *= d;
      }
      reinterpret_cast<uint4*>(zr)[i] = pack8_bf16_rn(p);
    }
  }
}

// Wide bf16 rows (V >= 16384): 256 threads per row and up to four rows per SM,
// so that one row's reductions overlap other rows' memory traffic.  Pass 1
// streams the row once for its maximum and sum of exponentials (online: the
// sum is rescaled when the maximum grows); pass 2 reads the row again, while
// it is still in L2, and writes dz in place.
#define CE2_THREADS 256
template <bool CAP>
__global__ void __launch_bounds__(CE2_THREADS, 4) k_cross_entropy_bf16_stream(int V, bf16* __restrict__ z, int64_t ldz,
                                                                             const int32_t* __restrict__ targets,
                                                                             float* __restrict__ row_loss, float scale,
                                                                             int32_t* __restrict__ err, float cap) {
  __shared__ float shm[CE2_THREADS / 32], shs[CE2_THREADS / 32];
  const int64_t row = blockIdx.x;
  bf16* zr = z + row * ldz;
  const uint4* zv = reinterpret_cast<const uint4*>(zr);
  const int nv = V / 8;
  const float L2E = 1.4426950408889634f;
  const float icap = CAP ? 1.f / cap : 0.f;
  auto capped = [&](float v) {
    float d;
    return CAP ? cap * tanh_sech2(v * icap, &d) : v;
  };
  float m = -INFINITY, sum = 0.f;   // m in log2 units
  for (int i0 = threadIdx.x; i0 < nv; i0 += 4 * CE2_THREADS) {
    uint4 u[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (i0 + q * CE2_THREADS < nv) u[q] = zv[i0 + q * CE2_THREADS];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (i0 + q * CE2_THREADS >= nv) break;
      const bf16* e = reinterpret_cast<const bf16*>(&u[q]);
      float x[8], cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        x[j] = capped(__bfloat162float(e[j])) * L2E;
        cm = fmaxf(cm, x[j]);
      }
      if (cm > m) {
        sum *= ex2_approx(m - cm);
        m = cm;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) sum += ex2_approx(x[j] - m);
    }
  }
  // (m, sum) over the block: warps by shuffles, then warp 0 over the warps
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, off), os = __shfl_xor_sync(0xffffffffu, sum, off);
    const float nm = fmaxf(m, om);
    sum = (m == -INFINITY ? 0.f : sum * ex2_approx(m - nm)) + (om == -INFINITY ? 0.f : os * ex2_approx(om - nm));
    m = nm;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { shm[warp] = m; shs[warp] = sum; }
  __syncthreads();
  if (warp == 0) {
    m = lane < CE2_THREADS / 32 ? shm[lane] : -INFINITY;
    sum = lane < CE2_THREADS / 32 ? shs[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, off), os = __shfl_xor_sync(0xffffffffu, sum, off);
      const float nm = fmaxf(m, om);
      sum = (m == -INFINITY ? 0.f : sum * ex2_approx(m - nm)) + (om == -INFINITY ? 0.f : os * ex2_approx(om - nm));
      m = nm;
    }
    if (lane == 0) { shm[0] = m; shs[0] = sum; }
  }
  __syncthreads();
  m = shm[0];
  sum = shs[0];
  const int tgt = targets[row];
  const bool ok = tgt >= 0 && tgt < V;
  if (threadIdx.x == 0) {
    const float ztgt = ok ? capped(__bfloat162float(zr[tgt])) : 0.f;
    if (!ok && err) atomicOr(err, NC_DEVERR_TOKEN);
    row_loss[row] = ok ? (m + log2f(sum)) * 0.69314718055994531f - ztgt : 0.f;
  }
  __syncthreads();   // zr[tgt] is read before pass 2 overwrites it
  const float inv = scale / sum;
  uint4* zw = reinterpret_cast<uint4*>(zr);
  for (int i = threadIdx.x; i < nv; i += CE2_THREADS) {
    const uint4 u = zv[i];
    const bf16* e = reinterpret_cast<const bf16*>(&u);
    float p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float zz = __bfloat162float(e[j]);
      float d = 1.f;
      const float t = CAP ? tanh_sech2(zz * icap, &d) : 0.f;
      p[j] = ex2_approx(fmaf(CAP ? cap * t : zz, L2E, -m)) * inv;
      if (i * 8 + j == tgt) p[j] -= scale;
      if (CAP) p[j] *= d;
    }
    zw[i] = pack8_bf16_rn(p);
  }
}

template <bool CAP>
static void launch_ce_t(int dtype, int64_t rows, int V, void* z, int64_t ldz, const int32_t* targets,
                        float* row_loss, float scale, int32_t* err, float cap, cudaStream_t st) {
  const bool vec = dtype == NC_BF16 && V % 8 == 0 && ldz % 8 == 0 && (((uintptr_t)z) & 15) == 0;
  const unsigned g = (unsigned)rows;
  if (vec && V >= 16384)
    k_cross_entropy_bf16_stream<CAP><<<g, CE2_THREADS, 0, st>>>(V, (bf16*)z, ldz, targets, row_loss, scale, err, cap);
  else if (vec && V <= 8 * CE_THREADS * CE_VEC)
    k_cross_entropy_bf16<CAP><<<g, CE_THREADS, 0, st>>>(V, (bf16*)z, ldz, targets, row_loss, scale, err, cap);
  else if (dtype == NC_BF16)
    k_cross_entropy<bf16, CAP><<<g, 512, 0, st>>>(V, (bf16*)z, ldz, targets, row_loss, scale, err, cap);
  else
    k_cross_entropy<float, CAP><<<g, 512, 0, st>>>(V, (float*)z, ldz, targets, row_loss, scale, err, cap);
}

nc_status launch_cross_entropy(int dtype, int64_t rows, int V, void* z, int64_t ldz,
                               const int32_t* targets, float* row_loss, float scale, int32_t* err,
                               cudaStream_t st, float softcap) {
  if (rows <= 0) return NC_OK;
  if (rows > 0x7fffffff) return NC_ERR_ARG;
  if (!(softcap >= 0.f) || softcap == INFINITY) return NC_ERR_ARG;
  if (softcap > 0.f) launch_ce_t<true>(dtype, rows, V, z, ldz, targets, row_loss, scale, err, softcap, st);
  else launch_ce_t<false>(dtype, rows, V, z, ldz, targets, row_loss, scale, err, 0.f, st);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// z <- c tanh(z / c) in place on n fp32 logits (the soft-cap variant's
// logits, for the entry points that return them).  Grid-stride, tanhf.
__global__ void k_softcap_f32(int64_t n, float* __restrict__ z, float cap) {
  const float icap = 1.f / cap;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    z[i] = cap * tanhf(z[i] * icap);
}

nc_status launch_softcap_f32(int64_t n, float* z, float cap, cudaStream_t st) {
  if (n <= 0 || cap <= 0.f) return NC_OK;
  const int64_t blocks = std::min<int64_t>(cdiv(n, 256), 148 * 16);
  k_softcap_f32<<<(unsigned)blocks, 256, 0, st>>>(n, z, cap);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

// Mean of row_loss[0..n) in a fixed order (fp64 partials), written to out[0].
__global__ void __launch_bounds__(1024) k_mean(int64_t n, const float* __restrict__ x, float* __restrict__ out) {
  __shared__ double part[1024];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += 1024) s += (double)x[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int off = 512; off > 0; off >>= 1) {
    if (threadIdx.x < off) part[threadIdx.x] += part[threadIdx.x + off];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[0] = (float)(part[0] / (double)n);
}

nc_status launch_mean(int64_t n, const float* x, float* out, cudaStream_t st) {
  k_mean<<<1, 1024, 0, st>>>(n, x, out);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}
