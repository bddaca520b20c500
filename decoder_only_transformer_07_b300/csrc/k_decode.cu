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
__global__ void k_kv_store(int64_t rows, int T, int t0, int H, int Hkv, int hd, const E* __restrict__ qkv, int64_t ld,
                           E* __restrict__ kc, E* __restrict__ vc, int max_len) {
  const int64_t per_row = (int64_t)Hkv * hd;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * per_row) return;
  const int64_t r = i / per_row;
  const int rem = (int)(i % per_row);
  const int g = rem / hd, d = rem % hd;
  const int64_t b = r / T;
  const int t = t0 + (int)(r % T);
  const int64_t dst = ((b * Hkv + g) * max_len + t) * hd + d;
  kc[dst] = qkv[r * ld + (int64_t)(H + g) * hd + d];
  vc[dst] = qkv[r * ld + (int64_t)(H + Hkv + g) * hd + d];
}

constexpr int DEC_CHUNK = 256;
constexpr int DEC_WARPS = 4;

// Partials: part[((b * H + h) * nsplit + s) * (HD + 2) + {0: max (log2 units), 1: sum, 2..: output}]
template <typename E, int HD, int G>
__global__ void __launch_bounds__(DEC_WARPS * 32)
    k_decode_attn(int H, int Hkv, int len, int nsplit, const E* __restrict__ qkv, int64_t ld,
                  const E* __restrict__ kc, const E* __restrict__ vc, int max_len, float scale_log2,
                  float* __restrict__ part) {
  constexpr int DPL = HD / 32;
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
nc_status decode_attn_t(int B, int H, int Hkv, int len, const E* qkv, int64_t ld, const E* kc, const E* vc,
                        int max_len, float* part, E* o, int64_t ldo, cudaStream_t st) {
  const int nsplit = (len + DEC_CHUNK - 1) / DEC_CHUNK;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  k_decode_attn<E, HD, G><<<dim3((unsigned)(B * Hkv), (unsigned)nsplit), DEC_WARPS * 32, 0, st>>>(
      H, Hkv, len, nsplit, qkv, ld, kc, vc, max_len, scale_log2, part);
  NC_CUDA_TRY(cudaGetLastError());
  const int64_t rows = (int64_t)B * H;
  k_decode_combine<E, HD><<<cdiv(rows, 8), 256, 0, st>>>(rows, nsplit, part, o, ldo, H);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

template <typename E, int HD>
nc_status decode_attn_g(int G, int B, int H, int Hkv, int len, const E* qkv, int64_t ld, const E* kc, const E* vc,
                        int max_len, float* part, E* o, int64_t ldo, cudaStream_t st) {
  switch (G) {
    case 1: return decode_attn_t<E, HD, 1>(B, H, Hkv, len, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 2: return decode_attn_t<E, HD, 2>(B, H, Hkv, len, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 3: return decode_attn_t<E, HD, 3>(B, H, Hkv, len, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 4: return decode_attn_t<E, HD, 4>(B, H, Hkv, len, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    case 8: return decode_attn_t<E, HD, 8>(B, H, Hkv, len, qkv, ld, kc, vc, max_len, part, o, ldo, st);
    default: return NC_ERR_UNSUPPORTED;
  }
}

}  // namespace

size_t decode_part_floats(int B, int H, int hd, int max_len) {
  return (size_t)B * H * ((max_len + DEC_CHUNK - 1) / DEC_CHUNK) * (hd + 2);
}

nc_status launch_kv_store(int dtype, int64_t rows, int T, int t0, int H, int Hkv, int hd, const void* qkv, int64_t ld,
                          void* kc, void* vc, int max_len, cudaStream_t st) {
  const int64_t n = rows * Hkv * hd;
  if (n <= 0) return NC_OK;
  if (dtype == NC_BF16)
    k_kv_store<bf16><<<cdiv(n, 256), 256, 0, st>>>(rows, T, t0, H, Hkv, hd, (const bf16*)qkv, ld, (bf16*)kc,
                                                    (bf16*)vc, max_len);
  else
    k_kv_store<float><<<cdiv(n, 256), 256, 0, st>>>(rows, T, t0, H, Hkv, hd, (const float*)qkv, ld, (float*)kc,
                                                     (float*)vc, max_len);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status launch_decode_attn(int dtype, int B, int H, int Hkv, int hd, int len, const void* qkv, int64_t ld,
                             const void* kc, const void* vc, int max_len, float* part, void* o, int64_t ldo,
                             cudaStream_t st) {
  if (B <= 0 || len <= 0 || len > max_len || H % Hkv || (hd != 64 && hd != 128)) return NC_ERR_ARG;
  const int G = H / Hkv;
  if (dtype == NC_BF16)
    return hd == 128 ? decode_attn_g<bf16, 128>(G, B, H, Hkv, len, (const bf16*)qkv, ld, (const bf16*)kc,
                                                (const bf16*)vc, max_len, part, (bf16*)o, ldo, st)
                     : decode_attn_g<bf16, 64>(G, B, H, Hkv, len, (const bf16*)qkv, ld, (const bf16*)kc,
                                               (const bf16*)vc, max_len, part, (bf16*)o, ldo, st);
  return hd == 128 ? decode_attn_g<float, 128>(G, B, H, Hkv, len, (const float*)qkv, ld, (const float*)kc,
                                               (const float*)vc, max_len, part, (float*)o, ldo, st)
                   : decode_attn_g<float, 64>(G, B, H, Hkv, len, (const float*)qkv, ld, (const float*)kc,
                                              (const float*)vc, max_len, part, (float*)o, ldo, st);
}
