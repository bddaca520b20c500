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
// (b, g, s) takes the CK keys [CK s, CK s + CK) of kv head g for every query
// head of its group.  It stages their K and V rows in shared memory with
// 16-byte asynchronous copies (rows padded by 16 bytes, so that lanes reading
// different rows hit different banks), computes every (head, key) score at
// once, one per thread, then the chunk's softmax statistics per head, then the
// unnormalised output with one output column per thread, and leaves a partial
// (max, sum, output) per head; a second kernel merges the partials of a row.
// Scores are q.k / sqrt(hd) in fp32 (exp2 form), as in the training attention.
// With a RoPE table the kernel also does the decode step's RoPE + QK norm: each
// CTA rotates and normalises the G query heads of its group from the raw
// projection, and the CTA whose chunk holds the new position does the same for
// its key head and appends key and value to the cache (and to its staged rows)
// - with the RoPE/QK-norm kernel's arithmetic, so the values are the same.
#include "nc_kernels.cuh"
#include "nc_ptx.cuh"

int g_decode_pdl = 1;   // test hook: 0 launches the decode kernels with plain stream order

namespace {
// The decode kernels (skinny GEMM, attention, combine) are launched with
// programmatic stream serialization: each may start while the previous kernel
// drains, and waits (griddep_wait) before touching that kernel's data.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = g_decode_pdl ? 1 : 0;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
}  // namespace

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

constexpr int DEC_THREADS = 128;
// Keys per CTA: 64 rows of bf16, 32 of fp32, so that K and V stay within the
// static shared-memory limit; the partial buffer is sized for the smaller.
template <typename E>
__host__ __device__ constexpr int dec_chunk() { return sizeof(E) == 2 ? 64 : 32; }
constexpr int DEC_CHUNK_MIN = 32;

__device__ __forceinline__ void ld_unit(const uint8_t* p, const float*, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}
__device__ __forceinline__ void ld_unit(const uint8_t* p, const bf16*, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(h[e]);
}

// Partials: part[((b * H + h) * nsplit + s) * (HD + 2) + {0: max (log2 units), 1: sum, 2..: output}]
// len_dev (device, may be NULL): the key count is *len_dev + 1 (the position of
// the token just appended, plus one); chunks past it leave empty partials.
// tab (may be NULL): RoPE table [T][HD/2] of (cos, sin); then qkv holds the raw
// projection of the new position len - 1 and its k, v are not yet cached.
template <typename E, int HD, int G>
__global__ void __launch_bounds__(DEC_THREADS)
    k_decode_attn(int H, int Hkv, int len, const int32_t* __restrict__ len_dev, int nsplit,
                  const E* __restrict__ qkv, int64_t ld, E* __restrict__ kc, E* __restrict__ vc,
                  int max_len, float scale_log2, float* __restrict__ part, const float2* __restrict__ tab,
                  float eps) {
  constexpr int CK = dec_chunk<E>();
  constexpr int EPU = 16 / (int)sizeof(E);              // elements per 16-byte unit
  constexpr int UPR = HD / EPU;                         // units per row
  constexpr int RB = HD * (int)sizeof(E) + 16;          // padded row bytes in shared memory
  static_assert(HD <= DEC_THREADS && DEC_THREADS % HD == 0, "one output column per thread");
  __shared__ __align__(16) uint8_t ks[CK * RB];
  __shared__ __align__(16) uint8_t vs[CK * RB];
  __shared__ float qs[G][HD];
  __shared__ float ps[G][CK];
  __shared__ float mh[G], sh[G];
  griddep_wait();   // the projection's q/k/v, and `part` the previous combine read
  if (len_dev) len = *len_dev + 1;
  const int bg = blockIdx.x, s = blockIdx.y;
  const int b = bg / Hkv, g = bg % Hkv;
  const int tid = threadIdx.x;
  const int k0 = s * CK;
  const int nk = min(len - k0, CK);
  // head g * G + h of row b: partial at pbase + h * nsplit * (HD + 2)
  float* pbase = part + ((int64_t)(b * H + g * G) * nsplit + s) * (HD + 2);
  if (nk <= 0) {
    if (tid < G) {
      pbase[(int64_t)tid * nsplit * (HD + 2)] = -INFINITY;
      pbase[(int64_t)tid * nsplit * (HD + 2) + 1] = 0.f;
    }
    griddep_launch_dependents();
    return;
  }
  const int pos = len - 1;                             // the position just appended
  const int rp = tab ? pos - k0 : -1;                  // its row in this chunk (fused RoPE), if < nk
  const bool owner = rp >= 0 && rp < nk;
  const int64_t row0 = ((int64_t)(b * Hkv + g) * max_len + k0) * HD;
  const uint8_t* kg = reinterpret_cast<const uint8_t*>(kc + row0);
  const uint8_t* vg = reinterpret_cast<const uint8_t*>(vc + row0);
  for (int i = tid; i < nk * UPR; i += DEC_THREADS) {
    const int r = i / UPR, u = i - r * UPR;
    if (r == rp) continue;                             // computed below
    cp_async16(ks + r * RB + u * 16, kg + (int64_t)i * 16);
    cp_async16(vs + r * RB + u * 16, vg + (int64_t)i * 16);
  }
  cp_async_commit();
  if (tab) {
    // item j < G: query head g*G + j; j == G: key head g; j == G + 1: value head g (the last two in the owner only)
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t crow = ((int64_t)(b * Hkv + g) * max_len + pos) * HD;   // the new position in the cache
    for (int j = warp; j < G + (owner ? 2 : 0); j += DEC_THREADS / 32) {
      if (j == G + 1) {
        const E* src = qkv + (int64_t)b * ld + (int64_t)(H + Hkv + g) * HD;
        E* sv = reinterpret_cast<E*>(vs + rp * RB);
        for (int i = lane; i < HD; i += 32) {
          const E v = src[i];
          vc[crow + i] = v;
          sv[i] = v;
        }
        continue;
      }
      const E* src = qkv + (int64_t)b * ld + (int64_t)(j < G ? g * G + j : H + g) * HD;
      constexpr int D2 = HD / 2;
      const float2* cs = tab + (int64_t)pos * D2;
      float y[2][4];
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = 2 * lane + 64 * k;
        y[k][0] = y[k][1] = y[k][2] = y[k][3] = 0.f;
        if (i < D2) {
          const float ax = ld_f(src + i), ay = ld_f(src + i + 1);
          const float bx = ld_f(src + i + D2), by = ld_f(src + i + D2 + 1);
          const float4 c = *reinterpret_cast<const float4*>(cs + i);   // cos_i, sin_i, cos_i+1, sin_i+1
          y[k][0] = ax * c.x + bx * c.y;
          y[k][2] = -ax * c.y + bx * c.x;
          y[k][1] = ay * c.z + by * c.w;
          y[k][3] = -ay * c.w + by * c.z;
          ss += y[k][0] * y[k][0] + y[k][1] * y[k][1] + y[k][2] * y[k][2] + y[k][3] * y[k][3];
        }
      }
      ss = warp_sum(ss);
      const float r = rsqrtf(ss / (float)HD + eps);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = 2 * lane + 64 * k;
        if (i < D2) {
          const E e[4] = {from_f32<E>(y[k][0] * r), from_f32<E>(y[k][1] * r), from_f32<E>(y[k][2] * r),
                          from_f32<E>(y[k][3] * r)};
          const int at[4] = {i, i + 1, i + D2, i + D2 + 1};
          if (j < G) {
#pragma unroll
            for (int t = 0; t < 4; ++t) qs[j][at[t]] = to_f32(e[t]) * scale_log2;
          } else {
            E* sk = reinterpret_cast<E*>(ks + rp * RB);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              kc[crow + at[t]] = e[t];
              sk[at[t]] = e[t];
            }
          }
        }
      }
    }
  } else {
    for (int i = tid; i < G * HD; i += DEC_THREADS) {
      const int h = i / HD, d = i - h * HD;
      qs[h][d] = ld_f(qkv + (int64_t)b * ld + (int64_t)(g * G + h) * HD + d) * scale_log2;
    }
  }
  cp_async_wait_all();
  __syncthreads();
  // scores, one (head, key) per thread
  for (int i = tid; i < G * CK; i += DEC_THREADS) {
    const int h = i / CK, key = i - h * CK;
    if (key < nk) {
      const uint8_t* kr = ks + key * RB;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < UPR; ++u) {
        float kf[EPU];
        ld_unit(kr + u * 16, (const E*)nullptr, kf);
#pragma unroll
        for (int e = 0; e < EPU; ++e) acc = fmaf(qs[h][u * EPU + e], kf[e], acc);
      }
      ps[h][key] = acc;
    }
  }
  __syncthreads();
  // per head: the chunk's maximum, p = 2^(s - max) in place, and their sum
  const int warp = tid >> 5, lane = tid & 31;
  for (int h = warp; h < G; h += DEC_THREADS / 32) {
    float m = -INFINITY;
    for (int key = lane; key < nk; key += 32) m = fmaxf(m, ps[h][key]);
    m = warp_max(m);
    float sum = 0.f;
    for (int key = lane; key < nk; key += 32) {
      const float p = exp2f(ps[h][key] - m);
      ps[h][key] = p;
      sum += p;
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      mh[h] = m;
      sh[h] = sum;
    }
  }
  __syncthreads();
  // output column d of heads h0, h0 + STEP, ... (STEP = threads / HD)
  constexpr int STEP = DEC_THREADS / HD;
  constexpr int NJ = (G + STEP - 1) / STEP;
  const int d = tid % HD, h0 = tid / HD;
  float acc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) acc[j] = 0.f;
  for (int key = 0; key < nk; ++key) {
    const float v = ld_f(reinterpret_cast<const E*>(vs + key * RB) + d);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int h = h0 + STEP * j;
      if (h < G) acc[j] = fmaf(ps[h][key], v, acc[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int h = h0 + STEP * j;
    if (h < G) {
      float* pp = pbase + (int64_t)h * nsplit * (HD + 2);
      pp[2 + d] = acc[j];
      if (d == 0) {
        pp[0] = mh[h];
        pp[1] = sh[h];
      }
    }
  }
  griddep_launch_dependents();   // the combine may launch now; it waits for this grid to complete
}

// o[b, h*HD + d] = merged output of row (b, h); one block of HD threads per
// row: the splits' weights 2^(max_s - max) and the total sum in parallel, then
// output column d per thread over all splits (independent loads).  Dynamic
// shared memory: nsplit floats.
template <typename E, int HD>
__global__ void __launch_bounds__(HD) k_decode_combine(int nsplit, const float* __restrict__ part,
                                                       E* __restrict__ out, int64_t ldo, int H) {
  extern __shared__ float fw[];
  __shared__ float red[32];
  griddep_wait();
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const float* pr = part + r * nsplit * (HD + 2);
  float m = -INFINITY;
  for (int s = tid; s < nsplit; s += HD) m = fmaxf(m, pr[(int64_t)s * (HD + 2)]);
  m = block_max(m, red);
  float S = 0.f;
  for (int s = tid; s < nsplit; s += HD) {
    const float ms = pr[(int64_t)s * (HD + 2)];
    const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - m);   // an empty split weighs nothing
    fw[s] = f;
    S = fmaf(pr[(int64_t)s * (HD + 2) + 1], f, S);
  }
  S = block_sum(S, red);
  __syncthreads();
  float acc = 0.f;
#pragma unroll 8
  for (int s = 0; s < nsplit; ++s) acc = fmaf(fw[s], pr[(int64_t)s * (HD + 2) + 2 + tid], acc);
  griddep_launch_dependents();
  const int64_t b = r / H;
  const int h = (int)(r % H);
  st_f(out + b * ldo + (int64_t)h * HD + tid, S > 0.f ? acc / S : 0.f);
}

template <typename E, int HD, int G>
nc_status decode_attn_t(int B, int H, int Hkv, int len, const int32_t* len_dev, const E* qkv, int64_t ld, E* kc,
                        E* vc, int max_len, float* part, E* o, int64_t ldo, const float2* tab, float eps,
                        cudaStream_t st) {
  // with the length on the device the grid covers the whole capacity
  constexpr int CK = dec_chunk<E>();
  const int nsplit = ((len_dev ? max_len : len) + CK - 1) / CK;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  if ((size_t)nsplit * sizeof(float) > 48 * 1024) return NC_ERR_UNSUPPORTED;   // the combine's split weights
  NC_CUDA_TRY(launch_pdl(k_decode_attn<E, HD, G>, dim3((unsigned)(B * Hkv), (unsigned)nsplit), dim3(DEC_THREADS), 0,
                         st, H, Hkv, len, len_dev, nsplit, qkv, ld, kc, vc, max_len, scale_log2, part, tab, eps));
  NC_CUDA_TRY(launch_pdl(k_decode_combine<E, HD>, dim3((unsigned)(B * H)), dim3(HD), nsplit * sizeof(float), st,
                         nsplit, (const float*)part, o, ldo, H));
  return NC_OK;
}

template <typename E, int HD>
nc_status decode_attn_g(int G, int B, int H, int Hkv, int len, const int32_t* len_dev, const E* qkv, int64_t ld,
                        E* kc, E* vc, int max_len, float* part, E* o, int64_t ldo, const float2* tab, float eps,
                        cudaStream_t st) {
#define NC_DEC_ARGS B, H, Hkv, len, len_dev, qkv, ld, kc, vc, max_len, part, o, ldo, tab, eps, st
  switch (G) {
    case 1: return decode_attn_t<E, HD, 1>(NC_DEC_ARGS);
    case 2: return decode_attn_t<E, HD, 2>(NC_DEC_ARGS);
    case 3: return decode_attn_t<E, HD, 3>(NC_DEC_ARGS);
    case 4: return decode_attn_t<E, HD, 4>(NC_DEC_ARGS);
    case 8: return decode_attn_t<E, HD, 8>(NC_DEC_ARGS);
#undef NC_DEC_ARGS
    default: return NC_ERR_UNSUPPORTED;
  }
}

}  // namespace

size_t decode_part_floats(int B, int H, int hd, int max_len) {
  return (size_t)B * H * ((max_len + DEC_CHUNK_MIN - 1) / DEC_CHUNK_MIN) * (hd + 2);
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
                             void* kc, void* vc, int max_len, float* part, void* o, int64_t ldo, cudaStream_t st,
                             const int32_t* len_dev, const float* rope_tab, float eps) {
  if (B <= 0 || (!len_dev && (len <= 0 || len > max_len)) || H % Hkv || (hd != 64 && hd != 128)) return NC_ERR_ARG;
  if (rope_tab && (((uintptr_t)rope_tab) & 15)) return NC_ERR_ARG;
  const int G = H / Hkv;
  const float2* tab = reinterpret_cast<const float2*>(rope_tab);
  if (dtype == NC_BF16)
    return hd == 128 ? decode_attn_g<bf16, 128>(G, B, H, Hkv, len, len_dev, (const bf16*)qkv, ld, (bf16*)kc,
                                                (bf16*)vc, max_len, part, (bf16*)o, ldo, tab, eps, st)
                     : decode_attn_g<bf16, 64>(G, B, H, Hkv, len, len_dev, (const bf16*)qkv, ld, (bf16*)kc,
                                               (bf16*)vc, max_len, part, (bf16*)o, ldo, tab, eps, st);
  return hd == 128 ? decode_attn_g<float, 128>(G, B, H, Hkv, len, len_dev, (const float*)qkv, ld, (float*)kc,
                                               (float*)vc, max_len, part, (float*)o, ldo, tab, eps, st)
                   : decode_attn_g<float, 64>(G, B, H, Hkv, len, len_dev, (const float*)qkv, ld, (float*)kc,
                                              (float*)vc, max_len, part, (float*)o, ldo, tab, eps, st);
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
// pieces, eight in flight per lane.  The grid is persistent (two CTAs per SM):
// a CTA stages A in shared memory once (all of K when it fits in the dynamic
// shared-memory budget, else chunk by chunk for every column group) and walks
// column groups of 8, each warp issuing the next batch of pieces - of this
// column or of its next column - before it uses the current one.
// Accumulation is fp32 in a fixed order.
namespace {

constexpr int SK_WARPS = 8;
constexpr int SK_PIECES = 8;                 // 16-byte pieces of W in flight per lane
constexpr int SK_SMEM_MAX = 100 * 1024;      // dynamic shared memory of a CTA: two CTAs per SM

__device__ __forceinline__ void ld8(const bf16* p, float* f) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(h[e]);
}
__device__ __forceinline__ void unpack(const uint4& u, const float*, float* f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint4& u, const bf16*, float* f) {
  const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(h[e]);
}

// Pieces u < SK_PIECES of the batch at column kb: lane l's piece u covers
// columns kb + (32 u + l) EPU ..+EPU (32 lanes read 512 contiguous bytes);
// pieces at or past kc are not loaded.
template <typename E>
__device__ __forceinline__ void sk_load(const E* wr, int kb, int kc, int lane, uint4* w) {
  constexpr int EPU = 16 / (int)sizeof(E);
#pragma unroll
  for (int u = 0; u < SK_PIECES; ++u) {
    const int k = kb + (32 * u + lane) * EPU;
    if (k < kc) w[u] = __ldg(reinterpret_cast<const uint4*>(wr + k));
  }
}

// acc[m] += the batch at column kb (pieces below kc) times rows m of xs (row pitch ldx)
template <typename E, int MB>
__device__ __forceinline__ void sk_fma(const E* xs, int ldx, int M, int kb, int kc, int lane, const uint4* w,
                                       float* acc) {
  constexpr int EPU = 16 / (int)sizeof(E);
#pragma unroll
  for (int u = 0; u < SK_PIECES; ++u) {
    const int k = kb + (32 * u + lane) * EPU;
    if (k < kc) {
      float wf[EPU];
      unpack(w[u], (const E*)nullptr, wf);
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (m < M) {
          float x[EPU];
          if constexpr (EPU == 8) {
            ld8(xs + (int64_t)m * ldx + k, x);
          } else {
            const float4 a = *reinterpret_cast<const float4*>(xs + (int64_t)m * ldx + k);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
          }
#pragma unroll
          for (int e = 0; e < EPU; ++e) acc[m] = fmaf(x[e], wf[e], acc[m]);
        }
      }
    }
  }
}

// Warp-wide sums of acc[m] and the epilogue of column n.
template <typename E, int MB>
__device__ __forceinline__ void sk_store(const float* acc, int M, int n, int lane, int ep, void* D, int64_t ldd) {
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

// NORM: the rows come from the fp32 residual stream and are normalised on the
// way in, A = act(x * rstd(x)), rstd = 1/sqrt(mean(x^2) + eps) in fp32 (the
// RMSNorm kernel's formula; the sum of squares is taken in another order, so
// rstd may differ from that kernel's in the last bit); M <= SK_WARPS then.
// Dynamic shared memory: xs [MB][KC] then rs [MB] and red [SK_WARPS][MB].
template <typename E, int MB, bool NORM>
__global__ void __launch_bounds__(SK_WARPS * 32)
    k_gemm_skinny(int M, int N, int K, int KC, const void* __restrict__ Ain, int64_t lda, const E* __restrict__ W,
                  int64_t ldw, int ep, void* __restrict__ D, int64_t ldd, float eps) {
  constexpr int EPU = 16 / (int)sizeof(E);
  constexpr int BATCH = 32 * SK_PIECES * EPU;          // K columns per batch of pieces
  extern __shared__ __align__(16) uint8_t sk_smem[];
  E* xs = reinterpret_cast<E*>(sk_smem);
  float* rs = reinterpret_cast<float*>(sk_smem + (size_t)MB * KC * sizeof(E));
  float* red = rs + MB;
  const E* A = reinterpret_cast<const E*>(Ain);
  const float* X = reinterpret_cast<const float*>(Ain);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = (N + SK_WARPS - 1) / SK_WARPS;
  const int nchunks = (K + KC - 1) / KC;

  // columns [k0, k0 + kc) of the M rows of A into xs
  auto stage = [&](int k0, int kc) {
    for (int i = threadIdx.x * 8; i < MB * KC; i += SK_WARPS * 32 * 8) {
      const int m = i / KC, k = i - m * KC;
      if (m < M && k < kc) {
        if (NORM) {
          const float r = rs[m];
          const float4 a = *reinterpret_cast<const float4*>(X + (int64_t)m * lda + k0 + k);
          const float4 b = *reinterpret_cast<const float4*>(X + (int64_t)m * lda + k0 + k + 4);
          const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) st_f(&xs[m * KC + k + e], v[e] * r);
        } else {
          *reinterpret_cast<uint4*>(&xs[m * KC + k]) = *reinterpret_cast<const uint4*>(A + (int64_t)m * lda + k0 + k);
          if (sizeof(E) == 4) *reinterpret_cast<uint4*>(&xs[m * KC + k + 4]) =
              *reinterpret_cast<const uint4*>(A + (int64_t)m * lda + k0 + k + 4);
        }
      }
    }
  };

  uint4 w[SK_PIECES], wn[SK_PIECES];
  int g = blockIdx.x;
  // the first pieces of W are in flight while the previous kernel finishes and A is prepared
  if (g * SK_WARPS + warp < N) sk_load(W + (int64_t)(g * SK_WARPS + warp) * ldw, 0, min(KC, K), lane, w);
  griddep_wait();   // A (or X) and D are the previous kernels' data
  if (NORM) {
    // sum of squares of each row: every thread a strided share, then the warps' partials in order
    float ss[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) ss[m] = 0.f;
    for (int c = threadIdx.x; c < K / 4; c += SK_WARPS * 32) {
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (m < M) {
          const float4 v = *reinterpret_cast<const float4*>(X + (int64_t)m * lda + 4 * c);
          ss[m] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      float v = ss[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp * MB + m] = v;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      float t = 0.f;
      for (int q = 0; q < SK_WARPS; ++q) t += red[q * MB + threadIdx.x];
      rs[threadIdx.x] = rsqrtf(t / (float)K + eps);
    }
  }
  float acc[MB];
#pragma unroll
  for (int m = 0; m < MB; ++m) acc[m] = 0.f;
  if (nchunks == 1) {
    __syncthreads();
    stage(0, K);
    __syncthreads();
    // this warp's sequence of (column group, batch), the next one's pieces always in flight
    const int nb = (K + BATCH - 1) / BATCH;
    int b = 0;
    while (g < ngroups) {
      const int n = g * SK_WARPS + warp;
      int g2 = g, b2 = b + 1;
      if (b2 == nb) {
        b2 = 0;
        g2 = g + gridDim.x;
      }
      const int n2 = g2 * SK_WARPS + warp;
      if (g2 < ngroups && n2 < N) sk_load(W + (int64_t)n2 * ldw, b2 * BATCH, K, lane, wn);
      if (n < N) sk_fma<E, MB>(xs, KC, M, b * BATCH, K, lane, w, acc);
      if (b == nb - 1) {
        if (n < N) sk_store<E, MB>(acc, M, n, lane, ep, D, ldd);
#pragma unroll
        for (int m = 0; m < MB; ++m) acc[m] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < SK_PIECES; ++u) w[u] = wn[u];
      g = g2;
      b = b2;
      if (g >= ngroups) griddep_launch_dependents();   // this warp's last store is issued
    }
    return;
  }
  // A larger than the budget: every column group walks the K chunks, restaging A
  for (; g < ngroups; g += gridDim.x) {
    const int n = g * SK_WARPS + warp;
    const bool has_n = n < N;
    const E* wrow = W + (int64_t)(has_n ? n : 0) * ldw;
    for (int k0 = 0; k0 < K; k0 += KC) {
      const int kc = min(KC, K - k0);
      if ((k0 > 0 || g != (int)blockIdx.x) && has_n) sk_load(wrow + k0, 0, kc, lane, w);
      __syncthreads();
      stage(k0, kc);
      __syncthreads();
      if (has_n) {
        for (int kb = 0; kb < kc; kb += BATCH) {
          const bool more = kb + BATCH < kc;
          if (more) sk_load(wrow + k0, kb + BATCH, kc, lane, wn);
          sk_fma<E, MB>(xs, KC, M, kb, kc, lane, w, acc);
          if (more) {
#pragma unroll
            for (int u = 0; u < SK_PIECES; ++u) w[u] = wn[u];
          }
        }
      }
    }
    if (has_n) sk_store<E, MB>(acc, M, n, lane, ep, D, ldd);
#pragma unroll
    for (int m = 0; m < MB; ++m) acc[m] = 0.f;
  }
  griddep_launch_dependents();
}

// The bf16 skinny GEMM for 2 <= M <= 8 rows: each warp streams NCOL = 4
// weight columns at once over a slice of K, so that every shared-memory load
// and conversion of the A rows serves four columns, and the products run two
// lanes per instruction (fma.rn.f32x2).  A CTA's 8 warps are 8 / ks column
// groups times ks K slices; slice partials are summed through shared memory in
// slice order (deterministic).  All of A is staged once (it must fit); with
// NORM, A = act(x * rstd(x)) as in k_gemm_skinny.  W loads before griddep_wait.
constexpr int SC_NCOL = 4;
constexpr int SC_P = 2;   // 16-byte pieces per column and lane in one batch
template <int MB, bool NORM>
__global__ void __launch_bounds__(SK_WARPS * 32)
    k_gemm_skinny_cols(int M, int N, int K, int ks, const void* __restrict__ Ain, int64_t lda,
                       const bf16* __restrict__ W, int64_t ldw, int ep, void* __restrict__ D, int64_t ldd, float eps) {
  constexpr int EPU = 8;
  constexpr int BATCH = 32 * SC_P * EPU;                // K columns of one batch of a slice
  extern __shared__ __align__(16) uint8_t sk_smem[];
  bf16* xs = reinterpret_cast<bf16*>(sk_smem);          // [MB][K]
  float* rs = reinterpret_cast<float*>(sk_smem + (size_t)MB * K * sizeof(bf16));
  float* red = rs + MB;                                 // [SK_WARPS][MB] (NORM) then [SK_WARPS][NCOL][MB]
  const bf16* A = reinterpret_cast<const bf16*>(Ain);
  const float* X = reinterpret_cast<const float*>(Ain);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = warp / ks, sl = warp - cg * ks;        // column group and K slice of this warp
  const int cpc = SC_NCOL * (SK_WARPS / ks);            // columns per CTA group
  const int ngroups = (N + cpc - 1) / cpc;
  const int ksl = ((K + ks - 1) / ks + EPU - 1) / EPU * EPU;
  const int k_lo = min(K, sl * ksl), k_hi = min(K, k_lo + ksl);
  const int nb = (ksl + BATCH - 1) / BATCH;   // the same for every warp: the group's end is a CTA barrier
  auto load = [&](int g, int b, uint4 (*w)[SC_P]) {
#pragma unroll
    for (int c = 0; c < SC_NCOL; ++c) {
      const int n = g * cpc + cg * SC_NCOL + c;
#pragma unroll
      for (int u = 0; u < SC_P; ++u) {
        const int k = k_lo + b * BATCH + (32 * u + lane) * EPU;
        if (n < N && k < k_hi) w[c][u] = __ldg(reinterpret_cast<const uint4*>(W + (int64_t)n * ldw + k));
      }
    }
  };
  uint4 w[SC_NCOL][SC_P], wn[SC_NCOL][SC_P];
  int g = blockIdx.x;
  if (g < ngroups) load(g, 0, w);   // in flight while the previous kernel finishes and A is prepared
  griddep_wait();
  if (NORM) {
    float ss[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) ss[m] = 0.f;
    for (int c = threadIdx.x; c < K / 4; c += SK_WARPS * 32) {
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        if (m < M) {
          const float4 v = *reinterpret_cast<const float4*>(X + (int64_t)m * lda + 4 * c);
          ss[m] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      float v = ss[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp * MB + m] = v;
    }
    __syncthreads();
    if (threadIdx.x < M) {
      float t = 0.f;
      for (int q = 0; q < SK_WARPS; ++q) t += red[q * MB + threadIdx.x];
      rs[threadIdx.x] = rsqrtf(t / (float)K + eps);
    }
    __syncthreads();
  }
  for (int i = threadIdx.x * 8; i < MB * K; i += SK_WARPS * 32 * 8) {   // all of A into xs
    const int m = i / K, k = i - m * K;
    if (m < M) {
      if (NORM) {
        const float r = rs[m];
        const float4 a = *reinterpret_cast<const float4*>(X + (int64_t)m * lda + k);
        const float4 b = *reinterpret_cast<const float4*>(X + (int64_t)m * lda + k + 4);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) st_f(&xs[m * K + k + e], v[e] * r);
      } else {
        *reinterpret_cast<uint4*>(&xs[m * K + k]) = *reinterpret_cast<const uint4*>(A + (int64_t)m * lda + k);
      }
    }
  }
  __syncthreads();
  float* part = red + SK_WARPS * MB;   // [SK_WARPS][NCOL][MB]
  int b = 0;
  float2 acc[SC_NCOL][MB];
#pragma unroll
  for (int c = 0; c < SC_NCOL; ++c)
#pragma unroll
    for (int m = 0; m < MB; ++m) acc[c][m] = make_float2(0.f, 0.f);
  while (g < ngroups) {
    int g2 = g, b2 = b + 1;
    if (b2 == nb) {
      b2 = 0;
      g2 = g + gridDim.x;
    }
    if (g2 < ngroups) load(g2, b2, wn);
#pragma unroll
    for (int u = 0; u < SC_P; ++u) {
      const int k = k_lo + b * BATCH + (32 * u + lane) * EPU;
      if (k < k_hi) {
        float2 wf[SC_NCOL][4];
#pragma unroll
        for (int c = 0; c < SC_NCOL; ++c) {
          const uint32_t* q = reinterpret_cast<const uint32_t*>(&w[c][u]);
#pragma unroll
          for (int e = 0; e < 4; ++e) wf[c][e] = make_float2(__uint_as_float(q[e] << 16), __uint_as_float(q[e] & 0xffff0000u));
        }
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          if (m < M) {
            const uint4 xa = *reinterpret_cast<const uint4*>(xs + (int64_t)m * K + k);
            const uint32_t* q = reinterpret_cast<const uint32_t*>(&xa);
            float2 x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = make_float2(__uint_as_float(q[e] << 16), __uint_as_float(q[e] & 0xffff0000u));
#pragma unroll
            for (int c = 0; c < SC_NCOL; ++c)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[c][m] = fma2(x[e], wf[c][e], acc[c][m]);
          }
        }
      }
    }
    if (b == nb - 1) {
      // lane sums, then the slices' partials in slice order
#pragma unroll
      for (int c = 0; c < SC_NCOL; ++c) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          float v = acc[c][m].x + acc[c][m].y;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) part[(warp * SC_NCOL + c) * MB + m] = v;
          acc[c][m] = make_float2(0.f, 0.f);
        }
      }
      __syncthreads();
      if (sl == 0 && lane < SC_NCOL * MB) {
        const int c = lane / MB, m = lane - c * MB;
        const int n = g * cpc + cg * SC_NCOL + c;
        if (m < M && n < N) {
          float v = 0.f;
          for (int q = 0; q < ks; ++q) v += part[((cg * ks + q) * SC_NCOL + c) * MB + m];
          if (ep == NC_EP_STORE_F32) reinterpret_cast<float*>(D)[(int64_t)m * ldd + n] = v;
          else if (ep == NC_EP_ACCUM_F32) reinterpret_cast<float*>(D)[(int64_t)m * ldd + n] += v;
          else {
            if (ep == NC_EP_RELU2_SQ) { v = fmaxf(v, 0.f); v *= v; }
            st_f(reinterpret_cast<bf16*>(D) + (int64_t)m * ldd + n, v);
          }
        }
      }
      __syncthreads();   // part is rewritten by the next group
      if (g2 >= ngroups) griddep_launch_dependents();
    }
#pragma unroll
    for (int c = 0; c < SC_NCOL; ++c)
#pragma unroll
      for (int u = 0; u < SC_P; ++u) w[c][u] = wn[c][u];
    g = g2;
    b = b2;
  }
  griddep_launch_dependents();
}

template <int MB>
size_t sc_smem_bytes(int K) {
  return (size_t)MB * K * sizeof(bf16) + (size_t)(MB + SK_WARPS * MB + SK_WARPS * SC_NCOL * MB) * sizeof(float);
}
constexpr int SC_SMEM_MAX = 110 * 1024;   // two CTAs per SM

template <int MB, bool NORM>
nc_status skinny_cols_t(int M, int N, int K, const void* A, int64_t lda, const bf16* W, int64_t ldw, int ep, void* D,
                        int64_t ldd, float eps, cudaStream_t st) {
  // K slices per column group: doubled while the CTAs do not cover the SMs and
  // a slice keeps at least one 16-byte piece per lane
  int ks = 1;
  while (ks < SK_WARPS && (int64_t)((N + SC_NCOL * (SK_WARPS / ks) - 1) / (SC_NCOL * (SK_WARPS / ks))) < g_num_sms &&
         K / (2 * ks) >= 32 * 8)
    ks *= 2;
  const int cpc = SC_NCOL * (SK_WARPS / ks);
  const int ngroups = (N + cpc - 1) / cpc;
  const int grid = std::min(ngroups, 2 * g_num_sms);
  NC_CUDA_TRY(launch_pdl(k_gemm_skinny_cols<MB, NORM>, dim3(grid), dim3(SK_WARPS * 32), sc_smem_bytes<MB>(K), st,
                         M, N, K, ks, A, lda, W, ldw, ep, D, ldd, eps));
  return NC_OK;
}

template <int MB, bool NORM>
cudaError_t sc_attr() {
  return cudaFuncSetAttribute(k_gemm_skinny_cols<MB, NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, SC_SMEM_MAX);
}

template <typename E, int MB>
size_t sk_smem_bytes(int KC) {
  return (size_t)MB * KC * sizeof(E) + (size_t)(MB + SK_WARPS * MB) * sizeof(float);
}

template <typename E, int MB, bool NORM>
nc_status skinny_t(int M, int N, int K, const void* A, int64_t lda, const E* W, int64_t ldw, int ep, void* D,
                   int64_t ldd, float eps, cudaStream_t st) {
  // K chunk: all of K (rounded up to 8) if it fits the budget, else the largest multiple of 8 that does
  const int64_t fit = (int64_t)((SK_SMEM_MAX - sk_smem_bytes<E, MB>(0)) / (MB * sizeof(E))) / 8 * 8;
  const int KC = (int)std::min<int64_t>((K + 7) / 8 * 8, fit);
  const int ngroups = (N + SK_WARPS - 1) / SK_WARPS;
  const int grid = std::min(ngroups, 2 * g_num_sms);
  NC_CUDA_TRY(launch_pdl(k_gemm_skinny<E, MB, NORM>, dim3(grid), dim3(SK_WARPS * 32), sk_smem_bytes<E, MB>(KC), st,
                         M, N, K, KC, A, lda, W, ldw, ep, D, ldd, eps));
  return NC_OK;
}

template <typename E, int MB, bool NORM>
cudaError_t sk_attr() {
  return cudaFuncSetAttribute(k_gemm_skinny<E, MB, NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM_MAX);
}

template <typename E, bool NORM>
nc_status skinny_e(int M, int N, int K, const void* A, int64_t lda, const E* W, int64_t ldw, int ep, void* D,
                   int64_t ldd, float eps, cudaStream_t st) {
  if (M <= 1) return skinny_t<E, 1, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if constexpr (sizeof(E) == 2) {
    if (M <= 8 && sc_smem_bytes<8>(K) <= (size_t)SC_SMEM_MAX) {
      if (M <= 2) return skinny_cols_t<2, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
      if (M <= 4) return skinny_cols_t<4, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
      return skinny_cols_t<8, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
    }
  }
  if (M <= 2) return skinny_t<E, 2, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if (M <= 4) return skinny_t<E, 4, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if (M <= 8 || NORM) return skinny_t<E, 8, NORM>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  if (M <= 16) return skinny_t<E, 16, false>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
  return skinny_t<E, 32, false>(M, N, K, A, lda, W, ldw, ep, D, ldd, eps, st);
}

// Raise the dynamic shared-memory limit of every skinny instantiation once
// (outside any stream capture: the decode graph is captured later).
nc_status skinny_prepare() {
  static bool done = false;
  if (done) return NC_OK;
  if (!g_num_sms) {
    int dev = 0;
    NC_CUDA_TRY(cudaGetDevice(&dev));
    NC_CUDA_TRY(cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev));
  }
  const cudaError_t e[] = {
      sk_attr<bf16, 1, false>(), sk_attr<bf16, 2, false>(), sk_attr<bf16, 4, false>(), sk_attr<bf16, 8, false>(),
      sk_attr<bf16, 16, false>(), sk_attr<bf16, 32, false>(), sk_attr<bf16, 1, true>(), sk_attr<bf16, 2, true>(),
      sk_attr<bf16, 4, true>(), sk_attr<bf16, 8, true>(), sk_attr<float, 1, false>(), sk_attr<float, 2, false>(),
      sk_attr<float, 4, false>(), sk_attr<float, 8, false>(), sk_attr<float, 16, false>(),
      sk_attr<float, 32, false>(), sk_attr<float, 1, true>(), sk_attr<float, 2, true>(), sk_attr<float, 4, true>(),
      sk_attr<float, 8, true>(), sc_attr<2, false>(), sc_attr<4, false>(), sc_attr<8, false>(),
      sc_attr<2, true>(), sc_attr<4, true>(), sc_attr<8, true>()};
  for (cudaError_t x : e)
    if (x != cudaSuccess) return NC_ERR_CUDA;
  done = true;
  return NC_OK;
}

}  // namespace

nc_status decode_kernels_prepare() { return skinny_prepare(); }

nc_status launch_gemm_skinny(int dtype, int M, int N, int K, const void* A, int64_t lda, const void* W, int64_t ldw,
                             int ep, void* D, int64_t ldd, cudaStream_t st) {
  if (M < 1 || M > SKINNY_MAX_M || N < 1 || K < 8 || K % 8 || lda % 8 || ldw % 8 ||
      (ep != NC_EP_STORE && ep != NC_EP_STORE_F32 && ep != NC_EP_ACCUM_F32 && ep != NC_EP_RELU2_SQ))
    return NC_ERR_ARG;
  if ((((uintptr_t)A) & 15) || (((uintptr_t)W) & 15)) return NC_ERR_ARG;
  NC_TRY(skinny_prepare());
  if (dtype == NC_BF16) return skinny_e<bf16, false>(M, N, K, A, lda, (const bf16*)W, ldw, ep, D, ldd, 0.f, st);
  return skinny_e<float, false>(M, N, K, A, lda, (const float*)W, ldw, ep, D, ldd, 0.f, st);
}

nc_status launch_gemm_skinny_norm(int dtype, int M, int N, int K, const float* x, int64_t ldx, const void* W,
                                  int64_t ldw, int ep, void* D, int64_t ldd, float eps, cudaStream_t st) {
  if (M < 1 || M > SK_WARPS || N < 1 || K < 8 || K % 8 || ldx % 4 || ldw % 8 ||
      (ep != NC_EP_STORE && ep != NC_EP_STORE_F32 && ep != NC_EP_ACCUM_F32 && ep != NC_EP_RELU2_SQ))
    return NC_ERR_ARG;
  if ((((uintptr_t)x) & 15) || (((uintptr_t)W) & 15)) return NC_ERR_ARG;
  NC_TRY(skinny_prepare());
  if (dtype == NC_BF16) return skinny_e<bf16, true>(M, N, K, x, ldx, (const bf16*)W, ldw, ep, D, ldd, eps, st);
  return skinny_e<float, true>(M, N, K, x, ldx, (const float*)W, ldw, ep, D, ldd, eps, st);
}
