// bf16 GEMM on the 5th-generation tensor cores: D[M,N] (op)= sum_k A(m,k) B(n,k)
// with fp32 accumulation in tensor memory, and the training step's epilogues
// fused (bf16 store, fp32 store / accumulate for residual adds and weight
// gradients, relu^2 with its saved input, relu^2 backward).
//
// Structure (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: loads 128 x 64 A and BN x 64 B tiles (128-byte
//               swizzle) into a STAGES-deep shared-memory ring;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16)
//               and tcgen05.commit to free ring slots / publish accumulators;
//   warp 2      allocates / frees 2*BN TMEM columns (two accumulators, so the
//               epilogue of tile i overlaps the main loop of tile i+1);
//   warps 4..11 epilogue: tcgen05.ld of their 32-lane quarter (warps w and
//               w+4 share a quarter and split the tile's columns), fused op,
//               vector stores to global memory.
// Operands may be K-major ([rows][K]) or MN-major ([K][rows]); the forward
// uses K-major A and B, dX = dY W uses an MN-major B, and dW = dY^T X uses
// MN-major A and B.  The F8 instantiations take E4M3 operands (K-major only)
// through tcgen05.mma kind::f8f6f4: a 128-byte swizzled row then holds 128
// elements instead of 64, so every shared-memory offset and descriptor is the
// same as for bf16 and only the K coordinates double; the epilogue multiplies
// the fp32 accumulator by the two operands' dequantisation factors.  Every mbarrier wait is bounded in time: on expiry the
// kernel raises the timeout bit of the error flag, drains its own TMA loads
// and MMAs (again bounded) and frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "nc_kernels.cuh"
#include "nc_ptx.cuh"

#define TC_BM 128
#define TC_BK 64
#define TC_EPI_WARPS 8                          // two per TMEM lane quarter
#define TC_THREADS (128 + 32 * TC_EPI_WARPS)

#ifndef NC_MN_SWAP_LBO_SBO
#define NC_MN_SWAP_LBO_SBO 0
#endif

struct TcParams {
  int M, N, K;
  int a_mn, b_mn;          // 1 = operand stored MN-major
  int ep;
  void* D;
  int64_t ldd;
  void* aux;
  int64_t ldaux;
  int tiles_m, tiles_n, num_kb;
  // Batched products (the NC_EP_STORE epilogue only): `batch` independent
  // problems of the same shape stacked along the outer (row) dimension of each
  // tensor map, problem b's rows starting b * {a,b,d}_bro rows further.  0 or 1:
  // a single problem.
  int batch, a_bro, b_bro, d_bro;
  int32_t* err;
  uint64_t wait_ns;
  int stall;               // test hook: the MMA issuer waits on a barrier nothing completes (single-CTA kernel)
  // split-K: work unit u covers k-blocks [s*kps, (s+1)*kps) of tile t, with
  // s = u / tiles and t = u % tiles, so CTAs running together stream the same
  // K slice (L2 reuse).  With splits > 1 every unit writes its fp32 partial
  // to ws[s][t][128][BN] and a fix-up kernel sums the slices in order.
  int splits, kps;
  float* ws;
  // NC_EP_QKV_ROPE (the fused q/k/v projection): heads < rope_nh are rotated
  // (RoPE, cos/sin table [T][hd/2][2]) and RMS-normalised per head, their
  // rstd stored to rstd_qk[row * rope_nh + head]; the other heads are stored as is.
  int tma_epi;             // 1: epilogue staged in smem and written by TMA (tmD / tmAux valid)
  const float* rope_tab;
  float* rstd_qk;
  int rope_T, rope_nh, rope_hd;
  int rope_pair_rows;      // 0: table [T][hd/2][2]; > 0: pair-major [hd/4][rope_pair_rows][4]
  float rope_eps;
  // F8 kernels: D = (*scale_a) (*scale_b) sum_k A8(m,k) B8(n,k)
  const float* scale_a;
  const float* scale_b;
  // optional (bf16 outputs of the staged epilogue): atomic maximum of |D| as
  // stored, as float bits, for a per-tensor quantiser of D
  unsigned* amax;
};

// One unit of work of a CTA: k-blocks [k0, k1) of output tile t (slice s).
struct TcSeg {
  int t, s, k0, k1;
};

// Iterates the units a CTA owns, identically in every role.
struct TcSegIter {
  int u, stride, units, tiles;
  __device__ TcSegIter(const TcParams& p, int cta, int grid) {
    tiles = p.tiles_m * p.tiles_n * (p.batch > 1 ? p.batch : 1);
    units = tiles * p.splits;
    u = cta - grid;
    stride = grid;
  }
  __device__ bool next(const TcParams& p, TcSeg& g) {
    u += stride;
    if (u >= units) return false;
    g.s = u / tiles;
    g.t = u - g.s * tiles;
    g.k0 = g.s * p.kps;
    g.k1 = min(p.num_kb, g.k0 + p.kps);
    return true;
  }
};

template <int BN>
struct TcCfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;         // 16 KB
  static constexpr int B_BYTES = BN * TC_BK * 2;            // 32 KB or 16 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  // epilogue staging: one [32 rows][128 B] 128B-swizzled box per epilogue warp
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int STG_BYTES = TC_EPI_WARPS * 4096;
  static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
  static constexpr size_t SMEM = 1024 + (size_t)BAR_OFF + 256;
};

// Instruction descriptor of tcgen05.mma: fp32 accumulator (bits 4-5 = 1); A and
// B formats (bits 7-9, 10-12) bf16 = 1 for kind::f16, E4M3 = 0 for
// kind::f8f6f4; operand majorness, N/8 and M/16.
__device__ __forceinline__ uint32_t tc_idesc(int bn, int a_mn, int b_mn, bool f8 = false) {
  return (1u << 4) | (f8 ? 0u : ((1u << 7) | (1u << 10))) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(TC_BM >> 4) << 24);
}

// Descriptor of the k-th 16-deep slice of a staged operand tile.
//  K-major: rows of 64 elements (128 B), 8-row swizzle atoms 1024 B apart;
//           the k-th slice starts 32 bytes further.
//  MN-major: 64-element (128 B) MN chunks, each a [64 k-rows][128 B] block of
//           8 KB; chunks 8 KB apart (leading offset), 8-deep k groups 1 KB
//           apart (stride offset); the k-th slice starts 16 rows = 2 KB further.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn, int k) {
  if (!mn) return smem_desc(base + 32u * k, 16u, 1024u);
#if NC_MN_SWAP_LBO_SBO
  return smem_desc(base + 2048u * k, 1024u, 8192u);
#else
  return smem_desc(base + 2048u * k, 8192u, 1024u);
#endif
}

__device__ __forceinline__ void tile_coords(const TcParams& p, int t, int& tm, int& tn);
// Tile t of a batched launch: problem b, then the problem's own tile order.
__device__ __forceinline__ void tile_coords_b(const TcParams& p, int t, int& b, int& tm, int& tn) {
  const int per = p.tiles_m * p.tiles_n;
  b = t / per;
  tile_coords(p, t - b * per, tm, tn);
}

__device__ __forceinline__ void tile_coords(const TcParams& p, int t, int& tm, int& tn) {
  // Groups of 16 row tiles sweep all column tiles, so concurrently running
  // CTAs share A row blocks and B column blocks through L2.
  const int G = 16;
  const int per_group = G * p.tiles_n;
  const int g = t / per_group;
  const int first_m = g * G;
  const int gm = min(G, p.tiles_m - first_m);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Apply the epilogue to one row segment: 32 fp32 values for columns n0 .. n0+31.
__device__ __forceinline__ void tc_epilogue_row(const TcParams& p, int64_t m, int n0, const uint32_t* r) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  const bool full = (n0 + 32 <= p.N);
  if (p.ep == NC_EP_STORE_F32 || p.ep == NC_EP_ACCUM_F32) {
    float* d = (float*)p.D + m * p.ldd + n0;
    if (full && ((((uintptr_t)d) & 15) == 0)) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 o = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        if (p.ep == NC_EP_ACCUM_F32) {
          float4 c = *reinterpret_cast<float4*>(d + i);
          o.x += c.x; o.y += c.y; o.z += c.z; o.w += c.w;
        }
        *reinterpret_cast<float4*>(d + i) = o;
      }
    } else {
      for (int i = 0; i < 32 && n0 + i < p.N; ++i) d[i] = (p.ep == NC_EP_ACCUM_F32) ? d[i] + v[i] : v[i];
    }
    return;
  }
  if (p.ep == NC_EP_RELU2) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.f);
  } else if (p.ep == NC_EP_RELU2_SQ) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.f) * fmaxf(v[i], 0.f);
  } else if (p.ep == NC_EP_RELU2_BWD || p.ep == NC_EP_RELU2_SQ_BWD) {
    // aux holds relu(u) (RELU2_BWD) or relu(u)^2 (RELU2_SQ_BWD, whose root is relu(u))
    const bool sq = p.ep == NC_EP_RELU2_SQ_BWD;
    const bf16* a = (const bf16*)p.aux + m * p.ldaux + n0;
    if (full && ((((uintptr_t)a) & 15) == 0)) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 u = *reinterpret_cast<const uint4*>(a + i);
        const bf16* h = reinterpret_cast<const bf16*>(&u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float x = __bfloat162float(h[j]);
          v[i + j] *= 2.f * (sq ? sqrt_approx(x) : x);
        }
      }
    } else {
      for (int i = 0; i < 32; ++i) {
        const float x = (n0 + i < p.N) ? __bfloat162float(a[i]) : 0.f;
        v[i] = (n0 + i < p.N) ? v[i] * 2.f * (sq ? sqrt_approx(x) : x) : 0.f;
      }
    }
  }
  bf16* d = (bf16*)p.D + m * p.ldd + n0;
  bf16* h = (p.ep == NC_EP_RELU2) ? (bf16*)p.aux + m * p.ldaux + n0 : nullptr;
  if (full && ((((uintptr_t)d) & 15) == 0) && (!h || ((((uintptr_t)h) & 15) == 0))) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 o;
      o.x = pack_bf16x2(v[i], v[i + 1]);
      o.y = pack_bf16x2(v[i + 2], v[i + 3]);
      o.z = pack_bf16x2(v[i + 4], v[i + 5]);
      o.w = pack_bf16x2(v[i + 6], v[i + 7]);
      *reinterpret_cast<uint4*>(d + i) = o;
      if (h) {
        uint4 q;
        q.x = pack_bf16x2(v[i] * v[i], v[i + 1] * v[i + 1]);
        q.y = pack_bf16x2(v[i + 2] * v[i + 2], v[i + 3] * v[i + 3]);
        q.z = pack_bf16x2(v[i + 4] * v[i + 4], v[i + 5] * v[i + 5]);
        q.w = pack_bf16x2(v[i + 6] * v[i + 6], v[i + 7] * v[i + 7]);
        *reinterpret_cast<uint4*>(h + i) = q;
      }
    }
  } else {
    for (int i = 0; i < 32 && n0 + i < p.N; ++i) {
      d[i] = __float2bfloat16_rn(v[i]);
      if (h) h[i] = __float2bfloat16_rn(v[i] * v[i]);
    }
  }
}

__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
  uint4 o;
  o.x = pack_bf16x2(v[0], v[1]);
  o.y = pack_bf16x2(v[2], v[3]);
  o.z = pack_bf16x2(v[4], v[5]);
  o.w = pack_bf16x2(v[6], v[7]);
  return o;
}

// Byte offset of 16-byte unit u of row r in a [32 rows][128 B] box stored
// with the TMA 128-byte swizzle (unit index XOR row mod 8): the 32 lanes of a
// warp, one row each, write a unit column in 4 conflict-free wavefronts.
__device__ __forceinline__ uint32_t stg_off(int r, int u) {
  return (uint32_t)(r * 128 + ((((u ^ r) & 7)) << 4));
}

// Staged epilogue of one warp: its 32 rows x (BN/2) accumulator columns pass
// through the warp's [32][128 B] shared-memory box, 128 bytes of output per
// row at a time (32 fp32 or 64 bf16 columns), and leave by TMA store - or
// TMA reduce-add for the fp32 accumulate - as whole lines.  The relu^2
// backward's aux input arrives in the same box by TMA load and is replaced in
// place by the result.  Returns false if a bounded wait expired.
// `ep` is the epilogue kind (p.ep, or NC_EP_STORE_F32 for a split-K partial);
// columns n_base.. of the box row m0 in tmD's coordinates, clipped at n_lim.
template <int BN, bool F8 = false>
__device__ __forceinline__ bool tc_epilogue_staged(const TcParams& p, int ep, const CUtensorMap* tmD,
                                                   const CUtensorMap* tmAux, uint8_t* stg, uint64_t* aux_bar,
                                                   uint32_t& aux_phase, uint32_t taddr, int n_base, int n_lim, int m0,
                                                   int lane) {
  const bool f32o = (ep == NC_EP_STORE_F32 || ep == NC_EP_ACCUM_F32);
  const bool aux_in = (ep == NC_EP_RELU2_BWD || ep == NC_EP_RELU2_SQ_BWD);
  const bool sq_bwd = (ep == NC_EP_RELU2_SQ_BWD);
  const int cc = f32o ? 32 : 64;
  const uint32_t sa = smem_u32(stg);
  const int r = lane;
  const float alpha = F8 ? __ldg(p.scale_a) * __ldg(p.scale_b) : 1.f;
  float am = 0.f;   // maximum |value| this warp stores (p.amax)
#pragma unroll 1
  for (int oc = 0; oc < BN / 2; oc += cc) {
    const int n_out = n_base + oc;
    if (n_out >= n_lim) break;
    // first accumulator piece into registers before the wait: the TMEM read
    // overlaps the previous store still reading the box
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + oc, v);
    tmem_ld_wait();
    if (lane == 0) bulk_wait_read();   // the previous store has read the box
    __syncwarp();
    if (aux_in) {
      if (lane == 0) {
        mbar_arrive_expect_tx(aux_bar, 4096);
        tma_load_2d(stg, tmAux, aux_bar, n_out, m0);
      }
      const uint32_t ph = aux_phase;
      const bool ok = mbar_wait_bounded(aux_bar, ph, p.wait_ns);
      aux_phase ^= 1;
      if (!__all_sync(0xffffffffu, ok)) {
        // the load was issued: it lands in the box before this warp gives up
        if (lane == 0) mbar_wait_bounded(aux_bar, ph, NC_DRAIN_NS);
        __syncwarp();
        return false;
      }
    }
#pragma unroll 1
    for (int pc = 0; pc < cc; pc += 32) {
      if (pc > 0) {
        tmem_ld_32x32b_x32(taddr + oc + pc, v);
        tmem_ld_wait();
      }
      if (F8) {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
      }
      if (f32o) {
#pragma unroll
        for (int u = 0; u < 8; ++u) st_shared_v4(sa + stg_off(r, u), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int u = (pc >> 3) + k;
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[8 * k + e]);
          if (ep == NC_EP_RELU2 || ep == NC_EP_RELU2_SQ) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = fmaxf(f[e], 0.f);
            if (ep == NC_EP_RELU2_SQ) {
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] *= f[e];
            }
          } else if (aux_in) {
            const uint4 a = ld_shared_v4(sa + stg_off(r, u));
            const bf16* h = reinterpret_cast<const bf16*>(&a);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float x = __bfloat162float(h[e]);
              f[e] *= 2.f * (sq_bwd ? sqrt_approx(x) : x);
            }
          }
          if (p.amax) {
#pragma unroll
            for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(f[e]));
          }
          const uint4 o = pack8_bf16(f);
          st_shared_v4(sa + stg_off(r, u), o.x, o.y, o.z, o.w);
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (ep == NC_EP_ACCUM_F32) tma_reduce_add_2d(tmD, stg, n_out, m0);
      else tma_store_2d(tmD, stg, n_out, m0);
      bulk_commit();
    }
    if (ep == NC_EP_RELU2) {   // second output: aux = relu(acc)^2
      if (lane == 0) bulk_wait_read();
      __syncwarp();
#pragma unroll 1
      for (int pc = 0; pc < cc; pc += 32) {
        tmem_ld_32x32b_x32(taddr + oc + pc, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = fmaxf(__uint_as_float(v[8 * k + e]), 0.f) * fmaxf(__uint_as_float(v[8 * k + e]), 0.f);
          const uint4 o = pack8_bf16(f);
          st_shared_v4(sa + stg_off(r, (pc >> 3) + k), o.x, o.y, o.z, o.w);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmAux, stg, n_out, m0);
        bulk_commit();
      }
    }
  }
  if (p.amax) {
    // rounding to bf16 is monotonic, so the rounded maximum is the maximum of the stored values
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (lane == 0 && am > 0.f) atomicMax(p.amax, __float_as_uint(__bfloat162float(__float2bfloat16_rn(am))));
  }
  return true;
}

// NC_EP_QKV_ROPE through the staging box: per head of the warp's columns,
// q/k heads get rstd from the fp32 accumulator (the rotation keeps the sum of
// squares) and the rotated, scaled values; v heads are stored as computed.
// The projection output is alpha * accumulator (alpha = 1 for bf16 operands,
// the two dequantisation factors for 8-bit ones; multiplying by 1 is exact).
__device__ __forceinline__ void tc_epilogue_qkv_rope_staged(const TcParams& p, const CUtensorMap* tmD, uint8_t* stg,
                                                            uint32_t tcol0, int n_base, int ncols, int m0,
                                                            int64_t m, int lane, float alpha) {
  const int hd = p.rope_hd, d = hd >> 1;
  const uint32_t sa = smem_u32(stg);
  const int r = lane;
  const bool row_ok = m < p.M;
  // float4 (cos_i, sin_i, cos_i+1, sin_i+1) of pair i (even) at this row's position: element
  // (i / 2) * cs_step of cs (pair-major table: consecutive rows are consecutive in memory)
  const int pos = (int)(m % p.rope_T);
  const float4* cs = reinterpret_cast<const float4*>(p.rope_tab) +
                     (p.rope_pair_rows ? (size_t)pos : (size_t)pos * (hd / 4));
  const size_t cs_step = p.rope_pair_rows ? (size_t)p.rope_pair_rows : 1;
#pragma unroll 1
  for (int hc = 0; hc < ncols; hc += hd) {
    const int n0 = n_base + hc;
    if (n0 >= p.N) break;
    const int head = n0 / hd;
    const uint32_t tc = tcol0 + hc;
    const bool qk = head < p.rope_nh;
    float rs = 1.f;
    if (qk) {
      float ss = 0.f;
#pragma unroll 1
      for (int c = 0; c < hd; c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tc + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float u = __uint_as_float(v[e]) * alpha;
          ss += u * u;
        }
      }
      rs = rsqrtf(ss / (float)hd + p.rope_eps);
    }
#pragma unroll 1
    for (int oc = 0; oc < hd; oc += 64) {
      if (lane == 0) bulk_wait_read();
      __syncwarp();
#pragma unroll 1
      for (int pc = oc; pc < oc + 64; pc += 32) {
        float y[32];
        if (!qk) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tc + pc, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) y[e] = __uint_as_float(v[e]) * alpha;
        } else {
          // first half: y_i = (u_i cos + u_{i+d} sin) rs; second: y_{i+d} = (-u_i sin + u_{i+d} cos) rs
          const bool first = pc < d;
          const int i0 = first ? pc : pc - d;
          uint32_t a[32], b[32];
          tmem_ld_32x32b_x32(tc + i0, a);
          tmem_ld_32x32b_x32(tc + i0 + d, b);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float4 q = __ldg(cs + ((i0 + e) >> 1) * cs_step);   // cos_i, sin_i, cos_i+1, sin_i+1
            const float a0 = __uint_as_float(a[e]) * alpha, a1 = __uint_as_float(a[e + 1]) * alpha;
            const float b0 = __uint_as_float(b[e]) * alpha, b1 = __uint_as_float(b[e + 1]) * alpha;
            y[e] = (first ? (a0 * q.x + b0 * q.y) : (-a0 * q.y + b0 * q.x)) * rs;
            y[e + 1] = (first ? (a1 * q.z + b1 * q.w) : (-a1 * q.w + b1 * q.z)) * rs;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 o = pack8_bf16(y + 8 * k);
          st_shared_v4(sa + stg_off(r, ((pc - oc) >> 3) + k), o.x, o.y, o.z, o.w);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmD, stg, n0 + oc, m0);
        bulk_commit();
      }
    }
    if (qk && row_ok) p.rstd_qk[m * p.rope_nh + head] = rs;
  }
}

template <int BN, bool F8>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmAux, TcParams p) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full_bar = (uint64_t*)(smem + Cfg::BAR_OFF);
  uint64_t* empty_bar = full_bar + S;
  uint64_t* acc_full = empty_bar + S;      // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain_bar = acc_empty + 2;     // [1]
  uint64_t* aux_bar = drain_bar + 1;       // [TC_EPI_WARPS] TMA loads of the epilogue's aux input
  uint32_t* tmem_slot = (uint32_t*)(aux_bar + TC_EPI_WARPS);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], TC_EPI_WARPS); }
    mbar_init(drain_bar, 1);
    for (int w = 0; w < TC_EPI_WARPS; ++w) mbar_init(&aux_bar[w], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (p.tma_epi) prefetch_tmap(&tmD);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    if (p.err) atomicOr(p.err, NC_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    TcSegIter it(p, blockIdx.x, gridDim.x);
    TcSeg sg;
    while (!*abort_flag && it.next(p, sg)) {
      int b, tm, tn;
      tile_coords_b(p, sg.t, b, tm, tn);
      const int ya = b * p.a_bro, yb = b * p.b_bro;   // the problem's first row in each map
      for (int kb = sg.k0; kb < sg.k1; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, p.wait_ns)) { fail(); break; }
        if (*abort_flag) break;
        uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
        uint8_t* sb = sa + Cfg::A_BYTES;
        mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
        const int k0 = kb * (F8 ? 2 * TC_BK : TC_BK);   // elements: 128 bytes of K per slot
        if (!p.a_mn) {
          tma_load_2d(sa, &tmA, &full_bar[stage], k0, tm * TC_BM + ya);
        } else {
          tma_load_2d(sa, &tmA, &full_bar[stage], tm * TC_BM, k0 + ya);
          tma_load_2d(sa + 8192, &tmA, &full_bar[stage], tm * TC_BM + 64, k0 + ya);
        }
        if (!p.b_mn) {
          tma_load_2d(sb, &tmB, &full_bar[stage], k0, tn * BN + yb);
        } else {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(sb + 8192 * j, &tmB, &full_bar[stage], tn * BN + 64 * j, k0 + yb);
        }
        ++issued;
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
    // Drain: every load this thread issued must land before the CTA exits
    // (already true on the normal path, where the MMA issuer consumed them all).
    for (int s = 0; s < S; ++s) {
      long long n_s = issued / S + ((issued % S) > s ? 1 : 0);
      if (n_s > 0) mbar_wait_bounded(&full_bar[s], (uint32_t)((n_s - 1) & 1), NC_DRAIN_NS);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    const uint32_t idesc = tc_idesc(BN, p.a_mn, p.b_mn, F8);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    TcSegIter it(p, blockIdx.x, gridDim.x);
    TcSeg sg;
    // Test hook (p.stall): first wait for drain_bar, which nothing completes
    // before this thread's own drain commit below, so the wait runs out after
    // the wait limit and the kernel takes its timeout path.
    if (p.stall && !mbar_wait_bounded(drain_bar, 0, p.wait_ns)) fail();
    for (; !*abort_flag && it.next(p, sg); ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1, p.wait_ns)) { fail(); break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = sg.k0; kb < sg.k1; ++kb) {
        if (!mbar_wait_bounded(&full_bar[stage], phase, p.wait_ns)) { fail(); break; }
        if (*abort_flag) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
        const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
        for (int k = 0; k < TC_BK / 16; ++k) {
          if constexpr (F8)
            tc_mma_f8(d_tmem, operand_desc(sa, 0, k), operand_desc(sb, 0, k), idesc, (kb > sg.k0 || k > 0) ? 1u : 0u);
          else
            tc_mma_f16(d_tmem, operand_desc(sa, p.a_mn, k), operand_desc(sb, p.b_mn, k), idesc,
                       (kb > sg.k0 || k > 0) ? 1u : 0u);
        }
        tc_commit(&empty_bar[stage]);
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag) break;
      tc_commit(&acc_full[acc]);
    }
    // Drain: all MMAs issued by this thread complete before TMEM is freed.
    tc_commit(drain_bar);
    mbar_wait_bounded(drain_bar, 0, NC_DRAIN_NS);
  } else if (warp >= 4) {
    // ---------------- epilogue
    const int quarter = warp & 3;
    const int c_lo = ((warp - 4) >> 2) * (BN / 2);   // this warp's half of the columns
    uint8_t* stg = smem + Cfg::STG_OFF + (warp - 4) * 4096;
    uint32_t aux_phase = 0;
    int local = 0;
    TcSegIter it(p, blockIdx.x, gridDim.x);
    TcSeg sg;
    for (; !*abort_flag && it.next(p, sg); ++local) {
      int b, tm, tn;
      tile_coords_b(p, sg.t, b, tm, tn);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait_bounded(&acc_full[acc], acc_phase, p.wait_ns)) { fail(); break; }
      tc_fence_after();
      const int64_t m = (int64_t)tm * TC_BM + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      // split-K: this unit's fp32 partial goes to the workspace
      float* part = (p.splits > 1)
                        ? p.ws + ((size_t)sg.s * (p.tiles_m * p.tiles_n) + sg.t) * TC_BM * BN +
                              (size_t)(quarter * 32 + lane) * BN
                        : nullptr;
      const int m0 = tm * TC_BM + quarter * 32;
      if (m0 >= p.M && (p.ep == NC_EP_QKV_ROPE || (p.tma_epi && !part))) {
        // all 32 rows of this warp are past the end: nothing to store
      } else if (p.ep == NC_EP_QKV_ROPE) {
        tc_epilogue_qkv_rope_staged(p, &tmD, stg, taddr + c_lo, tn * BN + c_lo, BN / 2, m0, m, lane,
                                    F8 ? __ldg(p.scale_a) * __ldg(p.scale_b) : 1.f);
      } else if (p.tma_epi && !part) {
        if (!tc_epilogue_staged<BN, F8>(p, p.ep, &tmD, &tmAux, stg, &aux_bar[warp - 4], aux_phase, taddr + c_lo,
                                        tn * BN + c_lo, p.N, m0 + b * p.d_bro, lane)) {
          fail();
          break;
        }
      } else
#pragma unroll 1
      for (int c = c_lo; c < c_lo + BN / 2; c += 32) {
        const int n0 = tn * BN + c;
        const bool row_ok = (m < p.M) && (n0 < p.N);
        // residual / accumulate target loaded before the TMEM read so that
        // the two latencies overlap
        float4 prev[8];
        const bool pre = !part && row_ok && p.ep == NC_EP_ACCUM_F32 && (n0 + 32 <= p.N) &&
                         ((((uintptr_t)((float*)p.D + m * p.ldd + n0)) & 15) == 0);
        if (pre) {
          const float4* src = reinterpret_cast<const float4*>((float*)p.D + m * p.ldd + n0);
#pragma unroll
          for (int i = 0; i < 8; ++i) prev[i] = src[i];
        }
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c, r);
        tmem_ld_wait();
        if (part) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(part + c + i) =
                make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                            __uint_as_float(r[i + 3]));
        } else if (pre) {
          float4* dst = reinterpret_cast<float4*>((float*)p.D + m * p.ldd + n0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(prev[i].x + __uint_as_float(r[4 * i]), prev[i].y + __uint_as_float(r[4 * i + 1]),
                                 prev[i].z + __uint_as_float(r[4 * i + 2]), prev[i].w + __uint_as_float(r[4 * i + 3]));
        } else if (row_ok) {
          tc_epilogue_row(p, m, n0, r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
    if (lane == 0) bulk_wait_all();   // TMA stores of this warp complete before the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------- CTA-pair kernel
// The same GEMM over 256 x 256 output tiles computed by a pair of CTAs (a
// cluster of 2) with tcgen05 cta_group::2: CTA rank r stages rows
// [128 r, 128 r + 128) of the A tile and rows [128 r, 128 r + 128) of the B
// tile; one thread of rank 0 issues M = 256, N = 256 MMAs that read both
// CTAs' shared memory, and each CTA's tensor memory holds its 128 rows of the
// accumulator.  Per SM this stages 32 KB per 64 of depth instead of 48 KB for
// the same multiply-adds as the single-CTA 128 x 256 tile.  A ring slot holds
// two 64-column (128 B) swizzled chunks along K: K-major [2][128 rows][128 B],
// MN-major [2][2 mn-chunks][64 k-rows][128 B].  Ring slots are
// released (and accumulators published) to both CTAs by multicast commits;
// both CTAs' epilogue warps release an accumulator on rank 0's barrier.
struct Tc2Cfg {
  // 128-deep k-blocks: eight MMAs per ring slot, so the issuing thread's per-slot
  // wait / commit / loop overhead is spread over twice the work of a 64-deep slot.
  static constexpr int BK = 128;
  static constexpr int STAGES = 3;
  static constexpr int A_BYTES = TC_BM * BK * 2;            // 32 KB: this CTA's 128 rows of A
  static constexpr int B_BYTES = 128 * BK * 2;              // 32 KB: this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 512;                     // two 256-column accumulators
  static constexpr int STG_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + TC_EPI_WARPS * 4096;
  static constexpr size_t SMEM = 1024 + (size_t)BAR_OFF + 256;
};

template <bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
    k_gemm_tc2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmAux, TcParams p) {
  using Cfg = Tc2Cfg;
  constexpr int S = Cfg::STAGES;
  constexpr int BN = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full_bar = (uint64_t*)(smem + Cfg::BAR_OFF);   // rank 0: both CTAs' loads land here
  uint64_t* empty_bar = full_bar + S;                       // each CTA: its slot is free again
  uint64_t* acc_full = empty_bar + S;                       // [2] each CTA: accumulator ready
  uint64_t* acc_empty = acc_full + 2;                       // [2] rank 0: both epilogues done
  uint64_t* drain_bar = acc_empty + 2;
  uint64_t* aux_bar = drain_bar + 1;                        // [TC_EPI_WARPS]
  uint32_t* tmem_slot = (uint32_t*)(aux_bar + TC_EPI_WARPS);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], 2 * TC_EPI_WARPS); }
    mbar_init(drain_bar, 1);
    for (int w = 0; w < TC_EPI_WARPS; ++w) mbar_init(&aux_bar[w], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (p.tma_epi) prefetch_tmap(&tmD);
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();    // barriers of both CTAs initialised before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t full_rank0 = mapa_shared(smem_u32(full_bar), 0);
  const uint32_t acc_empty_rank0 = mapa_shared(smem_u32(acc_empty), 0);

  auto fail = [&]() {
    if (p.err) atomicOr(p.err, NC_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs): own A rows and own half of B
    int stage = 0;
    uint32_t phase = 0;
    TcSegIter it(p, cluster, nclusters);
    TcSeg sg;
    while (!*abort_flag && it.next(p, sg)) {
      int b, tm, tn;
      tile_coords_b(p, sg.t, b, tm, tn);
      const int arow = tm * 256 + (int)rank * 128, brow = tn * BN + (int)rank * 128;
      const int ya = b * p.a_bro, yb = b * p.b_bro;   // the problem's first row in each map
      for (int kb = sg.k0; kb < sg.k1; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, p.wait_ns)) { fail(); break; }
        if (*abort_flag) break;
        uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
        uint8_t* sb = sa + Cfg::A_BYTES;
        const uint32_t fb = full_rank0 + stage * 8;
        if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * Cfg::STAGE_BYTES);
        constexpr int KE = F8 ? 2 : 1;            // a 128-byte chunk holds 64 bf16 or 128 E4M3 values
        const int k0 = kb * Cfg::BK * KE;
#pragma unroll
        for (int kc = 0; kc < 2; ++kc) {
          if (!p.a_mn) {
            tma_load_2d_pair(sa + kc * 16384, &tmA, fb, k0 + 64 * KE * kc, arow + ya);
          } else {
            tma_load_2d_pair(sa + kc * 16384, &tmA, fb, arow, k0 + 64 * kc + ya);
            tma_load_2d_pair(sa + kc * 16384 + 8192, &tmA, fb, arow + 64, k0 + 64 * kc + ya);
          }
          if (!p.b_mn) {
            tma_load_2d_pair(sb + kc * 16384, &tmB, fb, k0 + 64 * KE * kc, brow + yb);
          } else {
            tma_load_2d_pair(sb + kc * 16384, &tmB, fb, brow, k0 + 64 * kc + yb);
            tma_load_2d_pair(sb + kc * 16384 + 8192, &tmB, fb, brow + 64, k0 + 64 * kc + yb);
          }
        }
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------- MMA issuer (rank 0 only): M = 256, N = 256
    const uint32_t idesc = (1u << 4) | (F8 ? 0u : ((1u << 7) | (1u << 10))) | ((uint32_t)p.a_mn << 15) |
                           ((uint32_t)p.b_mn << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    TcSegIter it(p, cluster, nclusters);
    TcSeg sg;
    for (; !*abort_flag && it.next(p, sg); ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1, p.wait_ns)) { fail(); break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = sg.k0; kb < sg.k1; ++kb) {
        if (!mbar_wait_bounded(&full_bar[stage], phase, p.wait_ns)) { fail(); break; }
        if (*abort_flag) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
        const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
        for (int k = 0; k < Cfg::BK / 16; ++k) {  // k-chunk k/4 sits 16 KB further
          if constexpr (F8)
            tc_mma_f8_pair(d_tmem, operand_desc(sa + (k >> 2) * 16384, 0, k & 3),
                           operand_desc(sb + (k >> 2) * 16384, 0, k & 3), idesc, (kb > sg.k0 || k > 0) ? 1u : 0u);
          else
            tc_mma_f16_pair(d_tmem, operand_desc(sa + (k >> 2) * 16384, p.a_mn, k & 3),
                            operand_desc(sb + (k >> 2) * 16384, p.b_mn, k & 3), idesc,
                            (kb > sg.k0 || k > 0) ? 1u : 0u);
        }
        tc_commit_pair(&empty_bar[stage], 0x3);
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag) break;
      tc_commit_pair(&acc_full[acc], 0x3);
    }
    tc_commit_pair(drain_bar, 0x1);
    mbar_wait_bounded(drain_bar, 0, NC_DRAIN_NS);
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs): this CTA's 128 rows of the tile
    const int quarter = warp & 3;
    const int c_lo = ((warp - 4) >> 2) * (BN / 2);
    uint8_t* stg = smem + Cfg::STG_OFF + (warp - 4) * 4096;
    uint32_t aux_phase = 0;
    int local = 0;
    TcSegIter it(p, cluster, nclusters);
    TcSeg sg;
    for (; !*abort_flag && it.next(p, sg); ++local) {
      int b, tm, tn;
      tile_coords_b(p, sg.t, b, tm, tn);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait_bounded(&acc_full[acc], acc_phase, p.wait_ns)) { fail(); break; }
      tc_fence_after();
      const int m0 = tm * 256 + (int)rank * 128 + quarter * 32;
      const int64_t m = (int64_t)m0 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (m0 >= p.M) {
        // all 32 rows of this warp are past the end: nothing to store
      } else if (p.splits > 1) {
        // split-K slice: this CTA's 128 x 256 fp32 partial into the workspace
        // ws[s][t][256][256] (tensor map tmAux), summed in slice order afterwards
        // (8-bit operands: the partial carries the dequantisation factor)
        const int wrow = (sg.s * (p.tiles_m * p.tiles_n) + sg.t) * 256 + (int)rank * 128 + quarter * 32;
        if (!tc_epilogue_staged<BN, F8>(p, NC_EP_STORE_F32, &tmAux, &tmAux, stg, &aux_bar[warp - 4], aux_phase,
                                        taddr + c_lo, c_lo, BN, wrow, lane)) {
          fail();
          break;
        }
      } else if (p.ep == NC_EP_QKV_ROPE) {
        tc_epilogue_qkv_rope_staged(p, &tmD, stg, taddr + c_lo, tn * BN + c_lo, BN / 2, m0, m, lane,
                                    F8 ? __ldg(p.scale_a) * __ldg(p.scale_b) : 1.f);
      } else if (p.tma_epi) {
        if (!tc_epilogue_staged<BN, F8>(p, p.ep, &tmD, &tmAux, stg, &aux_bar[warp - 4], aux_phase, taddr + c_lo,
                                        tn * BN + c_lo, p.N, m0 + b * p.d_bro, lane)) {
          fail();
          break;
        }
      } else {
#pragma unroll 1
        for (int c = c_lo; c < c_lo + BN / 2; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c, r);
          tmem_ld_wait();
          if (m < p.M && tn * BN + c < p.N) tc_epilogue_row(p, m, tn * BN + c, r);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_rank0 + acc * 8);
    }
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();    // the peer's shared memory and barriers stay alive until both CTAs are done
  tc_fence_after();
  if (warp == 2) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
}

// Split-K fix-up: out (op)= sum over slices s = 0..splits-1, in that order
// (bitwise reproducible), of the fp32 partial tiles.  One block per tile.
// One block per 32-row slab of a tile (BM / 32 blocks per tile), so that
// the few tiles of a weight-gradient GEMM still spread over every SM.
template <int BM, int BN>
__global__ void __launch_bounds__(256) k_gemm_tc_fixup(TcParams p) {
  constexpr int RB = 32;
  const int t = blockIdx.x / (BM / RB), rb = blockIdx.x % (BM / RB);
  const int tiles = p.tiles_m * p.tiles_n;
  int tm, tn;
  tile_coords(p, t, tm, tn);
  for (int i = threadIdx.x; i < RB * BN / 4; i += blockDim.x) {
    const int r = rb * RB + (i * 4) / BN, cc = (i * 4) % BN;
    const int64_t m = (int64_t)tm * BM + r;
    const int n = tn * BN + cc;
    if (m >= p.M || n >= p.N) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sl = 0; sl < p.splits; ++sl) {
      const float4 v = *reinterpret_cast<const float4*>(p.ws + ((size_t)sl * tiles + t) * BM * BN +
                                                        (size_t)r * BN + cc);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    float* d = (float*)p.D + m * p.ldd + n;
    const float a[4] = {acc.x, acc.y, acc.z, acc.w};
    for (int j = 0; j < 4 && n + j < p.N; ++j) d[j] = (p.ep == NC_EP_ACCUM_F32) ? d[j] + a[j] : a[j];
  }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  }
  return fn;
}

// 2D tensor map over a row-major [outer][inner] matrix of 2- or 4-byte
// elements with leading dimension ld (elements), box {box_inner, box_outer},
// 128-byte swizzle.
static bool make_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
                         uint64_t outer, int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  auto enc = get_encode();
  if (!enc) return false;
  if ((((uintptr_t)base) & 15) || ((ld * esize) % 16)) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, int64_t ld,
                       uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, ld, box_inner, box_outer);
}

// 3-D bf16 tensor map over [d2][d1][inner] with row pitch ld elements and
// d1 rows per d2 slice (a [B][T][cols] view of a [B*T, ld] matrix), box
// {box_inner, box_mid, 1}, 128-byte swizzle.  Boxes are clipped at d1, so a
// tile that runs past the end of one sequence never touches the next.
bool make_tmap_bf16_3d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t d1, uint64_t d2, int64_t ld,
                       uint32_t box_inner, uint32_t box_mid) {
  auto enc = get_encode();
  if (!enc) return false;
  if ((((uintptr_t)base) & 15) || ((ld * 2) % 16)) return false;
  cuuint64_t dims[3] = {inner, d1, d2};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * d1};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int g_num_sms = 0;
uint64_t g_tc_wait_ns = 4000000000ull;   // bounded-wait limit of the tensor-core kernels
int g_tc_stall_next = 0;                 // test hook: the next single-CTA GEMM launch times out

template <int BN, bool F8 = false>
static nc_status launch_tc_bn(TcParams p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                              const CUtensorMap& tx, size_t ws_bytes, cudaStream_t st) {
  static bool attr_set = false;
  auto kern = k_gemm_tc<BN, F8>;
  if (!attr_set) {
    NC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<BN>::SMEM));
    attr_set = true;
  }
  const int tiles = p.tiles_m * p.tiles_n * (p.batch > 1 ? p.batch : 1);
  // Split K when whole tiles would leave the last wave badly filled (fp32
  // outputs only: the weight gradients and the lm_head input gradient, whose
  // K is the token count or the vocabulary).  Cost model per split count S:
  // waves(S) * (k-blocks per slice) * t_kb + partial-tile traffic.
  p.splits = 1;
  p.kps = p.num_kb;
  const bool f32_out = (p.ep == NC_EP_STORE_F32 || p.ep == NC_EP_ACCUM_F32);
  if (f32_out && p.ws && tiles < 4 * g_num_sms) {
    const double t_kb = 0.35e-6;                                   // s per 128 x BN x 64 block, one SM
    const double tile_bytes = 2.0 * TC_BM * BN * sizeof(float);    // write + read of one partial
    double best = 1e30;
    for (int S = 1; S <= 16; ++S) {
      const int kps = (p.num_kb + S - 1) / S;
      if (S > 1 && (kps < 16 || (size_t)S * tiles * TC_BM * BN * sizeof(float) > ws_bytes)) break;
      const int waves = (tiles * S + g_num_sms - 1) / g_num_sms;
      const double cost = waves * kps * t_kb + (S > 1 ? S * tiles * tile_bytes / 6.0e12 : 0.0);
      if (cost < best * 0.98) { best = cost; p.splits = S; p.kps = kps; }
    }
    p.splits = (p.num_kb + p.kps - 1) / p.kps;
  }
  const int grid = std::min(tiles * p.splits, g_num_sms);
  p.stall = g_tc_stall_next;
  g_tc_stall_next = 0;
  kern<<<grid, TC_THREADS, TcCfg<BN>::SMEM, st>>>(ta, tb, td, tx, p);
  NC_CUDA_TRY(cudaGetLastError());
  if (p.splits > 1) {
    k_gemm_tc_fixup<TC_BM, BN><<<tiles * (TC_BM / 32), 256, 0, st>>>(p);
    NC_CUDA_TRY(cudaGetLastError());
  }
  return NC_OK;
}

int g_gemm_pair = 1;       // CTA-pair kernel for eligible shapes (test hook can turn it off)

// 256 x 256 tiles on CTA pairs: persistent grid of co-resident clusters.
template <bool F8 = false>
static nc_status launch_tc_pair(TcParams p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                                const CUtensorMap& tx, size_t ws_bytes, cudaStream_t st) {
  static int max_clusters = 0;
  auto kern = k_gemm_tc2<F8>;
  if (!max_clusters) {
    NC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Tc2Cfg::SMEM));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (g_num_sms / 2));
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = Tc2Cfg::SMEM;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = g_num_sms / 2;
    }
    max_clusters = std::min(n, g_num_sms / 2);
  }
  const int bk = Tc2Cfg::BK * (F8 ? 2 : 1);                   // K elements per ring slot
  p.num_kb = (p.K + bk - 1) / bk;
  p.splits = 1;
  p.kps = p.num_kb;
  const int tiles = p.tiles_m * p.tiles_n * (p.batch > 1 ? p.batch : 1);
  // Split K when whole 256 x 256 tiles would leave the last wave of clusters
  // badly filled (fp32 outputs only: the weight gradients, whose K is the token
  // count).  Cost per split count S: waves(S) * (k-blocks per slice) * t_kb plus
  // the partial tiles' write and read.
  const bool f32_out = (p.ep == NC_EP_STORE_F32 || p.ep == NC_EP_ACCUM_F32);
  if (f32_out && p.ws && tiles < 4 * max_clusters) {
    const double t_kb = 0.9e-6;                                 // s per 256 x 256 x 128 block, one pair
    const double tile_bytes = 2.0 * 256 * 256 * sizeof(float);  // write + read of one partial
    double best = 1e30;
    int kps_best = p.num_kb;
    for (int S = 1; S <= 16; ++S) {
      const int kps = (p.num_kb + S - 1) / S;
      if (S > 1 && (kps < 8 || (size_t)S * tiles * 256 * 256 * sizeof(float) > ws_bytes)) break;
      const int waves = (tiles * S + max_clusters - 1) / max_clusters;
      const double cost = waves * kps * t_kb + (S > 1 ? S * tiles * tile_bytes / 6.0e12 : 0.0);
      if (cost < best * 0.98) { best = cost; kps_best = kps; }
    }
    p.kps = kps_best;
    p.splits = (p.num_kb + p.kps - 1) / p.kps;
  }
  CUtensorMap tw = tx;
  if (p.splits > 1) {
    // partial tiles ws[s][t][256][256] as one fp32 matrix of 256 columns
    if (!make_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.ws, 256, (uint64_t)p.splits * tiles * 256, 256, 32,
                      32))
      return NC_ERR_CUDA;
  }
  const int grid = 2 * std::min(tiles * p.splits, max_clusters);
  kern<<<grid, TC_THREADS, Tc2Cfg::SMEM, st>>>(ta, tb, td, tw, p);
  NC_CUDA_TRY(cudaGetLastError());
  if (p.splits > 1) {
    k_gemm_tc_fixup<256, 256><<<tiles * (256 / 32), 256, 0, st>>>(p);
    NC_CUDA_TRY(cudaGetLastError());
  }
  return NC_OK;
}

// Split-K partials: up to 4 waves of 128 x 256 fp32 tiles per slice set.
size_t gemm_tc_workspace_bytes() { return (size_t)256 << 20; }

struct TcRope {
  const float* tab;
  float* rstd;
  int T, nh, hd, pair_rows;
  float eps;
};

static nc_status gemm_tc_impl(int M, int N, int K, const bf16* A, int64_t lda, int a_kmajor, const bf16* B,
                              int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd, void* aux, int64_t ldaux,
                              const TcRope* rope, int32_t* err, void* ws, size_t ws_bytes, cudaStream_t st,
                              int batch = 1, int64_t a_bro = 0, int64_t b_bro = 0, int64_t d_bro = 0) {
  if (M <= 0 || N <= 0 || batch <= 0) return NC_OK;
  if (K <= 0) return NC_ERR_ARG;
  if ((lda % 8) || (ldb % 8) || (((uintptr_t)A) & 15) || (((uintptr_t)B) & 15)) return NC_ERR_ARG;
  if (!D || ((ep == NC_EP_RELU2 || ep == NC_EP_RELU2_BWD || ep == NC_EP_RELU2_SQ_BWD) && !aux))
    return NC_ERR_ARG;
  if (!g_num_sms) {
    int dev = 0;
    NC_CUDA_TRY(cudaGetDevice(&dev));
    NC_CUDA_TRY(cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev));
  }
  const int BN = (N > 128) ? 256 : 128;
  TcParams p;
  p.M = M; p.N = N; p.K = K;
  p.a_mn = a_kmajor ? 0 : 1;
  p.b_mn = b_kmajor ? 0 : 1;
  p.ep = ep; p.D = D; p.ldd = ldd; p.aux = aux; p.ldaux = ldaux;
  p.tiles_m = (M + TC_BM - 1) / TC_BM;
  p.tiles_n = (N + BN - 1) / BN;
  p.num_kb = (K + TC_BK - 1) / TC_BK;
  p.batch = batch;
  p.a_bro = (int)a_bro; p.b_bro = (int)b_bro; p.d_bro = (int)d_bro;
  p.err = err;
  p.wait_ns = g_tc_wait_ns;
  p.stall = 0;
  p.ws = (float*)ws;
  p.splits = 1;
  p.kps = 0;
  p.rope_tab = nullptr; p.rstd_qk = nullptr; p.rope_T = 1; p.rope_nh = 0; p.rope_hd = 0; p.rope_pair_rows = 0;
  p.rope_eps = 0.f;
  p.scale_a = nullptr; p.scale_b = nullptr;
  p.amax = nullptr;
  if (rope) {
    // whole heads in each epilogue warp's 128 columns, 16-byte row segments
    if (ep != NC_EP_QKV_ROPE || BN != 256 || (rope->hd != 64 && rope->hd != 128) || (N % rope->hd) ||
        rope->nh * rope->hd > N || rope->T <= 0 || (ldd % 8) || (((uintptr_t)D) & 15) ||
        (((uintptr_t)rope->tab) & 15) || !rope->rstd)
      return NC_ERR_ARG;
    if (rope->pair_rows < 0 || (rope->pair_rows > 0 && rope->pair_rows < rope->T)) return NC_ERR_ARG;
    p.rope_tab = rope->tab; p.rstd_qk = rope->rstd; p.rope_T = rope->T; p.rope_nh = rope->nh;
    p.rope_hd = rope->hd; p.rope_pair_rows = rope->pair_rows; p.rope_eps = rope->eps;
  } else if (ep == NC_EP_QKV_ROPE) {
    return NC_ERR_ARG;
  }
  if (ws && (((uintptr_t)ws) & 15)) return NC_ERR_ARG;
  // CTA pairs (256 x 256 tiles, split-K for few-tile fp32 outputs) whenever N > 128
  // and M >= 256; the single-CTA kernel otherwise
  const bool f32_out = (ep == NC_EP_STORE_F32 || ep == NC_EP_ACCUM_F32);
  const bool pair = g_gemm_pair && BN == 256 && M >= 256;
  if (pair) p.tiles_m = (M + 255) / 256;
  // outer (row) extents of the maps: the operand itself, or every problem's rows of a batch
  const uint64_t ra = batch > 1 ? (uint64_t)batch * a_bro : (uint64_t)(a_kmajor ? M : K);
  const uint64_t rb = batch > 1 ? (uint64_t)batch * b_bro : (uint64_t)(b_kmajor ? N : K);
  const uint64_t rd = batch > 1 ? (uint64_t)batch * d_bro : (uint64_t)M;
  CUtensorMap ta, tb;
  bool ok;
  if (a_kmajor) ok = make_tmap_bf16_2d(&ta, A, K, ra, lda, TC_BK, TC_BM);
  else ok = make_tmap_bf16_2d(&ta, A, M, ra, lda, 64, TC_BK);
  if (!ok) return NC_ERR_CUDA;
  if (b_kmajor) ok = make_tmap_bf16_2d(&tb, B, K, rb, ldb, TC_BK, pair ? 128 : BN);
  else ok = make_tmap_bf16_2d(&tb, B, N, rb, ldb, 64, TC_BK);
  if (!ok) return NC_ERR_CUDA;
  // Epilogue tensor maps: D (and aux for the relu^2 modes) in boxes of 32 rows
  // x 128 bytes; without them (unaligned D) the epilogue stores per thread.
  CUtensorMap td, tx;
  memset(&td, 0, sizeof(td));
  memset(&tx, 0, sizeof(tx));
  p.tma_epi = f32_out ? make_tmap_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, N, rd, ldd, 32, 32)
                      : make_tmap_bf16_2d(&td, D, N, rd, ldd, 64, 32);
  if (batch > 1 && !p.tma_epi) return NC_ERR_ARG;
  if (p.tma_epi && (ep == NC_EP_RELU2 || ep == NC_EP_RELU2_BWD || ep == NC_EP_RELU2_SQ_BWD))
    p.tma_epi = make_tmap_bf16_2d(&tx, aux, N, M, ldaux, 64, 32);
  if (ep == NC_EP_QKV_ROPE && !p.tma_epi) return NC_ERR_ARG;
  if (pair) return launch_tc_pair(p, ta, tb, td, tx, ws_bytes, st);
  if (BN == 256) return launch_tc_bn<256>(p, ta, tb, td, tx, ws_bytes, st);
  return launch_tc_bn<128>(p, ta, tb, td, tx, ws_bytes, st);
}

nc_status launch_gemm_tc(int M, int N, int K, const bf16* A, int64_t lda, int a_kmajor, const bf16* B,
                         int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd, void* aux, int64_t ldaux,
                         int32_t* err, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (ep == NC_EP_QKV_ROPE) return NC_ERR_ARG;
  return gemm_tc_impl(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, ep, D, ldd, aux, ldaux, nullptr, err, ws,
                      ws_bytes, st);
}

nc_status launch_gemm_tc_batched(int batch, int M, int N, int K, const bf16* A, int64_t lda, int a_kmajor,
                                 int64_t a_bro, const bf16* B, int64_t ldb, int b_kmajor, int64_t b_bro, bf16* D,
                                 int64_t ldd, int64_t d_bro, int32_t* err, cudaStream_t st) {
  if (batch <= 0 || M <= 0 || N <= 0) return NC_OK;
  if (K <= 0 || !A || !B || !D) return NC_ERR_ARG;
  // every problem's own rows inside its stride; output tiles (up to 256 rows)
  // inside the problem's output rows; K-rows of an MN-major operand in whole
  // 128-row k-blocks, so that no load reaches the next problem
  const int64_t ra = a_kmajor ? M : K, rb = b_kmajor ? N : K;
  if (a_bro < ra || b_bro < rb || d_bro < (int64_t)(M + 255) / 256 * 256) return NC_ERR_ARG;
  if ((!a_kmajor || !b_kmajor) && (K % 128)) return NC_ERR_ARG;
  if ((int64_t)batch * std::max(std::max(a_bro, b_bro), d_bro) >= ((int64_t)1 << 31)) return NC_ERR_ARG;
  return gemm_tc_impl(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, NC_EP_STORE, D, ldd, nullptr, 0, nullptr, err,
                      nullptr, 0, st, batch, a_bro, b_bro, d_bro);
}

// E4M3 GEMM: D[M,N] = (*scale_a) (*scale_b) A8 B8^T, both operands K-major
// bytes ([M][lda], [N][ldb]), fp32 accumulation, through the TMA-staged
// epilogue `ep`: NC_EP_STORE (bf16 D), NC_EP_STORE_F32, NC_EP_ACCUM_F32 (fp32
// D += ...), NC_EP_RELU2_SQ (bf16 relu(.)^2) or NC_EP_QKV_ROPE (with `rope`,
// bf16 D).  CTA pairs (256 x 256 tiles) when N > 128 and M >= 256, the
// single-CTA kernel otherwise; no split-K.
static nc_status gemm_fp8_impl(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                               const float* scale_a, const float* scale_b, int ep, void* D, int64_t ldd,
                               const TcRope* rope, int32_t* err, cudaStream_t st, const void* aux = nullptr,
                               int64_t ldaux = 0, unsigned* amax = nullptr, void* ws = nullptr,
                               size_t ws_bytes = 0) {
  if (M <= 0 || N <= 0) return NC_OK;
  if (K <= 0 || !A || !B || !D || !scale_a || !scale_b) return NC_ERR_ARG;
  if ((lda % 16) || (ldb % 16) || lda < K || ldb < K || (((uintptr_t)A) & 15) || (((uintptr_t)B) & 15))
    return NC_ERR_ARG;
  if (ep != NC_EP_STORE && ep != NC_EP_STORE_F32 && ep != NC_EP_ACCUM_F32 && ep != NC_EP_RELU2_SQ &&
      ep != NC_EP_RELU2_SQ_BWD && ep != NC_EP_QKV_ROPE)
    return NC_ERR_ARG;
  if ((ep == NC_EP_RELU2_SQ_BWD) != (aux != nullptr)) return NC_ERR_ARG;
  if ((ep == NC_EP_QKV_ROPE) != (rope != nullptr)) return NC_ERR_ARG;
  const bool out_f32 = (ep == NC_EP_STORE_F32 || ep == NC_EP_ACCUM_F32);
  if (amax && (out_f32 || ep == NC_EP_QKV_ROPE)) return NC_ERR_ARG;   // bf16 staged outputs only
  if (ldd < N || ((ldd * (out_f32 ? 4 : 2)) % 16) || (((uintptr_t)D) & 15)) return NC_ERR_ARG;
  if (!g_num_sms) {
    int dev = 0;
    NC_CUDA_TRY(cudaGetDevice(&dev));
    NC_CUDA_TRY(cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev));
  }
  const int BN = (N > 128) ? 256 : 128;
  const bool pair = g_gemm_pair && BN == 256 && M >= 256;
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.M = M; p.N = N; p.K = K;
  p.a_mn = 0; p.b_mn = 0;
  p.ep = ep;
  p.D = D; p.ldd = ldd;
  p.tiles_m = pair ? (M + 255) / 256 : (M + TC_BM - 1) / TC_BM;
  p.tiles_n = (N + BN - 1) / BN;
  p.num_kb = (K + 2 * TC_BK - 1) / (2 * TC_BK);
  p.err = err;
  p.wait_ns = g_tc_wait_ns;
  p.ws = nullptr;
  p.splits = 1;
  p.rope_T = 1;
  p.scale_a = scale_a; p.scale_b = scale_b;
  p.amax = amax;
  if (rope) {
    if (BN != 256 || (rope->hd != 64 && rope->hd != 128) || (N % rope->hd) || rope->nh * rope->hd > N ||
        rope->T <= 0 || (((uintptr_t)rope->tab) & 15) || !rope->rstd)
      return NC_ERR_ARG;
    if (rope->pair_rows < 0 || (rope->pair_rows > 0 && rope->pair_rows < rope->T)) return NC_ERR_ARG;
    p.rope_tab = rope->tab; p.rstd_qk = rope->rstd; p.rope_T = rope->T; p.rope_nh = rope->nh;
    p.rope_hd = rope->hd; p.rope_pair_rows = rope->pair_rows; p.rope_eps = rope->eps;
  }
  // 128-byte (128-element) K boxes; rows 128 (A), BN or 128 per CTA of a pair (B)
  CUtensorMap ta, tb, td, tx;
  memset(&tx, 0, sizeof(tx));
  if (!make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, M, lda, 128, TC_BM)) return NC_ERR_CUDA;
  if (!make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, N, ldb, 128, pair ? 128 : BN)) return NC_ERR_CUDA;
  p.tma_epi = out_f32 ? make_tmap_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, N, M, ldd, 32, 32)
                      : make_tmap_bf16_2d(&td, D, N, M, ldd, 64, 32);
  if (p.tma_epi && aux) {   // relu^2 backward: the saved relu(u)^2 arrives by TMA in the epilogue
    if ((ldaux % 8) || (((uintptr_t)aux) & 15)) return NC_ERR_ARG;
    p.aux = const_cast<void*>(aux);
    p.ldaux = ldaux;
    p.tma_epi = make_tmap_bf16_2d(&tx, aux, N, M, ldaux, 64, 32);
  }
  if (!p.tma_epi) return NC_ERR_CUDA;
  // split K (fp32 outputs, CTA pairs only, with a workspace): partials carry the factor
  if (pair && ws && out_f32) {
    if (((uintptr_t)ws) & 15) return NC_ERR_ARG;
    p.ws = (float*)ws;
    return launch_tc_pair<true>(p, ta, tb, td, tx, ws_bytes, st);
  }
  if (pair) return launch_tc_pair<true>(p, ta, tb, td, tx, 0, st);
  if (BN == 256) return launch_tc_bn<256, true>(p, ta, tb, td, tx, 0, st);
  return launch_tc_bn<128, true>(p, ta, tb, td, tx, 0, st);
}

nc_status launch_gemm_fp8(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                          const float* scale_a, const float* scale_b, int out_f32, void* D, int64_t ldd,
                          int32_t* err, cudaStream_t st) {
  return gemm_fp8_impl(M, N, K, A, lda, B, ldb, scale_a, scale_b, out_f32 ? NC_EP_STORE_F32 : NC_EP_STORE, D, ldd,
                       nullptr, err, st);
}

nc_status launch_gemm_fp8_ep(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                             const float* scale_a, const float* scale_b, int ep, void* D, int64_t ldd, int T, int nh,
                             int hd, const float* tab, int pair_rows, float* rstd, float eps, int32_t* err,
                             cudaStream_t st, const void* aux, int64_t ldaux, unsigned* amax, void* ws,
                             size_t ws_bytes) {
  if (ep != NC_EP_QKV_ROPE)
    return gemm_fp8_impl(M, N, K, A, lda, B, ldb, scale_a, scale_b, ep, D, ldd, nullptr, err, st, aux, ldaux, amax,
                         ws, ws_bytes);
  TcRope r{tab, rstd, T, nh, hd, pair_rows, eps};
  return gemm_fp8_impl(M, N, K, A, lda, B, ldb, scale_a, scale_b, ep, D, ldd, &r, err, st);
}

nc_status launch_gemm_tc_qkv_rope(int M, int N, int K, const bf16* A, int64_t lda, const bf16* Wqkv, int64_t ldb,
                                  bf16* qkv, int64_t ldd, int T, int nh, int hd, const float* tab, int pair_rows,
                                  float* rstd, float eps, int32_t* err, cudaStream_t st) {
  TcRope r{tab, rstd, T, nh, hd, pair_rows, eps};
  if (N <= 128) return NC_ERR_UNSUPPORTED;
  return gemm_tc_impl(M, N, K, A, lda, 1, Wqkv, ldb, 1, NC_EP_QKV_ROPE, qkv, ldd, nullptr, 0, &r, err, nullptr, 0,
                      st);
}
