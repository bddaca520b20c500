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
// MN-major A and B.  Every mbarrier wait is bounded in time: on expiry the
// kernel raises the timeout bit of the error flag, drains its own TMA loads
// and MMAs (again bounded) and frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

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
  int32_t* err;
  uint64_t wait_ns;
  // split-K: work unit u covers k-blocks [s*kps, (s+1)*kps) of tile t, with
  // s = u / tiles and t = u % tiles, so CTAs running together stream the same
  // K slice (L2 reuse).  With splits > 1 every unit writes its fp32 partial
  // to ws[s][t][128][BN] and a fix-up kernel sums the slices in order.
  int splits, kps;
  float* ws;
  // NC_EP_QKV_ROPE (the fused q/k/v projection): heads < rope_nh are rotated
  // (RoPE, cos/sin table [T][hd/2][2]) and RMS-normalised per head, their
  // rstd stored to rstd_qk[row * rope_nh + head]; the other heads are stored as is.
  const float* rope_tab;
  float* rstd_qk;
  int rope_T, rope_nh, rope_hd;
  float rope_eps;
};

// One unit of work of a CTA: k-blocks [k0, k1) of output tile t (slice s).
struct TcSeg {
  int t, s, k0, k1;
};

// Iterates the units a CTA owns, identically in every role.
struct TcSegIter {
  int u, stride, units, tiles;
  __device__ TcSegIter(const TcParams& p, int cta, int grid) {
    tiles = p.tiles_m * p.tiles_n;
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
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
};

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, bf16 A and
// B, operand majorness, N/8 and M/16.
__device__ __forceinline__ uint32_t tc_idesc(int bn, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
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
          v[i + j] *= 2.f * (sq ? sqrtf(x) : x);
        }
      }
    } else {
      for (int i = 0; i < 32; ++i) {
        const float x = (n0 + i < p.N) ? __bfloat162float(a[i]) : 0.f;
        v[i] = (n0 + i < p.N) ? v[i] * 2.f * (sq ? sqrtf(x) : x) : 0.f;
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

// NC_EP_QKV_ROPE epilogue of one row over `ncols` accumulator columns (whole
// heads) starting at output column n_base / TMEM column tcol0.  For a q or k
// head: rstd = 1/sqrt(mean(u^2) + eps) from the fp32 accumulator u (the
// rotation preserves the sum of squares, so this is the RMS of rope(u)), then
// y_i = (u_i cos + u_{i+d} sin) rstd, y_{i+d} = (-u_i sin + u_{i+d} cos) rstd
// with d = hd/2 and the angle of the row's position (cosmicrealm
// "noao-chat-0-项目总体介绍" §2.1 items 1-2: rotary embedding, then QK norm).
__device__ __forceinline__ void tc_epilogue_qkv_rope(const TcParams& p, int64_t m, int n_base, int ncols,
                                                     uint32_t tcol0) {
  const int hd = p.rope_hd, d = hd >> 1;
  const bool row_ok = m < p.M;
  const int t = (int)(m % p.rope_T);
#pragma unroll 1
  for (int hc = 0; hc < ncols; hc += hd) {
    const int n0 = n_base + hc;
    if (n0 >= p.N) break;
    const int head = n0 / hd;
    const uint32_t tc = tcol0 + hc;
    bf16* dst = (bf16*)p.D + m * p.ldd + n0;
    if (head >= p.rope_nh) {   // v head
#pragma unroll 1
      for (int c = 0; c < hd; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tc + c, r);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(r[e + k]);
            *reinterpret_cast<uint4*>(dst + c + e) = pack8_bf16(v);
          }
        }
      }
      continue;
    }
    float ss = 0.f;
#pragma unroll 1
    for (int c = 0; c < hd; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tc + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) ss += __uint_as_float(r[e]) * __uint_as_float(r[e]);
    }
    const float rs = rsqrtf(ss / (float)hd + p.rope_eps);
    const float4* cs = reinterpret_cast<const float4*>(p.rope_tab + (size_t)t * hd);
#pragma unroll 1
    for (int c = 0; c < d; c += 32) {
      uint32_t a[32], b[32];
      tmem_ld_32x32b_x32(tc + c, a);
      tmem_ld_32x32b_x32(tc + d + c, b);
      tmem_ld_wait();
      if (row_ok) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float y1[8], y2[8];
#pragma unroll
          for (int k = 0; k < 8; k += 2) {
            const float4 q = __ldg(cs + ((c + e + k) >> 1));   // cos_i, sin_i, cos_i+1, sin_i+1
            const float a0 = __uint_as_float(a[e + k]), a1 = __uint_as_float(a[e + k + 1]);
            const float b0 = __uint_as_float(b[e + k]), b1 = __uint_as_float(b[e + k + 1]);
            y1[k] = (a0 * q.x + b0 * q.y) * rs;
            y2[k] = (-a0 * q.y + b0 * q.x) * rs;
            y1[k + 1] = (a1 * q.z + b1 * q.w) * rs;
            y2[k + 1] = (-a1 * q.w + b1 * q.z) * rs;
          }
          *reinterpret_cast<uint4*>(dst + c + e) = pack8_bf16(y1);
          *reinterpret_cast<uint4*>(dst + d + c + e) = pack8_bf16(y2);
        }
      }
    }
    if (row_ok) p.rstd_qk[m * p.rope_nh + head] = rs;
  }
}

template <int BN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcParams p) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full_bar = (uint64_t*)(smem + S * Cfg::STAGE_BYTES);
  uint64_t* empty_bar = full_bar + S;
  uint64_t* acc_full = empty_bar + S;      // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* drain_bar = acc_empty + 2;     // [1]
  uint32_t* tmem_slot = (uint32_t*)(drain_bar + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], TC_EPI_WARPS); }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
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
      int tm, tn;
      tile_coords(p, sg.t, tm, tn);
      for (int kb = sg.k0; kb < sg.k1; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, p.wait_ns)) { fail(); break; }
        if (*abort_flag) break;
        uint8_t* sa = smem + stage * Cfg::STAGE_BYTES;
        uint8_t* sb = sa + Cfg::A_BYTES;
        mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
        const int k0 = kb * TC_BK;
        if (!p.a_mn) {
          tma_load_2d(sa, &tmA, &full_bar[stage], k0, tm * TC_BM);
        } else {
          tma_load_2d(sa, &tmA, &full_bar[stage], tm * TC_BM, k0);
          tma_load_2d(sa + 8192, &tmA, &full_bar[stage], tm * TC_BM + 64, k0);
        }
        if (!p.b_mn) {
          tma_load_2d(sb, &tmB, &full_bar[stage], k0, tn * BN);
        } else {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + 8192 * j, &tmB, &full_bar[stage], tn * BN + 64 * j, k0);
        }
        ++issued;
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
    // Drain: every load this thread issued must land before the CTA exits
    // (already true on the normal path, where the MMA issuer consumed them all).
    for (int s = 0; s < S; ++s) {
      long long n_s = issued / S + ((issued % S) > s ? 1 : 0);
      if (n_s > 0) mbar_wait_bounded(&full_bar[s], (uint32_t)((n_s - 1) & 1), p.wait_ns);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    const uint32_t idesc = tc_idesc(BN, p.a_mn, p.b_mn);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    TcSegIter it(p, blockIdx.x, gridDim.x);
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
        for (int k = 0; k < TC_BK / 16; ++k) {
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
    mbar_wait_bounded(drain_bar, 0, p.wait_ns);
  } else if (warp >= 4) {
    // ---------------- epilogue
    const int quarter = warp & 3;
    const int c_lo = ((warp - 4) >> 2) * (BN / 2);   // this warp's half of the columns
    int local = 0;
    TcSegIter it(p, blockIdx.x, gridDim.x);
    TcSeg sg;
    for (; !*abort_flag && it.next(p, sg); ++local) {
      int tm, tn;
      tile_coords(p, sg.t, tm, tn);
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
      if (p.ep == NC_EP_QKV_ROPE) {
        tc_epilogue_qkv_rope(p, m, tn * BN + c_lo, BN / 2, taddr + c_lo);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// Split-K fix-up: out (op)= sum over slices s = 0..splits-1, in that order
// (bitwise reproducible), of the fp32 partial tiles.  One block per tile.
template <int BN>
__global__ void __launch_bounds__(256) k_gemm_tc_fixup(TcParams p) {
  const int t = blockIdx.x;
  const int tiles = p.tiles_m * p.tiles_n;
  int tm, tn;
  tile_coords(p, t, tm, tn);
  for (int i = threadIdx.x; i < TC_BM * BN / 4; i += blockDim.x) {
    const int r = (i * 4) / BN, cc = (i * 4) % BN;
    const int64_t m = (int64_t)tm * TC_BM + r;
    const int n = tn * BN + cc;
    if (m >= p.M || n >= p.N) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sl = 0; sl < p.splits; ++sl) {
      const float4 v = *reinterpret_cast<const float4*>(p.ws + ((size_t)sl * tiles + t) * TC_BM * BN +
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
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &f, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  }
  return fn;
}

// 2D bf16 tensor map over a row-major [outer][inner] matrix with leading
// dimension ld (elements), box {box_inner, box_outer}, 128-byte swizzle.
bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, int64_t ld,
                      uint32_t box_inner, uint32_t box_outer) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int g_num_sms = 0;
uint64_t g_tc_wait_ns = 4000000000ull;   // bounded-wait limit of the tensor-core kernels

template <int BN>
static nc_status launch_tc_bn(TcParams p, const CUtensorMap& ta, const CUtensorMap& tb, size_t ws_bytes,
                              cudaStream_t st) {
  static bool attr_set = false;
  auto kern = k_gemm_tc<BN>;
  if (!attr_set) {
    NC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<BN>::SMEM));
    attr_set = true;
  }
  const int tiles = p.tiles_m * p.tiles_n;
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
  kern<<<grid, TC_THREADS, TcCfg<BN>::SMEM, st>>>(ta, tb, p);
  NC_CUDA_TRY(cudaGetLastError());
  if (p.splits > 1) {
    k_gemm_tc_fixup<BN><<<tiles, 256, 0, st>>>(p);
    NC_CUDA_TRY(cudaGetLastError());
  }
  return NC_OK;
}

// Split-K partials: up to 4 waves of 128 x 256 fp32 tiles per slice set.
size_t gemm_tc_workspace_bytes() { return (size_t)256 << 20; }

struct TcRope {
  const float* tab;
  float* rstd;
  int T, nh, hd;
  float eps;
};

static nc_status gemm_tc_impl(int M, int N, int K, const bf16* A, int64_t lda, int a_kmajor, const bf16* B,
                              int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd, void* aux, int64_t ldaux,
                              const TcRope* rope, int32_t* err, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (M <= 0 || N <= 0) return NC_OK;
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
  p.err = err;
  p.wait_ns = g_tc_wait_ns;
  p.ws = (float*)ws;
  p.splits = 1;
  p.kps = 0;
  p.rope_tab = nullptr; p.rstd_qk = nullptr; p.rope_T = 1; p.rope_nh = 0; p.rope_hd = 0; p.rope_eps = 0.f;
  if (rope) {
    // whole heads in each epilogue warp's 128 columns, 16-byte row segments
    if (ep != NC_EP_QKV_ROPE || BN != 256 || (rope->hd != 64 && rope->hd != 128) || (N % rope->hd) ||
        rope->nh * rope->hd > N || rope->T <= 0 || (ldd % 8) || (((uintptr_t)D) & 15) ||
        (((uintptr_t)rope->tab) & 15) || !rope->rstd)
      return NC_ERR_ARG;
    p.rope_tab = rope->tab; p.rstd_qk = rope->rstd; p.rope_T = rope->T; p.rope_nh = rope->nh;
    p.rope_hd = rope->hd; p.rope_eps = rope->eps;
  } else if (ep == NC_EP_QKV_ROPE) {
    return NC_ERR_ARG;
  }
  if (ws && (((uintptr_t)ws) & 15)) return NC_ERR_ARG;
  CUtensorMap ta, tb;
  bool ok;
  if (a_kmajor) ok = make_tmap_bf16_2d(&ta, A, K, M, lda, TC_BK, TC_BM);
  else ok = make_tmap_bf16_2d(&ta, A, M, K, lda, 64, TC_BK);
  if (!ok) return NC_ERR_CUDA;
  if (b_kmajor) ok = make_tmap_bf16_2d(&tb, B, K, N, ldb, TC_BK, BN);
  else ok = make_tmap_bf16_2d(&tb, B, N, K, ldb, 64, TC_BK);
  if (!ok) return NC_ERR_CUDA;
  if (BN == 256) return launch_tc_bn<256>(p, ta, tb, ws_bytes, st);
  return launch_tc_bn<128>(p, ta, tb, ws_bytes, st);
}

nc_status launch_gemm_tc(int M, int N, int K, const bf16* A, int64_t lda, int a_kmajor, const bf16* B,
                         int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd, void* aux, int64_t ldaux,
                         int32_t* err, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (ep == NC_EP_QKV_ROPE) return NC_ERR_ARG;
  return gemm_tc_impl(M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, ep, D, ldd, aux, ldaux, nullptr, err, ws,
                      ws_bytes, st);
}

nc_status launch_gemm_tc_qkv_rope(int M, int N, int K, const bf16* A, int64_t lda, const bf16* Wqkv, int64_t ldb,
                                  bf16* qkv, int64_t ldd, int T, int nh, int hd, const float* tab, float* rstd,
                                  float eps, int32_t* err, cudaStream_t st) {
  TcRope r{tab, rstd, T, nh, hd, eps};
  if (N <= 128) return NC_ERR_UNSUPPORTED;
  return gemm_tc_impl(M, N, K, A, lda, 1, Wqkv, ldb, 1, NC_EP_QKV_ROPE, qkv, ldd, nullptr, 0, &r, err, nullptr, 0,
                      st);
}
