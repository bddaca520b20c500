// Causal grouped-query flash attention on bf16 tensor cores (warp-level
// mma.sync m16n8k16, fp32 accumulation), forward and backward, head_dim 64 or
// 128.  Query head h reads kv head h / (H / Hkv) (cosmicrealm
// "noao-chat-0-项目总体介绍" §2.1 item 6); scores are q.k / sqrt(hd) under a
// causal mask.
//
// Layout: q, k, v are column blocks of the fused projection output
// qkv[B*T, (H + 2 Hkv) * hd]; o and do are [B*T, H * hd]; lse and the
// backward's rowsum(do * o) are fp32 [B, H, T].
//
// Forward: one CTA = 4 warps = 64 query rows (16 per warp) of one (b, h);
// key/value tiles of 64 rows stream through a double-buffered, XOR-swizzled
// shared-memory ring (cp.async); online softmax in registers with quad
// shuffles; P is re-packed from the score accumulators into mma A operands.
//
// Backward (deterministic, no atomics):
//   dq kernel    per 64-query tile: S = Q K^T, P = exp(S - lse),
//                dP = dO V^T, dS = P (dP - D), dQ += dS K;
//   dk/dv kernel per 64-key tile, over the group's query heads and the query
//                tiles at or after the diagonal: S^T = K Q^T, P^T,
//                dV += P^T dO, dP^T = V dO^T, dS^T, dK += dS^T Q.
#include "nc_kernels.cuh"
#include "nc_ptx.cuh"

namespace {

constexpr int FA_BM = 64;        // rows per CTA (16 per warp)
constexpr int FA_BN = 64;        // columns (keys or queries) per streamed tile
constexpr int FA_THREADS = 128;

struct FaShape {
  int B, T, H, Hkv, G;
  int64_t ld_qkv, ld_o;
  float scale_log2;   // log2(e) / sqrt(hd)
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, bool valid) {
  int n = valid ? 16 : 0;   // zero-fill rows past the sequence end
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Byte offset of element (row, col) in a [rows][HD] bf16 tile whose 16-byte
// chunks are XOR-swizzled by (row & 7), so that ldmatrix rows of one chunk
// column fall in distinct banks.
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * HD * 2 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}

// Load a [64][HD] tile: global rows row0.. (stride ld elements), rows >= nvalid zero-filled.
template <int HD>
__device__ __forceinline__ void load_tile(uint32_t sbase, const bf16* g, int64_t ld, int nvalid) {
  constexpr int CH = HD / 8;   // 16-byte chunks per row
  for (int i = threadIdx.x; i < FA_BN * CH; i += FA_THREADS) {
    int r = i / CH, c = i % CH;
    bool ok = r < nvalid;
    const bf16* src = g + (int64_t)(ok ? r : 0) * ld + c * 8;
    cp_async16(sbase + swz<HD>(r, c * 8), src, ok);
  }
}

// A fragments (16 rows x 16 cols, k-step kk) of a swizzled [rows][HD] tile, rows row0..row0+15.
template <int HD>
__device__ __forceinline__ void ld_a(uint32_t* a, uint32_t sbase, int row0, int kk) {
  const int lane = threadIdx.x & 31;
  int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
  int c = kk * 16 + (lane >> 4) * 8;
  ldsm_x4(a, sbase + swz<HD>(r, c));
}
// B fragments for C = A X^T where X is a swizzled [cols][HD] tile: n-tiles
// (8 cols) j and j+1 starting at col0, k-step kk.  b[0],b[1] -> n-tile j;
// b[2],b[3] -> n-tile j+1.
template <int HD>
__device__ __forceinline__ void ld_b_nt(uint32_t* b, uint32_t sbase, int col0, int kk) {
  const int lane = threadIdx.x & 31;
  int r = col0 + (lane & 7) + (lane >> 4) * 8;
  int c = kk * 16 + ((lane >> 3) & 1) * 8;
  ldsm_x4(b, sbase + swz<HD>(r, c));
}
// B fragments for C = P X where X is a swizzled [k rows][HD] tile: k-step
// rows kr..kr+15, output d-tiles dt and dt+1 (8 cols each).
template <int HD>
__device__ __forceinline__ void ld_b_nn(uint32_t* b, uint32_t sbase, int kr, int dt) {
  const int lane = threadIdx.x & 31;
  int r = kr + (lane & 7) + ((lane >> 3) & 1) * 8;
  int c = dt * 8 + (lane >> 4) * 8;
  ldsm_x4_t(b, sbase + swz<HD>(r, c));
}

// acc[8][4] (16 x 64) = A(16 x HD, swizzled smem rows arow0..) * X(64 x HD)^T
template <int HD>
__device__ __forceinline__ void gemm_abt(float (*acc)[4], uint32_t sa, int arow0, uint32_t sx) {
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    uint32_t a[4];
    ld_a<HD>(a, sa, arow0, kk);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      uint32_t b[4];
      ld_b_nt<HD>(b, sx, j * 8, kk);
      mma_bf16(acc[j], a, b[0], b[1]);
      mma_bf16(acc[j + 1], a, b[2], b[3]);
    }
  }
}

// out[HD/8][4] (16 x HD) += P(16 x 64, as packed bf16 A fragments p[4][4]) * X(64 x HD)
template <int HD>
__device__ __forceinline__ void gemm_pv(float (*out)[4], const uint32_t (*p)[4], uint32_t sx) {
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
    for (int dt = 0; dt < HD / 8; dt += 2) {
      uint32_t b[4];
      ld_b_nn<HD>(b, sx, ks * 16, dt);
      mma_bf16(out[dt], p[ks], b[0], b[1]);
      mma_bf16(out[dt + 1], p[ks], b[2], b[3]);
    }
  }
}

// Re-pack a 16 x 64 fp32 accumulator (C layout) as bf16 A fragments.
__device__ __forceinline__ void pack_a(uint32_t (*p)[4], const float (*s)[4]) {
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    p[ks][0] = pack_bf16(s[2 * ks][0], s[2 * ks][1]);
    p[ks][1] = pack_bf16(s[2 * ks][2], s[2 * ks][3]);
    p[ks][2] = pack_bf16(s[2 * ks + 1][0], s[2 * ks + 1][1]);
    p[ks][3] = pack_bf16(s[2 * ks + 1][2], s[2 * ks + 1][3]);
  }
}

// ---------------------------------------------------------------- forward
template <int HD>
__global__ void __launch_bounds__(FA_THREADS) k_fa_fwd(FaShape sh, const bf16* __restrict__ qkv,
                                                       bf16* __restrict__ o, float* __restrict__ lse) {
  extern __shared__ __align__(128) uint8_t fa_smem[];
  constexpr int TILE = FA_BN * HD * 2;
  const uint32_t sq = smem_u32(fa_smem);
  const uint32_t skv = sq + TILE;          // [2 stages][K, V]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (sh.T + FA_BM - 1) / FA_BM;
  const int qt = n_qt - 1 - blockIdx.x;   // heaviest (longest causal) tiles first
  const int bh = blockIdx.y, b = bh / sh.H, h = bh % sh.H, g = h / sh.G;
  const int q0 = qt * FA_BM;
  const int64_t rowb = (int64_t)b * sh.T;
  const bf16* Qg = qkv + (rowb + q0) * sh.ld_qkv + (int64_t)h * HD;
  const bf16* Kg = qkv + rowb * sh.ld_qkv + (int64_t)(sh.H + g) * HD;
  const bf16* Vg = qkv + rowb * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * HD;

  load_tile<HD>(sq, Qg, sh.ld_qkv, sh.T - q0);
  const int n_kt = qt + 1;   // causal: key tiles 0..qt (FA_BM == FA_BN)
  load_tile<HD>(skv, Kg, sh.ld_qkv, sh.T);
  load_tile<HD>(skv + TILE, Vg, sh.ld_qkv, sh.T);
  cp_async_commit();

  float acc_o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) acc_o[i][0] = acc_o[i][1] = acc_o[i][2] = acc_o[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  const int row_a = q0 + warp * 16 + (lane >> 2);   // this thread's two query rows: row_a, row_a + 8

  for (int kt = 0; kt < n_kt; ++kt) {
    const int st = kt & 1;
    if (kt + 1 < n_kt) {
      const uint32_t nx = skv + (st ^ 1) * 2 * TILE;
      const int k1 = (kt + 1) * FA_BN;
      load_tile<HD>(nx, Kg + (int64_t)k1 * sh.ld_qkv, sh.ld_qkv, sh.T - k1);
      load_tile<HD>(nx + TILE, Vg + (int64_t)k1 * sh.ld_qkv, sh.ld_qkv, sh.T - k1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sk = skv + st * 2 * TILE, sv = sk + TILE;
    float s[8][4];
    gemm_abt<HD>(s, sq, warp * 16, sk);
    const int k0 = kt * FA_BN;
    const bool diag = (kt == n_kt - 1) || (k0 + FA_BN > sh.T);
    float mx[2] = {m_r[0], m_r[1]};
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = k0 + j * 8 + (lane & 3) * 2 + (e & 1);
        const int row = row_a + (e >> 1) * 8;
        float v = s[j][e] * sh.scale_log2;
        if (diag && (col > row || col >= sh.T)) v = -INFINITY;
        s[j][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float corr[2], base[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      base[r] = (mx[r] == -INFINITY) ? 0.f : mx[r];
      corr[r] = exp2f(m_r[r] - base[r]);
      m_r[r] = mx[r];
      l_r[r] *= corr[r];
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float p = exp2f(s[j][e] - base[e >> 1]);
        s[j][e] = p;
        rs[e >> 1] += p;
      }
    l_r[0] += rs[0];
    l_r[1] += rs[1];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      acc_o[i][0] *= corr[0]; acc_o[i][1] *= corr[0];
      acc_o[i][2] *= corr[1]; acc_o[i][3] *= corr[1];
    }
    uint32_t p[4][4];
    pack_a(p, s);
    gemm_pv<HD>(acc_o, p, sv);
    __syncthreads();   // the stage is refilled by the next iteration's loads
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = row_a + r * 8;
    if (row >= sh.T) continue;
    const float inv = 1.f / l_r[r];
    bf16* orow = o + (rowb + row) * sh.ld_o + (int64_t)h * HD;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      const int c = i * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(orow + c) = pack_bf16(acc_o[i][2 * r] * inv, acc_o[i][2 * r + 1] * inv);
    }
    if ((lane & 3) == 0)   // natural-log logsumexp of the scaled scores
      lse[(int64_t)bh * sh.T + row] = (m_r[r] + log2f(l_r[r])) * 0.69314718055994531f;
  }
}

// ---------------------------------------------------------------- backward: dQ
template <int HD>
__global__ void __launch_bounds__(FA_THREADS) k_fa_bwd_dq(FaShape sh, const bf16* __restrict__ qkv,
                                                          const bf16* __restrict__ dout, const float* __restrict__ lse,
                                                          const float* __restrict__ Dv, bf16* __restrict__ dqkv) {
  extern __shared__ __align__(128) uint8_t fa_smem[];
  constexpr int TILE = FA_BN * HD * 2;
  const uint32_t sq = smem_u32(fa_smem);
  const uint32_t sdo = sq + TILE;
  const uint32_t skv = sdo + TILE;         // [2 stages][K, V]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (sh.T + FA_BM - 1) / FA_BM;
  const int qt = n_qt - 1 - blockIdx.x;
  const int bh = blockIdx.y, b = bh / sh.H, h = bh % sh.H, g = h / sh.G;
  const int q0 = qt * FA_BM;
  const int64_t rowb = (int64_t)b * sh.T;
  const bf16* Kg = qkv + rowb * sh.ld_qkv + (int64_t)(sh.H + g) * HD;
  const bf16* Vg = qkv + rowb * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * HD;
  load_tile<HD>(sq, qkv + (rowb + q0) * sh.ld_qkv + (int64_t)h * HD, sh.ld_qkv, sh.T - q0);
  load_tile<HD>(sdo, dout + (rowb + q0) * sh.ld_o + (int64_t)h * HD, sh.ld_o, sh.T - q0);
  load_tile<HD>(skv, Kg, sh.ld_qkv, sh.T);
  load_tile<HD>(skv + TILE, Vg, sh.ld_qkv, sh.T);
  cp_async_commit();
  const int row_a = q0 + warp * 16 + (lane >> 2);
  float L2[2], Dr[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = min(row_a + r * 8, sh.T - 1);
    L2[r] = lse[(int64_t)bh * sh.T + row] * 1.4426950408889634f;
    Dr[r] = Dv[(int64_t)bh * sh.T + row];
  }
  float acc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const int n_kt = qt + 1;
  const float scale = sh.scale_log2 * 0.69314718055994531f;   // 1/sqrt(hd)
  for (int kt = 0; kt < n_kt; ++kt) {
    const int st = kt & 1;
    if (kt + 1 < n_kt) {
      const uint32_t nx = skv + (st ^ 1) * 2 * TILE;
      const int k1 = (kt + 1) * FA_BN;
      load_tile<HD>(nx, Kg + (int64_t)k1 * sh.ld_qkv, sh.ld_qkv, sh.T - k1);
      load_tile<HD>(nx + TILE, Vg + (int64_t)k1 * sh.ld_qkv, sh.ld_qkv, sh.T - k1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sk = skv + st * 2 * TILE, sv = sk + TILE;
    float s[8][4], dp[8][4];
    gemm_abt<HD>(s, sq, warp * 16, sk);
    gemm_abt<HD>(dp, sdo, warp * 16, sv);
    const int k0 = kt * FA_BN;
    const bool diag = (kt == n_kt - 1) || (k0 + FA_BN > sh.T);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = k0 + j * 8 + (lane & 3) * 2 + (e & 1);
        const int row = row_a + (e >> 1) * 8;
        float p = exp2f(s[j][e] * sh.scale_log2 - L2[e >> 1]);
        if (diag && (col > row || col >= sh.T)) p = 0.f;
        s[j][e] = p * (dp[j][e] - Dr[e >> 1]) * scale;     // dS, with the 1/sqrt(hd) of dQ folded in
      }
    uint32_t ds[4][4];
    pack_a(ds, s);
    gemm_pv<HD>(acc, ds, sk);
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = row_a + r * 8;
    if (row >= sh.T) continue;
    bf16* dst = dqkv + (rowb + row) * sh.ld_qkv + (int64_t)h * HD;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      const int c = i * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16(acc[i][2 * r], acc[i][2 * r + 1]);
    }
  }
}

// ---------------------------------------------------------------- backward: dK, dV
template <int HD>
__global__ void __launch_bounds__(FA_THREADS) k_fa_bwd_dkv(FaShape sh, const bf16* __restrict__ qkv,
                                                           const bf16* __restrict__ dout,
                                                           const float* __restrict__ lse,
                                                           const float* __restrict__ Dv, bf16* __restrict__ dqkv) {
  extern __shared__ __align__(128) uint8_t fa_smem[];
  constexpr int TILE = FA_BN * HD * 2;
  const uint32_t sk = smem_u32(fa_smem);
  const uint32_t sv = sk + TILE;
  const uint32_t sqd = sv + TILE;          // [2 stages][Q, dO]
  float* sLD = reinterpret_cast<float*>(fa_smem + 6 * TILE);   // [2 stages][64 lse*log2e, 64 D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = (sh.T + FA_BN - 1) / FA_BN;
  const int kt = blockIdx.x;    // this CTA's key tile; the first tiles see the most queries, so go first
  const int bg = blockIdx.y, b = bg / sh.Hkv, g = bg % sh.Hkv;
  const int k0 = kt * FA_BN;
  const int64_t rowb = (int64_t)b * sh.T;
  load_tile<HD>(sk, qkv + (rowb + k0) * sh.ld_qkv + (int64_t)(sh.H + g) * HD, sh.ld_qkv, sh.T - k0);
  load_tile<HD>(sv, qkv + (rowb + k0) * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * HD, sh.ld_qkv, sh.T - k0);
  const int n_q = n_t - kt;                 // query tiles kt .. n_t-1 (causal)
  const int n_it = sh.G * n_q;              // over the group's query heads
  auto issue = [&](int it, int stage) {
    const int hh = it / n_q, qt = kt + it % n_q;
    const int h = g * sh.G + hh;
    const int q0 = qt * FA_BM;
    const uint32_t dst = sqd + stage * 2 * TILE;
    load_tile<HD>(dst, qkv + (rowb + q0) * sh.ld_qkv + (int64_t)h * HD, sh.ld_qkv, sh.T - q0);
    load_tile<HD>(dst + TILE, dout + (rowb + q0) * sh.ld_o + (int64_t)h * HD, sh.ld_o, sh.T - q0);
    float* ld = sLD + stage * 128;
    for (int i = threadIdx.x; i < FA_BM; i += FA_THREADS) {
      const int q = min(q0 + i, sh.T - 1);
      ld[i] = lse[((int64_t)b * sh.H + h) * sh.T + q] * 1.4426950408889634f;
      ld[64 + i] = Dv[((int64_t)b * sh.H + h) * sh.T + q];
    }
  };
  issue(0, 0);
  cp_async_commit();
  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }
  const int key_a = k0 + warp * 16 + (lane >> 2);   // this thread's two key rows
  const float scale = sh.scale_log2 * 0.69314718055994531f;
  for (int it = 0; it < n_it; ++it) {
    const int st = it & 1;
    if (it + 1 < n_it) {
      __syncthreads();   // the other stage's lse/D words are rewritten below
      issue(it + 1, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int q0 = (kt + it % n_q) * FA_BM;
    const uint32_t sq = sqd + st * 2 * TILE, sdo = sq + TILE;
    const float* ld = sLD + st * 128;
    float s[8][4], dp[8][4];
    gemm_abt<HD>(s, sk, warp * 16, sq);     // S^T: rows = keys, cols = queries
    gemm_abt<HD>(dp, sv, warp * 16, sdo);   // dP^T = V dO^T
    const bool diag = (q0 == k0) || (q0 + FA_BM > sh.T);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qc = j * 8 + (lane & 3) * 2 + (e & 1);
        const int q = q0 + qc;
        const int key = key_a + (e >> 1) * 8;
        float p = exp2f(s[j][e] * sh.scale_log2 - ld[qc]);
        if (diag && (q < key || q >= sh.T)) p = 0.f;
        s[j][e] = p;
        dp[j][e] = p * (dp[j][e] - ld[64 + qc]) * scale;
      }
    uint32_t pa[4][4];
    pack_a(pa, s);
    gemm_pv<HD>(dv, pa, sdo);       // dV += P^T dO
    pack_a(pa, dp);
    gemm_pv<HD>(dk, pa, sq);        // dK += dS^T Q
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int key = key_a + r * 8;
    if (key >= sh.T) continue;
    bf16* dkr = dqkv + (rowb + key) * sh.ld_qkv + (int64_t)(sh.H + g) * HD;
    bf16* dvr = dqkv + (rowb + key) * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * HD;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      const int c = i * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(dkr + c) = pack_bf16(dk[i][2 * r], dk[i][2 * r + 1]);
      *reinterpret_cast<uint32_t*>(dvr + c) = pack_bf16(dv[i][2 * r], dv[i][2 * r + 1]);
    }
  }
}

template <typename T>
__global__ void k_fa_rowdot(int64_t rows, int H, int hd, int T_, int64_t ld_o, const T* __restrict__ o,
                            const T* __restrict__ dout, float* __restrict__ Dv) {
  int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int lane = threadIdx.x & 31;
  if (w >= rows * H) return;
  int64_t row = w / H;
  int h = (int)(w % H);
  const T* a = o + row * ld_o + (int64_t)h * hd;
  const T* c = dout + row * ld_o + (int64_t)h * hd;
  float s = 0.f;
  for (int i = lane; i < hd; i += 32) s += to_f32(a[i]) * to_f32(c[i]);
  s = warp_sum(s);
  int b = (int)(row / T_), t = (int)(row % T_);
  if (lane == 0) Dv[((int64_t)b * H + h) * T_ + t] = s;
}

bool fa_shape(int B, int T, int H, int Hkv, int hd, FaShape* sh) {
  if (B <= 0 || T <= 0 || H <= 0 || Hkv <= 0 || H % Hkv || (hd != 64 && hd != 128)) return false;
  if ((int64_t)B * H > 65535) return false;
  sh->B = B; sh->T = T; sh->H = H; sh->Hkv = Hkv; sh->G = H / Hkv;
  sh->ld_qkv = (int64_t)(H + 2 * Hkv) * hd;
  sh->ld_o = (int64_t)H * hd;
  sh->scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  return true;
}

template <int HD>
nc_status fa_fwd(const FaShape& sh, const bf16* qkv, bf16* o, float* lse, cudaStream_t st) {
  const size_t smem = 5 * FA_BN * HD * 2;
  NC_CUDA_TRY(cudaFuncSetAttribute(k_fa_fwd<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  dim3 grid(cdiv(sh.T, FA_BM), sh.B * sh.H);
  k_fa_fwd<HD><<<grid, FA_THREADS, smem, st>>>(sh, qkv, o, lse);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

template <int HD>
nc_status fa_bwd(const FaShape& sh, const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, bf16* dqkv,
                 float* Dv, cudaStream_t st) {
  const int64_t rows = (int64_t)sh.B * sh.T;
  k_fa_rowdot<bf16><<<cdiv(rows * sh.H, 8), 256, 0, st>>>(rows, sh.H, HD, sh.T, sh.ld_o, o, dout, Dv);
  NC_CUDA_TRY(cudaGetLastError());
  const size_t smem_q = 6 * FA_BN * HD * 2;
  NC_CUDA_TRY(cudaFuncSetAttribute(k_fa_bwd_dq<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q));
  k_fa_bwd_dq<HD><<<dim3(cdiv(sh.T, FA_BM), sh.B * sh.H), FA_THREADS, smem_q, st>>>(sh, qkv, dout, lse, Dv, dqkv);
  NC_CUDA_TRY(cudaGetLastError());
  const size_t smem_k = 6 * FA_BN * HD * 2 + 2 * 128 * sizeof(float);
  NC_CUDA_TRY(cudaFuncSetAttribute(k_fa_bwd_dkv<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_k));
  k_fa_bwd_dkv<HD><<<dim3(cdiv(sh.T, FA_BN), sh.B * sh.Hkv), FA_THREADS, smem_k, st>>>(sh, qkv, dout, lse, Dv,
                                                                                      dqkv);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

}  // namespace

nc_status launch_attn_fwd_tc(int B, int T, int H, int Hkv, int hd, const bf16* qkv, bf16* o, float* lse,
                             cudaStream_t st) {
  FaShape sh;
  if (!fa_shape(B, T, H, Hkv, hd, &sh)) return NC_ERR_ARG;
  return hd == 128 ? fa_fwd<128>(sh, qkv, o, lse, st) : fa_fwd<64>(sh, qkv, o, lse, st);
}

nc_status launch_attn_bwd_tc(int B, int T, int H, int Hkv, int hd, const bf16* qkv, const bf16* o, const float* lse,
                             const bf16* dout, bf16* dqkv, float* Dv, cudaStream_t st) {
  FaShape sh;
  if (!fa_shape(B, T, H, Hkv, hd, &sh)) return NC_ERR_ARG;
  return hd == 128 ? fa_bwd<128>(sh, qkv, o, lse, dout, dqkv, Dv, st)
                   : fa_bwd<64>(sh, qkv, o, lse, dout, dqkv, Dv, st);
}
