// Causal grouped-query flash attention on the 5th-generation tensor cores:
// tcgen05.mma with fp32 accumulators in tensor memory (TMEM), operand tiles
// staged by TMA into 128-byte-swizzled shared memory, bf16 in and out,
// head_dim 64 or 128.  Query head h reads kv head h / (H / Hkv) (cosmicrealm
// "noao-chat-0-项目总体介绍" §2.1 item 6); scores are q.k / sqrt(hd) under a
// causal mask; the forward saves the natural-log logsumexp of every row.
//
// Layout: q, k, v are column blocks of the fused projection output
// qkv[B*T, (H + 2 Hkv) * hd]; o and do are [B*T, H * hd]; lse and the
// backward's D = rowsum(do * o) are fp32 [B, H, T].
//
// Every kernel is warp-specialised, 12 warps, one CTA per SM:
//   warp 0      TMA producer (one elected thread)
//   warps 1-3   MMA issuers (one thread each issues tcgen05.mma / tcgen05.commit;
//               a single thread issues only about one MMA per ~100 cycles, so
//               independent product chains get their own issuer); warp 2 also
//               allocates and frees the 512 TMEM columns
//   warps 4-11  "softmax" warps: each thread owns one TMEM lane = one row of
//               the score tile, so row reductions need no shuffles.
//
// Forward: a CTA takes 256 queries (two 128-row tiles i = 0, 1, issuers warps 1
//   and 3) of one (b, h) and streams the 128-key K and V tiles through a 4-slot
//   ring.  Per key tile j the tensor core computes S_i = Q_i K_j^T into TMEM;
//   warpgroup i turns its row of S_i into P = exp2(S * log2e/sqrt(hd) - m),
//   writes P as bf16 over the first 64 columns of S_i, and the tensor core
//   accumulates O_i += P V_j with P read from TMEM.  Tile 1 runs half a step
//   behind tile 0, so one tile's products overlap the other's softmax.  The
//   running max m is raised only when a row's new maximum exceeds it by more
//   than 8 (log2 units), in which case the warp rescales its rows of O in
//   TMEM; otherwise P <= 2^8, which bf16 and fp32 hold exactly enough.
// Backward (deterministic, no atomics), with P recomputed from lse:
//   dQ kernel    per 128-query tile, over key tiles 0..diagonal:
//                S = Q K^T (warp 1, double-buffered in TMEM, so S_{j+1} is
//                computed while the softmax works on step j), dP = dO V^T
//                (warp 2) into TMEM, dS = P (dP - D) as bf16 over S's
//                columns, dQ += dS K (warp 3);
//   dK/dV kernel per 128-key tile, over the group's query heads and the
//                64-query tiles from the diagonal on: S^T = K Q^T (warp 1),
//                dP^T = V dO^T (warp 2), double-buffered in TMEM; P^T and dS^T
//                as bf16 over their own product's columns; dV += P^T dO and
//                dK += dS^T Q (warp 3).
// The 1/sqrt(hd) of dQ and dK is applied to the fp32 accumulators on output.
// A TMEM region is only ever overwritten by the issuer whose earlier product
// reads it, or by softmax warps after a barrier that follows that read.
//
// Every mbarrier wait is bounded in time (the GEMM's limit): on expiry the
// kernel raises the timeout bit of the error flag, stops issuing work, drains
// its own TMA loads and MMAs (bounded again) and frees its TMEM.
#include <cuda.h>

#include "nc_kernels.cuh"
#include "nc_ptx.cuh"

extern uint64_t g_tc_wait_ns;

namespace {

constexpr int AT_THREADS = 384;
constexpr uint32_t CHUNK128 = 128 * 128;   // one [128 rows][64 bf16] swizzled chunk
constexpr uint32_t CHUNK64 = 64 * 128;     // one [64 rows][64 bf16] swizzled chunk
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.69314718055994531f;

struct AtShape {
  int B, T, H, Hkv, G;
  int64_t ld_qkv, ld_o;
  float scale_log2;   // log2(e) / sqrt(hd)
  float scale;        // 1 / sqrt(hd)
  int32_t* err;
  uint64_t wait_ns;
  // Backward only: with rope_tab set, dq and dk leave through the per-head
  // RMSNorm backward and the transposed rotation (rstd_qk [B*T, H+Hkv],
  // cos/sin table [T][hd/2][2]), i.e. as gradients of the projection output.
  const float* rope_tab;
  const float* rstd_qk;
  int rope_pair_rows;   // 0: rope_tab is [T][hd/2][2]; else pair-major [hd/4][rope_pair_rows][4]
  // Optional: atomic maximum of |output| as stored (bf16), as float bits, over
  // the rows inside T - O in the forward, all of dq, dk and dv in the backward -
  // for a per-tensor quantiser of that output.
  unsigned* amax;
};

// Commits a lane's maximum |value| (its row's, 0 past T) into sh.amax: warp
// maximum, rounded to bf16 (monotonic, so the maximum of the stored values),
// one atomic per warp.  The whole warp calls it.
__device__ __forceinline__ void at_amax_commit(const AtShape& sh, float am) {
  if (!sh.amax) return;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  if ((threadIdx.x & 31) == 0 && am > 0.f)
    atomicMax(sh.amax, __float_as_uint(__bfloat162float(__float2bfloat16_rn(am))));
}

// tcgen05.mma kind::f16 instruction descriptor: fp32 accumulator, bf16 A and
// B, A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128, N = n.
__device__ __forceinline__ uint32_t at_idesc(int n, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) | (8u << 24);
}
// K-major operand: rows of 64 elements (128 B) per chunk, chunks of `chunk`
// bytes along K; the kk-th 16-deep slice starts 32 B further in its chunk.
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk, uint32_t chunk) {
  return smem_desc(base + (uint32_t)(kk >> 2) * chunk + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
}
// MN-major operand read from a [K rows][64-element MN chunks] tile: MN chunks
// `chunk` bytes apart, 8-row K groups 1 KB apart, slice kk 16 rows further.
__device__ __forceinline__ uint64_t mndesc(uint32_t base, int kk, uint32_t chunk) {
  return smem_desc(base + (uint32_t)kk * 2048u, chunk, 1024u);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ bool at_wait(uint64_t* bar, uint32_t parity, const AtShape& sh, volatile int* abort_flag) {
  if (mbar_wait_bounded(bar, parity, sh.wait_ns)) return true;
  if (sh.err) atomicOr(sh.err, NC_DEVERR_TIMEOUT);
  *abort_flag = 1;
  return false;
}
// Every lane waits; the warp proceeds only if all lanes saw the phase.
__device__ __forceinline__ bool at_wait_warp(uint64_t* bar, uint32_t parity, const AtShape& sh,
                                             volatile int* abort_flag) {
  const bool ok = at_wait(bar, parity, sh, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait for a shared-memory counter written by another warp to reach
// `target` (counters only grow, so there is no phase to alias).
__device__ __forceinline__ bool at_wait_count(volatile int* cnt, int target, const AtShape& sh,
                                              volatile int* abort_flag) {
  if (*cnt >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (*cnt >= target) return true;
    if (*abort_flag) return false;
    if ((it & 255u) == 0 && globaltimer_ns() - t0 > sh.wait_ns) {
      if (sh.err) atomicOr(sh.err, NC_DEVERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// CTA order: heads in chunks of 16, and within a chunk the most expensive
// tile of every head first.  The chunk's K / V stays in L2 while its CTAs run,
// and the cheap tiles of one chunk overlap the expensive tiles of the next, so
// only the last chunk ends on short work.  Returns (rank, head): rank 0 is the
// most expensive tile.
__device__ __forceinline__ void at_cta_order(int idx, int heads, int ntiles, int& rank, int& head) {
  constexpr int HG = 16;
  const int chunk = idx / (HG * ntiles);
  const int hg = min(HG, heads - chunk * HG);
  const int within = idx - chunk * HG * ntiles;
  rank = within / hg;
  head = chunk * HG + within % hg;
}

// ======================================================================= forward
template <int HD>
struct FwdSmem {
  static constexpr uint32_t TILE = 128 * HD * 2;          // one [128][HD] bf16 tile
  static constexpr int NSLOT = 4;
  static constexpr uint32_t OFF_Q = 0;                    // Q0, Q1
  static constexpr uint32_t OFF_KV = 2 * TILE;            // 4-slot ring: K0 V0 K1 V1 ...
  static constexpr uint32_t OFF_BAR = OFF_KV + NSLOT * TILE;
  static constexpr size_t BYTES = 1024 + OFF_BAR + 256;
};

template <int HD, bool AMAX>
__global__ void __launch_bounds__(AT_THREADS, 1)
    k_attn_fwd_tc(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_o, AtShape sh,
                  bf16* __restrict__ o, float* __restrict__ lse) {
  using L = FwdSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = (uint64_t*)(smem + L::OFF_BAR);
  constexpr int NS = L::NSLOT;
  uint64_t* q_full = bar;          // [1]
  uint64_t* kv_full = bar + 1;     // [NS]
  uint64_t* kv_empty = kv_full + NS;
  uint64_t* s_full = kv_empty + NS;   // [2] S_i in TMEM (and every earlier MMA of the CTA done)
  uint64_t* p_full = s_full + 2;      // [2] P_i in TMEM, O_i rescaled (4 warps)
  uint64_t* pv_done = p_full + 2;     // [2] O_i += P_i V complete
  uint64_t* drain = pv_done + 2;      // [2] one per issuer
  uint32_t* tmem_slot = (uint32_t*)(drain + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  volatile int* s0_seen = abort_flag + 1;   // key tiles whose S_0 tile 0's softmax has seen

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (sh.T + 255) >> 8;
  int rank, bh;
  at_cta_order((int)blockIdx.x, sh.B * sh.H, nqb, rank, bh);
  const int qb = nqb - 1 - rank;                       // longest causal rows first
  const int b = bh / sh.H, h = bh - b * sh.H, g = h / sh.G;
  const int nt = (sh.T + 127) >> 7;
  const int n0 = 2 * qb + 1;                           // key tiles of query tile 0
  const int n1 = (2 * qb + 1 < nt) ? 2 * qb + 2 : 0;   // of query tile 1 (0: past the end)
  const int nmax = n1 > 0 ? n1 : n0;
  const int row0 = b * sh.T;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    // every K / V slot is released by both issuers when query tile 1 exists
    for (int s = 0; s < NS; ++s) { mbar_init(&kv_full[s], 1); mbar_init(&kv_empty[s], n1 > 0 ? 2 : 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1); mbar_init(&p_full[i], 4); mbar_init(&pv_done[i], 1); mbar_init(&drain[i], 1);
    }
    *abort_flag = 0;
    *s0_seen = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_qkv);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S0 cols 0-127, S1 128-255 (P_i overwrites the first 64 columns of S_i), O0 256.., O1 256+HD..
  const uint32_t tbase = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    mbar_arrive_expect_tx(q_full, 2 * L::TILE);
    for (int i = 0; i < 2; ++i)
      for (int c = 0; c < HD / 64; ++c)
        tma_load_2d(smem + L::OFF_Q + i * L::TILE + c * CHUNK128, &tm_qkv, q_full, h * HD + 64 * c,
                    row0 + (2 * qb + i) * 128);
    int issued = 0;
    for (int c = 0; c < 2 * nmax && !*abort_flag; ++c) {
      const int s = c % NS;
      if (!at_wait(&kv_empty[s], ((c / NS) & 1) ^ 1, sh, abort_flag)) break;
      const int col = ((c & 1) ? (sh.H + sh.Hkv + g) : (sh.H + g)) * HD;
      mbar_arrive_expect_tx(&kv_full[s], L::TILE);
      for (int cc = 0; cc < HD / 64; ++cc)
        tma_load_2d(smem + L::OFF_KV + s * L::TILE + cc * CHUNK128, &tm_qkv, &kv_full[s], col + 64 * cc,
                    row0 + (c >> 1) * 128);
      ++issued;
    }
    // every load lands before the CTA exits (already so unless aborted)
    mbar_wait_bounded(q_full, 0, NC_DRAIN_NS);
    for (int s = 0; s < NS; ++s) {
      const int uses = issued / NS + ((issued % NS) > s ? 1 : 0);
      if (uses > 0) mbar_wait_bounded(&kv_full[s], (uses - 1) & 1, NC_DRAIN_NS);
    }
  } else if ((warp == 1 || warp == 3) && lane == 0) {
    // ---------------- MMA issuers: warp 1 for query tile 0, warp 3 for tile 1.
    // A single thread issues at most about one MMA per ~100 cycles, less than
    // an M = 128, N = 128 product takes, so each tile has its own issuer and
    // the tensor pipe interleaves two independent chains
    //   S_i = Q_i K_j^T  ->  (softmax writes P_i over S_i)  ->  O_i += P_i V_j
    // In-order execution per issuer keeps S_i of tile j+1 behind O_i += P_i V_j.
    const int i = warp == 1 ? 0 : 1;
    const int n = i ? n1 : n0;
    const uint32_t id_s = at_idesc(128, 0), id_pv = at_idesc(HD, 1);
    const uint32_t sq = smem_u32(smem + L::OFF_Q) + i * L::TILE, skv = smem_u32(smem + L::OFF_KV);
    auto kv_ready = [&](int c) { return at_wait(&kv_full[c % NS], (c / NS) & 1, sh, abort_flag); };
    // (an inactive tile 1, n1 = 0, takes no part: the slots then count one release)
    bool ok = (n > 0) && at_wait(q_full, 0, sh, abort_flag);
    for (int j = 0; ok && j < nmax; ++j) {
      const int cK = 2 * j, cV = 2 * j + 1;
      if (j >= n) {
        // key tile only the other query tile uses: release its slots once filled
        if (kv_ready(cK)) mbar_arrive(&kv_empty[cK % NS]);
        if (kv_ready(cV)) mbar_arrive(&kv_empty[cV % NS]);
        continue;
      }
      if (!(ok = kv_ready(cK))) break;
      // Tile 1 runs half a step behind tile 0: its S is issued once tile 0's S of
      // the same key tile has completed, so the tensor core computes it while tile
      // 0's softmax runs (and tile 0's O += P V and next S during tile 1's softmax)
      // instead of both softmaxes running at once with the tensor core idle.  The
      // signal is a count, not s_full[0]'s phase parity, which would alias if
      // tile 0 were ever two key tiles ahead.
      if (i == 1 && j < n0 && !(ok = at_wait_count(s0_seen, j + 1, sh, abort_flag))) break;
      tc_fence_after();
      const uint32_t kb = skv + (cK % NS) * L::TILE;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        tc_mma_f16(tbase + i * 128, kdesc(sq, kk, CHUNK128), kdesc(kb, kk, CHUNK128), id_s, kk > 0 ? 1u : 0u);
      tc_commit(&s_full[i]);
      tc_commit(&kv_empty[cK % NS]);
      if (!(ok = kv_ready(cV)) || !(ok = at_wait(&p_full[i], j & 1, sh, abort_flag))) break;
      tc_fence_after();
      const uint32_t vb = skv + (cV % NS) * L::TILE;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)   // O_i += P_i V_j, P_i from tensor memory
        tc_mma_f16_ts(tbase + 256 + i * HD, tbase + i * 128 + 8 * kk, mndesc(vb, kk, CHUNK128), id_pv,
                      (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&pv_done[i]);
      tc_commit(&kv_empty[cV % NS]);
      if (*abort_flag) ok = false;
    }
    tc_commit(&drain[i]);
    mbar_wait_bounded(&drain[i], 0, NC_DRAIN_NS);
  } else if (warp >= 4) {
    // ---------------- softmax warpgroups: warps 4-7 own query tile 0, 8-11 tile 1
    const int i = (warp - 4) >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qt = 2 * qb + i;
    const int qpos = qt * 128 + r;
    const int n = i ? n1 : n0;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tbase + lane_off + i * 128;
    const uint32_t tO = tbase + lane_off + 256 + i * HD;
    float m = 0.f, l = 0.f;                        // running max (raw score units), row sum
    const float thresh = 8.f / sh.scale_log2;      // raise m only when it grows by > 2^8 in P
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!(ok = at_wait_warp(&s_full[i], j & 1, sh, abort_flag))) break;
      if (i == 0 && quarter == 0 && lane == 0) *s0_seen = j + 1;
      tc_fence_after();
      uint32_t x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tS + 32 * c, x + 32 * c);
      tmem_ld_wait();
      const int k0 = j * 128;
      if ((j == qt) || (k0 + 128 > sh.T)) {   // diagonal / ragged tile: mask in raw units
        const int lim = min(qpos - k0, sh.T - 1 - k0);   // last visible column
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) x[c] = __float_as_uint(-INFINITY);
      }
      // row max with 8 independent chains (raw score units)
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = __uint_as_float(x[e]);
#pragma unroll
      for (int c = 8; c < 128; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(x[c]));
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      // O_i += P_i V_{j-1} was issued before S_i of this tile, so it completed
      // with it: O_i is stable and may be rescaled here.
      if (j == 0) {
        m = (mx == -INFINITY) ? 0.f : mx;
      } else {
        const bool need = mx > m + thresh;
        if (__any_sync(0xffffffffu, need)) {
          const float mn = need ? mx : m;
          const float alpha = ex2_approx((m - mn) * sh.scale_log2);
          l *= alpha;
          m = mn;
#pragma unroll 1
          for (int c = 0; c < HD / 16; ++c) {
            uint32_t ov[16];
            tmem_ld_32x32b_x16(tO + 16 * c, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st_32x32b_x16(tO + 16 * c, ov);
          }
          tmem_st_wait();
        }
      }
      // p = 2^(s c - m c): one FFMA and one ex2 per score; 8 partial row sums.
      // (Moving a quarter of the exponentials to an FMA-pipe polynomial measured
      // 10 % slower: the softmax warps' issue slots, shared with the MMA-issuing
      // threads, bound this loop rather than the SFU.)
      // (two scores per FFMA2 / FADD2 instruction)
      const float mc = m * sh.scale_log2;
      const float2 sl2 = make_float2(sh.scale_log2, sh.scale_log2), nmc = make_float2(-mc, -mc);
      float2 s4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < 64; ++c) {   // packed in place: x[c] <- bf16x2(p[2c], p[2c+1])
        const float2 a = fma2(make_float2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])), sl2, nmc);
        const float2 p = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        s4[c & 3] = add2(s4[c & 3], p);
        x[c] = pack2(p.x, p.y);
      }
      const float sum = ((s4[0].x + s4[0].y) + (s4[1].x + s4[1].y)) + ((s4[2].x + s4[2].y) + (s4[3].x + s4[3].y));
      // P_i into the first 64 columns of S_i (this warp's lanes, already read)
      tmem_st_32x32b_x32(tS, x);
      tmem_st_32x32b_x32(tS + 32, x + 32);
      tmem_st_wait();
      l += sum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[i]);
    }
    if (ok && n > 0 && at_wait_warp(&pv_done[i], (n - 1) & 1, sh, abort_flag)) {
      tc_fence_after();
      const float inv = 1.f / l;
      float am = 0.f;   // max |O| of this row before the 1/l scale (a positive factor keeps the maximum)
      if constexpr (HD == 128) {
        // two 32 x 64 boxes per warp, staged in this tile's Q buffer (its last
        // S has completed) and stored by TMA
        const uint32_t sbox = smem_u32(smem + L::OFF_Q + i * L::TILE + quarter * 8192) + (uint32_t)lane * 128u;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t ovp[64];   // a box's two accumulator loads under one wait
          tmem_ld_32x32b_x32(tO + 64 * c, ovp);
          tmem_ld_32x32b_x32(tO + 64 * c + 32, ovp + 32);
          tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint32_t* ov = ovp + 32 * cc;
            if (AMAX) {
#pragma unroll
              for (int e = 0; e < 32; ++e) am = fmaxf(am, fabsf(__uint_as_float(ov[e])));
            }
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              const uint32_t chunk = (uint32_t)(4 * cc + e / 8);
              st_shared_v4(sbox + c * 4096u + (((chunk ^ (uint32_t)lane) & 7u) << 4),
                           pack2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv),
                           pack2(__uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv),
                           pack2(__uint_as_float(ov[e + 4]) * inv, __uint_as_float(ov[e + 5]) * inv),
                           pack2(__uint_as_float(ov[e + 6]) * inv, __uint_as_float(ov[e + 7]) * inv));
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && qt * 128 + quarter * 32 < sh.T) {
          for (int c = 0; c < 2; ++c)
            tma_store_3d(&tm_o, smem + L::OFF_Q + i * L::TILE + quarter * 8192 + c * 4096, h * HD + 64 * c,
                         qt * 128 + quarter * 32, b);
          bulk_commit();
          bulk_wait_all();
        }
      } else {
      bf16* orow = o + (int64_t)(row0 + qpos) * sh.ld_o + (int64_t)h * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tO + 32 * c, ov);
        tmem_ld_wait();
        if (qpos < sh.T) {
          if (AMAX) {
#pragma unroll
            for (int e = 0; e < 32; ++e) am = fmaxf(am, fabsf(__uint_as_float(ov[e])));
          }
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
            w.y = pack2(__uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
            w.z = pack2(__uint_as_float(ov[e + 4]) * inv, __uint_as_float(ov[e + 5]) * inv);
            w.w = pack2(__uint_as_float(ov[e + 6]) * inv, __uint_as_float(ov[e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c + e) = w;
          }
        }
      }
      }
      if (AMAX) at_amax_commit(sh, qpos < sh.T ? am * inv : 0.f);
      if (qpos < sh.T) lse[(int64_t)bh * sh.T + qpos] = (m * sh.scale_log2 + log2f(l)) * LN2;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 512);
}

// Output of a dQ or dK tile (128 rows x HD in TMEM, fp32) by the 8 epilogue
// warps (quarter = TMEM lane group, hf = half).  Plain: dst = scale * acc in
// bf16, each half-warp group writing HD/2 columns.  With rope_tab: g = scale *
// acc is the gradient of the normalised, rotated head y (the bf16 tile in
// shared memory, [128][HD] as 64-column 128B-swizzled chunks); the thread
// forms dot = mean(g * y) over the whole row, dr = rstd * (g - y * dot)
// (RMSNorm backward), and for its half of the rotation pairs (i, i + HD/2)
// writes dx_i = dr_i cos - dr_{i+d} sin, dx_{i+d} = dr_i sin + dr_{i+d} cos
// (the transpose of the forward rotation at the row's position).
// What the fused output reads from global memory besides the accumulator: the
// row's q/k-norm rstd and its half of the rotation table.  at_out_prefetch
// loads them before the last products complete, so that their L2 round trips
// overlap the tensor core's tail instead of following it.
template <int HD>
struct AtOutPre {
  float rr;
  float4 t[HD / 8];   // (cos_i, sin_i, cos_i+1, sin_i+1) for the thread's HD / 4 rotation pairs
};
template <int HD>
__device__ __forceinline__ void at_out_prefetch(const AtShape& sh, int hf, bool valid, int pos, int64_t token,
                                                int head, AtOutPre<HD>& pre) {
  constexpr int PW = HD / 4;
  pre.rr = 0.f;
#pragma unroll
  for (int k = 0; k < PW / 2; ++k) pre.t[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!sh.rope_tab || !valid) return;   // rows past the end read nothing (the table may end at T)
  pre.rr = sh.rstd_qk[token * (sh.H + sh.Hkv) + head];
  const size_t cstep = sh.rope_pair_rows ? (size_t)sh.rope_pair_rows : 1;
  const float4* cs = reinterpret_cast<const float4*>(sh.rope_tab) +
                     (sh.rope_pair_rows ? (size_t)pos : (size_t)pos * (HD / 4)) + (size_t)((hf * PW) >> 1) * cstep;
#pragma unroll
  for (int k = 0; k < PW / 2; ++k) pre.t[k] = __ldg(cs + (size_t)k * cstep);
}

template <int HD, bool AMAX>
__device__ __forceinline__ void at_out_tile(const AtShape& sh, uint32_t tacc, const uint8_t* ytile, int r, int hf,
                                            bool valid, const AtOutPre<HD>& pre, bf16* dst, float& am) {
  if (!sh.rope_tab) {
#pragma unroll 1
    for (int c = 0; c < HD / 64; ++c) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tacc + hf * (HD / 2) + 32 * c, v);
      tmem_ld_wait();
      if (valid) {
        if (AMAX) {
#pragma unroll
          for (int e = 0; e < 32; ++e) am = fmaxf(am, fabsf(__uint_as_float(v[e])) * sh.scale);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 w;
          w.x = pack2(__uint_as_float(v[e]) * sh.scale, __uint_as_float(v[e + 1]) * sh.scale);
          w.y = pack2(__uint_as_float(v[e + 2]) * sh.scale, __uint_as_float(v[e + 3]) * sh.scale);
          w.z = pack2(__uint_as_float(v[e + 4]) * sh.scale, __uint_as_float(v[e + 5]) * sh.scale);
          w.w = pack2(__uint_as_float(v[e + 6]) * sh.scale, __uint_as_float(v[e + 7]) * sh.scale);
          *reinterpret_cast<uint4*>(dst + hf * (HD / 2) + 32 * c + e) = w;
        }
      }
    }
    return;
  }
  constexpr int D = HD / 2, PW = D / 2;   // pairs per thread
  const uint32_t ybase = smem_u32(ytile) + r * 128;
  auto y8 = [&](int col, float* f) {      // 8 bf16 of row r from column col (multiple of 8)
    const uint4 u = ld_shared_v4(ybase + (col >> 6) * CHUNK128 + (((((uint32_t)col >> 3) & 7u) ^ (r & 7)) << 4));
    const bf16* b = reinterpret_cast<const bf16*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(b[e]);
  };
  float dot = 0.f;
#pragma unroll 1
  for (int c = 0; c < HD; c += 64) {   // two loads under one wait
    uint32_t v[64];
    tmem_ld_32x32b_x32(tacc + c, v);
    tmem_ld_32x32b_x32(tacc + c + 32, v + 32);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 64; q += 8) {
      float y[8];
      y8(c + q, y);
#pragma unroll
      for (int e = 0; e < 8; ++e) dot += __uint_as_float(v[q + e]) * y[e];
    }
  }
  dot *= sh.scale / (float)HD;
  const float rr = pre.rr;
  const int i0 = hf * PW;
  uint32_t g1[PW], g2[PW];
  if constexpr (PW == 32) {
    tmem_ld_32x32b_x32(tacc + i0, g1);
    tmem_ld_32x32b_x32(tacc + D + i0, g2);
  } else {
    tmem_ld_32x32b_x16(tacc + i0, g1);
    tmem_ld_32x32b_x16(tacc + D + i0, g2);
  }
  tmem_ld_wait();
  if (!valid) return;
#pragma unroll
  for (int q = 0; q < PW; q += 8) {
    float y1[8], y2[8], o1[8], o2[8];
    y8(i0 + q, y1);
    y8(D + i0 + q, y2);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float4 t = pre.t[(q + e) >> 1];   // cos_i, sin_i, cos_i+1, sin_i+1
      const float a0 = rr * (__uint_as_float(g1[q + e]) * sh.scale - y1[e] * dot);
      const float a1 = rr * (__uint_as_float(g1[q + e + 1]) * sh.scale - y1[e + 1] * dot);
      const float b0 = rr * (__uint_as_float(g2[q + e]) * sh.scale - y2[e] * dot);
      const float b1 = rr * (__uint_as_float(g2[q + e + 1]) * sh.scale - y2[e + 1] * dot);
      o1[e] = a0 * t.x - b0 * t.y;
      o2[e] = a0 * t.y + b0 * t.x;
      o1[e + 1] = a1 * t.z - b1 * t.w;
      o2[e + 1] = a1 * t.w + b1 * t.z;
    }
    if (AMAX) {
#pragma unroll
      for (int e = 0; e < 8; ++e) am = fmaxf(am, fmaxf(fabsf(o1[e]), fabsf(o2[e])));
    }
    uint4 w1, w2;
    w1.x = pack2(o1[0], o1[1]); w1.y = pack2(o1[2], o1[3]); w1.z = pack2(o1[4], o1[5]); w1.w = pack2(o1[6], o1[7]);
    w2.x = pack2(o2[0], o2[1]); w2.y = pack2(o2[2], o2[3]); w2.z = pack2(o2[4], o2[5]); w2.w = pack2(o2[6], o2[7]);
    *reinterpret_cast<uint4*>(dst + i0 + q) = w1;
    *reinterpret_cast<uint4*>(dst + D + i0 + q) = w2;
  }
}

// Plain output (mul * acc) of a 128 x 128 tile through shared memory and TMA.
// Warp (quarter, hf) writes columns [64 hf, 64 hf + 64) of its 32 rows as bf16
// into `box` (4 KB, 1024-aligned, 128-byte swizzled rows); one lane stores it
// by TMA at {x, y, bz} of a [B][T][cols] tensor map, which drops rows at or
// past T.  Every lane of the warp takes part, and the warp is converged again
// on return (the caller may issue aligned tcgen05 instructions next).
__device__ __forceinline__ void at_out_box128(uint32_t tacc, int hf, float mul, uint8_t* box, const CUtensorMap* tm,
                                              int x, int y, int bz, int T, float& am, bool track) {
  const int lane = threadIdx.x & 31;
  const uint32_t srow = smem_u32(box) + (uint32_t)lane * 128u;
  uint32_t v[64];   // both loads under one wait
  tmem_ld_32x32b_x32(tacc + hf * 64, v);
  tmem_ld_32x32b_x32(tacc + hf * 64 + 32, v + 32);
  tmem_ld_wait();
  if (track && y + lane < T) {   // rows past the end are not stored
#pragma unroll
    for (int e = 0; e < 64; ++e) am = fmaxf(am, fabsf(__uint_as_float(v[e])) * mul);
  }
#pragma unroll
  for (int e = 0; e < 64; e += 8)
    st_shared_v4(srow + ((((uint32_t)(e / 8) ^ (uint32_t)lane) & 7u) << 4),
                 pack2(__uint_as_float(v[e]) * mul, __uint_as_float(v[e + 1]) * mul),
                 pack2(__uint_as_float(v[e + 2]) * mul, __uint_as_float(v[e + 3]) * mul),
                 pack2(__uint_as_float(v[e + 4]) * mul, __uint_as_float(v[e + 5]) * mul),
                 pack2(__uint_as_float(v[e + 6]) * mul, __uint_as_float(v[e + 7]) * mul));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && y < T) {
    tma_store_3d(tm, box, x, y, bz);
    bulk_commit();
  }
  __syncwarp();
}

// ======================================================================= backward: dQ
template <int HD>
struct DqSmem {
  static constexpr uint32_t TILE = 128 * HD * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = TILE;
  // K_j is held until dQ += dS K_j completes, late in step j, so its ring is one
  // slot deeper than V's (V_j is released right after dP = dO V_j^T).
  static constexpr int NK = 3, NV = 2;
  static constexpr uint32_t OFF_K = 2 * TILE;               // NK slots
  static constexpr uint32_t OFF_V = OFF_K + NK * TILE;      // NV slots
  static constexpr uint32_t OFF_BAR = OFF_V + NV * TILE;
  static constexpr size_t BYTES = 1024 + OFF_BAR + 256;
};

template <int HD, bool AMAX>
__global__ void __launch_bounds__(AT_THREADS, 1)
    k_attn_bwd_dq_tc(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_out, AtShape sh, const float* __restrict__ lse,
                     const float* __restrict__ Dv, bf16* __restrict__ dqkv) {
  using L = DqSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = (uint64_t*)(smem + L::OFF_BAR);
  constexpr int NK = L::NK, NV = L::NV;
  uint64_t* qd_full = bar;            // [1]
  uint64_t* k_full = qd_full + 1;     // [NK]
  uint64_t* k_empty = k_full + NK;    // [NK]
  uint64_t* v_full = k_empty + NK;    // [NV]
  uint64_t* v_empty = v_full + NV;    // [NV]
  uint64_t* s_full = v_empty + NV;    // [2] S_j in TMEM buffer j & 1
  uint64_t* dp_full = s_full + 2;     // dP_j in TMEM
  uint64_t* sdp_free = dp_full + 1;   // S_j and dP_j read (8 warps)
  uint64_t* ds_full = sdp_free + 1;   // [2] dS_j written over S_j's columns (8 warps)
  uint64_t* buf_free = ds_full + 2;   // [2] dQ += dS_j K_j complete: buffer j & 1 may take S_{j+2}
  uint64_t* dq_done = buf_free + 2;
  uint64_t* drain = dq_done + 1;      // [3] one per issuer
  uint32_t* tmem_slot = (uint32_t*)(drain + 3);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = (sh.T + 127) >> 7;
  int rank, bh;
  at_cta_order((int)blockIdx.x, sh.B * sh.H, nt, rank, bh);
  const int qt = nt - 1 - rank;                        // longest causal rows first
  const int b = bh / sh.H, h = bh - b * sh.H, g = h / sh.G;
  const int n = qt + 1;
  const int row0 = b * sh.T;

  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    for (int s = 0; s < NK; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < NV; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&ds_full[i], 8); mbar_init(&buf_free[i], 1); }
    mbar_init(dp_full, 1); mbar_init(sdp_free, 8);
    mbar_init(dq_done, 1);
    for (int r = 0; r < 3; ++r) mbar_init(&drain[r], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_qkv);
    prefetch_tmap(&tm_do);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S_j in buffer j & 1 (columns 0-127 or 128-255), dP 256-383, dQ 384.. .  The
  // softmax warp of half hf reads S columns [64 hf, 64 hf + 64) of its buffer and
  // writes dS_j there as 32 bf16-pair columns, [64 hf, 64 hf + 32); dQ += dS_j K_j
  // reads them.  S_{j+2} overwrites the buffer only after buf_free signals that
  // dQ_j completed (the S issuer waits for it), so a buffer is written by the
  // tensor core only when no product reads it and by the softmax warps only
  // between S_j's completion and S_{j+2}'s issue.
  const uint32_t tbase = *tmem_slot;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(qd_full, 2 * L::TILE);
    for (int c = 0; c < HD / 64; ++c) {
      tma_load_2d(smem + L::OFF_Q + c * CHUNK128, &tm_qkv, qd_full, h * HD + 64 * c, row0 + qt * 128);
      tma_load_2d(smem + L::OFF_DO + c * CHUNK128, &tm_do, qd_full, h * HD + 64 * c, row0 + qt * 128);
    }
    int k_issued = 0, v_issued = 0;
    for (int j = 0; j < n && !*abort_flag; ++j) {
      const int sk_ = j % NK, sv_ = j % NV;
      if (!at_wait(&k_empty[sk_], ((j / NK) & 1) ^ 1, sh, abort_flag)) break;
      mbar_arrive_expect_tx(&k_full[sk_], L::TILE);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_2d(smem + L::OFF_K + sk_ * L::TILE + c * CHUNK128, &tm_qkv, &k_full[sk_],
                    (sh.H + g) * HD + 64 * c, row0 + j * 128);
      ++k_issued;
      if (!at_wait(&v_empty[sv_], ((j / NV) & 1) ^ 1, sh, abort_flag)) break;
      mbar_arrive_expect_tx(&v_full[sv_], L::TILE);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_2d(smem + L::OFF_V + sv_ * L::TILE + c * CHUNK128, &tm_qkv, &v_full[sv_],
                    (sh.H + sh.Hkv + g) * HD + 64 * c, row0 + j * 128);
      ++v_issued;
    }
    mbar_wait_bounded(qd_full, 0, NC_DRAIN_NS);
    for (int s = 0; s < NK; ++s) {
      const int ku = k_issued / NK + ((k_issued % NK) > s ? 1 : 0);
      if (ku > 0) mbar_wait_bounded(&k_full[s], (ku - 1) & 1, NC_DRAIN_NS);
    }
    for (int s = 0; s < NV; ++s) {
      const int vu = v_issued / NV + ((v_issued % NV) > s ? 1 : 0);
      if (vu > 0) mbar_wait_bounded(&v_full[s], (vu - 1) & 1, NC_DRAIN_NS);
    }
  } else if ((warp == 1 || warp == 2 || warp == 3) && lane == 0) {
    // ---------------- three MMA issuers (one thread issues about one MMA per ~100
    // cycles): warp 1 S_j = Q K_j^T into buffer j & 1, up to two steps ahead of the
    // softmax; warp 2 dP_j = dO V_j^T, once the softmax has read dP_{j-1}; warp 3
    // dQ += dS_j K_j.
    const int role = warp - 1;
    const uint32_t id_s = at_idesc(128, 0), id_q = at_idesc(HD, 1);
    const uint32_t sq = smem_u32(smem + L::OFF_Q), sdo = smem_u32(smem + L::OFF_DO);
    const uint32_t sk = smem_u32(smem + L::OFF_K), sv = smem_u32(smem + L::OFF_V);
    bool ok = at_wait(qd_full, 0, sh, abort_flag);
    if (role == 0) {
      for (int j = 0; ok && j < n; ++j) {
        if (!(ok = at_wait(&k_full[j % NK], (j / NK) & 1, sh, abort_flag))) break;
        if (j >= 2 && !(ok = at_wait(&buf_free[j & 1], ((j - 2) >> 1) & 1, sh, abort_flag))) break;
        tc_fence_after();
        const uint32_t kb = sk + (j % NK) * L::TILE;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma_f16(tbase + (j & 1) * 128, kdesc(sq, kk, CHUNK128), kdesc(kb, kk, CHUNK128), id_s, kk > 0 ? 1u : 0u);
        tc_commit(&s_full[j & 1]);
        if (*abort_flag) ok = false;
      }
    } else if (role == 1) {
      for (int j = 0; ok && j < n; ++j) {
        if (!(ok = at_wait(&v_full[j % NV], (j / NV) & 1, sh, abort_flag))) break;
        if (j > 0 && !(ok = at_wait(sdp_free, (j - 1) & 1, sh, abort_flag))) break;
        tc_fence_after();
        const uint32_t vb = sv + (j % NV) * L::TILE;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma_f16(tbase + 256, kdesc(sdo, kk, CHUNK128), kdesc(vb, kk, CHUNK128), id_s, kk > 0 ? 1u : 0u);
        tc_commit(dp_full);
        tc_commit(&v_empty[j % NV]);
        if (*abort_flag) ok = false;
      }
    } else {
      for (int j = 0; ok && j < n; ++j) {   // dQ += dS_j K_j, dS from tensor memory
        if (!(ok = at_wait(&ds_full[j & 1], (j >> 1) & 1, sh, abort_flag))) break;
        tc_fence_after();
        const uint32_t kb = sk + (j % NK) * L::TILE;
        const uint32_t ds = tbase + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // keys [16 kk, 16 kk + 16): half kk / 4, pair column 8 (kk % 4)
          tc_mma_f16_ts(tbase + 384, ds + 64 * (kk >> 2) + 8 * (kk & 3), mndesc(kb, kk, CHUNK128), id_q,
                        (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&buf_free[j & 1]);
        tc_commit(&k_empty[j % NK]);
        if (*abort_flag) ok = false;
      }
      if (ok) tc_commit(dq_done);
    }
    tc_commit(&drain[role]);
    mbar_wait_bounded(&drain[role], 0, NC_DRAIN_NS);
  } else if (warp >= 4) {
    const int quarter = warp & 3, hf = (warp - 4) >> 2;   // hf: key columns [64 hf, 64 hf + 64)
    const int r = quarter * 32 + lane;
    const int qpos = qt * 128 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tP = tbase + lane_off + 256 + 64 * hf;
    const bool valid = qpos < sh.T;
    const float lse2 = valid ? lse[(int64_t)bh * sh.T + qpos] * LOG2E : INFINITY;
    const float Dr = valid ? Dv[(int64_t)bh * sh.T + qpos] : 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!(ok = at_wait_warp(&s_full[j & 1], (j >> 1) & 1, sh, abort_flag))) break;
      if (!(ok = at_wait_warp(dp_full, j & 1, sh, abort_flag))) break;
      tc_fence_after();
      const uint32_t tS = tbase + lane_off + (j & 1) * 128 + 64 * hf;
      uint32_t s[64], dp[64];
      tmem_ld_32x32b_x32(tS, s);
      tmem_ld_32x32b_x32(tS + 32, s + 32);
      tmem_ld_32x32b_x32(tP, dp);
      tmem_ld_32x32b_x32(tP + 32, dp + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sdp_free);
      const int k0 = j * 128 + 64 * hf;
      const bool diag = (j == qt) || (j * 128 + 128 > sh.T);
      // two scores per FFMA2 / FADD2 / FMUL2 instruction
      const float2 sl2 = make_float2(sh.scale_log2, sh.scale_log2), nl2 = make_float2(-lse2, -lse2),
                   d2 = make_float2(Dr, Dr);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 a = fma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2, nl2);
        float2 p = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        if (diag) {
          if (k0 + c > qpos || k0 + c >= sh.T) p.x = 0.f;
          if (k0 + c + 1 > qpos || k0 + c + 1 >= sh.T) p.y = 0.f;
        }
        const float2 ds = mul2(p, sub2(make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), d2));
        s[c] = __float_as_uint(ds.x);
        s[c + 1] = __float_as_uint(ds.y);
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) s[c] = pack2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1]));
      tmem_st_32x32b_x32(tS, s);            // dS_j over the S columns this warp read
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[j & 1]);
    }
    AtOutPre<HD> pre;
    at_out_prefetch<HD>(sh, hf, ok && valid, qpos, (int64_t)row0 + qpos, h, pre);
    float am = 0.f;
    if (ok && at_wait_warp(dq_done, 0, sh, abort_flag)) {
      tc_fence_after();
      if (HD == 128 && !sh.rope_tab) {
        // staged in the K ring, free once every dQ product has completed
        at_out_box128(tbase + lane_off + 384, hf, sh.scale, smem + L::OFF_K + (hf * 4 + quarter) * 4096, &tm_out,
                      h * HD + hf * 64, qt * 128 + quarter * 32, b, sh.T, am, AMAX);
        if (lane == 0) bulk_wait_all();
      } else {
        at_out_tile<HD, AMAX>(sh, tbase + lane_off + 384, smem + L::OFF_Q, r, hf, valid, pre,
                        dqkv + (int64_t)(row0 + qpos) * sh.ld_qkv + (int64_t)h * HD, am);
      }
      if (AMAX) at_amax_commit(sh, am);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 512);
}

// ======================================================================= backward: dK, dV
template <int HD>
struct DkvSmem {
  static constexpr uint32_t KT = 128 * HD * 2;       // one [128][HD] tile
  static constexpr uint32_t QT = 64 * HD * 2;        // one [64][HD] tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = KT;
  static constexpr int NS = 4;
  static constexpr uint32_t OFF_QS = 2 * KT;                // NS stages of {Q, dO}
  static constexpr uint32_t OFF_LD = OFF_QS + NS * 2 * QT;  // per softmax warp {lse*log2e[32], D[32]}
  static constexpr uint32_t OFF_BAR = OFF_LD + 8 * 64 * 4;
  static constexpr size_t BYTES = 1024 + OFF_BAR + 256;
};

template <int HD, bool AMAX>
__global__ void __launch_bounds__(AT_THREADS, 1)
    k_attn_bwd_dkv_tc(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_out,
                      AtShape sh, const float* __restrict__ lse, const float* __restrict__ Dv,
                      bf16* __restrict__ dqkv) {
  using L = DkvSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = (uint64_t*)(smem + L::OFF_BAR);
  constexpr int NS = L::NS;
  uint64_t* kv_full = bar;              // [1]
  uint64_t* q_full = bar + 1;           // [NS] TMA bytes of {Q, dO}
  uint64_t* q_empty = q_full + NS;      // [NS] step's dV and dK products complete
  uint64_t* st_full = q_empty + NS;     // [2] S^T and dP^T in TMEM buffer (two issuers)
  uint64_t* pt_full = st_full + 2;      // [2] P^T, dS^T in that buffer (8 warps)
  uint64_t* buf_free = pt_full + 2;     // [2] dV, dK of the buffer's step complete: it may take step i+2
  uint64_t* dkv_done = buf_free + 2;    // every product complete
  uint64_t* drain = dkv_done + 1;       // [3] one per issuer
  uint32_t* tmem_slot = (uint32_t*)(drain + 3);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntk = (sh.T + 127) >> 7;
  int kt, bg;
  at_cta_order((int)blockIdx.x, sh.B * sh.Hkv, ntk, kt, bg);   // key tile 0 sees the most queries: first
  const int b = bg / sh.Hkv, g = bg - b * sh.Hkv;
  const int nq = (sh.T + 63) >> 6;
  const int per = nq - 2 * kt;                        // 64-query tiles from the diagonal on
  const int n = sh.G * per;
  const int row0 = b * sh.T;
  auto step_q0 = [&](int i) { return (2 * kt + i % per) * 64; };
  auto step_h = [&](int i) { return g * sh.G + i / per; };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NS; ++s) { mbar_init(&q_full[s], 1); mbar_init(&q_empty[s], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&st_full[i], 2); mbar_init(&pt_full[i], 8); mbar_init(&buf_free[i], 1); }
    mbar_init(dkv_done, 1);
    for (int r = 0; r < 3; ++r) mbar_init(&drain[r], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_kv);
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S^T[2] cols 0,64; dP^T[2] 128,192; dV 256..; dK 256+HD.  Warp half hf reads
  // columns [32 hf, 32 hf + 32) of S^T[buf] and of dP^T[buf] and overwrites the
  // first 16 of them with P^T and dS^T respectively, bf16 pairs of its 32
  // queries.  Three issuers: warp 1 writes S^T, warp 2 dP^T, and warp 3 reads
  // P^T and dS^T back (dV += P^T dO, dK += dS^T Q).  A buffer is written again
  // (S^T, dP^T of step i+2) only after buf_free signals that warp 3's products
  // of step i completed, and those were issued after the softmax warps had
  // read the buffer and written P^T, dS^T into it.
  const uint32_t tbase = *tmem_slot;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(kv_full, 2 * L::KT);
    for (int c = 0; c < HD / 64; ++c) {
      tma_load_2d(smem + L::OFF_K + c * CHUNK128, &tm_kv, kv_full, (sh.H + g) * HD + 64 * c, row0 + kt * 128);
      tma_load_2d(smem + L::OFF_V + c * CHUNK128, &tm_kv, kv_full, (sh.H + sh.Hkv + g) * HD + 64 * c,
                  row0 + kt * 128);
    }
    int issued = 0;
    for (int i = 0; i < n && !*abort_flag; ++i) {
      const int s = i % NS;
      if (!at_wait(&q_empty[s], ((i / NS) & 1) ^ 1, sh, abort_flag)) break;
      const int h = step_h(i), q0 = step_q0(i);
      uint8_t* dst = smem + L::OFF_QS + s * 2 * L::QT;
      mbar_arrive_expect_tx(&q_full[s], 2 * L::QT);
      for (int c = 0; c < HD / 64; ++c) {
        tma_load_2d(dst + c * CHUNK64, &tm_q, &q_full[s], h * HD + 64 * c, row0 + q0);
        tma_load_2d(dst + L::QT + c * CHUNK64, &tm_do, &q_full[s], h * HD + 64 * c, row0 + q0);
      }
      ++issued;
    }
    mbar_wait_bounded(kv_full, 0, NC_DRAIN_NS);
    for (int s = 0; s < NS; ++s) {
      const int uses = issued / NS + ((issued % NS) > s ? 1 : 0);
      if (uses > 0) mbar_wait_bounded(&q_full[s], (uses - 1) & 1, NC_DRAIN_NS);
    }
  } else if ((warp == 1 || warp == 2) && lane == 0) {
    // ---------------- two product issuers (a single thread issues about one MMA per
    // ~100 cycles, so each chain has its own): warp 1 S^T = K Q^T, warp 2
    // dP^T = V dO^T, into buffer i & 1, up to two steps ahead of the softmax
    const int role = warp - 1;
    const uint32_t id_s = at_idesc(64, 0);
    const uint32_t a_op = smem_u32(smem + (role ? L::OFF_V : L::OFF_K));
    const uint32_t sqs = smem_u32(smem + L::OFF_QS);
    bool ok = at_wait(kv_full, 0, sh, abort_flag);
    for (int i = 0; ok && i < n; ++i) {
      const int s = i % NS, buf = i & 1;
      if (!(ok = at_wait(&q_full[s], (i / NS) & 1, sh, abort_flag))) break;
      if (i >= 2 && !(ok = at_wait(&buf_free[buf], ((i - 2) >> 1) & 1, sh, abort_flag))) break;
      tc_fence_after();
      const uint32_t bop = sqs + s * 2 * L::QT + (role ? L::QT : 0u);   // Q (S^T) or dO (dP^T)
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk)
        tc_mma_f16(tbase + role * 128 + buf * 64, kdesc(a_op, kk, CHUNK128), kdesc(bop, kk, CHUNK64), id_s,
                   kk > 0 ? 1u : 0u);
      tc_commit(&st_full[buf]);
      if (*abort_flag) ok = false;
    }
    tc_commit(&drain[role]);
    mbar_wait_bounded(&drain[role], 0, NC_DRAIN_NS);
  } else if (warp == 3 && lane == 0) {
    // ---------------- the accumulating issuer: dV += P^T dO and dK += dS^T Q, A from TMEM
    const uint32_t id_kv = at_idesc(HD, 1);
    const uint32_t sqs = smem_u32(smem + L::OFF_QS);
    bool ok = true;
    for (int i = 0; ok && i < n; ++i) {
      const int s = i % NS, buf = i & 1;
      if (!(ok = at_wait(&pt_full[buf], (i >> 1) & 1, sh, abort_flag))) break;
      tc_fence_after();
      const uint32_t sq = sqs + s * 2 * L::QT;
#pragma unroll
      for (int role = 0; role < 2; ++role) {
        // P^T (in S^T's columns) or dS^T (in dP^T's); query slice kk at 32 (kk/2) + 8 (kk%2)
        const uint32_t pt = tbase + role * 128 + buf * 64;
        const uint32_t bop = sq + (role ? 0u : L::QT);    // dO (dV) or Q (dK), MN-major
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f16_ts(tbase + 256 + role * HD, pt + 32 * (kk >> 1) + 8 * (kk & 1), mndesc(bop, kk, CHUNK64),
                        id_kv, (i > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(&buf_free[buf]);
      tc_commit(&q_empty[s]);
      if (*abort_flag) ok = false;
    }
    if (ok) tc_commit(dkv_done);
    tc_commit(&drain[2]);
    mbar_wait_bounded(&drain[2], 0, NC_DRAIN_NS);
  } else if (warp >= 4) {
    const int quarter = warp & 3, hf = (warp - 4) >> 2;   // hf: query columns [32 hf, 32 hf + 32)
    const int r = quarter * 32 + lane;
    const int key = kt * 128 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // -lse * log2(e) and D of this warp's 32 queries: lane e fetches query e's
    // pair one step ahead (into registers), and the warp shares them through its
    // own 256-byte slot of shared memory (rows past the end get P = 0)
    float* ld = reinterpret_cast<float*>(smem + L::OFF_LD) + (warp - 4) * 64;
    auto fetch = [&](int i, float& l2, float& d) {
      const int q = step_q0(i) + 32 * hf + lane;
      const int64_t base = ((int64_t)b * sh.H + step_h(i)) * sh.T;
      l2 = q < sh.T ? __ldg(lse + base + q) * LOG2E : INFINITY;
      d = q < sh.T ? __ldg(Dv + base + q) : 0.f;
    };
    float nl = 0.f, nd = 0.f;
    if (n > 0) fetch(0, nl, nd);
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int buf = i & 1;
      if (!(ok = at_wait_warp(&st_full[buf], (i >> 1) & 1, sh, abort_flag))) break;
      tc_fence_after();
      uint32_t st[32], dp[32];
      tmem_ld_32x32b_x32(tbase + lane_off + buf * 64 + 32 * hf, st);
      tmem_ld_32x32b_x32(tbase + lane_off + 128 + buf * 64 + 32 * hf, dp);
      ld[lane] = -nl;
      ld[32 + lane] = nd;
      __syncwarp();
      if (i + 1 < n) fetch(i + 1, nl, nd);
      tmem_ld_wait();
      const int q0 = step_q0(i) + 32 * hf;
      const bool diag = step_q0(i) < kt * 128 + 128;
      const float4* ld4 = reinterpret_cast<const float4*>(ld);
      const float4* dd4 = reinterpret_cast<const float4*>(ld + 32);
      // two queries per FFMA2 / FADD2 / FMUL2 instruction
      const float2 sl2 = make_float2(sh.scale_log2, sh.scale_log2);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l4 = ld4[c4], d4 = dd4[c4];
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int c = 4 * c4 + e;
          const float2 nl2 = e ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
          const float2 dv2 = e ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
          const float2 a = fma2(make_float2(__uint_as_float(st[c]), __uint_as_float(st[c + 1])), sl2, nl2);
          float2 p = make_float2(ex2_approx(a.x), ex2_approx(a.y));
          if (diag) {
            if (q0 + c < key) p.x = 0.f;
            if (q0 + c + 1 < key) p.y = 0.f;
          }
          const float2 ds = mul2(p, sub2(make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), dv2));
          st[c] = __float_as_uint(p.x);
          st[c + 1] = __float_as_uint(p.y);
          dp[c] = __float_as_uint(ds.x);
          dp[c + 1] = __float_as_uint(ds.y);
        }
      }
      // P^T and dS^T as bf16 pairs into the S^T and dP^T columns this warp just read
#pragma unroll
      for (int c = 0; c < 16; ++c) st[c] = pack2(__uint_as_float(st[2 * c]), __uint_as_float(st[2 * c + 1]));
#pragma unroll
      for (int c = 0; c < 16; ++c) dp[c] = pack2(__uint_as_float(dp[2 * c]), __uint_as_float(dp[2 * c + 1]));
      tmem_st_32x32b_x16(tbase + lane_off + buf * 64 + 32 * hf, st);
      tmem_st_32x32b_x16(tbase + lane_off + 128 + buf * 64 + 32 * hf, dp);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();   // also: every lane has read the slot before the next step overwrites it
      if (lane == 0) mbar_arrive(&pt_full[buf]);
    }
    const bool valid = key < sh.T;
    AtOutPre<HD> pre;
    at_out_prefetch<HD>(sh, hf, ok && valid, key, (int64_t)row0 + key, sh.H + g, pre);
    float am = 0.f;
    if (ok && at_wait_warp(dkv_done, 0, sh, abort_flag)) {
      tc_fence_after();
      if constexpr (HD == 128) {
        // dV, then dK (carries 1/sqrt(hd)), staged in the Q / dO stages, free
        // once every product has completed; a fused dK leaves through the k-norm
        // and rotation backward with per-thread stores
        const int w8 = hf * 4 + quarter;
        at_out_box128(tbase + lane_off + 256, hf, 1.f, smem + L::OFF_QS + w8 * 4096, &tm_out,
                      (sh.H + sh.Hkv + g) * HD + hf * 64, kt * 128 + quarter * 32, b, sh.T, am, AMAX);
        if (!sh.rope_tab)
          at_out_box128(tbase + lane_off + 256 + HD, hf, sh.scale, smem + L::OFF_QS + 32768 + w8 * 4096, &tm_out,
                        (sh.H + g) * HD + hf * 64, kt * 128 + quarter * 32, b, sh.T, am, AMAX);
        else
          at_out_tile<HD, AMAX>(sh, tbase + lane_off + 256 + HD, smem + L::OFF_K, r, hf, valid, pre,
                          dqkv + (int64_t)(row0 + key) * sh.ld_qkv + (int64_t)(sh.H + g) * HD, am);
        if (lane == 0) bulk_wait_all();
      } else {
      bf16* dv = dqkv + (int64_t)(row0 + key) * sh.ld_qkv + (int64_t)(sh.H + sh.Hkv + g) * HD + hf * (HD / 2);
#pragma unroll 1
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tbase + lane_off + 256 + hf * (HD / 2) + 32 * c, v);
        tmem_ld_wait();
        if (valid) {
          if (AMAX) {
#pragma unroll
            for (int e = 0; e < 32; ++e) am = fmaxf(am, fabsf(__uint_as_float(v[e])));
          }
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack2(__uint_as_float(v[e]), __uint_as_float(v[e + 1]));
            w.y = pack2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
            w.z = pack2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
            w.w = pack2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
            *reinterpret_cast<uint4*>(dv + 32 * c + e) = w;
          }
        }
      }
      // dK (carries 1/sqrt(hd)), through the k-norm and rotation backward when fused
      at_out_tile<HD, AMAX>(sh, tbase + lane_off + 256 + HD, smem + L::OFF_K, r, hf, valid, pre,
                      dqkv + (int64_t)(row0 + key) * sh.ld_qkv + (int64_t)(sh.H + g) * HD, am);
      }
      if (AMAX) at_amax_commit(sh, am);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 512);
}

// D = rowsum(dO * O) per (row, head), fp32 [B, H, T].  One warp per row reads
// O and dO in 16-byte pieces (HD / 8 per head, held by a group of as many
// consecutive lanes), and each group reduces its head's sum.
template <int HD>
__global__ void k_attn_rowdot(int64_t rows, int H, int T_, int64_t ld_o, const bf16* __restrict__ o,
                              const bf16* __restrict__ dout, float* __restrict__ Dv) {
  constexpr int CPH = HD / 8;   // 16-byte pieces per head (divides 32)
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int nchunk = H * CPH;
  const uint4* a = reinterpret_cast<const uint4*>(o + row * ld_o);
  const uint4* c = reinterpret_cast<const uint4*>(dout + row * ld_o);
  const int64_t b = row / T_;
  const int t = (int)(row % T_);
  for (int c0 = 0; c0 < nchunk; c0 += 32) {
    const int ci = c0 + lane;
    float s = 0.f;
    if (ci < nchunk) {
      const uint4 x = a[ci], y = c[ci];
      const bf16* xe = reinterpret_cast<const bf16*>(&x);
      const bf16* ye = reinterpret_cast<const bf16*>(&y);
#pragma unroll
      for (int e = 0; e < 8; ++e) s = fmaf(__bfloat162float(xe[e]), __bfloat162float(ye[e]), s);
    }
#pragma unroll
    for (int off = CPH / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (ci < nchunk && (lane % CPH) == 0) Dv[(b * H + ci / CPH) * T_ + t] = s;
  }
}

bool at_shape(int B, int T, int H, int Hkv, int hd, int32_t* err, AtShape* sh) {
  if (B <= 0 || T <= 0 || H <= 0 || Hkv <= 0 || H % Hkv || (hd != 64 && hd != 128)) return false;
  if ((int64_t)B * T >= (1ll << 31) || (int64_t)B * H * ((T + 127) / 128) >= (1ll << 31)) return false;
  sh->B = B; sh->T = T; sh->H = H; sh->Hkv = Hkv; sh->G = H / Hkv;
  sh->ld_qkv = (int64_t)(H + 2 * Hkv) * hd;
  sh->ld_o = (int64_t)H * hd;
  sh->scale = 1.f / sqrtf((float)hd);
  sh->scale_log2 = LOG2E * sh->scale;
  sh->err = err;
  sh->wait_ns = g_tc_wait_ns;
  sh->rope_tab = nullptr;
  sh->rstd_qk = nullptr;
  sh->rope_pair_rows = 0;
  sh->amax = nullptr;
  return true;
}

bool aligned16(const void* p) { return (((uintptr_t)p) & 15) == 0; }

template <int HD>
nc_status attn_fwd_tc(const AtShape& sh, const bf16* qkv, bf16* o, float* lse, cudaStream_t st) {
  CUtensorMap tm, tm_o;
  if (!make_tmap_bf16_2d(&tm, qkv, sh.ld_qkv, (uint64_t)sh.B * sh.T, sh.ld_qkv, 64, 128) ||
      !make_tmap_bf16_3d(&tm_o, o, sh.ld_o, sh.T, sh.B, sh.ld_o, 64, 32))
    return NC_ERR_CUDA;
  static bool attr = false;
  if (!attr) {
    NC_CUDA_TRY(cudaFuncSetAttribute(k_attn_fwd_tc<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)FwdSmem<HD>::BYTES));
    NC_CUDA_TRY(cudaFuncSetAttribute(k_attn_fwd_tc<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)FwdSmem<HD>::BYTES));
    attr = true;
  }
  const unsigned grid = (unsigned)((sh.T + 255) / 256) * (unsigned)(sh.B * sh.H);
  // the instantiation with the output maximum only when it is asked for
  if (sh.amax) k_attn_fwd_tc<HD, true><<<grid, AT_THREADS, FwdSmem<HD>::BYTES, st>>>(tm, tm_o, sh, o, lse);
  else k_attn_fwd_tc<HD, false><<<grid, AT_THREADS, FwdSmem<HD>::BYTES, st>>>(tm, tm_o, sh, o, lse);
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

template <int HD>
nc_status attn_bwd_tc(const AtShape& sh, const bf16* qkv, const bf16* o, const float* lse, const bf16* dout,
                      bf16* dqkv, float* Dv, cudaStream_t st) {
  const int64_t rows = (int64_t)sh.B * sh.T;
  k_attn_rowdot<HD><<<cdiv(rows, 8), 256, 0, st>>>(rows, sh.H, sh.T, sh.ld_o, o, dout, Dv);
  NC_CUDA_TRY(cudaGetLastError());
  CUtensorMap tm_qkv128, tm_qkv64, tm_do128, tm_do64, tm_out;
  if (!make_tmap_bf16_3d(&tm_out, dqkv, sh.ld_qkv, sh.T, sh.B, sh.ld_qkv, 64, 32) ||
      !make_tmap_bf16_2d(&tm_qkv128, qkv, sh.ld_qkv, rows, sh.ld_qkv, 64, 128) ||
      !make_tmap_bf16_2d(&tm_qkv64, qkv, sh.ld_qkv, rows, sh.ld_qkv, 64, 64) ||
      !make_tmap_bf16_2d(&tm_do128, dout, sh.ld_o, rows, sh.ld_o, 64, 128) ||
      !make_tmap_bf16_2d(&tm_do64, dout, sh.ld_o, rows, sh.ld_o, 64, 64))
    return NC_ERR_CUDA;
  static bool attr = false;
  if (!attr) {
    NC_CUDA_TRY(cudaFuncSetAttribute(k_attn_bwd_dq_tc<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)DqSmem<HD>::BYTES));
    NC_CUDA_TRY(cudaFuncSetAttribute(k_attn_bwd_dkv_tc<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)DkvSmem<HD>::BYTES));
    NC_CUDA_TRY(cudaFuncSetAttribute(k_attn_bwd_dq_tc<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)DqSmem<HD>::BYTES));
    NC_CUDA_TRY(cudaFuncSetAttribute(k_attn_bwd_dkv_tc<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)DkvSmem<HD>::BYTES));
    attr = true;
  }
  const unsigned nt = (unsigned)((sh.T + 127) / 128);
  const dim3 gq(nt * (unsigned)(sh.B * sh.H)), gkv(nt * (unsigned)(sh.B * sh.Hkv));
  if (sh.amax) {   // the instantiations with the output maximum only when it is asked for
    k_attn_bwd_dq_tc<HD, true><<<gq, AT_THREADS, DqSmem<HD>::BYTES, st>>>(tm_qkv128, tm_do128, tm_out, sh, lse, Dv,
                                                                          dqkv);
    NC_CUDA_TRY(cudaGetLastError());
    k_attn_bwd_dkv_tc<HD, true><<<gkv, AT_THREADS, DkvSmem<HD>::BYTES, st>>>(tm_qkv128, tm_qkv64, tm_do64, tm_out,
                                                                             sh, lse, Dv, dqkv);
  } else {
    k_attn_bwd_dq_tc<HD, false><<<gq, AT_THREADS, DqSmem<HD>::BYTES, st>>>(tm_qkv128, tm_do128, tm_out, sh, lse,
                                                                           Dv, dqkv);
    NC_CUDA_TRY(cudaGetLastError());
    k_attn_bwd_dkv_tc<HD, false><<<gkv, AT_THREADS, DkvSmem<HD>::BYTES, st>>>(tm_qkv128, tm_qkv64, tm_do64, tm_out,
                                                                              sh, lse, Dv, dqkv);
  }
  return cudaGetLastError() == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

}  // namespace

nc_status launch_attn_fwd_tc(int B, int T, int H, int Hkv, int hd, const bf16* qkv, bf16* o, float* lse,
                             int32_t* err, cudaStream_t st, unsigned* amax) {
  AtShape sh;
  if (!at_shape(B, T, H, Hkv, hd, err, &sh)) return NC_ERR_ARG;
  sh.amax = amax;
  if (!aligned16(qkv) || !aligned16(o)) return NC_ERR_ARG;
  return hd == 128 ? attn_fwd_tc<128>(sh, qkv, o, lse, st) : attn_fwd_tc<64>(sh, qkv, o, lse, st);
}

nc_status launch_attn_bwd_tc(int B, int T, int H, int Hkv, int hd, const bf16* qkv, const bf16* o, const float* lse,
                             const bf16* dout, bf16* dqkv, float* Dv, const float* rstd_qk, const float* rope_tab,
                             int rope_pair_rows, int32_t* err, cudaStream_t st, unsigned* amax) {
  AtShape sh;
  if (!at_shape(B, T, H, Hkv, hd, err, &sh)) return NC_ERR_ARG;
  sh.amax = amax;
  if ((rstd_qk == nullptr) != (rope_tab == nullptr) || (rope_tab && !aligned16(rope_tab))) return NC_ERR_ARG;
  if (rope_pair_rows < 0 || (rope_pair_rows > 0 && (rope_pair_rows < T || hd % 4))) return NC_ERR_ARG;
  sh.rstd_qk = rstd_qk;
  sh.rope_tab = rope_tab;
  sh.rope_pair_rows = rope_pair_rows;
  if (!aligned16(qkv) || !aligned16(o) || !aligned16(dout) || !aligned16(dqkv)) return NC_ERR_ARG;
  return hd == 128 ? attn_bwd_tc<128>(sh, qkv, o, lse, dout, dqkv, Dv, st)
                   : attn_bwd_tc<64>(sh, qkv, o, lse, dout, dqkv, Dv, st);
}
