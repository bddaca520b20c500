// Launch functions of every kernel of the step (host side, enqueue only).
#pragma once
#include <algorithm>
#include "nc_common.cuh"
#include <cuda.h>

nc_status launch_init_normal(float* out, int64_t count, uint64_t seed, int tensor_index, float std,
                             cudaStream_t st);
nc_status launch_cast_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t st);
// tab [T][hd/2][2] and/or pairs [hd/4][T][4] (pair-major copy); either may be NULL.
nc_status launch_rope_table(int T, int hd, float base, float* tab, float* pairs, cudaStream_t st);

// amax_bits (optional, pre-zeroed): atomic maximum of |y| as stored, float bits (8-bit quantiser input).
nc_status launch_rmsnorm_fwd(int dtype, int64_t rows, int C, const float* x, void* y, float* rstd,
                             float eps, cudaStream_t st, unsigned* amax_bits = nullptr);
// amax_bits (optional, with dx_act): atomic maximum of |dx_act| as stored, float bits.
nc_status launch_rmsnorm_bwd(int dtype, int64_t rows, int C, const float* dy, const void* y,
                             const float* rstd, float* dx, void* dx_act, cudaStream_t st,
                             unsigned* amax_bits = nullptr);
// pos0 (device, may be NULL): positions are *pos0 + row % T instead of row % T.
// kc, vc (both or neither): also write every row's rotated, normalised k heads
// and its v heads into a [B][Hkv][max_len][hd] cache at the row's position.
nc_status launch_rope_qknorm_fwd(int dtype, int B, int T, int H, int Hkv, int hd, void* qkv,
                                 float* rstd, const float* tab, float eps, cudaStream_t st,
                                 const int32_t* pos0 = nullptr, void* kc = nullptr, void* vc = nullptr,
                                 int max_len = 0);
nc_status launch_rope_qknorm_bwd(int dtype, int B, int T, int H, int Hkv, int hd, void* dqkv,
                                 const void* qkv, const float* rstd, const float* tab,
                                 cudaStream_t st);

// rstd != NULL: the variant with a norm after the embedding (x = e * rstd, rstd saved per row).
nc_status launch_embed_fwd(int dtype, int64_t n, int C, int V, const int32_t* tokens,
                           const float* wte, float* x, int32_t* err, cudaStream_t st, float* rstd = nullptr,
                           float eps = 0.f);
// In place on dx [n, C]: the backward of that norm, its output recomputed from wte.
nc_status launch_embed_norm_bwd(int dtype, int64_t n, int C, int V, const int32_t* tokens, const float* wte,
                                const float* rstd, float* dx, cudaStream_t st);
size_t embed_bwd_scratch_bytes(int64_t n, int C, int V);
// accumulate != 0: dwte += the scatter (rows of absent ids untouched); else dwte = it.
// Positions whose id lies outside [0, V) add to no row and set the token bit of
// *err (when err is not NULL).
nc_status launch_embed_bwd(int64_t n, int C, int V, const int32_t* tokens, const float* dx,
                           float* dwte, void* scratch, cudaStream_t st, int accumulate = 0,
                           int32_t* err = nullptr);
// softcap > 0: the logits enter as softcap * tanh(z / softcap) (dz is taken with respect to z).
nc_status launch_cross_entropy(int dtype, int64_t rows, int V, void* z, int64_t ldz,
                               const int32_t* targets, float* row_loss, float scale, int32_t* err,
                               cudaStream_t st, float softcap = 0.f);
// z <- cap * tanh(z / cap) on n fp32 logits (no-op for cap <= 0).
nc_status launch_softcap_f32(int64_t n, float* z, float cap, cudaStream_t st);
nc_status launch_mean(int64_t n, const float* x, float* out, cudaStream_t st);

nc_status launch_gemm_simt(int dtype, int M, int N, int K, const void* A, int64_t lda, int a_kmajor,
                           const void* B, int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd,
                           void* aux, int64_t ldaux, cudaStream_t st);
// tcgen05 tensor-core GEMM (bf16 operands, fp32 accumulation in TMEM).
// ws (optional, 16-byte aligned): stream-K partial tiles for fp32-output GEMMs
// with few output tiles; gemm_tc_workspace_bytes() is enough for any shape.
nc_status launch_gemm_tc(int M, int N, int K, const bf16* A, int64_t lda, int a_kmajor,
                         const bf16* B, int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd,
                         void* aux, int64_t ldaux, int32_t* err, void* ws, size_t ws_bytes, cudaStream_t st);
size_t gemm_tc_workspace_bytes();
// Internal epilogue of the fused q/k/v projection (not part of the public enum).
#define NC_EP_QKV_ROPE 100
// qkv[M, N] = A[M, K] Wqkv[N, K]^T in bf16 with RoPE and the per-head RMSNorm
// of the first nh heads (q and k) applied in the epilogue (rstd [M, nh] fp32);
// the remaining heads (v) are stored as computed.  Rows are positions m % T.
// NC_ERR_UNSUPPORTED for N <= 128; hd 64 or 128.
// tab: [T][hd/2][2] (pair_rows = 0) or pair-major [hd/4][pair_rows][4] with
// pair_rows >= T (the coalesced layout the epilogue prefers).
// `batch` products of the same shape, D_b = A_b B_b^T in bf16 (NC_EP_STORE),
// operands as for launch_gemm_tc; problem b's rows start b * a_bro (A),
// b * b_bro (B) and b * d_bro (D) rows after the first problem's, where a
// row is the operand's outer dimension (M or N for K-major, K for MN-major).
// Needs a_bro and b_bro at least the operand's rows, d_bro at least M rounded
// up to 256 (output tiles past M land in that padding), and K a multiple of
// 128 when an operand is MN-major.  The buffers hold batch * bro rows each.
nc_status launch_gemm_tc_batched(int batch, int M, int N, int K, const bf16* A, int64_t lda, int a_kmajor,
                                 int64_t a_bro, const bf16* B, int64_t ldb, int b_kmajor, int64_t b_bro, bf16* D,
                                 int64_t ldd, int64_t d_bro, int32_t* err, cudaStream_t st);
nc_status launch_gemm_tc_qkv_rope(int M, int N, int K, const bf16* A, int64_t lda, const bf16* Wqkv, int64_t ldb,
                                  bf16* qkv, int64_t ldd, int T, int nh, int hd, const float* tab, int pair_rows,
                                  float* rstd, float eps, int32_t* err, cudaStream_t st);

// E4M3 GEMM on the tensor cores (kind::f8f6f4): D[M, N] = (*scale_a) (*scale_b)
// A[M, K] B[N, K]^T, operands K-major bytes (lda, ldb multiples of 16, bases
// 16-byte aligned), fp32 accumulation, D bf16 (out_f32 = 0) or fp32.
nc_status launch_gemm_fp8(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                          const float* scale_a, const float* scale_b, int out_f32, void* D, int64_t ldd,
                          int32_t* err, cudaStream_t st);
// The 8-bit GEMM through a step epilogue: NC_EP_STORE, NC_EP_STORE_F32,
// NC_EP_ACCUM_F32, NC_EP_RELU2_SQ, NC_EP_RELU2_SQ_BWD (with aux, bf16
// relu(u)^2, row pitch ldaux), or NC_EP_QKV_ROPE (then T, nh, hd, tab,
// pair_rows, rstd and eps as for launch_gemm_tc_qkv_rope; ignored otherwise).
// amax (bf16 outputs but QKV_ROPE): atomic maximum of |D| as stored, as float
// bits, for the per-tensor quantiser of D.  ws (fp32 outputs on CTA pairs): a
// split-K workspace of ws_bytes, as for launch_gemm_tc.
nc_status launch_gemm_fp8_ep(int M, int N, int K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                             const float* scale_a, const float* scale_b, int ep, void* D, int64_t ldd, int T, int nh,
                             int hd, const float* tab, int pair_rows, float* rstd, float eps, int32_t* err,
                             cudaStream_t st, const void* aux = nullptr, int64_t ldaux = 0,
                             unsigned* amax = nullptr, void* ws = nullptr, size_t ws_bytes = 0);
// Per-tensor E4M3 quantisation of n fp32 / bf16 values: stats (device, 3
// floats) gets {amax, scale, scale_inv}; y the codes.
nc_status launch_quantize_fp8(int dtype, const void* x, int64_t n, uint8_t* y, float* stats, cudaStream_t st);
// The step's 8-bit cast.  stats = {amax bits, scale, scale_inv}, stats[0]
// holding the maximum |x| its producer took (as float bits): scale = fl32(448
// / amax) (1 if not finite and positive), formed by every block; the codes of
// fl32(x * scale) of a [rows][cols] bf16 tensor go to y [rows][cols] (equal
// to launch_quantize_fp8's) and transposed into yt [cols][ldt] (ldt >= rows, a
// multiple of 16): the codes of a product that contracts over the rows;
// stats[1], stats[2] are written.
nc_status launch_fp8_cast_dual(const void* x, int rows, int cols, float* stats, uint8_t* y, uint8_t* yt, int64_t ldt,
                               cudaStream_t st);

nc_status launch_attn_fwd_simt(int dtype, int B, int T, int H, int Hkv, int hd, const void* qkv, void* o,
                               float* lse, cudaStream_t st);
nc_status launch_attn_bwd_simt(int dtype, int B, int T, int H, int Hkv, int hd, const void* qkv,
                               const void* o, const float* lse, const void* dout, void* dqkv, float* Dv,
                               cudaStream_t st);
// bf16 causal GQA flash attention on tcgen05 tensor cores (head_dim 64 or 128).
// err (device int32, may be NULL) receives NC_DEVERR_TIMEOUT if a bounded wait expires.
nc_status launch_attn_fwd_tc(int B, int T, int H, int Hkv, int hd, const bf16* qkv, bf16* o, float* lse,
                             int32_t* err, cudaStream_t st,
                             unsigned* amax = nullptr);
// With rstd_qk and rope_tab (both or neither), dq and dk are returned through the
// per-head RMSNorm backward and the transposed rotation (the RoPE + QK-norm
// backward fused into the output epilogue).  rope_tab is [T][hd/2][2]
// (rope_pair_rows = 0) or pair-major [hd/4][rope_pair_rows][4] (rope_pair_rows >= T).
// amax (both directions, may be NULL): atomic maximum of |output| as stored (O;
// dq, dk and dv), as float bits, for the per-tensor quantiser of that output.
nc_status launch_attn_bwd_tc(int B, int T, int H, int Hkv, int hd, const bf16* qkv, const bf16* o, const float* lse,
                             const bf16* dout, bf16* dqkv, float* Dv, const float* rstd_qk, const float* rope_tab,
                             int rope_pair_rows, int32_t* err, cudaStream_t st,
                             unsigned* amax = nullptr);

// 2D bf16 TMA descriptor over a row-major [outer][inner] matrix with leading
// dimension ld (elements), box {box_inner, box_outer}, 128-byte swizzle.
bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, int64_t ld,
                       uint32_t box_inner, uint32_t box_outer);
// 3D bf16 TMA descriptor viewing a [d2*d1, ld] matrix as [d2][d1][inner], box
// {box_inner, box_mid, 1}, 128-byte swizzle; stores are clipped at d1.
bool make_tmap_bf16_3d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t d1, uint64_t d2, int64_t ld,
                       uint32_t box_inner, uint32_t box_mid);

// ---------------------------------------------------------------- optimizer (k_optim.cu)
extern int g_num_sms;
// The weight matrices one Muon launch covers, passed by value as a kernel
// parameter.  Block b works on chunk b - chunk0[t] of tensor t, where
// chunk0[t] <= b < chunk0[t + 1]; each chunk is OPT_CHUNK elements.
#define NC_OPT_MAXT 384
#define OPT_CHUNK 16384
struct OptTensors {
  int32_t n;
  int32_t chunk0[NC_OPT_MAXT + 1];
  int64_t off[NC_OPT_MAXT];    // element offset in the packed parameter / gradient vectors
  int64_t soff[NC_OPT_MAXT];   // element offset in the optimizer's state buffers
  int64_t len[NC_OPT_MAXT];    // elements
  float* norm;                 // device [n]: ||U||_F per tensor (written by launch_muon_momentum)
};
// Tensors whose 8-bit codes are transposed for the backward: tensor t is
// [rows[t]][cols[t]] bytes at offset off[t]; tile0 counts 64 x 64 tiles.
struct Fp8Transposes {
  int32_t n;
  int32_t tile0[NC_OPT_MAXT + 1];
  int64_t off[NC_OPT_MAXT];
  int32_t rows[NC_OPT_MAXT], cols[NC_OPT_MAXT];
};
nc_status launch_fp8_transpose_multi(const Fp8Transposes& tt, const uint8_t* src, uint8_t* dst, cudaStream_t st);
// Every tensor t of tl at once (fp32 master + tl.off[t], tl.len[t] elements):
// stats + 4 t as above (stats[4 t] zeroed beforehand), codes at y + tl.soff[t].
nc_status launch_fp8_quantize_multi(const OptTensors& tl, const float* master, float* stats, uint8_t* y,
                                    cudaStream_t st);
// M <- mu M + G; U = nesterov ? G + mu M : M; then tl.norm[t] = ||U_t||_F.
// partial: one float per chunk.
nc_status launch_muon_momentum(const OptTensors& tl, const float* G, float* M, float* U, float mu, int nesterov,
                               float* partial, cudaStream_t st);
// X = U / (norm + eps) in the compute dtype.
nc_status launch_ns_init(int dtype, const OptTensors& tl, const float* U, float eps, void* X, cudaStream_t st);
// `steps` Newton-Schulz iterations on X0[rows, cols]; the result is left in ping0
// or ping1 (*out).  A and A2 hold min(rows, cols)^2 elements.
nc_status newton_schulz_run(int dtype, int rows, int cols, int steps, const void* x0, void* ping0, void* ping1,
                            void* A, void* A2, const void** out, int32_t* err, void* gemm_ws, size_t gemm_ws_bytes,
                            cudaStream_t st);
// newton_schulz_run on `batch` bf16 matrices of one shape at once: X_b starts
// b * xr rows into ping0, the n x n products b * nr rows into A and A2 (xr,
// nr at least rows and n rounded up to 256; rows a multiple of 128).
nc_status newton_schulz_batched(int batch, int rows, int cols, int steps, void* ping0, void* ping1, int64_t xr,
                                void* A, void* A2, int64_t nr, const void** out, int32_t* err, cudaStream_t st);
// W <- W - lr X (n elements, X in the compute dtype).
nc_status launch_muon_apply(int dtype, int64_t n, float* W, const void* X, float lr, cudaStream_t st);
// W <- W - lr X for every tensor t of tl at once: W = master + tl.off[t], X (compute
// dtype) at X + tl.soff[t] elements, tl.len[t] elements each.
nc_status launch_muon_apply_multi(int dtype, const OptTensors& tl, float* W, const void* X, float lr, cudaStream_t st);
nc_status launch_cast_out(int dtype, int64_t n, const void* X, float* out, cudaStream_t st);
// One bias-corrected AdamW step (t >= 1) with decoupled weight decay.
nc_status launch_adamw(int64_t n, float* W, const float* G, float* m, float* v, float lr, float b1, float b2,
                       float eps, float wd, int64_t t, cudaStream_t st);

// ---------------------------------------------------------------- KV-cache decoding (k_decode.cu)
// Row r of qkv[rows, ld] = sequence r / T, position t0 + r % T: its k and v heads
// go to kc / vc ([B][Hkv][max_len][hd], compute dtype).
// t0_dev (device, may be NULL) replaces t0.
nc_status launch_kv_store(int dtype, int64_t rows, int T, int t0, int H, int Hkv, int hd, const void* qkv, int64_t ld,
                          void* kc, void* vc, int max_len, cudaStream_t st, const int32_t* t0_dev = nullptr);
// o[b, h*hd..] = softmax(q_bh . K[b, h/G, 0..len) / sqrt(hd)) V for the single
// query row b of qkv (ld), H/Hkv in {1, 2, 3, 4, 8}, hd 64 or 128.  part holds
// decode_part_floats(B, H, hd, max_len) floats.
// len_dev (device, may be NULL): the keys are 0..*len_dev (inclusive) and the
// grid covers max_len (for a graph that replays at growing lengths).
// rope_tab (may be NULL; [T][hd/2][2] cos/sin, 16-byte aligned): qkv holds the
// raw projection of position len - 1; the kernel applies RoPE + the per-head
// RMSNorm (eps) to q and k itself and appends k and v to the cache.
nc_status launch_decode_attn(int dtype, int B, int H, int Hkv, int hd, int len, const void* qkv, int64_t ld,
                             void* kc, void* vc, int max_len, float* part, void* o, int64_t ldo, cudaStream_t st,
                             const int32_t* len_dev = nullptr, const float* rope_tab = nullptr, float eps = 0.f);
// *p = v (add = false) or *p += v, on the device.
nc_status launch_set_i32(int32_t* p, int32_t v, bool add, cudaStream_t st);
size_t decode_part_floats(int B, int H, int hd, int max_len);
// One-time launch attributes of the decode kernels (call outside stream capture).
nc_status decode_kernels_prepare();
// D[m, n] (op)= sum_k A[m, k] W[n, k] for 1 <= M <= SKINNY_MAX_M rows on the
// CUDA cores (memory-bound on W); K, lda, ldw multiples of 8, 16-byte aligned
// A and W; ep one of NC_EP_STORE, NC_EP_STORE_F32, NC_EP_ACCUM_F32, NC_EP_RELU2_SQ.
#define SKINNY_MAX_M 32
nc_status launch_gemm_skinny(int dtype, int M, int N, int K, const void* A, int64_t lda, const void* W, int64_t ldw,
                             int ep, void* D, int64_t ldd, cudaStream_t st);
// The same with A = act(rmsnorm(x)) of the fp32 rows x (ldx a multiple of 4),
// the normalisation done in the kernel; 1 <= M <= 8.
nc_status launch_gemm_skinny_norm(int dtype, int M, int N, int K, const float* x, int64_t ldx, const void* W,
                                  int64_t ldw, int ep, void* D, int64_t ldd, float eps, cudaStream_t st);
