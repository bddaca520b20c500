// The C ABI of libnc: model lifetime, parameter layout, the forward+backward
// training step and the kernel-level entry points.  See include/nc.h.
//
// One step enqueues, on the caller's stream: the weight cast, the embedding
// gather, per layer {RMSNorm, QKV GEMM, RoPE + QK-norm, attention, output
// projection GEMM + residual, RMSNorm, fc GEMM + relu^2, c_proj GEMM +
// residual}, the final RMSNorm, the chunked lm_head + cross-entropy (forward
// and backward per chunk), then per layer in reverse the matching backward
// kernels, and the embedding scatter.  The only synchronisation is the final
// read of the loss and the device error flag.
#include <algorithm>
#include <cmath>
#include <cfloat>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "nc_kernels.cuh"

extern uint64_t g_tc_wait_ns;

struct ParamTensor {
  std::string name;
  int64_t rows, cols, off;
};

struct nc_model {
  nc_config cfg;
  int L, C, H, Hkv, hd, F, V, Tmax, Bmax, qkvw, dtype;
  int64_t Nmax, P;
  size_t act;                        // bytes per compute-dtype element
  std::vector<ParamTensor> layout;
  std::vector<void*> allocs;
  float* master = nullptr;           // fp32 [P]
  void* wact = nullptr;              // compute-dtype weights [P] (== master in fp32 mode)
  float* rope_tab = nullptr;         // [Tmax, hd/2, 2]
  float* rope_pairs = nullptr;       // the same, pair-major [hd/4, Tmax, 4] (bf16 QKV GEMM epilogue)
  float softcap = 0.f;               // logit soft-cap c (0: off)
  bool emb_norm = false;             // RMSNorm after the embedding lookup
  float* rstd_e = nullptr;           // [Nmax] its per-row rstd (emb_norm only)
  bool fp8 = false;                  // the blocks' forward and dX linears on E4M3 operands
  uint8_t* q8a = nullptr;            // E4M3 codes of a linear layer's input [Nmax, max(C, F)]
  uint8_t* q8w = nullptr;            // E4M3 codes of every block weight operand, quantised once per step
  uint8_t* q8wT = nullptr;           // the same codes transposed ([in][out]): B operands of the dX products
  uint8_t* q8xT = nullptr;           // per layer, the four linears' input codes transposed [in][q8np]: dW operands
  uint8_t* q8dyT = nullptr;          // one output gradient's codes transposed [out][q8np]
  int64_t q8np = 0;                  // row pitch of the transposed codes: the token count rounded up to 16
  float* q8s = nullptr;              // per layer and linear {amax bits, scale, scale_inv, -}: inputs [L][4],
                                     // weights [L][4], output gradients dY [L][4]
  OptTensors* q8tl = nullptr;        // the 4 L weight operands (fp32 master offset, code offset, length)
  Fp8Transposes* q8tt = nullptr;     // the same operands as [out][in] byte matrices, for the transpose
  int32_t* err = nullptr;            // device error flag
  float* result = nullptr;           // device: [0] loss, [1] error flag copy
  float* result_host = nullptr;      // pinned host copy
  // forward activations (per layer, strides sized for Nmax tokens)
  float* x = nullptr;                // residual stream [N, C]
  uint8_t *xn1, *xn2, *qkv, *o, *h;      // h = relu(u)^2 (relu(u) = sqrt(h) in the backward)
  float *rstd1, *rstd2, *rstdqk, *lse;
  void* xf = nullptr;
  float* rstd_f = nullptr;
  void* logits = nullptr;            // [Nc, V] chunk of logits / dlogits
  int64_t chunk_rows = 0;
  float* rowloss = nullptr;
  // backward scratch
  float* dx = nullptr;
  void* dx_act = nullptr;
  void* du = nullptr;
  float* dxn = nullptr;
  void* dout = nullptr;
  void* dqkv = nullptr;
  float* Dv = nullptr;
  void* emb_scratch = nullptr;
  void* gemm_ws = nullptr;           // stream-K partial tiles
  size_t gemm_ws_bytes = 0;
  int32_t *tok_dev = nullptr, *tgt_dev = nullptr;
  int64_t launches = 0;
  // optimizer state, allocated and zeroed by the first nc_optimizer_step
  bool opt_ready = false;
  int64_t opt_t = 0;                 // optimizer steps taken
  OptTensors* opt_tl = nullptr;      // the Muon matrices (host copy of the kernel parameter)
  float *opt_mom = nullptr, *opt_u = nullptr, *opt_partial = nullptr, *opt_norm = nullptr;
  void* opt_x0 = nullptr;
  float *adam_m = nullptr, *adam_v = nullptr;   // [wte | lm_head] moments
  // The matrices' Newton-Schulz iterations are independent: they run on
  // NC_OPT_STREAMS side streams (fork / join through events on the caller's
  // stream), each with its own ping-pong and A buffers; matrices are assigned
  // largest first to the least-loaded stream.
  static constexpr int NC_OPT_STREAMS = 4;
  cudaStream_t opt_st[NC_OPT_STREAMS] = {};
  cudaEvent_t opt_fork = nullptr, opt_join[NC_OPT_STREAMS] = {};
  void *opt_ping0[NC_OPT_STREAMS] = {}, *opt_ping1[NC_OPT_STREAMS] = {};
  void *opt_a[NC_OPT_STREAMS] = {}, *opt_a2[NC_OPT_STREAMS] = {};
  std::vector<int> opt_order, opt_lane;    // matrices by decreasing work, and each one's stream
  // bf16 with every matrix's rows a multiple of 128: the matrices of one shape
  // iterate together (batched GEMMs on the caller's stream) instead
  struct NsGroup {
    int rows, cols;
    int64_t xr, nr;                        // row strides of the stacked X and n x n buffers
    std::vector<int> members;              // optimizer tensor indices
    OptTensors* apply = nullptr;           // the members' master offsets and stacked result offsets
  };
  std::vector<NsGroup> ns_groups;
  void *nsb_ping0 = nullptr, *nsb_ping1 = nullptr, *nsb_a = nullptr, *nsb_a2 = nullptr;
  // key/value cache for incremental decoding (nc_kv_cache_create)
  void *kcache = nullptr, *vcache = nullptr;   // per layer [kv_b][Hkv][kv_max][hd], compute dtype
  float* dec_part = nullptr;                   // decode-attention partials
  int kv_b = 0, kv_max = 0;                    // capacity
  int kv_batch = 0, kv_len = 0;                // sequences and positions held
  // A decode step reads its position from dec_pos (device) and its tokens /
  // writes its logits through fixed buffers, so the same CUDA graph replays
  // every step; it is captured on dec_st once per batch size.
  int32_t *dec_pos = nullptr, *dec_tok = nullptr;
  float* dec_logits = nullptr;
  cudaStream_t dec_st = nullptr;
  cudaEvent_t dec_ev0 = nullptr, dec_ev1 = nullptr;
  cudaGraphExec_t dec_exec = nullptr;
  int dec_graph_b = 0;                         // batch of dec_exec (0: none, -1: capture failed)
  // profiling (nc_profile_enable)
  struct Rec { int cls, sub; int ev; double flops, bytes; };
  bool prof_on = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  std::vector<Rec> recs;
  double prof_ms[NC_PROF_CLASSES] = {}, prof_flops[NC_PROF_CLASSES] = {}, prof_bytes[NC_PROF_CLASSES] = {};
  int64_t prof_n[NC_PROF_CLASSES] = {};
};

// ------------------------------------------------------------------ profiling

static int prof_event(nc_model* m) {
  if (m->ev_used == m->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return -1;
    m->ev_pool.push_back(e);
  }
  return (int)m->ev_used++;
}

static int prof_begin(nc_model* m, cudaStream_t st) {
  if (!m->prof_on) return -1;
  int e = prof_event(m);
  if (e >= 0) cudaEventRecord(m->ev_pool[e], st);
  return e;
}

static void prof_end(nc_model* m, int e0, int cls, double flops, double bytes, cudaStream_t st, int sub = -1) {
  if (!m->prof_on || e0 < 0) return;
  int e1 = prof_event(m);
  if (e1 < 0) return;
  cudaEventRecord(m->ev_pool[e1], st);
  m->recs.push_back({cls, sub, e0, flops, bytes});
}

// Fold recorded event pairs into the per-class totals and recycle the events.
static void prof_flush(nc_model* m) {
  if (m->recs.empty()) { m->ev_used = 0; return; }
  cudaEventSynchronize(m->ev_pool[m->ev_used - 1]);
  for (const auto& r : m->recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, m->ev_pool[r.ev], m->ev_pool[r.ev + 1]) == cudaSuccess) {
      for (int c : {r.cls, r.sub}) {
        if (c < 0) continue;
        m->prof_ms[c] += ms;
        m->prof_flops[c] += r.flops;
        m->prof_bytes[c] += r.bytes;
        m->prof_n[c] += 1;
      }
    }
  }
  m->recs.clear();
  m->ev_used = 0;
}

#define PROF_SUB(cls, sub, flops, bytes, call)                            \
  do {                                                                     \
    int e0_ = prof_begin(m, st);                                           \
    nc_status s_ = (call);                                                 \
    prof_end(m, e0_, (cls), (double)(flops), (double)(bytes), st, (sub));  \
    if (s_ != NC_OK) return s_;                                            \
  } while (0)
#define PROF(cls, flops, bytes, call) PROF_SUB(cls, -1, flops, bytes, call)

// ------------------------------------------------------------------ helpers

static nc_status dalloc(nc_model* m, size_t bytes, void** out) {
  void* p = nullptr;
  if (bytes == 0) bytes = 256;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    *out = nullptr;
    return NC_ERR_ALLOC;
  }
  m->allocs.push_back(p);
  *out = p;
  return NC_OK;
}
template <typename T>
static nc_status dalloc_t(nc_model* m, size_t count, T** out) {
  void* p;
  nc_status s = dalloc(m, count * sizeof(T), &p);
  *out = (T*)p;
  return s;
}

static const ParamTensor& tensor(const nc_model* m, int layer, int which) {
  // which: 0 q, 1 k, 2 v, 3 o, 4 fc, 5 proj
  return m->layout[1 + layer * 6 + which];
}

static nc_status gemm(nc_model* m, int role, int M, int N, int K, const void* A, int64_t lda, int a_kmajor,
                      const void* B, int64_t ldb, int b_kmajor, int ep, void* D, int64_t ldd, void* aux,
                      int64_t ldaux, cudaStream_t st) {
  m->launches += 1;
  const double a = (double)m->act;
  const double out = (ep == NC_EP_STORE_F32) ? 4.0 : (ep == NC_EP_ACCUM_F32) ? 8.0
                   : (ep == NC_EP_STORE || ep == NC_EP_RELU2_SQ) ? a : 2.0 * a;
  const double bytes = ((double)M * K + (double)N * K) * a + (double)M * N * out;
  const double flops = 2.0 * M * N * K;
  if (m->dtype == NC_BF16)
    PROF_SUB(NC_PROF_GEMM, role, flops, bytes,
         launch_gemm_tc(M, N, K, (const bf16*)A, lda, a_kmajor, (const bf16*)B, ldb, b_kmajor, ep, D, ldd, aux,
                        ldaux, m->err, m->gemm_ws, m->gemm_ws_bytes, st));
  else
    PROF_SUB(NC_PROF_GEMM, role, flops, bytes,
         launch_gemm_simt(NC_FP32, M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, ep, D, ldd, aux, ldaux, st));
  return NC_OK;
}

// Attention: bf16 runs on the tensor cores, fp32 on CUDA cores in fp32.
static nc_status attn_fwd(int dtype, int B, int T, int H, int Hkv, int hd, const void* qkv, void* o, float* lse,
                          int32_t* err, cudaStream_t st, unsigned* amax = nullptr) {
  if (dtype == NC_BF16) return launch_attn_fwd_tc(B, T, H, Hkv, hd, (const bf16*)qkv, (bf16*)o, lse, err, st, amax);
  return launch_attn_fwd_simt(dtype, B, T, H, Hkv, hd, qkv, o, lse, st);
}
// rstd_qk / rope_tab (bf16 only): fold the RoPE + QK-norm backward into the output;
// pair_rows > 0 selects the pair-major table layout.
static nc_status attn_bwd(int dtype, int B, int T, int H, int Hkv, int hd, const void* qkv, const void* o,
                          const float* lse, const void* dout, void* dqkv, float* Dv, const float* rstd_qk,
                          const float* rope_tab, int pair_rows, int32_t* err, cudaStream_t st,
                          unsigned* amax = nullptr) {
  if (dtype == NC_BF16)
    return launch_attn_bwd_tc(B, T, H, Hkv, hd, (const bf16*)qkv, (const bf16*)o, lse, (const bf16*)dout,
                              (bf16*)dqkv, Dv, rstd_qk, rope_tab, pair_rows, err, st, amax);
  if (rstd_qk || rope_tab) return NC_ERR_UNSUPPORTED;
  return launch_attn_bwd_simt(dtype, B, T, H, Hkv, hd, qkv, o, lse, dout, dqkv, Dv, st);
}

static void* wptr(const nc_model* m, const ParamTensor& t) { return (uint8_t*)m->wact + t.off * m->act; }
static uint8_t* layer_act(const nc_model* m, uint8_t* base, int l, int64_t width) {
  return base + (size_t)l * m->Nmax * width * m->act;
}

// The transposed input codes of layer l's linear k (0 qkv, 1 proj, 2 fc, 3
// c_proj) in q8xT: [in][q8np] bytes, the layer's four blocks back to back.
static uint8_t* q8x_t(const nc_model* m, int l, int k) {
  const int64_t C = m->C, Hd = (int64_t)m->H * m->hd, F = m->F;
  const int64_t off[4] = {0, C, C + Hd, 2 * C + Hd};
  return m->q8xT + ((int64_t)l * (2 * C + Hd + F) + off[k]) * m->q8np;
}

// ------------------------------------------------------------------ config

static nc_status validate(const nc_config* c, nc_config* out) {
  if (!c) return NC_ERR_ARG;
  nc_config k = *c;
  if (k.rope_base <= 0.f) k.rope_base = 10000.f;
  if (k.norm_eps < 0.f) k.norm_eps = FLT_EPSILON;
  if (k.init_std <= 0.f) k.init_std = 0.02f;
  if (k.depth <= 0 || k.n_embd <= 0 || k.n_head <= 0 || k.n_kv_head <= 0 || k.head_dim <= 0 ||
      k.mlp_hidden <= 0 || k.vocab <= 0 || k.seq_len <= 0 || k.batch <= 0)
    return NC_ERR_CONFIG;
  if (k.dtype != NC_FP32 && k.dtype != NC_BF16) return NC_ERR_CONFIG;
  if (k.n_embd != k.n_head * k.head_dim) return NC_ERR_CONFIG;
  if (k.n_head % k.n_kv_head) return NC_ERR_CONFIG;
  if (k.head_dim % 16 || k.head_dim > 256) return NC_ERR_CONFIG;
  if (k.dtype == NC_BF16 && k.head_dim != 64 && k.head_dim != 128) return NC_ERR_CONFIG;
  if (k.n_embd % 8 || k.mlp_hidden % 8 || k.vocab % 8) return NC_ERR_CONFIG;
  if (k.n_embd > 8192) return NC_ERR_CONFIG;
  if (!(k.logit_softcap >= 0.f) || k.logit_softcap == INFINITY) return NC_ERR_CONFIG;
  if (k.embed_norm != 0 && k.embed_norm != 1) return NC_ERR_CONFIG;
  if (k.fp8 != 0 && k.fp8 != 1) return NC_ERR_CONFIG;
  if (k.fp8 && (k.dtype != NC_BF16 || k.n_embd % 16 || k.mlp_hidden % 16)) return NC_ERR_CONFIG;
  if ((int64_t)k.batch * k.seq_len > (1 << 20)) return NC_ERR_CONFIG;
  *out = k;
  return NC_OK;
}

static void build_layout(nc_model* m) {
  int64_t off = 0;
  auto add = [&](const std::string& n, int64_t r, int64_t c) {
    m->layout.push_back({n, r, c, off});
    off += r * c;
  };
  add("wte", m->V, m->C);
  for (int l = 0; l < m->L; ++l) {
    std::string p = "h" + std::to_string(l) + ".";
    add(p + "wq", (int64_t)m->H * m->hd, m->C);
    add(p + "wk", (int64_t)m->Hkv * m->hd, m->C);
    add(p + "wv", (int64_t)m->Hkv * m->hd, m->C);
    add(p + "wo", m->C, (int64_t)m->H * m->hd);
    add(p + "wfc", m->F, m->C);
    add(p + "wproj", m->C, m->F);
  }
  add("lm_head", m->V, m->C);
  m->P = off;
}

static nc_status allocate(nc_model* m) {
  const int64_t N = m->Nmax;
  const size_t a = m->act;
  const int L = m->L;
  NC_TRY(dalloc_t(m, (size_t)m->P, &m->master));
  if (m->dtype == NC_BF16) NC_TRY(dalloc(m, (size_t)m->P * 2, &m->wact));
  else m->wact = m->master;
  NC_TRY(dalloc_t(m, (size_t)m->Tmax * m->hd, &m->rope_tab));
  if (m->hd % 4 == 0) NC_TRY(dalloc_t(m, (size_t)m->Tmax * m->hd, &m->rope_pairs));
  NC_TRY(dalloc_t(m, 4, &m->err));
  NC_TRY(dalloc_t(m, 4, &m->result));
  if (cudaMallocHost((void**)&m->result_host, 16) != cudaSuccess) { cudaGetLastError(); return NC_ERR_ALLOC; }
  NC_TRY(dalloc_t(m, (size_t)N * m->C, &m->x));
  NC_TRY(dalloc(m, (size_t)L * N * m->C * a, (void**)&m->xn1));
  NC_TRY(dalloc(m, (size_t)L * N * m->C * a, (void**)&m->xn2));
  NC_TRY(dalloc(m, (size_t)L * N * m->qkvw * a, (void**)&m->qkv));
  NC_TRY(dalloc(m, (size_t)L * N * m->H * m->hd * a, (void**)&m->o));
  NC_TRY(dalloc(m, (size_t)L * N * m->F * a, (void**)&m->h));
  NC_TRY(dalloc_t(m, (size_t)L * N, &m->rstd1));
  NC_TRY(dalloc_t(m, (size_t)L * N, &m->rstd2));
  NC_TRY(dalloc_t(m, (size_t)L * N * (m->H + m->Hkv), &m->rstdqk));
  NC_TRY(dalloc_t(m, (size_t)L * N * m->H, &m->lse));
  NC_TRY(dalloc(m, (size_t)N * m->C * a, &m->xf));
  if (m->emb_norm) NC_TRY(dalloc_t(m, (size_t)N, &m->rstd_e));
  if (m->fp8) {
    const int64_t kmax = std::max<int64_t>(std::max<int64_t>(m->C, m->F), std::max<int64_t>(m->qkvw, m->H * m->hd));
    NC_TRY(dalloc(m, (size_t)(N * kmax), (void**)&m->q8a));
    // the blocks' weight operands [Wq; Wk; Wv], Wo, Wfc, Wproj, each its own tensor
    if (4 * L > NC_OPT_MAXT) return NC_ERR_UNSUPPORTED;
    m->q8tl = new (std::nothrow) OptTensors;
    if (!m->q8tl) return NC_ERR_ALLOC;
    memset(m->q8tl, 0, sizeof(OptTensors));
    m->q8tl->n = 4 * L;
    m->q8tt = new (std::nothrow) Fp8Transposes;
    if (!m->q8tt) return NC_ERR_ALLOC;
    memset(m->q8tt, 0, sizeof(Fp8Transposes));
    m->q8tt->n = 4 * L;
    int32_t c = 0, tiles = 0;
    int64_t so = 0;
    for (int l = 0; l < L; ++l) {
      const int64_t len[4] = {(int64_t)m->qkvw * m->C, (int64_t)m->C * m->H * m->hd, (int64_t)m->F * m->C,
                              (int64_t)m->C * m->F};
      const int which[4] = {0, 3, 4, 5};
      const int rows[4] = {m->qkvw, m->C, m->F, m->C}, cols[4] = {m->C, m->H * m->hd, m->C, m->F};
      for (int k = 0; k < 4; ++k) {
        const int t = 4 * l + k;
        m->q8tt->tile0[t] = tiles;
        m->q8tt->off[t] = so;
        m->q8tt->rows[t] = rows[k];
        m->q8tt->cols[t] = cols[k];
        tiles += ((rows[k] + 63) / 64) * ((cols[k] + 63) / 64);
        m->q8tl->chunk0[t] = c;
        m->q8tl->off[t] = tensor(m, l, which[k]).off;
        m->q8tl->soff[t] = so;
        m->q8tl->len[t] = len[k];
        c += (int32_t)((len[k] + OPT_CHUNK - 1) / OPT_CHUNK);
        so += (len[k] + 255) / 256 * 256;
      }
    }
    m->q8tl->chunk0[4 * L] = c;
    m->q8tt->tile0[4 * L] = tiles;
    NC_TRY(dalloc(m, (size_t)so, (void**)&m->q8w));
    NC_TRY(dalloc(m, (size_t)so, (void**)&m->q8wT));
    m->q8np = (N + 15) / 16 * 16;
    const int64_t xrows = 2 * (int64_t)m->C + (int64_t)m->H * m->hd + m->F;   // the four inputs' widths
    NC_TRY(dalloc(m, (size_t)(L * xrows * m->q8np), (void**)&m->q8xT));
    NC_TRY(dalloc(m, (size_t)(kmax * m->q8np), (void**)&m->q8dyT));
    NC_TRY(dalloc_t(m, (size_t)48 * L, &m->q8s));
  }
  NC_TRY(dalloc_t(m, (size_t)N, &m->rstd_f));
  // logits chunk: at most 1 GiB of compute-dtype logits per chunk, whole 128-row tiles
  int64_t rows = ((int64_t)1 << 30) / ((int64_t)m->V * (int64_t)a);
  rows = std::max<int64_t>(128, rows / 128 * 128);
  m->chunk_rows = std::min<int64_t>(rows, N);
  NC_TRY(dalloc(m, (size_t)m->chunk_rows * m->V * a, &m->logits));
  NC_TRY(dalloc_t(m, (size_t)N, &m->rowloss));
  NC_TRY(dalloc_t(m, (size_t)N * m->C, &m->dx));
  if (m->dtype == NC_BF16) NC_TRY(dalloc(m, (size_t)N * m->C * a, &m->dx_act));
  else m->dx_act = m->dx;
  NC_TRY(dalloc(m, (size_t)N * m->F * a, &m->du));
  NC_TRY(dalloc_t(m, (size_t)N * m->C, &m->dxn));
  NC_TRY(dalloc(m, (size_t)N * m->H * m->hd * a, &m->dout));
  NC_TRY(dalloc(m, (size_t)N * m->qkvw * a, &m->dqkv));
  NC_TRY(dalloc_t(m, (size_t)N * m->H, &m->Dv));
  NC_TRY(dalloc(m, embed_bwd_scratch_bytes(N, m->C, m->V), &m->emb_scratch));
  if (m->dtype == NC_BF16) {
    m->gemm_ws_bytes = gemm_tc_workspace_bytes();
    NC_TRY(dalloc(m, m->gemm_ws_bytes, &m->gemm_ws));
  }
  NC_TRY(dalloc_t(m, (size_t)N, &m->tok_dev));
  NC_TRY(dalloc_t(m, (size_t)N, &m->tgt_dev));
  return NC_OK;
}

// ------------------------------------------------------------------ ABI: misc

extern "C" const char* nc_status_string(nc_status s) {
  switch (s) {
    case NC_OK: return "ok";
    case NC_ERR_CONFIG: return "invalid config";
    case NC_ERR_ALLOC: return "device allocation failed";
    case NC_ERR_ARG: return "invalid argument";
    case NC_ERR_TOKEN_RANGE: return "token or target outside [0, vocab)";
    case NC_ERR_CUDA: return "CUDA error";
    case NC_ERR_TIMEOUT: return "bounded device wait expired";
    case NC_ERR_UNSUPPORTED: return "unsupported shape or mode";
  }
  return "unknown status";
}

extern "C" const char* nc_version(void) {
  return "libnc 0.3 sm_103a (tcgen05 GEMM and flash attention, Muon + AdamW optimizer)";
}

extern "C" void nc_model_destroy(nc_model* m) {
  if (!m) return;
  for (cudaEvent_t e : m->ev_pool) cudaEventDestroy(e);
  for (void* p : m->allocs) cudaFree(p);
  if (m->result_host) cudaFreeHost(m->result_host);
  delete m->opt_tl;
  for (auto& g : m->ns_groups) delete g.apply;
  delete m->q8tl;
  delete m->q8tt;
  for (int k = 0; k < nc_model::NC_OPT_STREAMS; ++k) {
    if (m->opt_st[k]) cudaStreamDestroy(m->opt_st[k]);
    if (m->opt_join[k]) cudaEventDestroy(m->opt_join[k]);
  }
  if (m->opt_fork) cudaEventDestroy(m->opt_fork);
  if (m->dec_exec) cudaGraphExecDestroy(m->dec_exec);
  if (m->dec_st) cudaStreamDestroy(m->dec_st);
  if (m->dec_ev0) cudaEventDestroy(m->dec_ev0);
  if (m->dec_ev1) cudaEventDestroy(m->dec_ev1);
  delete m;
}

extern "C" nc_status nc_model_create(const nc_config* cfg, uint64_t seed, nc_model** out) {
  if (!out) return NC_ERR_ARG;
  *out = nullptr;
  nc_config c;
  NC_TRY(validate(cfg, &c));
  nc_model* m = new (std::nothrow) nc_model();
  if (!m) return NC_ERR_ALLOC;
  m->cfg = c;
  m->L = c.depth; m->C = c.n_embd; m->H = c.n_head; m->Hkv = c.n_kv_head; m->hd = c.head_dim;
  m->F = c.mlp_hidden; m->V = c.vocab; m->Tmax = c.seq_len; m->Bmax = c.batch;
  m->qkvw = (m->H + 2 * m->Hkv) * m->hd;
  m->dtype = c.dtype;
  m->act = (c.dtype == NC_BF16) ? 2 : 4;
  m->Nmax = (int64_t)c.batch * c.seq_len;
  m->softcap = c.logit_softcap;
  m->emb_norm = c.embed_norm != 0;
  m->fp8 = c.fp8 != 0;
  build_layout(m);
  nc_status s = allocate(m);
  cudaStream_t st = 0;
  if (s == NC_OK) {
    for (size_t j = 0; j < m->layout.size() && s == NC_OK; ++j) {
      const ParamTensor& t = m->layout[j];
      s = launch_init_normal(m->master + t.off, t.rows * t.cols, seed, (int)j, c.init_std, st);
    }
  }
  if (s == NC_OK) s = launch_rope_table(m->Tmax, m->hd, c.rope_base, m->rope_tab, m->rope_pairs, st);
  if (s == NC_OK && cudaMemsetAsync(m->err, 0, sizeof(int32_t), st) != cudaSuccess) s = NC_ERR_CUDA;
  if (s == NC_OK && cudaStreamSynchronize(st) != cudaSuccess) s = NC_ERR_CUDA;
  if (s != NC_OK) {
    nc_model_destroy(m);
    return s;
  }
  *out = m;
  return NC_OK;
}

extern "C" nc_status nc_model_config(const nc_model* m, nc_config* out) {
  if (!m || !out) return NC_ERR_ARG;
  *out = m->cfg;
  return NC_OK;
}

extern "C" nc_status nc_param_layout(const nc_model* m, int32_t* n_tensors, int64_t* n_elems) {
  if (!m) return NC_ERR_ARG;
  if (n_tensors) *n_tensors = (int32_t)m->layout.size();
  if (n_elems) *n_elems = m->P;
  return NC_OK;
}

extern "C" nc_status nc_param_count(const nc_model* m, int32_t* n_tensors, int64_t* n_elems) {
  return nc_param_layout(m, n_tensors, n_elems);
}

extern "C" nc_status nc_param_info(const nc_model* m, int32_t i, const char** name, int64_t* rows, int64_t* cols,
                                   int64_t* offset) {
  if (!m || i < 0 || i >= (int32_t)m->layout.size()) return NC_ERR_ARG;
  const ParamTensor& t = m->layout[i];
  if (name) *name = t.name.c_str();
  if (rows) *rows = t.rows;
  if (cols) *cols = t.cols;
  if (offset) *offset = t.off;
  return NC_OK;
}

extern "C" nc_status nc_get_params(const nc_model* m, float* dst, void* stream) {
  if (!m || !dst) return NC_ERR_ARG;
  NC_CUDA_TRY(cudaMemcpyAsync(dst, m->master, (size_t)m->P * 4, cudaMemcpyDeviceToDevice, as_stream(stream)));
  return NC_OK;
}

extern "C" nc_status nc_set_params(nc_model* m, const float* src, void* stream) {
  if (!m || !src) return NC_ERR_ARG;
  NC_CUDA_TRY(cudaMemcpyAsync(m->master, src, (size_t)m->P * 4, cudaMemcpyDeviceToDevice, as_stream(stream)));
  return NC_OK;
}

extern "C" int64_t nc_last_launch_count(const nc_model* m) { return m ? m->launches : 0; }

static nc_status read_flag_status(nc_model* m, cudaStream_t st) {
  NC_CUDA_TRY(cudaMemcpyAsync(m->result_host + 1, m->err, 4, cudaMemcpyDeviceToHost, st));
  NC_CUDA_TRY(cudaStreamSynchronize(st));
  int32_t f;
  memcpy(&f, m->result_host + 1, 4);
  NC_CUDA_TRY(cudaMemsetAsync(m->err, 0, 4, st));
  if (f & NC_DEVERR_TIMEOUT) return NC_ERR_TIMEOUT;
  if (f & NC_DEVERR_TOKEN) return NC_ERR_TOKEN_RANGE;
  return NC_OK;
}

extern "C" nc_status nc_last_error(nc_model* m, void* stream) {
  if (!m) return NC_ERR_ARG;
  return read_flag_status(m, as_stream(stream));
}

// ------------------------------------------------------------------ the step

static nc_status check_bt(const nc_model* m, int32_t B, int32_t T) {
  if (B < 1 || B > m->Bmax || T < 1 || T > m->Tmax) return NC_ERR_ARG;
  return NC_OK;
}

// Weight cast, embedding and all L blocks; leaves xf = norm(x) and rstd_f.
static nc_status forward_trunk(nc_model* m, const int32_t* tokens, int B, int T, cudaStream_t st) {
  const int64_t N = (int64_t)B * T;
  const int C = m->C, F = m->F, Hd = m->H * m->hd, W = m->qkvw;
  const float eps = m->cfg.norm_eps;
  if (m->dtype == NC_BF16) {
    // every tensor except wte is read by a GEMM in bf16
    const ParamTensor& w0 = m->layout[1];
    PROF(NC_PROF_CAST, 0, 6.0 * (m->P - w0.off),
         launch_cast_bf16(m->master + w0.off, (bf16*)m->wact + w0.off, m->P - w0.off, st));
    m->launches += 1;
  }
  PROF(NC_PROF_EMBED, 0, (double)N * (8.0 * C + 4),
       launch_embed_fwd(m->dtype, N, C, m->V, tokens, m->master, m->x, m->err, st, m->rstd_e, eps));
  m->launches += 1;
  const double a = (double)m->act;
  const int nh = m->H + m->Hkv;
  const double attn_fl = 4.0 * B * m->H * m->hd * ((double)T * (T + 1) / 2.0);
  const double nrm_by = (double)N * (4.0 * C + a * C + 4);
  // The 8-bit step: every block weight operand is quantised once per step (two
  // launches over all of them); a linear layer's bf16 input is quantised into
  // q8a with its own statistics slot (the cast only, when the RMSNorm that
  // produced it has taken its maximum), then the E4M3 GEMM runs through the
  // layer's epilogue (RoPE + QK-norm with NC_EP_QKV_ROPE, else `ep`).
  if (m->fp8) {
    NC_CUDA_TRY(cudaMemsetAsync(m->q8s, 0, (size_t)48 * m->L * sizeof(float), st));
    PROF(NC_PROF_QUANT, 0, 9.0 * (double)m->q8tl->soff[4 * m->L - 1],
         launch_fp8_quantize_multi(*m->q8tl, m->master, m->q8s + 16 * m->L, m->q8w, st));
    m->launches += 2;
  }
  // (the input's maximum is already in its slot: its producer took it)
  auto lin8 = [&](int l, int k, const void* act_in, int K, int Nout, int ep, void* D, int64_t ldd, float* rstdqk,
                  unsigned* amax_out = nullptr) -> nc_status {
    float* as = m->q8s + (4 * l + k) * 4;
    float* ws = m->q8s + 16 * m->L + (4 * l + k) * 4;
    const uint8_t* w8 = m->q8w + m->q8tl->soff[4 * l + k];
    // the codes in both layouts: row-major for this product, transposed for its weight gradient
    PROF(NC_PROF_QUANT, 0, 4.0 * N * K,
         launch_fp8_cast_dual(act_in, (int)N, K, as, m->q8a, q8x_t(m, l, k), m->q8np, st));
    const double out = ep == NC_EP_ACCUM_F32 ? 8.0 : 2.0;
    PROF_SUB(NC_PROF_GEMM, NC_PROF_GEMM_FWD, 2.0 * N * Nout * K, (double)N * K + (double)Nout * K + (double)N * Nout * out,
             launch_gemm_fp8_ep((int)N, Nout, K, m->q8a, K, w8, K, as + 2, ws + 2, ep, D, ldd, T, nh, m->hd,
                                m->rope_pairs ? m->rope_pairs : m->rope_tab, m->rope_pairs ? m->Tmax : 0, rstdqk,
                                eps, m->err, st, nullptr, 0, amax_out));
    m->launches += 2;
    return NC_OK;
  };
  for (int l = 0; l < m->L; ++l) {
    uint8_t* xn1 = layer_act(m, m->xn1, l, C);
    uint8_t* xn2 = layer_act(m, m->xn2, l, C);
    uint8_t* qkv = layer_act(m, m->qkv, l, W);
    uint8_t* o = layer_act(m, m->o, l, Hd);
    uint8_t* h = layer_act(m, m->h, l, F);
    float* rstd1 = m->rstd1 + (size_t)l * m->Nmax;
    float* rstd2 = m->rstd2 + (size_t)l * m->Nmax;
    float* rstdqk = m->rstdqk + (size_t)l * m->Nmax * (m->H + m->Hkv);
    float* lse = m->lse + (size_t)l * m->Nmax * m->H;
    if (m->fp8) {
      // the norms take the maximum of the bf16 values they store: their inputs' quantisation is one cast
      PROF(NC_PROF_NORM, 0, nrm_by,
           launch_rmsnorm_fwd(m->dtype, N, C, m->x, xn1, rstd1, eps, st, (unsigned*)(m->q8s + (4 * l + 0) * 4)));
      NC_TRY(lin8(l, 0, xn1, C, W, NC_EP_QKV_ROPE, qkv, W, rstdqk));
      // the attention epilogue takes the maximum of O for the output projection's quantiser
      PROF(NC_PROF_ATTN_FWD, attn_fl, (double)N * (W + Hd) * a + 4.0 * N * m->H,
           attn_fwd(m->dtype, B, T, m->H, m->Hkv, m->hd, qkv, o, lse, m->err, st,
                    (unsigned*)(m->q8s + (4 * l + 1) * 4)));
      NC_TRY(lin8(l, 1, o, Hd, C, NC_EP_ACCUM_F32, m->x, C, nullptr));
      PROF(NC_PROF_NORM, 0, nrm_by,
           launch_rmsnorm_fwd(m->dtype, N, C, m->x, xn2, rstd2, eps, st, (unsigned*)(m->q8s + (4 * l + 2) * 4)));
      // the up-projection's epilogue takes the maximum of relu(u)^2 for the down-projection's quantiser
      NC_TRY(lin8(l, 2, xn2, C, F, NC_EP_RELU2_SQ, h, F, nullptr, (unsigned*)(m->q8s + (4 * l + 3) * 4)));
      NC_TRY(lin8(l, 3, h, F, C, NC_EP_ACCUM_F32, m->x, C, nullptr));
      m->launches += 3;
      continue;
    }
    PROF(NC_PROF_NORM, 0, nrm_by, launch_rmsnorm_fwd(m->dtype, N, C, m->x, xn1, rstd1, eps, st));
    if (m->dtype == NC_BF16) {
      // q/k/v projection with RoPE and the q/k RMSNorm in the GEMM epilogue
      PROF_SUB(NC_PROF_GEMM, NC_PROF_GEMM_FWD, 2.0 * N * W * C, ((double)N * C + (double)W * C + (double)N * W) * a,
               launch_gemm_tc_qkv_rope((int)N, W, C, (const bf16*)xn1, C, (const bf16*)wptr(m, tensor(m, l, 0)), C,
                                       (bf16*)qkv, W, T, nh, m->hd, m->rope_pairs ? m->rope_pairs : m->rope_tab,
                                       m->rope_pairs ? m->Tmax : 0, rstdqk, eps, m->err, st));
      m->launches += 1;
    } else {
      NC_TRY(gemm(m, NC_PROF_GEMM_FWD, (int)N, W, C, xn1, C, 1, wptr(m, tensor(m, l, 0)), C, 1, NC_EP_STORE, qkv, W,
                  nullptr, 0, st));
      PROF(NC_PROF_ROPE, 0, (double)N * nh * (2.0 * a * m->hd + 4),
           launch_rope_qknorm_fwd(m->dtype, B, T, m->H, m->Hkv, m->hd, qkv, rstdqk, m->rope_tab, eps, st));
    }
    PROF(NC_PROF_ATTN_FWD, attn_fl, (double)N * (W + Hd) * a + 4.0 * N * m->H,
         attn_fwd(m->dtype, B, T, m->H, m->Hkv, m->hd, qkv, o, lse, m->err, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_FWD, (int)N, C, Hd, o, Hd, 1, wptr(m, tensor(m, l, 3)), Hd, 1, NC_EP_ACCUM_F32, m->x, C, nullptr, 0,
                st));
    PROF(NC_PROF_NORM, 0, nrm_by, launch_rmsnorm_fwd(m->dtype, N, C, m->x, xn2, rstd2, eps, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_FWD, (int)N, F, C, xn2, C, 1, wptr(m, tensor(m, l, 4)), C, 1, NC_EP_RELU2_SQ, h, F, nullptr, 0, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_FWD, (int)N, C, F, h, F, 1, wptr(m, tensor(m, l, 5)), F, 1, NC_EP_ACCUM_F32, m->x, C, nullptr, 0, st));
    m->launches += 4;
  }
  PROF(NC_PROF_NORM, 0, nrm_by, launch_rmsnorm_fwd(m->dtype, N, C, m->x, m->xf, m->rstd_f, eps, st));
  m->launches += 1;
  return NC_OK;
}

// One block's backward in the 8-bit step.  Each linear's output gradient dY
// is quantised once, per tensor, with its own statistics slot (its producer
// has taken the maximum), into q8a and transposed into q8dyT.  The input
// gradient dX = dY W multiplies those codes with W's forward codes read
// transposed; the weight gradient dW = dY^T X multiplies the transposed codes
// of dY and of X (kept from the forward), each with its own factor, split
// over K (the tokens) when the output has few tiles.
static nc_status backward_layer_fp8(nc_model* m, int l, int B, int T, float* grads, int gw, cudaStream_t st) {
  const int64_t N = (int64_t)B * T;
  const int C = m->C, F = m->F, Hd = m->H * m->hd, W = m->qkvw;
  const int n = (int)N;
  const double a = (double)m->act;
  const double attn_fl = 8.0 * B * m->H * m->hd * ((double)T * (T + 1) / 2.0);
  const double nb_by = (double)N * (4.0 * C + a * C + 4 + 8.0 * C + a * C);
  uint8_t* xn1 = layer_act(m, m->xn1, l, C);
  uint8_t* xn2 = layer_act(m, m->xn2, l, C);
  uint8_t* qkv = layer_act(m, m->qkv, l, W);
  uint8_t* o = layer_act(m, m->o, l, Hd);
  uint8_t* h = layer_act(m, m->h, l, F);
  float* rstd1 = m->rstd1 + (size_t)l * m->Nmax;
  float* rstd2 = m->rstd2 + (size_t)l * m->Nmax;
  float* rstdqk = m->rstdqk + (size_t)l * m->Nmax * (m->H + m->Hkv);
  float* lse = m->lse + (size_t)l * m->Nmax * m->H;
  const ParamTensor &tq = tensor(m, l, 0), &to = tensor(m, l, 3), &tfc = tensor(m, l, 4), &tpj = tensor(m, l, 5);
  auto slot = [&](int ll, int k) { return m->q8s + 32 * m->L + (4 * ll + k) * 4; };
  // k: the linear (0 qkv, 1 proj, 2 fc, 3 c_proj); dy [N][K]; Nout: its input width
  auto bwd8 = [&](int k, const void* dy, int K, int Nout, int ep, void* D, const void* aux, float* dw,
                  unsigned* amax_out = nullptr) -> nc_status {
    float* ys = slot(l, k);
    const float* ws = m->q8s + 16 * m->L + (4 * l + k) * 4;
    const float* xs = m->q8s + (4 * l + k) * 4;   // the forward input's factor
    const uint8_t* wT = m->q8wT + m->q8tl->soff[4 * l + k];
    PROF(NC_PROF_QUANT, 0, 4.0 * N * K, launch_fp8_cast_dual(dy, n, K, ys, m->q8a, m->q8dyT, m->q8np, st));
    const double out = ep == NC_EP_STORE_F32 ? 4.0 : (aux ? 4.0 : 2.0);
    PROF_SUB(NC_PROF_GEMM, NC_PROF_GEMM_DX, 2.0 * N * Nout * K,
             (double)N * K + (double)Nout * K + (double)N * Nout * out,
             launch_gemm_fp8_ep(n, Nout, K, m->q8a, K, wT, K, ys + 2, ws + 2, ep, D, Nout, 0, 0, 0, nullptr, 0,
                                nullptr, 0.f, m->err, st, aux, aux ? Nout : 0, amax_out));
    PROF_SUB(NC_PROF_GEMM, NC_PROF_GEMM_DW, 2.0 * N * Nout * K,
             (double)N * K + (double)Nout * N + (double)K * Nout * (gw == NC_EP_ACCUM_F32 ? 8.0 : 4.0),
             launch_gemm_fp8_ep(K, Nout, n, m->q8dyT, m->q8np, q8x_t(m, l, k), m->q8np, ys + 2, xs + 2, gw, dw, Nout,
                                0, 0, 0, nullptr, 0, nullptr, 0.f, m->err, st, nullptr, 0, nullptr, m->gemm_ws,
                                m->gemm_ws_bytes));
    m->launches += 3;
    return NC_OK;
  };
  // MLP: x2 = x1 + relu(xn2 Wfc^T)^2 Wproj^T; the relu^2-backward epilogue
  // takes the maximum of du for the up-projection's quantiser
  NC_TRY(bwd8(3, m->dx_act, C, F, NC_EP_RELU2_SQ_BWD, m->du, h, grads + tpj.off, (unsigned*)slot(l, 2)));
  NC_TRY(bwd8(2, m->du, F, C, NC_EP_STORE_F32, m->dxn, nullptr, grads + tfc.off));
  PROF(NC_PROF_NORM, 0, nb_by,
       launch_rmsnorm_bwd(m->dtype, N, C, m->dxn, xn2, rstd2, m->dx, m->dx_act, st, (unsigned*)slot(l, 1)));
  // attention: x1 = x + o Wo^T
  NC_TRY(bwd8(1, m->dx_act, C, Hd, NC_EP_STORE, m->dout, nullptr, grads + to.off));
  // the attention backward's epilogues take the maximum of dq, dk and dv for the dX quantiser
  PROF(NC_PROF_ATTN_BWD, attn_fl, (double)N * (2.0 * W + 2.0 * Hd) * a + 8.0 * N * m->H,
       attn_bwd(m->dtype, B, T, m->H, m->Hkv, m->hd, qkv, o, lse, m->dout, m->dqkv, m->Dv, rstdqk,
                m->rope_pairs ? m->rope_pairs : m->rope_tab, m->rope_pairs ? m->Tmax : 0, m->err, st,
                (unsigned*)slot(l, 0)));
  NC_TRY(bwd8(0, m->dqkv, W, C, NC_EP_STORE_F32, m->dxn, nullptr, grads + tq.off));
  // the block's input gradient is the previous block's output gradient: its maximum, for that block's Wproj product
  PROF(NC_PROF_NORM, 0, nb_by,
       launch_rmsnorm_bwd(m->dtype, N, C, m->dxn, xn1, rstd1, m->dx, m->dx_act, st,
                          l > 0 ? (unsigned*)slot(l - 1, 3) : nullptr));
  m->launches += 2 + 3;   // the two norms and the attention backward's three kernels
  return NC_OK;
}

// accumulate: the weight gradients are added to `grads` instead of stored.
static nc_status backward_layers(nc_model* m, const int32_t* tokens, int B, int T, float* grads, bool accumulate,
                                 cudaStream_t st) {
  const int gw = accumulate ? NC_EP_ACCUM_F32 : NC_EP_STORE_F32;
  const int64_t N = (int64_t)B * T;
  const int C = m->C, F = m->F, Hd = m->H * m->hd, W = m->qkvw;
  const int n = (int)N;
  const double a = (double)m->act;
  const int nh = m->H + m->Hkv;
  const double attn_fl = 8.0 * B * m->H * m->hd * ((double)T * (T + 1) / 2.0);
  const double nb_by = (double)N * (4.0 * C + a * C + 4 + 8.0 * C + (m->dtype == NC_BF16 ? a * C : 0));
  for (int l = m->L - 1; l >= 0; --l) {
    uint8_t* xn1 = layer_act(m, m->xn1, l, C);
    uint8_t* xn2 = layer_act(m, m->xn2, l, C);
    uint8_t* qkv = layer_act(m, m->qkv, l, W);
    uint8_t* o = layer_act(m, m->o, l, Hd);
    uint8_t* h = layer_act(m, m->h, l, F);
    float* rstd1 = m->rstd1 + (size_t)l * m->Nmax;
    float* rstd2 = m->rstd2 + (size_t)l * m->Nmax;
    float* rstdqk = m->rstdqk + (size_t)l * m->Nmax * (m->H + m->Hkv);
    float* lse = m->lse + (size_t)l * m->Nmax * m->H;
    const ParamTensor &tq = tensor(m, l, 0), &to = tensor(m, l, 3), &tfc = tensor(m, l, 4),
                      &tpj = tensor(m, l, 5);
    if (m->fp8) {
      NC_TRY(backward_layer_fp8(m, l, B, T, grads, gw, st));
      continue;
    }
    // MLP: x2 = x1 + relu(xn2 Wfc^T)^2 Wproj^T
    NC_TRY(gemm(m, NC_PROF_GEMM_DW, C, F, n, m->dx_act, C, 0, h, F, 0, gw, grads + tpj.off, F, nullptr, 0, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_DX, n, F, C, m->dx_act, C, 1, wptr(m, tpj), F, 0, NC_EP_RELU2_SQ_BWD, m->du, F, h, F, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_DW, F, C, n, m->du, F, 0, xn2, C, 0, gw, grads + tfc.off, C, nullptr, 0, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_DX, n, C, F, m->du, F, 1, wptr(m, tfc), C, 0, NC_EP_STORE_F32, m->dxn, C, nullptr, 0, st));
    PROF(NC_PROF_NORM, 0, nb_by,
         launch_rmsnorm_bwd(m->dtype, N, C, m->dxn, xn2, rstd2, m->dx, m->dtype == NC_BF16 ? m->dx_act : nullptr,
                            st));
    // attention: x1 = x + o Wo^T
    NC_TRY(gemm(m, NC_PROF_GEMM_DW, C, Hd, n, m->dx_act, C, 0, o, Hd, 0, gw, grads + to.off, Hd, nullptr, 0, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_DX, n, Hd, C, m->dx_act, C, 1, wptr(m, to), Hd, 0, NC_EP_STORE, m->dout, Hd, nullptr, 0, st));
    if (m->dtype == NC_BF16) {
      // attention backward with the q/k RMSNorm + RoPE backward in its output epilogue
      PROF(NC_PROF_ATTN_BWD, attn_fl, (double)N * (2.0 * W + 2.0 * Hd) * a + 8.0 * N * m->H,
           attn_bwd(m->dtype, B, T, m->H, m->Hkv, m->hd, qkv, o, lse, m->dout, m->dqkv, m->Dv, rstdqk,
                    m->rope_pairs ? m->rope_pairs : m->rope_tab, m->rope_pairs ? m->Tmax : 0, m->err, st));
    } else {
      PROF(NC_PROF_ATTN_BWD, attn_fl, (double)N * (2.0 * W + 2.0 * Hd) * a + 8.0 * N * m->H,
           attn_bwd(m->dtype, B, T, m->H, m->Hkv, m->hd, qkv, o, lse, m->dout, m->dqkv, m->Dv, nullptr, nullptr, 0,
                    m->err, st));
      PROF(NC_PROF_ROPE, 0, (double)N * nh * (3.0 * a * m->hd + 4),
           launch_rope_qknorm_bwd(m->dtype, B, T, m->H, m->Hkv, m->hd, m->dqkv, qkv, rstdqk, m->rope_tab, st));
    }
    NC_TRY(gemm(m, NC_PROF_GEMM_DW, W, C, n, m->dqkv, W, 0, xn1, C, 0, gw, grads + tq.off, C, nullptr, 0, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_DX, n, C, W, m->dqkv, W, 1, wptr(m, tq), C, 0, NC_EP_STORE_F32, m->dxn, C, nullptr, 0, st));
    PROF(NC_PROF_NORM, 0, nb_by,
         launch_rmsnorm_bwd(m->dtype, N, C, m->dxn, xn1, rstd1, m->dx, m->dtype == NC_BF16 ? m->dx_act : nullptr,
                            st));
    m->launches += 3 + 1 + 2;
  }
  const ParamTensor& te = m->layout[0];
  if (m->emb_norm) {   // through the norm after the embedding, in place on dx
    PROF(NC_PROF_EMBED, 0, (double)N * (12.0 * C + 8),
         launch_embed_norm_bwd(m->dtype, N, C, m->V, tokens, m->master, m->rstd_e, m->dx, st));
    m->launches += 1;
  }
  PROF(NC_PROF_EMBED, 0, 4.0 * N * C + 4.0 * m->V * C,
       launch_embed_bwd(N, C, m->V, tokens, m->dx, grads + te.off, m->emb_scratch, st, accumulate ? 1 : 0,
                        m->err));
  m->launches += 4;
  return NC_OK;
}

// grads = (accumulate ? grads : 0) + gscale * d(mean CE)/d(params); the scale
// enters through the cross-entropy gradient, which every gradient is linear in.
static nc_status step(nc_model* m, const int32_t* tokens, const int32_t* targets, int B, int T, float* loss_host,
                      float* grads, float gscale, bool accumulate, cudaStream_t st) {
  const int64_t N = (int64_t)B * T;
  const int C = m->C, V = m->V;
  m->launches = 0;
  prof_flush(m);
  NC_TRY(forward_trunk(m, tokens, B, T, st));
  const ParamTensor& tl = m->layout.back();
  const void* Wlm = wptr(m, tl);
  NC_CUDA_TRY(cudaMemsetAsync(m->dx, 0, (size_t)N * C * sizeof(float), st));
  const float scale = gscale / (float)N;
  for (int64_t c0 = 0; c0 < N; c0 += m->chunk_rows) {
    const int nc = (int)std::min<int64_t>(m->chunk_rows, N - c0);
    const void* xfc = (const uint8_t*)m->xf + (size_t)c0 * C * m->act;
    NC_TRY(gemm(m, NC_PROF_GEMM_LM, nc, V, C, xfc, C, 1, Wlm, C, 1, NC_EP_STORE, m->logits, V, nullptr, 0, st));
    PROF(NC_PROF_CE, 0, (double)nc * (2.0 * V * m->act + 8),
         launch_cross_entropy(m->dtype, nc, V, m->logits, V, targets + c0, m->rowloss + c0, scale, m->err, st,
                              m->softcap));
    NC_TRY(gemm(m, NC_PROF_GEMM_LM, nc, C, V, m->logits, V, 1, Wlm, C, 0, NC_EP_STORE_F32, m->dxn + c0 * C, C, nullptr, 0, st));
    NC_TRY(gemm(m, NC_PROF_GEMM_LM, V, C, nc, m->logits, V, 0, xfc, C, 0,
                (c0 == 0 && !accumulate) ? NC_EP_STORE_F32 : NC_EP_ACCUM_F32,
                grads + tl.off, C, nullptr, 0, st));
    m->launches += 1;
  }
  // the 8-bit step's dX products read the weight codes transposed, and the
  // final norm takes the maximum of the last block's output gradient
  unsigned* amax_last = nullptr;
  if (m->fp8) {
    PROF(NC_PROF_QUANT, 0, 2.0 * (double)m->q8tl->soff[4 * m->L - 1],
         launch_fp8_transpose_multi(*m->q8tt, m->q8w, m->q8wT, st));
    m->launches += 1;
    amax_last = (unsigned*)(m->q8s + 32 * m->L + (4 * (m->L - 1) + 3) * 4);
  }
  PROF(NC_PROF_NORM, 0, (double)N * (4.0 * C + m->act * C + 4 + 8.0 * C + (m->dtype == NC_BF16 ? m->act * C : 0)),
       launch_rmsnorm_bwd(m->dtype, N, C, m->dxn, m->xf, m->rstd_f, m->dx, m->dtype == NC_BF16 ? m->dx_act : nullptr,
                          st, amax_last));
  m->launches += 1;
  NC_TRY(backward_layers(m, tokens, B, T, grads, accumulate, st));
  PROF(NC_PROF_OTHER, 0, 4.0 * N, launch_mean(N, m->rowloss, m->result, st));
  m->launches += 1;
  NC_CUDA_TRY(cudaMemcpyAsync(m->result_host, m->result, 4, cudaMemcpyDeviceToHost, st));
  nc_status s = read_flag_status(m, st);   // synchronises the stream
  if (loss_host) memcpy(loss_host, m->result_host, 4);
  return s;
}

extern "C" nc_status nc_forward_backward(nc_model* m, const int32_t* tokens, const int32_t* targets, int32_t B,
                                         int32_t T, float* loss_host, float* grads, void* stream) {
  if (!m || !tokens || !targets || !loss_host || !grads) return NC_ERR_ARG;
  NC_TRY(check_bt(m, B, T));
  return step(m, tokens, targets, B, T, loss_host, grads, 1.f, false, as_stream(stream));
}

extern "C" nc_status nc_forward_backward_accumulate(nc_model* m, const int32_t* tokens, const int32_t* targets,
                                                    int32_t B, int32_t T, float grad_scale, int32_t accumulate,
                                                    float* loss_host, float* grads, void* stream) {
  if (!m || !tokens || !targets || !loss_host || !grads || !std::isfinite(grad_scale)) return NC_ERR_ARG;
  NC_TRY(check_bt(m, B, T));
  return step(m, tokens, targets, B, T, loss_host, grads, grad_scale, accumulate != 0, as_stream(stream));
}

extern "C" nc_status nc_forward_backward_host(nc_model* m, const int32_t* tokens_host, const int32_t* targets_host,
                                              int32_t B, int32_t T, float* loss_host, float* grads, void* stream) {
  if (!m || !tokens_host || !targets_host || !loss_host || !grads) return NC_ERR_ARG;
  NC_TRY(check_bt(m, B, T));
  cudaStream_t st = as_stream(stream);
  size_t bytes = (size_t)B * T * sizeof(int32_t);
  NC_CUDA_TRY(cudaMemcpyAsync(m->tok_dev, tokens_host, bytes, cudaMemcpyHostToDevice, st));
  NC_CUDA_TRY(cudaMemcpyAsync(m->tgt_dev, targets_host, bytes, cudaMemcpyHostToDevice, st));
  return step(m, m->tok_dev, m->tgt_dev, B, T, loss_host, grads, 1.f, false, st);
}

extern "C" nc_status nc_forward_logits(nc_model* m, const int32_t* tokens, int32_t B, int32_t T, float* logits,
                                       void* stream) {
  if (!m || !tokens || !logits) return NC_ERR_ARG;
  NC_TRY(check_bt(m, B, T));
  cudaStream_t st = as_stream(stream);
  m->launches = 0;
  NC_TRY(forward_trunk(m, tokens, B, T, st));
  const int64_t N = (int64_t)B * T;
  NC_TRY(gemm(m, NC_PROF_GEMM_LM, (int)N, m->V, m->C, m->xf, m->C, 1, wptr(m, m->layout.back()), m->C, 1, NC_EP_STORE_F32, logits,
              m->V, nullptr, 0, st));
  return launch_softcap_f32(N * m->V, logits, m->softcap, st);
}

extern "C" nc_status nc_forward_row_losses(nc_model* m, const int32_t* tokens, const int32_t* targets, int32_t B,
                                           int32_t T, float* losses, void* stream) {
  if (!m || !tokens || !targets || !losses) return NC_ERR_ARG;
  NC_TRY(check_bt(m, B, T));
  cudaStream_t st = as_stream(stream);
  m->launches = 0;
  NC_TRY(forward_trunk(m, tokens, B, T, st));
  const int64_t N = (int64_t)B * T;
  for (int64_t c0 = 0; c0 < N; c0 += m->chunk_rows) {
    const int nc = (int)std::min<int64_t>(m->chunk_rows, N - c0);
    const void* xfc = (const uint8_t*)m->xf + (size_t)c0 * m->C * m->act;
    NC_TRY(gemm(m, NC_PROF_GEMM_LM, nc, m->V, m->C, xfc, m->C, 1, wptr(m, m->layout.back()), m->C, 1, NC_EP_STORE, m->logits, m->V,
                nullptr, 0, st));
    NC_TRY(launch_cross_entropy(m->dtype, nc, m->V, m->logits, m->V, targets + c0, losses + c0, 1.f, m->err, st,
                                m->softcap));
  }
  return NC_OK;
}

// ------------------------------------------------------------------ kernel-level entry points

static bool dtype_ok(int32_t d) { return d == NC_FP32 || d == NC_BF16; }

extern "C" size_t nc_gemm_workspace_bytes(void) { return gemm_tc_workspace_bytes(); }

extern "C" nc_status nc_op_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* A, int64_t lda,
                                int32_t a_kmajor, const void* B, int64_t ldb, int32_t b_kmajor, int32_t ep, void* D,
                                int64_t ldd, void* aux, int64_t ldaux, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (!dtype_ok(dtype) || !A || !B || !D || ep < 0 || ep > NC_EP_RELU2_SQ_BWD) return NC_ERR_ARG;
  if (M < 0 || N < 0 || K < 0) return NC_ERR_ARG;
  if (dtype == NC_BF16)
    return launch_gemm_tc(M, N, K, (const bf16*)A, lda, a_kmajor, (const bf16*)B, ldb, b_kmajor, ep, D, ldd, aux,
                          ldaux, nullptr, workspace, workspace ? workspace_bytes : 0, as_stream(stream));
  return launch_gemm_simt(dtype, M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, ep, D, ldd, aux, ldaux,
                          as_stream(stream));
}

extern "C" nc_status nc_op_rmsnorm_fwd(int32_t dtype, int64_t rows, int32_t C, const float* x, void* y, float* rstd,
                                       float eps, void* stream) {
  if (!dtype_ok(dtype) || !x || !y || !rstd || C <= 0) return NC_ERR_ARG;
  return launch_rmsnorm_fwd(dtype, rows, C, x, y, rstd, eps, as_stream(stream));
}

extern "C" nc_status nc_op_rmsnorm_bwd(int32_t dtype, int64_t rows, int32_t C, const float* dy, const void* y,
                                       const float* rstd, float* dx, void* dx_act, void* stream) {
  if (!dtype_ok(dtype) || !dy || !y || !rstd || !dx || C <= 0) return NC_ERR_ARG;
  return launch_rmsnorm_bwd(dtype, rows, C, dy, y, rstd, dx, dx_act, as_stream(stream));
}

extern "C" nc_status nc_op_rope_table(int32_t T, int32_t hd, float rope_base, float* cos_sin, void* stream) {
  return launch_rope_table(T, hd, rope_base, cos_sin, nullptr, as_stream(stream));
}

extern "C" nc_status nc_op_rope_table_pairs(int32_t T, int32_t hd, float rope_base, float* pairs, void* stream) {
  return launch_rope_table(T, hd, rope_base, nullptr, pairs, as_stream(stream));
}

extern "C" nc_status nc_op_rope_qknorm_fwd(int32_t dtype, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                           void* qkv, float* rstd, const float* cos_sin, float eps, void* stream) {
  if (!dtype_ok(dtype) || !qkv || !rstd || !cos_sin || B <= 0 || T <= 0 || H <= 0 || Hkv <= 0) return NC_ERR_ARG;
  return launch_rope_qknorm_fwd(dtype, B, T, H, Hkv, hd, qkv, rstd, cos_sin, eps, as_stream(stream));
}

extern "C" nc_status nc_op_gemm_qkv_rope(int32_t M, int32_t K, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                         const void* x, int64_t ldx, const void* wqkv, void* qkv, int64_t ldqkv,
                                         float* rstd, const float* cos_sin, int32_t pair_rows, float eps,
                                         void* stream) {
  if (!x || !wqkv || !qkv || !rstd || !cos_sin || M < 0 || K <= 0 || T <= 0 || H <= 0 || Hkv <= 0 || H % Hkv)
    return NC_ERR_ARG;
  const int N = (H + 2 * Hkv) * hd;
  return launch_gemm_tc_qkv_rope(M, N, K, (const bf16*)x, ldx, (const bf16*)wqkv, K, (bf16*)qkv, ldqkv, T, H + Hkv,
                                 hd, cos_sin, pair_rows, rstd, eps, nullptr, as_stream(stream));
}

extern "C" nc_status nc_op_rope_qknorm_bwd(int32_t dtype, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                           void* dqkv, const void* qkv, const float* rstd, const float* cos_sin,
                                           void* stream) {
  if (!dtype_ok(dtype) || !dqkv || !qkv || !rstd || !cos_sin || B <= 0 || T <= 0 || H <= 0 || Hkv <= 0)
    return NC_ERR_ARG;
  return launch_rope_qknorm_bwd(dtype, B, T, H, Hkv, hd, dqkv, qkv, rstd, cos_sin, as_stream(stream));
}

extern "C" nc_status nc_op_attention_fwd(int32_t dtype, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                         const void* qkv, void* o, float* lse, void* stream) {
  if (!dtype_ok(dtype) || !qkv || !o || !lse) return NC_ERR_ARG;
  return attn_fwd(dtype, B, T, H, Hkv, hd, qkv, o, lse, nullptr, as_stream(stream));
}

extern "C" nc_status nc_op_attention_bwd(int32_t dtype, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                         const void* qkv, const void* o, const float* lse, const void* do_,
                                         void* dqkv, float* workspace, void* stream) {
  if (!dtype_ok(dtype) || !qkv || !o || !lse || !do_ || !dqkv || !workspace) return NC_ERR_ARG;
  return attn_bwd(dtype, B, T, H, Hkv, hd, qkv, o, lse, do_, dqkv, workspace, nullptr, nullptr, 0, nullptr,
                  as_stream(stream));
}

extern "C" nc_status nc_op_attention_bwd_rope(int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                              const void* qkv, const void* o, const float* lse, const void* do_,
                                              void* dqkv, float* workspace, const float* rstd, const float* cos_sin,
                                              int32_t pair_rows, void* stream) {
  if (!qkv || !o || !lse || !do_ || !dqkv || !workspace || !rstd || !cos_sin) return NC_ERR_ARG;
  if (pair_rows < 0 || (pair_rows > 0 && pair_rows < T)) return NC_ERR_ARG;
  return attn_bwd(NC_BF16, B, T, H, Hkv, hd, qkv, o, lse, do_, dqkv, workspace, rstd, cos_sin, pair_rows, nullptr,
                  as_stream(stream));
}

extern "C" nc_status nc_op_cross_entropy(int32_t dtype, int64_t rows, int32_t V, void* z, const int32_t* targets,
                                         float* row_loss, float grad_scale, int32_t* err_dev, void* stream) {
  if (!dtype_ok(dtype) || !z || !targets || !row_loss || V <= 0) return NC_ERR_ARG;
  return launch_cross_entropy(dtype, rows, V, z, V, targets, row_loss, grad_scale, err_dev, as_stream(stream));
}

extern "C" nc_status nc_op_cross_entropy_softcap(int32_t dtype, int64_t rows, int32_t V, void* z,
                                                 const int32_t* targets, float* row_loss, float grad_scale,
                                                 float softcap, int32_t* err_dev, void* stream) {
  if (!dtype_ok(dtype) || !z || !targets || !row_loss || V <= 0) return NC_ERR_ARG;
  if (!(softcap >= 0.f) || softcap == INFINITY) return NC_ERR_ARG;
  return launch_cross_entropy(dtype, rows, V, z, V, targets, row_loss, grad_scale, err_dev, as_stream(stream),
                              softcap);
}

extern "C" nc_status nc_op_embed_fwd(int32_t dtype, int64_t n, int32_t C, int32_t V, const int32_t* tokens,
                                     const float* wte, float* x, int32_t* err_dev, void* stream) {
  if (!dtype_ok(dtype) || !tokens || !wte || !x || C <= 0 || V <= 0) return NC_ERR_ARG;
  return launch_embed_fwd(dtype, n, C, V, tokens, wte, x, err_dev, as_stream(stream));
}

extern "C" size_t nc_embed_bwd_scratch_bytes(int64_t n, int32_t C, int32_t V) {
  return embed_bwd_scratch_bytes(n, C, V);
}

extern "C" nc_status nc_op_embed_bwd(int64_t n, int32_t C, int32_t V, const int32_t* tokens, const float* dx,
                                     float* dwte, void* scratch, void* stream) {
  if (!tokens || !dx || !dwte || !scratch || n < 0) return NC_ERR_ARG;
  return launch_embed_bwd(n, C, V, tokens, dx, dwte, scratch, as_stream(stream));
}

extern "C" nc_status nc_profile_enable(nc_model* m, int32_t on) {
  if (!m) return NC_ERR_ARG;
  prof_flush(m);
  for (int c = 0; c < NC_PROF_CLASSES; ++c) {
    m->prof_ms[c] = m->prof_flops[c] = m->prof_bytes[c] = 0.0;
    m->prof_n[c] = 0;
  }
  m->prof_on = on != 0;
  return NC_OK;
}

extern "C" nc_status nc_profile_read(nc_model* m, int32_t cls, double* ms, int64_t* launches, double* flops,
                                     double* bytes) {
  if (!m || cls < 0 || cls >= NC_PROF_CLASSES) return NC_ERR_ARG;
  prof_flush(m);
  if (ms) *ms = m->prof_ms[cls];
  if (launches) *launches = m->prof_n[cls];
  if (flops) *flops = m->prof_flops[cls];
  if (bytes) *bytes = m->prof_bytes[cls];
  return NC_OK;
}

// Test hook: the time limit (ns) of every bounded wait in the tensor-core kernels.
extern "C" void nc_debug_set_wait_limit_ns(uint64_t ns) { g_tc_wait_ns = ns; }

extern int g_gemm_pair;
extern "C" void nc_debug_set_gemm_pair(int32_t on) { g_gemm_pair = on != 0; }

extern int g_tc_stall_next;
extern "C" void nc_debug_stall_next_gemm(int32_t on) { g_tc_stall_next = on != 0; }

static int g_ns_batched = 1;
extern "C" void nc_debug_set_ns_batched(int32_t on) { g_ns_batched = on != 0; }

// ------------------------------------------------------------------ optimizer
// Muon for every weight matrix, AdamW for wte and lm_head (cosmicrealm
// "noao-chat-0-项目总体介绍" §2.2, §4.2).

extern "C" void nc_optim_config_default(nc_optim_config* oc) {
  if (!oc) return;
  oc->matrix_lr = 0.02f;
  oc->embedding_lr = 0.2f;
  oc->unembedding_lr = 0.004f;
  oc->momentum = 0.95f;
  oc->nesterov = 1;
  oc->ns_steps = 5;
  oc->beta1 = 0.9f;
  oc->beta2 = 0.999f;
  oc->adam_eps = 1e-8f;
  oc->weight_decay = 0.f;
}

static void opt_fill(OptTensors* tl, const int64_t* off, const int64_t* len, int n) {
  memset(tl, 0, sizeof(*tl));
  tl->n = n;
  int32_t c = 0;
  int64_t so = 0;
  for (int i = 0; i < n; ++i) {
    tl->chunk0[i] = c;
    tl->off[i] = off[i];
    tl->soff[i] = so;
    tl->len[i] = len[i];
    c += (int32_t)((len[i] + OPT_CHUNK - 1) / OPT_CHUNK);
    so += len[i];
  }
  tl->chunk0[n] = c;
}

static nc_status opt_alloc(nc_model* m) {
  const int nm = 6 * m->L;
  if (nm > NC_OPT_MAXT) return NC_ERR_UNSUPPORTED;
  std::vector<int64_t> off(nm), len(nm);
  int64_t total = 0, maxrc = 0, maxn = 0;
  for (int i = 0; i < nm; ++i) {
    const ParamTensor& t = m->layout[1 + i];
    off[i] = t.off;
    len[i] = t.rows * t.cols;
    total += len[i];
    maxrc = std::max(maxrc, len[i]);
    maxn = std::max(maxn, std::min(t.rows, t.cols));
  }
  m->opt_tl = new OptTensors;
  opt_fill(m->opt_tl, off.data(), len.data(), nm);
  const int64_t nchunks = m->opt_tl->chunk0[nm];
  const ParamTensor& te = m->layout.front();
  const ParamTensor& tl = m->layout.back();
  const int64_t na = te.rows * te.cols + tl.rows * tl.cols;
  NC_TRY(dalloc_t(m, (size_t)total, &m->opt_mom));
  NC_TRY(dalloc_t(m, (size_t)total, &m->opt_u));
  NC_TRY(dalloc_t(m, (size_t)std::max<int64_t>(nchunks, 1), &m->opt_partial));
  NC_TRY(dalloc_t(m, (size_t)nm, &m->opt_norm));
  NC_TRY(dalloc(m, (size_t)total * m->act, &m->opt_x0));
  // matrices of one shape in one group, in order of first appearance
  bool batched = g_ns_batched && m->dtype == NC_BF16;
  m->ns_groups.clear();
  for (int i = 0; i < nm; ++i) {
    const ParamTensor& t = m->layout[1 + i];
    if (t.rows % 128) batched = false;
    size_t g = 0;
    while (g < m->ns_groups.size() && (m->ns_groups[g].rows != t.rows || m->ns_groups[g].cols != t.cols)) ++g;
    if (g == m->ns_groups.size()) {
      nc_model::NsGroup ng;
      ng.rows = (int)t.rows;
      ng.cols = (int)t.cols;
      ng.xr = (t.rows + 255) / 256 * 256;
      ng.nr = (std::min(t.rows, t.cols) + 255) / 256 * 256;
      m->ns_groups.push_back(ng);
    }
    m->ns_groups[g].members.push_back(i);
  }
  if (!batched) m->ns_groups.clear();
  for (auto& g : m->ns_groups) {
    const int nb = (int)g.members.size();
    if (nb > NC_OPT_MAXT) return NC_ERR_UNSUPPORTED;
    g.apply = new (std::nothrow) OptTensors;
    if (!g.apply) return NC_ERR_ALLOC;
    memset(g.apply, 0, sizeof(OptTensors));
    g.apply->n = nb;
    int32_t c = 0;
    for (int b = 0; b < nb; ++b) {
      const ParamTensor& t = m->layout[1 + g.members[b]];
      g.apply->chunk0[b] = c;
      g.apply->off[b] = t.off;
      g.apply->soff[b] = (int64_t)b * g.xr * g.cols;
      g.apply->len[b] = t.rows * t.cols;
      c += (int32_t)((g.apply->len[b] + OPT_CHUNK - 1) / OPT_CHUNK);
    }
    g.apply->chunk0[nb] = c;
  }
  if (batched) {
    int64_t xmax = 0, amax = 0;
    for (const auto& g : m->ns_groups) {
      const int64_t nb = (int64_t)g.members.size();
      xmax = std::max(xmax, nb * g.xr * g.cols);
      amax = std::max(amax, nb * g.nr * std::min(g.rows, g.cols));
    }
    NC_TRY(dalloc(m, (size_t)xmax * m->act, &m->nsb_ping0));
    NC_TRY(dalloc(m, (size_t)xmax * m->act, &m->nsb_ping1));
    NC_TRY(dalloc(m, (size_t)amax * m->act, &m->nsb_a));
    NC_TRY(dalloc(m, (size_t)amax * m->act, &m->nsb_a2));
  }
  for (int k = 0; k < nc_model::NC_OPT_STREAMS; ++k) {
    if (!batched) {
      NC_TRY(dalloc(m, (size_t)maxrc * m->act, &m->opt_ping0[k]));
      NC_TRY(dalloc(m, (size_t)maxrc * m->act, &m->opt_ping1[k]));
      NC_TRY(dalloc(m, (size_t)(maxn * maxn) * m->act, &m->opt_a[k]));
      NC_TRY(dalloc(m, (size_t)(maxn * maxn) * m->act, &m->opt_a2[k]));
    }
    NC_CUDA_TRY(cudaStreamCreateWithFlags(&m->opt_st[k], cudaStreamNonBlocking));
    NC_CUDA_TRY(cudaEventCreateWithFlags(&m->opt_join[k], cudaEventDisableTiming));
  }
  NC_CUDA_TRY(cudaEventCreateWithFlags(&m->opt_fork, cudaEventDisableTiming));
  NC_TRY(dalloc_t(m, (size_t)na, &m->adam_m));
  NC_TRY(dalloc_t(m, (size_t)na, &m->adam_v));
  // longest-processing-time-first assignment of matrices to the side streams
  std::vector<double> work(nm);
  for (int i = 0; i < nm; ++i) {
    const ParamTensor& t = m->layout[1 + i];
    const double n = (double)std::min(t.rows, t.cols), k = (double)std::max(t.rows, t.cols);
    work[i] = 4.0 * n * n * k + 2.0 * n * n * n;
  }
  m->opt_order.resize(nm);
  m->opt_lane.assign(nm, 0);
  for (int i = 0; i < nm; ++i) m->opt_order[i] = i;
  std::stable_sort(m->opt_order.begin(), m->opt_order.end(), [&](int a, int b) { return work[a] > work[b]; });
  double load[nc_model::NC_OPT_STREAMS] = {};
  for (int i : m->opt_order) {
    int best = 0;
    for (int k = 1; k < nc_model::NC_OPT_STREAMS; ++k)
      if (load[k] < load[best]) best = k;
    m->opt_lane[i] = best;
    load[best] += work[i];
  }
  m->opt_tl->norm = m->opt_norm;
  m->opt_ready = true;
  return NC_OK;
}

extern "C" nc_status nc_optimizer_reset(nc_model* m, void* stream) {
  if (!m) return NC_ERR_ARG;
  m->opt_t = 0;
  if (!m->opt_ready) return NC_OK;
  cudaStream_t st = as_stream(stream);
  const int64_t total = m->opt_tl->soff[m->opt_tl->n - 1] + m->opt_tl->len[m->opt_tl->n - 1];
  const ParamTensor& te = m->layout.front();
  const ParamTensor& tl = m->layout.back();
  const int64_t na = te.rows * te.cols + tl.rows * tl.cols;
  NC_CUDA_TRY(cudaMemsetAsync(m->opt_mom, 0, (size_t)total * sizeof(float), st));
  NC_CUDA_TRY(cudaMemsetAsync(m->adam_m, 0, (size_t)na * sizeof(float), st));
  NC_CUDA_TRY(cudaMemsetAsync(m->adam_v, 0, (size_t)na * sizeof(float), st));
  return NC_OK;
}

extern "C" int64_t nc_optimizer_steps(const nc_model* m) { return m ? m->opt_t : -1; }

// Newton-Schulz + apply for every matrix.  Batched (bf16, rows multiples of
// 128): per shape group, the members' X0 are copied into one stacked buffer,
// iterate together and are applied one by one, on `st`.  Otherwise each
// matrix runs on a side stream, forked from and joined back into `st`; no
// split-K workspace, since the side streams run concurrently and must not
// share one.
static nc_status opt_matrices(nc_model* m, const nc_optim_config* oc, float lr_mult, cudaStream_t st) {
  const OptTensors& tl = *m->opt_tl;
  if (!m->ns_groups.empty()) {
    for (const auto& g : m->ns_groups) {
      const int nb = (int)g.members.size();
      const size_t xbytes = (size_t)g.xr * g.cols * m->act;   // one stacked matrix with its padding rows
      for (int b = 0; b < nb; ++b)
        NC_CUDA_TRY(cudaMemcpyAsync((uint8_t*)m->nsb_ping0 + b * xbytes,
                                    (const uint8_t*)m->opt_x0 + tl.soff[g.members[b]] * m->act,
                                    (size_t)g.rows * g.cols * m->act, cudaMemcpyDeviceToDevice, st));
      const void* x = m->nsb_ping0;
      if (oc->ns_steps > 0)
        NC_TRY(newton_schulz_batched(nb, g.rows, g.cols, oc->ns_steps, m->nsb_ping0, m->nsb_ping1, g.xr, m->nsb_a,
                                     m->nsb_a2, g.nr, &x, m->err, st));
      const float scale = sqrtf(std::max(1.f, (float)g.rows / (float)g.cols));
      NC_TRY(launch_muon_apply_multi(m->dtype, *g.apply, m->master, x, oc->matrix_lr * lr_mult * scale, st));
    }
    return NC_OK;
  }
  NC_CUDA_TRY(cudaEventRecord(m->opt_fork, st));
  for (int k = 0; k < nc_model::NC_OPT_STREAMS; ++k) NC_CUDA_TRY(cudaStreamWaitEvent(m->opt_st[k], m->opt_fork, 0));
  nc_status s = NC_OK;
  for (int i : m->opt_order) {
    const ParamTensor& t = m->layout[1 + i];
    const int k = m->opt_lane[i];
    cudaStream_t sk = m->opt_st[k];
    const void* x = (const uint8_t*)m->opt_x0 + tl.soff[i] * m->act;
    if (oc->ns_steps > 0)
      s = newton_schulz_run(m->dtype, (int)t.rows, (int)t.cols, oc->ns_steps, x, m->opt_ping0[k], m->opt_ping1[k],
                            m->opt_a[k], m->opt_a2[k], &x, m->err, nullptr, 0, sk);
    if (s != NC_OK) break;
    const float scale = sqrtf(std::max(1.f, (float)t.rows / (float)t.cols));
    s = launch_muon_apply(m->dtype, t.rows * t.cols, m->master + t.off, x, oc->matrix_lr * lr_mult * scale, sk);
    if (s != NC_OK) break;
  }
  // always join, so that `st` orders after everything already enqueued on the side streams
  for (int k = 0; k < nc_model::NC_OPT_STREAMS; ++k) {
    if (cudaEventRecord(m->opt_join[k], m->opt_st[k]) != cudaSuccess ||
        cudaStreamWaitEvent(st, m->opt_join[k], 0) != cudaSuccess)
      s = NC_ERR_CUDA;
  }
  return s;
}

extern "C" nc_status nc_optimizer_step(nc_model* m, const nc_optim_config* oc, const float* grads, float lr_mult,
                                       void* stream) {
  if (!m || !oc || !grads) return NC_ERR_ARG;
  if (oc->ns_steps < 0 || oc->ns_steps > 64 || !(oc->momentum >= 0.f && oc->momentum < 1.f) ||
      !(oc->beta1 >= 0.f && oc->beta1 < 1.f) || !(oc->beta2 >= 0.f && oc->beta2 < 1.f) || !(oc->adam_eps > 0.f))
    return NC_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  if (!m->opt_ready) {
    NC_TRY(opt_alloc(m));
    NC_TRY(nc_optimizer_reset(m, stream));
  }
  prof_flush(m);
  m->opt_t += 1;
  const OptTensors& tl = *m->opt_tl;
  const int64_t total = tl.soff[tl.n - 1] + tl.len[tl.n - 1];
  const double act = (double)m->act;
  // Muon: momentum, Nesterov update and its norm for every matrix at once
  PROF(NC_PROF_OPT_EW, 0, 16.0 * total,
       launch_muon_momentum(tl, grads, m->opt_mom, m->opt_u, oc->momentum, oc->nesterov, m->opt_partial, st));
  PROF(NC_PROF_OPT_EW, 0, (4.0 + act) * total, launch_ns_init(m->dtype, tl, m->opt_u, 1e-7f, m->opt_x0, st));
  // per matrix: Newton-Schulz and the apply, on the side streams (profiled as one phase)
  double ns_flops = 0.0, ns_bytes = 0.0;
  for (int i = 0; i < tl.n; ++i) {
    const ParamTensor& t = m->layout[1 + i];
    const double n = (double)std::min(t.rows, t.cols), k = (double)std::max(t.rows, t.cols);
    ns_flops += oc->ns_steps * (4.0 * n * n * k + 2.0 * n * n * n);
    ns_bytes += oc->ns_steps * (4.0 * n * k + 4.0 * n * n) * act + (8.0 + act) * n * k;
  }
  PROF(NC_PROF_OPT_NS, ns_flops, ns_bytes, opt_matrices(m, oc, lr_mult, st));
  // AdamW on the embedding and the output head
  const ParamTensor& te = m->layout.front();
  const ParamTensor& th = m->layout.back();
  const int64_t ne = te.rows * te.cols, nh = th.rows * th.cols;
  PROF(NC_PROF_OPT_EW, 0, 28.0 * ne,
       launch_adamw(ne, m->master + te.off, grads + te.off, m->adam_m, m->adam_v, oc->embedding_lr * lr_mult,
                    oc->beta1, oc->beta2, oc->adam_eps, oc->weight_decay, m->opt_t, st));
  PROF(NC_PROF_OPT_EW, 0, 28.0 * nh,
       launch_adamw(nh, m->master + th.off, grads + th.off, m->adam_m + ne, m->adam_v + ne,
                    oc->unembedding_lr * lr_mult, oc->beta1, oc->beta2, oc->adam_eps, oc->weight_decay, m->opt_t,
                    st));
  return NC_OK;
}

static int64_t align_up(int64_t b) { return (b + 255) & ~(int64_t)255; }

extern "C" size_t nc_newton_schulz_workspace_bytes(int32_t dtype, int32_t rows, int32_t cols) {
  if (!dtype_ok(dtype) || rows <= 0 || cols <= 0) return 0;
  const int64_t rc = (int64_t)rows * cols, n = std::min(rows, cols);
  const int64_t act = dtype == NC_BF16 ? 2 : 4;
  const int64_t nchunks = (rc + OPT_CHUNK - 1) / OPT_CHUNK;
  return (size_t)(align_up(nchunks * 4) + align_up(4) + 2 * align_up(rc * 4) + 3 * align_up(rc * act) +
                  2 * align_up(n * n * act));
}

extern "C" nc_status nc_op_newton_schulz(int32_t dtype, int32_t rows, int32_t cols, int32_t steps, const float* u,
                                         float* x, void* workspace, void* stream) {
  if (!dtype_ok(dtype) || rows <= 0 || cols <= 0 || steps < 0 || steps > 64 || !u || !x || !workspace)
    return NC_ERR_ARG;
  if ((((uintptr_t)workspace) & 255)) return NC_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  const int64_t rc = (int64_t)rows * cols, n = std::min(rows, cols);
  const int64_t act = dtype == NC_BF16 ? 2 : 4;
  uint8_t* p = (uint8_t*)workspace;
  OptTensors tl;
  const int64_t off0 = 0;
  opt_fill(&tl, &off0, &rc, 1);
  float* partial = (float*)p; p += align_up((int64_t)tl.chunk0[1] * 4);
  tl.norm = (float*)p; p += align_up(4);
  float* mom = (float*)p; p += align_up(rc * 4);
  float* uu = (float*)p; p += align_up(rc * 4);
  void* x0 = p; p += align_up(rc * act);
  void* ping0 = p; p += align_up(rc * act);
  void* ping1 = p; p += align_up(rc * act);
  void* A = p; p += align_up(n * n * act);
  void* A2 = p;
  // momentum 0 from a zero buffer gives U = u; this also forms ||u||_F
  NC_CUDA_TRY(cudaMemsetAsync(mom, 0, (size_t)rc * 4, st));
  NC_TRY(launch_muon_momentum(tl, u, mom, uu, 0.f, 0, partial, st));
  NC_TRY(launch_ns_init(dtype, tl, uu, 1e-7f, x0, st));
  const void* out = x0;
  if (steps > 0)
    NC_TRY(newton_schulz_run(dtype, rows, cols, steps, x0, ping0, ping1, A, A2, &out, nullptr, nullptr, 0, st));
  return launch_cast_out(dtype, rc, out, x, st);
}

// ------------------------------------------------------------------ KV-cache decoding
// Prefill runs the forward over B prompts and keeps every layer's (rotated,
// normalised) keys and values; each decode step then feeds one token per
// sequence at the next position: one row of every projection and one
// attention row over the cache (woshipm nanochat analysis §三 item 4).

static size_t kv_layer_elems(const nc_model* m) { return (size_t)m->kv_b * m->Hkv * m->kv_max * m->hd; }

extern "C" nc_status nc_kv_cache_create(nc_model* m, int32_t max_batch, int32_t max_len) {
  if (!m || max_batch < 1 || max_batch > m->Bmax || max_len < 1 || max_len > m->Tmax) return NC_ERR_ARG;
  if ((m->hd != 64 && m->hd != 128) || (m->H / m->Hkv != 1 && m->H / m->Hkv != 2 && m->H / m->Hkv != 3 &&
                                        m->H / m->Hkv != 4 && m->H / m->Hkv != 8))
    return NC_ERR_UNSUPPORTED;
  if (m->fp8) return NC_ERR_UNSUPPORTED;   // decode steps have no 8-bit projections
  NC_TRY(decode_kernels_prepare());
  if (m->kcache && max_batch <= m->kv_b && max_len <= m->kv_max) {
    m->kv_batch = m->kv_len = 0;
    return NC_OK;
  }
  m->kv_b = max_batch;
  m->kv_max = max_len;
  const size_t n = kv_layer_elems(m) * m->L;
  NC_TRY(dalloc(m, n * m->act, &m->kcache));
  NC_TRY(dalloc(m, n * m->act, &m->vcache));
  NC_TRY(dalloc_t(m, decode_part_floats(max_batch, m->H, m->hd, max_len), &m->dec_part));
  NC_TRY(dalloc_t(m, (size_t)max_batch, &m->dec_tok));
  NC_TRY(dalloc_t(m, (size_t)max_batch * m->V, &m->dec_logits));
  if (!m->dec_pos) NC_TRY(dalloc_t(m, 1, &m->dec_pos));
  if (!m->dec_st) {
    NC_CUDA_TRY(cudaStreamCreateWithFlags(&m->dec_st, cudaStreamNonBlocking));
    NC_CUDA_TRY(cudaEventCreateWithFlags(&m->dec_ev0, cudaEventDisableTiming));
    NC_CUDA_TRY(cudaEventCreateWithFlags(&m->dec_ev1, cudaEventDisableTiming));
  }
  if (m->dec_exec) cudaGraphExecDestroy(m->dec_exec);   // it baked in the old buffers
  m->dec_exec = nullptr;
  m->dec_graph_b = 0;
  m->kv_batch = m->kv_len = 0;
  return NC_OK;
}

extern "C" int32_t nc_kv_cache_length(const nc_model* m) { return m ? m->kv_len : -1; }

static void* kv_layer(const nc_model* m, void* base, int l) {
  return (uint8_t*)base + kv_layer_elems(m) * l * m->act;
}

extern "C" nc_status nc_prefill(nc_model* m, const int32_t* tokens, int32_t B, int32_t T, float* logits,
                                void* stream) {
  if (!m || !tokens || !logits) return NC_ERR_ARG;
  if (!m->kcache) return NC_ERR_ARG;
  if (B < 1 || B > m->kv_b || T < 1 || T > m->kv_max) return NC_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  m->launches = 0;
  NC_TRY(forward_trunk(m, tokens, B, T, st));
  for (int l = 0; l < m->L; ++l)
    NC_TRY(launch_kv_store(m->dtype, (int64_t)B * T, T, 0, m->H, m->Hkv, m->hd, layer_act(m, m->qkv, l, m->qkvw),
                           m->qkvw, kv_layer(m, m->kcache, l), kv_layer(m, m->vcache, l), m->kv_max, st));
  // logits of each prompt's last position: rows b*T + T-1 of xf
  const void* last = (const uint8_t*)m->xf + (size_t)(T - 1) * m->C * m->act;
  NC_TRY(gemm(m, NC_PROF_GEMM_LM, B, m->V, m->C, last, (int64_t)T * m->C, 1, wptr(m, m->layout.back()), m->C, 1,
              NC_EP_STORE_F32, logits, m->V, nullptr, 0, st));
  NC_TRY(launch_softcap_f32((int64_t)B * m->V, logits, m->softcap, st));
  NC_TRY(launch_set_i32(m->dec_pos, T, false, st));
  m->kv_batch = B;
  m->kv_len = T;
  return NC_OK;
}

// One decode step for B sequences at position *dec_pos: tokens from dec_tok,
// logits to dec_logits; ends by advancing *dec_pos.  Every argument is fixed
// for a given B, so the enqueued work can be captured once and replayed.
static nc_status decode_body(nc_model* m, int B, cudaStream_t st) {
  const int C = m->C, F = m->F, Hd = m->H * m->hd, W = m->qkvw;
  const float eps = m->cfg.norm_eps;
  // Projections of B <= 8 rows are bound by reading the weights once: CUDA-core
  // skinny GEMM, with the RMSNorm of its input rows done inside it when the
  // input is the residual stream.  Beyond that, the tensor-core GEMM after a
  // separate RMSNorm.
  const bool skinny = B <= 8;
  auto proj = [&](int role, int N, int K, const void* a, const void* w, int ep, void* d, int64_t ldd) -> nc_status {
    if (skinny) return launch_gemm_skinny(m->dtype, B, N, K, a, K, w, K, ep, d, ldd, st);
    return gemm(m, role, B, N, K, a, K, 1, w, K, 1, ep, d, ldd, nullptr, 0, st);
  };
  auto norm_proj = [&](int role, int N, const void* w, int ep, void* d, int64_t ldd, void* xn,
                       float* rstd) -> nc_status {   // d = op(norm(x) W^T)
    if (skinny) return launch_gemm_skinny_norm(m->dtype, B, N, C, m->x, C, w, C, ep, d, ldd, eps, st);
    NC_TRY(launch_rmsnorm_fwd(m->dtype, B, C, m->x, xn, rstd, eps, st));
    return proj(role, N, C, xn, w, ep, d, ldd);
  };
  NC_TRY(launch_embed_fwd(m->dtype, B, C, m->V, m->dec_tok, m->master, m->x, m->err, st, m->rstd_e, eps));
  uint8_t* xn1 = layer_act(m, m->xn1, 0, C);
  uint8_t* xn2 = layer_act(m, m->xn2, 0, C);
  uint8_t* qkv = layer_act(m, m->qkv, 0, W);
  uint8_t* o = layer_act(m, m->o, 0, Hd);
  uint8_t* h = layer_act(m, m->h, 0, F);
  for (int l = 0; l < m->L; ++l) {
    NC_TRY(norm_proj(NC_PROF_GEMM_FWD, W, wptr(m, tensor(m, l, 0)), NC_EP_STORE, qkv, W, xn1, m->rstd1));
    // RoPE + QK norm at position *dec_pos, the cache append of k and v, and attention in one kernel
    NC_TRY(launch_decode_attn(m->dtype, B, m->H, m->Hkv, m->hd, 0, qkv, W, kv_layer(m, m->kcache, l),
                              kv_layer(m, m->vcache, l), m->kv_max, m->dec_part, o, Hd, st, m->dec_pos,
                              m->rope_tab, eps));
    NC_TRY(proj(NC_PROF_GEMM_FWD, C, Hd, o, wptr(m, tensor(m, l, 3)), NC_EP_ACCUM_F32, m->x, C));
    NC_TRY(norm_proj(NC_PROF_GEMM_FWD, F, wptr(m, tensor(m, l, 4)), NC_EP_RELU2_SQ, h, F, xn2, m->rstd2));
    NC_TRY(proj(NC_PROF_GEMM_FWD, C, F, h, wptr(m, tensor(m, l, 5)), NC_EP_ACCUM_F32, m->x, C));
  }
  NC_TRY(norm_proj(NC_PROF_GEMM_LM, m->V, wptr(m, m->layout.back()), NC_EP_STORE_F32, m->dec_logits, m->V, m->xf,
                   m->rstd_f));
  NC_TRY(launch_softcap_f32((int64_t)B * m->V, m->dec_logits, m->softcap, st));
  return launch_set_i32(m->dec_pos, 1, true, st);
}

int g_decode_graph = 1;   // test hook: 0 runs decode steps eagerly

static nc_status decode_capture(nc_model* m, int B) {
  cudaGraph_t g = nullptr;
  NC_CUDA_TRY(cudaStreamBeginCapture(m->dec_st, cudaStreamCaptureModeRelaxed));
  nc_status s = decode_body(m, B, m->dec_st);
  cudaError_t e = cudaStreamEndCapture(m->dec_st, &g);
  if (s == NC_OK && e == cudaSuccess) e = cudaGraphInstantiate(&m->dec_exec, g, 0);
  if (g) cudaGraphDestroy(g);
  if (s != NC_OK || e != cudaSuccess) {
    cudaGetLastError();
    m->dec_exec = nullptr;
    return s != NC_OK ? s : NC_ERR_CUDA;
  }
  m->dec_graph_b = B;
  return NC_OK;
}

extern "C" nc_status nc_decode_step(nc_model* m, const int32_t* tokens, int32_t B, float* logits, void* stream) {
  if (!m || !tokens || !logits) return NC_ERR_ARG;
  if (!m->kcache || m->kv_len < 1 || B != m->kv_batch || m->kv_len >= m->kv_max) return NC_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  NC_CUDA_TRY(cudaMemcpyAsync(m->dec_tok, tokens, (size_t)B * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
  const bool graph = g_decode_graph && !m->prof_on && m->dec_graph_b >= 0;
  if (graph && m->dec_graph_b != B) {
    if (m->dec_exec) cudaGraphExecDestroy(m->dec_exec);
    m->dec_exec = nullptr;
    if (decode_capture(m, B) != NC_OK) m->dec_graph_b = -1;   // run eagerly from now on
  }
  if (graph && m->dec_exec) {
    NC_CUDA_TRY(cudaEventRecord(m->dec_ev0, st));
    NC_CUDA_TRY(cudaStreamWaitEvent(m->dec_st, m->dec_ev0, 0));
    NC_CUDA_TRY(cudaGraphLaunch(m->dec_exec, m->dec_st));
    NC_CUDA_TRY(cudaEventRecord(m->dec_ev1, m->dec_st));
    NC_CUDA_TRY(cudaStreamWaitEvent(st, m->dec_ev1, 0));
  } else {
    NC_TRY(decode_body(m, B, st));
  }
  NC_CUDA_TRY(cudaMemcpyAsync(logits, m->dec_logits, (size_t)B * m->V * sizeof(float), cudaMemcpyDeviceToDevice, st));
  m->kv_len += 1;
  return NC_OK;
}

// Test hook: 0 makes decode steps run eagerly instead of through the captured graph.
extern "C" void nc_debug_set_decode_graph(int32_t on) { g_decode_graph = on != 0; }

extern int g_decode_pdl;
extern "C" void nc_debug_set_decode_pdl(int32_t on) { g_decode_pdl = on != 0; }

extern "C" nc_status nc_op_gemm_rows(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* A, int64_t lda,
                                     const void* W, int64_t ldw, int32_t ep, void* D, int64_t ldd, void* stream) {
  if (!dtype_ok(dtype) || !A || !W || !D) return NC_ERR_ARG;
  return launch_gemm_skinny(dtype, M, N, K, A, lda, W, ldw, ep, D, ldd, as_stream(stream));
}

extern "C" nc_status nc_op_quantize_fp8(int32_t dtype, const void* x_dev, int64_t n, uint8_t* codes_dev,
                                        float* stats_dev, void* stream) {
  return launch_quantize_fp8(dtype, x_dev, n, codes_dev, stats_dev, as_stream(stream));
}

extern "C" nc_status nc_op_gemm_fp8(int32_t M, int32_t N, int32_t K, const uint8_t* a_dev, int64_t lda,
                                    const uint8_t* b_dev, int64_t ldb, const float* a_scale_inv_dev,
                                    const float* b_scale_inv_dev, int32_t out_dtype, void* d_dev, int64_t ldd,
                                    void* stream) {
  if (M < 0 || N < 0 || K < 0 || (out_dtype != NC_BF16 && out_dtype != NC_FP32)) return NC_ERR_ARG;
  return launch_gemm_fp8(M, N, K, a_dev, lda, b_dev, ldb, a_scale_inv_dev, b_scale_inv_dev, out_dtype == NC_FP32,
                         d_dev, ldd, nullptr, as_stream(stream));
}
