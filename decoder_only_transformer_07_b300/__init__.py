"""Python binding of libnc: a B300 (sm_103a) forward+backward training step
of a nanochat-style decoder-only GPT.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libnc.so`` (built in-tree by ``build.py``).  PyTorch supplies
device memory (tensors) and the current CUDA stream.  If the library is
missing, importing this package fails loudly; there is no CPU path.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python decoder_only_transformer_07_b300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

NC_FP32, NC_BF16 = 0, 1
EP_STORE, EP_STORE_F32, EP_ACCUM_F32, EP_RELU2, EP_RELU2_BWD, EP_RELU2_SQ, EP_RELU2_SQ_BWD = range(7)
STATUS = {0: "NC_OK", 1: "NC_ERR_CONFIG", 2: "NC_ERR_ALLOC", 3: "NC_ERR_ARG",
          4: "NC_ERR_TOKEN_RANGE", 5: "NC_ERR_CUDA", 6: "NC_ERR_TIMEOUT", 7: "NC_ERR_UNSUPPORTED"}


class NcError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.nc_status_string(status).decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


class nc_config(ctypes.Structure):
    _fields_ = [("depth", ctypes.c_int32), ("n_embd", ctypes.c_int32), ("n_head", ctypes.c_int32),
                ("n_kv_head", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("mlp_hidden", ctypes.c_int32), ("vocab", ctypes.c_int32), ("seq_len", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("dtype", ctypes.c_int32), ("rope_base", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("init_std", ctypes.c_float), ("logit_softcap", ctypes.c_float),
                ("embed_norm", ctypes.c_int32), ("fp8", ctypes.c_int32)]


class nc_optim_config(ctypes.Structure):
    _fields_ = [("matrix_lr", ctypes.c_float), ("embedding_lr", ctypes.c_float),
                ("unembedding_lr", ctypes.c_float), ("momentum", ctypes.c_float), ("nesterov", ctypes.c_int32),
                ("ns_steps", ctypes.c_int32), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("adam_eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


_p, _i32, _i64, _f32, _u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_uint64
_sz = ctypes.c_size_t
_SIGS = {
    "nc_status_string": (ctypes.c_char_p, [_i32]),
    "nc_version": (ctypes.c_char_p, []),
    "nc_model_create": (_i32, [ctypes.POINTER(nc_config), _u64, ctypes.POINTER(_p)]),
    "nc_model_destroy": (None, [_p]),
    "nc_model_config": (_i32, [_p, ctypes.POINTER(nc_config)]),
    "nc_param_layout": (_i32, [_p, ctypes.POINTER(_i32), ctypes.POINTER(_i64)]),
    "nc_param_count": (_i32, [_p, ctypes.POINTER(_i32), ctypes.POINTER(_i64)]),
    "nc_param_info": (_i32, [_p, _i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_i64),
                             ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    "nc_get_params": (_i32, [_p, _p, _p]),
    "nc_set_params": (_i32, [_p, _p, _p]),
    "nc_forward_backward": (_i32, [_p, _p, _p, _i32, _i32, ctypes.POINTER(_f32), _p, _p]),
    "nc_forward_backward_host": (_i32, [_p, _p, _p, _i32, _i32, ctypes.POINTER(_f32), _p, _p]),
    "nc_forward_backward_accumulate": (_i32, [_p, _p, _p, _i32, _i32, _f32, _i32, ctypes.POINTER(_f32), _p, _p]),
    "nc_forward_logits": (_i32, [_p, _p, _i32, _i32, _p, _p]),
    "nc_forward_row_losses": (_i32, [_p, _p, _p, _i32, _i32, _p, _p]),
    "nc_last_error": (_i32, [_p, _p]),
    "nc_last_launch_count": (_i64, [_p]),
    "nc_op_gemm": (_i32, [_i32, _i32, _i32, _i32, _p, _i64, _i32, _p, _i64, _i32, _i32, _p, _i64, _p, _i64, _p,
                          _sz, _p]),
    "nc_gemm_workspace_bytes": (_sz, []),
    "nc_op_rmsnorm_fwd": (_i32, [_i32, _i64, _i32, _p, _p, _p, _f32, _p]),
    "nc_op_rmsnorm_bwd": (_i32, [_i32, _i64, _i32, _p, _p, _p, _p, _p, _p]),
    "nc_op_rope_table": (_i32, [_i32, _i32, _f32, _p, _p]),
    "nc_op_rope_qknorm_fwd": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _f32, _p]),
    "nc_op_gemm_qkv_rope": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _p, _i64, _p, _p, _i64, _p, _p, _i32, _f32,
                                   _p]),
    "nc_op_rope_table_pairs": (_i32, [_i32, _i32, _f32, _p, _p]),
    "nc_op_rope_qknorm_bwd": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _p]),
    "nc_op_attention_fwd": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p]),
    "nc_op_attention_bwd": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _p, _p, _p]),
    "nc_op_attention_bwd_rope": (_i32, [_i32, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _p, _p, _p, _p, _i32, _p]),
    "nc_op_cross_entropy": (_i32, [_i32, _i64, _i32, _p, _p, _p, _f32, _p, _p]),
    "nc_op_cross_entropy_softcap": (_i32, [_i32, _i64, _i32, _p, _p, _p, _f32, _f32, _p, _p]),
    "nc_op_embed_fwd": (_i32, [_i32, _i64, _i32, _i32, _p, _p, _p, _p, _p]),
    "nc_embed_bwd_scratch_bytes": (_sz, [_i64, _i32, _i32]),
    "nc_optim_config_default": (None, [ctypes.POINTER(nc_optim_config)]),
    "nc_kv_cache_create": (_i32, [_p, _i32, _i32]),
    "nc_prefill": (_i32, [_p, _p, _i32, _i32, _p, _p]),
    "nc_decode_step": (_i32, [_p, _p, _i32, _p, _p]),
    "nc_kv_cache_length": (_i32, [_p]),
    "nc_optimizer_step": (_i32, [_p, ctypes.POINTER(nc_optim_config), _p, _f32, _p]),
    "nc_optimizer_reset": (_i32, [_p, _p]),
    "nc_optimizer_steps": (_i64, [_p]),
    "nc_newton_schulz_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "nc_op_newton_schulz": (_i32, [_i32, _i32, _i32, _i32, _p, _p, _p, _p]),
    "nc_op_embed_bwd": (_i32, [_i64, _i32, _i32, _p, _p, _p, _p, _p]),
    "nc_debug_set_wait_limit_ns": (None, [_u64]),
    "nc_debug_set_gemm_pair": (None, [_i32]),
    "nc_debug_set_ns_batched": (None, [_i32]),
    "nc_debug_stall_next_gemm": (None, [_i32]),
    "nc_debug_set_decode_graph": (None, [_i32]),
    "nc_debug_set_decode_pdl": (None, [_i32]),
    "nc_op_gemm_rows": (_i32, [_i32, _i32, _i32, _i32, _p, _i64, _p, _i64, _i32, _p, _i64, _p]),
    "nc_op_quantize_fp8": (_i32, [_i32, _p, _i64, _p, _p, _p]),
    "nc_op_gemm_fp8": (_i32, [_i32, _i32, _i32, _p, _i64, _p, _i64, _p, _p, _i32, _p, _i64, _p]),
    "nc_profile_enable": (_i32, [_p, _i32]),
    "nc_profile_read": (_i32, [_p, _i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i64),
                                ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def lib():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib


def _check(status, where):
    if status != 0:
        raise NcError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return NC_BF16
    if t.dtype == torch.float32:
        return NC_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_config(depth, n_embd, n_head, n_kv_head, head_dim, mlp_hidden, vocab, seq_len, batch,
                dtype="bf16", rope_base=10000.0, norm_eps=-1.0, init_std=0.02, logit_softcap=0.0, embed_norm=False,
                fp8=False):
    d = NC_BF16 if dtype in ("bf16", NC_BF16) else NC_FP32
    return nc_config(depth, n_embd, n_head, n_kv_head, head_dim, mlp_hidden, vocab, seq_len, batch, d,
                     rope_base, norm_eps, init_std, logit_softcap, 1 if embed_norm else 0, 1 if fp8 else 0)


def optim_config(**kw):
    """nc_optim_config with the library defaults, fields overridden by keyword."""
    oc = nc_optim_config()
    _lib.nc_optim_config_default(ctypes.byref(oc))
    for k, v in kw.items():
        setattr(oc, k, v)
    return oc


def config_from_workload(w, **kw):
    return make_config(w.depth, w.n_embd, w.n_head, w.n_kv_head, w.head_dim, w.mlp_hidden, w.vocab,
                       w.seq_len, w.batch, w.dtype, **kw)


class Model:
    """One GPT model resident on the current CUDA device."""

    def __init__(self, cfg, seed=1):
        self._h = ctypes.c_void_p()
        self.cfg = cfg
        _check(_lib.nc_model_create(ctypes.byref(cfg), ctypes.c_uint64(seed), ctypes.byref(self._h)),
               "nc_model_create")
        nt, ne = _i32(), _i64()
        _check(_lib.nc_param_layout(self._h, ctypes.byref(nt), ctypes.byref(ne)), "nc_param_layout")
        self.n_tensors, self.n_params = nt.value, ne.value
        self.layout = []
        for i in range(self.n_tensors):
            name, r, c, o = ctypes.c_char_p(), _i64(), _i64(), _i64()
            _check(_lib.nc_param_info(self._h, i, ctypes.byref(name), ctypes.byref(r), ctypes.byref(c),
                                      ctypes.byref(o)), "nc_param_info")
            self.layout.append((name.value.decode(), r.value, c.value, o.value))

    def close(self):
        if self._h:
            _lib.nc_model_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def get_params(self, out=None):
        import torch
        if out is None:
            out = torch.empty(self.n_params, dtype=torch.float32, device="cuda")
        _check(_lib.nc_get_params(self._h, _ptr(out), _stream()), "nc_get_params")
        return out

    def set_params(self, flat):
        import torch
        flat = flat.to(device="cuda", dtype=torch.float32).contiguous()
        _check(_lib.nc_set_params(self._h, _ptr(flat), _stream()), "nc_set_params")
        torch.cuda.current_stream().synchronize()

    def forward_backward(self, tokens, targets, grads=None):
        """tokens, targets: int32 CUDA tensors [B, T].  Returns (loss, grads)."""
        import torch
        B, T = tokens.shape
        if grads is None:
            grads = torch.empty(self.n_params, dtype=torch.float32, device="cuda")
        loss = _f32()
        _check(_lib.nc_forward_backward(self._h, _ptr(tokens), _ptr(targets), B, T, ctypes.byref(loss),
                                        _ptr(grads), _stream()), "nc_forward_backward")
        return loss.value, grads

    def forward_backward_accumulate(self, tokens, targets, grads, grad_scale=1.0, accumulate=True):
        """grads (+)= grad_scale * d(mean CE of this micro-batch)/d(params).  Returns the loss."""
        B, T = tokens.shape
        loss = _f32()
        _check(_lib.nc_forward_backward_accumulate(self._h, _ptr(tokens), _ptr(targets), B, T, grad_scale,
                                                   1 if accumulate else 0, ctypes.byref(loss), _ptr(grads),
                                                   _stream()), "nc_forward_backward_accumulate")
        return loss.value

    def forward_backward_host(self, tokens, targets, grads):
        """tokens, targets: int32 host (pinned) tensors [B, T]."""
        B, T = tokens.shape
        loss = _f32()
        _check(_lib.nc_forward_backward_host(self._h, _ptr(tokens), _ptr(targets), B, T, ctypes.byref(loss),
                                             _ptr(grads), _stream()), "nc_forward_backward_host")
        return loss.value

    def forward_logits(self, tokens, out=None):
        import torch
        B, T = tokens.shape
        if out is None:
            out = torch.empty((B, T, self.cfg.vocab), dtype=torch.float32, device="cuda")
        _check(_lib.nc_forward_logits(self._h, _ptr(tokens), B, T, _ptr(out), _stream()), "nc_forward_logits")
        self.check()
        return out

    def row_losses(self, tokens, targets, out=None):
        import torch
        B, T = tokens.shape
        if out is None:
            out = torch.empty((B, T), dtype=torch.float32, device="cuda")
        _check(_lib.nc_forward_row_losses(self._h, _ptr(tokens), _ptr(targets), B, T, _ptr(out), _stream()),
               "nc_forward_row_losses")
        self.check()
        return out

    def check(self):
        _check(_lib.nc_last_error(self._h, _stream()), "device error flag")

    def optimizer_step(self, grads, config=None, lr_mult=1.0):
        """One Muon (matrices) + AdamW (wte, lm_head) step on the fp32 master weights."""
        oc = config if config is not None else optim_config()
        _check(_lib.nc_optimizer_step(self._h, ctypes.byref(oc), _ptr(grads), lr_mult, _stream()),
               "nc_optimizer_step")

    def optimizer_reset(self):
        _check(_lib.nc_optimizer_reset(self._h, _stream()), "nc_optimizer_reset")

    def optimizer_steps(self):
        return int(_lib.nc_optimizer_steps(self._h))

    def kv_cache_create(self, max_batch, max_len):
        _check(_lib.nc_kv_cache_create(self._h, max_batch, max_len), "nc_kv_cache_create")

    def prefill(self, tokens, out=None):
        """tokens: int32 CUDA [B, T].  Returns fp32 logits [B, V] of the last positions."""
        import torch
        B, T = tokens.shape
        if out is None:
            out = torch.empty((B, self.cfg.vocab), dtype=torch.float32, device="cuda")
        _check(_lib.nc_prefill(self._h, _ptr(tokens), B, T, _ptr(out), _stream()), "nc_prefill")
        return out

    def decode_step(self, tokens, out=None):
        """tokens: int32 CUDA [B] at the next position.  Returns fp32 logits [B, V]."""
        import torch
        B = tokens.shape[0]
        if out is None:
            out = torch.empty((B, self.cfg.vocab), dtype=torch.float32, device="cuda")
        _check(_lib.nc_decode_step(self._h, _ptr(tokens), B, _ptr(out), _stream()), "nc_decode_step")
        return out

    def kv_cache_length(self):
        return int(_lib.nc_kv_cache_length(self._h))

    def last_launch_count(self):
        return int(_lib.nc_last_launch_count(self._h))

    def unpack(self, flat):
        """Dict name -> [rows, cols] view of a packed vector (torch or numpy)."""
        return {n: flat[o:o + r * c].reshape(r, c) for n, r, c, o in self.layout}


# ---------------------------------------------------------------- kernel-level ops
class ops:
    """Single-kernel entry points on torch CUDA tensors (for parity tests)."""

    @staticmethod
    def gemm(A, a_kmajor, B, b_kmajor, M, N, K, D, ep=EP_STORE, aux=None, dtype=None, workspace=None):
        dt = _dtype_code(A) if dtype is None else dtype
        lda = A.stride(0)
        ldb = B.stride(0)
        ldd = D.stride(0)
        ldaux = aux.stride(0) if aux is not None else 0
        wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(_lib.nc_op_gemm(dt, M, N, K, _ptr(A), lda, int(a_kmajor), _ptr(B), ldb, int(b_kmajor), ep,
                               _ptr(D), ldd, _ptr(aux), ldaux, _ptr(workspace), wsb, _stream()), "nc_op_gemm")

    @staticmethod
    def gemm_workspace_bytes():
        return int(_lib.nc_gemm_workspace_bytes())

    @staticmethod
    def rmsnorm_fwd(x, y, rstd, eps):
        rows, C = x.shape
        _check(_lib.nc_op_rmsnorm_fwd(_dtype_code(y), rows, C, _ptr(x), _ptr(y), _ptr(rstd), eps, _stream()),
               "nc_op_rmsnorm_fwd")

    @staticmethod
    def rmsnorm_bwd(dy, y, rstd, dx, dx_act=None):
        rows, C = dy.shape
        _check(_lib.nc_op_rmsnorm_bwd(_dtype_code(y), rows, C, _ptr(dy), _ptr(y), _ptr(rstd), _ptr(dx),
                                      _ptr(dx_act), _stream()), "nc_op_rmsnorm_bwd")

    @staticmethod
    def rope_table(T, hd, base, out):
        _check(_lib.nc_op_rope_table(T, hd, base, _ptr(out), _stream()), "nc_op_rope_table")

    @staticmethod
    def rope_qknorm_fwd(qkv, B, T, H, Hkv, hd, rstd, table, eps):
        _check(_lib.nc_op_rope_qknorm_fwd(_dtype_code(qkv), B, T, H, Hkv, hd, _ptr(qkv), _ptr(rstd), _ptr(table),
                                          eps, _stream()), "nc_op_rope_qknorm_fwd")

    @staticmethod
    def gemm_qkv_rope(x, wqkv, qkv, T, H, Hkv, hd, rstd, table, eps, pair_rows=0):
        M, K = x.shape
        _check(_lib.nc_op_gemm_qkv_rope(M, K, T, H, Hkv, hd, _ptr(x), x.stride(0), _ptr(wqkv), _ptr(qkv),
                                        qkv.stride(0), _ptr(rstd), _ptr(table), pair_rows, eps, _stream()),
               "nc_op_gemm_qkv_rope")

    @staticmethod
    def rope_table_pairs(T, hd, base, pairs):
        _check(_lib.nc_op_rope_table_pairs(T, hd, base, _ptr(pairs), _stream()), "nc_op_rope_table_pairs")

    @staticmethod
    def rope_qknorm_bwd(dqkv, qkv, B, T, H, Hkv, hd, rstd, table):
        _check(_lib.nc_op_rope_qknorm_bwd(_dtype_code(qkv), B, T, H, Hkv, hd, _ptr(dqkv), _ptr(qkv), _ptr(rstd),
                                          _ptr(table), _stream()), "nc_op_rope_qknorm_bwd")

    @staticmethod
    def attention_fwd(qkv, B, T, H, Hkv, hd, o, lse):
        _check(_lib.nc_op_attention_fwd(_dtype_code(qkv), B, T, H, Hkv, hd, _ptr(qkv), _ptr(o), _ptr(lse),
                                        _stream()), "nc_op_attention_fwd")

    @staticmethod
    def attention_bwd(qkv, o, lse, do, B, T, H, Hkv, hd, dqkv, ws):
        _check(_lib.nc_op_attention_bwd(_dtype_code(qkv), B, T, H, Hkv, hd, _ptr(qkv), _ptr(o), _ptr(lse),
                                        _ptr(do), _ptr(dqkv), _ptr(ws), _stream()), "nc_op_attention_bwd")

    @staticmethod
    def attention_bwd_rope(qkv, o, lse, do, B, T, H, Hkv, hd, dqkv, workspace, rstd, table, pair_rows=0):
        _check(_lib.nc_op_attention_bwd_rope(B, T, H, Hkv, hd, _ptr(qkv), _ptr(o), _ptr(lse), _ptr(do), _ptr(dqkv),
                                             _ptr(workspace), _ptr(rstd), _ptr(table), pair_rows, _stream()),
               "nc_op_attention_bwd_rope")

    @staticmethod
    def cross_entropy(z, targets, row_loss, scale, err=None):
        rows, V = z.shape
        _check(_lib.nc_op_cross_entropy(_dtype_code(z), rows, V, _ptr(z), _ptr(targets), _ptr(row_loss), scale,
                                        _ptr(err), _stream()), "nc_op_cross_entropy")

    @staticmethod
    def cross_entropy_softcap(z, targets, row_loss, scale, softcap, err=None):
        rows, V = z.shape
        _check(_lib.nc_op_cross_entropy_softcap(_dtype_code(z), rows, V, _ptr(z), _ptr(targets), _ptr(row_loss),
                                                scale, softcap, _ptr(err), _stream()), "nc_op_cross_entropy_softcap")

    @staticmethod
    def embed_fwd(tokens, wte, x, dtype, err=None):
        V, C = wte.shape
        _check(_lib.nc_op_embed_fwd(dtype, tokens.numel(), C, V, _ptr(tokens), _ptr(wte), _ptr(x), _ptr(err),
                                    _stream()), "nc_op_embed_fwd")

    @staticmethod
    def gemm_rows(A, W, D, ep=EP_STORE_F32):
        """D[m, n] (op)= sum_k A[m, k] W[n, k] for at most 32 rows (CUDA-core skinny GEMM)."""
        M, K = A.shape
        N = W.shape[0]
        _check(_lib.nc_op_gemm_rows(_dtype_code(A), M, N, K, _ptr(A), A.stride(0), _ptr(W), W.stride(0), ep, _ptr(D),
                                    D.stride(0), _stream()), "nc_op_gemm_rows")

    @staticmethod
    def quantize_fp8(x, codes=None, stats=None):
        """Per-tensor E4M3 codes of x (fp32 / bf16, contiguous): returns (codes uint8, stats fp32[3] =
        amax, scale, scale_inv), both on x's device."""
        import torch
        if codes is None:
            codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        if stats is None:
            stats = torch.empty(3, dtype=torch.float32, device=x.device)
        _check(_lib.nc_op_quantize_fp8(_dtype_code(x), _ptr(x), x.numel(), _ptr(codes), _ptr(stats), _stream()),
               "nc_op_quantize_fp8")
        return codes, stats

    @staticmethod
    def gemm_fp8(a8, b8, a_scale_inv, b_scale_inv, D):
        """D[m, n] = a_scale_inv b_scale_inv sum_k a8[m, k] b8[n, k]; a8, b8 uint8 E4M3 codes (row-major, K
        innermost); the scales are one-element fp32 device tensors (views); D bf16 or fp32."""
        M, K = a8.shape
        N = b8.shape[0]
        _check(_lib.nc_op_gemm_fp8(M, N, K, _ptr(a8), a8.stride(0), _ptr(b8), b8.stride(0), _ptr(a_scale_inv),
                                   _ptr(b_scale_inv), _dtype_code(D), _ptr(D), D.stride(0), _stream()),
               "nc_op_gemm_fp8")

    @staticmethod
    def newton_schulz(u, x, steps=5, dtype=None, workspace=None):
        """x (float [rows, cols]) = Newton-Schulz orthogonalisation of u in `dtype`."""
        import torch
        rows, cols = u.shape
        d = NC_BF16 if dtype in (None, "bf16", NC_BF16) else NC_FP32
        if workspace is None:
            nb = int(_lib.nc_newton_schulz_workspace_bytes(d, rows, cols))
            workspace = torch.empty(nb, dtype=torch.uint8, device="cuda")
        _check(_lib.nc_op_newton_schulz(d, rows, cols, steps, _ptr(u), _ptr(x), _ptr(workspace), _stream()),
               "nc_op_newton_schulz")

    @staticmethod
    def embed_bwd_scratch_bytes(n, C, V):
        return int(_lib.nc_embed_bwd_scratch_bytes(n, C, V))

    @staticmethod
    def embed_bwd(tokens, dx, dwte, scratch):
        n, C = dx.shape
        V = dwte.shape[0]
        _check(_lib.nc_op_embed_bwd(n, C, V, _ptr(tokens), _ptr(dx), _ptr(dwte), _ptr(scratch), _stream()),
               "nc_op_embed_bwd")


def version():
    return _lib.nc_version().decode()
