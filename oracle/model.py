"""Plain fp64 forward and hand-written backward of one GPT training step.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Slow on purpose: every
operation is the textbook definition, matrix products go through NumPy's
``@`` (BLAS dgemm), attention loops over batch rows and heads, and nothing is
fused or reordered.

Readings of the pages used here (each is repeated where it applies):

* pre-norm residual block ``x += attn(norm(x)); x += mlp(norm(x))`` and a final
  ``norm`` before ``lm_head``: the pages say "standard decoder block with
  normalisation" (devpress §4.1) for a GPT-2-lineage model;
* no normalisation directly after the embedding lookup (not in the block
  description);
* RoPE frequencies ``omega_i = base**(-2 i / hd)`` for pair ``i`` of the
  half-split layout, ``base = 10000`` (the pages give only the rotation);
* attention scale ``1/sqrt(hd)`` with a causal mask;
* GQA query head ``h`` reads key/value head ``h // (H / Hkv)``;
* RMSNorm ``eps`` is a config field, float32 machine epsilon by default;
* cross-entropy is the mean over all B*T positions, no ignore index;
* two variants, both off by default: the pages' "logit stabilisation"
  (woshipm nanochat analysis §三.3 item 1) read as the tanh soft-cap
  ``z <- c tanh(z / c)`` on the lm_head output (``logit_softcap = c > 0``),
  and a parameter-free RMSNorm right after the embedding lookup
  (``embed_norm``).
"""
from dataclasses import dataclass

import numpy as np

from . import fp8 as _fp8

FLT_EPSILON = float(np.finfo(np.float32).eps)


@dataclass(frozen=True)
class Config:
    depth: int
    n_embd: int
    n_head: int
    n_kv_head: int
    head_dim: int
    mlp_hidden: int
    vocab: int
    rope_base: float = 10000.0
    norm_eps: float = FLT_EPSILON
    init_std: float = 0.02
    logit_softcap: float = 0.0      # c > 0: logits z <- c * tanh(z / c) before the loss
    embed_norm: bool = False        # RMSNorm of the embedding rows before the first block
    fp8: bool = False               # the blocks' four linear layers multiply E4M3 operands (forward)

    @staticmethod
    def from_workload(w, **kw):
        return Config(w.depth, w.n_embd, w.n_head, w.n_kv_head, w.head_dim,
                      w.mlp_hidden, w.vocab, **kw)


def param_layout(cfg):
    """Packed parameter order: (name, rows, cols, offset) per tensor.

    Linear weights are stored ``W[out, in]`` and applied as ``y = x W^T``
    (bias-free, cosmicrealm "noao-chat-0" §2.1 item 5).  The embedding and the
    output head are separate tensors (untied, §2.1 item 3).
    """
    C, H, Hkv, hd, F, V = (cfg.n_embd, cfg.n_head, cfg.n_kv_head, cfg.head_dim,
                           cfg.mlp_hidden, cfg.vocab)
    shapes = [("wte", V, C)]
    for l in range(cfg.depth):
        shapes += [(f"h{l}.wq", H * hd, C), (f"h{l}.wk", Hkv * hd, C),
                   (f"h{l}.wv", Hkv * hd, C), (f"h{l}.wo", C, H * hd),
                   (f"h{l}.wfc", F, C), (f"h{l}.wproj", C, F)]
    shapes.append(("lm_head", V, C))
    out, off = [], 0
    for name, r, c in shapes:
        out.append((name, r, c, off))
        off += r * c
    return out


def n_params(cfg):
    return sum(r * c for _, r, c, _ in param_layout(cfg))


def unpack(cfg, flat):
    """Dict of fp64 matrices (copies) from a packed vector."""
    return {name: np.array(flat[off:off + r * c], dtype=np.float64).reshape(r, c)
            for name, r, c, off in param_layout(cfg)}


def pack(cfg, mats):
    flat = np.zeros(n_params(cfg), dtype=np.float64)
    for name, r, c, off in param_layout(cfg):
        flat[off:off + r * c] = mats[name].reshape(-1)
    return flat


# --------------------------------------------------------------------------
# RMSNorm without gain: y = x / sqrt(mean(x^2) + eps) over the last axis.
# cosmicrealm "noao-chat-0" §2.1 item 5 (a functional rms_norm, no parameters).

def rms_norm(x, eps):
    """Returns (y, rstd) with rstd = 1/sqrt(mean(x^2) + eps) per row."""
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * rstd, rstd


def rms_norm_bwd(dy, y, rstd):
    """dx = rstd * (dy - y * mean(dy * y)), the derivative of ``rms_norm``."""
    return rstd * (dy - y * np.mean(dy * y, axis=-1, keepdims=True))


# --------------------------------------------------------------------------
# Rotary embedding by half-split rotation, cosmicrealm "noao-chat-0" §2.1
# item 1 and §5.3: with x1, x2 the two halves of a head vector,
# y1 = x1 cos + x2 sin and y2 = -x1 sin + x2 cos.

def rope_tables(T, hd, base):
    """cos, sin of theta[t, i] = t * base**(-2 i / hd), shapes [T, hd/2]."""
    d = hd // 2
    omega = base ** (-(2.0 * np.arange(d, dtype=np.float64)) / hd)
    theta = np.arange(T, dtype=np.float64)[:, None] * omega[None, :]
    return np.cos(theta), np.sin(theta)


def rope(x, cos, sin):
    """x: [..., T, hd]; cos, sin: [T, hd/2]."""
    d = x.shape[-1] // 2
    x1, x2 = x[..., :d], x[..., d:]
    return np.concatenate([x1 * cos + x2 * sin, -x1 * sin + x2 * cos], axis=-1)


def rope_bwd(dy, cos, sin):
    """Transpose of ``rope``: the rotation by the opposite angle."""
    d = dy.shape[-1] // 2
    dy1, dy2 = dy[..., :d], dy[..., d:]
    return np.concatenate([dy1 * cos - dy2 * sin, dy1 * sin + dy2 * cos], axis=-1)


# --------------------------------------------------------------------------
# Causal scaled-dot-product attention for one sequence and one head.

def attention(q, k, v):
    """q, k, v: [T, hd].  Returns (o [T, hd], lse [T]).

    s[t, u] = q_t . k_u / sqrt(hd) for u <= t, -inf otherwise;
    p = softmax over u; o = p v.  ``lse`` is the natural-log sum of
    exp(s) per query row.
    """
    T, hd = q.shape
    s = (q @ k.T) / np.sqrt(hd)
    s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=1, keepdims=True)
    p = e / z
    return p @ v, (m + np.log(z))[:, 0]


def attention_bwd(q, k, v, do):
    """Gradients (dq, dk, dv) of ``attention`` for upstream ``do``."""
    T, hd = q.shape
    scale = 1.0 / np.sqrt(hd)
    s = (q @ k.T) * scale
    s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    e = np.exp(s - np.max(s, axis=1, keepdims=True))
    p = e / np.sum(e, axis=1, keepdims=True)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - np.sum(dp * p, axis=1, keepdims=True))
    dq = (ds @ k) * scale
    dk = (ds.T @ q) * scale
    return dq, dk, dv


# --------------------------------------------------------------------------
# Next-token cross-entropy (devpress §2.2 item 2; cosmicrealm §6.2 snippet).

def cross_entropy(z, tgt):
    """z: [n, V] logits, tgt: [n].  Returns (per-row losses, dlogits of their sum)."""
    m = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - m)
    ssum = np.sum(e, axis=1, keepdims=True)
    lse = (m + np.log(ssum))[:, 0]
    rows = np.arange(z.shape[0])
    loss = lse - z[rows, tgt]
    dz = e / ssum
    dz[rows, tgt] -= 1.0
    return loss, dz


def bf16_round(x):
    """Round to bfloat16 (round to nearest, ties to even) through float32,
    returned as fp64: the top 16 bits of the float32 pattern after adding
    0x7fff plus the lowest kept bit (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def quantize_dequantize(x):
    """Per-tensor E4M3 quantisation (of the float32 values of x, which are
    exact for the bf16 activations and fp32 weights it receives) and the
    values it stands for: decode(codes) * scale_inv (``oracle/fp8.py``)."""
    codes, _, _, scale_inv = _fp8.quantize(x)
    return _fp8.e4m3_decode(codes) * float(scale_inv)


def linear(cfg, x, w):
    """A bias-free linear layer y = x w^T (w stored [out, in]).

    With cfg.fp8 (the 8-bit reading of woshipm nanochat analysis §一.2 / §六.2,
    which name FP8 without a recipe): both operands are quantised per tensor
    to E4M3 with current scaling, the activation from its bfloat16 value (the
    tensor the layer reads) and the weight from its float32 master value, and
    the product of the decoded values is taken exactly (fp32 accumulation on
    the device).  The gradient passes through each quantiser as the identity
    (straight-through); the backward's own products dX = dY w and
    dW = dY^T x multiply E4M3 operands too (``linear_dx``, ``linear_dw``).
    """
    if not cfg.fp8:
        return x @ w.T
    xq = quantize_dequantize(bf16_round(x))
    wq = quantize_dequantize(w)
    return xq @ wq.T


def linear_dx(cfg, dy, w):
    """The input gradient of ``linear``: dX = dY w.

    With cfg.fp8 both operands are E4M3 as well: the bf16 value of dY
    quantised per tensor with current scaling (its own absolute maximum), and
    the weight with the same codes and factor as in the forward (the same
    tensor, read transposed)."""
    if not cfg.fp8:
        return dy @ w
    return quantize_dequantize(bf16_round(dy)) @ quantize_dequantize(w)


def linear_dw(cfg, dy, x):
    """The weight gradient of ``linear``: dW = dY^T x (rows of dy and x are tokens).

    With cfg.fp8 both operands are E4M3: dY with the codes and factor of its
    input-gradient product (``linear_dx``), x with the codes and factor of the
    forward product (``linear``), so each tensor is quantised once; the
    products of the decoded values accumulate exactly (fp32 on the device)."""
    if not cfg.fp8:
        return dy.T @ x
    return quantize_dequantize(bf16_round(dy)).T @ quantize_dequantize(bf16_round(x))


def softcap(z, c):
    """Logit soft-cap: (c tanh(z / c), dzc/dz = 1 - tanh(z / c)^2); identity for c <= 0.

    The reading of woshipm nanochat analysis §三.3 item 1 ("logit
    stabilisation", not defined there): a smooth bound |z| < c on every logit.
    """
    if not c or c <= 0:
        return z, None
    t = np.tanh(z / c)
    return c * t, 1.0 - t * t


# --------------------------------------------------------------------------
# One block.  cosmicrealm §2.1 items 2, 4, 6 and devpress §4.1.

def _kv_head_of(cfg, h):
    return h // (cfg.n_head // cfg.n_kv_head)


def block_forward(cfg, W, l, x, cos, sin, keep=False):
    """x: [B, T, C] residual stream entering layer l; returns the stream leaving it."""
    B, T, C = x.shape
    H, Hkv, hd = cfg.n_head, cfg.n_kv_head, cfg.head_dim
    p = f"h{l}."
    a, rstd1 = rms_norm(x, cfg.norm_eps)
    if cfg.fp8:
        # one operand tensor [Wq; Wk; Wv] for the three projections, as multiplied together
        qkv = linear(cfg, a, np.concatenate([W[p + "wq"], W[p + "wk"], W[p + "wv"]], axis=0))
        q2, k2, v2 = np.split(qkv, [H * hd, (H + Hkv) * hd], axis=-1)
    else:
        q2, k2, v2 = a @ W[p + "wq"].T, a @ W[p + "wk"].T, a @ W[p + "wv"].T
    q = q2.reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    k = k2.reshape(B, T, Hkv, hd).transpose(0, 2, 1, 3)
    v = v2.reshape(B, T, Hkv, hd).transpose(0, 2, 1, 3)
    qr, kr = rope(q, cos, sin), rope(k, cos, sin)          # RoPE first ...
    qn, rq = rms_norm(qr, cfg.norm_eps)                     # ... then QK norm
    kn, rk = rms_norm(kr, cfg.norm_eps)
    o = np.empty((B, H, T, hd))
    for b in range(B):
        for h in range(H):
            g = _kv_head_of(cfg, h)
            o[b, h], _ = attention(qn[b, h], kn[b, g], v[b, g])
    o2 = o.transpose(0, 2, 1, 3).reshape(B, T, H * hd)
    x1 = x + linear(cfg, o2, W[p + "wo"])
    bn, rstd2 = rms_norm(x1, cfg.norm_eps)
    u = linear(cfg, bn, W[p + "wfc"])
    r = np.maximum(u, 0.0)
    hmid = r * r                                            # relu(u)^2
    x2 = x1 + linear(cfg, hmid, W[p + "wproj"])
    if not keep:
        return x2
    return x2, dict(a=a, rstd1=rstd1, qn=qn, kn=kn, rq=rq, rk=rk, v=v, o2=o2,
                    x1=x1, bn=bn, rstd2=rstd2, r=r, hmid=hmid)


def block_backward(cfg, W, l, x, dx2, cos, sin, G):
    """Backward of ``block_forward`` for layer l, recomputing its forward from x.

    Adds the weight gradients into G and returns d(loss)/dx.
    """
    B, T, C = x.shape
    H, Hkv, hd = cfg.n_head, cfg.n_kv_head, cfg.head_dim
    p = f"h{l}."
    _, s = block_forward(cfg, W, l, x, cos, sin, keep=True)
    N = B * T
    # MLP: x2 = x1 + relu(bn Wfc^T)^2 Wproj^T
    G[p + "wproj"] += linear_dw(cfg, dx2.reshape(N, C), s["hmid"].reshape(N, -1))
    dh = linear_dx(cfg, dx2, W[p + "wproj"])
    du = dh * 2.0 * s["r"]
    G[p + "wfc"] += linear_dw(cfg, du.reshape(N, -1), s["bn"].reshape(N, C))
    dbn = linear_dx(cfg, du, W[p + "wfc"])
    dx1 = dx2 + rms_norm_bwd(dbn, s["bn"], s["rstd2"])
    # attention output projection: x1 = x + o2 Wo^T
    G[p + "wo"] += linear_dw(cfg, dx1.reshape(N, C), s["o2"].reshape(N, -1))
    do2 = linear_dx(cfg, dx1, W[p + "wo"])
    do = do2.reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    dqn = np.zeros((B, H, T, hd))
    dkn = np.zeros((B, Hkv, T, hd))
    dv = np.zeros((B, Hkv, T, hd))
    for b in range(B):
        for h in range(H):
            g = _kv_head_of(cfg, h)
            dq_, dk_, dv_ = attention_bwd(s["qn"][b, h], s["kn"][b, g], s["v"][b, g], do[b, h])
            dqn[b, h] = dq_
            dkn[b, g] += dk_          # a shared kv head sums its group's gradients
            dv[b, g] += dv_
    dq = rope_bwd(rms_norm_bwd(dqn, s["qn"], s["rq"]), cos, sin)
    dk = rope_bwd(rms_norm_bwd(dkn, s["kn"], s["rk"]), cos, sin)
    dq2 = dq.transpose(0, 2, 1, 3).reshape(N, H * hd)
    dk2 = dk.transpose(0, 2, 1, 3).reshape(N, Hkv * hd)
    dv2 = dv.transpose(0, 2, 1, 3).reshape(N, Hkv * hd)
    a = s["a"].reshape(N, C)
    if cfg.fp8:   # one operand [dq | dk | dv], as the fused projection's weight gradient multiplies it
        gqkv = linear_dw(cfg, np.concatenate([dq2, dk2, dv2], axis=-1), a)
        nq, nk = dq2.shape[1], dk2.shape[1]
        G[p + "wq"] += gqkv[:nq]
        G[p + "wk"] += gqkv[nq:nq + nk]
        G[p + "wv"] += gqkv[nq + nk:]
    else:
        G[p + "wq"] += dq2.T @ a
        G[p + "wk"] += dk2.T @ a
        G[p + "wv"] += dv2.T @ a
    if cfg.fp8:   # one operand [dq | dk | dv] against [Wq; Wk; Wv], as the fused projection's backward multiplies them
        da = linear_dx(cfg, np.concatenate([dq2, dk2, dv2], axis=-1),
                       np.concatenate([W[p + "wq"], W[p + "wk"], W[p + "wv"]], axis=0))
    else:
        da = dq2 @ W[p + "wq"] + dk2 @ W[p + "wk"] + dv2 @ W[p + "wv"]
    return dx1 + rms_norm_bwd(da.reshape(B, T, C), s["a"], s["rstd1"])


# --------------------------------------------------------------------------
# Whole model.

def _embed(W, tokens):
    return W["wte"][tokens]


def embed_norm_bwd(cfg, W, tokens, dx):
    """Gradient with respect to the embedding rows e = wte[tok] of x0 = norm(e)."""
    y0, r0 = rms_norm(_embed(W, tokens), cfg.norm_eps)
    return rms_norm_bwd(dx, y0, r0)


def _trunk(cfg, W, tokens, keep_inputs):
    B, T = tokens.shape
    cos, sin = rope_tables(T, cfg.head_dim, cfg.rope_base)
    x = _embed(W, tokens)
    if cfg.embed_norm:
        x, _ = rms_norm(x, cfg.norm_eps)
    xs = []
    for l in range(cfg.depth):
        if keep_inputs:
            xs.append(x)
        x = block_forward(cfg, W, l, x, cos, sin)
    return x, xs, cos, sin


def forward_logits(cfg, params, tokens, rows=None):
    """fp64 logits [B, T, V] (or only the flat rows listed in ``rows``)."""
    W = unpack(cfg, params) if not isinstance(params, dict) else params
    x, _, _, _ = _trunk(cfg, W, np.asarray(tokens), False)
    xf, _ = rms_norm(x, cfg.norm_eps)
    B, T, C = xf.shape
    xf = xf.reshape(B * T, C)
    if rows is not None:
        return softcap(xf[np.asarray(rows)] @ W["lm_head"].T, cfg.logit_softcap)[0]
    return softcap(xf @ W["lm_head"].T, cfg.logit_softcap)[0].reshape(B, T, -1)


def row_losses(cfg, params, tokens, targets):
    """Per-position cross-entropy [B, T] (forward only)."""
    W = unpack(cfg, params) if not isinstance(params, dict) else params
    tokens, targets = np.asarray(tokens), np.asarray(targets)
    x, _, _, _ = _trunk(cfg, W, tokens, False)
    xf, _ = rms_norm(x, cfg.norm_eps)
    B, T, C = xf.shape
    xf = xf.reshape(B * T, C)
    t = targets.reshape(-1)
    out = np.empty(B * T)
    for a in range(0, B * T, 512):
        z, _ = softcap(xf[a:a + 512] @ W["lm_head"].T, cfg.logit_softcap)
        out[a:a + 512], _ = cross_entropy(z, t[a:a + 512])
    return out.reshape(B, T)


def forward_backward(cfg, params, tokens, targets, chunk=512, grad_scale=1.0):
    """Mean next-token cross-entropy and its gradient for every parameter.

    Returns (loss, grads) with grads a dict of fp64 matrices in layout order
    (use ``pack`` for the flat vector); the gradients are those of
    grad_scale * loss.  Only the residual stream entering each layer is kept;
    each layer's forward is recomputed in the backward.
    """
    W = unpack(cfg, params) if not isinstance(params, dict) else params
    tokens, targets = np.asarray(tokens), np.asarray(targets)
    B, T = tokens.shape
    N = B * T
    G = {k: np.zeros_like(v) for k, v in W.items()}
    x, xs, cos, sin = _trunk(cfg, W, tokens, True)
    xf, rstd = rms_norm(x, cfg.norm_eps)
    C = xf.shape[-1]
    xf2 = xf.reshape(N, C)
    t = targets.reshape(-1)
    total = 0.0
    dxf = np.empty((N, C))
    for a in range(0, N, chunk):
        z, dcap = softcap(xf2[a:a + chunk] @ W["lm_head"].T, cfg.logit_softcap)
        l_rows, dz = cross_entropy(z, t[a:a + chunk])
        total += float(np.sum(l_rows))
        dz *= grad_scale / N                      # the loss is a mean over B*T
        if dcap is not None:
            dz *= dcap                            # through the soft-cap
        G["lm_head"] += dz.T @ xf2[a:a + chunk]
        dxf[a:a + chunk] = dz @ W["lm_head"]
    dx = rms_norm_bwd(dxf.reshape(B, T, C), xf, rstd)
    for l in reversed(range(cfg.depth)):
        dx = block_backward(cfg, W, l, xs[l], dx, cos, sin, G)
    if cfg.embed_norm:
        dx = embed_norm_bwd(cfg, W, tokens, dx)
    np.add.at(G["wte"], tokens.reshape(-1), dx.reshape(N, C))
    return total / N, G
