"""The optimizer step that follows the gradients, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It shares no code with
the CUDA path.

What the pages fix (cosmicrealm "noao-chat-0-项目总体介绍" §2.2 and §4.2;
woshipm nanochat analysis §六.1): the transformer's weight matrices are
updated by Muon, the embedding and the output head by AdamW, with learning
rates 0.02 (matrices), 0.2 (embedding) and 0.004 (output head) and a warmup +
cosine schedule applied on top.  Muon is SGD with momentum whose update is
orthogonalised by a Newton-Schulz iteration and then scaled by a factor that
depends on the matrix's aspect ratio.

What they leave open, and the reading taken here (the published methods):

* Muon (Jordan et al., "Muon: an optimizer for hidden layers in neural
  networks", 2024): momentum mu = 0.95 with the Nesterov form U = G + mu M of
  the buffer M <- mu M + G; the iteration starts from X = U / (||U||_F + 1e-7),
  works on the wide orientation (rows <= cols, transposing a tall matrix), and
  repeats X <- a X + (b A + c A^2) X with A = X X^T five times, with the
  quintic's coefficients (a, b, c) = (3.4445, -4.7750, 2.0315); the step is
  W <- W - lr * sqrt(max(1, rows / cols)) * X.
* AdamW (Loshchilov & Hutter, "Decoupled weight decay regularization", 2019):
  m <- b1 m + (1 - b1) g, v <- b2 v + (1 - b2) g^2, bias-corrected by
  1 - b^t, W <- W - lr (m_hat / (sqrt(v_hat) + eps) + wd W), with the Adam
  paper's b1 = 0.9, b2 = 0.999, eps = 1e-8 and wd = 0 by default.
* The schedule's value at a step is the caller's: every learning rate is
  multiplied by ``lr_mult``.
"""
from dataclasses import dataclass

import numpy as np

from .model import param_layout

NS_COEFFS = (3.4445, -4.7750, 2.0315)


@dataclass(frozen=True)
class OptimConfig:
    matrix_lr: float = 0.02
    embedding_lr: float = 0.2
    unembedding_lr: float = 0.004
    momentum: float = 0.95
    nesterov: bool = True
    ns_steps: int = 5
    beta1: float = 0.9
    beta2: float = 0.999
    adam_eps: float = 1e-8
    weight_decay: float = 0.0


def newton_schulz(U, steps=5, coeffs=NS_COEFFS, eps=1e-7):
    """Approximately orthogonalise U: every singular value s of U / ||U||_F is
    mapped through the quintic p(s) = a s + b s^3 + c s^5 `steps` times while the
    singular vectors are kept.  Tall matrices are iterated on their transpose."""
    a, b, c = coeffs
    X = np.asarray(U, dtype=np.float64)
    X = X / (np.linalg.norm(X) + eps)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tall else X


def muon_matrix(W, G, M, lr, momentum=0.95, nesterov=True, steps=5):
    """One Muon step on one weight matrix W[out, in] with gradient G and
    momentum buffer M.  Returns (new W, new M)."""
    G = np.asarray(G, dtype=np.float64)
    M = momentum * np.asarray(M, dtype=np.float64) + G
    U = G + momentum * M if nesterov else M
    rows, cols = G.shape
    scale = np.sqrt(max(1.0, rows / cols))
    return np.asarray(W, dtype=np.float64) - lr * scale * newton_schulz(U, steps), M


def adamw(W, G, m, v, t, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0):
    """One AdamW step (t counts from 1).  Returns (new W, new m, new v)."""
    W = np.asarray(W, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * G
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * G * G
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    return W - lr * (m_hat / (np.sqrt(v_hat) + eps) + weight_decay * W), m, v


def new_state(cfg):
    """Zero optimizer state for the packed parameter vector: a momentum buffer
    per matrix, Adam moments for wte and lm_head, and the step count."""
    st = {"t": 0}
    for name, r, c, _ in param_layout(cfg):
        if name in ("wte", "lm_head"):
            st[name + ".m"] = np.zeros((r, c))
            st[name + ".v"] = np.zeros((r, c))
        else:
            st[name + ".M"] = np.zeros((r, c))
    return st


def optimizer_step(cfg, params, grads, state, oc=OptimConfig(), lr_mult=1.0):
    """Apply one step to the packed fp64 parameter vector `params` given the
    packed gradient; `state` (from new_state) is updated in place.  Returns the
    new packed parameters."""
    out = np.array(params, dtype=np.float64)
    state["t"] += 1
    t = state["t"]
    for name, r, c, off in param_layout(cfg):
        W = out[off:off + r * c].reshape(r, c)
        G = np.asarray(grads[off:off + r * c], dtype=np.float64).reshape(r, c)
        if name in ("wte", "lm_head"):
            lr = (oc.embedding_lr if name == "wte" else oc.unembedding_lr) * lr_mult
            W2, state[name + ".m"], state[name + ".v"] = adamw(
                W, G, state[name + ".m"], state[name + ".v"], t, lr, oc.beta1, oc.beta2, oc.adam_eps,
                oc.weight_decay)
        else:
            W2, state[name + ".M"] = muon_matrix(W, G, state[name + ".M"], oc.matrix_lr * lr_mult, oc.momentum,
                                                 oc.nesterov, oc.ns_steps)
        out[off:off + r * c] = W2.reshape(-1)
    return out
