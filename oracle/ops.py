"""Single-operation definitions used by the kernel-level parity tests.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Each is the plain
definition in fp64; the whole-step oracle in ``model.py`` applies the same
definitions inline.  Every function is pinned in
``tests/test_oracle_ops_pins.py`` against a statement that shares no code with
it (explicit loops, conservation, exact special cases), on non-square shapes
so that a transposed operand or a wrong axis fails.
"""
import numpy as np


def gemm(a, b):
    """D[m, n] = sum_k A[m, k] B[n, k] (a bias-free linear layer is gemm(x, W)).

    Pin: an explicit triple loop; identity and column-selecting weights; an
    exact integer case."""
    return np.asarray(a, dtype=np.float64) @ np.asarray(b, dtype=np.float64).T


def relu2(u):
    """relu(u)^2 and relu(u) (cosmicrealm "noao-chat-0-项目总体介绍" §2.1 item 4)."""
    r = np.maximum(np.asarray(u, dtype=np.float64), 0.0)
    return r * r, r


def relu2_bwd(dh, r):
    """d/du of relu(u)^2 is 2 relu(u).  Pin: exact values, and central
    differences in ``tests/test_oracle_pins.py``."""
    return np.asarray(dh, dtype=np.float64) * 2.0 * np.asarray(r, dtype=np.float64)


def relu2_bwd_from_square(dh, h):
    """The same derivative written with h = relu(u)^2: relu(u) = sqrt(h), since relu(u) >= 0."""
    return np.asarray(dh, dtype=np.float64) * 2.0 * np.sqrt(np.asarray(h, dtype=np.float64))


def embed(wte, tokens):
    """Row tokens[...] of the embedding table (cosmicrealm "noao-chat-0-项目总体介绍"
    §2.1 item 3).  Pin: a per-position lookup loop."""
    return np.asarray(wte)[np.asarray(tokens)]


def embed_bwd(tokens, dx, vocab):
    """Sum of dx rows per token id; ids not present get zero rows.

    Pin: a per-position accumulation loop; column conservation
    (sum_v dwte[v] = sum_n dx[n]); the adjoint identity
    <embed(wte), dx> = <wte, embed_bwd(dx)>."""
    tokens = np.asarray(tokens).reshape(-1)
    dx = np.asarray(dx, dtype=np.float64).reshape(tokens.size, -1)
    out = np.zeros((vocab, dx.shape[1]))
    np.add.at(out, tokens, dx)
    return out
