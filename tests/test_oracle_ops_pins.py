"""Pins for the single-operation definitions in ``oracle/ops.py``.

The kernel-level parity tests compare CUDA kernels with these functions, so
each is checked here against a statement of the same operation that shares no
code with it: explicit Python loops on small cases, conservation laws, and
special cases with a known answer.  Shapes are non-square throughout, so that a
transposed operand or a wrong axis changes the result (or fails outright).
The second half plants such mistakes and checks that a pin catches each.
"""
import numpy as np
import pytest

from oracle import ops as OO


def _loop_gemm(a, b):
    """D[m][n] = sum_k A[m][k] * B[n][k], one scalar product at a time
    (a bias-free linear layer y = x W^T, W stored [out][in]: cosmicrealm
    "noao-chat-0-项目总体介绍" §2.1 item 5)."""
    M, K = len(a), len(a[0])
    N = len(b)
    out = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += float(a[m][k]) * float(b[n][k])
            out[m][n] = s
    return np.array(out)


def test_gemm_matches_explicit_triple_loop():
    rng = np.random.default_rng(11)
    for M, N, K in ((3, 5, 7), (1, 4, 2), (6, 2, 9)):
        a = rng.standard_normal((M, K))
        b = rng.standard_normal((N, K))
        got = OO.gemm(a, b)
        assert got.shape == (M, N)
        np.testing.assert_allclose(got, _loop_gemm(a.tolist(), b.tolist()), rtol=1e-13, atol=1e-13)


def test_gemm_special_cases():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((4, 6))
    # a linear layer with the identity weight returns its input
    np.testing.assert_array_equal(OO.gemm(x, np.eye(6)), x)
    # a weight that picks input column j into output column i
    W = np.zeros((3, 6))
    W[0, 5] = W[1, 0] = W[2, 2] = 1.0
    np.testing.assert_array_equal(OO.gemm(x, W), x[:, [5, 0, 2]])
    # exact small integers: [[1,2],[3,4]] times W^T with W = [[1,0],[1,1],[0,2]]
    got = OO.gemm(np.array([[1.0, 2.0], [3.0, 4.0]]), np.array([[1.0, 0.0], [1.0, 1.0], [0.0, 2.0]]))
    np.testing.assert_array_equal(got, [[1.0, 3.0, 4.0], [3.0, 7.0, 8.0]])


def test_embed_matches_row_lookup_loop():
    rng = np.random.default_rng(13)
    V, C = 9, 5
    wte = rng.standard_normal((V, C))
    tokens = np.array([[3, 0, 8, 3], [1, 1, 7, 2]], dtype=np.int32)
    got = OO.embed(wte, tokens)
    assert got.shape == (2, 4, C)
    for b in range(2):
        for t in range(4):
            np.testing.assert_array_equal(got[b, t], wte[tokens[b, t]])


def _loop_embed_bwd(tokens, dx, vocab):
    """dwte[v] = sum of dx[i] over positions i holding id v, one position at a time."""
    C = len(dx[0])
    out = [[0.0] * C for _ in range(vocab)]
    for i, v in enumerate(tokens):
        for c in range(C):
            out[v][c] += float(dx[i][c])
    return np.array(out)


def test_embed_bwd_matches_per_token_loop_and_conserves_columns():
    rng = np.random.default_rng(14)
    V, C, n = 11, 3, 40
    tokens = rng.integers(0, V, size=n).astype(np.int32)
    tokens[:5] = 4                                 # a repeated id
    tokens[tokens == 9] = 0                        # an id that never occurs
    dx = rng.standard_normal((n, C))
    got = OO.embed_bwd(tokens, dx, V)
    assert got.shape == (V, C)
    np.testing.assert_allclose(got, _loop_embed_bwd(tokens.tolist(), dx.tolist(), V), rtol=1e-13, atol=1e-13)
    # conservation: every position's gradient lands in exactly one row
    np.testing.assert_allclose(got.sum(axis=0), dx.sum(axis=0), rtol=1e-12, atol=1e-12)
    # rows of absent ids are exactly zero
    assert np.all(got[9] == 0.0)
    # the derivative of the gather: <embed(wte), dx> = <wte, embed_bwd(dx)> for every wte
    wte = rng.standard_normal((V, C))
    lhs = float(np.sum(OO.embed(wte, tokens) * dx))
    rhs = float(np.sum(wte * got))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_embed_bwd_accepts_batch_shaped_tokens():
    rng = np.random.default_rng(15)
    tokens = np.array([[2, 2, 0], [1, 2, 4]], dtype=np.int32)
    dx = rng.standard_normal((2, 3, 4))
    got = OO.embed_bwd(tokens, dx, 5)
    np.testing.assert_allclose(got[2], dx[0, 0] + dx[0, 1] + dx[1, 1], rtol=1e-14)
    np.testing.assert_allclose(got[4], dx[1, 2], rtol=1e-14)
    assert np.all(got[3] == 0.0)


def test_relu2_and_its_backward_forms():
    u = np.array([-2.0, -0.5, 0.0, 0.25, 3.0])
    h, r = OO.relu2(u)
    np.testing.assert_array_equal(r, [0.0, 0.0, 0.0, 0.25, 3.0])
    np.testing.assert_array_equal(h, [0.0, 0.0, 0.0, 0.0625, 9.0])
    dh = np.array([1.0, 2.0, 3.0, 4.0, 5.0])
    np.testing.assert_array_equal(OO.relu2_bwd(dh, r), [0.0, 0.0, 0.0, 2.0, 30.0])
    np.testing.assert_array_equal(OO.relu2_bwd_from_square(dh, h), [0.0, 0.0, 0.0, 2.0, 30.0])


# ---------------------------------------------------------------- planted mistakes

def _gemm_transposed_b(a, b):
    return np.asarray(a, dtype=np.float64) @ np.asarray(b, dtype=np.float64)


def _gemm_swapped(a, b):
    return (np.asarray(b, dtype=np.float64) @ np.asarray(a, dtype=np.float64).T).T.T


def _embed_bwd_wrong_axis(tokens, dx, vocab):
    tokens = np.asarray(tokens).reshape(-1)
    dx = np.asarray(dx, dtype=np.float64).reshape(tokens.size, -1)
    out = np.zeros((vocab, dx.shape[1]))
    np.add.at(out.T, tokens % dx.shape[1], dx.T)
    return out


def _embed_bwd_last_write_wins(tokens, dx, vocab):
    tokens = np.asarray(tokens).reshape(-1)
    dx = np.asarray(dx, dtype=np.float64).reshape(tokens.size, -1)
    out = np.zeros((vocab, dx.shape[1]))
    out[tokens] += dx                              # repeated ids keep only one position
    return out


def _embed_off_by_one(wte, tokens):
    return np.asarray(wte)[(np.asarray(tokens) + 1) % np.asarray(wte).shape[0]]


OPS_MUTANTS = {
    "gemm without the transpose": ("gemm", _gemm_transposed_b),
    "gemm operands swapped": ("gemm", _gemm_swapped),
    "embed_bwd on the wrong axis": ("embed_bwd", _embed_bwd_wrong_axis),
    "embed_bwd drops repeated ids": ("embed_bwd", _embed_bwd_last_write_wins),
    "embed off by one row": ("embed", _embed_off_by_one),
}

OPS_PINS = [
    test_gemm_matches_explicit_triple_loop,
    test_gemm_special_cases,
    test_embed_matches_row_lookup_loop,
    test_embed_bwd_matches_per_token_loop_and_conserves_columns,
    test_embed_bwd_accepts_batch_shaped_tokens,
]


@pytest.mark.parametrize("name", sorted(OPS_MUTANTS))
def test_planted_ops_mistake_is_caught(name, monkeypatch):
    attr, fn = OPS_MUTANTS[name]
    monkeypatch.setattr(OO, attr, fn)
    failed = 0
    for pin in OPS_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake '{name}'"
