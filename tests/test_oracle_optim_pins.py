"""Pins of the optimizer oracle (``oracle/optim.py``) to facts outside it, and
planted mistakes that those pins must catch.

* The Newton-Schulz iteration is a matrix polynomial in U U^T, so it acts on
  the singular values alone: for U = P diag(s) Q^T the result must be
  P diag(q(s / ||s||)) Q^T with q the quintic applied five times to a scalar.
* The published coefficients make the result approximately orthogonal:
  every singular value of the output of a full-rank input lies near 1.
* With a constant gradient the momentum buffer has the closed form
  G (1 - mu^t) / (1 - mu), and since the iteration ignores the scale of its
  input every Muon step moves W by the same lr * sqrt(max(1, rows/cols)) X.
* AdamW's bias correction makes the first step (and every step of a
  constant gradient) move each weight by lr * g / (|g| + eps), and with a zero
  gradient the decoupled decay scales W by (1 - lr wd).
"""
import numpy as np
import pytest

from oracle import model as M
from oracle import optim as O


def _orthonormal(n, k, seed):
    q, r = np.linalg.qr(np.random.default_rng(seed).standard_normal((n, k)))
    return q * np.sign(np.diag(r))


def _quintic_scalar(s, steps=5):
    a, b, c = 3.4445, -4.7750, 2.0315     # the published Muon coefficients
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


@pytest.mark.parametrize("shape", [(8, 20), (20, 8), (12, 12)])
def test_newton_schulz_acts_on_singular_values(shape):
    r, c = shape
    k = min(r, c)
    P, Q = _orthonormal(r, k, 1), _orthonormal(c, k, 2)
    s = 7.0 * np.geomspace(1.0, 1e-3, k)
    U = (P * s) @ Q.T
    want = (P * _quintic_scalar(s / (np.linalg.norm(s) + 1e-7))) @ Q.T
    got = O.newton_schulz(U)
    assert got.shape == U.shape
    assert np.max(np.abs(got - want)) < 1e-12


def test_newton_schulz_output_is_nearly_orthogonal():
    for shape, seed in (((32, 96), 3), ((96, 32), 4), ((64, 64), 5)):
        G = np.random.default_rng(seed).standard_normal(shape)
        sv = np.linalg.svd(O.newton_schulz(G), compute_uv=False)
        assert sv.min() > 0.5 and sv.max() < 1.5, (shape, sv.min(), sv.max())
        # and the input's singular vectors are kept: X and G are positively aligned
        assert np.sum(O.newton_schulz(G) * G) > 0


@pytest.mark.parametrize("shape", [(6, 15), (15, 6)])
def test_muon_momentum_closed_form_and_aspect_scale(shape):
    rng = np.random.default_rng(6)
    G = rng.standard_normal(shape)
    W0 = rng.standard_normal(shape)
    W, Mb = W0.copy(), np.zeros(shape)
    mu, lr = 0.95, 0.02
    X = O.newton_schulz(G)
    scale = np.sqrt(max(1.0, shape[0] / shape[1]))
    for t in range(1, 5):
        W, Mb = O.muon_matrix(W, G, Mb, lr, mu, True, 5)
        assert np.allclose(Mb, G * (1 - mu ** t) / (1 - mu), rtol=1e-13, atol=0)
        # U is a positive multiple of G; the 1e-7 in the normalisation makes the
        # iteration scale-invariant only to ~1e-8 per step
        assert np.allclose(W, W0 - t * lr * scale * X, rtol=0, atol=1e-7)


def test_muon_without_nesterov_uses_the_buffer():
    rng = np.random.default_rng(7)
    G1, G2 = rng.standard_normal((5, 9)), rng.standard_normal((5, 9))
    W = np.zeros((5, 9))
    W, Mb = O.muon_matrix(W, G1, np.zeros((5, 9)), 1.0, 0.9, False, 5)
    W, Mb = O.muon_matrix(W, G2, Mb, 1.0, 0.9, False, 5)
    assert np.allclose(W, -O.newton_schulz(G1) - O.newton_schulz(0.9 * G1 + G2), atol=1e-12)


def test_adamw_closed_forms():
    rng = np.random.default_rng(8)
    W0, g = rng.standard_normal(50), rng.standard_normal(50)
    lr, eps, wd = 0.1, 1e-8, 0.01
    m = v = np.zeros(50)
    W1, m, v = O.adamw(W0, g, m, v, 1, lr, 0.9, 0.999, eps, wd)
    assert np.allclose(W1, W0 - lr * (g / (np.abs(g) + eps) + wd * W0), rtol=0, atol=1e-14)
    W2, m, v = O.adamw(W1, g, m, v, 2, lr, 0.9, 0.999, eps, wd)
    assert np.allclose(W2, W1 - lr * (g / (np.abs(g) + eps) + wd * W1), rtol=0, atol=1e-13)
    W3, _, _ = O.adamw(W0, np.zeros(50), np.zeros(50), np.zeros(50), 1, lr, 0.9, 0.999, eps, wd)
    assert np.allclose(W3, W0 * (1 - lr * wd), rtol=1e-15, atol=0)


def _tiny():
    return M.Config(depth=2, n_embd=8, n_head=2, n_kv_head=1, head_dim=4, mlp_hidden=32, vocab=11)


def test_optimizer_step_routes_each_tensor():
    cfg = _tiny()
    rng = np.random.default_rng(9)
    P = rng.standard_normal(M.n_params(cfg))
    Gr = rng.standard_normal(M.n_params(cfg))
    oc = O.OptimConfig()
    st = O.new_state(cfg)
    out = O.optimizer_step(cfg, P, Gr, st, oc, lr_mult=0.5)
    for name, r, c, off in M.param_layout(cfg):
        W0 = P[off:off + r * c].reshape(r, c)
        g = Gr[off:off + r * c].reshape(r, c)
        W1 = out[off:off + r * c].reshape(r, c)
        if name in ("wte", "lm_head"):
            lr = 0.5 * (oc.embedding_lr if name == "wte" else oc.unembedding_lr)
            assert np.allclose(W1, W0 - lr * g / (np.abs(g) + oc.adam_eps), atol=1e-14), name
        else:
            lr = 0.5 * oc.matrix_lr * np.sqrt(max(1.0, r / c))
            assert np.allclose(W1, W0 - lr * O.newton_schulz(g), atol=1e-12), name
    assert st["t"] == 1


# ---------------------------------------------------------------- planted mistakes

def _ns_coeffs_reversed(U, steps=5, coeffs=O.NS_COEFFS, eps=1e-7):
    return O.__dict__["_orig_newton_schulz"](U, steps, coeffs[::-1], eps)


def _ns_no_normalisation(U, steps=5, coeffs=O.NS_COEFFS, eps=1e-7):
    a, b, c = coeffs
    X = np.asarray(U, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    X = X.T if tall else X
    for _ in range(steps):
        A = X @ X.T
        X = a * X + (b * A + c * A @ A) @ X
    return X.T if tall else X


def _ns_four_steps(U, steps=5, coeffs=O.NS_COEFFS, eps=1e-7):
    return O.__dict__["_orig_newton_schulz"](U, steps - 1, coeffs, eps)


def _muon_inverted_scale(W, G, Mb, lr, momentum=0.95, nesterov=True, steps=5):
    W2, M2 = O.__dict__["_orig_muon_matrix"](W, G, Mb, lr, momentum, nesterov, steps)
    r, c = np.shape(G)
    return W - (W - W2) * np.sqrt(max(1.0, r / c)) ** -1 * np.sqrt(max(1.0, c / r)), M2


def _muon_buffer_not_decayed(W, G, Mb, lr, momentum=0.95, nesterov=True, steps=5):
    W2, M2 = O.__dict__["_orig_muon_matrix"](W, G, Mb, lr, 1.0, nesterov, steps)
    return W2, M2


def _adam_no_bias_correction(W, G, m, v, t, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0):
    m = beta1 * np.asarray(m) + (1 - beta1) * np.asarray(G)
    v = beta2 * np.asarray(v) + (1 - beta2) * np.asarray(G) ** 2
    return np.asarray(W) - lr * (m / (np.sqrt(v) + eps) + weight_decay * np.asarray(W)), m, v


MUTANTS = {
    "ns coefficients reversed": ("newton_schulz", _ns_coeffs_reversed),
    "ns without normalisation": ("newton_schulz", _ns_no_normalisation),
    "ns four steps": ("newton_schulz", _ns_four_steps),
    "muon aspect scale inverted": ("muon_matrix", _muon_inverted_scale),
    "muon momentum not decayed": ("muon_matrix", _muon_buffer_not_decayed),
    "adam without bias correction": ("adamw", _adam_no_bias_correction),
}

PINS = [
    lambda: [test_newton_schulz_acts_on_singular_values(s) for s in ((8, 20), (20, 8), (12, 12))],
    test_newton_schulz_output_is_nearly_orthogonal,
    lambda: [test_muon_momentum_closed_form_and_aspect_scale(s) for s in ((6, 15), (15, 6))],
    test_muon_without_nesterov_uses_the_buffer,
    test_adamw_closed_forms,
    test_optimizer_step_routes_each_tensor,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_optimizer_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setitem(O.__dict__, "_orig_" + attr, getattr(O, attr))
    monkeypatch.setattr(O, attr, fn)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, FloatingPointError, np.linalg.LinAlgError):
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake '{name}'"
