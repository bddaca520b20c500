"""Pins of the oracle's 8-bit training step (``Config(fp8=True)``).

The reading (woshipm nanochat analysis §一.2 and §六.2 name FP8 without a
recipe): each block's four linear layers multiply E4M3 operands, the bf16
activation and the fp32 master weight, each quantised per tensor with
current scaling (one tensor [Wq; Wk; Wv] for the fused projection); the
input-gradient products dX = dY W multiply E4M3 operands as well (dY's bf16
value with its own per-tensor scale, W with its forward codes), and so do the
weight-gradient products dW = dY^T X (dY with those codes, X with its forward
codes); the quantisers pass gradients through unchanged.

Pins from outside the oracle:
* with the quantiser and the bf16 rounding replaced by identities the step is
  the fp64 step (the hooks sit in the four forward products only, and the
  backward is the fp64 one);
* per-tensor scaling makes the quantised model exactly invariant when wte,
  Wo and Wproj are scaled by a power of two (the codes do not change, the
  dequantisation factors scale exactly, and the norms remove the scale);
* every quantised product lies within the E4M3 error bound of the exact one;
* the 8-bit step's loss stays close to the fp64 loss;
* the input-gradient products dX = dY w and the weight-gradient products
  dW = dY^T x are E4M3 too (dY with its own per-tensor scale): within the same
  bound, and scaling the loss by a power of two scales every gradient exactly.
Planted mistakes in the dequantisation and in the scaling of dY are caught.
"""
import numpy as np
import pytest

from oracle import fp8 as F8
from oracle import model as M


def small_cfg(**kw):
    base = dict(depth=2, n_embd=16, n_head=2, n_kv_head=1, head_dim=8, mlp_hidden=64, vocab=13, fp8=True)
    base.update(kw)
    return M.Config(**base)


def rand_params(cfg, seed, std=0.3):
    return np.random.default_rng(seed).normal(0.0, std, size=M.n_params(cfg)).astype(np.float32).astype(np.float64)


def rand_tokens(cfg, B, T, seed):
    g = np.random.default_rng(seed)
    return g.integers(0, cfg.vocab, size=(B, T)), g.integers(0, cfg.vocab, size=(B, T))


def test_identity_quantiser_gives_the_fp64_step(monkeypatch):
    cfg8 = small_cfg()
    cfg = small_cfg(fp8=False)
    params = rand_params(cfg, 41)
    tok, tgt = rand_tokens(cfg, 2, 6, 42)
    l0, G0 = M.forward_backward(cfg, params, tok, tgt)
    monkeypatch.setattr(M, "quantize_dequantize", lambda x: np.asarray(x, dtype=np.float64))
    monkeypatch.setattr(M, "bf16_round", lambda x: np.asarray(x, dtype=np.float64))
    l8, G8 = M.forward_backward(cfg8, params, tok, tgt)
    assert l8 == pytest.approx(l0, rel=1e-12)
    for k in G0:
        np.testing.assert_allclose(G8[k], G0[k], rtol=1e-9, atol=1e-13)


def test_power_of_two_scaling_leaves_the_8bit_model_unchanged():
    cfg = small_cfg(norm_eps=0.0)
    W = M.unpack(cfg, rand_params(cfg, 43))
    tok, _ = rand_tokens(cfg, 2, 7, 44)
    for k in (3, -2):
        W2 = {n: (v * 2.0 ** k if (n == "wte" or n.endswith(".wo") or n.endswith(".wproj")) else v)
              for n, v in W.items()}
        assert np.array_equal(M.forward_logits(cfg, W, tok), M.forward_logits(cfg, W2, tok))
    # a scale that is not a power of two changes the codes of those weights
    W3 = {n: (v * 3.0 if n.endswith(".wo") else v) for n, v in W.items()}
    assert not np.array_equal(M.forward_logits(cfg, W, tok), M.forward_logits(cfg, W3, tok))


def test_quantised_product_within_the_e4m3_bound():
    """|lin8(x, w) - x w^T| <= sum_k |x||w| ((1 + 2^-9)(1 + 2^-4)^2 - 1) + the
    subnormal quanta: each operand is within half a quantum, 2^-4 relative for
    E4M3 normals and 2^-10 / scale absolute for subnormals, and the activation
    first rounds to bf16 (2^-9)."""
    rng = np.random.default_rng(45)
    cfg = small_cfg()
    x = rng.normal(0.0, 1.0, size=(37, 48)) * np.exp(rng.normal(0.0, 1.0, size=(37, 1)))
    w = rng.normal(0.0, 0.05, size=(29, 48)).astype(np.float32).astype(np.float64)
    got = M.linear(cfg, x, w)
    exact = x @ w.T
    _, _, xs, _ = F8.quantize(M.bf16_round(x).astype(np.float32))
    _, _, ws, _ = F8.quantize(w.astype(np.float32))
    qx, qw = 2.0 ** -10 / float(xs), 2.0 ** -10 / float(ws)      # half of a subnormal quantum, in value units
    ax, aw = np.abs(x), np.abs(w)
    rel = (1 + 2.0 ** -9) * (1 + 2.0 ** -4) ** 2 - 1
    bound = rel * (ax @ aw.T) + qx * (1 + 2.0 ** -4) * aw.sum(axis=1)[None, :] + \
        qw * (1 + 2.0 ** -4) * ax.sum(axis=1)[:, None] * (1 + 2.0 ** -9) + qx * qw * x.shape[1]
    err = np.abs(got - exact)
    assert np.all(err <= bound)
    # and the quantisation is really there: errors of the order of 2^-4 relative
    assert np.median(err / (ax @ aw.T)) > 2.0 ** -9


def test_8bit_step_loss_close_to_fp64():
    """E4M3 operands carry ~2^-5 relative rms error each; at std-0.1 weights the
    loss moves by about 1e-2, far inside 0.05, and every gradient keeps its
    direction; a wrong dequantisation factor moves them by orders of magnitude."""
    cfg = small_cfg()
    params = rand_params(cfg, 46, std=0.1)
    tok, tgt = rand_tokens(cfg, 2, 8, 47)
    l8, G8 = M.forward_backward(cfg, params, tok, tgt)
    l0, G0 = M.forward_backward(small_cfg(fp8=False), params, tok, tgt)
    assert abs(l8 - l0) < 0.05 and l8 != l0
    for k in G0:
        a, b = G8[k].ravel(), G0[k].ravel()
        assert a @ b / (np.linalg.norm(a) * np.linalg.norm(b)) > 0.95, k


def test_quantised_input_gradient_within_the_e4m3_bound():
    """dX = dY w with both operands E4M3 (dY from its bf16 value): within the same bound as the forward product."""
    rng = np.random.default_rng(48)
    cfg = small_cfg()
    dy = rng.normal(0.0, 1e-3, size=(41, 29)) * np.exp(rng.normal(0.0, 1.0, size=(41, 1)))
    w = rng.normal(0.0, 0.05, size=(29, 48)).astype(np.float32).astype(np.float64)
    got = M.linear_dx(cfg, dy, w)
    exact = dy @ w
    _, _, ys, _ = F8.quantize(M.bf16_round(dy).astype(np.float32))
    _, _, ws, _ = F8.quantize(w.astype(np.float32))
    qy, qw = 2.0 ** -10 / float(ys), 2.0 ** -10 / float(ws)
    ay, aw = np.abs(dy), np.abs(w)
    rel = (1 + 2.0 ** -9) * (1 + 2.0 ** -4) ** 2 - 1
    bound = rel * (ay @ aw) + qy * (1 + 2.0 ** -4) * aw.sum(axis=0)[None, :] + \
        qw * (1 + 2.0 ** -4) * ay.sum(axis=1)[:, None] * (1 + 2.0 ** -9) + qy * qw * dy.shape[1]
    err = np.abs(got - exact)
    assert np.all(err <= bound)
    assert np.median(err / (ay @ aw)) > 2.0 ** -9


def test_quantised_weight_gradient_within_the_e4m3_bound():
    """dW = dY^T x with both operands E4M3 (dY and x from their bf16 values): the
    bound of the forward product with the token sum as the contraction."""
    rng = np.random.default_rng(51)
    cfg = small_cfg()
    dy = rng.normal(0.0, 1e-3, size=(53, 29)) * np.exp(rng.normal(0.0, 1.0, size=(53, 1)))
    x = rng.normal(0.0, 1.0, size=(53, 48)) * np.exp(rng.normal(0.0, 1.0, size=(53, 1)))
    got = M.linear_dw(cfg, dy, x)
    exact = dy.T @ x
    _, _, ys, _ = F8.quantize(M.bf16_round(dy).astype(np.float32))
    _, _, xs, _ = F8.quantize(M.bf16_round(x).astype(np.float32))
    qy, qx = 2.0 ** -10 / float(ys), 2.0 ** -10 / float(xs)
    ay, ax = np.abs(dy), np.abs(x)
    rel = (1 + 2.0 ** -9) ** 2 * (1 + 2.0 ** -4) ** 2 - 1
    bound = rel * (ay.T @ ax) + qy * (1 + 2.0 ** -4) * (1 + 2.0 ** -9) * ax.sum(axis=0)[None, :] + \
        qx * (1 + 2.0 ** -4) * (1 + 2.0 ** -9) * ay.sum(axis=0)[:, None] + qy * qx * dy.shape[0]
    err = np.abs(got - exact)
    assert np.all(err <= bound)
    assert np.median(err / (ay.T @ ax)) > 2.0 ** -9
    # and it is the plain product without the 8-bit reading
    assert np.array_equal(M.linear_dw(small_cfg(fp8=False), dy, x), exact)


def test_weight_gradient_lies_on_the_e4m3_product_grid():
    """Every E4M3 value is a multiple of 2^-9 (the subnormal step), so a sum of
    products of two of them is a multiple of 2^-18: dW divided by both
    dequantisation factors lands on that grid (to fp64 rounding), which a dW
    with either operand left unquantised does not."""
    rng = np.random.default_rng(52)
    cfg = small_cfg()
    dy = rng.normal(0.0, 1e-3, size=(37, 21))
    x = rng.normal(0.0, 1.0, size=(37, 19))
    _, _, _, siy = F8.quantize(M.bf16_round(dy).astype(np.float32))
    _, _, _, six = F8.quantize(M.bf16_round(x).astype(np.float32))
    v = M.linear_dw(cfg, dy, x) / (float(siy) * float(six)) * 2.0 ** 18
    assert np.max(np.abs(v - np.round(v))) < 1e-3
    assert np.max(np.abs(v)) > 1e6          # far from trivially small


def test_gradient_scale_by_a_power_of_two_is_exact():
    """Current (per-tensor) scaling of every dY: scaling the loss by 2^k scales
    every dY by 2^k, which leaves its codes unchanged and its factor exact, so
    the 8-bit step's gradients are exactly 2^k times; a factor of 3 changes the
    codes and the gradients are not exactly 3 times."""
    cfg = small_cfg()
    params = rand_params(cfg, 49, std=0.1)
    tok, tgt = rand_tokens(cfg, 2, 6, 50)
    _, G1 = M.forward_backward(cfg, params, tok, tgt)
    _, G8 = M.forward_backward(cfg, params, tok, tgt, grad_scale=2.0 ** 5)
    for k in G1:
        assert np.array_equal(G8[k], G1[k] * 2.0 ** 5), k
    _, G3 = M.forward_backward(cfg, params, tok, tgt, grad_scale=3.0)
    assert any(not np.allclose(G3[k], 3.0 * G1[k], rtol=1e-9, atol=0) for k in G1 if not k.startswith("lm_head"))


# ---------------------------------------------------------------- planted mistakes

def _dequantise_with_scale(x):
    codes, _, scale, _ = F8.quantize(x)
    return F8.e4m3_decode(codes) * float(scale)


def _no_dequantisation(x):
    codes, _, _, _ = F8.quantize(x)
    return F8.e4m3_decode(codes)


def _linear_dx_fixed_scale(cfg, dy, w):
    """dY quantised with a fixed unit scale instead of its own maximum."""
    if not cfg.fp8:
        return dy @ w
    codes = F8.e4m3_encode(np.clip(M.bf16_round(dy).astype(np.float32), -448, 448))
    return F8.e4m3_decode(codes) @ M.quantize_dequantize(w)


def _linear_dw_fixed_scale(cfg, dy, x):
    """dY quantised with a fixed unit scale in the weight gradient."""
    if not cfg.fp8:
        return dy.T @ x
    codes = F8.e4m3_encode(np.clip(M.bf16_round(dy).astype(np.float32), -448, 448))
    return F8.e4m3_decode(codes).T @ M.quantize_dequantize(M.bf16_round(x))


def _linear_dw_x_unquantised(cfg, dy, x):
    """The weight gradient with x left at its bf16 value."""
    if not cfg.fp8:
        return dy.T @ x
    return M.quantize_dequantize(M.bf16_round(dy)).T @ M.bf16_round(x)


MUTANTS = {"dequantised with the scale": ("quantize_dequantize", _dequantise_with_scale),
           "codes used without their factor": ("quantize_dequantize", _no_dequantisation),
           "input gradient with a fixed scale": ("linear_dx", _linear_dx_fixed_scale),
           "weight gradient with a fixed scale": ("linear_dw", _linear_dw_fixed_scale),
           "weight gradient with x unquantised": ("linear_dw", _linear_dw_x_unquantised)}

PINS = [test_power_of_two_scaling_leaves_the_8bit_model_unchanged, test_quantised_product_within_the_e4m3_bound,
        test_8bit_step_loss_close_to_fp64, test_quantised_input_gradient_within_the_e4m3_bound,
        test_quantised_weight_gradient_within_the_e4m3_bound, test_weight_gradient_lies_on_the_e4m3_product_grid,
        test_gradient_scale_by_a_power_of_two_is_exact]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_8bit_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(M, attr, fn)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake '{name}'"
