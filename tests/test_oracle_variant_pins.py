"""Pins of the oracle's two off-by-default variants (woshipm nanochat analysis
§三.3 item 1, "logit stabilisation", read as the tanh soft-cap
z <- c tanh(z / c); and a parameter-free RMSNorm after the embedding lookup).

Each pin comes from outside the oracle: central finite differences of the
whole step, the limit c -> infinity (the uncapped model), the bound |z| < c,
the closed form ln V at zero logits, and the scale invariance that a norm
after the embedding adds.  The last tests plant mistakes in the variants'
backward and check that a pin catches each.
"""
import math

import numpy as np
import pytest

from oracle import model as M


def small_cfg(**kw):
    base = dict(depth=2, n_embd=8, n_head=2, n_kv_head=2, head_dim=4, mlp_hidden=32, vocab=11)
    base.update(kw)
    return M.Config(**base)


def rand_params(cfg, seed, std=0.5):
    return np.random.default_rng(seed).normal(0.0, std, size=M.n_params(cfg))


def rand_tokens(cfg, B, T, seed):
    g = np.random.default_rng(seed)
    return g.integers(0, cfg.vocab, size=(B, T)), g.integers(0, cfg.vocab, size=(B, T))


def _fd_check(cfg, seed):
    params = rand_params(cfg, seed)
    tok, tgt = rand_tokens(cfg, 2, 5, seed + 1)
    loss, G = M.forward_backward(cfg, params, tok, tgt)
    g = M.pack(cfg, G)
    h = 1e-6
    fd = np.empty_like(params)
    for i in range(params.size):
        old = params[i]
        params[i] = old + h
        lp = float(np.mean(M.row_losses(cfg, params, tok, tgt)))
        params[i] = old - h
        lm = float(np.mean(M.row_losses(cfg, params, tok, tgt)))
        params[i] = old
        fd[i] = (lp - lm) / (2 * h)
    scale = np.sqrt(np.mean(g * g))
    err = np.abs(fd - g) / np.maximum(np.abs(g), 1e-2 * scale)
    # central differences with h = 1e-6 carry a roundoff of about eps * |loss| / h
    # (~5e-10 absolute), up to ~1e-6 of the smallest gradients the floor admits;
    # a wrong or missing term is off by O(1)
    assert err.max() < 1e-5, (err.max(), int(err.argmax()))
    assert loss == pytest.approx(float(np.mean(M.row_losses(cfg, params, tok, tgt))), rel=1e-14)


@pytest.mark.parametrize("kw", [dict(logit_softcap=1.0), dict(embed_norm=True),
                                dict(logit_softcap=0.7, embed_norm=True, n_kv_head=1)],
                         ids=["softcap", "embed_norm", "both_gqa"])
def test_variant_step_central_finite_differences(kw):
    _fd_check(small_cfg(**kw), 31)


def test_softcap_function_values_and_derivative():
    z = np.array([-30.0, -2.0, -0.1, 0.0, 0.1, 2.0, 30.0])
    c = 3.0
    zc, d = M.softcap(z, c)
    assert np.all(np.abs(zc) < c) and zc[3] == 0.0
    np.testing.assert_allclose(zc, [c * math.tanh(v / c) for v in z], rtol=1e-15)
    h = 1e-6
    fd = (M.softcap(z + h, c)[0] - M.softcap(z - h, c)[0]) / (2 * h)
    np.testing.assert_allclose(d, fd, rtol=1e-8, atol=1e-10)   # FD roundoff ~ eps * c / h
    # odd, increasing, and the identity to first order at 0
    assert np.allclose(M.softcap(-z, c)[0], -zc) and np.all(np.diff(zc) > 0) and d[3] == 1.0
    # c <= 0 switches it off
    assert M.softcap(z, 0.0)[0] is z and M.softcap(z, 0.0)[1] is None


def test_softcap_limit_is_the_uncapped_model():
    cfg0 = small_cfg()
    cfgc = small_cfg(logit_softcap=1e6)
    params = rand_params(cfg0, 32)
    tok, tgt = rand_tokens(cfg0, 2, 6, 33)
    l0, G0 = M.forward_backward(cfg0, params, tok, tgt)
    lc, Gc = M.forward_backward(cfgc, params, tok, tgt)
    assert lc == pytest.approx(l0, rel=1e-10)
    for k in G0:
        np.testing.assert_allclose(Gc[k], G0[k], rtol=1e-8, atol=1e-12)


def test_softcap_bounds_logits_and_zero_head_gives_ln_vocab():
    cfg = small_cfg(logit_softcap=0.5)
    W = M.unpack(cfg, rand_params(cfg, 34, std=2.0))
    tok, tgt = rand_tokens(cfg, 2, 6, 35)
    z = M.forward_logits(cfg, W, tok)
    assert np.all(np.abs(z) <= 0.5) and np.abs(z).max() > 0.4     # large logits are squeezed to c (tanh rounds to 1 in fp64 past ~19)
    W["lm_head"][:] = 0.0
    loss, G = M.forward_backward(cfg, W, tok, tgt)
    assert loss == pytest.approx(math.log(cfg.vocab), rel=1e-15)
    assert all(np.all(G[k] == 0.0) for k in G if k != "lm_head")


def test_embed_norm_makes_the_model_invariant_to_the_embedding_scale():
    """With the norm after the lookup, wte -> a wte (a > 0) leaves every logit
    unchanged (exactly with eps = 0) and scales dwte by 1/a; without it the
    logits change."""
    for norm in (True, False):
        cfg = small_cfg(norm_eps=0.0, embed_norm=norm)
        W = M.unpack(cfg, rand_params(cfg, 36))
        tok, tgt = rand_tokens(cfg, 2, 5, 37)
        W2 = {k: (v * 4.0 if k == "wte" else v) for k, v in W.items()}
        same = np.allclose(M.forward_logits(cfg, W, tok), M.forward_logits(cfg, W2, tok), rtol=1e-12, atol=1e-14)
        assert same == norm
        if norm:
            _, G = M.forward_backward(cfg, W, tok, tgt)
            _, G2 = M.forward_backward(cfg, W2, tok, tgt)
            np.testing.assert_allclose(G2["wte"], G["wte"] / 4.0, rtol=1e-10, atol=1e-15)
            for k in G:
                if k != "wte":
                    np.testing.assert_allclose(G2[k], G[k], rtol=1e-10, atol=1e-15)


def test_embed_norm_rows_have_unit_rms():
    cfg = small_cfg(depth=1, embed_norm=True, norm_eps=0.0)
    W = M.unpack(cfg, rand_params(cfg, 38))
    tok, _ = rand_tokens(cfg, 1, 6, 39)
    x0 = M.rms_norm(M._embed(W, tok), 0.0)[0]
    np.testing.assert_allclose(np.sqrt(np.mean(x0 * x0, axis=-1)), 1.0, rtol=1e-14)


# ---------------------------------------------------------------- planted mistakes

def _softcap_no_derivative(z, c):
    zc, _ = M.__dict__["_orig_softcap"](z, c)
    return zc, (None if _ is None else np.ones_like(zc))


def _softcap_wrong_derivative(z, c):
    zc, d = M.__dict__["_orig_softcap"](z, c)
    return zc, (None if d is None else 1.0 - (zc / c))


def _embed_norm_bwd_dropped(cfg, W, tokens, dx):
    return dx


MUTANTS = {
    "softcap backward without its factor": ("softcap", _softcap_no_derivative),
    "softcap derivative 1 - t": ("softcap", _softcap_wrong_derivative),
    "embedding norm backward dropped": ("embed_norm_bwd", _embed_norm_bwd_dropped),
}

PINS = [
    lambda: test_variant_step_central_finite_differences(dict(logit_softcap=1.0)),
    lambda: test_variant_step_central_finite_differences(dict(embed_norm=True)),
    test_softcap_function_values_and_derivative,
    test_embed_norm_makes_the_model_invariant_to_the_embedding_scale,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_variant_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setitem(M.__dict__, "_orig_" + attr, getattr(M, attr))
    monkeypatch.setattr(M, attr, fn)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake '{name}'"
