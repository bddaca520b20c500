"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a value the pages print, a closed form, an
invariant of the mathematics, or central finite differences.  They are chosen
so that a dropped term, a wrong sign or index, or a transposed operand in any
oracle function fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import model as M
from oracle import rng as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_cfg(**kw):
    base = dict(depth=2, n_embd=8, n_head=2, n_kv_head=2, head_dim=4,
                mlp_hidden=32, vocab=11)
    base.update(kw)
    return M.Config(**base)


def rand_params(cfg, seed, std=0.5):
    g = np.random.default_rng(seed)
    return g.normal(0.0, std, size=M.n_params(cfg))


def rand_tokens(cfg, B, T, seed):
    g = np.random.default_rng(seed)
    return g.integers(0, cfg.vocab, size=(B, T)), g.integers(0, cfg.vocab, size=(B, T))


# ---------------------------------------------------------------- RNG

def test_splitmix64_published_vectors():
    want = [int(l) for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt"))
            if l.strip() and not l.startswith("#")]
    got = [int(x) for x in R.splitmix64_outputs(1234567, 5)]
    assert got == want


def test_splitmix64_offset_continues_stream():
    a = R.splitmix64_outputs(99, 10)
    b = R.splitmix64_outputs(99, 4, start=6)
    assert np.array_equal(a[6:], b)


def test_box_muller_closed_form_and_moments():
    # top 24 bits = 2^23 -> u1 = (2^23 + 0.5)/2^24; bits 16..39 = 0 -> u2 = 0.5/2^24
    w = np.array([np.uint64(1) << np.uint64(63)], dtype=np.uint64)
    u1 = (2.0 ** 23 + 0.5) / 2.0 ** 24
    u2 = 0.5 / 2.0 ** 24
    want = math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2)
    assert R.box_muller(w)[0] == pytest.approx(want, rel=1e-15)
    z = R.normal_init(5, 3, 1 << 20, 0.02)
    assert z.dtype == np.float32
    assert abs(z.mean()) < 0.02 * 5 / 1024
    assert abs(z.std() / 0.02 - 1) < 5e-3
    # tensors use different streams
    assert not np.array_equal(R.normal_init(5, 3, 64, 1.0), R.normal_init(5, 4, 64, 1.0))


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_unit_rms_and_scale_invariance():
    x = np.random.default_rng(0).normal(size=(7, 33)) * 3.0
    y, rstd = M.rms_norm(x, 1e-6)
    ms = np.mean(x * x, axis=1)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(ms / (ms + 1e-6)), rtol=1e-14)
    y2, _ = M.rms_norm(2.5 * x, 0.0)
    y1, _ = M.rms_norm(x, 0.0)
    assert np.allclose(y1, y2, rtol=1e-14)
    assert np.allclose(rstd[:, 0], 1 / np.sqrt(ms + 1e-6))


def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = f()
        x[i] = old - h
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


def test_rms_norm_bwd_matches_fd():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(3, 6))
    w = rng.normal(size=(3, 6))
    f = lambda: float(np.sum(w * M.rms_norm(x, 1e-3)[0]))
    y, rstd = M.rms_norm(x, 1e-3)
    assert np.allclose(M.rms_norm_bwd(w, y, rstd), _fd(f, x), rtol=1e-7, atol=1e-9)


# ---------------------------------------------------------------- RoPE

def test_rope_golden_unit_pair():
    """Sign convention of the half-split rotation, from the pages' formula."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "rope_unit_pair.txt"))
            if l.strip() and not l.startswith("#")]
    cos, sin = M.rope_tables(4, 2, 10000.0)
    for t, x1, x2, y1, y2 in rows:
        t = int(t)
        x = np.zeros((4, 2))
        x[t] = [float(x1), float(x2)]
        y = M.rope(x, cos, sin)
        assert y[t] == pytest.approx([float(y1), float(y2)], abs=1e-15)


def test_rope_identity_at_zero_norm_and_relative_position():
    hd, T = 16, 9
    cos, sin = M.rope_tables(T, hd, 10000.0)
    rng = np.random.default_rng(2)
    x = rng.normal(size=(T, hd))
    y = M.rope(x, cos, sin)
    assert np.array_equal(y[0], x[0])
    d = hd // 2
    assert np.allclose(x[:, :d] ** 2 + x[:, d:] ** 2, y[:, :d] ** 2 + y[:, d:] ** 2, rtol=1e-14)
    q, k = rng.normal(size=hd), rng.normal(size=hd)
    Q, K = M.rope(np.tile(q, (T, 1)), cos, sin), M.rope(np.tile(k, (T, 1)), cos, sin)
    # <R_m q, R_n k> depends only on m - n
    assert Q[5] @ K[3] == pytest.approx(Q[4] @ K[2], rel=1e-12)
    assert Q[8] @ K[1] == pytest.approx(Q[7] @ K[0], rel=1e-12)
    # frequencies: pair i at position 1 turns by base**(-2i/hd)
    assert np.allclose(np.arccos(cos[1]), 10000.0 ** (-2 * np.arange(d) / hd), rtol=1e-10)


def test_rope_bwd_is_inverse_and_commutes_with_norm():
    hd, T = 8, 6
    cos, sin = M.rope_tables(T, hd, 500.0)
    x = np.random.default_rng(3).normal(size=(2, T, hd))
    assert np.allclose(M.rope_bwd(M.rope(x, cos, sin), cos, sin), x, atol=1e-14)
    # RoPE is orthogonal, so QK-norm after it equals QK-norm before it
    a = M.rms_norm(M.rope(x, cos, sin), 1e-6)[0]
    b = M.rope(M.rms_norm(x, 1e-6)[0], cos, sin)
    assert np.allclose(a, b, atol=1e-13)


# ---------------------------------------------------------------- attention

def test_attention_T1_returns_v_and_constant_keys_give_running_mean():
    rng = np.random.default_rng(4)
    q, k, v = rng.normal(size=(1, 8)), rng.normal(size=(1, 8)), rng.normal(size=(1, 8))
    o, lse = M.attention(q, k, v)
    assert np.array_equal(o, v)
    assert lse[0] == pytest.approx(float(q[0] @ k[0]) / math.sqrt(8), rel=1e-14)
    T = 7
    q = rng.normal(size=(T, 8))
    k = np.tile(rng.normal(size=(1, 8)), (T, 1))
    v = rng.normal(size=(T, 8))
    o, lse = M.attention(q, k, v)
    want = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.allclose(o, want, rtol=1e-13, atol=1e-14)
    # constant scores: lse = s + ln(t + 1)
    s = (q @ k[0]) / math.sqrt(8)
    assert np.allclose(lse, s + np.log(np.arange(1, T + 1)), rtol=1e-13)


def test_attention_is_causal():
    rng = np.random.default_rng(5)
    q, k, v = (rng.normal(size=(6, 4)) for _ in range(3))
    o1, _ = M.attention(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[4:] += 10.0
    v2[4:] -= 3.0
    o2, _ = M.attention(q, k2, v2)
    assert np.array_equal(o1[:4], o2[:4])
    assert not np.allclose(o1[4:], o2[4:])


def test_attention_bwd_matches_fd():
    rng = np.random.default_rng(6)
    q, k, v = (rng.normal(size=(5, 4)) for _ in range(3))
    w = rng.normal(size=(5, 4))
    f = lambda: float(np.sum(w * M.attention(q, k, v)[0]))
    dq, dk, dv = M.attention_bwd(q, k, v, w)
    for got, x in ((dq, q), (dk, k), (dv, v)):
        assert np.allclose(got, _fd(f, x), rtol=1e-7, atol=1e-9)


# ---------------------------------------------------------------- cross-entropy

def test_cross_entropy_zero_logits_and_row_sums():
    z = np.zeros((3, 512))
    loss, dz = M.cross_entropy(z, np.array([0, 7, 511]))
    assert np.allclose(loss, math.log(512), rtol=0, atol=1e-15)
    z = np.random.default_rng(7).normal(size=(4, 9))
    t = np.array([1, 2, 8, 0])
    loss, dz = M.cross_entropy(z, t)
    assert np.allclose(dz.sum(axis=1), 0.0, atol=1e-15)
    want = np.log(np.exp(z).sum(axis=1)) - z[np.arange(4), t]
    assert np.allclose(loss, want, rtol=1e-14)
    f = lambda: float(np.sum(M.cross_entropy(z, t)[0]))
    assert np.allclose(dz, _fd(f, z), rtol=1e-7, atol=1e-9)


def test_zero_lm_head_gives_ln_vocab_and_only_head_grad():
    cfg = small_cfg()
    W = M.unpack(cfg, rand_params(cfg, 8))
    W["lm_head"][:] = 0.0
    tok, tgt = rand_tokens(cfg, 2, 5, 9)
    loss, G = M.forward_backward(cfg, W, tok, tgt)
    assert loss == pytest.approx(math.log(cfg.vocab), abs=1e-15)
    for name, g in G.items():
        if name == "lm_head":
            assert np.abs(g).max() > 0
        else:
            assert np.all(g == 0.0), name


# ---------------------------------------------------------------- MLP (relu^2)

def test_relu_squared_mlp_properties():
    cfg = small_cfg(depth=1)
    W = M.unpack(cfg, rand_params(cfg, 10))
    x = np.random.default_rng(11).normal(size=(1, 5, cfg.n_embd))
    cos, sin = M.rope_tables(5, cfg.head_dim, cfg.rope_base)

    def mlp_delta(Wfc):
        W2 = dict(W)
        W2["h0.wfc"] = Wfc
        out, s = M.block_forward(cfg, W2, 0, x, cos, sin, keep=True)
        return out - s["x1"], s

    d_pos, s = mlp_delta(W["h0.wfc"])
    d_neg, _ = mlp_delta(-W["h0.wfc"])
    u = s["bn"] @ W["h0.wfc"].T
    # relu(u)^2 + relu(-u)^2 = u^2: the two halves add up to the pure square
    assert np.allclose(d_pos + d_neg, (u * u) @ W["h0.wproj"].T, rtol=1e-12, atol=1e-13)
    # degree-2 homogeneity in Wfc
    d2, _ = mlp_delta(3.0 * W["h0.wfc"])
    assert np.allclose(d2, 9.0 * d_pos, rtol=1e-12, atol=1e-13)


def test_relu_squared_derivative_single_ops():
    """The single-op definitions the GEMM epilogues are checked against: relu2
    returns (relu(u)^2, relu(u)); both backward forms equal the central
    difference of relu(u)^2 (away from the kink at 0)."""
    from oracle import ops as O
    u = np.random.default_rng(14).normal(size=200)
    u = u[np.abs(u) > 1e-3]
    dh = np.random.default_rng(15).normal(size=u.size)
    h, r = O.relu2(u)
    assert np.array_equal(r, np.where(u > 0, u, 0.0)) and np.array_equal(h, r * r)
    eps = 1e-6
    fd = dh * ((np.maximum(u + eps, 0) ** 2 - np.maximum(u - eps, 0) ** 2) / (2 * eps))
    assert np.allclose(O.relu2_bwd(dh, r), fd, rtol=1e-7, atol=1e-9)
    assert np.allclose(O.relu2_bwd_from_square(dh, h), fd, rtol=1e-7, atol=1e-9)
    assert np.all(O.relu2_bwd_from_square(dh, h)[u < 0] == 0.0)


# ---------------------------------------------------------------- whole step

@pytest.mark.parametrize("shape", [dict(n_kv_head=2), dict(n_kv_head=1),
                                   # three query heads per kv head, as in the d24 GQA workload
                                   dict(depth=1, n_embd=12, n_head=3, n_kv_head=1, mlp_hidden=48)],
                         ids=["mha", "gqa2", "gqa3"])
def test_whole_step_central_finite_differences(shape):
    cfg = small_cfg(**shape)
    params = rand_params(cfg, 12)
    tok, tgt = rand_tokens(cfg, 2, 5, 13)
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
    assert err.max() < 1e-6, (err.max(), int(err.argmax()))
    assert loss == pytest.approx(float(np.mean(M.row_losses(cfg, params, tok, tgt))), rel=1e-14)


def test_gqa_equals_mha_with_repeated_kv_heads():
    g_cfg = small_cfg(n_head=4, n_kv_head=2, n_embd=16, mlp_hidden=64)
    m_cfg = small_cfg(n_head=4, n_kv_head=4, n_embd=16, mlp_hidden=64)
    Wg = M.unpack(g_cfg, rand_params(g_cfg, 14))
    hd = g_cfg.head_dim
    Wm = {}
    for k, v in Wg.items():
        if k.endswith(".wk") or k.endswith(".wv"):
            heads = v.reshape(2, hd, -1)
            Wm[k] = np.repeat(heads, 2, axis=0).reshape(4 * hd, -1)   # kv head g serves q heads 2g, 2g+1
        else:
            Wm[k] = v.copy()
    tok, tgt = rand_tokens(g_cfg, 2, 6, 15)
    lg, Gg = M.forward_backward(g_cfg, Wg, tok, tgt)
    lm, Gm = M.forward_backward(m_cfg, Wm, tok, tgt)
    assert lg == pytest.approx(lm, rel=1e-13)
    for k in Gg:
        if k.endswith(".wk") or k.endswith(".wv"):
            summed = Gm[k].reshape(2, 2, hd, -1).sum(axis=1).reshape(2 * hd, -1)
            assert np.allclose(Gg[k], summed, rtol=1e-10, atol=1e-13), k
        else:
            assert np.allclose(Gg[k], Gm[k], rtol=1e-10, atol=1e-13), k


def test_gqa_three_groups_equals_mha_with_repeated_kv_heads():
    """Three query heads per kv head (the d24 GQA grouping): kv head g serves q heads 3g .. 3g+2."""
    g_cfg = small_cfg(n_head=6, n_kv_head=2, n_embd=24, mlp_hidden=96, depth=1)
    m_cfg = small_cfg(n_head=6, n_kv_head=6, n_embd=24, mlp_hidden=96, depth=1)
    Wg = M.unpack(g_cfg, rand_params(g_cfg, 18))
    hd = g_cfg.head_dim
    Wm = {}
    for k, v in Wg.items():
        if k.endswith(".wk") or k.endswith(".wv"):
            Wm[k] = np.repeat(v.reshape(2, hd, -1), 3, axis=0).reshape(6 * hd, -1)
        else:
            Wm[k] = v.copy()
    tok, tgt = rand_tokens(g_cfg, 2, 7, 19)
    lg, Gg = M.forward_backward(g_cfg, Wg, tok, tgt)
    lm, Gm = M.forward_backward(m_cfg, Wm, tok, tgt)
    assert lg == pytest.approx(lm, rel=1e-13)
    for k in Gg:
        if k.endswith(".wk") or k.endswith(".wv"):
            summed = Gm[k].reshape(2, 3, hd, -1).sum(axis=1).reshape(2 * hd, -1)
            assert np.allclose(Gg[k], summed, rtol=1e-10, atol=1e-13), k
        else:
            assert np.allclose(Gg[k], Gm[k], rtol=1e-10, atol=1e-13), k


def test_causality_and_batch_independence_of_the_model():
    cfg = small_cfg()
    params = rand_params(cfg, 16)
    tok, tgt = rand_tokens(cfg, 2, 6, 17)
    z1 = M.forward_logits(cfg, params, tok)
    tok2 = tok.copy()
    tok2[0, 4:] = (tok2[0, 4:] + 1) % cfg.vocab
    z2 = M.forward_logits(cfg, params, tok2)
    assert np.array_equal(z1[0, :4], z2[0, :4])
    assert not np.allclose(z1[0, 4:], z2[0, 4:])
    assert np.array_equal(z1[1], z2[1])


def test_residual_scale_invariance_of_prenorm_stack():
    """Scaling wte, Wo and Wproj by a > 0 scales the whole residual stream by a,
    which the pre-norms and the final norm remove (eps = 0 makes it exact)."""
    cfg = small_cfg(norm_eps=0.0)
    W = M.unpack(cfg, rand_params(cfg, 18))
    tok, _ = rand_tokens(cfg, 1, 5, 19)
    W2 = {k: (v * 3.0 if (k == "wte" or k.endswith(".wo") or k.endswith(".wproj")) else v)
          for k, v in W.items()}
    assert np.allclose(M.forward_logits(cfg, W, tok), M.forward_logits(cfg, W2, tok), rtol=1e-12)


def test_embedding_scatter_conservation():
    cfg = small_cfg()
    params = rand_params(cfg, 20)
    tok, tgt = rand_tokens(cfg, 2, 5, 21)
    _, G = M.forward_backward(cfg, params, tok, tgt)
    present = np.zeros(cfg.vocab, dtype=bool)
    present[tok.reshape(-1)] = True
    assert np.all(G["wte"][~present] == 0.0)
    assert np.all(np.abs(G["wte"][present]).sum(axis=1) > 0)


# ---------------------------------------------------------------- sizes (context)

def test_param_count_formula_and_pages_model_sizes():
    def count(d, hkv_div=1):
        C = 64 * d
        H = C // 128
        return M.n_params(M.Config(d, C, H, H // hkv_div, 128, 4 * C, 65536))
    for d in (12, 20, 24):
        C = 64 * d
        H = C // 128
        assert count(d) == 2 * 65536 * C + d * (4 * C * C + 8 * C * C)
    # woshipm nanochat analysis §五.2 quotes d16 ~343M, d20 ~566M, d24 ~860M;
    # the formula lands within a few percent of each (context, not a pin).
    for d, quoted in ((16, 343e6), (20, 566e6), (24, 860e6)):
        assert abs(count(d) / quoted - 1) < 0.05
