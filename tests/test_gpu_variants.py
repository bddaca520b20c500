"""The two off-by-default variants against the fp64 oracle: the logit soft-cap
z <- c tanh(z / c) (the reading of woshipm nanochat analysis §三.3 item 1,
"logit stabilisation") fused into the cross-entropy kernels, and the RMSNorm
after the embedding lookup.

Kernel level: the capped cross-entropy of all three kernels (generic, one
row in registers, vocabulary-wide streaming) against the oracle's
softcap + cross-entropy.  Step level, with the step's own tolerances: the
tiny fp32 workload (loss within 1e-5, gradients and logits within 1e-4
relative) and a small bf16 GQA model (loss within 2e-2, every gradient
tensor at cosine >= 0.999), each with both variants on; the capped logits of
nc_forward_logits and of prefill + decoding.
"""
import numpy as np
import pytest

import synthetic as S
from oracle import model as OM
from oracle import rng as OR
from tests.gpu_util import dev_tensor, to64, rel_close, cosine, norm_rel

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402

BF16, F32 = torch.bfloat16, torch.float32


def rnd(seed, shape, scale=1.0):
    return np.random.default_rng(seed).normal(0.0, scale, size=shape).astype(np.float32)


@pytest.mark.parametrize("dt,V", [(F32, 1000), (BF16, 1000), (BF16, 4096), (BF16, 32768)],
                         ids=["f32_generic", "bf16_generic", "bf16_registers", "bf16_streaming"])
def test_cross_entropy_softcap(dt, V):
    rows, c, scale = 48, 3.0, 0.5
    Z = dev_tensor(rnd(70, (rows, V), 2.5), dt)       # |z| up to ~10: the cap saturates some logits
    z = to64(Z)
    tgt = np.random.default_rng(71).integers(0, V, size=rows).astype(np.int32)
    RL = torch.empty(rows, dtype=F32, device="cuda")
    nc.ops.cross_entropy_softcap(Z, torch.from_numpy(tgt).cuda(), RL, scale, c)
    zc, dcap = OM.softcap(z, c)
    loss_ref, dzc = OM.cross_entropy(zc, tgt)
    torch.cuda.synchronize()
    assert np.allclose(to64(RL), loss_ref, rtol=1e-5, atol=2e-5)
    rtol = 1e-5 if dt == F32 else 2.0 ** -8
    ok, worst = rel_close(to64(Z), scale * dzc * dcap, rtol, 1e-3)
    assert ok, worst


def test_cross_entropy_softcap_rejects_bad_cap():
    Z = torch.zeros((2, 64), dtype=F32, device="cuda")
    TG = torch.zeros(2, dtype=torch.int32, device="cuda")
    RL = torch.empty(2, dtype=F32, device="cuda")
    for bad in (-1.0, float("inf"), float("nan")):
        with pytest.raises(nc.NcError) as e:
            nc.ops.cross_entropy_softcap(Z, TG, RL, 1.0, bad)
        assert e.value.status == 3


def _variant_model(w, softcap, embed_norm, std=None):
    kw = dict(logit_softcap=softcap, embed_norm=embed_norm)
    cfg = OM.Config.from_workload(w, **kw)
    m = nc.Model(nc.config_from_workload(w, **kw), seed=S.WEIGHT_SEED)
    params = OR.init_params(cfg, S.WEIGHT_SEED)
    if std is not None:
        params = params * np.float32(std / 0.02)
    m.set_params(torch.from_numpy(params))
    return cfg, m, params


def test_tiny_fp32_step_with_both_variants():
    w = S.workload("tiny")
    # c = 0.3 against logits of a few tenths: the cap bends them
    cfg, m, params = _variant_model(w, 0.3, True)
    tok, tgt = S.batch_tokens(w)
    loss, g = m.forward_backward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
    g = g.cpu().numpy().astype(np.float64)
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    g_ref = OM.pack(cfg, G)
    assert abs(loss - loss_ref) <= 1e-5, (loss, loss_ref)
    for name, r, c, off in m.layout:
        ok, worst = rel_close(g[off:off + r * c], g_ref[off:off + r * c], 1e-4)
        assert ok, (name, worst)
        assert norm_rel(g[off:off + r * c], g_ref[off:off + r * c]) <= 1e-5, name
    z = m.forward_logits(torch.from_numpy(tok).cuda()).cpu().numpy()
    z_ref = OM.forward_logits(cfg, params.astype(np.float64), tok)
    assert np.abs(z).max() <= 0.3 and np.abs(z_ref).max() > 0.1
    ok, worst = rel_close(z, z_ref, 1e-4)
    assert ok, worst
    m.close()


@pytest.mark.parametrize("softcap,embed_norm", [(0.5, False), (0.0, True), (0.5, True)],
                         ids=["softcap", "embed_norm", "both"])
def test_small_bf16_step_with_variants(softcap, embed_norm):
    w = S.Workload(name="small", dtype="bf16", tokens="zipf", depth=2, n_embd=256, n_head=4, n_kv_head=2,
                   head_dim=64, mlp_hidden=1024, vocab=1024, seq_len=200, batch=2)
    cfg, m, params = _variant_model(w, softcap, embed_norm, std=0.05)
    tok, tgt = S.batch_tokens(w)
    loss, g = m.forward_backward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
    g = g.cpu().numpy().astype(np.float64)
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    g_ref = OM.pack(cfg, G)
    assert abs(loss - loss_ref) <= 2e-2, (loss, loss_ref)
    for name, r, c, off in m.layout:
        cs = cosine(g[off:off + r * c], g_ref[off:off + r * c])
        assert cs >= 0.999, (name, cs)
    dwte = g[:w.vocab * w.n_embd].reshape(w.vocab, w.n_embd)
    present = np.zeros(w.vocab, dtype=bool)
    present[tok.reshape(-1)] = True
    assert np.all(dwte[~present] == 0.0)
    m.close()


def test_decode_fp32_tiny_with_both_variants():
    """Prefill + decoding give the capped logits of the whole-sequence forward."""
    w = S.workload("tiny")
    cfg, m, params = _variant_model(w, 0.3, True)
    t0, k = 40, 5
    tok, _ = S.batch_tokens(w, seq_len=t0 + k)
    m.kv_cache_create(tok.shape[0], t0 + k)
    got = [m.prefill(torch.from_numpy(np.ascontiguousarray(tok[:, :t0])).cuda()).cpu().numpy()]
    for j in range(k - 1):
        got.append(m.decode_step(torch.from_numpy(np.ascontiguousarray(tok[:, t0 + j])).cuda()).cpu().numpy())
    z = OM.forward_logits(cfg, params.astype(np.float64), tok)
    for j, gj in enumerate(got):
        ok, worst = rel_close(gj, z[:, t0 - 1 + j, :], 1e-4)
        assert ok, (j, worst)
    m.close()


def test_variant_config_validation():
    import ctypes
    base = dict(depth=1, n_embd=256, n_head=2, n_kv_head=2, head_dim=128, mlp_hidden=1024, vocab=512,
                seq_len=64, batch=1, dtype="bf16")
    for kw in (dict(logit_softcap=-1.0), dict(logit_softcap=float("inf")), dict(embed_norm=True)):
        cfg = nc.make_config(**base, **kw)
        if "embed_norm" in kw:
            cfg.embed_norm = 2
        h = ctypes.c_void_p()
        assert nc.lib().nc_model_create(ctypes.byref(cfg), 1, ctypes.byref(h)) == 1 and not h.value
