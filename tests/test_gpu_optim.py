"""The optimizer step (Muon for the matrices, AdamW for wte / lm_head) through
the C ABI against the fp64 oracle in ``oracle/optim.py``.

Tolerances come from the arithmetic.
* fp32 mode: the iteration's products are exact-fp32 FMA GEMMs.  An fp32
  emulation of the five iterations lands about 2e-7 (Frobenius, relative) from
  fp64, so the bound is 1e-5.
* bf16 mode: every product is rounded to bf16 (fp32 accumulation).  A bf16
  emulation lands 0.8-1.3e-2 from fp64 with cosine >= 0.9999, so the bounds
  are 3e-2 and cosine >= 0.999.
* A real model gradient is ill-conditioned (singular values spanning up to
  ~1e11 at initialisation) and the iteration magnifies its small directions,
  where the bf16 rounding lands: the same emulation on the oracle gradient of a
  small model reaches cosine 0.9977-0.9995 per matrix, so that case is bounded
  at 0.99.
* AdamW is fp32 elementwise: 1e-5 of the step.
Inputs are seeded host draws (weights N(0, 0.02), gradients standard normal);
nothing the GPU computes feeds the oracle.
"""
import numpy as np
import pytest

import synthetic as S
from oracle import model as OM
from oracle import optim as OO

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def _cos(a, b):
    return float(np.sum(a * b) / (np.linalg.norm(a) * np.linalg.norm(b)))


@pytest.mark.parametrize("shape", [(96, 200), (200, 96), (128, 128), (40, 24)])
def test_newton_schulz_fp32(shape):
    u = np.random.default_rng(11).standard_normal(shape)
    U = torch.from_numpy(u.astype(np.float32)).cuda()
    X = torch.empty_like(U)
    nc.ops.newton_schulz(U, X, 5, dtype="fp32")
    got = X.cpu().numpy().astype(np.float64)
    want = OO.newton_schulz(u.astype(np.float32).astype(np.float64))
    assert _rel(got, want) < 1e-5, _rel(got, want)


@pytest.mark.parametrize("shape", [(256, 512), (512, 256), (384, 384), (1280, 5120)])
def test_newton_schulz_bf16(shape):
    u = np.random.default_rng(12).standard_normal(shape)
    U = torch.from_numpy(u.astype(np.float32)).cuda()
    X = torch.empty_like(U)
    nc.ops.newton_schulz(U, X, 5, dtype="bf16")
    got = X.cpu().numpy().astype(np.float64)
    want = OO.newton_schulz(u.astype(np.float32).astype(np.float64))
    assert _rel(got, want) < 3e-2 and _cos(got, want) > 0.999, (_rel(got, want), _cos(got, want))


def test_newton_schulz_zero_steps_is_the_normalised_input():
    u = np.random.default_rng(13).standard_normal((64, 96))
    U = torch.from_numpy(u.astype(np.float32)).cuda()
    X = torch.empty_like(U)
    nc.ops.newton_schulz(U, X, 0, dtype="fp32")
    uf = u.astype(np.float32).astype(np.float64)
    assert _rel(X.cpu().numpy().astype(np.float64), uf / (np.linalg.norm(uf) + 1e-7)) < 1e-6


def _run_steps(w, dtype, steps, lr_mults, seed):
    cfg = OM.Config.from_workload(w)
    P = OM.n_params(cfg)
    rng = np.random.default_rng(seed)
    params = (rng.standard_normal(P) * 0.02).astype(np.float32)
    grads = [rng.standard_normal(P).astype(np.float32) for _ in range(steps)]
    assert w.dtype == dtype
    m = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    oc = nc.optim_config()
    got = []
    for g, lm in zip(grads, lr_mults):
        m.optimizer_step(torch.from_numpy(g).cuda(), oc, lm)
        got.append(m.get_params().cpu().numpy().astype(np.float64))
    assert m.optimizer_steps() == steps
    ref_state = OO.new_state(cfg)
    ref = []
    cur = params.astype(np.float64)
    for g, lm in zip(grads, lr_mults):
        cur = OO.optimizer_step(cfg, cur, g.astype(np.float64), ref_state, OO.OptimConfig(), lm)
        ref.append(cur)
    m.close()
    return cfg, params.astype(np.float64), got, ref


def _check(cfg, p0, got, ref, muon_rel, muon_cos):
    for k in range(len(got)):
        for name, r, c, off in OM.param_layout(cfg):
            d_got = got[k][off:off + r * c] - p0[off:off + r * c]
            d_ref = ref[k][off:off + r * c] - p0[off:off + r * c]
            if name in ("wte", "lm_head"):
                assert np.max(np.abs(d_got - d_ref)) <= 1e-5 * np.max(np.abs(d_ref)), (k, name)
            else:
                assert _rel(d_got, d_ref) < muon_rel and _cos(d_got, d_ref) > muon_cos, \
                    (k, name, _rel(d_got, d_ref), _cos(d_got, d_ref))


def test_optimizer_steps_fp32_tiny():
    cfg, p0, got, ref = _run_steps(S.workload("tiny"), "fp32", 3, [1.0, 0.5, 0.25], 21)
    _check(cfg, p0, got, ref, 1e-5, 0.99999)


def test_optimizer_steps_bf16_small_gqa():
    w = S.workload("d12", depth=2, n_embd=256, n_head=2, n_kv_head=1, head_dim=128, mlp_hidden=1024, vocab=512,
                   seq_len=128, batch=2)
    cfg, p0, got, ref = _run_steps(w, "bf16", 2, [1.0, 0.3], 22)
    _check(cfg, p0, got, ref, 3e-2, 0.999)


def test_batched_newton_schulz_equals_per_matrix():
    """The batched iteration (all matrices of a shape in one launch per product)
    computes, tile for tile, the products the per-matrix iteration computes:
    two bf16 steps leave bit-identical weights either way."""
    w = S.workload("d12", depth=2, n_embd=256, n_head=2, n_kv_head=1, head_dim=128, mlp_hidden=1024, vocab=512,
                   seq_len=128, batch=2)
    P = OM.n_params(OM.Config.from_workload(w))
    rng = np.random.default_rng(24)
    params = torch.from_numpy((rng.standard_normal(P) * 0.02).astype(np.float32))
    g = torch.from_numpy(rng.standard_normal(P).astype(np.float32)).cuda()
    out = []
    for batched in (1, 0):
        nc.lib().nc_debug_set_ns_batched(batched)
        try:
            m = nc.Model(nc.config_from_workload(w), seed=1)
            m.set_params(params)
            m.optimizer_step(g)
            m.optimizer_step(g, lr_mult=0.5)
            out.append(m.get_params().cpu())
            m.close()
        finally:
            nc.lib().nc_debug_set_ns_batched(1)
    assert not torch.equal(out[0], params)
    assert torch.equal(out[0], out[1])


def test_optimizer_is_deterministic_and_reset_restarts():
    w = S.workload("tiny")
    P = OM.n_params(OM.Config.from_workload(w))
    rng = np.random.default_rng(23)
    params = torch.from_numpy((rng.standard_normal(P) * 0.02).astype(np.float32))
    g = torch.from_numpy(rng.standard_normal(P).astype(np.float32)).cuda()
    out = []
    for _ in range(2):
        m = nc.Model(nc.config_from_workload(w), seed=1)
        m.set_params(params)
        m.optimizer_step(g)
        first = m.get_params().cpu()
        m.optimizer_step(g)
        m.set_params(params)
        m.optimizer_reset()
        assert m.optimizer_steps() == 0
        m.optimizer_step(g)
        assert torch.equal(m.get_params().cpu(), first), "reset did not restart the optimizer"
        out.append(first)
        m.close()
    assert torch.equal(out[0], out[1])


def test_optimizer_rejects_bad_settings():
    m = nc.Model(nc.config_from_workload(S.workload("tiny")), seed=1)
    g = torch.zeros(m.n_params, dtype=torch.float32, device="cuda")
    for bad in (dict(momentum=1.0), dict(beta2=1.5), dict(adam_eps=0.0), dict(ns_steps=-1)):
        with pytest.raises(nc.NcError):
            m.optimizer_step(g, nc.optim_config(**bad))
    m.close()


def test_optimizer_step_from_a_real_gradient_bf16():
    """Muon on the ill-conditioned gradient of an actual batch (the oracle's)."""
    from oracle import rng as OR
    w = S.Workload("realgrad", 2, 256, 4, 2, 64, 1024, 1024, 128, 2, "bf16", "zipf")
    cfg = OM.Config.from_workload(w)
    params = OR.init_params(cfg, S.WEIGHT_SEED)
    tok, tgt = S.batch_tokens(w)
    _, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    g32 = OM.pack(cfg, G).astype(np.float32)
    m = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    m.optimizer_step(torch.from_numpy(g32).cuda())
    d_got = m.get_params().cpu().numpy().astype(np.float64) - params
    d_ref = OO.optimizer_step(cfg, params.astype(np.float64), g32.astype(np.float64), OO.new_state(cfg)) - params
    for name, r, c, off in m.layout:
        a, b = d_got[off:off + r * c], d_ref[off:off + r * c]
        if name in ("wte", "lm_head"):
            assert np.max(np.abs(a - b)) <= 1e-5 * np.max(np.abs(b)), name
        else:
            assert _cos(a, b) > 0.99, (name, _cos(a, b))
    m.close()
