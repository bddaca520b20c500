"""Whole-step parity of nc_forward_backward / nc_forward_logits against the fp64
oracle on the same seeded inputs, plus the init RNG and error paths."""
import math

import numpy as np
import pytest

import synthetic as S
from oracle import model as OM
from oracle import rng as OR
from tests.gpu_util import rel_close, cosine, norm_rel

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402


def make(w, seed=S.WEIGHT_SEED):
    return nc.Model(nc.config_from_workload(w), seed=seed)


def oracle_cfg(w):
    return OM.Config.from_workload(w)


def run_step(model, tok, tgt):
    T = torch.from_numpy(tok).cuda()
    G = torch.from_numpy(tgt).cuda()
    loss, grads = model.forward_backward(T, G)
    return loss, grads.cpu().numpy().astype(np.float64)


def test_init_matches_oracle_rng():
    w = S.workload("tiny")
    m = make(w)
    got = m.get_params().cpu().numpy()
    want = OR.init_params(oracle_cfg(w), S.WEIGHT_SEED)
    diff = got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64)
    # the two sides evaluate log/cos in fp64 independently: allow a rare 1-ulp
    # difference after the single rounding to float32
    assert np.abs(diff).max() <= 1
    assert np.count_nonzero(diff) <= max(2, got.size // 100000)
    m.close()


def test_param_layout_matches_oracle():
    """nc_param_layout / nc_param_info give the oracle's packed order, shapes and offsets."""
    import ctypes
    w = S.Workload(name="gqa", dtype="bf16", tokens="zipf", depth=3, n_embd=256, n_head=4, n_kv_head=2,
                   head_dim=64, mlp_hidden=1024, vocab=1024, seq_len=64, batch=1)
    m = make(w)
    nt, ne = ctypes.c_int32(), ctypes.c_int64()
    assert nc.lib().nc_param_layout(m.handle, ctypes.byref(nt), ctypes.byref(ne)) == 0
    want = OM.param_layout(oracle_cfg(w))
    assert nt.value == len(want) == 2 + 6 * w.depth
    assert ne.value == OM.n_params(oracle_cfg(w))
    assert [tuple(t) for t in m.layout] == [tuple(t) for t in want]
    m.close()


def test_tiny_fp32_step_matches_oracle():
    w = S.workload("tiny")
    cfg = oracle_cfg(w)
    m = make(w)
    params = OR.init_params(cfg, S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    tok, tgt = S.batch_tokens(w)
    loss, g = run_step(m, tok, tgt)
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    g_ref = OM.pack(cfg, G)
    assert abs(loss - loss_ref) <= 1e-5, (loss, loss_ref)
    for name, r, c, off in m.layout:
        ok, worst = rel_close(g[off:off + r * c], g_ref[off:off + r * c], 1e-4)
        assert ok, (name, worst)
        assert norm_rel(g[off:off + r * c], g_ref[off:off + r * c]) <= 1e-5, name
    logits = m.forward_logits(torch.from_numpy(tok).cuda()).cpu().numpy()
    z_ref = OM.forward_logits(cfg, params.astype(np.float64), tok)
    ok, worst = rel_close(logits, z_ref, 1e-4)
    assert ok, worst
    m.close()


def test_tiny_fp32_ragged_batch_and_length():
    w = S.workload("tiny")
    cfg = oracle_cfg(w)
    m = make(w)
    params = OR.init_params(cfg, S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    tok, tgt = S.batch_tokens(w, batch=1, seq_len=37)
    loss, g = run_step(m, tok, tgt)
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    assert abs(loss - loss_ref) <= 1e-5
    g_ref = OM.pack(cfg, G)
    for name, r, c, off in m.layout:
        ok, worst = rel_close(g[off:off + r * c], g_ref[off:off + r * c], 1e-4)
        assert ok, (name, worst)
    m.close()


SMALL_BF16 = [
    dict(depth=2, n_embd=256, n_head=2, n_kv_head=2, head_dim=128, mlp_hidden=1024, vocab=2048,
         seq_len=256, batch=2),
    dict(depth=2, n_embd=256, n_head=4, n_kv_head=2, head_dim=64, mlp_hidden=1024, vocab=1024,
         seq_len=200, batch=2),
]


@pytest.mark.parametrize("shape", SMALL_BF16, ids=["mha_hd128", "gqa_hd64"])
def test_small_bf16_step_matches_oracle(shape):
    w = S.Workload(name="small", dtype="bf16", tokens="zipf", **shape)
    cfg = oracle_cfg(w)
    m = make(w)
    params = OR.init_params(cfg, S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    tok, tgt = S.batch_tokens(w)
    loss, g = run_step(m, tok, tgt)
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    g_ref = OM.pack(cfg, G)
    assert abs(loss - loss_ref) <= 2e-2, (loss, loss_ref)
    for name, r, c, off in m.layout:
        cs = cosine(g[off:off + r * c], g_ref[off:off + r * c])
        assert cs >= 0.999, (name, cs)
    # token-indexed rows of dwte: exactly the ids present are nonzero
    dwte = g[:w.vocab * w.n_embd].reshape(w.vocab, w.n_embd)
    present = np.zeros(w.vocab, dtype=bool)
    present[tok.reshape(-1)] = True
    assert np.all(dwte[~present] == 0.0)
    assert np.all(np.any(dwte[present] != 0.0, axis=1))
    m.close()


def test_step_is_deterministic():
    w = S.Workload(name="small", dtype="bf16", tokens="zipf", **SMALL_BF16[0])
    m = make(w)
    tok, tgt = S.batch_tokens(w)
    l1, g1 = run_step(m, tok, tgt)
    l2, g2 = run_step(m, tok, tgt)
    assert l1 == l2 and np.array_equal(g1, g2)
    m.close()


def test_token_out_of_range_is_reported():
    w = S.workload("tiny")
    m = make(w)
    tok, tgt = S.batch_tokens(w)
    tok = tok.copy()
    tok[1, 5] = w.vocab
    with pytest.raises(nc.NcError) as e:
        run_step(m, tok, tgt)
    assert e.value.status == 4
    tok, tgt = S.batch_tokens(w)
    tgt = tgt.copy()
    tgt[0, 0] = -3
    with pytest.raises(nc.NcError) as e:
        run_step(m, tok, tgt)
    assert e.value.status == 4
    # the model stays usable
    tok, tgt = S.batch_tokens(w)
    loss, _ = run_step(m, tok, tgt)
    assert math.isfinite(loss)
    m.close()


def test_bad_batch_shape_rejected():
    w = S.workload("tiny")
    m = make(w)
    tok = torch.zeros((3, 64), dtype=torch.int32, device="cuda")     # B > cfg.batch
    with pytest.raises(nc.NcError) as e:
        m.forward_backward(tok, tok)
    assert e.value.status == 3
    m.close()
