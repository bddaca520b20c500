"""The 8-bit training step (nc_config.fp8 = 1) against the oracle's 8-bit step.

Recipe (the reading of woshipm nanochat analysis §一.2 and §六.2, which name
FP8 without one): the blocks' four linear layers multiply E4M3 operands in
the forward, the bf16 activation and the fp32 master weight quantised per
tensor with current scaling; their input gradients dX = dY W multiply E4M3
operands too (dY's bf16 value with its own per-tensor scale, W's forward
codes read transposed), and so do their weight gradients dW = dY^T X (the
same codes of dY and of X, transposed).

Tolerances.  Both sides quantise the same fp32 master weights, so the weight
codes agree; the activation and output-gradient codes come from tensors that
differ by the bf16 path's rounding (about 2^-9 relative).  E4M3 codes are 2^-3 apart, so a
few per cent of the activation codes land one step apart between the two
evaluations: per element the two forwards then differ by about
sqrt(0.03) * 2^-3 ~ 2 % of an operand, some twenty times the bf16 path's
per-element noise, and 1 - cosine of a gradient grows with its square (the
bf16 step measures 1 - cos below 1e-5 here).  Hence: loss within 2e-2 as for
bf16, every gradient tensor at cosine >= 0.99, token rows exact.
"""
import ctypes

import numpy as np
import pytest

import synthetic as S
from oracle import model as OM
from oracle import rng as OR
from tests.gpu_util import cosine

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402

SHAPES = [
    dict(depth=2, n_embd=256, n_head=2, n_kv_head=2, head_dim=128, mlp_hidden=1024, vocab=2048, seq_len=256, batch=2),
    dict(depth=2, n_embd=256, n_head=4, n_kv_head=2, head_dim=64, mlp_hidden=1024, vocab=1024, seq_len=200, batch=2),
    # rows past one 256-row pair tile and a ragged tail: CTA-pair 8-bit GEMMs with every epilogue
    dict(depth=1, n_embd=384, n_head=3, n_kv_head=1, head_dim=128, mlp_hidden=1536, vocab=4096, seq_len=333, batch=3),
    # an MLP width that is a multiple of 16 but not of 64: partial column tiles in the casts and the weight-code
    # transposes, and N, K tails in the 8-bit products
    dict(depth=1, n_embd=256, n_head=2, n_kv_head=2, head_dim=128, mlp_hidden=1040, vocab=1024, seq_len=200, batch=2),
]


def _models(w):
    cfg8 = OM.Config.from_workload(w, fp8=True)
    m = nc.Model(nc.config_from_workload(w, fp8=True), seed=S.WEIGHT_SEED)
    params = OR.init_params(cfg8, S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    return cfg8, m, params


@pytest.mark.parametrize("shape", SHAPES, ids=["mha_hd128", "gqa_hd64", "gqa3_ragged", "mlp1040"])
def test_fp8_step_matches_oracle(shape):
    w = S.Workload(name="small", dtype="bf16", tokens="zipf", **shape)
    cfg8, m, params = _models(w)
    tok, tgt = S.batch_tokens(w)
    T_, G_ = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    loss, g = m.forward_backward(T_, G_)
    g = g.cpu().numpy().astype(np.float64)
    loss2, g2 = m.forward_backward(T_, G_)
    assert loss2 == loss and np.array_equal(g2.cpu().numpy().astype(np.float64), g)   # deterministic
    loss_ref, G = OM.forward_backward(cfg8, params.astype(np.float64), tok, tgt)
    g_ref = OM.pack(cfg8, G)
    assert abs(loss - loss_ref) <= 2e-2, (loss, loss_ref)
    worst = min((cosine(g[off:off + r * c], g_ref[off:off + r * c]), name) for name, r, c, off in m.layout)
    assert worst[0] >= 0.99, worst
    dwte = g[:w.vocab * w.n_embd].reshape(w.vocab, w.n_embd)
    present = np.zeros(w.vocab, dtype=bool)
    present[tok.reshape(-1)] = True
    assert np.all(dwte[~present] == 0.0)
    m.close()


def test_fp8_forward_differs_from_bf16_by_the_quantisation():
    """The 8-bit logits sit closer to the oracle's 8-bit logits than to the
    bf16 model's: the quantisation is really applied, where the recipe says."""
    w = S.Workload(name="small", dtype="bf16", tokens="zipf", **SHAPES[0])
    cfg8, m8, params = _models(w)
    m16 = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    m16.set_params(torch.from_numpy(params))
    tok, _ = S.batch_tokens(w, batch=1, seq_len=96)
    z8 = m8.forward_logits(torch.from_numpy(tok).cuda()).cpu().numpy().astype(np.float64)
    z16 = m16.forward_logits(torch.from_numpy(tok).cuda()).cpu().numpy().astype(np.float64)
    r8 = OM.forward_logits(cfg8, params.astype(np.float64), tok)
    r16 = OM.forward_logits(OM.Config.from_workload(w), params.astype(np.float64), tok)
    d = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
    assert d(z8, r8) < d(z8, r16)          # nearer its own reading than the bf16 model
    assert d(z16, r16) < d(z16, r8)
    assert d(z8, z16) > 1e-3               # the two paths differ by more than bf16 noise
    m8.close()
    m16.close()


def test_fp8_config_rules():
    base = dict(depth=1, n_embd=256, n_head=2, n_kv_head=2, head_dim=128, mlp_hidden=1024, vocab=512,
                seq_len=64, batch=1)
    # fp32 compute, and an MLP width whose 8-bit rows would not be 16-byte multiples
    for kw in (dict(dtype="fp32"), dict(dtype="bf16", mlp_hidden=1032)):
        cfg = nc.make_config(**{**base, **kw}, fp8=True)
        h = ctypes.c_void_p()
        assert nc.lib().nc_model_create(ctypes.byref(cfg), 1, ctypes.byref(h)) == 1 and not h.value
    m = nc.Model(nc.make_config(**base, dtype="bf16", fp8=True))
    with pytest.raises(nc.NcError) as e:
        m.kv_cache_create(1, 64)
    assert e.value.status == 7
    m.close()


def test_fp8_step_accumulates_micro_batches():
    """Accumulating a second micro-batch adds its 8-bit gradient to the first's:
    the buffer equals the sum of the two steps' gradients taken separately (each
    micro-batch quantised with its own per-tensor scales either way), through the
    reduce-add epilogues and the split-K fix-up of the 8-bit weight gradients."""
    w = S.Workload(name="small", dtype="bf16", tokens="zipf", **SHAPES[2])
    cfg8, m, params = _models(w)
    tok, tgt = S.batch_tokens(w)                          # [3, 333]
    parts = [(tok[:2], tgt[:2]), (tok[2:], tgt[2:])]
    dev = [(torch.from_numpy(np.ascontiguousarray(t)).cuda(), torch.from_numpy(np.ascontiguousarray(g)).cuda())
           for t, g in parts]
    separate = []
    for t, g in dev:
        _, grads = m.forward_backward(t, g)
        separate.append(grads.clone())
    acc = torch.empty(m.n_params, dtype=torch.float32, device="cuda")
    for i, (t, g) in enumerate(dev):
        m.forward_backward_accumulate(t, g, acc, 1.0, accumulate=i > 0)
    want = (separate[0] + separate[1]).cpu().numpy().astype(np.float64)
    got = acc.cpu().numpy().astype(np.float64)
    for name, r, c, off in m.layout:
        a, b = got[off:off + r * c], want[off:off + r * c]
        assert np.linalg.norm(a - b) <= 1e-6 * np.linalg.norm(b), name
    m.close()
