"""Gradient accumulation over micro-batches (nc_forward_backward_accumulate)
against the fp64 oracle's gradient of the whole batch.

With k equal micro-batches, grad_scale = 1/k and accumulation on all but the
first call, the buffer must hold the gradient of the mean loss over the union
(the mean of equal-size means).  Tolerances are the step's own: fp32 within
1e-4 (relative, normwise), bf16 per-tensor cosine >= 0.999.  Accumulating into
a non-zero buffer must leave the embedding rows of ids absent from the
micro-batch bitwise unchanged.
"""
import numpy as np
import pytest

import synthetic as S
from oracle import model as OM
from oracle import rng as OR

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402


def _setup(w):
    cfg = OM.Config.from_workload(w)
    m = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    params = OR.init_params(cfg, S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    return cfg, m, params


def _accumulate(m, tok, tgt, k):
    g = torch.empty(m.n_params, dtype=torch.float32, device="cuda")
    rows = np.array_split(np.arange(tok.shape[0]), k)
    losses = []
    for i, r in enumerate(rows):
        T_ = torch.from_numpy(np.ascontiguousarray(tok[r])).cuda()
        G_ = torch.from_numpy(np.ascontiguousarray(tgt[r])).cuda()
        losses.append(m.forward_backward_accumulate(T_, G_, g, 1.0 / k, accumulate=i > 0))
    return losses, g.cpu().numpy().astype(np.float64)


def test_accumulate_two_micro_batches_fp32():
    w = S.workload("tiny")
    cfg, m, params = _setup(w)
    tok, tgt = S.batch_tokens(w)                          # [2, 64]
    losses, g = _accumulate(m, tok, tgt, 2)
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    g_ref = OM.pack(cfg, G)
    for i in range(2):
        li, _ = OM.forward_backward(cfg, params.astype(np.float64), tok[i:i + 1], tgt[i:i + 1])
        assert abs(losses[i] - li) <= 1e-5
    assert abs(np.mean(losses) - loss_ref) <= 1e-5
    for name, r, c, off in m.layout:
        a, b = g[off:off + r * c], g_ref[off:off + r * c]
        assert np.linalg.norm(a - b) <= 1e-4 * np.linalg.norm(b), name
    m.close()


def test_accumulate_three_micro_batches_bf16_gqa():
    w = S.Workload("acc", 2, 256, 4, 2, 64, 1024, 1024, 96, 3, "bf16", "zipf")
    cfg, m, params = _setup(w)
    tok, tgt = S.batch_tokens(w)                          # [3, 96]
    losses, g = _accumulate(m, tok, tgt, 3)
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    g_ref = OM.pack(cfg, G)
    assert abs(np.mean(losses) - loss_ref) <= 2e-2
    for name, r, c, off in m.layout:
        a, b = g[off:off + r * c], g_ref[off:off + r * c]
        assert float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b))) >= 0.999, name
    m.close()


def test_accumulate_adds_onto_existing_buffer_and_leaves_absent_rows():
    w = S.workload("tiny")
    cfg, m, params = _setup(w)
    tok, tgt = S.batch_tokens(w, batch=1, seq_len=20)
    base = np.random.default_rng(31).standard_normal(m.n_params).astype(np.float32)
    g = torch.from_numpy(base.copy()).cuda()
    m.forward_backward_accumulate(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda(), g, 0.3, accumulate=True)
    got = g.cpu().numpy()
    _, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    want = base.astype(np.float64) + 0.3 * OM.pack(cfg, G)
    for name, r, c, off in m.layout:
        a, b = got[off:off + r * c].astype(np.float64), want[off:off + r * c]
        d = b - base[off:off + r * c]
        assert np.linalg.norm(a - b) <= 1e-4 * np.linalg.norm(d) + 1e-6, name
    V, C = w.vocab, w.n_embd
    present = np.zeros(V, dtype=bool)
    present[tok.reshape(-1)] = True
    wte_got, wte_base = got[:V * C].reshape(V, C), base[:V * C].reshape(V, C)
    assert np.array_equal(wte_got[~present], wte_base[~present])
    m.close()
