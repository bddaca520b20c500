"""KV-cache decoding (nc_prefill + nc_decode_step) against the fp64 oracle.

By causality the logits of position t depend only on tokens 0..t, so the
logits after prefilling t0 tokens and decoding k more must equal row t0+k-1 of
the oracle's forward over the whole sequence.  fp32 mode: within 1e-4
(relative, the step's own tolerance).  bf16 mode: per-row cosine >= 0.999 and
|dz| <= 0.02 + 0.02 |z| (logits here are O(0.3); bf16 activations carry ~1 %).
"""
import numpy as np
import pytest

import synthetic as S
from oracle import model as OM
from oracle import rng as OR
from tests.gpu_util import rel_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402


def _model(w):
    cfg = OM.Config.from_workload(w)
    m = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    params = OR.init_params(cfg, S.WEIGHT_SEED)
    m.set_params(torch.from_numpy(params))
    return cfg, m, params


def _decode_run(w, t0, k):
    cfg, m, params = _model(w)
    tok, _ = S.batch_tokens(w, seq_len=t0 + k)
    B = tok.shape[0]
    m.kv_cache_create(B, t0 + k)
    got = [m.prefill(torch.from_numpy(np.ascontiguousarray(tok[:, :t0])).cuda()).cpu().numpy()]
    for j in range(k - 1):
        got.append(m.decode_step(torch.from_numpy(np.ascontiguousarray(tok[:, t0 + j])).cuda()).cpu().numpy())
    assert m.kv_cache_length() == t0 + k - 1
    z = OM.forward_logits(cfg, params.astype(np.float64), tok)           # [B, t0 + k, V]
    want = [z[:, t0 - 1 + j, :] for j in range(k)]
    m.close()
    return got, want


def test_decode_fp32_tiny():
    got, want = _decode_run(S.workload("tiny"), 40, 6)
    for j, (g, z) in enumerate(zip(got, want)):
        ok, worst = rel_close(g, z, 1e-4)
        assert ok, (j, worst)


@pytest.mark.parametrize("shape", [dict(depth=2, n_embd=256, n_head=4, n_kv_head=2, head_dim=64, mlp_hidden=1024,
                                        vocab=1024, seq_len=320, batch=2),
                                   dict(depth=2, n_embd=384, n_head=3, n_kv_head=1, head_dim=128, mlp_hidden=1536,
                                        vocab=512, seq_len=320, batch=3)],
                         ids=["gqa2_hd64", "gqa3_hd128"])
def test_decode_bf16_matches_full_forward(shape):
    w = S.Workload(name="dec", dtype="bf16", tokens="zipf", **shape)
    # 300 prompt positions: the decode attention spans two key chunks of 256
    got, want = _decode_run(w, 300, 5)
    for j, (g, z) in enumerate(zip(got, want)):
        for b in range(g.shape[0]):
            cos = float(g[b] @ z[b] / (np.linalg.norm(g[b]) * np.linalg.norm(z[b])))
            assert cos >= 0.999, (j, b, cos)
        assert np.all(np.abs(g - z) <= 0.02 + 0.02 * np.abs(z)), (j, float(np.max(np.abs(g - z))))


def test_decode_bf16_wide_batch_tensor_core_projections():
    """12 sequences: beyond 8 rows the projections run on the tensor-core GEMM after a separate RMSNorm."""
    w = S.Workload(name="dec", dtype="bf16", tokens="zipf", depth=2, n_embd=256, n_head=4, n_kv_head=2, head_dim=64,
                   mlp_hidden=1024, vocab=1024, seq_len=128, batch=12)
    got, want = _decode_run(w, 100, 3)
    for j, (g, z) in enumerate(zip(got, want)):
        for b in range(g.shape[0]):
            cos = float(g[b] @ z[b] / (np.linalg.norm(g[b]) * np.linalg.norm(z[b])))
            assert cos >= 0.999, (j, b, cos)
        assert np.all(np.abs(g - z) <= 0.02 + 0.02 * np.abs(z)), (j, float(np.max(np.abs(g - z))))


def test_decode_errors_and_cache_reuse():
    w = S.workload("tiny")
    cfg, m, params = _model(w)
    tok, _ = S.batch_tokens(w, seq_len=8)
    T_ = torch.from_numpy(tok).cuda()
    with pytest.raises(nc.NcError):
        m.prefill(T_)                                   # no cache yet
    m.kv_cache_create(2, 10)
    with pytest.raises(nc.NcError):
        m.decode_step(T_[:, 0].contiguous())            # empty cache
    m.prefill(T_)
    with pytest.raises(nc.NcError):
        m.decode_step(T_[:1, 0].contiguous())           # batch differs from the prefill's
    m.decode_step(T_[:, 1].contiguous())
    m.decode_step(T_[:, 2].contiguous())
    assert m.kv_cache_length() == 10
    with pytest.raises(nc.NcError):
        m.decode_step(T_[:, 3].contiguous())            # full
    m.kv_cache_create(2, 10)                            # reused and emptied
    assert m.kv_cache_length() == 0
    z1 = m.prefill(T_[:, :5].contiguous()).cpu().numpy()
    z_ref = OM.forward_logits(cfg, params.astype(np.float64), tok[:, :5])[:, 4, :]
    ok, worst = rel_close(z1, z_ref, 1e-4)
    assert ok, worst
    m.close()


def test_decode_graph_replay_equals_eager():
    """The captured step and the eagerly enqueued one give bitwise the same logits."""
    w = S.Workload(name="dec", dtype="bf16", tokens="zipf", depth=2, n_embd=256, n_head=4, n_kv_head=2, head_dim=64,
                   mlp_hidden=1024, vocab=1024, seq_len=320, batch=2)
    cfg, m, params = _model(w)
    tok, _ = S.batch_tokens(w, seq_len=270)
    dev = torch.from_numpy(tok).cuda()
    outs = []
    for graph in (1, 0):
        nc.lib().nc_debug_set_decode_graph(graph)
        m.kv_cache_create(2, 270)
        z = [m.prefill(dev[:, :250].contiguous()).cpu()]
        for j in range(19):
            z.append(m.decode_step(dev[:, 250 + j].contiguous()).cpu())
        outs.append(torch.stack(z))
    nc.lib().nc_debug_set_decode_graph(1)
    assert torch.equal(outs[0], outs[1])
    m.close()


def test_decode_overlapped_launches_equal_stream_order():
    """Decode kernels launched to overlap their predecessor's tail (programmatic
    dependent launch, in the captured step) give bitwise the logits of plain
    stream order."""
    w = S.Workload(name="dec", dtype="bf16", tokens="zipf", depth=2, n_embd=256, n_head=4, n_kv_head=2, head_dim=64,
                   mlp_hidden=1024, vocab=1024, seq_len=320, batch=2)
    tok, _ = S.batch_tokens(w, seq_len=270)
    dev = torch.from_numpy(tok).cuda()
    outs = []
    for pdl in (1, 0):
        nc.lib().nc_debug_set_decode_pdl(pdl)
        try:
            cfg, m, params = _model(w)
            m.kv_cache_create(2, 270)
            z = [m.prefill(dev[:, :250].contiguous()).cpu()]
            for j in range(19):
                z.append(m.decode_step(dev[:, 250 + j].contiguous()).cpu())
            outs.append(torch.stack(z))
            m.close()
        finally:
            nc.lib().nc_debug_set_decode_pdl(1)
    assert torch.equal(outs[0], outs[1])
