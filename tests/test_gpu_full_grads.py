"""Whole-step gradients at full sequence length against the fp64 oracle.

The full-size tests elsewhere compare sampled losses at full length and
gradients only on short sequences.  Here the oracle computes the whole step
at the workloads' full sequence length, so every gradient tensor is compared
where the long-sequence paths run:

* d12 (full widths, T = 2048) on 5 sequences, 10,240 tokens: the lm_head and
  cross-entropy run in two row chunks (8,192 rows each at V = 65,536), so dWlm
  is accumulated across chunks by the TMA reduce-add; the weight-gradient
  GEMMs have K = 10,240 and split K with the ordered fix-up; the
  vocabulary-wide rows take the streaming cross-entropy kernel; the Zipf
  stream gives the embedding scatter its hot segments (id 0 on ~14 % of
  positions);
* d24 GQA (three query heads per kv head) on one sequence of T = 4096.

Bounds (bf16 compute against fp64): loss within 2e-2 absolute and every
tensor's gradient at cosine >= 0.999; embedding rows of absent ids exactly
zero.  Weights are N(0, 0.02) float32 from NumPy's seeded generator; tokens
are the workloads' seeded Zipf streams.
"""
import ctypes

import numpy as np
import pytest

import synthetic as S
from oracle import model as OM
from tests.gpu_util import cosine

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402

NC_PROF_GEMM_LM = 12
CASES = [("d12", 5), ("d24gqa", 1)]


@pytest.mark.parametrize("name,batch", CASES, ids=[f"{n}_b{b}" for n, b in CASES])
def test_full_length_step_gradients_match_oracle(name, batch):
    w = S.workload(name, batch=batch)
    cfg = OM.Config.from_workload(w)
    params = np.random.default_rng(4321).standard_normal(OM.n_params(cfg), dtype=np.float32)
    params *= np.float32(cfg.init_std)
    m = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    try:
        m.set_params(torch.from_numpy(params))
        tok, tgt = S.batch_tokens(w)
        lib = nc.lib()
        lib.nc_profile_enable(m.handle, 1)
        loss, g = m.forward_backward(torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda())
        n_lm = ctypes.c_int64()
        lib.nc_profile_read(m.handle, NC_PROF_GEMM_LM, None, ctypes.byref(n_lm), None, None)
        lib.nc_profile_enable(m.handle, 0)
        g = g.cpu().numpy().astype(np.float64)
    finally:
        m.close()
    n_tok = w.batch * w.seq_len
    chunks = -(-n_tok // 8192)
    assert n_lm.value == 3 * chunks          # logits, dx and dW GEMMs per lm_head row chunk
    if name == "d12":
        assert chunks >= 2
    loss_ref, G = OM.forward_backward(cfg, params.astype(np.float64), tok, tgt)
    assert abs(loss - loss_ref) <= 2e-2, (loss, loss_ref)
    g_ref = OM.pack(cfg, G)
    worst = (None, 1.0)
    for tname, r, c, off in OM.param_layout(cfg):
        cs = cosine(g[off:off + r * c], g_ref[off:off + r * c])
        if cs < worst[1]:
            worst = (tname, cs)
    assert worst[1] >= 0.999, worst
    V, C = w.vocab, w.n_embd
    dwte = g[:V * C].reshape(V, C)
    present = np.zeros(V, dtype=bool)
    present[tok.reshape(-1)] = True
    assert np.all(dwte[~present] == 0.0)
    assert np.all(np.abs(dwte[present]).max(axis=1) > 0)
