"""The bounded-wait timeout path of the tensor-core kernels.

The pages describe no fault tolerance of the training step (ssnai "核心分析":
the project lacks fault tolerance), so the library's own status path is the
only one.  Here one GEMM launch is made to wait on a barrier that nothing
completes (the nc_debug_stall_next_gemm hook) under a lowered wait limit: the
kernel must give up, drain what it issued, and the step must return
NC_ERR_TIMEOUT; the next step on the same model must then match a step taken
before the timeout bit for bit.  No GPU fault, trap or endless wait is
involved: the expiry is the kernel's own bounded wait.
"""
import numpy as np
import pytest

import synthetic as S

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402

NC_ERR_TIMEOUT = 6
DEFAULT_WAIT_NS = 4_000_000_000


def test_gemm_wait_timeout_is_reported_and_model_stays_usable():
    lib = nc.lib()
    w = S.Workload(name="timeout", dtype="bf16", tokens="zipf", depth=1, n_embd=256, n_head=2, n_kv_head=2,
                   head_dim=128, mlp_hidden=1024, vocab=1024, seq_len=128, batch=1)
    m = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    tok_np, tgt_np = S.batch_tokens(w)
    tok, tgt = torch.from_numpy(tok_np).cuda(), torch.from_numpy(tgt_np).cuda()
    lib.nc_debug_set_gemm_pair(0)            # every GEMM on the single-CTA kernel, which the hook arms
    try:
        loss0, g0 = m.forward_backward(tok, tgt)
        g0 = g0.clone()
        lib.nc_debug_set_wait_limit_ns(250_000_000)
        lib.nc_debug_stall_next_gemm(1)
        with pytest.raises(nc.NcError) as e:
            m.forward_backward(tok, tgt)
        assert e.value.status == NC_ERR_TIMEOUT
        lib.nc_debug_set_wait_limit_ns(DEFAULT_WAIT_NS)
        # the flag was cleared by the read, the context is usable, the model state intact
        m.check()
        loss1, g1 = m.forward_backward(tok, tgt)
        assert loss1 == loss0
        assert torch.equal(g1, g0)
    finally:
        lib.nc_debug_stall_next_gemm(0)
        lib.nc_debug_set_wait_limit_ns(DEFAULT_WAIT_NS)
        lib.nc_debug_set_gemm_pair(1)
        m.close()
