"""The embedding backward that allocates nothing (nc_op_embed_bwd_noalloc).

It exists for callers that cannot allocate device memory, such as a host that
hands the library only its input and output buffers under a fixed memory
budget.  Its result must equal that of nc_op_embed_bwd, which takes its
scratch from the caller, on consecutive calls that share the library's static
scratch array.  This file is collected last so that a run stopping at its
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402
import synthetic as S  # noqa: E402

NC_ERR_UNSUPPORTED = 7


def _noalloc():
    fn = nc.lib().nc_op_embed_bwd_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    return fn


def _case(seed, n, C, V):
    tok = S.token_stream(V, 1, n - 1, "zipf", seed=seed).reshape(-1)
    dx = np.random.default_rng(seed + 100).normal(size=(n, C)).astype(np.float32)
    return torch.from_numpy(tok).cuda(), torch.from_numpy(dx).cuda()


def test_noalloc_matches_scratch_entry_point_on_two_calls():
    fn = _noalloc()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two different calls in a row: the second must not see the first's leftovers
    for seed, (n, C, V) in ((31, (6000, 384, 4096)), (32, (4097, 256, 8192))):
        tok, dx = _case(seed, n, C, V)
        want = torch.full((V, C), float("nan"), dtype=torch.float32, device="cuda")
        scratch = torch.empty(nc.ops.embed_bwd_scratch_bytes(n, C, V), dtype=torch.uint8, device="cuda")
        nc.ops.embed_bwd(tok, dx, want, scratch)
        got = torch.full((V, C), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(n, C, V, ctypes.c_void_p(tok.data_ptr()), ctypes.c_void_p(dx.data_ptr()),
                ctypes.c_void_p(got.data_ptr()), stream)
        assert st == 0, nc.lib().nc_status_string(st)
        torch.cuda.synchronize()
        # same kernels, same summation order: bitwise equal
        assert torch.equal(got, want)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _noalloc()
    n, C, V = 1 << 16, 1280, 65536            # needs ~340 MB of scratch
    assert nc.ops.embed_bwd_scratch_bytes(n, C, V) > (64 << 20)
    dummy = torch.zeros(4, dtype=torch.int32, device="cuda")
    st = fn(n, C, V, ctypes.c_void_p(dummy.data_ptr()), ctypes.c_void_p(dummy.data_ptr()),
            ctypes.c_void_p(dummy.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == NC_ERR_UNSUPPORTED
