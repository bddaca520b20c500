"""CPU-side checks of the C ABI: the library loads, exports every function
include/nc.h declares, and rejects invalid configs before touching a GPU."""
import ctypes
import os
import re

import pytest

import decoder_only_transformer_07_b300 as nc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "nc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(nc_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_step_entry_points():
    names = declared_functions()
    for n in ("nc_model_create", "nc_forward_backward", "nc_forward_logits", "nc_model_destroy",
              "nc_op_gemm", "nc_op_attention_fwd", "nc_op_embed_bwd"):
        assert n in names
    assert len(names) >= 25


def test_library_exports_every_declared_function():
    lib = ctypes.CDLL(nc.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version():
    lib = nc.lib()
    for s in range(8):
        assert lib.nc_status_string(s)
    assert b"sm_103a" in lib.nc_version()


@pytest.mark.parametrize("field,value", [
    ("n_embd", 100),          # != n_head * head_dim
    ("n_kv_head", 3),         # n_head % n_kv_head != 0
    ("head_dim", 96),         # bf16 kernels take 64 or 128
    ("vocab", 0),
    ("seq_len", -1),
    ("dtype", 7),
    ("logit_softcap", -1.0),  # the cap is c >= 0 (0: off)
    ("logit_softcap", float("inf")),
    ("embed_norm", 2),        # a 0/1 switch
])
def test_invalid_config_rejected_without_gpu(field, value):
    kw = dict(depth=2, n_embd=256, n_head=2, n_kv_head=2, head_dim=128, mlp_hidden=1024, vocab=512,
              seq_len=64, batch=2, dtype="bf16")
    cfg = nc.make_config(**kw)
    setattr(cfg, field, value)
    h = ctypes.c_void_p()
    st = nc.lib().nc_model_create(ctypes.byref(cfg), 1, ctypes.byref(h))
    assert st == 1 and not h.value


def test_null_arguments_rejected():
    lib = nc.lib()
    assert lib.nc_model_create(None, 1, None) == 3
    assert lib.nc_forward_backward(None, None, None, 1, 1, None, None, None) == 3
    assert lib.nc_op_gemm(1, 4, 4, 4, None, 4, 1, None, 4, 1, 0, None, 4, None, 0, None, 0, None) == 3
    assert lib.nc_param_layout(None, None, None) == 3
    assert lib.nc_param_count(None, None, None) == 3


def test_fp8_and_row_gemm_arguments_rejected_without_gpu():
    lib = nc.lib()
    # E4M3 GEMM: null operands, a row pitch that is not a multiple of 16 bytes, an unknown output type
    assert lib.nc_op_gemm_fp8(64, 64, 64, None, 64, None, 64, None, None, 1, None, 64, None) == 3
    buf = ctypes.create_string_buffer(64 * 64 + 16)
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    assert lib.nc_op_gemm_fp8(64, 64, 40, p, 40, p, 40, p, p, 1, p, 64, None) == 3
    assert lib.nc_op_gemm_fp8(64, 64, 64, p, 64, p, 64, p, p, 9, p, 64, None) == 3
    # quantiser: missing stats, an unknown input type
    assert lib.nc_op_quantize_fp8(1, p, 16, p, None, None) == 3
    assert lib.nc_op_quantize_fp8(7, p, 16, p, p, None) == 3
    # skinny row GEMM: more than 32 rows
    assert lib.nc_op_gemm_rows(1, 33, 64, 64, p, 64, p, 64, 1, p, 64, None) == 3
