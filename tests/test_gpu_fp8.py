"""The 8-bit path (nc_op_quantize_fp8, nc_op_gemm_fp8) against the oracle.

* Quantisation is integer work decided in fp32 on both sides: the codes and
  the three statistics must match bit for bit.
* The GEMM's products of E4M3 values are exact; what is left is the order and
  precision of the tensor cores' fp32 accumulation and the output rounding.
  The bound per element is |D - O| <= 2^-10 * alpha * sum_k |A(m,k) B(n,k)|
  (an accumulator keeping 10 bits below the largest partial sum), plus half
  a bf16 ulp of |O| for bf16 outputs.  A transposed operand, a wrong scale or
  a dropped / repeated K block moves an element by a sizeable fraction of
  sqrt(K) typical products, far beyond that bound at these K.
"""
import numpy as np
import pytest

import synthetic as S
from oracle import fp8 as F

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("n", [1, 7, 8, 4096 * 13 + 5, 1_000_003])
def test_quantize_bitexact(dtype, n):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * 2.5).astype(np.float32)
    x[rng.integers(0, n, max(1, n // 1000))] *= 40.0          # a few outliers set the scale
    xt = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        xt = xt.to(torch.bfloat16)
        x = xt.float().cpu().numpy()                          # the values the kernel sees
    codes, stats = nc.ops.quantize_fp8(xt)
    want, amax, scale, scale_inv = F.quantize(x)
    st = stats.cpu().numpy()
    assert st[0] == amax and st[1] == scale and st[2] == scale_inv
    got = codes.cpu().numpy()
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (bad[:8], got[bad[:8]], want[bad[:8]], x[bad[:8]])


def test_quantize_degenerate():
    z = torch.zeros(1000, dtype=torch.float32, device="cuda")
    codes, stats = nc.ops.quantize_fp8(z)
    assert stats.cpu().tolist() == [0.0, 1.0, 1.0] and not codes.any()
    e = torch.zeros(0, dtype=torch.float32, device="cuda")
    codes, stats = nc.ops.quantize_fp8(e)
    assert stats.cpu().tolist() == [0.0, 1.0, 1.0]
    with pytest.raises(nc.NcError):
        nc.ops.quantize_fp8(torch.zeros(64, dtype=torch.float32, device="cuda")[1:])   # not 16-byte aligned


def _check_gemm(D, a, b, sa, sb, rows=None):
    """D: the GPU result (torch, fp32 or bf16), rows of the product given by `rows` (all if None)."""
    bf16_out = D.dtype == torch.bfloat16
    g = D.float().cpu().numpy().astype(np.float64)
    a = a if rows is None else a[rows]
    A, B = F.e4m3_decode(a), F.e4m3_decode(b)
    want = F.gemm(a, b, sa, sb)
    alpha = float(sa) * float(sb)
    bound = 2.0 ** -10 * alpha * (np.abs(A) @ np.abs(B).T)
    if bf16_out:
        bound = bound + 2.0 ** -8 * np.abs(want)
    err = np.abs(g - want)
    assert np.all(err <= bound), (float(np.max(err / np.maximum(bound, 1e-30))), np.argwhere(err > bound)[:5])


@pytest.mark.parametrize("M,N,K", [(300, 520, 400),      # CTA pairs, ragged M, N and K tails
                                   (100, 200, 272),      # single CTA, 128 x 256 tiles
                                   (130, 96, 144),       # single CTA, 128 x 128 tiles
                                   (512, 256, 1024)])
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_gemm_fp8_matches_oracle(M, N, K, out):
    a = S.fp8_codes(M, K, seed=11)
    b = S.fp8_codes(N, K, seed=12)
    sa, sb = np.float32(2.0 ** -5), np.float32(0.0123)
    sc = torch.tensor([sa, sb], dtype=torch.float32, device="cuda")
    D = torch.empty((M, N), dtype=torch.float32 if out == "fp32" else torch.bfloat16, device="cuda")
    nc.ops.gemm_fp8(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), sc[0:1], sc[1:2], D)
    _check_gemm(D, a, b, sa, sb)


@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_gemm_fp8_every_finite_code(out):
    """Operands over every finite E4M3 code, with rows of subnormals only and
    rows and columns of the saturated magnitude 448 (the quantiser's code for
    amax), on CTA pairs with ragged tails."""
    M, N, K = 384, 320, 512
    a = S.fp8_codes_all(M, K, seed=21)
    b = S.fp8_codes_all(N, K, seed=22)
    a[5] = np.where(np.arange(K) % 2, 0x7E, 0xFE)          # +-448
    b[7] = 0x7E
    a[9] = (np.arange(K) % 7 + 1).astype(np.uint8)         # subnormals 2^-9 .. 7 * 2^-9
    b[11] = (np.arange(K) % 7 + 0x81).astype(np.uint8)     # negative subnormals
    assert np.all(np.isin(np.arange(256)[(np.arange(256) != 0x7F) & (np.arange(256) != 0xFF)], a))
    sa, sb = np.float32(2.0 ** -7), np.float32(0.0371)
    sc = torch.tensor([sa, sb], dtype=torch.float32, device="cuda")
    D = torch.empty((M, N), dtype=torch.float32 if out == "fp32" else torch.bfloat16, device="cuda")
    nc.ops.gemm_fp8(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), sc[0:1], sc[1:2], D)
    _check_gemm(D, a, b, sa, sb)
    if out == "fp32":
        # 448 * 448 * K products of equal sign are exact in fp32: D(5, 7) is their alternating sum, 0
        assert float(D[5, 7]) == 0.0


def test_gemm_fp8_row_pitch_and_unaligned_k():
    """K = 40 inside rows of 48 bytes: the tail of each K block is read as zeros."""
    M, N, K = 260, 300, 40
    a = np.ascontiguousarray(S.fp8_codes(M, 48, seed=13))
    b = np.ascontiguousarray(S.fp8_codes(N, 48, seed=14))
    sc = torch.ones(2, dtype=torch.float32, device="cuda")
    D = torch.empty((M, N + 4), dtype=torch.float32, device="cuda")
    nc.ops.gemm_fp8(torch.from_numpy(a).cuda()[:, :K], torch.from_numpy(b).cuda()[:, :K], sc[0:1], sc[1:2],
                    D[:, :N])
    _check_gemm(D[:, :N], a[:, :K], b[:, :K], 1.0, 1.0)


def test_gemm_fp8_argument_errors():
    a = torch.zeros((64, 40), dtype=torch.uint8, device="cuda")
    b = torch.zeros((64, 40), dtype=torch.uint8, device="cuda")
    sc = torch.ones(2, dtype=torch.float32, device="cuda")
    D = torch.empty((64, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(nc.NcError):
        nc.ops.gemm_fp8(a, b, sc[0:1], sc[1:2], D)            # row pitch 40 bytes: not a multiple of 16
    with pytest.raises(nc.NcError):
        nc.ops.gemm_fp8(a[:, :0], b[:, :0], sc[0:1], sc[1:2], D)   # K = 0


def test_gemm_fp8_full_size_sampled():
    """The benchmark's launch: the d20 MLP up-projection shape, 65536 x 5120 x 1280, bf16 out,
    checked on sampled rows (tile edges and random ones) over every column."""
    M, N, K = 65536, 5120, 1280
    a = S.fp8_codes(M, K, seed=15)
    b = S.fp8_codes(N, K, seed=16)
    sa, sb = np.float32(2.0 ** -6), np.float32(2.0 ** -7)
    sc = torch.tensor([sa, sb], dtype=torch.float32, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    nc.ops.gemm_fp8(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), sc[0:1], sc[1:2], D)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 257, M - 1],
                                     np.random.default_rng(17).integers(0, M, 40)]))
    _check_gemm(D[torch.from_numpy(rows).cuda()], a, b, sa, sb, rows=rows)
