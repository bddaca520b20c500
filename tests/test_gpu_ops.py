"""Kernel-level parity: each CUDA kernel, called through the C ABI, against the
fp64 oracle definition of its operation on the same seeded inputs."""
import math

import numpy as np
import pytest

from oracle import model as OM
from oracle import ops as OO
from tests.gpu_util import dev_tensor, to64, rel_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decoder_only_transformer_07_b300 as nc  # noqa: E402

BF16, F32 = torch.bfloat16, torch.float32


def rnd(seed, shape, scale=1.0):
    return np.random.default_rng(seed).normal(0.0, scale, size=shape).astype(np.float32)


# ---------------------------------------------------------------- GEMM

def _gemm_case(M, N, K, a_kmajor, b_kmajor, ep, dt, seed=0, ws=False):
    a = rnd(seed, (M, K))
    b = rnd(seed + 1, (N, K))
    A = dev_tensor(a if a_kmajor else a.T.copy(), dt)
    B = dev_tensor(b if b_kmajor else b.T.copy(), dt)
    a64 = to64(A) if a_kmajor else to64(A).T
    b64 = to64(B) if b_kmajor else to64(B).T
    ref = OO.gemm(a64, b64)
    out_dt = F32 if ep in (nc.EP_STORE_F32, nc.EP_ACCUM_F32) else dt
    D = torch.zeros((M, N), dtype=out_dt, device="cuda")
    aux = None
    if ep == nc.EP_ACCUM_F32:
        base = rnd(seed + 2, (M, N))
        D.copy_(torch.from_numpy(base))
        ref = ref + base
    if ep == nc.EP_RELU2:
        aux = torch.zeros((M, N), dtype=dt, device="cuda")
    if ep in (nc.EP_RELU2_BWD, nc.EP_RELU2_SQ_BWD):
        aux = dev_tensor(np.abs(rnd(seed + 3, (M, N))), dt)
    W = torch.empty(nc.ops.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda") if ws else None
    nc.ops.gemm(A, a_kmajor, B, b_kmajor, M, N, K, D, ep=ep, aux=aux,
                dtype=nc.NC_BF16 if dt == BF16 else nc.NC_FP32, workspace=W)
    torch.cuda.synchronize()
    if ep == nc.EP_RELU2:
        h_ref, r_ref = OO.relu2(ref)
        return [(to64(D), r_ref), (to64(aux), h_ref)]
    if ep == nc.EP_RELU2_BWD:
        return [(to64(D), OO.relu2_bwd(ref, to64(aux)))]
    if ep == nc.EP_RELU2_SQ:
        return [(to64(D), OO.relu2(ref)[0])]
    if ep == nc.EP_RELU2_SQ_BWD:
        return [(to64(D), OO.relu2_bwd_from_square(ref, to64(aux)))]
    return [(to64(D), ref)]


def _assert_gemm(pairs, dt, K, ep):
    for got, want in pairs:
        scale = float(np.max(np.abs(want))) + 1e-30
        if dt == F32:
            tol = 1e-5 * math.sqrt(K) * scale / 8 + 1e-6 * scale
        elif ep in (nc.EP_STORE_F32, nc.EP_ACCUM_F32):
            tol = 2e-6 * math.sqrt(K) * scale + 1e-5 * scale
        else:
            tol = None
        if tol is not None:
            err = float(np.max(np.abs(got - want)))
            assert err <= tol, (err, tol)
        else:   # bf16 output: one rounding of a correct fp32 value
            err = np.abs(got - want)
            bound = 2.0 ** -8 * np.abs(want) + 1e-4 * scale
            assert np.all(err <= bound), float(np.max(err / bound))


LAYOUTS = [(1, 1), (1, 0), (0, 0), (0, 1)]


@pytest.mark.parametrize("a_kmajor,b_kmajor", LAYOUTS)
@pytest.mark.parametrize("dt", [BF16, F32])
def test_gemm_layouts_ragged(a_kmajor, b_kmajor, dt):
    M, N, K = 200, 328, 136
    _assert_gemm(_gemm_case(M, N, K, a_kmajor, b_kmajor, nc.EP_STORE_F32, dt), dt, K, nc.EP_STORE_F32)


@pytest.mark.parametrize("ep", [nc.EP_STORE, nc.EP_STORE_F32, nc.EP_ACCUM_F32, nc.EP_RELU2, nc.EP_RELU2_BWD,
                                nc.EP_RELU2_SQ, nc.EP_RELU2_SQ_BWD])
@pytest.mark.parametrize("dt", [BF16, F32])
def test_gemm_epilogues(ep, dt):
    M, N, K = 256, 384, 192
    _assert_gemm(_gemm_case(M, N, K, 1, 1, ep, dt, seed=10 + ep), dt, K, ep)


@pytest.mark.parametrize("a_kmajor,b_kmajor", LAYOUTS)
def test_gemm_bf16_many_tiles_long_k(a_kmajor, b_kmajor):
    # 32 x 8 = 256 output tiles (> one per SM) and 64 k-blocks: exercises the
    # persistent tile loop, both TMEM accumulators and many ring phases.
    M, N, K = 4096, 2048, 4096
    _assert_gemm(_gemm_case(M, N, K, a_kmajor, b_kmajor, nc.EP_STORE_F32, BF16, seed=7), BF16, K,
                 nc.EP_STORE_F32)


@pytest.mark.parametrize("M,N,K,ep", [(1280, 1280, 8192, nc.EP_STORE_F32),     # 50 tiles: stream-K
                                      (3840, 1280, 4096, nc.EP_STORE_F32),     # 150 tiles
                                      (640, 384, 20000, nc.EP_ACCUM_F32),      # ragged K, accumulate
                                      (1280, 5120, 2048, nc.EP_STORE_F32)])
def test_gemm_bf16_streamk_weight_gradient_shapes(M, N, K, ep):
    # dW = dY^T X: both operands MN-major, K = tokens; few output tiles
    pairs = _gemm_case(M, N, K, 0, 0, ep, BF16, seed=11, ws=True)
    _assert_gemm(pairs, BF16, K, ep)


def test_gemm_bf16_streamk_is_deterministic():
    M, N, K = 1280, 1280, 6144
    a = dev_tensor(rnd(1, (K, M)), BF16)
    b = dev_tensor(rnd(2, (K, N)), BF16)
    W = torch.empty(nc.ops.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        D = torch.empty((M, N), dtype=F32, device="cuda")
        nc.ops.gemm(a, 0, b, 0, M, N, K, D, ep=nc.EP_STORE_F32, workspace=W)
        outs.append(D)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("M", [1, 2, 5, 33])
@pytest.mark.parametrize("dt", [BF16, F32])
def test_gemm_few_rows(M, dt):
    # the decode step's projections: one row per sequence
    _assert_gemm(_gemm_case(M, 640, 256, 1, 1, nc.EP_STORE_F32, dt, seed=40 + M), dt, 256, nc.EP_STORE_F32)
    _assert_gemm(_gemm_case(M, 384, 256, 1, 1, nc.EP_ACCUM_F32, dt, seed=50 + M), dt, 256, nc.EP_ACCUM_F32)


@pytest.mark.parametrize("M", [1, 2, 5, 8, 17, 32])
@pytest.mark.parametrize("dt", [BF16, F32])
@pytest.mark.parametrize("ep", [nc.EP_STORE, nc.EP_STORE_F32, nc.EP_ACCUM_F32, nc.EP_RELU2_SQ])
@pytest.mark.parametrize("K", [1096, 4104])
def test_gemm_rows_skinny(M, dt, ep, K):
    # the decode step's CUDA-core projections: at most 32 rows, ragged N; K = 4104 spans
    # several batches of in-flight weight pieces and several staged chunks of A
    N = 333
    a, w = rnd(70 + M, (M, K)), rnd(71 + M, (N, K))
    A, W = dev_tensor(a, dt), dev_tensor(w, dt)
    out_f32 = ep in (nc.EP_STORE_F32, nc.EP_ACCUM_F32)
    d0 = rnd(72, (M, N)) if ep == nc.EP_ACCUM_F32 else np.zeros((M, N), np.float32)
    D = dev_tensor(d0, F32 if out_f32 else dt)
    nc.ops.gemm_rows(A, W, D, ep)
    acc = OO.gemm(to64(A), to64(W))
    want = {nc.EP_STORE: acc, nc.EP_STORE_F32: acc, nc.EP_ACCUM_F32: d0.astype(np.float64) + acc,
            nc.EP_RELU2_SQ: np.maximum(acc, 0.0) ** 2}[ep]
    got = to64(D)
    scale = np.abs(want).max()
    if dt == F32 or out_f32:   # fp32 accumulation of exact products of the inputs
        assert np.max(np.abs(got - want)) <= 1e-5 * scale, float(np.max(np.abs(got - want)) / scale)
    else:                      # one bf16 rounding of a correct fp32 value
        assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-4 * scale)


def test_gemm_bf16_narrow_n():
    _assert_gemm(_gemm_case(384, 64, 256, 1, 1, nc.EP_STORE_F32, BF16, seed=3), BF16, 256, nc.EP_STORE_F32)
    _assert_gemm(_gemm_case(136, 128, 72, 0, 0, nc.EP_STORE_F32, BF16, seed=4), BF16, 72, nc.EP_STORE_F32)


# ---------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("dt", [F32, BF16])
def test_rmsnorm_fwd_bwd(dt):
    rows, C, eps = 300, 768, 1.1920929e-07
    x = rnd(20, (rows, C), 0.3)
    X = dev_tensor(x, F32)
    Y = torch.empty((rows, C), dtype=dt, device="cuda")
    R = torch.empty(rows, dtype=F32, device="cuda")
    nc.ops.rmsnorm_fwd(X, Y, R, eps)
    y_ref, r_ref = OM.rms_norm(x.astype(np.float64), eps)
    torch.cuda.synchronize()
    rtol = 1e-5 if dt == F32 else 2.0 ** -8
    ok, worst = rel_close(to64(Y), y_ref, rtol, 1e-2)
    assert ok, worst
    assert np.allclose(to64(R), r_ref[:, 0], rtol=1e-5)
    dy = rnd(21, (rows, C))
    dx0 = rnd(22, (rows, C))
    DX = dev_tensor(dx0, F32)
    DXA = torch.empty((rows, C), dtype=dt, device="cuda") if dt == BF16 else None
    nc.ops.rmsnorm_bwd(dev_tensor(dy, F32), Y, R, DX, DXA)
    want = dx0 + OM.rms_norm_bwd(dy.astype(np.float64), to64(Y), to64(R)[:, None])
    torch.cuda.synchronize()
    ok, worst = rel_close(to64(DX), want, 1e-4, 1e-2)
    assert ok, worst
    if DXA is not None:
        assert torch.equal(DXA, DX.to(BF16))


# ---------------------------------------------------------------- RoPE + QK-norm

@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("dt", [F32, BF16])
def test_rope_qknorm_fwd_bwd(hd, dt):
    B, T, H, Hkv, eps, base = 2, 70, 4, 2, 1.1920929e-07, 10000.0
    W = (H + 2 * Hkv) * hd
    qkv = rnd(30, (B * T, W))
    tab = torch.empty((T, hd // 2, 2), dtype=F32, device="cuda")
    nc.ops.rope_table(T, hd, base, tab)
    cos, sin = OM.rope_tables(T, hd, base)
    torch.cuda.synchronize()
    assert np.allclose(to64(tab)[..., 0], cos, atol=1e-7) and np.allclose(to64(tab)[..., 1], sin, atol=1e-7)
    Q = dev_tensor(qkv, dt)
    q_in = to64(Q).reshape(B, T, H + 2 * Hkv, hd)
    R = torch.empty((B * T, H + Hkv), dtype=F32, device="cuda")
    nc.ops.rope_qknorm_fwd(Q, B, T, H, Hkv, hd, R, tab, eps)
    heads = q_in[:, :, :H + Hkv].transpose(0, 2, 1, 3)          # [B, nh, T, hd]
    y_ref, r_ref = OM.rms_norm(OM.rope(heads, cos, sin), eps)
    got = to64(Q).reshape(B, T, H + 2 * Hkv, hd)
    rtol = 1e-5 if dt == F32 else 2.0 ** -8
    ok, worst = rel_close(got[:, :, :H + Hkv].transpose(0, 2, 1, 3), y_ref, rtol, 1e-2)
    assert ok, worst
    assert np.array_equal(got[:, :, H + Hkv:], q_in[:, :, H + Hkv:])       # v untouched
    assert np.allclose(to64(R).reshape(B, T, H + Hkv).transpose(0, 2, 1), r_ref[..., 0], rtol=1e-5)
    # backward
    g = rnd(31, (B * T, W))
    G = dev_tensor(g, dt)
    g_in = to64(G).reshape(B, T, H + 2 * Hkv, hd)
    nc.ops.rope_qknorm_bwd(G, Q, B, T, H, Hkv, hd, R, tab)
    gh = g_in[:, :, :H + Hkv].transpose(0, 2, 1, 3)
    yh = got[:, :, :H + Hkv].transpose(0, 2, 1, 3)
    rh = to64(R).reshape(B, T, H + Hkv).transpose(0, 2, 1)[..., None]
    want = OM.rope_bwd(OM.rms_norm_bwd(gh, yh, rh), cos, sin)
    got_g = to64(G).reshape(B, T, H + 2 * Hkv, hd)
    rtol = 1e-4 if dt == F32 else 2e-2
    ok, worst = rel_close(got_g[:, :, :H + Hkv].transpose(0, 2, 1, 3), want, rtol, 1e-2)
    assert ok, worst


@pytest.mark.parametrize("pairs", [False, True])
@pytest.mark.parametrize("hd,H,Hkv", [(64, 4, 2), (128, 3, 1), (128, 2, 2)])
def test_gemm_qkv_rope_fused(hd, H, Hkv, pairs):
    """The q/k/v projection with RoPE + per-head RMSNorm in its epilogue, against
    gemm -> rope -> rms_norm of the oracle on the same bf16 inputs."""
    B, T, K, eps, base = 2, 100, 192, 1.1920929e-07, 10000.0
    M, W = B * T, (H + 2 * Hkv) * hd
    X = dev_tensor(rnd(50, (M, K)), BF16)
    Wq = dev_tensor(rnd(51, (W, K), 0.1), BF16)
    tab = torch.empty((T, hd // 2, 2), dtype=F32, device="cuda")
    nc.ops.rope_table(T, hd, base, tab)
    QKV = torch.full((M, W), float("nan"), dtype=BF16, device="cuda")
    R = torch.empty((M, H + Hkv), dtype=F32, device="cuda")
    if pairs:   # pair-major table built for more positions than T (row stride 160)
        tabp = torch.empty((hd // 4, 160, 4), dtype=F32, device="cuda")
        nc.ops.rope_table_pairs(160, hd, base, tabp)
        torch.cuda.synchronize()
        assert torch.equal(tabp[:, :T].reshape(hd // 4, T, 2, 2).permute(1, 0, 2, 3).reshape(T, hd // 2, 2), tab)
        nc.ops.gemm_qkv_rope(X, Wq, QKV, T, H, Hkv, hd, R, tabp, eps, pair_rows=160)
    else:
        nc.ops.gemm_qkv_rope(X, Wq, QKV, T, H, Hkv, hd, R, tab, eps)
    torch.cuda.synchronize()
    u = OO.gemm(to64(X), to64(Wq)).reshape(B, T, H + 2 * Hkv, hd)
    cos, sin = OM.rope_tables(T, hd, base)
    heads = u[:, :, :H + Hkv].transpose(0, 2, 1, 3)
    y_ref, r_ref = OM.rms_norm(OM.rope(heads, cos, sin), eps)
    got = to64(QKV).reshape(B, T, H + 2 * Hkv, hd)
    # one bf16 rounding of a value computed in fp32 from exact products
    ok, worst = rel_close(got[:, :, :H + Hkv].transpose(0, 2, 1, 3), y_ref, 2.0 ** -8, 1e-2)
    assert ok, worst
    ok, worst = rel_close(got[:, :, H + Hkv:], u[:, :, H + Hkv:], 2.0 ** -8, 1e-2)
    assert ok, worst
    assert np.allclose(to64(R).reshape(B, T, H + Hkv).transpose(0, 2, 1), r_ref[..., 0], rtol=1e-4)


# ---------------------------------------------------------------- attention

def _attn_ref(qkv, B, T, H, Hkv, hd, do=None):
    x = qkv.reshape(B, T, H + 2 * Hkv, hd)
    G = H // Hkv
    o = np.zeros((B, T, H, hd))
    lse = np.zeros((B, H, T))
    dqkv = np.zeros_like(x)
    for b in range(B):
        for h in range(H):
            g = h // G
            q, k, v = x[b, :, h], x[b, :, H + g], x[b, :, H + Hkv + g]
            o[b, :, h], lse[b, h] = OM.attention(q, k, v)
            if do is not None:
                dq, dk, dv = OM.attention_bwd(q, k, v, do.reshape(B, T, H, hd)[b, :, h])
                dqkv[b, :, h] = dq
                dqkv[b, :, H + g] += dk
                dqkv[b, :, H + Hkv + g] += dv
    return o.reshape(B * T, H * hd), lse, dqkv.reshape(B * T, -1)


@pytest.mark.parametrize("hd,H,Hkv,T", [(64, 4, 2, 100), (128, 3, 1, 100), (128, 2, 2, 100),
                                          (128, 6, 2, 300), (64, 2, 1, 257)])
@pytest.mark.parametrize("dt", [F32, BF16])
def test_attention_fwd_bwd(hd, H, Hkv, T, dt):
    B = 2
    W = (H + 2 * Hkv) * hd
    QKV = dev_tensor(rnd(40, (B * T, W)), dt)
    qkv = to64(QKV)
    O = torch.empty((B * T, H * hd), dtype=dt, device="cuda")
    L = torch.empty((B, H, T), dtype=F32, device="cuda")
    nc.ops.attention_fwd(QKV, B, T, H, Hkv, hd, O, L)
    DO = dev_tensor(rnd(41, (B * T, H * hd)), dt)
    o_ref, lse_ref, d_ref = _attn_ref(qkv, B, T, H, Hkv, hd, to64(DO))
    torch.cuda.synchronize()
    if dt == F32:
        ok, worst = rel_close(to64(O), o_ref, 1e-4, 1e-2)
    else:
        # bf16 path: P is rounded to bf16 (2^-9 relative) before P V, so the
        # error of an output element scales with rms(o), not with |o|
        # (sigma ~ 2^-9 rms(o) per element, 2^-9 relative for the bf16 store):
        # per element 2^-7 |o| + 2^-5 rms(o) (about 6 sigma over ~5e5
        # elements), and the aggregate cosine >= 0.99999.
        from tests.gpu_util import cosine
        ok, worst = rel_close(to64(O), o_ref, 2.0 ** -7, 4.0)
        assert cosine(to64(O), o_ref) > 0.99999
    assert ok, worst
    assert np.allclose(to64(L), lse_ref, rtol=1e-5, atol=1e-5)
    DQKV = torch.zeros((B * T, W), dtype=dt, device="cuda")
    ws = torch.empty(B * H * T, dtype=F32, device="cuda")
    nc.ops.attention_bwd(QKV, O, L, DO, B, T, H, Hkv, hd, DQKV, ws)
    torch.cuda.synchronize()
    if dt == F32:
        # the oracle backward uses the oracle forward's o; the kernel uses its own
        ok, worst = rel_close(to64(DQKV), d_ref, 1e-3, 1e-2)
        assert ok, worst
    else:
        # bf16 inputs, bf16 P and dS operands: compare per q/k/v block by cosine
        from tests.gpu_util import cosine
        got = to64(DQKV).reshape(B, T, H + 2 * Hkv, hd)
        ref = d_ref.reshape(B, T, H + 2 * Hkv, hd)
        for name, sl in (("dq", slice(0, H)), ("dk", slice(H, H + Hkv)), ("dv", slice(H + Hkv, None))):
            assert cosine(got[:, :, sl], ref[:, :, sl]) > 0.9999, name


@pytest.mark.parametrize("pairs", [False, True])
@pytest.mark.parametrize("hd,H,Hkv,T", [(128, 4, 2, 300), (64, 2, 1, 200), (128, 2, 2, 128), (128, 3, 1, 257)])
def test_attention_bwd_with_fused_rope_qknorm_bwd(hd, H, Hkv, T, pairs):
    """Attention backward whose dq / dk leave through the QK-norm and RoPE
    backward, against the oracle's attention backward followed by its RMSNorm
    and rotation backward on the same normalised bf16 q, k, v."""
    B, eps, base = 2, 1.1920929e-07, 10000.0
    W = (H + 2 * Hkv) * hd
    QKV = dev_tensor(rnd(60, (B * T, W)), BF16)
    tab = torch.empty((T, hd // 2, 2), dtype=F32, device="cuda")
    nc.ops.rope_table(T, hd, base, tab)
    R = torch.empty((B * T, H + Hkv), dtype=F32, device="cuda")
    nc.ops.rope_qknorm_fwd(QKV, B, T, H, Hkv, hd, R, tab, eps)      # q, k now rotated and normalised
    O = torch.empty((B * T, H * hd), dtype=BF16, device="cuda")
    L = torch.empty((B, H, T), dtype=F32, device="cuda")
    nc.ops.attention_fwd(QKV, B, T, H, Hkv, hd, O, L)
    DO = dev_tensor(rnd(61, (B * T, H * hd)), BF16)
    DQKV = torch.zeros((B * T, W), dtype=BF16, device="cuda")
    ws = torch.empty(B * H * T, dtype=F32, device="cuda")
    if pairs:   # the pair-major table, built for more positions than T
        ptab = torch.empty((hd // 4, T + 5, 4), dtype=F32, device="cuda")
        nc.ops.rope_table_pairs(T + 5, hd, base, ptab)
        nc.ops.attention_bwd_rope(QKV, O, L, DO, B, T, H, Hkv, hd, DQKV, ws, R, ptab, pair_rows=T + 5)
    else:
        nc.ops.attention_bwd_rope(QKV, O, L, DO, B, T, H, Hkv, hd, DQKV, ws, R, tab)
    torch.cuda.synchronize()
    qkv = to64(QKV)
    _, _, d_ref = _attn_ref(qkv, B, T, H, Hkv, hd, to64(DO))
    cos, sin = OM.rope_tables(T, hd, base)
    g = d_ref.reshape(B, T, H + 2 * Hkv, hd)[:, :, :H + Hkv].transpose(0, 2, 1, 3)
    y = qkv.reshape(B, T, H + 2 * Hkv, hd)[:, :, :H + Hkv].transpose(0, 2, 1, 3)
    rr = to64(R).reshape(B, T, H + Hkv).transpose(0, 2, 1)[..., None]
    want_qk = OM.rope_bwd(OM.rms_norm_bwd(g, y, rr), cos, sin)
    got = to64(DQKV).reshape(B, T, H + 2 * Hkv, hd)
    from tests.gpu_util import cosine
    got_qk = got[:, :, :H + Hkv].transpose(0, 2, 1, 3)
    assert cosine(got_qk[:, :H], want_qk[:, :H]) > 0.9999, "dq"
    assert cosine(got_qk[:, H:], want_qk[:, H:]) > 0.9999, "dk"
    want_v = d_ref.reshape(B, T, H + 2 * Hkv, hd)[:, :, H + Hkv:]
    assert cosine(got[:, :, H + Hkv:], want_v) > 0.9999, "dv"


# ---------------------------------------------------------------- cross-entropy

@pytest.mark.parametrize("dt", [F32, BF16])
def test_cross_entropy(dt):
    rows, V = 64, 1000
    Z = dev_tensor(rnd(50, (rows, V), 2.0), dt)
    z = to64(Z)
    tgt = np.random.default_rng(51).integers(0, V, size=rows).astype(np.int32)
    TG = torch.from_numpy(tgt).cuda()
    RL = torch.empty(rows, dtype=F32, device="cuda")
    nc.ops.cross_entropy(Z, TG, RL, 0.5)
    loss_ref, dz_ref = OM.cross_entropy(z, tgt)
    torch.cuda.synchronize()
    assert np.allclose(to64(RL), loss_ref, rtol=1e-5, atol=1e-5)
    rtol = 1e-5 if dt == F32 else 2.0 ** -8
    ok, worst = rel_close(to64(Z), 0.5 * dz_ref, rtol, 1e-3)
    assert ok, worst


@pytest.mark.parametrize("V", [16384, 65536])
def test_cross_entropy_wide_rows_bf16(V):
    # the vocabulary-sized rows of the step (two-pass streaming kernel)
    rows = 24
    Z = dev_tensor(rnd(52, (rows, V), 3.0), BF16)
    z = to64(Z)
    tgt = np.random.default_rng(53).integers(0, V, size=rows).astype(np.int32)
    TG = torch.from_numpy(tgt).cuda()
    RL = torch.empty(rows, dtype=F32, device="cuda")
    nc.ops.cross_entropy(Z, TG, RL, 0.25)
    loss_ref, dz_ref = OM.cross_entropy(z, tgt)
    torch.cuda.synchronize()
    assert np.allclose(to64(RL), loss_ref, rtol=1e-5, atol=1e-5)
    ok, worst = rel_close(to64(Z), 0.25 * dz_ref, 2.0 ** -8, 1e-3)
    assert ok, worst


def test_cross_entropy_flags_bad_target():
    Z = torch.zeros((4, 64), dtype=F32, device="cuda")
    TG = torch.tensor([0, 64, 3, -1], dtype=torch.int32, device="cuda")
    RL = torch.empty(4, dtype=F32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    nc.ops.cross_entropy(Z, TG, RL, 1.0, err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1


# ---------------------------------------------------------------- embedding

@pytest.mark.parametrize("dt_code", [nc.NC_FP32, nc.NC_BF16])
def test_embed_gather_bit_exact(dt_code):
    V, C, n = 5000, 256, 777
    wte = rnd(60, (V, C), 0.02)
    tok = np.random.default_rng(61).integers(0, V, size=n).astype(np.int32)
    WTE = dev_tensor(wte, F32)
    X = torch.empty((n, C), dtype=F32, device="cuda")
    nc.ops.embed_fwd(torch.from_numpy(tok).cuda(), WTE, X, dt_code)
    want = torch.from_numpy(OO.embed(wte, tok))
    if dt_code == nc.NC_BF16:
        want = want.to(BF16).float()
    torch.cuda.synchronize()
    assert torch.equal(X.cpu(), want)


def test_embed_scatter_deterministic_and_exact_rows():
    import synthetic as S
    V, C = 4096, 384
    n = 6000                                     # 24 chunks, ragged tail
    tok = S.token_stream(V, 1, n - 1, "zipf", seed=62).reshape(-1)
    dx = rnd(63, (n, C))
    TOK = torch.from_numpy(tok).cuda()
    DX = dev_tensor(dx, F32)
    scratch = torch.empty(nc.ops.embed_bwd_scratch_bytes(n, C, V), dtype=torch.uint8, device="cuda")
    out1 = torch.full((V, C), float("nan"), dtype=F32, device="cuda")
    out2 = torch.full((V, C), float("nan"), dtype=F32, device="cuda")
    nc.ops.embed_bwd(TOK, DX, out1, scratch)
    nc.ops.embed_bwd(TOK, DX, out2, scratch)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)                                   # bitwise reproducible
    got = to64(out1)
    want = OO.embed_bwd(tok, dx, V)
    present = np.zeros(V, dtype=bool)
    present[tok] = True
    assert np.all(got[~present] == 0.0) and not np.any(np.signbit(got[~present]))
    assert np.all(np.any(got[present] != 0.0, axis=1))
    assert np.allclose(got, want, rtol=1e-5, atol=1e-5 * np.sqrt(np.bincount(tok).max()))


def test_embed_scatter_skips_out_of_range_ids():
    """Ids outside [0, V) add to no row (no out-of-bounds write): every row
    equals the oracle's scatter of the same positions with the bad ones left out."""
    import synthetic as S
    V, C = 2048, 256
    n = 1500                                     # 6 chunks, ragged tail
    tok = S.token_stream(V, 1, n - 1, "zipf", seed=64).reshape(-1).copy()
    bad = np.array([3, 700, 701, 1499])
    tok[bad] = [V, -1, 1 << 30, V + 7]
    dx = rnd(65, (n, C))
    keep = np.ones(n, dtype=bool)
    keep[bad] = False
    scratch = torch.empty(nc.ops.embed_bwd_scratch_bytes(n, C, V), dtype=torch.uint8, device="cuda")
    got = torch.full((V, C), float("nan"), dtype=F32, device="cuda")
    nc.ops.embed_bwd(torch.from_numpy(tok).cuda(), dev_tensor(dx, F32), got, scratch)
    tk = np.ascontiguousarray(tok[keep])
    torch.cuda.synchronize()
    want = OO.embed_bwd(tk, dx[keep], V)
    g = to64(got)
    assert np.all(np.isfinite(g))
    assert np.allclose(g, want, rtol=1e-5, atol=1e-5 * np.sqrt(np.bincount(tk).max()))
    present = np.zeros(V, dtype=bool)
    present[tk] = True
    assert np.all(g[~present] == 0.0)
