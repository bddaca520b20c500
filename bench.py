"""Benchmark: training tokens/s and MFU of one forward+backward GPT step on B300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config d26] [--impl ours|reference]

Prints ONE JSON line (rank 0).  The default workload is d26, the largest
single-GPU configuration; on one GPU the d20, d24-GQA and d12 workloads are
measured in the same run and reported under "other_configs" with the same
fields.  A step is one nc_forward_backward call over a full batch of the
workload: weight cast, forward, chunked lm_head +
cross-entropy, backward, fp32 gradient write, loss read-back.  `value` is
timed with CUDA events on the launching stream with inputs already resident
in HBM; `e2e` times the same step through nc_forward_backward_host from
pinned host buffers (host->device token copies and the loss read inside the
timed region).  The working set (GBs of activations) is far larger than L2,
so no explicit L2 flush is needed between steps.

With N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the step has no data-path exchange here); `value` sums all ranks' tokens over
the slowest rank's time.

`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload on this host's cores (rank 0 only).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402

METRIC = "train tokens/sec and MFU at 1 B300 (fwd+bwd step), vs CPU oracle tok/s"
UNIT = "tokens/s"
DESCR = {
    "tiny": "tiny GPT L2 C128 H2/2 hd64 F512 V512 T64 B2 (fp32)",
    "d12": "d12 GPT L12 C768 H6/6 hd128 F3072 V65536 T2048 B32 (bf16)",
    "d20": "d20 GPT L20 C1280 H10/10 hd128 F5120 V65536 T2048 B32 (bf16)",
    "d26": "d26 GPT L26 C1664 H13/13 hd128 F6656 V65536 T2048 B16 (bf16)",
    "d24gqa": "d24 GQA GPT L24 C1536 H12/4 hd128 F6144 V65536 T4096 B8 (bf16)",
}
# DRAM traffic per GEMM call (main kernel + split-K fix-up) per workload: ncu
# dram__bytes_read.sum + dram__bytes_write.sum of every distinct GEMM launch of
# one step (`bench.py --op gemmset --config <w>`, each launch at full size),
# weighted by the step's call counts.  A workload is left out (null traffic)
# whenever the GEMM kernels change and the capture is not repeated.
GEMM_DRAM_BYTES_PER_CALL = {"d26": 9.104e+08, "d20": 1.262e+09, "d24gqa": 7.151e+08, "d12": 6.803e+08}
# CPU-oracle sample (tokens of one sequence) per workload: ~10-30 s of fp64 work
CPU_SAMPLE_T = {"tiny": 64, "d12": 128, "d20": 64, "d26": 48, "d24gqa": 48}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops", 1800.0), d.get("bf16_tflops_sustained", 1400.0), d.get("hbm_gbs", 6400.0), "measured"
    return 1800.0, 1400.0, 6400.0, "fallback"


def flops_per_token(w):
    """Algorithmic training FLOPs per token (forward + backward).

    6 * (matrix parameters: every weight except the embedding table, which is
    a gather) + causal attention 6 * L * H * hd * T (QK^T and PV, forward x3,
    each query attending to T/2 keys on average).  Also returns the
    full-square attention and 6 * N_total conventions.
    """
    C, H, Hkv, hd, F, V, L, T = (w.n_embd, w.n_head, w.n_kv_head, w.head_dim, w.mlp_hidden, w.vocab,
                                 w.depth, w.seq_len)
    n_layer = C * H * hd + 2 * C * Hkv * hd + H * hd * C + 2 * C * F
    n_mm = L * n_layer + V * C
    n_total = n_mm + V * C
    attn_causal = 6 * L * H * hd * T
    return {"causal": 6 * n_mm + attn_causal, "full_square": 6 * n_mm + 2 * attn_causal,
            "six_n_total": 6 * n_total, "n_mm": n_mm, "n_total": n_total}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        rows = [l.split(",") for l in open(self.f.name).read().strip().splitlines() if l.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample(w, t_sample, steps, warmup):
    """Time the fp64 oracle on one sequence of t_sample tokens (weights N(0, 0.02))."""
    from oracle import model as OM
    cfg = OM.Config.from_workload(w)
    rng = np.random.default_rng(S.WEIGHT_SEED)
    W = {name: rng.standard_normal((r, c)) * 0.02 for name, r, c, _ in OM.param_layout(cfg)}
    tok, tgt = S.batch_tokens(w, batch=1, seq_len=t_sample)
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        OM.forward_backward(cfg, W, tok, tgt)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    try:
        from threadpoolctl import threadpool_info
        threads = max([d.get("num_threads", 1) for d in threadpool_info()] or [1])
    except Exception:
        threads = os.cpu_count()
    return t_sample / statistics.median(times), threads, times


def sample_flops_per_token(w, t_sample):
    """Algorithmic FLOPs per token of the oracle's sample (one sequence of
    t_sample tokens): the matrix term plus causal attention at that length."""
    f = flops_per_token(w)
    return f["causal"] - 6 * w.depth * w.n_head * w.head_dim * (w.seq_len - t_sample)


def cpu_baseline(w, name):
    """The oracle on the host cores: one sequence of CPU_SAMPLE_T tokens.  At
    that length attention costs far less per token than at the workload's T,
    so the line also gives the sample's FLOPs per token and the rate scaled to
    the workload's FLOPs per token (the oracle's matrix products run at a
    roughly constant FLOP rate)."""
    t_sample = CPU_SAMPLE_T.get(name, 64)
    tps, threads, _ = oracle_sample(w, t_sample, 1, 0)
    fs, fw = sample_flops_per_token(w, t_sample), flops_per_token(w)["causal"]
    return {"value": tps, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"one sequence of {t_sample} tokens of the {name} workload, fp64 NumPy fwd+bwd",
            "sample_flops_per_token": fs, "workload_flops_per_token": fw,
            "value_at_workload_flops_per_token": tps * fs / fw}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    """The maximum of x over all ranks (every rank gets it); x itself when
    world == 1.  device: "cuda" under NCCL, "cpu" under gloo."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_step, steps, ms):
    """Whole-job tokens/s of `world` independent replicas that each ran `steps`
    steps of `tokens_per_step` tokens, timed by the slowest rank (ms)."""
    return world * tokens_per_step * steps / (ms / 1e3)


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    t_sample = CPU_SAMPLE_T.get(args.config, 64)
    tps, threads, times = oracle_sample(w, t_sample, args.steps, args.warmup)
    fs, fw = sample_flops_per_token(w, t_sample), flops_per_token(w)["causal"]
    # the host cores run it; n_gpus is the N the arm was launched for
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {**arm_config(args.config, w, world), "sample": f"1 x {t_sample} tokens"},
            "cpu_baseline": {"value": tps, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"one sequence of {t_sample} tokens of the {args.config} workload, "
                                       f"fp64 NumPy forward+backward",
                             "sample_flops_per_token": fs, "workload_flops_per_token": fw,
                             "value_at_workload_flops_per_token": tps * fs / fw},
            "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_optim(args):
    """Optimizer mode: times nc_optimizer_step (Muon for every weight matrix,
    AdamW for wte and lm_head) on the --config model with seeded synthetic
    gradients, then splits one profiled step into its Newton-Schulz products
    (tensor cores) and its elementwise kernels (HBM)."""
    import ctypes
    import statistics
    import torch
    import decoder_only_transformer_07_b300 as nc
    torch.cuda.set_device(0)
    w = S.workload(args.config)
    model = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    g = torch.Generator(device="cuda").manual_seed(3)
    grads = torch.randn(model.n_params, device="cuda", generator=g) * 1e-3
    oc = nc.optim_config()
    for _ in range(args.warmup):
        model.optimizer_step(grads, oc)
    torch.cuda.synchronize()
    times = []
    for _ in range(args.iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        model.optimizer_step(grads, oc)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    lib = nc.lib()
    lib.nc_profile_enable(model.handle, 1)
    model.optimizer_step(grads, oc)
    torch.cuda.synchronize()
    phases = {}
    for cls, name in ((13, "newton_schulz"), (14, "elementwise")):
        t, n, fl, by = ctypes.c_double(), ctypes.c_int64(), ctypes.c_double(), ctypes.c_double()
        lib.nc_profile_read(model.handle, cls, ctypes.byref(t), ctypes.byref(n), ctypes.byref(fl), ctypes.byref(by))
        phases[name] = {"ms": t.value, "launches": n.value, "tflops": fl.value / t.value / 1e9 if t.value else None,
                        "gbs": by.value / t.value / 1e6 if t.value else None}
    lib.nc_profile_enable(model.handle, 0)
    _, sustained, hbm, kind = load_peaks()
    ns, ew = phases["newton_schulz"], phases["elementwise"]
    print(json.dumps({"op": "optim", "config": args.config, "ms": statistics.median(times), "iters": args.iters,
                      "phases": phases,
                      "roofline": {"bound": "tensor", "achieved": ns["tflops"], "peak": sustained, "unit": "TFLOP/s",
                                   "frac": ns["tflops"] / sustained, "peak_kind": f"bf16 dense, sustained ({kind})",
                                   "kernel": "Newton-Schulz products (tcgen05 GEMM)"},
                      "elementwise_hbm_frac": ew["gbs"] / hbm if ew["gbs"] else None,
                      "optimizer_steps": model.optimizer_steps()}), flush=True)
    model.close()


def run_decode(args):
    """Decode mode: prefill --batch prompts of --seq tokens of the --config
    model, then time --iters decode steps (one token per sequence each).
    Decoding is memory-bound: every step reads each weight once (all but the
    embedding table) and the whole key/value cache, which is the algorithmic
    byte count the HBM roofline uses."""
    import statistics
    import numpy as np
    import torch
    import decoder_only_transformer_07_b300 as nc
    torch.cuda.set_device(0)
    w = S.workload(args.config)
    B, T0, K = args.batch, args.seq, args.iters
    model = nc.Model(nc.config_from_workload(w), seed=S.WEIGHT_SEED)
    model.kv_cache_create(B, T0 + K + args.warmup + 1)
    tok, _ = S.batch_tokens(w, batch=B, seq_len=T0 + K + args.warmup + 1)
    dev = torch.from_numpy(tok).cuda()
    model.prefill(dev[:, :T0].contiguous())
    steps = [dev[:, T0 + j].contiguous() for j in range(K + args.warmup)]
    for j in range(args.warmup):
        model.decode_step(steps[j])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for j in range(K):
        model.decode_step(steps[args.warmup + j])
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    act = 2 if w.dtype == "bf16" else 4
    n_w = model.n_params - w.vocab * w.n_embd
    avg_len = T0 + args.warmup + (K + 1) / 2.0
    kv_bytes = w.depth * B * w.n_kv_head * avg_len * w.head_dim * 2 * act
    step_bytes = n_w * act + kv_bytes
    _, _, hbm, kind = load_peaks()
    gbs = step_bytes / (ms / 1e3) / 1e9
    print(json.dumps({"op": "decode", "config": args.config, "batch": B, "prompt": T0, "steps": K,
                      "ms_per_step": ms, "tokens_per_s": B / (ms / 1e3),
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                                   "peak_kind": kind, "bytes_per_step": step_bytes,
                                   "kernel": "whole decode step (weights + KV cache read once)"}}), flush=True)
    model.close()


def run_gemm8(args):
    """The 8-bit GEMM against the bf16 GEMM on the same shape (default: the d20
    MLP up-projection, 65536 x 5120 x 1280, bf16 output), and the per-tensor
    quantisation of the bf16 A operand.  The 8-bit tensor-core peak is taken
    as twice the measured bf16 peak (the nominal fp8 : bf16 dense ratio)."""
    import torch
    import decoder_only_transformer_07_b300 as nc
    torch.cuda.set_device(0)
    bf16_peak, bf16_sus, hbm, kind = load_peaks()
    g = torch.Generator(device="cuda").manual_seed(0)
    M, N, K = args.m, args.n, args.k
    a8 = torch.randint(0x20, 0x60, (M, K), dtype=torch.uint8, device="cuda", generator=g)
    b8 = torch.randint(0x20, 0x60, (N, K), dtype=torch.uint8, device="cuda", generator=g)
    a8 |= torch.randint(0, 2, (M, K), dtype=torch.uint8, device="cuda", generator=g) << 7
    b8 |= torch.randint(0, 2, (N, K), dtype=torch.uint8, device="cuda", generator=g) << 7
    sc = torch.tensor([2.0 ** -6, 2.0 ** -7], dtype=torch.float32, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    A16 = torch.randn((M, K), device="cuda", generator=g).to(torch.bfloat16)
    B16 = torch.randn((N, K), device="cuda", generator=g).to(torch.bfloat16)
    W = torch.empty(nc.ops.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    codes = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    stats = torch.empty(3, dtype=torch.float32, device="cuda")

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    flops = 2.0 * M * N * K
    ms8 = timed(lambda: nc.ops.gemm_fp8(a8, b8, sc[0:1], sc[1:2], D))
    ms16 = timed(lambda: nc.ops.gemm(A16, True, B16, True, M, N, K, D, ep=0, workspace=W))
    msq = timed(lambda: nc.ops.quantize_fp8(A16, codes, stats))
    tf8, tf16 = flops / (ms8 / 1e3) / 1e12, flops / (ms16 / 1e3) / 1e12
    qbytes = 5.0 * M * K          # two passes: read 2 B per value twice, write 1 B
    qgbs = qbytes / (msq / 1e3) / 1e9
    print(json.dumps({"op": "gemm8", "shape": [M, N, K], "iters": args.iters,
                      "fp8": {"ms": ms8, "tflops": tf8, "peak": 2 * bf16_peak, "frac": tf8 / (2 * bf16_peak),
                              "frac_of_sustained": tf8 / (2 * bf16_sus)},
                      "bf16": {"ms": ms16, "tflops": tf16, "frac": tf16 / bf16_peak},
                      "speedup": ms16 / ms8,
                      "quantize_bf16": {"ms": msq, "gbs": qgbs, "frac_of_hbm": qgbs / hbm, "bytes": qbytes},
                      "peak_kind": kind + " (fp8 = 2 x bf16)"}), flush=True)


def run_op(args):
    """Single-kernel mode (for ncu captures of one kernel on a small case):
    times --iters launches of one GEMM or one attention forward+backward."""
    import torch
    import decoder_only_transformer_07_b300 as nc
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda").manual_seed(0)
    times = []
    if args.op == "gemm":
        M, N, K = args.m, args.n, args.k
        A = torch.randn((M, K) if args.a_major == "k" else (K, M), device="cuda", generator=g).to(torch.bfloat16)
        B = torch.randn((N, K) if args.b_major == "k" else (K, N), device="cuda", generator=g).to(torch.bfloat16)
        D = torch.empty((M, N), dtype=torch.float32 if args.ep in (1, 2) else torch.bfloat16, device="cuda")
        aux = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda") if args.ep in (3, 4, 6) else None
        W = torch.empty(nc.ops.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
        flops = 2.0 * M * N * K

        def once():
            nc.ops.gemm(A, args.a_major == "k", B, args.b_major == "k", M, N, K, D, ep=args.ep, aux=aux,
                        workspace=W)
    else:
        Bsz, T, H, Hkv, hd = args.batch, args.seq, args.heads, args.kv_heads, args.head_dim
        W_ = (H + 2 * Hkv) * hd
        qkv = (torch.randn((Bsz * T, W_), device="cuda", generator=g)).to(torch.bfloat16)
        o = torch.empty((Bsz * T, H * hd), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((Bsz, H, T), dtype=torch.float32, device="cuda")
        do = torch.randn((Bsz * T, H * hd), device="cuda", generator=g).to(torch.bfloat16)
        dqkv = torch.empty_like(qkv)
        ws = torch.empty(Bsz * H * T, dtype=torch.float32, device="cuda")
        # the training step's backward: dq, dk leave through the QK-norm and RoPE backward
        tab = torch.empty((hd // 4, T, 4), dtype=torch.float32, device="cuda")   # pair-major, as the step uses
        nc.ops.rope_table_pairs(T, hd, 10000.0, tab)
        rstd = torch.ones((Bsz * T, H + Hkv), dtype=torch.float32, device="cuda")
        flops = 4.0 * Bsz * H * hd * T * (T + 1) / 2 * (3 if args.op == "attn" else 1)

        def once():
            nc.ops.attention_fwd(qkv, Bsz, T, H, Hkv, hd, o, lse)
            if args.op == "attn":
                nc.ops.attention_bwd_rope(qkv, o, lse, do, Bsz, T, H, Hkv, hd, dqkv, ws, rstd, tab, pair_rows=T)
    for _ in range(args.warmup):
        once()
    torch.cuda.synchronize()
    for _ in range(args.iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        once()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    print(json.dumps({"op": args.op, "ms": ms, "tflops": flops / (ms / 1e3) / 1e12, "iters": args.iters,
                      "args": {k: v for k, v in vars(args).items() if k not in ("impl",)}}), flush=True)


def gemm_set(w):
    """The GEMM launches of one training step of workload w: (count, M, N, K,
    a_kmajor, b_kmajor, epilogue, fp32 output) per distinct launch, in the
    step's operand layouts (the forward, the chunked lm_head, then the
    backward of each layer)."""
    N = w.batch * w.seq_len
    C, F, V, L = w.n_embd, w.mlp_hidden, w.vocab, w.depth
    Hd, W = w.n_head * w.head_dim, (w.n_head + 2 * w.n_kv_head) * w.head_dim
    chunk = max(128, ((1 << 30) // (V * 2)) // 128 * 128)
    nchunks = -(-N // chunk)
    nc_rows = min(chunk, N)
    return [  # (tag, count, M, N, K, a_kmajor, b_kmajor, ep)
        ("qkv_rope", L, N, W, C, 1, 1, "qkv"), ("proj", L, N, C, Hd, 1, 1, 2), ("fc", L, N, F, C, 1, 1, 5),
        ("c_proj", L, N, C, F, 1, 1, 2),
        ("lm_logits", nchunks, nc_rows, V, C, 1, 1, 0), ("lm_dx", nchunks, nc_rows, C, V, 1, 0, 1),
        ("lm_dw", nchunks, V, C, nc_rows, 0, 0, 2),
        ("dw_proj", L, C, F, N, 0, 0, 1), ("du", L, N, F, C, 1, 0, 6), ("dw_fc", L, F, C, N, 0, 0, 1),
        ("dx_fc", L, N, C, F, 1, 0, 1), ("dw_o", L, C, Hd, N, 0, 0, 1), ("do", L, N, Hd, C, 1, 0, 0),
        ("dw_qkv", L, W, C, N, 0, 0, 1), ("dx_qkv", L, N, C, W, 1, 0, 1)]


def run_gemmset(args):
    """Launch every distinct GEMM of one --config training step once, at the
    step's full shapes (for a per-kernel DRAM capture of the GEMM kernels;
    a few GB on the device).  Prints the launch table with call counts."""
    import torch
    import decoder_only_transformer_07_b300 as nc
    torch.cuda.set_device(0)
    w = S.workload(args.config)
    g = torch.Generator(device="cuda").manual_seed(0)
    ws = torch.empty(nc.ops.gemm_workspace_bytes(), dtype=torch.uint8, device="cuda")
    rows = []
    for tag, count, M, N, K, ak, bk, ep in gemm_set(w):
        A = (torch.randn((M, K) if ak else (K, M), device="cuda", generator=g) * 0.1).to(torch.bfloat16)
        B = (torch.randn((N, K) if bk else (K, N), device="cuda", generator=g) * 0.1).to(torch.bfloat16)
        if ep == "qkv":
            T, H, Hkv, hd = w.seq_len, w.n_head, w.n_kv_head, w.head_dim
            D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            tab = torch.empty((hd // 4, T, 4), dtype=torch.float32, device="cuda")
            nc.ops.rope_table_pairs(T, hd, 10000.0, tab)
            rstd = torch.empty((M, H + Hkv), dtype=torch.float32, device="cuda")
            fn = (lambda A=A, B=B, D=D, tab=tab, rstd=rstd, T=T, H=H, Hkv=Hkv, hd=hd:
                  nc.ops.gemm_qkv_rope(A, B, D, T, H, Hkv, hd, rstd, tab, 1.1920929e-07, pair_rows=T))
        else:
            D = torch.zeros((M, N), dtype=torch.float32 if ep in (1, 2) else torch.bfloat16, device="cuda")
            aux = torch.rand((M, N), device="cuda", generator=g).to(torch.bfloat16) if ep == 6 else None
            fn = (lambda A=A, B=B, D=D, aux=aux, M=M, N=N, K=K, ak=ak, bk=bk, ep=ep:
                  nc.ops.gemm(A, ak, B, bk, M, N, K, D, ep=ep, aux=aux, workspace=ws))
        fn()
        torch.cuda.synchronize()
        rows.append({"tag": tag, "count": count, "M": M, "N": N, "K": K, "flops": 2.0 * M * N * K})
        del A, B, D
        torch.cuda.empty_cache()
    print(json.dumps({"op": "gemmset", "config": args.config, "launches": rows}), flush=True)


def measure(w, name, args, world, rank, dev, gpu_traffic=True, fp8=False):
    """Time `args.steps` training steps of workload w (device-resident inputs),
    then the same through the host-buffer entry point; returns the fields of
    the bench line for this workload.  fp8: the 8-bit step (the blocks'
    linear products on E4M3 operands)."""
    import ctypes
    import torch
    import decoder_only_transformer_07_b300 as nc

    model = nc.Model(nc.config_from_workload(w, fp8=fp8), seed=S.WEIGHT_SEED)
    tok_np, tgt_np = S.batch_tokens(w)
    tok = torch.from_numpy(tok_np).cuda()
    tgt = torch.from_numpy(tgt_np).cuda()
    grads = torch.empty(model.n_params, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        model.forward_backward(tok, tgt, grads)
    launches_per_step = model.last_launch_count()

    # ---- device-resident timing
    clocks = ClockSampler(dev)
    lib = nc.lib()
    lib.nc_profile_enable(model.handle, 1)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    losses = []
    for _ in range(args.steps):
        loss, _ = model.forward_backward(tok, tgt, grads)
        losses.append(loss)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    prof = {}
    for cls, pname in enumerate(["gemm", "attn_fwd", "attn_bwd", "norm", "rope", "ce", "embed", "cast", "other",
                                 "gemm_fwd", "gemm_dx", "gemm_dw", "gemm_lm_head", "opt_ns", "opt_ew", "quant"]):
        t, n, fl, by = ctypes.c_double(), ctypes.c_int64(), ctypes.c_double(), ctypes.c_double()
        lib.nc_profile_read(model.handle, cls, ctypes.byref(t), ctypes.byref(n), ctypes.byref(fl), ctypes.byref(by))
        prof[pname] = {"ms": t.value, "launches": n.value, "flops": fl.value, "bytes": by.value}
    lib.nc_profile_enable(model.handle, 0)
    ms = max_over_ranks(ms, world, "cuda")

    tokens_per_step = w.batch * w.seq_len
    value = replica_throughput(world, tokens_per_step, args.steps, ms)
    ms_step = ms / args.steps

    # ---- end-to-end through the host-buffer entry point
    tok_h = torch.from_numpy(tok_np).pin_memory()
    tgt_h = torch.from_numpy(tgt_np).pin_memory()
    for _ in range(2):
        model.forward_backward_host(tok_h, tgt_h, grads)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        model.forward_backward_host(tok_h, tgt_h, grads)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, "cuda")
    e2e = {"value": replica_throughput(world, tokens_per_step, args.steps, 1e3 * e2e_s), "unit": UNIT,
           "h2d_bytes_per_step": int(tok_np.nbytes + tgt_np.nbytes), "d2h_bytes_per_step": 8}
    model.close()
    del grads, tok, tgt
    torch.cuda.empty_cache()

    peak_burst, peak_sust, hbm, peak_src = load_peaks()
    fpt = flops_per_token(w)
    per_gpu_tps = value / world
    mfu = {k: per_gpu_tps * fpt[k] / (peak_burst * 1e12) for k in ("causal", "full_square", "six_n_total")}
    mfu["causal_vs_sustained"] = per_gpu_tps * fpt["causal"] / (peak_sust * 1e12)

    g = prof["gemm"]
    gemm_tflops = g["flops"] / (g["ms"] / 1e3) / 1e12 if g["ms"] > 0 else None
    traffic = GEMM_DRAM_BYTES_PER_CALL.get(name) if (gpu_traffic and not fp8) else None
    roofline = {"kernel": "k_gemm_tc2 / k_gemm_tc (tcgen05 bf16 GEMM, all 5 linear layers fwd + dX + dW)",
                "bound": "tensor", "achieved": gemm_tflops, "peak": peak_sust, "unit": "TFLOP/s",
                "frac": (gemm_tflops / peak_sust) if gemm_tflops else None,
                "traffic": traffic,
                "traffic_unit": "DRAM bytes per GEMM call (ncu dram__bytes_read.sum + write.sum of the step's "
                                "GEMM launches, each at full size, weighted by the step's call counts)",
                "algorithmic_bytes_per_call": (g["bytes"] / g["launches"]) if g["launches"] else None,
                "peak_kind": f"bf16 dense, sustained ({peak_src})"}
    total_prof_ms = sum(v["ms"] for k, v in prof.items() if not k.startswith(("gemm_", "opt_")))
    kernels = {k: {"ms_per_step": v["ms"] / args.steps, "share": (v["ms"] / total_prof_ms) if total_prof_ms else None,
                   "launches_per_step": v["launches"] / args.steps,
                   "tflops": (v["flops"] / (v["ms"] / 1e3) / 1e12) if v["ms"] > 0 and v["flops"] else None,
                   "gbs": (v["bytes"] / (v["ms"] / 1e3) / 1e9) if v["ms"] > 0 and v["bytes"] else None}
               for k, v in prof.items() if v["launches"]}
    return {"value": value, "ms_per_step": ms_step, "mfu": mfu, "flops_per_token": fpt["causal"],
            "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches_per_step * args.steps), "clocks": clk,
            "kernels": kernels, "loss": losses[-1],
            "config": arm_config(name, w, world)}


def arm_config(name, w, world):
    """The bench line's config for workload w on `world` GPUs (both arms)."""
    return {"workload": DESCR[name], "global_batch": world * w.batch, "seq_len": w.seq_len,
            "parallelism": "replicas" if world > 1 else "single", "l2": "working set >> L2 (no flush needed)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="d26", choices=sorted(S.WORKLOADS))
    ap.add_argument("--extra-configs", default=None,
                    help="comma-separated workloads measured after --config and reported under 'other_configs' "
                         "(default: the other bf16 workloads when --config is d26 on one GPU; '' for none)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--fp8-step", type=int, default=None,
                    help="1: also time the 8-bit step of --config (default: with the extra configs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-batch", type=int, default=0,
                    help="profiling only: run the step at this batch size instead of the workload's")
    # single-op mode (profiling)
    ap.add_argument("--op", choices=["gemm", "gemm8", "gemmset", "attn", "attn_fwd", "optim", "decode"])
    ap.add_argument("--m", type=int, default=65536)
    ap.add_argument("--n", type=int, default=None, help="default 3840 (--op gemm), 5120 (--op gemm8)")
    ap.add_argument("--k", type=int, default=1280)
    ap.add_argument("--a-major", choices=["k", "mn"], default="k")
    ap.add_argument("--b-major", choices=["k", "mn"], default="k")
    ap.add_argument("--ep", type=int, default=0)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--seq", type=int, default=2048)
    ap.add_argument("--heads", type=int, default=10)
    ap.add_argument("--kv-heads", type=int, default=10)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--iters", type=int, default=5)
    args = ap.parse_args()
    if args.n is None:
        args.n = 5120 if args.op == "gemm8" else 3840
    if args.op == "optim":
        return run_optim(args)
    if args.op == "decode":
        return run_decode(args)
    if args.op == "gemm8":
        return run_gemm8(args)
    if args.op == "gemmset":
        return run_gemmset(args)
    if args.op:
        return run_op(args)
    w = S.workload(args.config, **({"batch": args.step_batch} if args.step_batch else {}))
    if args.impl == "reference":
        return run_reference(args, w)

    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    res = measure(w, args.config, args, world, rank, dev, gpu_traffic=not args.step_batch)
    extras = args.extra_configs
    if extras is None:
        extras = "d20,d24gqa,d12" if (args.config == "d26" and world == 1 and not args.step_batch) else ""
    others = {}
    for name in [e for e in extras.split(",") if e]:
        others[name] = measure(S.workload(name), name, args, world, rank, dev)
    fp8_step = None
    if (args.fp8_step if args.fp8_step is not None else (extras != "")) and w.dtype == "bf16":
        fp8_step = measure(w, args.config, args, world, rank, dev, fp8=True)
        fp8_step["dtype"] = "e4m3 operands in the blocks' linear products (forward, dX, dW), bf16 elsewhere"
        fp8_step["note"] = ("the 8-bit training step (nc_config.fp8 = 1), same workload; MFU is quoted against the "
                            "bf16 peak, and the GEMM roofline mixes the blocks' 8-bit products with the bf16 lm_head")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.config)

    if rank == 0:
        line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
                "data": "synthetic: Zipf(1.1) token ids (seed 2), N(0,0.02) fp32 master weights (seed 1)",
                "config": res["config"], "mfu": res["mfu"], "flops_per_token": res["flops_per_token"],
                "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "kernels": res["kernels"],
                "loss": res["loss"]}
        if others:
            line["other_configs"] = others
        if fp8_step:
            line["fp8_step"] = fp8_step
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
