"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no arithmetic of the model: it only names the workload
shapes and draws token ids.  Both the CUDA path and the CPU oracle consume
what it produces.

Token streams stand in for the BPE-tokenised web text the nanochat pages
train on (devpress "用不到100美元，亲手训练一个属于你的GPT-2" §2.2 item 2;
woshipm nanochat analysis §四).  A Zipf(1.1) law over the vocabulary gives the
skewed id frequencies of real BPE text; the tiny parity case uses uniform ids.
"""
from dataclasses import dataclass, asdict

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    depth: int
    n_embd: int
    n_head: int
    n_kv_head: int
    head_dim: int
    mlp_hidden: int
    vocab: int
    seq_len: int
    batch: int
    dtype: str          # "fp32" or "bf16": the compute dtype of the CUDA path
    tokens: str         # "uniform" or "zipf"

    def as_dict(self):
        return asdict(self)

    @property
    def n_tokens(self):
        return self.batch * self.seq_len


WORKLOADS = {
    "tiny": Workload("tiny", 2, 128, 2, 2, 64, 512, 512, 64, 2, "fp32", "uniform"),
    "d12": Workload("d12", 12, 768, 6, 6, 128, 3072, 65536, 2048, 32, "bf16", "zipf"),
    "d20": Workload("d20", 20, 1280, 10, 10, 128, 5120, 65536, 2048, 32, "bf16", "zipf"),
    "d26": Workload("d26", 26, 1664, 13, 13, 128, 6656, 65536, 2048, 16, "bf16", "zipf"),
    "d24gqa": Workload("d24gqa", 24, 1536, 12, 4, 128, 6144, 65536, 4096, 8, "bf16", "zipf"),
}

WEIGHT_SEED = 1
TOKEN_SEED = 2
ZIPF_S = 1.1


def workload(name, **overrides):
    """Return a named workload, optionally with some fields replaced."""
    w = WORKLOADS[name]
    if overrides:
        d = w.as_dict()
        d.update(overrides)
        w = Workload(**d)
    return w


def zipf_cdf(vocab, s=ZIPF_S):
    """CDF of P(id = k-1) proportional to k^-s for k = 1..vocab."""
    k = np.arange(1, vocab + 1, dtype=np.float64)
    p = k ** (-s)
    c = np.cumsum(p)
    return c / c[-1]


def token_stream(vocab, batch, seq_len, kind="zipf", seed=TOKEN_SEED):
    """Draw a [batch, seq_len + 1] int32 stream of token ids.

    ``kind="uniform"``: ids uniform in [0, vocab).
    ``kind="zipf"``: inverse-CDF sampling of a Zipf(1.1) law truncated to the
    vocabulary, so id 0 is the most frequent.
    """
    rng = np.random.default_rng(seed)
    shape = (batch, seq_len + 1)
    if kind == "uniform":
        s = rng.integers(0, vocab, size=shape, dtype=np.int64)
    elif kind == "zipf":
        u = rng.random(size=shape)
        s = np.searchsorted(zipf_cdf(vocab), u, side="right")
        s = np.minimum(s, vocab - 1)
    else:
        raise ValueError(f"unknown token distribution {kind!r}")
    return s.astype(np.int32)


def batch_tokens(w, seed=TOKEN_SEED, batch=None, seq_len=None):
    """tokens, targets (each [B, T] int32) for a workload: the stream shifted by one."""
    B = w.batch if batch is None else batch
    T = w.seq_len if seq_len is None else seq_len
    s = token_stream(w.vocab, B, T, w.tokens, seed)
    return np.ascontiguousarray(s[:, :T]), np.ascontiguousarray(s[:, 1:])


FP8_SEED = 3


def fp8_codes(rows, cols, seed=FP8_SEED):
    """Random E4M3 byte codes for the 8-bit GEMM's operands: exponent fields
    4..11 (magnitudes 2^-3 .. 30, the range a per-tensor scale maps a
    normal-like activation's bulk into), any mantissa, random sign.  No NaN
    code (0x7f / 0xff) can occur."""
    rng = np.random.default_rng(seed)
    mag = rng.integers(0x20, 0x60, size=(rows, cols), dtype=np.uint8)
    sign = rng.integers(0, 2, size=(rows, cols), dtype=np.uint8) << 7
    return mag | sign


def fp8_codes_all(rows, cols, seed=FP8_SEED):
    """Random E4M3 byte codes drawn uniformly from every finite code: the
    subnormals (exponent field 0), the zeros, and the largest magnitude 448
    (0x7e / 0xfe) included; only the two NaN codes 0x7f / 0xff are left out."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 254, size=(rows, cols), dtype=np.int64)
    c = c + (c >= 0x7f)                   # skip 0x7f: 0..0x7e, 0x80..0xfe
    return c.astype(np.uint8)
