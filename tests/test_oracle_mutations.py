"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of an oracle function (on the CPU,
through monkeypatching) and checks that at least one pin in
``test_oracle_pins.py`` then fails.
"""
import numpy as np
import pytest

from oracle import model as M
import tests.test_oracle_pins as P


def _rope_wrong_sign(x, cos, sin):
    d = x.shape[-1] // 2
    x1, x2 = x[..., :d], x[..., d:]
    return np.concatenate([x1 * cos - x2 * sin, x1 * sin + x2 * cos], axis=-1)


def _rope_tables_wrong_freq(T, hd, base):
    d = hd // 2
    omega = base ** (-(np.arange(d, dtype=np.float64)) / hd)
    theta = np.arange(T, dtype=np.float64)[:, None] * omega[None, :]
    return np.cos(theta), np.sin(theta)


def _norm_bwd_dropped_term(dy, y, rstd):
    return rstd * dy


def _attention_no_scale(q, k, v):
    T, hd = q.shape
    s = q @ k.T
    s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    z = e.sum(axis=1, keepdims=True)
    return (e / z) @ v, (s.max(axis=1, keepdims=True) + np.log(z))[:, 0]


def _attention_bwd_transposed(q, k, v, do):
    dq, dk, dv = M.__dict__["_orig_attention_bwd"](q, k, v, do)
    return dq, dv, dk


def _kv_head_interleaved(cfg, h):
    return h % cfg.n_kv_head


def _ce_wrong_sign(z, tgt):
    loss, dz = M.__dict__["_orig_cross_entropy"](z, tgt)
    return loss, -dz


MUTANTS = {
    "rope sign": ("rope", _rope_wrong_sign),
    "rope frequency": ("rope_tables", _rope_tables_wrong_freq),
    "norm bwd term": ("rms_norm_bwd", _norm_bwd_dropped_term),
    "attention scale": ("attention", _attention_no_scale),
    "attention bwd operands": ("attention_bwd", _attention_bwd_transposed),
    "gqa mapping": ("_kv_head_of", _kv_head_interleaved),
    "ce grad sign": ("cross_entropy", _ce_wrong_sign),
}

PINS = [
    P.test_rope_golden_unit_pair,
    P.test_rope_identity_at_zero_norm_and_relative_position,
    P.test_rms_norm_bwd_matches_fd,
    P.test_attention_T1_returns_v_and_constant_keys_give_running_mean,
    P.test_attention_bwd_matches_fd,
    P.test_cross_entropy_zero_logits_and_row_sums,
    P.test_gqa_equals_mha_with_repeated_kv_heads,
    lambda: P.test_whole_step_central_finite_differences(dict(n_kv_head=1)),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setitem(M.__dict__, "_orig_" + attr, getattr(M, attr))
    monkeypatch.setattr(M, attr, fn)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake '{name}'"
