"""Helpers shared by the GPU parity tests (no model arithmetic here)."""
import numpy as np


def torch_mod():
    import torch
    return torch


def dev_tensor(a, dtype):
    """numpy array -> CUDA tensor of `dtype` (rounded once if narrower)."""
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dtype)


def to64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_close(got, want, rtol, floor_frac=0.1):
    """Per element |got - want| <= rtol * max(|want|, floor_frac * rms(want)).

    The floor keeps the bound meaningful for elements near zero, where any
    finite-precision evaluation has an absolute (not relative) error.  On the
    tiny fp32 step the largest error of any gradient or logit element
    measures 1.0e-5 * rms(tensor) (fp32 roundoff through ~20 chained
    operations), so the smallest floor every element meets is 0.059 * rms;
    0.1 * rms keeps a 1.7x margin on it while every element larger than
    0.1 * rms is held to the full relative bound.
    """
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    nz = want[want != 0]            # rms over the entries that carry a value (the
    rms = float(np.sqrt(np.mean(nz * nz))) if nz.size else 0.0   # zero rows of dwte are not a scale)
    bound = rtol * np.maximum(np.abs(want), floor_frac * rms)
    err = np.abs(got - want)
    bad = err > bound
    worst = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    return (not bad.any()), worst


def norm_rel(got, want):
    got = np.asarray(got, dtype=np.float64).ravel()
    want = np.asarray(want, dtype=np.float64).ravel()
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))
