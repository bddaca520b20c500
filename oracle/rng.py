"""Counter-based weight initialisation, written from published definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages do not say how weights are initialised; the workloads fix i.i.d.
N(0, 0.02) fp32 weights drawn from a seed.  The draw is specified so that two
independent implementations produce the same numbers:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state advances by the golden gamma
  0x9E3779B97F4A7C15 and each output is the state passed through the
  variant-13 mixing function.  Tensor ``j`` of the packed layout uses the
  stream whose initial state is ``seed XOR ((j + 1) * gamma)``; element ``e``
  of that tensor takes output number ``e`` (counting from 0), i.e.
  ``mix(state0 + (e + 1) * gamma)``.
* Box-Muller (Box & Muller, 1958), one normal per 64-bit output: the top 24
  bits give u1, bits 16..39 give u2, each as ``(k + 0.5) / 2**24``;
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)`` in fp64, times ``std``, rounded once
  to float32.  ``std`` is the float32 value a model configuration carries
  (0.02 becomes float32(0.02) = 0.0199999995529651...), widened exactly.
"""
import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK24 = np.uint64(0xFFFFFF)


def _mix(z):
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_outputs(state0, count, start=0):
    """Outputs number ``start .. start+count-1`` of SplitMix64 from ``state0``."""
    with np.errstate(over="ignore"):
        e = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(np.uint64(state0) + e * GAMMA)


def stream_state(seed, tensor_index):
    with np.errstate(over="ignore"):
        return np.uint64(seed) ^ (np.uint64(tensor_index + 1) * GAMMA)


def box_muller(u64):
    """One standard normal (fp64) per 64-bit word."""
    u1 = ((u64 >> np.uint64(40)).astype(np.float64) + 0.5) / 16777216.0
    u2 = (((u64 >> np.uint64(16)) & _MASK24).astype(np.float64) + 0.5) / 16777216.0
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def normal_init(seed, tensor_index, count, std, chunk=1 << 24):
    """float32 N(0, std) values for one tensor of the packed layout."""
    out = np.empty(count, dtype=np.float32)
    std = float(np.float32(std))
    s0 = stream_state(seed, tensor_index)
    for a in range(0, count, chunk):
        n = min(chunk, count - a)
        out[a:a + n] = (box_muller(splitmix64_outputs(s0, n, a)) * std).astype(np.float32)
    return out


def init_params(cfg, seed):
    """All parameters, packed in layout order, as one float32 vector."""
    from .model import param_layout
    layout = param_layout(cfg)
    total = sum(r * c for _, r, c, _ in layout)
    flat = np.empty(total, dtype=np.float32)
    for j, (_, r, c, off) in enumerate(layout):
        flat[off:off + r * c] = normal_init(seed, j, r * c, cfg.init_std)
    return flat
