"""Oracle for the rotary position embedding (RoPE) of Q and K — TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may
import this module.  The library never calls it, and it shares no code with the
CUDA path: a plain fp64 restatement of the rotation.

Page cited: [LC] "超长上下文技术" survey (intelliparadigm.com article 2061774),
§2.1.3 RoPE (rotary position embedding injects the position into query and key
through a rotation).  What the section fixes:
  * the frequencies: inv_freq over the even indices 0, 2, ..., D-2 divided by D,
    i.e. theta_i = 1 / base^(2i/D) for i = 0 .. D/2-1, with base 10000;
  * the angle of position t in pair i is t * theta_i (the outer product of the
    positions with inv_freq; the cache repeats the D/2 angles for both halves);
  * the pairing is "rotate half": x1 = the first D/2 features, x2 = the last D/2,
    and the result is [x1 cos - x2 sin, x1 sin + x2 cos].
Reading taken where the printed code is inconsistent: its cos/sin cache has D
columns (the angles concatenated twice) while x1 and x2 have D/2; since both
halves of the cache hold the same angles, feature i and feature i + D/2 are
rotated together by angle t * theta_i.  The cache's fp32 precision is not kept:
the rotation is evaluated at the exact angle (in fp64 here).

Every function is pinned by tests/oracle_pins.py (unit-vector closed forms with
the frequencies written out, the relative-position property, orthogonality).
"""
from __future__ import annotations

import numpy as np


def rope_frequencies(D: int, base: float = 10000.0) -> np.ndarray:
    """theta_i = 1 / base^(2i / D), i = 0 .. D/2-1 ([LC] §2.1.3, inv_freq)."""
    if D % 2:
        raise ValueError("RoPE needs an even head dim")
    even = np.arange(0, D, 2, dtype=np.float64)
    return 1.0 / base ** (even / D)


def rope_rotate(x, positions, *, base: float = 10000.0, inverse: bool = False):
    """Rotate the feature pairs (i, i + D/2) of every row of x by position * theta_i.

    x: [..., S, D] float64, rows in ORIGINAL order; positions: S numbers (the
    position of each row).  inverse=True applies the transpose (rotation by the
    negated angle): the inverse of the rotation and also its gradient map.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    pos = np.asarray(positions, dtype=np.float64)
    assert pos.shape == (x.shape[-2],)
    angle = pos[:, None] * rope_frequencies(D, base)[None, :]  # [S, D/2]
    if inverse:
        angle = -angle
    c, s = np.cos(angle), np.sin(angle)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)
