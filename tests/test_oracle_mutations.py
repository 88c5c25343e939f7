"""Planted mistakes: each plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand) must make at least one pin fail.

The mistakes are planted in a private copy of the oracle's source, on the CPU;
the oracle itself is never modified."""
import importlib.util
import os
import sys
import types

import pytest

from oracle_pins import ALL_PINS

ORACLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")
SOURCES = ("attention.py", "rope.py")  # executed in this order into one mutant module

MUTATIONS = {
    "dropped_scale": ("s = scale * (qrows @ kkeys.T)", "s = (qrows @ kkeys.T)"),
    "alibi_sign": ("s = s - slope * dist", "s = s + slope * dist"),
    "diagonal_masked": ("keys[None, :] <= rows[:, None]", "keys[None, :] < rows[:, None]"),
    "zigzag_pairing": ("shards[r].extend(chunks[2 * N - 1 - r])", "shards[r].extend(chunks[N + r])"),
    "zigzag_order": ("shards[r].extend(chunks[r])\n            shards[r].extend(chunks[2 * N - 1 - r])",
                     "shards[r].extend(chunks[2 * N - 1 - r])\n            shards[r].extend(chunks[r])"),
    "q_k_swapped": ("s = _scores(q[b, h, r], kk, r, keys, scale, slope, causal)\n                lse = _row_lse(s)",
                    "s = _scores(k[b, h, r], q[b, h][keys], r, keys, scale, slope, causal)\n                lse = _row_lse(s)"),
    "lse_no_log": ("lse = safe + np.log(tot)", "lse = safe + tot"),
    "ds_missing_D": ("ds = p * (dp - Dvec[r][:, None])", "ds = p * dp"),
    "dk_unscaled": ("dk[b, h] += scale * (ds.T @ q[b, h, r])\n    return dq, dk, dv",
                    "dk[b, h] += (ds.T @ q[b, h, r])\n    return dq, dk, dv"),
    "dv_wrong_operand": ("dv[b, h] += p.T @ dout[b, h, r]\n                dq[b, h, r]",
                         "dv[b, h] += p.T @ v[b, h, r]\n                dq[b, h, r]"),
    "merge_max": ("lse = np.logaddexp(lse_a, lse_b)", "lse = np.maximum(lse_a, lse_b)"),
    "online_alpha_inverted": ("alpha = np.where(np.isfinite(m), np.exp(m - ref), 0.0)",
                              "alpha = np.where(np.isfinite(m), np.exp(ref - m), 0.0)"),
    "ring_direction_skips": ("steps = [(r - t) % N for t in range(N)]", "steps = [(r - t) % N for t in range(1, N)]"),
    "pairs_off_by_one": ("int(sum(g + 1 for g in shard))", "int(sum(g for g in shard))"),
    "strided_blocks": ("shards[g % N].append(g)", "shards[g // (S // N)].append(g)"),
    # RoPE (rope.py)
    "rope_interleaved_pairs": ("rope.py", "x1, x2 = x[..., :half], x[..., half:]",
                               "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    "rope_exponent_halved": ("rope.py", "even = np.arange(0, D, 2, dtype=np.float64)",
                             "even = np.arange(0, D // 2, dtype=np.float64)"),
    "rope_rotation_sign": ("rope.py", "[x1 * c - x2 * s, x1 * s + x2 * c]", "[x1 * c + x2 * s, -x1 * s + x2 * c]"),
    "rope_inverse_ignored": ("rope.py", "angle = -angle", "angle = angle"),
    "rope_dropped_cos": ("rope.py", "x1 * s + x2 * c]", "x1 * s + x2]"),
}


def _load_mutant(name, target, old, new):
    mod = types.ModuleType(f"oracle_mutant_{name}")
    for src in SOURCES:
        with open(os.path.join(ORACLE, src)) as f:
            text = f.read()
        if src == target:
            assert text.count(old) == 1, f"mutation {name}: anchor not found exactly once"
            text = text.replace(old, new)
        exec(compile(text, f"<mutant {name}: {src}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    spec = MUTATIONS[name]
    target, old, new = spec if len(spec) == 3 else ("attention.py",) + spec
    mod = _load_mutant(name, target, old, new)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # an assertion or a crash both count as caught
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"
