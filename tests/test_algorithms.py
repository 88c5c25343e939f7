"""Two numerical methods of the kernels, restated here on the CPU and held to the
mathematics (not to the kernels' outputs):

1. The forward's online softmax moves its reference maximum only when a tile's
   maximum exceeds it by more than 8 (log2 units) and otherwise takes the
   probabilities against the stale reference (so they are at most 2^8), with O
   and l sharing that reference.  The result equals softmax attention by its
   definition ([LC] "超长上下文技术" §3.1.2 gives the blockwise recurrence; the
   threshold is this library's choice): checked against the fp64 oracle on
   adversarial score patterns, in fp64 and in fp32.

2. RoPE angles ([LC] §2.1.3, theta_i = 1/base^(2i/D)): the angle of position t is
   taken as a fraction of a turn, t * F_i mod 2^64 with F_i = theta_i / (2 pi) as
   a 64-bit binary fraction, its top 32 bits read as a signed fraction of a
   half-turn.  Against the exact angle (mpmath, 40 digits) that is within 4e-7
   rad at positions sampled up to 2^31, whereas the plain fp32 product
   t * theta_i is off by up to 7.8e-3 rad (about 2^-7) at t = 2^18."""
import math

import numpy as np
import pytest

import oracle

LOG2E = 1.0 / math.log(2.0)


def online_softmax_threshold(q, k, v, *, causal, scale, tile=128, dtype=np.float64, threshold=8.0):
    """The kernel's recurrence for one head: q [S, D], k/v [S, D] (original order,
    positions = indices).  Returns O [S, D], LSE [S] (natural log) and the largest
    probability formed against the reference."""
    S, D = q.shape
    q, k, v = (np.asarray(a, dtype=dtype) for a in (q, k, v))
    c2 = dtype(scale * LOG2E)
    O = np.zeros((S, D), dtype=dtype)
    l = np.zeros(S, dtype=dtype)
    m_ref = np.full(S, -np.inf, dtype=dtype)
    pmax = 0.0
    for j0 in range(0, S, tile):
        keys = np.arange(j0, min(S, j0 + tile))
        x = (q @ k[keys].T) * c2  # log2 domain
        if causal:
            x = np.where(keys[None, :] <= np.arange(S)[:, None], x, -np.inf)
        mt = x.max(axis=1)
        move = mt > m_ref + dtype(threshold)
        with np.errstate(over="ignore", invalid="ignore"):  # the unused branch may overflow
            alpha = np.where(move, np.where(np.isfinite(m_ref), np.exp2(m_ref - mt), 0.0), 1.0).astype(dtype)
        O *= alpha[:, None]
        l *= alpha
        m_ref = np.where(move, mt, m_ref)
        mu = np.where(np.isfinite(m_ref), m_ref, 0.0).astype(dtype)
        p = np.exp2(x - mu[:, None]).astype(dtype)
        pmax = max(pmax, float(p.max()))
        l += p.sum(axis=1, dtype=dtype)
        O += p @ v[keys]
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, (m_ref + np.log2(l)) / LOG2E, -np.inf)
    O = np.where(l[:, None] > 0, O / np.where(l > 0, l, 1.0)[:, None], 0.0)
    return O, lse, pmax


def _score_patterns(rng, S, D):
    """q, k pairs whose scores stress the recurrence."""
    q = rng.standard_normal((S, D))
    k = rng.standard_normal((S, D))
    yield "random", q, k
    # scores that grow tile after tile: the maximum creeps up, rescales are rare
    ramp = np.repeat(np.arange(S // 128), 128)[:S] * 5.0
    yield "creeping max", np.ones((S, D)) / math.sqrt(D), np.outer(ramp, np.ones(D)) / math.sqrt(D) * math.sqrt(D)
    # a late spike far above everything before it (alpha underflows to 0)
    k2 = k.copy()
    k2[S - 5] *= 60.0
    yield "late spike", q, k2
    # very wide range of scores
    yield "wide range", q * 12.0, k * 12.0
    # all scores equal
    yield "equal", np.ones((S, D)), np.ones((S, D))


@pytest.mark.parametrize("causal", [True, False])
def test_threshold_recurrence_is_exact_fp64(causal):
    rng = np.random.default_rng(3)
    S, D = 640, 16
    v = rng.standard_normal((S, D))
    scale = 1.0 / math.sqrt(D)
    for name, q, k in _score_patterns(rng, S, D):
        O, lse, pmax = online_softmax_threshold(q, k, v, causal=causal, scale=scale)
        O_ref, lse_ref = oracle.attention_forward(q[None, None], k[None, None], v[None, None], causal=causal,
                                                  scale=scale)
        assert pmax <= 2.0 ** 8 * (1 + 1e-12), name
        assert np.allclose(lse, lse_ref[0, 0], rtol=1e-12, atol=1e-12), name
        assert np.allclose(O, O_ref[0, 0], rtol=1e-10, atol=1e-12), name


def test_threshold_recurrence_fp32():
    """In fp32 the stale reference costs nothing measurable: against the fp64
    oracle its error is that of the textbook recurrence (threshold 0) at the same
    precision, and nothing overflows."""
    rng = np.random.default_rng(4)
    S, D = 1024, 32
    v = rng.standard_normal((S, D))
    scale = 1.0 / math.sqrt(D)
    for name, q, k in _score_patterns(rng, S, D):
        O_ref, lse_ref = oracle.attention_forward(q[None, None], k[None, None], v[None, None], causal=True,
                                                  scale=scale)
        errs = {}
        for th in (0.0, 8.0):
            O, lse, pmax = online_softmax_threshold(q, k, v, causal=True, scale=scale, dtype=np.float32,
                                                    threshold=th)
            assert np.all(np.isfinite(O)) and pmax <= 2.0 ** th * (1 + 1e-6), name
            errs[th] = (np.max(np.abs(O - O_ref[0, 0])), np.max(np.abs(lse - lse_ref[0, 0])))
        assert errs[8.0][0] <= 2.0 * errs[0.0][0] + 1e-6, (name, errs)
        assert errs[8.0][1] <= 2.0 * errs[0.0][1] + 1e-6, (name, errs)


def test_threshold_changes_nothing_but_the_reference():
    """Threshold 0 (always move the maximum: the textbook recurrence) and 8 give
    the same result to rounding."""
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((512, 8)) * 4 for _ in range(3))
    a = online_softmax_threshold(q, k, v, causal=True, scale=0.5, threshold=0.0)
    b = online_softmax_threshold(q, k, v, causal=True, scale=0.5, threshold=8.0)
    assert a[2] <= 1.0 + 1e-12 and b[2] > 1.0   # only the lazy form forms probabilities above 1
    assert np.allclose(a[0], b[0], rtol=1e-11, atol=1e-12) and np.allclose(a[1], b[1], rtol=1e-12)


# ---------------------------------------------------------------------------- RoPE angles
def _turns(D, base):
    """F_i: theta_i / (2 pi) as a 64-bit binary fraction, rounded to nearest."""
    return [int(round(math.ldexp((1.0 / base ** (2 * i / D)) * (1.0 / (2 * math.pi)), 64))) for i in range(D // 2)]


def _fixed_point_angle(t, F):
    """Angle (radians) of position t: bits 32..63 of t * F mod 2^64, read as a
    signed 32-bit fraction of a half-turn, through an fp32 conversion."""
    turn = ((t * F) >> 32) & 0xFFFFFFFF
    signed = turn - (1 << 32) if turn >= (1 << 31) else turn
    half_turns = float(np.float32(signed)) * 2.0 ** -31
    return half_turns * math.pi


@pytest.mark.parametrize("base", [10000.0, 500000.0])
def test_rope_fixed_point_angles(base):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    D = 128
    F = _turns(D, base)
    positions = [0, 1, 2, 7, 1000, 2 ** 18 - 1, 2 ** 18, 123457, 2 ** 24 + 3, 2 ** 31 - 1]
    worst = 0.0
    for i in range(0, D // 2, 3):
        theta = mpmath.mpf(1) / mpmath.power(mpmath.mpf(base), mpmath.mpf(2 * i) / D)
        for t in positions:
            exact = mpmath.fmod(t * theta, 2 * mpmath.pi)
            got = _fixed_point_angle(t, F[i])
            d = float(mpmath.fmod(mpmath.mpf(got) - exact + 3 * mpmath.pi, 2 * mpmath.pi) - mpmath.pi)
            worst = max(worst, abs(d))
    assert worst < 4e-7, worst


def test_rope_plain_fp32_angle_is_not_enough():
    """Why the angle is reduced in fixed point: the fp32 product t * theta_i at
    t = 2^18 is already off by far more than the bf16 tolerance allows."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    t = 2 ** 18
    errs = []
    for i in range(64):
        theta = 1.0 / 10000.0 ** (2 * i / 128)
        naive = float(np.float32(t) * np.float32(theta))
        exact = mpmath.mpf(t) / mpmath.power(10000, mpmath.mpf(2 * i) / 128)
        errs.append(abs(float(mpmath.mpf(naive) - exact)))
    assert max(errs) > 2.0 ** -8


# ---------------------------------------------------------------------------- ALiBi exponents
def _f32(x):
    return np.float32(x)


def _fma32(a, b, c):
    """fp32 fused multiply-add: the product of two fp32 numbers is exact in fp64,
    one rounding of the sum to fp32 (the second rounding through fp64 cannot
    matter at these magnitudes for this check)."""
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def test_alibi_exponent_precision_far_from_the_diagonal():
    """The forward's probability exponent on an ALiBi tile far below the diagonal:
    with the row's reference folded into the tile's bias base first, the exponent
    is formed from small numbers and keeps fp32 precision; adding the ~1e5 bias to
    the score first (and the reference after) loses it."""
    rng = np.random.default_rng(6)
    slope2 = 0.5 * LOG2E           # log2-domain slope of the steepest head
    c2 = _f32(LOG2E / math.sqrt(128))
    dist0 = 2 ** 18 - 256          # distance of the tile's first key from the query
    base = _f32(-slope2 * dist0)   # bias of column 0 (keys before the query)
    sl = _f32(slope2)              # the bias grows towards the diagonal
    raw = rng.standard_normal(128).astype(np.float32) * 8
    exact = np.array([np.float64(r) * np.float64(c2) + np.float64(base) + np.float64(sl) * u
                      for u, r in enumerate(raw)])
    mu = _f32(exact.max())         # the row's reference (any value near the max will do)
    folded, late = [], []
    for u, r in enumerate(raw):
        ch, uu = divmod(u, 32)
        bm = np.float32(np.float64(base) - np.float64(mu))
        lb = _fma32(sl, _f32(32 * ch), bm)
        folded.append(_fma32(r, c2, _fma32(sl, _f32(uu), lb)))
        lb0 = _fma32(sl, _f32(32 * ch), base)
        late.append(np.float32(np.float64(_fma32(r, c2, _fma32(sl, _f32(uu), lb0))) - np.float64(mu)))
    ref = exact - np.float64(mu)
    err_folded = np.max(np.abs(np.array(folded, dtype=np.float64) - ref))
    err_late = np.max(np.abs(np.array(late, dtype=np.float64) - ref))
    assert err_folded < 1e-4, err_folded            # relative error of 2^x below 1e-4
    assert err_late > 10 * err_folded, (err_late, err_folded)


def _bf16_round(x):
    """Round a float64 to the nearest bf16 value (ties to even), returned as float64."""
    import torch
    return float(torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).to(torch.float64))


def _column_term_parts(slope2, step, c2, u):
    """The causal-ALiBi column term of key u in raw-score units, taken relative to
    the tile's middle column, slope2*step*(u-64)/c2, as four successive bf16
    roundings (what the K-side block of the extra K step holds); their exact sum
    is what the tensor core adds to the score."""
    rest = float(slope2) * float(step) * (u - 64) / float(c2)
    parts = []
    for _ in range(4):
        p = _bf16_round(rest)
        parts.append(p)
        rest -= p
    return parts


def _mma_bias_exponents(raw, slope2, step, c2, dk, lim=127):
    """The forward's log2 exponents on a causal ALiBi tile whose column term rides on
    the Q K^T product: S'_u = raw_u + (sum of the four parts), one fp32 rounding;
    the row term slope2 * dk (dk = position of column 64 minus the query's) split
    exactly into bhi + blo; the reference mu = fl(max S' * c2 + bhi) over the
    visible columns u <= lim; x_u = fl(S'_u c2 - fl(fl(mu - bhi) - blo))."""
    s1 = np.array([np.float32(np.float64(r) + sum(_column_term_parts(slope2, step, c2, u)))
                   for u, r in enumerate(raw)], dtype=np.float32)
    dkf = _f32(dk)
    bhi = np.float32(np.float64(slope2) * np.float64(dkf))
    blo = np.float32(np.float64(slope2) * np.float64(dkf) - np.float64(bhi))  # exact remainder (fma)
    mu = np.float32(np.float64(np.float32(np.float64(s1[:lim + 1].max()) * np.float64(c2))) + np.float64(bhi))
    mub = np.float32(np.float64(np.float32(np.float64(mu) - np.float64(bhi))) - np.float64(blo))
    x = np.array([np.float32(np.float64(s) * np.float64(c2) - np.float64(mub)) for s in s1])
    exact = np.array([np.float64(r) * np.float64(c2) + np.float64(slope2) * (np.float64(dkf) + step * (u - 64))
                      for u, r in enumerate(raw)]) - np.float64(mu)
    return x.astype(np.float64), exact, mu, (bhi, blo)


@pytest.mark.parametrize("step", [1, 16])
def test_alibi_column_term_on_the_tensor_core(step):
    """Causal ALiBi with the column term added by the tensor core: for the
    steepest head of the page's slope formula (2^(-8/H) with H = 32) on a diagonal
    tile, whose visible keys matter most, the exponents of every key that carries
    weight (probability above 2^-64 of the row's reference) are within 1e-4 of
    exact (a relative error below 7e-5 in the probability, against 2^-9 for the
    bf16 rounding of P), with the token-strided step (16) as well."""
    rng = np.random.default_rng(11)
    slope2 = _f32(2.0 ** (-8.0 / 32) * LOG2E)
    c2 = _f32(LOG2E / math.sqrt(128))
    for trial in range(8):
        raw = (rng.standard_normal(128) * 11.3).astype(np.float32)
        for lim in (0, 40, 64, 100, 127):         # the query's column in the diagonal tile
            x, exact, _, _ = _mma_bias_exponents(raw, slope2, step, c2, dk=(64 - lim) * step, lim=lim)
            keep = exact[:lim + 1] > -64
            err = np.max(np.abs(x[:lim + 1] - exact[:lim + 1])[keep])
            assert err < 1e-4, (lim, err)


def test_alibi_row_term_split_far_from_the_diagonal():
    """A ring-step partial whose keys all lie far before the query (2^18 tokens):
    the row term slope2 * (gk0 - g_i) is ~3e5 in log2 units.  Taken as an exact
    two-float sum (fma remainder) it leaves the exponents within 1e-4 of exact;
    with the remainder dropped they are off by up to half an ulp of 3e5 (~1e-2)."""
    rng = np.random.default_rng(12)
    slope2 = _f32(2.0 ** (-8.0 / 32) * LOG2E)
    c2 = _f32(LOG2E / math.sqrt(128))
    errs, errs_nolo = [], []
    for trial in range(40):
        raw = (rng.standard_normal(128) * 11.3).astype(np.float32)
        dk = -(2 ** 18 - 256) - int(rng.integers(0, 4096))
        x, exact, mu, (bhi, blo) = _mma_bias_exponents(raw, slope2, 1, c2, dk=dk)
        keep = exact > -64
        errs.append(np.max(np.abs(x - exact)[keep]))
        # the same without the remainder of the row term
        mub = np.float32(np.float64(mu) - np.float64(bhi))
        s1 = x + np.float64(np.float32(np.float64(mu) - np.float64(bhi)) - np.float64(blo))  # S' * c2
        x_nolo = np.array([np.float32(np.float64(s) - np.float64(mub)) for s in s1])
        errs_nolo.append(np.max(np.abs(x_nolo - exact)[keep]))
    assert max(errs) < 1e-4, max(errs)
    assert max(errs_nolo) > 10 * max(errs), (max(errs_nolo), max(errs))
