"""CPU checks of the arithmetic shortcuts the encode kernel takes, each against the definition it
replaces (no GPU). The kernel never forms the quotients x / s16 or y / ||v||:

  * q8_0 keys (PolyKV abstract: int8 q8_0 keys): with a normal fp16 scale s16 the code is the low
    mantissa byte of RN(x * yb + 2^23 + 256), yb one ulp above RU(1 / s16);
  * 3-bit values (normalized FWHT, Lloyd-Max codes for N(0,1)): the code is
    3.5 + copysign(m + 0.5, y) with m = #{i in 4..6 : |y| >= RN(b_i * ||v||)}, using the symmetry
    of the codebook, and eight codes are packed by an fp32 Horner sum of half-codes.

Each test restates the shortcut in numpy (float64 arithmetic rounded to float32 where the kernel
rounds) and compares it with the definition the oracle implements."""
import numpy as np

from oracle import codebook

MAGIC_Q8 = np.float64(8388864.0)      # 2^23 + 256
HALF_CODE_BIAS = np.float64(8388607.5)  # 3.5 * (8^8 - 1) / 7


def _all_finite(dtype):
    if dtype == "fp16":
        x = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    else:
        x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    return x[np.isfinite(x)]


def _ru_recip(s):
    """Smallest float32 >= 1 / s (s a positive fp16 value), by exact float64 products."""
    y = np.float32(1.0 / float(s))
    if float(y) * float(s) < 1.0:
        y = np.nextafter(y, np.float32(np.inf))
    p = np.nextafter(y, np.float32(0))
    while float(p) * float(s) >= 1.0:
        y, p = p, np.nextafter(p, np.float32(0))
    return y


def _round_half_away(x, s):
    """The definition: the correctly rounded fp32 quotient, rounded half away from zero."""
    r = (x / np.float32(s)).astype(np.float32).astype(np.float64)
    return np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -127, 127)


def test_q8_fused_multiply_add_code_equals_round_half_away():
    rng = np.random.default_rng(7)
    normal = np.arange(0x0400, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    scales = np.concatenate([normal[:150], normal[-60:], rng.choice(normal, 190, replace=False)])
    checked = 0
    for dtype in ("fp16", "bf16"):
        xs = _all_finite(dtype)
        for s in scales:
            # a block whose scale rounds to s has amax < (s + ulp(s) / 2) * 127 (65504 covers < 65520)
            ulp = 32.0 if s == np.float32(65504.0) else float(np.spacing(np.float16(s)))
            x = xs[np.abs(xs) < (float(s) + ulp / 2) * 127]
            yb = np.nextafter(_ru_recip(s), np.float32(np.inf))
            f = (x.astype(np.float64) * np.float64(yb) + MAGIC_Q8).astype(np.float32)
            low = (f.view(np.uint32) & 0xFF).astype(np.int64)
            low = np.where(low > 127, low - 256, low)
            ref = _round_half_away(x, s)
            assert np.array_equal(f.astype(np.float64) - MAGIC_Q8, ref), (dtype, float(s))
            assert np.array_equal(low, ref), (dtype, float(s))
            checked += x.size
    assert checked > 2e7


def test_codebook_boundaries_symmetric():
    """The value decision folds the sign out: b_{6-i} = -b_i exactly and b_3 = 0 in fp32."""
    _, b32 = codebook.codebook_f32()
    assert b32.dtype == np.float32 and b32.size == 7
    assert b32[3] == 0.0
    for i in range(3):
        assert b32[6 - i].view(np.uint32) == (-b32[i]).view(np.uint32)


def test_value_half_code_decision_matches_definition_off_boundaries():
    _, b32 = codebook.codebook_f32()
    rng = np.random.default_rng(11)
    n = (np.abs(rng.standard_normal(200_000)) * 11.3 + 1e-3).astype(np.float32)
    # half of the coordinates are pushed to within a few ulps of a scaled boundary
    y = (rng.standard_normal(n.size) * n / np.sqrt(128.0)).astype(np.float32)
    near = rng.random(n.size) < 0.5
    bsel = b32[rng.integers(0, 7, n.size)]
    y_near = (bsel.astype(np.float64) * n).astype(np.float32)
    k = rng.integers(-3, 4, n.size).astype(np.float64)
    y_near = (y_near.astype(np.float64) + k * np.spacing(np.abs(y_near)).astype(np.float64)).astype(np.float32)
    y = np.where(near, y_near, y)
    # kernel: thresholds RN(b_i * n), magnitude compares, half-code with the sign of y
    t = (b32[4:].astype(np.float64)[None, :] * n.astype(np.float64)[:, None]).astype(np.float32)
    m = (np.abs(y)[:, None] >= t).sum(axis=1)
    got = 3.5 + np.copysign(m + 0.5, y)
    # definition: u = fp32(y / n), code = #{i : u >= b_i}
    u = (y / n).astype(np.float32)
    ref = (u[:, None] >= b32[None, :]).sum(axis=1)
    diff = got != ref
    if diff.any():
        ud = u[diff].astype(np.float64)
        dist = np.min(np.abs(ud[:, None] - b32.astype(np.float64)[None, :]) /
                      np.maximum(np.abs(b32.astype(np.float64)), 1.0)[None, :], axis=1)
        assert np.all(dist <= 1e-6), "a decision differs away from a boundary"
    # on the unperturbed half, differences are as rare as the parity contract allows
    assert diff[~near].sum() <= max(1, 1e-5 * (~near).sum())


def test_half_code_horner_packing_is_exact():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 8, (400_000, 8))
    codes[:8] = np.array([[0] * 8, [7] * 8, [0, 7] * 4, [7, 0] * 4, [3] * 8, [4] * 8,
                          [0, 0, 0, 0, 0, 0, 0, 7], [7, 0, 0, 0, 0, 0, 0, 0]])
    h = codes.astype(np.float64) - 3.5
    w = h[:, 7].astype(np.float32)
    for i in range(6, -1, -1):
        w = (w.astype(np.float64) * 8.0 + h[:, i]).astype(np.float32)   # one fma per step
    packed = (w.astype(np.float64) + HALF_CODE_BIAS).astype(np.float32)
    want = (codes * (8 ** np.arange(8))[None, :]).sum(axis=1)
    assert np.array_equal(packed.astype(np.int64), want)
