"""CPU checks of the arithmetic the GPU kernels rely on (numpy's IEEE fp16, no GPU)."""
import numpy as np


def test_router_hi_lo_split_error_bound():
    """The tensor-core router represents an fp32 router value w as hi = fp16(w) and
    lo = fp16((w - hi) * 2^11): |w - hi - 2^-11 lo| <= 2^-22 |w| for |w| in fp16's normal range
    (w - hi is exact in fp32, Sterbenz), and below 2^-35 absolutely for tiny w, where lo is subnormal
    (spacing 2^-24, scaled by 2^-11)."""
    rng = np.random.default_rng(7)
    w = np.concatenate([rng.normal(0, 0.02, 200000), rng.normal(0, 3.0, 20000),
                        rng.uniform(-1e-5, 1e-5, 20000)]).astype(np.float32)
    hi = w.astype(np.float16)
    lo = ((w.astype(np.float64) - hi.astype(np.float64)) * 2048.0).astype(np.float32).astype(np.float16)
    rec = hi.astype(np.float64) + lo.astype(np.float64) / 2048.0
    err = np.abs(w.astype(np.float64) - rec)
    big = np.abs(w) >= 2.0 ** -11  # here a subnormal lo (error <= 2^-36) is still within the relative bound
    assert np.all(err[big] <= 2.0 ** -22 * np.abs(w[big].astype(np.float64)) * (1 + 1e-12))
    assert np.all(err <= np.maximum(2.0 ** -22 * np.abs(w.astype(np.float64)), 2.0 ** -35))


def test_bf16_activations_are_exact_in_fp16_inside_its_range():
    """bf16 values with |x| in [2^-14, 65504] convert to fp16 without rounding (8 significant bits
    fit in 11); the fp16 operand of the tensor-core paths is then the activation itself."""
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 16, 400000, dtype=np.uint32).astype(np.uint32) << 16
    x = bits.view(np.float32)
    ok = np.isfinite(x) & (np.abs(x) >= 2.0 ** -14) & (np.abs(x) <= 65504.0)
    assert ok.sum() > 10000
    np.testing.assert_array_equal(x[ok].astype(np.float16).astype(np.float32), x[ok])


def test_int4_lop3_conversion_is_exact():
    """The int4 -> fp16 conversion of both tensor-core paths: mask ? (w ^ k) : k (truth table 0x6A)
    with k = 0x64086408 puts 1024 + (q + 8) under the exponent of 1024 for the codes in bits 0-3 and
    16-19; subtracting 1032 gives q exactly.  With k = 0x64806480 the codes in bits 4-7 and 20-23
    become 1024 + 16 (q + 8); times 1/16 minus 72 gives q exactly."""
    def lop3_6a(a, b, c):  # mask b selects a ^ c, else c
        return ((a ^ c) & b) | (c & ~b)
    for q in range(-8, 8):
        nib = q & 0xF
        w = nib | (nib << 4) | (nib << 16) | (nib << 20)
        lo = lop3_6a(w, 0x000F000F, 0x64086408) & 0xFFFFFFFF
        hi = lop3_6a(w, 0x00F000F0, 0x64806480) & 0xFFFFFFFF
        for word, conv in ((lo, lambda v: v - np.float16(1032)), (hi, lambda v: v * np.float16(1 / 16) - np.float16(72))):
            halves = np.array([word & 0xFFFF, word >> 16], dtype=np.uint16).view(np.float16)
            got = conv(halves.astype(np.float16)).astype(np.float16)
            np.testing.assert_array_equal(got.astype(np.float32), np.float32(q))
