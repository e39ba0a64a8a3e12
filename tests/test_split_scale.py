"""The group-32 tensor-core path folds each fp16 scale into the A operand as
an exact pair of fp16 values: hi = fp16_rn(s q), lo = fp16_rn(s q - hi), with
hi + lo = s q exactly. This checks that claim for every finite fp16 scale the
path takes unshifted (|s| <= 8188, so |s q| <= 65504) and every q in [-8, 7],
in exact (float64) arithmetic on the host; the kernel's fused fp16
multiply-add computes the same rounded residual."""
import numpy as np


def test_every_scale_splits_exactly():
    s = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    s = s[np.isfinite(s) & (np.abs(s.astype(np.float64)) <= 8188)].astype(np.float64)
    assert s.size == 57344
    for q in range(-8, 8):
        v = s * q                                    # exact
        hi = v.astype(np.float16)                    # round to nearest even
        assert np.all(np.isfinite(hi))
        lo = (v - hi.astype(np.float64)).astype(np.float16)
        assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), v), q


def test_a_larger_scale_would_overflow_without_the_shift():
    # |s| = 8190 with q = -8 rounds past the largest finite fp16 value; the
    # kernel halves such a row's scales (and doubles its result) first
    assert np.isinf(np.float16(np.float64(np.float16(8190.0)) * -8))
    assert np.isfinite(np.float16(np.float64(np.float16(8190.0)) * 0.5 * -8))
