"""Comparison helpers shared by the GPU parity tests (no layer arithmetic here)."""
import numpy as np

# Output tolerance for bf16 inputs with fp32 accumulation:
#   max|got - ref| <= REL * max|ref| + ABS
# The absolute floor is nearly vacuous for outputs of ~N(0, 0.02) inputs (their
# max|ref| is ~1e-3), so every check also applies the relative-only form
#   max|got - ref| <= REL * max|ref|
# and unit-scale cases (outputs of order 1) are run as well.
REL = 1e-2
ABS = 1e-3


def f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def assert_close_bf16(got_bits, ref_bits, what="output", rel=REL, atol=ABS):
    g = f32(got_bits).astype(np.float64)
    r = f32(ref_bits).astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    if r.size == 0:
        return 0.0
    err = float(np.max(np.abs(g - r)))
    scale = float(np.max(np.abs(r)))
    assert err <= rel * scale + atol, f"{what}: max|d|={err:.3e} > {rel}*{scale:.3e}+{atol}"
    assert err <= rel * scale, f"{what}: max|d|={err:.3e} > {rel}*max|ref|={rel * scale:.3e}"
    return err / max(scale, 1e-30)
