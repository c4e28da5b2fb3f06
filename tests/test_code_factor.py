"""The kernel's code factor 127 / a (a = a row's largest prologue magnitude)
is formed without a division routine: a fast reciprocal r, q = fl(127 r),
then one Newton step q + r (127 - a q) with both products fused (fma).  This
checks, on the host, the error bound that claim rests on: for every a in a
wide sweep and for any reciprocal within 2 ulp of 1/a (the fast reciprocal's
accuracy), the result is within 1 ulp of the correctly rounded 127 / a.

The fp32 steps are emulated in numpy: the product of two fp32 values is
exact in fp64; the residual 127 - a q is then exact in fp64 too, and the
final sum q + r e is formed in fp64 (within 2^-53, far below an fp32 ulp)
before the single rounding to fp32 that an fma makes.
"""
import numpy as np

F32 = np.float32


def _fma32(x, y, z):
    """fl32(x * y + z) for fp32 x, y, z: x*y exact in fp64, the sum in fp64,
    then one rounding to fp32."""
    return (x.astype(np.float64) * y.astype(np.float64) + z.astype(np.float64)).astype(F32)


def _newton_quotient(a, r):
    q = (F32(127.0) * r).astype(F32)
    e = _fma32(-a, q, np.full_like(a, F32(127.0)))
    return _fma32(e, r, q)


def _ulp_distance(x, y):
    xi = x.view(np.int32).astype(np.int64)
    yi = y.view(np.int32).astype(np.int64)
    return np.abs(xi - yi)


def test_code_factor_within_one_ulp():
    rng = np.random.default_rng(0)
    # a spans the magnitudes a row maximum takes (bf16 activations, RMSNorm
    # and SwiGLU values): 2^-20 .. 2^20, random mantissas, plus powers of two
    e = rng.uniform(-20, 20, 200_000)
    a = np.concatenate([(2.0 ** e).astype(F32), (2.0 ** np.arange(-20, 21)).astype(F32)])
    exact = (127.0 / a.astype(np.float64)).astype(F32)   # correctly rounded: 127/a is not a tie in fp32
    r0 = (1.0 / a.astype(np.float64)).astype(F32)
    worst = 0
    for k in range(-2, 3):  # any reciprocal within 2 ulp of 1/a
        r = (r0.view(np.int32) + k).view(F32)
        q = _newton_quotient(a, r)
        worst = max(worst, int(_ulp_distance(q, exact).max()))
    assert worst <= 1, worst


def test_code_factor_exact_where_the_quotient_is_representable():
    # 127 / a is an fp32 value for a = 127 * 2^-k and a = 127 / 2^k: the step
    # must return it exactly
    k = np.arange(-20, 21)
    for a in ((127.0 * 2.0 ** k).astype(F32), (127.0 / 2.0 ** k).astype(F32)):
        exact = (127.0 / a.astype(np.float64)).astype(F32)
        r = (1.0 / a.astype(np.float64)).astype(F32)
        assert np.array_equal(_newton_quotient(a, r), exact)
