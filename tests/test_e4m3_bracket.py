"""The rule behind the write kernels' E4M3 encode, checked on the host.

The kernels take two products x * lo and x * hi, where lo and hi are
RN(1/scale) scaled by (1 - 2^-20) and (1 + 2^-20), and use their common
E4M3 code when the two agree (IEEE division otherwise).  The claim is that
agreement implies the code of the IEEE binary32 quotient RN(x / scale):
the products bracket the quotient and E4M3 rounding is monotonic.  This
test restates the rule in numpy binary32 arithmetic and checks the claim
for every finite bf16 value and a spread of scales, with the oracle's
E4M3 encoder deciding every code.  (The kernels themselves are compared
with the oracle on every bf16 value by the GPU write tests.)
"""
import numpy as np
import pytest

import oracle

SCALES = [1.0, 0.5, 3.0, 7.0, 0.3, 1.1, 0.999, 0.0123, 4.7 / 448, 1e30, 3e-38]


@pytest.fixture(scope="module")
def enc():
    o = oracle.load()
    return np.vectorize(o.e4m3_from_float, otypes=[np.uint8])


def test_bracket_agreement_implies_the_quotient_code(enc):
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    disagree = 0
    with np.errstate(all="ignore"):
        for s in SCALES:
            s = np.float32(s)
            r = np.float32(1) / s
            assert np.isfinite(r) and r >= np.finfo(np.float32).tiny and r < 1e38
            lo = np.float32(r * np.float32(1 - 2.0 ** -20))
            hi = np.float32(r * np.float32(1 + 2.0 ** -20))
            c_lo = enc((x * lo).astype(np.float32))
            c_hi = enc((x * hi).astype(np.float32))
            agree = c_lo == c_hi
            q = (x[agree] / s).astype(np.float32)
            assert np.array_equal(enc(q), c_lo[agree]), float(s)
            disagree += int((~agree).sum())
    # the division fallback is rare: at most a few per thousand values
    assert disagree < 0.005 * x.size * len(SCALES)
