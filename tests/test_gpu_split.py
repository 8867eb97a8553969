"""The activation encoding of the expert kernels, on its own (moe_mxfp4_split_terms).

Every activation that reaches the tensor cores (the layer input x, and h = silu(g) * u)
is a sum of E2M1 terms with one E8M0 scale per term and 32-element block.  Each term at
least quarters the block's largest residual (its scale puts that residual at 3..6 times
the scale, where the E2M1 grid's half-spacing is at most one scale unit), so the first t
terms reproduce every value to within 4^-t of the block's largest magnitude, or 2^-119
absolute where the residual becomes that small.  The kernels use t = 8, and t = 4 for
the dense operand of larger blocks.  These tests check that bound on hard inputs
(magnitudes spread over 2^40 inside a block, tie values, saturation edges, tiny and huge
blocks), and check the first term's scale and codes against the conversion rule.
"""
import numpy as np
import pytest
import torch

import mxfp4_moe_expert_gb300 as pkg
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    if not os.path.exists(pkg.LIB_PATH):
        from mxfp4_moe_expert_gb300 import build
        build.build()
    pkg.load_library()


def _blocks(seed=0):
    rng = np.random.default_rng(seed)
    out = [rng.standard_normal((4096, 32)),
           rng.standard_normal((4096, 32)) * np.exp2(rng.integers(-20, 21, (4096, 32))),   # 2^40 spread
           rng.standard_normal((512, 32)) * np.exp2(rng.integers(-60, 61, (512, 1)))]       # tiny .. huge blocks
    edge = np.zeros((16, 32))
    edge[1, 5] = 3.0                                                       # one non-zero value
    edge[2, :] = 1.0                                                       # all equal
    edge[3, :] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4)   # E2M1 midpoints, then 6 = max
    edge[4, :] = np.linspace(-6.0, 6.0, 32)
    edge[5, :] = 6.5 * np.linspace(0.0, 1.0, 32)                           # max / X just over 6: doubled scale
    edge[6, :] = 7.99 * np.linspace(-1.0, 1.0, 32)
    edge[7, :] = 1e-37 * np.linspace(-1.0, 1.0, 32)                        # close to the fp32 floor
    edge[8, :] = 1e37 * np.linspace(-1.0, 1.0, 32)
    edge[9, 0], edge[9, 1:] = 1.0, 2.0 ** -30                              # one large value, the rest far below
    edge[10, :] = -np.abs(rng.standard_normal(32))
    out.append(edge)
    return np.concatenate(out).astype(np.float32)


def _split(x):
    codes, scales = pkg.split_terms(torch.from_numpy(x).to(DEV))
    torch.cuda.synchronize()
    return codes.cpu().numpy().view(np.uint32), scales.cpu().numpy()


def _partial_sums(codes, scales, terms):
    val = np.zeros(codes.shape, np.float64)
    for j in range(terms):
        c = (codes >> (4 * j)) & 0xF
        val += O.E2M1_VALUES[c] * np.ldexp(1.0, scales[:, j].astype(np.int64) - 127)[:, None]
    return val


@pytest.mark.parametrize("terms", [4, 8])
def test_first_terms_are_within_their_bound(terms):
    x = _blocks()
    codes, scales = _split(x)
    err = np.abs(_partial_sums(codes, scales, terms) - x.astype(np.float64))
    bound = np.maximum(np.abs(x).max(axis=1, keepdims=True).astype(np.float64) * 4.0 ** -terms, 2.0 ** -119)
    assert np.all(err <= bound), np.max(err / bound)


def test_first_term_follows_the_conversion_rule():
    """Term 0: scale 2^(floor(log2 amax) - 2), doubled when amax exceeds 6 times it;
    codes = the E2M1 value nearest to x / scale, ties to the even code."""
    x = _blocks(1)
    codes, scales = _split(x)
    amax = np.abs(x).max(axis=1).astype(np.float64)
    nz = amax >= 2.0 ** -119
    e = np.floor(np.log2(np.where(nz, amax, 1.0)))
    X = np.exp2(e - 2)
    X = np.where(amax > 6 * X, 2 * X, X)
    assert np.array_equal(scales[nz, 0].astype(np.int64), (np.log2(X[nz]) + 127).astype(np.int64))
    v = x[nz].astype(np.float64) / X[nz, None]
    mag = O._round_e2m1_magnitude(np.abs(v))                     # the oracle's pinned rounding
    got = codes[nz] & 0xF
    assert np.array_equal(got & 7, mag)
    sign = (got >> 3) & 1
    nzm = mag > 0   # (a code of magnitude 0 may carry either sign)
    assert np.array_equal(sign[nzm], (v[nzm] < 0).astype(sign.dtype))
