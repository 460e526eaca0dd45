"""The number format of the tensor-core router, checked on the CPU in fp64.

From 256 rows the router multiplies X and Wr on the bf16 tensor cores. Every
fp32 value is split into three bf16 parts, each the round-to-nearest-even bf16
of what the earlier parts leave, and six of the nine part products are
accumulated: x1 w1 + x1 w2 + x2 w1 + x1 w3 + x3 w1 + x2 w2. These tests pin
the two facts that make that fp32-accurate: the split is exact to 2^-24, and
the six products reproduce x . w to about 2^-22 of sum |x||w|."""

import numpy as np
import torch


def split3(v: np.ndarray):
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    p1 = t.to(torch.bfloat16).to(torch.float32)
    r1 = t - p1
    p2 = r1.to(torch.bfloat16).to(torch.float32)
    r2 = r1 - p2
    p3 = r2.to(torch.bfloat16).to(torch.float32)
    return p1.numpy(), p2.numpy(), p3.numpy(), r1.numpy(), r2.numpy()


def test_split_is_exact_to_2_minus_24():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(100_000), rng.normal(0, 0.02, 100_000),
                        rng.uniform(-1e4, 1e4, 1_000), [0.0, 1.0, -3.0, 2.0 ** -100]]).astype(np.float32)
    p1, p2, p3, r1, r2 = split3(v)
    v64 = v.astype(np.float64)
    # the remainders are exact fp32 subtractions
    assert np.array_equal(r1.astype(np.float64), v64 - p1)
    assert np.array_equal(r2.astype(np.float64), r1.astype(np.float64) - p2)
    # each part is at most 2^-8 of what it splits
    assert np.all(np.abs(r1) <= 2.0 ** -8 * np.abs(v))
    assert np.all(np.abs(r2) <= 2.0 ** -8 * np.abs(r1))
    err = np.abs(v64 - p1 - p2 - p3)
    assert np.all(err <= 2.0 ** -24 * np.abs(v64))


def test_six_part_products_match_the_fp64_dot_product():
    rng = np.random.default_rng(6)
    H = 2048
    x = rng.standard_normal((64, H)).astype(np.float32)
    w = rng.normal(0.0, 0.02, (H, 32)).astype(np.float32)
    x1, x2, x3, _, _ = split3(x)
    w1, w2, w3, _, _ = split3(w)

    def mm(a, b):  # bf16 x bf16 products are exact in fp64
        return a.astype(np.float64) @ b.astype(np.float64)

    six = mm(x1, w1) + mm(x1, w2) + mm(x2, w1) + mm(x1, w3) + mm(x3, w1) + mm(x2, w2)
    exact = mm(x, w)
    scale = np.abs(x).astype(np.float64) @ np.abs(w).astype(np.float64)
    rel = np.max(np.abs(six - exact) / scale)
    assert rel < 2.0 ** -21, rel
    # the leading product alone is only good to about 2^-8: the other five matter
    assert np.max(np.abs(mm(x1, w1) - exact) / scale) > 2.0 ** -12
