"""The error budget of the tensor-core path's number format, on the CPU.

The tensor-core path multiplies bf16 operands: each weight is formed in fp32
as f * (256 d s_j) - (128 d s_j + dmin m_j) with f = 0.5 + q/256 (exact),
one fp32 FMA, and rounded once to bf16; the token rows are rounded to bf16,
and h is rounded to bf16 between the two projections; products are
accumulated in fp32. This module models those roundings in numpy (float64
arithmetic with explicit fp32 and bf16 rounding, torch's round-to-nearest-even)
and checks the reading's two claims: the per-weight error of the dequant is
that of rounding the exact weight to bf16 (the fp32 stage adds next to
nothing), and a layer computed this way stays well inside the 1e-2 * max|ref|
tolerance of that path. It models the format, not the kernels, and no GPU
test uses it as a reference.
"""

import numpy as np
import torch

from quantized_moe_transformer_gb300 import inputs
from tests import kquant_ref as kq


def bf16(x) -> np.ndarray:
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def fields(blocks: np.ndarray):
    """d, dmin, s [.., 8], m [.., 8], q [.., 256] of Q4_K/Q5_K super-blocks."""
    d = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float32)
    dmin = blocks[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float32)
    bits = np.unpackbits(blocks[..., 4:16], axis=-1, bitorder="little").reshape(*blocks.shape[:-1], 16, 6)
    vals = (bits.astype(np.int64) * (1 << np.arange(6))).sum(-1)
    i = np.arange(256)
    nb = blocks.shape[-1]
    qs = blocks[..., 16:144] if nb == 144 else blocks[..., 48:176]
    q = (qs[..., i // 2].astype(np.int64) >> (4 * (i % 2))) & 15
    if nb == 176:
        q = q + 16 * ((blocks[..., 16 + i // 8].astype(np.int64) >> (i % 8)) & 1)
    return d, dmin, vals[..., :8], vals[..., 8:], q


def f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_dequant(blocks: np.ndarray) -> np.ndarray:
    """The tensor-core path's weights: bf16(fp32 FMA of f = 0.5 + q/256 with
    256 d s_j and the fp32 constant -(128 d s_j + dmin m_j))."""
    d, dmin, s, m, q = fields(blocks)
    j = np.arange(256) // 32
    ds = f32(d[..., None].astype(np.float64) * s)           # exact: 11 x 6 bits
    dm = f32(dmin[..., None].astype(np.float64) * m)
    a = 256.0 * ds                                           # exact
    c = -f32(128.0 * ds + dm)                                # fp32 FMA: one rounding
    f = 0.5 + q / 256.0                                      # exact
    return bf16(f32(f * a[..., j] + c[..., j]))              # product exact in fp64; fp32 FMA, then bf16


def test_bf16_dequant_error_is_that_of_plain_rounding():
    rng = inputs.generator(9, "Wg")
    for qt in ("q4k", "q5k"):
        blocks = inputs.packed_blocks(rng, (8192,), qt)
        exact = kq.decode(blocks)
        mask = np.abs(exact) > 1e-3 * np.abs(exact).max()
        rel_tc = np.abs(bf16_dequant(blocks) - exact)[mask] / np.abs(exact)[mask]
        rel_rn = np.abs(bf16(exact) - exact)[mask] / np.abs(exact)[mask]
        assert rel_rn.mean() < 0.0016
        assert rel_tc.mean() / rel_rn.mean() < 1.05, qt
        # the fp32 stage moves a weight across a bf16 rounding boundary rarely
        assert np.mean(bf16_dequant(blocks) != bf16(exact)) < 0.01, qt


def test_layer_in_the_tensor_core_format_is_inside_its_tolerance():
    """A Qwen3.5-35B-A3B-width layer at 16 rows, every expert dense, in the
    path's format: max|err| stays a few times below 1e-2 * max|ref|."""
    from oracle import qmoe_oracle as oracle

    layer = inputs.moe_layer(4, 2048, 16, 512, shared=True)
    k = 2
    X = inputs.hidden(4, 16, 2048)
    ref = oracle.moe_forward(X, layer, k)
    ids, w, _, _ = oracle.route(X, layer["Wr"], k)

    def dense(W):
        v = bf16_dequant(W)
        return v.reshape(*W.shape[:-2], W.shape[-2] * 256)

    xb = bf16(X)

    def ffn(e_g, e_u, e_d, rows):
        g = xb[rows] @ dense(e_g).T
        u = xb[rows] @ dense(e_u).T
        h = bf16(g / (1.0 + np.exp(-g)) * u)
        return h @ dense(e_d).T

    out = ffn(layer["Sg"], layer["Su"], layer["Sd"], np.arange(16))
    for t in range(16):
        for s in range(k):
            e = ids[t, s]
            out[t] += w[t, s] * ffn(layer["Wg"][e], layer["Wu"][e], layer["Wd"][e], np.array([t]))[0]
    ratio = np.max(np.abs(out - ref)) / np.max(np.abs(ref))
    assert ratio < 5e-3, ratio  # 3.0e-3 at these seeds
