"""Pins of the fp64 oracle against things other than itself.

Hand-constructed super-blocks, a second dequantiser, brute force over all
experts, closed forms, the pages' printed sizes and the rank-split invariants of
"CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights" ("What PR #382 Now
Splits"). A plausible slip in the oracle (a swapped field, a wrong nibble order,
a dropped term, a sign, an index) fails at least one of these.
"""

import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from quantized_moe_transformer_gb300 import inputs
from tests import kquant_ref as kq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ dequant

def test_q4k_hand_block(oracle):
    s = [1, 2, 3, 4, 5, 6, 7, 63]
    m = [0, 1, 2, 3, 4, 5, 6, 63]
    q = [i % 16 for i in range(256)]
    blk = kq.encode_q4k(0.5, 0.25, s, m, q)
    w = oracle.dequant_q4k(blk)
    for idx, val in _golden("q4k_hand_block.txt"):
        assert w[int(idx)] == float(val), idx


def test_q4k_all_zero(oracle):
    assert np.all(oracle.dequant_q4k(np.zeros(144, np.uint8)) == 0.0)
    assert np.all(oracle.dequant_q5k(np.zeros(176, np.uint8)) == 0.0)


def test_q4k_identity_scales(oracle):
    q = [(7 * i + 3) % 16 for i in range(256)]
    blk = kq.encode_q4k(1.0, 0.0, [1] * 8, [0] * 8, q)
    assert np.array_equal(oracle.dequant_q4k(blk), np.array(q, dtype=np.float64))


@pytest.mark.parametrize("d", [65504.0, 2.0**-14, 2.0**-10])
def test_q4k_field_maxima(oracle, d):
    q = [15] * 256
    blk = kq.encode_q4k(d, d, [63] * 8, [63] * 8, q)
    exp = kq.expected_weights(d, d, [63] * 8, [63] * 8, q)
    assert np.array_equal(oracle.dequant_q4k(blk), exp)
    q5 = [31] * 256
    blk5 = kq.encode_q5k(d, d / 2, [63] * 8, [0] * 8, q5)
    assert np.array_equal(oracle.dequant_q5k(blk5), kq.expected_weights(d, d / 2, [63] * 8, [0] * 8, q5))


def test_six_bit_field_walk(oracle):
    """Every bit of every 6-bit field, alone: with d = dmin = 1 and q = 1, the
    block decodes to s_j - m_j, which names the field and bit that was set."""
    q = [1] * 256
    for f in range(16):
        for b in range(6):
            s = [0] * 8
            m = [0] * 8
            (s if f < 8 else m)[f % 8] = 1 << b
            blk = kq.encode_q4k(1.0, 1.0, s, m, q)
            w = oracle.dequant_q4k(blk).reshape(8, 32)
            exp = np.zeros((8, 32))
            exp[f % 8, :] = (1 << b) * (1 if f < 8 else -1)
            assert np.array_equal(w, exp), (f, b)


def test_nibble_and_high_bit_walk(oracle):
    """Every nibble bit of every weight (Q4_K and Q5_K) and every Q5_K high bit."""
    for i in range(256):
        for b in range(4):
            q = [0] * 256
            q[i] = 1 << b
            w = oracle.dequant_q4k(kq.encode_q4k(1.0, 0.0, [1] * 8, [0] * 8, q))
            assert np.array_equal(w, np.array(q, np.float64)), (i, b)
        q = [0] * 256
        q[i] = 16 + (i % 16)
        w5 = oracle.dequant_q5k(kq.encode_q5k(1.0, 0.0, [1] * 8, [0] * 8, q))
        assert np.array_equal(w5, np.array(q, np.float64)), i


def test_dequant_matches_second_decoder(oracle):
    rng = inputs.generator(5, "Wg")
    for qt, fn in (("q4k", oracle.dequant_q4k), ("q5k", oracle.dequant_q5k)):
        blocks = inputs.packed_blocks(rng, (64, 3), qt)
        assert np.array_equal(fn(blocks), kq.decode(blocks))


# Q6_K (the format a Q4_K_M file keeps some tensors in; no GPU kernel takes it
# yet): the oracle's reading of the library's layout, pinned the same way.

def test_q6k_hand_block(oracle):
    s = [j - 8 for j in range(16)]
    q = [i % 64 for i in range(256)]
    w = oracle.dequant_q6k(kq.encode_q6k(0.5, s, q))
    for idx, val in _golden("q6k_hand_block.txt"):
        assert w[int(idx)] == float(val), idx
    assert np.array_equal(w, kq.expected_weights_q6k(0.5, s, q))


def test_q6k_zero_and_midpoint(oracle):
    assert np.all(oracle.dequant_q6k(np.zeros(210, np.uint8)) == 0.0)
    # q = 32 is the zero of every sub-block, whatever d and the scales
    blk = kq.encode_q6k(3.0, [127, -128] * 8, [32] * 256)
    assert np.all(oracle.dequant_q6k(blk) == 0.0)


@pytest.mark.parametrize("d", [65504.0, 2.0**-14, -1.5])
def test_q6k_scale_extremes(oracle, d):
    s = [127, -128, 1, -1] * 4
    q = [0, 63, 31, 33] * 64
    blk = kq.encode_q6k(d, s, q)
    assert np.array_equal(oracle.dequant_q6k(blk), kq.expected_weights_q6k(d, s, q))


def test_q6k_quant_bit_and_scale_walk(oracle):
    """Every one of the 6 quant bits of every weight alone (the others at the
    zero point 32), and every sub-block scale alone."""
    for i in range(256):
        for b in range(6):
            q = [32] * 256
            q[i] = 1 << b
            w = oracle.dequant_q6k(kq.encode_q6k(1.0, [1] * 16, q))
            exp = np.zeros(256)
            exp[i] = (1 << b) - 32
            assert np.array_equal(w, exp), (i, b)
    for j in range(16):
        s = [0] * 16
        s[j] = -3
        w = oracle.dequant_q6k(kq.encode_q6k(1.0, s, [33] * 256)).reshape(16, 16)
        exp = np.zeros((16, 16))
        exp[j, :] = -3.0
        assert np.array_equal(w, exp), j


def test_q6k_matches_second_decoder(oracle):
    rng = np.random.default_rng(66)
    blocks = rng.integers(0, 256, (64, 3, 210), dtype=np.uint8)
    blocks[..., 1] &= 0x3B  # keep d a finite fp16
    assert np.array_equal(oracle.dequant_q6k(blocks), kq.decode_q6k(blocks))
    dense = oracle.dequant_matrix(blocks)
    assert dense.shape == (64, 3 * 256)
    assert np.array_equal(dense, kq.decode_q6k(blocks).reshape(64, 768))


# MXFP4 (the MXFP4-class format the pages name for the target model class; no
# GPU kernel takes it yet)

def test_mxfp4_code_table(oracle):
    """All 16 E2M1 codes at scale 1 (e = 127): the format's value table."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    codes = [i % 16 for i in range(256)]
    w = oracle.dequant_mxfp4(kq.encode_mxfp4([127] * 8, codes))
    assert np.array_equal(w, np.array([table[c] for c in codes]))
    assert all(kq.e2m1_value(c) == table[c] for c in range(16))


def test_mxfp4_scale_walk(oracle):
    """Every E8M0 exponent 0..254 is 2^(e - 127) exactly; 255 is NaN."""
    for e in list(range(0, 255, 7)) + [254, 127, 0]:
        w = oracle.dequant_mxfp4(kq.encode_mxfp4([e] + [127] * 7, [2] * 256))  # code 2 = 1.0
        assert np.all(w[:32] == 2.0 ** (e - 127)) and np.all(w[32:] == 1.0), e
    w = oracle.dequant_mxfp4(kq.encode_mxfp4([127, 255] + [127] * 6, [2] * 256))
    assert np.all(np.isnan(w[32:64])) and np.all(w[:32] == 1.0) and np.all(w[64:] == 1.0)


def test_mxfp4_matches_second_decoder(oracle):
    rng = np.random.default_rng(77)
    blocks = rng.integers(0, 256, (16, 2, 136), dtype=np.uint8)
    blocks[..., 0:8] = rng.integers(100, 150, (16, 2, 8), dtype=np.uint8)
    assert np.array_equal(oracle.dequant_mxfp4(blocks), kq.decode_mxfp4(blocks))
    assert oracle.dequant_matrix(blocks).shape == (16, 512)


def test_generator_ranges(oracle):
    blocks = inputs.packed_blocks(inputs.generator(0, "Wg"), (4096,), "q4k")
    d = blocks[:, 0:2].copy().view(np.float16).astype(np.float64)
    assert d.min() >= 2.0**-12 and d.max() <= 2.0**-10
    w = oracle.dequant_q4k(blocks)
    assert np.isfinite(w).all()
    # the formats without a kernel yet: finite, and weights of the same size
    ref = np.abs(w).max()
    for qt, fn in (("q6k", oracle.dequant_q6k), ("mxfp4", oracle.dequant_mxfp4)):
        wq = fn(inputs.packed_blocks(inputs.generator(0, "Wg"), (4096,), qt))
        assert np.isfinite(wq).all()
        assert ref / 4 < np.abs(wq).max() < 4 * ref, qt


# ------------------------------------------------------------------ router

def _brute_route(X, Wr, k):
    L = X.astype(np.float64) @ Wr.astype(np.float64)
    P = scipy.special.softmax(L, axis=1)
    ids = np.stack([sorted(range(L.shape[1]), key=lambda e: (-L[t, e], e))[:k]
                    for t in range(L.shape[0])])
    sel = np.take_along_axis(P, ids, axis=1)
    return ids, sel / sel.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("k", [1, 2, 8])
def test_router_brute_force(oracle, k):
    X = inputs.hidden(0, 16, 256)
    Wr = inputs.generator(0, "Wr").normal(0, 0.02, size=(256, 32)).astype(np.float32)
    ids, w, gap, _ = oracle.route(X, Wr, k)
    bids, bw = _brute_route(X, Wr, k)
    assert np.array_equal(ids, bids)
    np.testing.assert_allclose(w, bw, rtol=1e-12, atol=0)
    if k == 1:
        assert np.all(w == 1.0)
    L = X.astype(np.float64) @ Wr.astype(np.float64)
    srt = -np.sort(-L, axis=1)
    np.testing.assert_allclose(gap, srt[:, k - 1] - srt[:, k], rtol=0, atol=1e-15)


def test_router_k_equals_e_is_softmax(oracle):
    X = inputs.hidden(1, 4, 256)
    Wr = inputs.generator(1, "Wr").normal(0, 0.02, size=(256, 8)).astype(np.float32)
    ids, w, gap, L = oracle.route(X, Wr, 8)
    P = scipy.special.softmax(L, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(P, ids, axis=1), rtol=1e-12)
    assert np.all(np.isinf(gap))


def test_router_ties_take_lower_index(oracle):
    X = inputs.hidden(2, 6, 256)
    Wr = inputs.generator(2, "Wr").normal(0, 0.02, size=(256, 8)).astype(np.float32)
    Wr[:, 5] = Wr[:, 1]          # experts 1 and 5 always tie
    Wr[:, 6] = Wr[:, 2]
    ids, w, gap, L = oracle.route(X, Wr, 4)
    for t in range(6):
        row = list(ids[t])
        for a, b in ((1, 5), (2, 6)):
            if b in row:
                assert a in row and row.index(a) < row.index(b)
    # equal logits give equal weights
    for t in range(6):
        row = list(ids[t])
        if 1 in row and 5 in row:
            assert w[t, row.index(1)] == w[t, row.index(5)]


# ------------------------------------------------------------------ MoE layer

def _brute_moe(X, layer, k, R=None, f_half=None):
    """All E experts for every row, then a mask: a different loop structure and
    a different dequantiser from the oracle's."""
    x = X.astype(np.float64)
    E, F = layer["E"], layer["F"]
    cols = slice(None) if f_half is None else slice(f_half * F // 2, (f_half + 1) * F // 2)
    def ffn(Wg, Wu, Wd):
        g = np.einsum("th,fh->tf", x, kq.dense(Wg)[cols])
        u = np.einsum("th,fh->tf", x, kq.dense(Wu)[cols])
        h = g / (1 + np.exp(-g)) * u
        return np.einsum("tf,hf->th", h, kq.dense(Wd)[:, cols])
    Y = np.stack([ffn(layer["Wg"][e], layer["Wu"][e], layer["Wd"][e]) for e in range(E)], axis=1)
    ids, w = _brute_route(X, layer["Wr"], k)
    gate = np.zeros((x.shape[0], E))
    np.put_along_axis(gate, ids, w, axis=1)
    out = np.einsum("te,teh->th", gate, Y)
    if "Sg" in layer:
        out = out + ffn(layer["Sg"], layer["Su"], layer["Sd"])
    if R is not None and f_half is None:
        out = out + R
    return out


@pytest.mark.parametrize("shared,down,routing", [(True, "q6k", "uniform"), (False, "mxfp4", "uniform"),
                                                  (False, "q4k", "uniform"), (True, "q5k", "uniform"),
                                                 (True, "q5k", "zipf")])
def test_moe_brute_force(oracle, shared, down, routing):
    layer = inputs.moe_layer(3, 256, 8, 256, shared=shared, down_type=down, routing=routing)
    X = inputs.hidden(3, 5, 256, routing)
    R = inputs.residual(3, 5, 256)
    got = oracle.moe_forward(X, layer, 2, R)
    exp = _brute_moe(X, layer, 2, R)
    assert np.max(np.abs(got - exp)) <= 1e-12 * np.max(np.abs(exp))


def test_moe_zero_scales_give_residual(oracle):
    layer = inputs.moe_layer(4, 256, 4, 256, shared=True)
    for name in ("Wg", "Wu", "Wd", "Sg", "Su", "Sd"):
        layer[name][..., 0:4] = 0                   # d = dmin = 0
    X = inputs.hidden(4, 3, 256)
    R = inputs.residual(4, 3, 256)
    assert np.array_equal(oracle.moe_forward(X, layer, 2, R), R.astype(np.float64))


def test_moe_closed_form_swiglu(oracle):
    """Constant weights a, b, c (gate, up, down) and a one-hot row give
    y = F * silu(a) * b * c in every output, whichever experts are chosen."""
    H, E, F = 256, 2, 256
    a, b, c = 1.0, 0.5, 0.25
    layer = inputs.moe_layer(0, H, E, F, shared=False, down_type="q4k")
    for name, val in (("Wg", a), ("Wu", b), ("Wd", c)):
        blk = kq.encode_q4k(val, 0.0, [1] * 8, [0] * 8, [1] * 256)
        layer[name][...] = blk
    X = np.zeros((1, H), np.float32)
    X[0, 7] = 1.0
    out = oracle.moe_forward(X, layer, 1)
    silu_a = 1.0 / (1.0 + math.exp(-1.0))            # silu(1) = 1 * sigmoid(1)
    assert np.allclose(out, F * silu_a * b * c, rtol=1e-15, atol=0)


def test_moe_f_split_invariant(oracle):
    """Rank 0 + rank 1 partials of the 256/256 intermediate split equal the
    unsplit layer (routed and shared experts split the same way)."""
    layer = inputs.moe_layer(6, 256, 8, 512, shared=True)
    X = inputs.hidden(6, 7, 256)
    full = oracle.moe_forward(X, layer, 2)
    p0 = oracle.moe_forward(X, layer, 2, f_half=0)
    p1 = oracle.moe_forward(X, layer, 2, f_half=1)
    assert np.max(np.abs(p0 + p1 - full)) <= 1e-12 * np.max(np.abs(full))
    assert np.max(np.abs(p0 - _brute_moe(X, layer, 2, f_half=0))) <= 1e-12 * np.max(np.abs(p0))
    assert not np.allclose(p0, p1)


# ------------------------------------------------------------------ page pins

def test_page_shape_pins():
    pins = {r[0]: int(r[1]) for r in _golden("page_shape_pins.txt")}
    T, H = 4096, 2048
    assert T * H * np.dtype(np.float32).itemsize == pins["hidden_collective_bytes_at_4096_rows"]
    k = pins["selected_per_token"]
    route_record = np.dtype(np.int32).itemsize + np.dtype(np.float32).itemsize
    assert T * k * route_record == pins["router_sync_bytes_at_4096_rows"]
    assert pins["f_split_rank0"] + pins["f_split_rank1"] == 512
    assert pins["routed_experts"] == 256
    assert pins["query_heads"] // pins["query_heads_per_rank"] == 2
    assert pins["kv_heads"] // pins["kv_heads_per_rank"] == 2
    assert 8192 * 2 == pins["hidden_partial_bytes_per_token_8192_bf16"]
    # super-block sizes: 4.5 and 5.5 bits per weight
    assert inputs.Q4K_BYTES * 8 / 256 == 4.5 and inputs.Q5K_BYTES * 8 / 256 == 5.5
    # one expert's gate+up (Q4_K) and down (Q5_K) bytes at H=2048, F=512
    assert 2 * 512 * (H // 256) * 144 + H * (512 // 256) * 176 == 1900544


# ------------------------------------------------------------------ block pieces

def test_round_bf16_matches_torch(oracle):
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), ref)
    ties = np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8)])
    assert np.array_equal(oracle.round_bf16(ties), np.array([1.0, 1 + 2**-6, -1.0]))


def test_rmsnorm_closed_forms(oracle):
    g = np.ones(64)
    x = np.full((1, 64), 3.0)
    assert np.allclose(oracle.rmsnorm(x, g, 0.0), 1.0, rtol=1e-15)
    assert np.allclose(oracle.rmsnorm(x, g, 1e-6), 3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-15)
    y = inputs.hidden(0, 2, 64).astype(np.float64)
    gam = np.arange(1, 65, dtype=np.float64)
    r = oracle.rmsnorm(y, gam, 0.0)
    assert np.allclose(np.sqrt(np.mean((r / gam) ** 2, axis=1)), 1.0, rtol=1e-14)


def test_rope_pairs_and_relative_position(oracle):
    d, theta = 4, 100.0
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    got = oracle.rope(x, np.array([1]), theta)[0, 0]
    a0, a1 = 1.0, theta ** (-2.0 / 4)                # angles of pairs (0,2), (1,3)
    exp = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
           3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    assert np.allclose(got, exp, rtol=0, atol=1e-15)
    assert np.array_equal(oracle.rope(x, np.array([0]), theta), x)
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    dots = [float(np.sum(oracle.rope(q, np.array([m]), 1e7) * oracle.rope(k, np.array([m - 5]), 1e7)))
            for m in (5, 50, 4095)]
    assert np.allclose(dots, dots[0], rtol=1e-10)


def test_attention_closed_forms(oracle):
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 2, 8))
    K = rng.standard_normal((1, 1, 8))
    V = rng.standard_normal((1, 1, 8))
    out = oracle.attention(q, K, V, np.array([0]), np.array([0, 0]))
    assert np.allclose(out[0, 0], V[0, 0]) and np.allclose(out[0, 1], V[0, 0])
    # equal keys: the mean of the visible values
    K = np.repeat(rng.standard_normal((1, 1, 8)), 10, axis=0)
    V = rng.standard_normal((10, 1, 8))
    out = oracle.attention(q.repeat(3, axis=0)[:3, :1], K, V, np.array([0, 4, 9]), np.array([0]))
    for t, p in enumerate([0, 4, 9]):
        assert np.allclose(out[t, 0], V[:p + 1, 0].mean(axis=0), rtol=1e-13)


def test_attention_context_split_merge(oracle):
    """Merging per-shard (max, normaliser, output) statistics reproduces
    unsplit softmax attention ("Two-Dimensional Attention at Long Context")."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((3, 16))
    K = rng.standard_normal((40, 16)) * 3
    V = rng.standard_normal((40, 16))
    full = oracle.attention(q[:, None, :], K[:, None, :], V[:, None, :],
                            np.array([39, 39, 39]), np.array([0]))[:, 0]
    parts = [oracle.attention_shard_stats(q, K[a:b], V[a:b]) for a, b in ((0, 7), (7, 30), (30, 40))]
    assert np.allclose(oracle.attention_merge(parts), full, rtol=1e-13, atol=1e-14)
    # brute force of the definition
    S = q @ K.T / 4.0
    P = np.exp(S) / np.exp(S).sum(axis=1, keepdims=True)
    assert np.allclose(full, P @ V, rtol=1e-13)


def _small_block(seed=0, T=6, ctx=32):
    blk = inputs.block(seed, H=256, n_heads=8, n_kv=2, head_dim=64, ctx=ctx, F=512, E=8)
    X = inputs.hidden(seed, T, 256)
    return blk, X


def test_block_split_invariant(oracle):
    """Two rank partials (half the query heads, one KV head each, with the
    matching O-projection columns; F split 256/256) sum to the unsplit block."""
    blk, X = _small_block()
    kc = oracle.bf16_bits_to_f64(blk["k_cache"])
    vc = oracle.bf16_bits_to_f64(blk["v_cache"])
    out, parts = oracle.block_forward(X, blk, 2, 10, kc.copy(), vc.copy())
    out_s, parts_s = oracle.block_forward(X, blk, 2, 10, kc.copy(), vc.copy(), split=True)
    assert np.max(np.abs(out_s - out)) <= 1e-12 * np.max(np.abs(out))
    a = parts["attn"][0]
    assert np.max(np.abs(parts_s["attn"][0] + parts_s["attn"][1] - a)) <= 1e-12 * np.max(np.abs(a))
    m = parts["moe"][0]
    assert np.max(np.abs(parts_s["moe"][0] + parts_s["moe"][1] - m)) <= 1e-12 * np.max(np.abs(m))


def test_block_decode_step_matches_prefill_row(oracle):
    """Decoding the last row after prefilling the others gives the prefill's
    last row (causality of the cache path)."""
    blk, X = _small_block(1, T=5, ctx=16)
    kc = oracle.bf16_bits_to_f64(blk["k_cache"])
    vc = oracle.bf16_bits_to_f64(blk["v_cache"])
    full, _ = oracle.block_forward(X, blk, 2, 0, kc.copy(), vc.copy())
    kc2, vc2 = kc.copy(), vc.copy()
    oracle.block_forward(X[:4], blk, 2, 0, kc2, vc2)
    last, _ = oracle.block_forward(X[4:], blk, 2, 4, kc2, vc2)
    assert np.allclose(last[0], full[4], rtol=1e-12, atol=1e-12 * np.abs(full).max())


def test_block_rows_restriction(oracle):
    """Evaluating only some query rows gives those rows of the full block."""
    blk, X = _small_block(2, T=7, ctx=16)
    kc = oracle.bf16_bits_to_f64(blk["k_cache"])
    vc = oracle.bf16_bits_to_f64(blk["v_cache"])
    full, _ = oracle.block_forward(X, blk, 2, 3, kc.copy(), vc.copy())
    rows = np.array([0, 4, 6])
    part, _ = oracle.block_forward_rows(X, blk, 2, 3, kc.copy(), vc.copy(), rows)
    assert np.max(np.abs(part - full[rows])) <= 1e-12 * np.max(np.abs(full))


# ------------------------------------------------------------------ block composition
# The block is h1 = X + attn(X), out = h1 + moe(RMSNorm(h1; g2)) ("CKE Zip: From
# Splitting Tokens To Splitting Qwen3.5 Weights", "What PR #382 Now Splits": attention
# partials, then the residual, then the router and MoE on the new state, then the
# residual). Each case below reduces the block to parts pinned above, so that a
# composition slip fails one of them: the second norm reading X instead of h1, using
# g1 instead of g2, or either residual dropped.

def _zero_scales(packed):
    packed[..., 0:4] = 0            # d = dmin = 0: every weight of the matrix is 0


def _composition_cases(oracle, blk, X, pos0, rows=None):
    kc = oracle.bf16_bits_to_f64(blk["k_cache"])
    vc = oracle.bf16_bits_to_f64(blk["v_cache"])
    if rows is None:
        out, _ = oracle.block_forward(X, blk, 2, pos0, kc.copy(), vc.copy())
        return out, kc, vc
    out, _ = oracle.block_forward_rows(X, blk, 2, pos0, kc.copy(), vc.copy(), rows)
    return out, kc, vc


@pytest.mark.parametrize("rows", [None, np.array([1, 4, 5])])
def test_block_zero_attention_is_residual_plus_moe(oracle, rows):
    """Attention weights all zero: the attention branch is 0, so the block is
    X + moe(RMSNorm(X; g2)) (with g1 != g2, a norm with g1 fails this)."""
    blk, X = _small_block(4, T=6, ctx=32)
    for name in ("Wq", "Wk", "Wv", "Wo"):
        _zero_scales(blk[name])
    assert not np.allclose(blk["g1"], blk["g2"])
    out, _, _ = _composition_cases(oracle, blk, X, 10, rows)
    sel = np.arange(6) if rows is None else rows
    exp = X[sel].astype(np.float64) + oracle.moe_forward(
        oracle.rmsnorm(X[sel], blk["g2"]), blk["moe"], 2)
    assert np.max(np.abs(out - exp)) <= 1e-12 * np.max(np.abs(exp))
    wrong = X[sel].astype(np.float64) + oracle.moe_forward(
        oracle.rmsnorm(X[sel], blk["g1"]), blk["moe"], 2)
    assert np.max(np.abs(out - wrong)) > 1e-6 * np.max(np.abs(exp))


@pytest.mark.parametrize("rows", [None, np.array([0, 5])])
def test_block_zero_moe_is_residual_plus_attention(oracle, rows):
    """Every routed and shared expert weight zero: the MoE branch is 0, so the
    block is X + attn(X)."""
    blk, X = _small_block(5, T=6, ctx=32)
    for name in ("Wg", "Wu", "Wd", "Sg", "Su", "Sd"):
        _zero_scales(blk["moe"][name])
    out, kc, vc = _composition_cases(oracle, blk, X, 10, rows)
    a = oracle.attn_sublayer(X, blk, 10, kc.copy(), vc.copy(), rows=rows)
    sel = np.arange(6) if rows is None else rows
    exp = X[sel].astype(np.float64) + a
    assert np.max(np.abs(out - exp)) <= 1e-12 * np.max(np.abs(exp))
    assert np.max(np.abs(a)) > 1e-3 * np.max(np.abs(X))


def _constant_moe(blk, a, b, c):
    """Every gate weight a, up weight b, down weight c (routed and shared)."""
    from tests import kquant_ref as kq2
    moe = blk["moe"]
    for name, val in (("Wg", a), ("Wu", b), ("Sg", a), ("Su", b)):
        moe[name][...] = kq2.encode_q4k(val, 0.0, [1] * 8, [0] * 8, [1] * 256)
    for name in ("Wd", "Sd"):
        moe[name][...] = kq2.encode_q5k(c, 0.0, [1] * 8, [0] * 8, [1] * 256)


@pytest.mark.parametrize("rows", [None, np.array([2, 3])])
def test_block_second_norm_reads_h1(oracle, rows):
    """Attention live, every expert with constant weights a (gate), b (up),
    c (down): each expert maps a row r to c F silu(a S) b S in every output,
    S = sum_i r_i, and the renormalised weights sum to 1, so with the shared
    expert the block is h1 + 2 c F silu(a S) b S with S summed over
    RMSNorm(h1; g2), h1 = X + attn(X). Norming X instead of h1 fails this."""
    blk, X = _small_block(6, T=6, ctx=32)
    a, b, c = 2.0**-4, 2.0**-4, 2.0**-6
    _constant_moe(blk, a, b, c)
    F = blk["moe"]["F"]
    out, kc, vc = _composition_cases(oracle, blk, X, 10, rows)
    att = oracle.attn_sublayer(X, blk, 10, kc.copy(), vc.copy(), rows=rows)
    sel = np.arange(6) if rows is None else rows
    h1 = X[sel].astype(np.float64) + att

    def closed(state):
        S = oracle.rmsnorm(state, blk["g2"]).sum(axis=1, keepdims=True)
        return 2.0 * c * F * (a * S) / (1.0 + np.exp(-a * S)) * (b * S)

    exp = h1 + closed(h1)
    assert np.max(np.abs(out - exp)) <= 1e-12 * np.max(np.abs(exp))
    wrong = h1 + closed(X[sel].astype(np.float64))
    assert np.max(np.abs(out - wrong)) > 1e-6 * np.max(np.abs(exp))
