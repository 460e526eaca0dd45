"""GPU parity of the attention + MoE block (Qwen3.5-35B-A3B-shaped: H=2048,
16 query heads, 2 KV heads, head_dim 128, RoPE theta 1e7, bf16 KV cache, the
decode MoE layer) against the fp64 oracle, at T=1 against a 4095-entry cache,
at prefill T=4096 (sampled rows), at ragged T, and as two rank partials (8
query heads + 1 KV head each; intermediate split 256/256) summed."""

import numpy as np
import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs
from tests.parity import GAP, TOL_GEMV, TOL_TC, assert_close

pytestmark = pytest.mark.gpu
K_TOP = 8


@pytest.fixture(scope="module")
def blk_pair():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    arr = inputs.block(0, ctx=4096)
    return arr, qb.Block.from_arrays(arr, K_TOP)


def _caches(arr, oracle):
    kd = qb.cache_from_bits(arr["k_cache"])
    vd = qb.cache_from_bits(arr["v_cache"])
    return kd, vd, oracle.bf16_bits_to_f64(arr["k_cache"]), oracle.bf16_bits_to_f64(arr["v_cache"])


def _check_rows(got, ref, parts, tol):
    ok = parts["gap"] >= GAP
    assert_close(got, ref, tol, rows=ok)


@pytest.mark.parametrize("seed", [0, 1])
def test_block_decode_against_long_cache(oracle, blk_pair, seed):
    arr, blk = blk_pair
    kd, vd, kc, vc = _caches(arr, oracle)
    pos0 = 4095
    X = inputs.hidden(50 + seed, 1, 2048)
    out = qb.block_forward(blk, torch.from_numpy(X).cuda(), kd, vd, pos0)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    ref, parts = oracle.block_forward_rows(X, arr, K_TOP, pos0, kc, vc, np.array([0]))
    _check_rows(out.cpu().numpy(), ref, parts, TOL_GEMV)
    # the new key and value went into the cache at pos0, bf16
    kref = oracle.round_bf16(kc[pos0])
    kgot = kd[pos0].float().cpu().numpy()
    assert np.max(np.abs(kgot - kref)) <= 2 ** -7 * np.max(np.abs(kref))


@pytest.mark.parametrize("T,pos0", [(5, 100), (37, 0), (100, 3000)])
def test_block_ragged(oracle, blk_pair, T, pos0):
    arr, blk = blk_pair
    kd, vd, kc, vc = _caches(arr, oracle)
    X = inputs.hidden(60 + T, T, 2048)
    out = qb.block_forward(blk, torch.from_numpy(X).cuda(), kd, vd, pos0)
    torch.cuda.synchronize()
    rows = np.array(sorted({0, T // 2, T - 1}))
    ref, parts = oracle.block_forward_rows(X, arr, K_TOP, pos0, kc, vc, rows)
    tol = TOL_TC if T > qb.get_gemm_threshold() else TOL_GEMV
    _check_rows(out.cpu().numpy()[rows], ref, parts, tol)


def test_block_prefill_4096(oracle, blk_pair):
    arr, blk = blk_pair
    kd, vd, kc, vc = _caches(arr, oracle)
    T = 4096
    X = inputs.hidden(70, T, 2048)
    out = qb.block_forward(blk, torch.from_numpy(X).cuda(), kd, vd, 0)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    rows = np.array([0, 1, 63, 64, 2047, 4094, 4095])
    ref, parts = oracle.block_forward_rows(X, arr, K_TOP, 0, kc, vc, rows)
    _check_rows(out.cpu().numpy()[rows], ref, parts, TOL_TC)


def test_decode_after_prefill_matches_prefill(blk_pair):
    """Prefill 20 rows, then decode row 20 alone: equals row 20 of a 21-row
    prefill (the fp32 GEMV kernels for the projections and the MoE layer at
    every size here, the threshold raised for the test)."""
    arr, blk = blk_pair
    X = torch.from_numpy(inputs.hidden(80, 21, 2048)).cuda()
    old = qb.get_gemm_threshold()
    qb.set_gemm_threshold(64)
    try:
        k1, v1 = qb.cache_from_bits(arr["k_cache"]), qb.cache_from_bits(arr["v_cache"])
        full = qb.block_forward(blk, X, k1, v1, 0)
        k2, v2 = qb.cache_from_bits(arr["k_cache"]), qb.cache_from_bits(arr["v_cache"])
        qb.block_forward(blk, X[:20].contiguous(), k2, v2, 0)
        last = qb.block_forward(blk, X[20:].contiguous(), k2, v2, 20)
        torch.cuda.synchronize()
    finally:
        qb.set_gemm_threshold(old)
    assert_close(last.cpu().numpy(), full[20:].cpu().numpy(), TOL_GEMV)


def _slice_block(arr, r):
    """Rank r's weights: query heads 8r..8r+7, KV head r, O input columns
    [1024r, 1024r+1024) (4 super-blocks), the MoE intermediate half r."""
    hd = 128
    q_rows = slice(8 * r * hd, 8 * (r + 1) * hd)
    kv_rows = slice(r * hd, (r + 1) * hd)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    moe = arr["moe"]
    half = qb.MoeLayer(2048, 256, K_TOP, 256, d(moe["Wr"]), d(moe["Wg"][:, 256 * r:256 * (r + 1)]),
                       d(moe["Wu"][:, 256 * r:256 * (r + 1)]), d(moe["Wd"][:, :, r:r + 1]),
                       d(moe["Sg"][256 * r:256 * (r + 1)]), d(moe["Su"][256 * r:256 * (r + 1)]),
                       d(moe["Sd"][:, r:r + 1]))
    return qb.Block(2048, 8, 1, hd, d(arr["g1"]), d(arr["g2"]), d(arr["Wq"][q_rows]), d(arr["Wk"][kv_rows]),
                    d(arr["Wv"][kv_rows]), d(arr["Wo"][:, 4 * r:4 * (r + 1)]), half)


@pytest.fixture
def fp32_path():
    """The fp32 GEMV kernels at every size the test uses: the split invariant
    is checked at the fp32 tolerance. (With random weights the block's
    attention scores are large, so bf16 rounding of the K/V projections on the
    tensor-core path moves the softmax by more than that; the tensor-core path
    is checked against the oracle in test_block_ragged and
    test_block_prefill_4096.)"""
    old = qb.get_gemm_threshold()
    qb.set_gemm_threshold(64)
    yield
    qb.set_gemm_threshold(old)


@pytest.mark.parametrize("T,pos0", [(1, 4095), (8, 200)])
def test_rank_partials_sum_to_block(oracle, blk_pair, fp32_path, T, pos0):
    arr, blk = blk_pair
    X = inputs.hidden(90 + T, T, 2048)
    Xd = torch.from_numpy(X).cuda()
    kc_full = qb.cache_from_bits(arr["k_cache"])
    vc_full = qb.cache_from_bits(arr["v_cache"])
    whole = qb.block_forward(blk, Xd, kc_full.clone(), vc_full.clone(), pos0)
    # attention partials, each rank with its own KV head's cache
    h1 = Xd.clone()
    for r in range(2):
        rb = _slice_block(arr, r)
        kc_r = kc_full[:, r:r + 1].contiguous()
        vc_r = vc_full[:, r:r + 1].contiguous()
        h1 += qb.attn_forward(rb, Xd, None, kc_r, vc_r, pos0)
    r2 = qb.rmsnorm(h1, blk.g2)
    ids, w = qb.moe_route(r2, blk.moe.Wr, K_TOP)   # one synchronised routing decision
    out = h1.clone()
    for r in range(2):
        rb = _slice_block(arr, r)
        out += qb.moe_forward(rb.moe, r2, ids=ids, w=w)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), whole.cpu().numpy(), TOL_GEMV)
    kc = oracle.bf16_bits_to_f64(arr["k_cache"])
    vc = oracle.bf16_bits_to_f64(arr["v_cache"])
    ref, parts = oracle.block_forward_rows(X, arr, K_TOP, pos0, kc, vc, np.arange(T))
    _check_rows(out.cpu().numpy(), ref, parts, TOL_GEMV)
