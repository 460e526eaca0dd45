"""GPU parity of the causal prefill attention (the tcgen05 kernel: S and O in
tensor memory) through the attention sub-layer entry point, on every row.

"CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "What PR #382
Now Splits": 16 query heads over 2 KV heads, query head h reading KV head
h / 8, causal, scale 1/sqrt(128). "Distributed CPU: Zip Fusion Beyond Tensor
Parallelism", "Two-Dimensional Attention at Long Context": the softmax over
key blocks is carried by a running maximum, normaliser and weighted output.

Most cases run the projections on the fp32 GEMV kernels (the tensor-core threshold
is raised), so the attention kernel's own bf16 operands (the scaled queries,
the bf16 cache, the bf16 probabilities) are the only roundings besides the
cache's; the tolerance is the tensor-core one. Shapes cross the kernel's
128-row query tiles and 128-key blocks at unaligned offsets: one partial tile
(T = 17), exactly one tile, one tile plus a row, three tiles with the last
partial, a cache offset that is not a multiple of 128, and one KV head for
8 query heads (a rank's slice of the block).
"""

import numpy as np
import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs
from tests.parity import TOL_TC, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def blk_pair():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    arr = inputs.block(3, ctx=2048)
    return arr, qb.Block.from_arrays(arr, 8)


@pytest.fixture
def fp32_projections():
    old = qb.get_gemm_threshold()
    qb.set_gemm_threshold(1 << 20)
    yield
    qb.set_gemm_threshold(old)


@pytest.mark.parametrize("T,pos0", [(17, 0), (128, 0), (129, 77), (300, 77), (300, 1000)])
def test_prefill_attention_every_row(oracle, blk_pair, fp32_projections, T, pos0):
    arr, blk = blk_pair
    X = inputs.hidden(300 + T + pos0, T, 2048)
    kd = qb.cache_from_bits(arr["k_cache"])
    vd = qb.cache_from_bits(arr["v_cache"])
    got = qb.attn_forward(blk, torch.from_numpy(X).cuda(), None, kd, vd, pos0)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    kc = oracle.bf16_bits_to_f64(arr["k_cache"])
    vc = oracle.bf16_bits_to_f64(arr["v_cache"])
    ref = oracle.attn_sublayer(X, arr, pos0, kc, vc)
    assert_close(got.cpu().numpy(), ref, TOL_TC)


def test_prefill_attention_one_kv_head(oracle, blk_pair, fp32_projections):
    """8 query heads on one KV head: rank 1's slice (query heads 8..15, KV head
    1, O input columns 1024..2047) against the oracle's rank partial."""
    arr, _ = blk_pair
    hd = 128
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    moe = arr["moe"]
    half = qb.MoeLayer(2048, 256, 8, 512, d(moe["Wr"]), d(moe["Wg"]), d(moe["Wu"]), d(moe["Wd"]),
                       d(moe["Sg"]), d(moe["Su"]), d(moe["Sd"]))
    rb = qb.Block(2048, 8, 1, hd, d(arr["g1"]), d(arr["g2"]), d(arr["Wq"][8 * hd:16 * hd]),
                  d(arr["Wk"][hd:2 * hd]), d(arr["Wv"][hd:2 * hd]), d(arr["Wo"][:, 4:8]), half)
    T, pos0 = 200, 130
    X = inputs.hidden(401, T, 2048)
    kd = qb.cache_from_bits(arr["k_cache"])[:, 1:2].contiguous()
    vd = qb.cache_from_bits(arr["v_cache"])[:, 1:2].contiguous()
    got = qb.attn_forward(rb, torch.from_numpy(X).cuda(), None, kd, vd, pos0)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    kc = oracle.bf16_bits_to_f64(arr["k_cache"])
    vc = oracle.bf16_bits_to_f64(arr["v_cache"])
    ref = oracle.attn_sublayer(X, arr, pos0, kc, vc, rank=1)
    assert_close(got.cpu().numpy(), ref, TOL_TC)


def test_prefill_attention_repeatable(blk_pair, fp32_projections):
    """Two runs of the same call give the same bits."""
    arr, blk = blk_pair
    X = torch.from_numpy(inputs.hidden(402, 257, 2048)).cuda()
    outs = []
    for _ in range(2):
        kd = qb.cache_from_bits(arr["k_cache"])
        vd = qb.cache_from_bits(arr["v_cache"])
        outs.append(qb.attn_forward(blk, X, None, kd, vd, 5))
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_prefill_attention_one_kv_head_mixed_paths(blk_pair):
    """The same rank slice at the default tensor-core threshold: the Q and O
    projections (1024 and 2048 outputs) run on the tensor cores, the K and V
    projections (128 outputs, not a whole 256-row weight block) on the fp32
    kernels, which read the fp32 RMSNorm rows. The K/V cache rows the call
    writes must be the bits the all-fp32 projections write, and the call with
    a residual must give the bits of X + the sub-layer without it. (Against the oracle, bf16 queries move this slice's
    large synthetic attention scores beyond the tensor-core bound; the
    all-tensor-core block is checked against the oracle in test_gpu_block.)"""
    arr, _ = blk_pair
    hd = 128
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    moe = arr["moe"]
    half = qb.MoeLayer(2048, 256, 8, 512, d(moe["Wr"]), d(moe["Wg"]), d(moe["Wu"]), d(moe["Wd"]),
                       d(moe["Sg"]), d(moe["Su"]), d(moe["Sd"]))
    rb = qb.Block(2048, 8, 1, hd, d(arr["g1"]), d(arr["g2"]), d(arr["Wq"][8 * hd:16 * hd]),
                  d(arr["Wk"][hd:2 * hd]), d(arr["Wv"][hd:2 * hd]), d(arr["Wo"][:, 4:8]), half)
    T, pos0 = 200, 130
    assert T > qb.get_gemm_threshold()
    Xd = torch.from_numpy(inputs.hidden(403, T, 2048)).cuda()

    def caches():
        return (qb.cache_from_bits(arr["k_cache"])[:, 1:2].contiguous(),
                qb.cache_from_bits(arr["v_cache"])[:, 1:2].contiguous())

    kd, vd = caches()
    with_res = qb.attn_forward(rb, Xd, Xd, kd, vd, pos0)
    kd2, vd2 = caches()
    no_res = qb.attn_forward(rb, Xd, None, kd2, vd2, pos0)
    old = qb.get_gemm_threshold()
    qb.set_gemm_threshold(1 << 20)
    try:
        kf, vf = caches()
        qb.attn_forward(rb, Xd, None, kf, vf, pos0)
    finally:
        qb.set_gemm_threshold(old)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    assert torch.isfinite(with_res).all()
    rows = slice(pos0, pos0 + T)
    assert torch.equal(kd[rows], kf[rows]) and torch.equal(vd[rows], vf[rows])
    assert torch.equal(with_res, Xd + no_res)
