"""GPU parity of the Q6_K and MXFP4 weight formats (through the C ABI) against
the fp64 oracle's dequant_q6k / dequant_mxfp4.

"CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", opening
paragraphs: the pages run a Q4_K_M model file, a file type that keeps some
tensors (typically the down projections) in Q6_K. "Distributed CPU: Zip Fusion
Beyond Tensor Parallelism", "Decode vs Prefill: Same Weights, Different
Bottlenecks": the model class it targets carries MXFP4-class weights. Layers
with either format run on the grouped GEMV kernels (fp32 accumulation, the
fp32 tolerance), except Q6_K or MXFP4 down projections next to Q4_K gate/up
above the tensor-core threshold: those take the tcgen05 kernels (whole
weight rows by bulk copies, bf16 operands, the tensor-core tolerance).
"""

import numpy as np
import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs
from tests.parity import GAP, TOL_GEMV, TOL_TC, assert_close, check_routes

pytestmark = pytest.mark.gpu

H, E, F, K = 2048, 256, 512, 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    qb.lib()


_layers = {}


def layer(gate, down, seed=3):
    key = (gate, down, seed)
    if key not in _layers:
        if len(_layers) > 2:
            _layers.clear()
            torch.cuda.empty_cache()
        arr = inputs.moe_layer(seed, H, E, F, shared=True, gate_type=gate, down_type=down)
        _layers[key] = (arr, qb.MoeLayer.from_arrays(arr, K))
    return _layers[key]


def expected_path(arr, T):
    tc = (arr["Wg"].shape[-1] == 144 and arr["Wd"].shape[-1] in (210, 136) and T > qb.get_gemm_threshold())
    return "gemm_tc" if tc else "gemv"


def run(oracle, arr, lay, T, seed, rows=None):
    X = inputs.hidden(seed, T, H)
    R = inputs.residual(seed, T, H)
    ws = lay.workspace(T)
    out = qb.moe_forward(lay, torch.from_numpy(X).cuda(), torch.from_numpy(R).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    path = expected_path(arr, T)
    assert qb.last_path() == path
    if rows is None:
        rows = np.arange(T)
    L = lay.workspace_layout(T)
    ids = ws[L.ids:L.ids + 4 * T * K].view(torch.int32).reshape(T, K).cpu().numpy()
    ref, parts = oracle.moe_forward_rows(X, arr, K, rows, R)
    ok = check_routes(ids[rows], parts["ids"], parts["gap"], parts["logits"])
    assert_close(out.cpu().numpy()[rows], ref, TOL_TC if path == "gemm_tc" else TOL_GEMV, rows=ok)


@pytest.mark.parametrize("down", ["q6k", "mxfp4"])
@pytest.mark.parametrize("T", [1, 4, 37, 300])
def test_down_format(oracle, down, T):
    """Q4_K gate/up with a Q6_K or MXFP4 down projection (the Q4_K_M mix)."""
    arr, lay = layer("q4k", down)
    rows = None if T <= 4 else np.array([0, T // 2, T - 1])
    run(oracle, arr, lay, T, 200 + T, rows)


@pytest.mark.parametrize("fmt", ["q6k", "mxfp4"])
def test_gate_up_and_down_same_format(oracle, fmt):
    """Every matrix of the layer in one of the two formats."""
    arr, lay = layer(fmt, fmt)
    run(oracle, arr, lay, 3, 11)
    run(oracle, arr, lay, 65, 12, rows=np.array([0, 40, 64]))


def test_tiny_layer_all_rows(oracle):
    """H=256, E=8, top-2, F=256 (one super-block per row), no shared expert."""
    for down in ("q6k", "mxfp4"):
        arr = inputs.moe_layer(5, 256, 8, 256, shared=False, gate_type="q4k", down_type=down)
        lay = qb.MoeLayer.from_arrays(arr, 2)
        X = inputs.hidden(6, 33, 256)
        out = qb.moe_forward(lay, torch.from_numpy(X).cuda())
        torch.cuda.synchronize()
        path = expected_path(arr, 33)
        assert qb.query_status() == 0 and qb.last_path() == path
        assert_close(out.cpu().numpy(), oracle.moe_forward(X, arr, 2), TOL_TC if path == "gemm_tc" else TOL_GEMV)


def test_q6k_down_tensor_cores_large(oracle):
    """Q6_K down weights on the tensor-core path at T = 4096 (every expert cut
    into token chunks, many work items per SM), sampled rows, and the same
    layer through the GEMV kernels (threshold raised) on one row."""
    arr, lay = layer("q4k", "q6k")
    run(oracle, arr, lay, 4096, 31, rows=np.array([0, 1, 2047, 4095]))
    old = qb.get_gemm_threshold()
    qb.set_gemm_threshold(1 << 20)
    try:
        run(oracle, arr, lay, 6, 32)
    finally:
        qb.set_gemm_threshold(old)


def test_q6k_field_extremes(oracle):
    """Q6_K down blocks at the field extremes: every quant 63 or 0 (all low
    nibbles and high parts set, or none), scales +127 and -128, fp16 d at its
    largest normal; on the GEMV kernels (T = 2) and the tensor-core kernels
    (T = 37, sampled rows)."""
    arr, _ = layer("q4k", "q6k")
    arr = dict(arr)
    Wd = arr["Wd"].copy()
    d = np.frombuffer(np.float16(2.0**-6).tobytes(), np.uint8)
    Wd[..., 0:2] = d
    Wd[..., 2:18] = np.array([127, 128] * 8, np.uint8)      # int8 +127, -128
    Wd[:E // 2, :, :, 18:210] = 0xFF                          # q = 63
    Wd[E // 2:, :, :, 18:210] = 0x00                          # q = 0
    arr["Wd"] = Wd
    Sd = arr["Sd"].copy()
    Sd[..., 0:2] = np.frombuffer(np.float16(65504.0).tobytes(), np.uint8)
    Sd[..., 2:18] = 1
    arr["Sd"] = Sd
    lay = qb.MoeLayer.from_arrays(arr, K)
    run(oracle, arr, lay, 2, 21)
    run(oracle, arr, lay, 37, 23, rows=np.array([0, 18, 36]))  # the tensor-core path


def test_mxfp4_every_code_and_scale(oracle):
    """MXFP4 down blocks cycling through all 16 E2M1 codes (both zeros and the
    negative half) with E8M0 scales 2^-12 .. 2^-1; GEMV kernels (T = 3) and
    tensor-core kernels (T = 37, sampled rows)."""
    arr, _ = layer("q4k", "mxfp4")
    arr = dict(arr)
    Wd = arr["Wd"].copy()
    Wd[..., 0:8] = np.arange(115, 123, dtype=np.uint8) + (np.arange(8, dtype=np.uint8) % 4)
    codes = np.arange(256, dtype=np.uint8) % 16
    Wd[..., 8:136] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    arr["Wd"] = Wd
    lay = qb.MoeLayer.from_arrays(arr, K)
    run(oracle, arr, lay, 3, 22)
    run(oracle, arr, lay, 37, 24, rows=np.array([0, 18, 36]))


def test_mxfp4_down_tensor_cores_large(oracle):
    """MXFP4 down weights on the tensor-core path at T = 4096, sampled rows."""
    arr, lay = layer("q4k", "mxfp4")
    run(oracle, arr, lay, 4096, 33, rows=np.array([0, 1, 2047, 4095]))
