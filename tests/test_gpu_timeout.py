"""Bounded device waits, driven to run out without faulting the GPU.

"Meet Dis-Tract 0.1.0": a participant that waits on another gives up after a
bounded time and reports the failure instead of hanging. Here every device
wait of the library (a copy's mbarrier, a counter another CTA advances) gives
up after a time limit and records QMOE_ERR_TIMEOUT. The test-only entry point
qmoe_test_inject makes the next calls withhold one copy (decode path), one
producer arrival (tensor-core gate/up kernel) or the prefill attention's
final-output signal with a short limit; the call must return, report the
time-out through qmoe_query_status, and the next normal call must be clean
and correct.
"""

import time

import numpy as np
import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs
from tests.parity import TOL_GEMV, TOL_TC, assert_close

pytestmark = pytest.mark.gpu

_layer = {}


@pytest.fixture(scope="module")
def layer():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    if "l" not in _layer:
        _layer["l"] = qb.MoeLayer.from_arrays(inputs.moe_layer(4, 2048, 256, 512, shared=True), 8)
    return _layer["l"]


def _timed_out_call(layer, X, site, wait_us):
    qb.test_inject(site, wait_us)
    try:
        t0 = time.perf_counter()
        qb.moe_forward(layer, X, X)
        st = qb.query_status()
        dt = time.perf_counter() - t0
    finally:
        qb.test_inject("none")
    return st, dt


@pytest.mark.parametrize("T", [1, 4])
def test_decode_copy_withheld_times_out_then_recovers(layer, T):
    X = torch.from_numpy(inputs.hidden(60 + T, T, 2048)).cuda()
    ref = qb.moe_forward(layer, X, X)
    torch.cuda.synchronize()
    assert qb.query_status() == 0 and qb.last_path() == "decode"
    st, dt = _timed_out_call(layer, X, "decode_copy", 20000)
    assert st == -7, st
    assert dt < 5.0
    again = qb.moe_forward(layer, X, X)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    assert torch.equal(again, ref)


@pytest.mark.parametrize("T", [16, 300])
def test_tensor_core_arrival_withheld_times_out_then_recovers(layer, T):
    X = torch.from_numpy(inputs.hidden(70 + T, T, 2048)).cuda()
    ref = qb.moe_forward(layer, X, X)
    torch.cuda.synchronize()
    assert qb.query_status() == 0 and qb.last_path() == "gemm_tc"
    st, dt = _timed_out_call(layer, X, "tc_arrive", 20000)
    assert st == -7, st
    assert dt < 5.0
    again = qb.moe_forward(layer, X, X)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    assert torch.equal(again, ref)


@pytest.mark.parametrize("T", [17, 300])
def test_attention_final_withheld_times_out_then_recovers(T):
    """The first attention CTA's P V issuer never marks its output final: its
    softmax warps give up, every MMA is drained, TMEM is freed, the call
    reports the time-out, and the next call gives the same bits as before."""
    from quantized_moe_transformer_gb300 import build
    build.build()
    arr = inputs.block(3, ctx=1024)
    blk = qb.Block.from_arrays(arr, 8)
    X = torch.from_numpy(inputs.hidden(80 + T, T, 2048)).cuda()

    def run():
        kd = qb.cache_from_bits(arr["k_cache"])
        vd = qb.cache_from_bits(arr["v_cache"])
        return qb.attn_forward(blk, X, None, kd, vd, 40)

    ref = run()
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    qb.test_inject("attn_final", 20000)
    try:
        t0 = time.perf_counter()
        run()
        st = qb.query_status()
        dt = time.perf_counter() - t0
    finally:
        qb.test_inject("none")
    assert st == -7, st
    assert dt < 5.0
    again = run()
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    assert torch.equal(again, ref)


def test_inject_rejects_unknown_site():
    r = qb.lib().qmoe_test_inject(9, 0)
    assert r == -1
    assert qb.lib().qmoe_test_inject(0, 0) == 0
