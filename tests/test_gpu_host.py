"""The host-buffer entry point qmoe_moe_forward_host against the device one.

The host call copies X (and R) in, runs the layer and copies the result out;
from the second call with the same arguments it replays a captured graph of
that work. Every call must give the bits of qmoe_moe_forward on the same rows
(the layer is deterministic), on the decode path (T = 1, 4) and the tensor-core
path (T = 64), with and without a residual, and a call on other buffers must
not replay another call's graph.
"""

import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs

pytestmark = pytest.mark.gpu

_layer = {}


@pytest.fixture(scope="module")
def layer():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    if "l" not in _layer:
        _layer["l"] = qb.MoeLayer.from_arrays(inputs.moe_layer(8, 2048, 256, 512, shared=True), 8)
    return _layer["l"]


@pytest.mark.parametrize("T", [1, 4, 64])
@pytest.mark.parametrize("with_res", [False, True])
def test_host_forward_matches_device_forward(layer, T, with_res):
    X = torch.from_numpy(inputs.hidden(500 + T, T, 2048))
    R = torch.from_numpy(inputs.hidden(600 + T, T, 2048)) if with_res else None
    Xd = X.cuda()
    Rd = R.cuda() if with_res else None
    ref = qb.moe_forward(layer, Xd, Rd).cpu()
    Xh = X.pin_memory()
    Rh = R.pin_memory() if with_res else None
    ws = torch.empty(qb.host_workspace_bytes(layer, T), dtype=torch.uint8, device="cuda")
    outs = [torch.full_like(Xh, float("nan")).pin_memory() for _ in range(2)]
    for call in range(4):  # direct, capture, replay, replay
        o = outs[0]
        o.fill_(float("nan"))
        qb.moe_forward_host(layer, Xh, Rh, out=o, ws=ws)
        assert torch.equal(o, ref), f"call {call}"
        assert qb.query_status() == 0
    # other output buffer: its own key
    qb.moe_forward_host(layer, Xh, Rh, out=outs[1], ws=ws)
    assert torch.equal(outs[1], ref)
    # new input values in the same pinned buffer are read by the replay
    X2 = torch.from_numpy(inputs.hidden(700 + T, T, 2048))
    Xh.copy_(X2)
    ref2 = qb.moe_forward(layer, X2.cuda(), Rd).cpu()
    qb.moe_forward_host(layer, Xh, Rh, out=outs[0], ws=ws)
    assert torch.equal(outs[0], ref2)


def test_host_forward_pageable_buffers(layer):
    """Pageable host buffers run directly every call and give the same bits."""
    T = 4
    X = torch.from_numpy(inputs.hidden(801, T, 2048))
    ref = qb.moe_forward(layer, X.cuda()).cpu()
    ws = torch.empty(qb.host_workspace_bytes(layer, T), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(X)
    for _ in range(3):
        out.fill_(float("nan"))
        qb.moe_forward_host(layer, X, out=out, ws=ws)
        assert torch.equal(out, ref)
