"""GPU parity of the routed-MoE layer (through the C ABI) against the fp64 oracle.

Workloads: the tiny layer (T=4, H=256, E=8, top-2, F=256, Q4_K down, no shared
expert), the Qwen3.5-35B-A3B-shaped decode layer (T=1, H=2048, E=256, top-8,
F=512, Q4_K gate/up, Q5_K down, shared expert), the batched-decode sweep
T = 1..64 under uniform and Zipf(1.1) routing, prefill T = 512 and 4096, and
ragged and degenerate cases.
"""

import numpy as np
import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs
from tests.parity import GAP, TOL_GEMV, TOL_TC, assert_close, check_routes

pytestmark = pytest.mark.gpu

FULL = dict(H=2048, E=256, F=512)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    qb.lib()


_layers = {}


def layer_pair(seed, routing="uniform", tiny=False):
    key = (seed, routing, tiny)
    if key not in _layers:
        if tiny:
            arr = inputs.moe_layer(seed, 256, 8, 256, shared=False, down_type="q4k", routing=routing)
            k = 2
        else:
            arr = inputs.moe_layer(seed, **FULL, shared=True, routing=routing)
            k = 8
        if len(_layers) > 3:
            _layers.clear()
            torch.cuda.empty_cache()
        _layers[key] = (arr, qb.MoeLayer.from_arrays(arr, k), k)
    return _layers[key]


def tol_for_path():
    return TOL_TC if qb.last_path() == "gemm_tc" else TOL_GEMV


def run_and_check(oracle, seed, T, routing="uniform", tiny=False, rows=None, R_mode="none"):
    arr, lay, k = layer_pair(seed, routing, tiny)
    X = inputs.hidden(seed + 100 * T, T, arr["H"], routing)
    R = None
    if R_mode == "x":
        R = X
    elif R_mode == "sep":
        R = inputs.residual(seed, T, arr["H"])
    Xd = torch.from_numpy(X).cuda()
    Rd = None if R is None else torch.from_numpy(R).cuda()
    ws = lay.workspace(T)
    out = qb.moe_forward(lay, Xd, Rd, ws=ws)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    tol = tol_for_path()
    L = lay.workspace_layout(T)
    ids_gpu = ws[L.ids:L.ids + 4 * T * k].view(torch.int32).reshape(T, k).cpu().numpy()
    if rows is None:
        rows = np.arange(T)
    ref, parts = oracle.moe_forward_rows(X, arr, k, rows, R)
    ok = check_routes(ids_gpu[rows], parts["ids"], parts["gap"], parts["logits"])
    assert_close(out.cpu().numpy()[rows], ref, tol, rows=ok)
    return out, ws, parts


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("R_mode", ["none", "x", "sep"])
def test_tiny_layer(oracle, seed, R_mode):
    run_and_check(oracle, seed, 4, tiny=True, R_mode=R_mode)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_layer(oracle, seed):
    run_and_check(oracle, seed, 1, R_mode="x")
    assert qb.last_path() == "decode"


@pytest.mark.parametrize("routing", ["uniform", "zipf"])
@pytest.mark.parametrize("T", [1, 2, 4, 8, 16, 32, 64])
def test_decode_sweep(oracle, T, routing):
    rows = np.unique(np.linspace(0, T - 1, min(T, 6)).astype(int))
    run_and_check(oracle, 0, T, routing, rows=rows)


@pytest.mark.parametrize("routing", ["uniform", "zipf"])
@pytest.mark.parametrize("T", [512, 4096])
def test_prefill_sampled_rows(oracle, T, routing):
    rows = np.array([0, 1, T // 3, T // 2 + 7, T - 2, T - 1])
    run_and_check(oracle, 1, T, routing, rows=rows, R_mode="sep")


@pytest.mark.parametrize("T", [3, 37, 100, 300])
def test_ragged_rows(oracle, T):
    rows = np.array(sorted({0, T // 2, T - 1}))
    run_and_check(oracle, 2, T, rows=rows)


def test_tiny_ragged_all_rows(oracle):
    for T in (1, 5, 33, 130):
        run_and_check(oracle, 0, T, tiny=True, R_mode="sep")


def test_zero_rows():
    arr, lay, k = layer_pair(0, tiny=True)
    X = torch.empty((0, 256), device="cuda")
    out = qb.moe_forward(lay, X, ws=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert out.shape == (0, 256)


def test_route_entry_point(oracle):
    for T, seed in ((1, 0), (64, 1), (4096, 2)):
        arr, lay, k = layer_pair(0)
        X = inputs.hidden(seed, T, 2048)
        ids, w = qb.moe_route(torch.from_numpy(X).cuda(), lay.Wr, k)
        torch.cuda.synchronize()
        oids, ow, gap, logits = oracle.route(X, arr["Wr"], k)
        ok = check_routes(ids.cpu().numpy(), oids, gap, logits)
        np.testing.assert_allclose(w.cpu().numpy()[ok], ow[ok], rtol=0, atol=2e-6)


@pytest.mark.parametrize("T", [256, 300, 1000])
@pytest.mark.parametrize("routing", ["uniform", "zipf"])
def test_route_entry_point_tensor_core_router(oracle, T, routing):
    """From 256 rows the router runs on the tensor cores (three-part bf16 split,
    several H slices); row tiles of 128 end ragged at T = 300 and 1000."""
    arr, lay, k = layer_pair(0, routing=routing)
    X = inputs.hidden(11 + T, T, 2048, routing=routing)
    ids, w = qb.moe_route(torch.from_numpy(X).cuda(), lay.Wr, k)
    torch.cuda.synchronize()
    oids, ow, gap, logits = oracle.route(X, arr["Wr"], k)
    ok = check_routes(ids.cpu().numpy(), oids, gap, logits)
    np.testing.assert_allclose(w.cpu().numpy()[ok], ow[ok], rtol=0, atol=2e-6)


def test_caller_supplied_routes(oracle):
    """One routing decision fed to the layer (the synchronised-router case)."""
    arr, lay, k = layer_pair(0)
    X = inputs.hidden(7, 16, 2048)
    oids, ow, _, _ = oracle.route(X, arr["Wr"], k)
    ids = torch.from_numpy(oids.astype(np.int32)).cuda()
    w = torch.from_numpy(ow.astype(np.float32)).cuda()
    out = qb.moe_forward(lay, torch.from_numpy(X).cuda(), ids=ids, w=w)
    ref = oracle.moe_forward(X, arr, k)
    assert_close(out.cpu().numpy(), ref, tol_for_path())


def test_run_to_run_bit_identical():
    arr, lay, k = layer_pair(1)
    X = torch.from_numpy(inputs.hidden(3, 64, 2048)).cuda()
    a = qb.moe_forward(lay, X)
    b = qb.moe_forward(lay, X)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_stagewise_expert_outputs(oracle):
    """Per-(row, slot) expert outputs y in the workspace against the oracle's."""
    arr, lay, k = layer_pair(0)
    T = 2
    X = inputs.hidden(11, T, 2048)
    ws = lay.workspace(T)
    qb.set_decode_max_rows(0)
    try:
        qb.moe_forward(lay, torch.from_numpy(X).cuda(), ws=ws)
        assert qb.last_path() == "gemv"
    finally:
        qb.set_decode_max_rows(-1)
    torch.cuda.synchronize()
    L = lay.workspace_layout(T)
    rows = T * k + T
    y = ws[L.y:L.y + 4 * rows * 2048].view(torch.float32).reshape(rows, 2048).cpu().numpy()
    ref, parts = oracle.moe_forward(X, arr, k, return_parts=True)
    for t in range(T):
        for s in range(k):
            assert_close(y[t * k + s], parts["y"][t, s], tol_for_path())
        assert_close(y[T * k + t], parts["y_shared"][t], tol_for_path())
    offs = ws[L.offsets:L.offsets + 4 * (256 + 2)].view(torch.int32).cpu().numpy()
    assert offs[0] == 0 and offs[256] == T * k and offs[257] == T * k + T
    perm = ws[L.perm:L.perm + 4 * rows].view(torch.int32).cpu().numpy()
    assert sorted(perm.tolist()) == list(range(rows))


def _half(t: torch.Tensor, dim: int, r: int, n: int) -> torch.Tensor:
    return t.narrow(dim, r * n, n).contiguous()


def test_f_split_partials_sum_to_layer(oracle):
    """Rank partials of the 256/256 intermediate split, each run through the
    library with its slices of the packed tensors and one shared routing
    decision, sum to the whole layer."""
    arr, lay, k = layer_pair(2)
    T = 8
    X = inputs.hidden(5, T, 2048)
    Xd = torch.from_numpy(X).cuda()
    ids, w = qb.moe_route(Xd, lay.Wr, k)
    full = qb.moe_forward(lay, Xd, ids=ids, w=w)
    parts = []
    for r in range(2):
        half = qb.MoeLayer(2048, 256, k, 256, lay.Wr, _half(lay.Wg, 1, r, 256), _half(lay.Wu, 1, r, 256),
                           _half(lay.Wd, 2, r, 1), _half(lay.Sg, 0, r, 256), _half(lay.Su, 0, r, 256),
                           _half(lay.Sd, 1, r, 1))
        parts.append(qb.moe_forward(half, Xd, ids=ids, w=w))
    torch.cuda.synchronize()
    tot = (parts[0] + parts[1]).cpu().numpy()
    tol = tol_for_path()
    assert_close(tot, full.cpu().numpy(), tol)
    for r in range(2):
        assert_close(parts[r].cpu().numpy(), oracle.moe_forward(X, arr, k, f_half=r), tol)


def test_out_of_range_route_is_reported_not_faulted():
    arr, lay, k = layer_pair(0, tiny=True)
    X = torch.from_numpy(inputs.hidden(0, 4, 256)).cuda()
    ids = torch.tensor([[0, 1], [2, 99], [3, 4], [5, -1]], dtype=torch.int32, device="cuda")
    w = torch.full((4, 2), 0.5, device="cuda")
    qb.moe_forward(lay, X, ids=ids, w=w)
    assert qb.query_status() == -8
    assert qb.query_status() == 0


def test_argument_errors():
    arr, lay, k = layer_pair(0, tiny=True)
    X = torch.from_numpy(inputs.hidden(0, 4, 256)).cuda()
    ws = lay.workspace(4)
    with pytest.raises(qb.QmoeError, match="workspace"):
        qb.moe_forward(lay, X, ws=ws[: ws.numel() // 2])
    with pytest.raises(qb.QmoeError, match="aligned"):
        qb.moe_forward(lay, X, ws=ws[1:])
    with pytest.raises(qb.QmoeError):
        qb.moe_forward(lay, X, out=X)


@pytest.mark.parametrize("T", [65, 200])
def test_gemv_and_tensor_core_paths_agree(oracle, T):
    """The same rows through both paths (threshold forced each way)."""
    arr, lay, k = layer_pair(0)
    X = inputs.hidden(21, T, 2048)
    Xd = torch.from_numpy(X).cuda()
    old = qb.get_gemm_threshold()
    try:
        qb.set_gemm_threshold(10**9)
        a = qb.moe_forward(lay, Xd)
        assert qb.last_path() == "gemv"
        qb.set_gemm_threshold(0)
        b = qb.moe_forward(lay, Xd)
        assert qb.last_path() == "gemm_tc"
    finally:
        qb.set_gemm_threshold(old)
    torch.cuda.synchronize()
    assert_close(b.cpu().numpy(), a.cpu().numpy(), TOL_TC)
    rows = np.array([0, T // 2, T - 1])
    ref, parts = oracle.moe_forward_rows(X, arr, k, rows)
    ok = parts["gap"] >= GAP
    assert_close(a.cpu().numpy()[rows], ref, TOL_GEMV, rows=ok)
    assert_close(b.cpu().numpy()[rows], ref, TOL_TC, rows=ok)


def test_tensor_core_path_bit_identical():
    arr, lay, k = layer_pair(1)
    X = torch.from_numpy(inputs.hidden(4, 512, 2048)).cuda()
    a = qb.moe_forward(lay, X)
    assert qb.last_path() == "gemm_tc"
    b = qb.moe_forward(lay, X)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("routing", ["uniform", "zipf"])
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_decode_path_matches_gemv_path(oracle, T, routing):
    """The PDL-chained decode path and the grouped GEMV path on the same rows;
    both against the oracle; the decode path's routes and per-pair outputs."""
    arr, lay, k = layer_pair(1, routing)
    X = inputs.hidden(31 + T, T, 2048, routing)
    R = inputs.residual(5, T, 2048)
    Xd, Rd = torch.from_numpy(X).cuda(), torch.from_numpy(R).cuda()
    ws = lay.workspace(T)
    a = qb.moe_forward(lay, Xd, Rd, ws=ws)
    assert qb.last_path() == "decode"
    torch.cuda.synchronize()
    L = lay.workspace_layout(T)
    ids = ws[L.ids:L.ids + 4 * T * k].view(torch.int32).reshape(T, k).cpu().numpy()
    w = ws[L.w:L.w + 4 * T * k].view(torch.float32).reshape(T, k).cpu().numpy()
    rows = T * k + T
    y = ws[L.y:L.y + 4 * rows * 2048].view(torch.float32).reshape(rows, 2048).cpu().numpy()
    qb.set_decode_max_rows(0)
    try:
        b = qb.moe_forward(lay, Xd, Rd)
        assert qb.last_path() == "gemv"
    finally:
        qb.set_decode_max_rows(-1)
    torch.cuda.synchronize()
    assert_close(a.cpu().numpy(), b.cpu().numpy(), TOL_GEMV)
    ref, parts = oracle.moe_forward(X, arr, k, R, return_parts=True)
    ok = check_routes(ids, parts["ids"], parts["gap"], parts["logits"])
    assert_close(a.cpu().numpy(), ref, TOL_GEMV, rows=ok)
    np.testing.assert_allclose(w[ok], parts["w"][ok], rtol=0, atol=2e-6)
    for t in np.nonzero(ok)[0]:
        for s2 in range(k):
            assert_close(y[t * k + s2], parts["y"][t, s2], TOL_GEMV)
        assert_close(y[T * k + t], parts["y_shared"][t], TOL_GEMV)


def test_decode_path_bit_identical_and_chained():
    """Run to run bit identity, and a chain of layers where each output is the
    next input (the previous kernel's output read after the PDL wait)."""
    arr, lay, k = layer_pair(2)
    X = torch.from_numpy(inputs.hidden(8, 1, 2048)).cuda()
    a = qb.moe_forward(lay, X, X)
    b = qb.moe_forward(lay, X, X)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    h1 = qb.moe_forward(lay, X, X)
    h2 = qb.moe_forward(lay, h1 / h1.abs().max(), h1 / h1.abs().max())
    torch.cuda.synchronize()
    qb.set_decode_max_rows(0)
    try:
        g1 = qb.moe_forward(lay, X, X)
        g2 = qb.moe_forward(lay, g1 / g1.abs().max(), g1 / g1.abs().max())
    finally:
        qb.set_decode_max_rows(-1)
    torch.cuda.synchronize()
    assert_close(h2.cpu().numpy(), g2.cpu().numpy(), TOL_GEMV)
