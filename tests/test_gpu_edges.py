"""GPU parity at the edges of the routed-MoE layer, through the C ABI, against
the fp64 oracle.

* Planted exact ties: router columns duplicated in groups of three give
  bit-identical logits on the GPU and in the oracle, so the lower-index rule
  decides both the selected set (a tie across the k-th/(k+1)-th boundary) and
  the slot order, on all three router paths (the decode path's router, the
  CUDA-core router below 256 rows, the tensor-core router from 256 rows).
* Field extremes of the packed super-blocks: fp16 d and dmin at 65504 and at
  2^-14 (the largest and smallest normal), every 6-bit scale and min at 63,
  every Q5_K high bit set, quants at their maximum.
* Zero scales: routed experts with d = dmin = 0 leave R + y_shared; every
  expert zero leaves R exactly.
* Extreme skew: every row routed to the same eight experts (4096 rows), and
  caller-supplied routes sending every slot of every row to one expert.
* The permutation and offsets against a stable sort of the routes.
* Rows of NaN logits: the k lowest indices, never a repeated id.

Sources: "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights",
"What The First Prototype Split" (selected top-k ids and weights, rows
independent) and "What PR #382 Now Splits" (the layer's shapes and formats).
"""

import numpy as np
import pytest
import torch

from quantized_moe_transformer_gb300 import binding as qb
from quantized_moe_transformer_gb300 import inputs
from tests import kquant_ref as kq
from tests.parity import GAP, TOL_GEMV, TOL_TC, assert_close

pytestmark = pytest.mark.gpu

H, E, F, K = 2048, 256, 512, 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_moe_transformer_gb300 import build
    build.build()
    qb.lib()


def tol():
    return TOL_TC if qb.last_path() == "gemm_tc" else TOL_GEMV


def triplet_router(seed, routing="uniform"):
    """Router weights whose columns come in groups of three equal columns
    (3m, 3m+1, 3m+2), so that the three experts of a group have equal logits
    on every row: k = 8 then always cuts through a group."""
    Wr = inputs.generator(seed, "Wr").normal(0.0, 0.02, size=(H, E)).astype(np.float32)
    for m in range(E // 3):
        Wr[:, 3 * m + 1] = Wr[:, 3 * m]
        Wr[:, 3 * m + 2] = Wr[:, 3 * m]
    return Wr


def check_tied_routes(ids_gpu, w_gpu, X, Wr, oracle):
    """Exact ids and slot order on every row, where the only near-ties among
    the top k+1 logits are the planted exact ones; rows with an accidental
    gap in (0, 1e-5) are excused (and counted)."""
    oids, ow, _, L = oracle.route(X, Wr, K)
    T = X.shape[0]
    counted = 0
    for t in range(T):
        srt = -np.sort(-L[t])[: K + 1]
        gaps = -np.diff(srt)
        if np.any((gaps > 0) & (gaps < GAP)):
            continue
        counted += 1
        assert list(ids_gpu[t]) == list(oids[t]), (t, ids_gpu[t], oids[t])
        np.testing.assert_allclose(w_gpu[t], ow[t], rtol=0, atol=2e-6)
        # the planted ties really are in play: the k-th and (k+1)-th are equal
        assert srt[K - 1] == srt[K]
    assert counted >= max(1, int(0.99 * T)), (counted, T)


@pytest.mark.parametrize("T", [1, 3, 16, 64, 200, 256, 300])
def test_planted_ties_router(oracle, T):
    """qmoe_moe_route: T < 256 on the CUDA-core router, T >= 256 on the
    tensor-core router (three-part bf16 split); equal columns give equal fp32
    logits on either."""
    Wr = triplet_router(1)
    X = inputs.hidden(50 + T, T, H)
    ids, w = qb.moe_route(torch.from_numpy(X).cuda(), torch.from_numpy(Wr).cuda(), K)
    torch.cuda.synchronize()
    check_tied_routes(ids.cpu().numpy(), w.cpu().numpy(), X, Wr, oracle)


_tie_layer = {}


def tie_layer():
    if "l" not in _tie_layer:
        arr = inputs.moe_layer(2, H, E, F, shared=True)
        arr["Wr"] = triplet_router(2)
        _tie_layer["l"] = (arr, qb.MoeLayer.from_arrays(arr, K))
    return _tie_layer["l"]


@pytest.mark.parametrize("T", [1, 2, 3, 4, 8])
def test_planted_ties_layer(oracle, T):
    """The whole layer with planted ties: the decode path (T <= 4) and the
    tensor-core path take the same ids, in the same slot order, as the oracle,
    and the same output."""
    arr, lay = tie_layer()
    X = inputs.hidden(70 + T, T, H)
    ws = lay.workspace(T)
    out = qb.moe_forward(lay, torch.from_numpy(X).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    L = lay.workspace_layout(T)
    ids = ws[L.ids:L.ids + 4 * T * K].view(torch.int32).reshape(T, K).cpu().numpy()
    w = ws[L.w:L.w + 4 * T * K].view(torch.float32).reshape(T, K).cpu().numpy()
    check_tied_routes(ids, w, X, arr["Wr"], oracle)
    ref = oracle.moe_forward(X, arr, K)
    assert_close(out.cpu().numpy(), ref, tol())


def test_nan_rows_take_lowest_indices():
    """A row whose logits are all NaN selects experts 0..k-1, each once, on the
    CUDA-core and tensor-core routers and in the decode path."""
    Wr = torch.from_numpy(inputs.generator(3, "Wr").normal(0, 0.02, size=(H, E)).astype(np.float32)).cuda()
    for T in (2, 300):
        X = torch.from_numpy(inputs.hidden(9, T, H)).cuda()
        X[1] = float("nan")
        ids, _ = qb.moe_route(X, Wr, K)
        torch.cuda.synchronize()
        assert ids[1].tolist() == list(range(K)), (T, ids[1].tolist())
        others = ids.cpu().numpy()
        for t in range(T):
            assert len(set(others[t].tolist())) == K


# ------------------------------------------------------------------ field extremes

def extreme_layer(kind):
    """Layer whose super-blocks hold extreme header fields: d = dmin = 65504
    ("large") or 2^-14 ("small") with every s_j = m_j = 63 and every Q5_K high
    bit set (quants random); or ("max") every quant at its maximum (q = 15,
    31), s = m = 63, d = 2^-10 and dmin = (q_max - 1) d, so that every weight
    is 63 d, a value bf16 holds exactly (a constant weight that bf16 rounded
    would put the same rounding error on every product, which no tolerance
    built on independent roundings covers)."""
    arr = inputs.moe_layer(5, H, E, F, shared=True)
    d = {"large": 65504.0, "small": 2.0**-14, "max": 2.0**-10}[kind]
    for name in ("Wg", "Wu", "Sg", "Su", "Wd", "Sd"):
        a = arr[name]
        q5 = a.shape[-1] == 176
        dmin = d if kind != "max" else (30.0 if q5 else 14.0) * d
        a[..., 0:16] = np.frombuffer(kq.encode_header(d, dmin, [63] * 8, [63] * 8), dtype=np.uint8)
        if q5:
            a[..., 16:48] = 0xFF
        if kind == "max":
            a[..., -128:] = 0xFF
    return arr


@pytest.mark.parametrize("kind", ["large", "small", "max"])
@pytest.mark.parametrize("T", [1, 3, 16, 300])
def test_field_extremes(oracle, kind, T):
    """Decode path (T = 1, 3), GEMV path (T = 3 with the decode path off) and
    tensor-core path (T = 16, 300) on extreme super-blocks."""
    arr = extreme_layer(kind)
    lay = qb.MoeLayer.from_arrays(arr, K)
    X = inputs.hidden(80 + T, T, H)
    R = inputs.residual(8, T, H)
    rows = np.unique(np.array([0, T // 2, T - 1]))
    ref, parts = oracle.moe_forward_rows(X, arr, K, rows, R)
    variants = [None] if T != 3 else [None, "gemv"]
    for v in variants:
        if v == "gemv":
            qb.set_decode_max_rows(0)
        try:
            out = qb.moe_forward(lay, torch.from_numpy(X).cuda(), torch.from_numpy(R).cuda())
            path = qb.last_path()
        finally:
            qb.set_decode_max_rows(-1)
        torch.cuda.synchronize()
        assert qb.query_status() == 0
        if v == "gemv":
            assert path == "gemv"
        got = out.cpu().numpy()[rows]
        assert np.all(np.isfinite(got))
        assert_close(got, ref, TOL_TC if path == "gemm_tc" else TOL_GEMV, rows=parts["gap"] >= GAP)


@pytest.mark.parametrize("T", [1, 4, 64])
def test_zero_routed_scales_leave_residual_plus_shared(oracle, T):
    arr = inputs.moe_layer(6, H, E, F, shared=True)
    for name in ("Wg", "Wu", "Wd"):
        arr[name][..., 0:4] = 0
    lay = qb.MoeLayer.from_arrays(arr, K)
    X = inputs.hidden(90 + T, T, H)
    R = inputs.residual(9, T, H)
    out = qb.moe_forward(lay, torch.from_numpy(X).cuda(), torch.from_numpy(R).cuda())
    torch.cuda.synchronize()
    ref = oracle.moe_forward(X, arr, K, R)
    assert_close(out.cpu().numpy() - R, ref - R, tol())
    # every expert zero: the output is R itself, bit for bit
    for name in ("Sg", "Su", "Sd"):
        arr[name][..., 0:4] = 0
    lay0 = qb.MoeLayer.from_arrays(arr, K)
    out0 = qb.moe_forward(lay0, torch.from_numpy(X).cuda(), torch.from_numpy(R).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(out0.cpu().numpy(), R)


# ------------------------------------------------------------------ extreme skew

def test_every_row_same_eight_experts(oracle):
    """Router bias making experts 40..47 the top eight of every row: 4096 rows
    each for eight experts (32 token chunks each), 248 experts idle."""
    arr = inputs.moe_layer(7, H, E, F, shared=True)
    bias = np.full(E, -50.0, np.float32)
    bias[40:48] = 50.0 + 10.0 * np.arange(8, dtype=np.float32)  # spaced far beyond the logit noise
    arr["Wr"][0] = bias
    lay = qb.MoeLayer.from_arrays(arr, K)
    T = 4096
    X = inputs.hidden(11, T, H)
    X[:, 0] = 1.0
    ws = lay.workspace(T)
    out = qb.moe_forward(lay, torch.from_numpy(X).cuda(), ws=ws)
    torch.cuda.synchronize()
    assert qb.query_status() == 0 and qb.last_path() == "gemm_tc"
    Lw = lay.workspace_layout(T)
    offs = ws[Lw.offsets:Lw.offsets + 4 * (E + 2)].view(torch.int32).cpu().numpy()
    counts = np.diff(offs[:E + 1])
    assert np.all(counts[40:48] == T) and counts.sum() == T * K
    rows = np.array([0, 1, 2047, 4095])
    ref, parts = oracle.moe_forward_rows(X, arr, K, rows)
    assert np.all(parts["ids"] == np.arange(47, 39, -1))
    assert_close(out.cpu().numpy()[rows], ref, TOL_TC)


def test_every_slot_one_expert_caller_routes(oracle):
    """Caller-supplied routes with all eight slots of all 4096 rows on expert
    13 (weights 1/8): one expert with 32768 rows (256 chunks of 128). The
    expected rows are the oracle's expert function of expert 13 plus the
    shared expert."""
    arr = inputs.moe_layer(8, H, E, F, shared=True)
    lay = qb.MoeLayer.from_arrays(arr, K)
    T = 4096
    X = inputs.hidden(12, T, H)
    ids = torch.full((T, K), 13, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), 1.0 / K, dtype=torch.float32, device="cuda")
    out = qb.moe_forward(lay, torch.from_numpy(X).cuda(), ids=ids, w=w)
    torch.cuda.synchronize()
    assert qb.query_status() == 0
    rows = np.array([0, 777, 4095])
    x = X[rows].astype(np.float64)
    dm = oracle.dequant_matrix
    y13 = oracle.expert_ffn(x, dm(arr["Wg"][13]), dm(arr["Wu"][13]), dm(arr["Wd"][13]))
    ysh = oracle.expert_ffn(x, dm(arr["Sg"]), dm(arr["Su"]), dm(arr["Sd"]))
    assert_close(out.cpu().numpy()[rows], y13 + ysh, tol())


# ------------------------------------------------------------------ permutation

@pytest.mark.parametrize("T,path", [(2, "gemv"), (64, "gemm_tc"), (4096, "gemm_tc")])
def test_permutation_is_stable_sort_of_routes(T, path):
    """offsets = exclusive scan of the per-expert counts (the shared expert's
    T rows last) and perm = the pairs t*k+s stably sorted by expert, then the
    shared pairs T*k+t, exactly."""
    arr = inputs.moe_layer(1, H, E, F, shared=True, routing="zipf")
    lay = qb.MoeLayer.from_arrays(arr, K)
    X = inputs.hidden(13 + T, T, H, "zipf")
    ws = lay.workspace(T)
    if path == "gemv":
        qb.set_decode_max_rows(0)
    try:
        qb.moe_forward(lay, torch.from_numpy(X).cuda(), ws=ws)
        assert qb.last_path() == path
    finally:
        qb.set_decode_max_rows(-1)
    torch.cuda.synchronize()
    L = lay.workspace_layout(T)
    ids = ws[L.ids:L.ids + 4 * T * K].view(torch.int32).cpu().numpy()
    offs = ws[L.offsets:L.offsets + 4 * (E + 2)].view(torch.int32).cpu().numpy()
    perm = ws[L.perm:L.perm + 4 * (T * K + T)].view(torch.int32).cpu().numpy()
    counts = np.bincount(ids, minlength=E)
    exp_offs = np.concatenate([[0], np.cumsum(counts), [T * K + T]])
    assert np.array_equal(offs, exp_offs)
    exp_perm = np.concatenate([np.argsort(ids, kind="stable"), T * K + np.arange(T)])
    assert np.array_equal(perm, exp_perm)
