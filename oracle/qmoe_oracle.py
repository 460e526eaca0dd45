"""fp64 CPU oracle for the k-quant routed-MoE layer and its transformer block.

TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the bench's
CPU-baseline leg may import this module. The library's CUDA path never calls
it, and this module imports nothing from the library.

It is the plain, slow definition of what the path computes, written from these
pages:

* [CKE-Zip] "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights"
  (shivasnotes.com): the routed-MoE layer of Qwen3.5-35B-A3B with Q4_K gate/up
  and Q5_K down weights, 256 experts, top-8, a shared expert, SwiGLU branches
  (sections "What The First Prototype Split" and "What PR #382 Now Splits"),
  the block recombination order (same section), and the slot-order merge of the
  eight routes ("A Separate Decode Result Shows Why Axis Choice Matters").
* [CKE-Dist] "Distributed CPU: Zip Fusion Beyond Tensor Parallelism"
  (c-kernel-engine.github.io): the column-split reduction algebra (section "What
  Must Cross the Fabric: The Reduction Algebra"), the fixed reduction order
  ("Streaming reductions: keep the pipeline moving"), GQA head grouping ("The
  Zip Schedule", GQA note) and the exact online-softmax merge ("Two-Dimensional
  Attention at Long Context").

Every value is widened to float64 before any arithmetic (fp32 hidden rows and
router weights, fp16 d/dmin, bf16 cache entries), and every step is done in
float64 in the order the pages give. The pages print no byte layout for Q4_K or
Q5_K, no routing formula, no RMSNorm epsilon and no RoPE variant; the readings
taken here are:

* Q4_K super-block (144 B): fp16 d, fp16 dmin, sixteen 6-bit fields packed
  little-endian (s_0..s_7 then m_0..m_7), 128 bytes of nibbles (byte b: weight
  2b low nibble, 2b+1 high nibble). Q5_K (176 B): the same header, 32 bytes of
  high bits (bit i = weight i), then the nibbles. Weight i of sub-block
  j = i // 32 is d*s_j*q_i - dmin*m_j with q_i = nibble (+16*high bit for Q5_K).
* Q6_K super-block (210 B; no GPU kernel takes it yet): fp16 d, sixteen signed
  8-bit scales (16 weights each), 64 bytes of 2-bit high parts, 128 bytes of
  low nibbles; w_i = d*s_{i//16}*(q_i - 32), q_i = nibble + 16*high part.
* MXFP4 super-block (136 B; no GPU kernel yet): eight E8M0 scales for the
  32-weight blocks, 128 bytes of FP4 E2M1 codes; w_i = 2^(e - 127) * E2M1.
* Routing: logits l = x Wr; the k experts with the largest logits (ties to the
  lower index), in descending-logit slot order, with weights softmax over the
  whole row renormalised over the selected k, which equals
  exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0).
* SwiGLU h = silu(g) * u with silu(z) = z / (1 + exp(-z)); the shared expert is
  added with weight 1, without a gate.
* Combine: out = R + y_shared + sum over slots s = 0..k-1 of w_s y_s, in slot
  order.
* Block: RMSNorm x / sqrt(mean(x^2) + eps) * gamma with eps = 1e-6; rotate-half
  RoPE pairing (i, i + d/2) with inverse frequency theta^(-2i/d); keys and
  values rounded to bf16 (nearest, ties to even) when written to the cache;
  scores scaled by 1/sqrt(d); query head h reads KV head h // (n_heads/n_kv);
  no biases; no QK-norm.
"""

from __future__ import annotations

import math

import numpy as np

QK = 256
SUB = 32
Q4K_BYTES = 144
Q5K_BYTES = 176
Q6K_BYTES = 210
MXFP4_BYTES = 136


# --------------------------------------------------------------------------
# k-quant dequantisation  ([CKE-Zip] "What PR #382 Now Splits": Q4_K gate and
# up, Q5_K down; [CKE-Dist] "Prior Art, Candidly": packed-weight unpack and
# scale decode are part of each lane's local work)
# --------------------------------------------------------------------------

def _header(blocks: np.ndarray):
    """d, dmin (float64) and the sixteen 6-bit fields of each super-block."""
    hdr = np.ascontiguousarray(blocks[..., 0:4])
    d = hdr.view(np.float16)[..., 0].astype(np.float64)
    dmin = hdr.view(np.float16)[..., 1].astype(np.float64)
    # bytes 4..15 form one little-endian bit stream; field f is bits 6f..6f+5
    bits = np.unpackbits(blocks[..., 4:16], axis=-1, bitorder="little")
    fields = bits.reshape(*bits.shape[:-1], 16, 6)
    place = np.array([1, 2, 4, 8, 16, 32], dtype=np.int64)
    vals = (fields.astype(np.int64) * place).sum(axis=-1)
    return d, dmin, vals[..., 0:8], vals[..., 8:16]


def _nibbles(qs: np.ndarray) -> np.ndarray:
    """128 quant bytes -> 256 values; weight 2b is the low nibble of byte b."""
    lo = (qs & 0x0F).astype(np.int64)
    hi = (qs >> 4).astype(np.int64)
    return np.stack([lo, hi], axis=-1).reshape(*qs.shape[:-1], 256)


def _apply_scales(q: np.ndarray, d, dmin, s, m) -> np.ndarray:
    j = np.arange(QK) // SUB                       # sub-block of each weight
    scale = d[..., None] * s[..., j].astype(np.float64)
    offset = dmin[..., None] * m[..., j].astype(np.float64)
    return scale * q.astype(np.float64) - offset


def dequant_q4k(blocks: np.ndarray) -> np.ndarray:
    """[..., 144] uint8 -> [..., 256] float64."""
    assert blocks.shape[-1] == Q4K_BYTES and blocks.dtype == np.uint8
    d, dmin, s, m = _header(blocks)
    q = _nibbles(blocks[..., 16:144])
    return _apply_scales(q, d, dmin, s, m)


def dequant_q5k(blocks: np.ndarray) -> np.ndarray:
    """[..., 176] uint8 -> [..., 256] float64; q = nibble + 16 * high bit."""
    assert blocks.shape[-1] == Q5K_BYTES and blocks.dtype == np.uint8
    d, dmin, s, m = _header(blocks)
    high = np.unpackbits(blocks[..., 16:48], axis=-1, bitorder="little").astype(np.int64)
    q = _nibbles(blocks[..., 48:176]) + 16 * high
    return _apply_scales(q, d, dmin, s, m)


def dequant_q6k(blocks: np.ndarray) -> np.ndarray:
    """[..., 210] uint8 -> [..., 256] float64.

    Q6_K, the format a Q4_K_M model file ([CKE-Zip], opening paragraphs: "a
    real Qwen3.5-35B-A3B Q4_K_M prefill") keeps some of its tensors in. The
    pages print no layout; the library's own reading: fp16 d, sixteen signed
    8-bit sub-block scales s_0..s_15 (16 weights each), 64 bytes of 2-bit high
    parts (weight i: bits 2(i % 4), 2(i % 4) + 1 of byte i // 4), 128 bytes of
    low nibbles (byte b: weight 2b low, 2b+1 high); q_i = low + 16 * high in
    0..63 and w_i = d * s_{i // 16} * (q_i - 32). No min, no second scale."""
    assert blocks.shape[-1] == Q6K_BYTES and blocks.dtype == np.uint8
    d = np.ascontiguousarray(blocks[..., 0:2]).view(np.float16)[..., 0].astype(np.float64)
    s = np.ascontiguousarray(blocks[..., 2:18]).view(np.int8).astype(np.int64)
    hb = blocks[..., 18:82]
    high = np.stack([(hb >> (2 * r)) & 3 for r in range(4)], axis=-1)
    high = high.reshape(*hb.shape[:-1], QK).astype(np.int64)
    q = _nibbles(blocks[..., 82:210]) + 16 * high
    j = np.arange(QK) // 16                        # sub-block of each weight
    return d[..., None] * s[..., j].astype(np.float64) * (q - 32).astype(np.float64)


# FP4 E2M1 (sign, 2 exponent bits with bias 1, 1 mantissa bit; exponent 0 is
# subnormal): the value of each 4-bit code
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                  -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def dequant_mxfp4(blocks: np.ndarray) -> np.ndarray:
    """[..., 136] uint8 -> [..., 256] float64.

    The MXFP4-class format that "Distributed CPU: Zip Fusion Beyond Tensor
    Parallelism", section "Decode vs Prefill: Same Weights, Different
    Bottlenecks", names for the packed weights of the model class it targets,
    with the element and scale types of the OCP microscaling format (blocks of
    32 FP4 E2M1 values sharing one E8M0 scale), in the library's own
    256-weight super-block: eight E8M0 scales
    (one per 32 weights, value 2^(e - 127), e = 255 is NaN), then 128 bytes of
    FP4 E2M1 codes (byte b: weight 2b low nibble, 2b+1 high);
    w_i = 2^(e_{i//32} - 127) * E2M1(code_i)."""
    assert blocks.shape[-1] == MXFP4_BYTES and blocks.dtype == np.uint8
    e = blocks[..., 0:8].astype(np.int64)
    scale = np.where(e == 255, np.nan, np.ldexp(1.0, e - 127))
    codes = _nibbles(blocks[..., 8:136])
    j = np.arange(QK) // 32
    return scale[..., j] * _E2M1[codes]


def dequant_matrix(W: np.ndarray) -> np.ndarray:
    """Packed [..., rows, n_blocks, bytes] -> dense [..., rows, n_blocks*256].

    Row r of the result is output feature r; its columns run along the input
    axis, which is the axis the super-blocks cover."""
    nb = W.shape[-1]
    dense = {Q4K_BYTES: dequant_q4k, Q5K_BYTES: dequant_q5k, Q6K_BYTES: dequant_q6k,
             MXFP4_BYTES: dequant_mxfp4}[nb](W)
    return dense.reshape(*W.shape[:-2], W.shape[-2] * QK)


# --------------------------------------------------------------------------
# Router ([CKE-Zip] "What The First Prototype Split": the selected top-k expert
# indices and their routing weights; "What PR #382 Now Splits": 256 routed
# experts, eight selected per token, one synchronised router decision)
# --------------------------------------------------------------------------

def route(X: np.ndarray, Wr: np.ndarray, k: int):
    """Returns ids [T,k] int64, w [T,k] float64, gap [T] and logits [T,E].

    gap is the k-th minus the (k+1)-th largest logit (inf when k == E): the
    margin by which the selected set is decided."""
    L = X.astype(np.float64) @ Wr.astype(np.float64)
    T, E = L.shape
    ids = np.empty((T, k), dtype=np.int64)
    w = np.empty((T, k), dtype=np.float64)
    gap = np.full(T, np.inf)
    index = np.arange(E)
    for t in range(T):
        order = np.lexsort((index, -L[t]))         # logit descending, then index
        sel = order[:k]
        ids[t] = sel
        e = np.exp(L[t, sel] - L[t, sel[0]])
        w[t] = e / e.sum()
        if k < E:
            gap[t] = L[t, order[k - 1]] - L[t, order[k]]
    return ids, w, gap, L


# --------------------------------------------------------------------------
# Expert FFN with SwiGLU ([CKE-Zip] "What The First Prototype Split": routed and
# shared SwiGLU branches; "What PR #382 Now Splits": gate, up, SwiGLU, down)
# --------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_ffn(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray,
               f_cols: slice | None = None) -> np.ndarray:
    """x [n,H] float64; dense Wg, Wu [F,H], Wd [H,F] -> y [n,H].

    ``f_cols`` keeps only that slice of the intermediate axis: gate and up rows
    and the matching down columns, i.e. one rank's partial of the F split."""
    if f_cols is not None:
        Wg, Wu, Wd = Wg[f_cols], Wu[f_cols], Wd[:, f_cols]
    g = x @ Wg.T
    u = x @ Wu.T
    h = silu(g) * u
    return h @ Wd.T


def moe_forward(X: np.ndarray, layer: dict, k: int, R: np.ndarray | None = None,
                f_half: int | None = None, return_parts: bool = False):
    """The routed-MoE layer on rows X [T,H]; float64 result [T,H].

    out_t = R_t + y_shared,t + sum_{s=0}^{k-1} w_{t,s} y_{t,s}, summed in slot
    order. ``f_half`` in {0, 1} computes one rank's partial of the 256/256 split
    of every expert's intermediate axis (routed and shared); routing still uses
    the whole row, as the pages' synchronised router does, and R is left out of
    partials."""
    T, H = X.shape
    F = layer["F"]
    x = X.astype(np.float64)
    ids, w, gap, L = route(X, layer["Wr"], k)
    f_cols = None
    if f_half is not None:
        half = F // 2
        f_cols = slice(f_half * half, (f_half + 1) * half)
    # y[t, s] for every (row, slot); each expert is dequantised once and applied
    # to the rows that selected it -- the same per-row products, grouped.
    y = np.zeros((T, k, H))
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        Wg = dequant_matrix(layer["Wg"][e])
        Wu = dequant_matrix(layer["Wu"][e])
        Wd = dequant_matrix(layer["Wd"][e])
        y[rows, slots] = expert_ffn(x[rows], Wg, Wu, Wd, f_cols)
    out = np.zeros((T, H))
    if R is not None and f_half is None:
        out += R.astype(np.float64)
    y_sh = None
    if "Sg" in layer:
        y_sh = expert_ffn(x, dequant_matrix(layer["Sg"]), dequant_matrix(layer["Su"]),
                          dequant_matrix(layer["Sd"]), f_cols)
        out += y_sh
    for s in range(k):
        out += w[:, s:s + 1] * y[:, s, :]
    if return_parts:
        return out, {"ids": ids, "w": w, "gap": gap, "logits": L, "y": y, "y_shared": y_sh}
    return out


def moe_forward_rows(X: np.ndarray, layer: dict, k: int, rows: np.ndarray,
                     R: np.ndarray | None = None):
    """moe_forward restricted to the listed rows (rows are independent through
    the layer: [CKE-Zip] "What The First Prototype Split")."""
    Rs = None if R is None else R[rows]
    return moe_forward(X[rows], layer, k, Rs, return_parts=True)


# --------------------------------------------------------------------------
# Block pieces ([CKE-Zip] "What PR #382 Now Splits": the attention + MoE block,
# 16 query heads and 2 KV heads, recombined as attention partials + residual +
# synchronised router + MoE partials + residual)
# --------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = x.astype(np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gamma.astype(np.float64)


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE on x [T, heads, d] at positions pos [T]."""
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = pos.astype(np.float64)[:, None] * inv_freq[None, :]      # [T, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value of each float64 (ties to even), as float64.

    bf16 keeps 8 significant bits; the float64 value is split as m * 2^e with
    0.5 <= |m| < 1 and m is rounded to a multiple of 2^-8 (numpy's rint rounds
    ties to even), with no intermediate float32 rounding. Values are assumed to
    lie in bf16's normal range, which every value of this path does."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
              q_pos: np.ndarray, kv_head_of: np.ndarray) -> np.ndarray:
    """Causal attention: q [T, nh, d] float64; caches [ctx, nkv, d] float64.

    Query t at position q_pos[t] attends to cache positions 0..q_pos[t]."""
    T, nh, d = q.shape
    out = np.zeros((T, nh, d))
    scale = 1.0 / math.sqrt(d)
    for h in range(nh):
        g = kv_head_of[h]
        K = k_cache[:, g, :]
        V = v_cache[:, g, :]
        S = (q[:, h, :] @ K.T) * scale            # [T, ctx]
        ctx = K.shape[0]
        mask = np.arange(ctx)[None, :] > q_pos[:, None]
        S = np.where(mask, -np.inf, S)
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[:, h, :] = P @ V
    return out


def attention_merge(parts):
    """Exact merge of attention computed over disjoint context shards from each
    shard's (max m, normaliser l, weighted output o), [CKE-Dist] "Two-Dimensional
    Attention at Long Context": each shard's statistics are rescaled to the
    common maximum before summing."""
    M = np.max([m for m, _, _ in parts], axis=0)
    L = sum(l * np.exp(m - M) for m, l, _ in parts)
    O = sum(o * (np.exp(m - M))[..., None] for m, _, o in parts)
    return O / L[..., None]


def attention_shard_stats(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """(m, l, o) of one context shard for queries q [n, d] against K, V [c, d]
    (no mask): m the row max of the scaled scores, l = sum exp(s - m),
    o = sum exp(s - m) v."""
    d = q.shape[-1]
    S = (q @ K.T) / math.sqrt(d)
    m = S.max(axis=1)
    P = np.exp(S - m[:, None])
    return m, P.sum(axis=1), P @ V


def attn_sublayer(X: np.ndarray, blk: dict, pos0: int, k_cache: np.ndarray,
                  v_cache: np.ndarray, theta: float = 1e7, eps: float = 1e-6,
                  rank: int | None = None, n_ranks: int = 2,
                  rows: np.ndarray | None = None) -> np.ndarray:
    """Attention branch of the block without its residual: O(attn(RoPE(QKV(rms(X))))).

    Writes the rows' bf16-rounded keys and values into the float64 caches
    (positions pos0..pos0+T-1). With ``rank`` set, computes that rank's partial:
    query heads [rank*nh/n_ranks, ...), its KV heads, and the matching input
    columns of the O projection ([CKE-Zip] "What PR #382 Now Splits"). With
    ``rows``, keys and values are still computed and cached for every row but
    the output is formed only for those query rows."""
    T, H = X.shape
    nh, nkv, d = blk["n_heads"], blk["n_kv"], blk["head_dim"]
    r = rmsnorm(X, blk["g1"], eps)
    Wq = dequant_matrix(blk["Wq"])
    Wk = dequant_matrix(blk["Wk"])
    Wv = dequant_matrix(blk["Wv"])
    Wo = dequant_matrix(blk["Wo"])
    heads = np.arange(nh)
    kvh = np.arange(nkv)
    if rank is not None:
        heads = heads[rank * nh // n_ranks:(rank + 1) * nh // n_ranks]
        kvh = kvh[rank * nkv // n_ranks:(rank + 1) * nkv // n_ranks]
    group = nh // nkv
    if rows is None:
        rows = np.arange(T)
    q = (r[rows] @ Wq.T).reshape(len(rows), nh, d)[:, heads]
    kk = (r @ Wk.T).reshape(T, nkv, d)[:, kvh]
    vv = (r @ Wv.T).reshape(T, nkv, d)[:, kvh]
    pos = pos0 + np.arange(T)
    q = rope(q, pos[rows], theta)
    kk = rope(kk, pos, theta)
    k_cache[pos0:pos0 + T, kvh] = round_bf16(kk)
    v_cache[pos0:pos0 + T, kvh] = round_bf16(vv)
    # local KV head index for each local query head
    kv_local = np.array([list(kvh).index(h // group) for h in heads])
    o = attention(q, k_cache[:pos0 + T, kvh], v_cache[:pos0 + T, kvh], pos[rows], kv_local)
    cols = np.concatenate([np.arange(h * d, (h + 1) * d) for h in heads])
    return o.reshape(len(rows), len(heads) * d) @ Wo[:, cols].T


def block_forward(X: np.ndarray, blk: dict, k: int, pos0: int, k_cache: np.ndarray,
                  v_cache: np.ndarray, theta: float = 1e7, eps: float = 1e-6,
                  split: bool = False):
    """One block: h1 = X + attn(X); out = h1 + moe(rms(h1)).

    With ``split`` the attention and MoE branches are each computed as two rank
    partials and summed, in the recombination order of [CKE-Zip] "What PR #382
    Now Splits": attention partial 0 + partial 1, + residual, routing on the
    whole state, MoE partial 0 + partial 1, + residual. Returns (out, parts)."""
    x = X.astype(np.float64)
    if split:
        a_parts = [attn_sublayer(X, blk, pos0, k_cache, v_cache, theta, eps, rank=r)
                   for r in range(2)]
        h1 = x + (a_parts[0] + a_parts[1])
    else:
        a_parts = [attn_sublayer(X, blk, pos0, k_cache, v_cache, theta, eps)]
        h1 = x + a_parts[0]
    r2 = rmsnorm(h1, blk["g2"], eps)
    if split:
        m_parts = [moe_forward(r2, blk["moe"], k, f_half=r) for r in range(2)]
        out = h1 + (m_parts[0] + m_parts[1])
    else:
        m_parts = [moe_forward(r2, blk["moe"], k)]
        out = h1 + m_parts[0]
    return out, {"attn": a_parts, "moe": m_parts, "h1": h1}


def block_forward_rows(X: np.ndarray, blk: dict, k: int, pos0: int, k_cache: np.ndarray,
                       v_cache: np.ndarray, rows: np.ndarray, theta: float = 1e7,
                       eps: float = 1e-6):
    """block_forward for the listed query rows only (every row's keys and values
    still enter the cache; given the cache, rows are independent). Returns
    (out[rows], moe parts of those rows incl. the routing gap)."""
    a = attn_sublayer(X, blk, pos0, k_cache, v_cache, theta, eps, rows=rows)
    h1 = X[rows].astype(np.float64) + a
    r2 = rmsnorm(h1, blk["g2"], eps)
    m, parts = moe_forward(r2, blk["moe"], k, return_parts=True)
    return h1 + m, parts
