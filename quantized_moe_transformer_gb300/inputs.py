"""Seeded synthetic inputs for the k-quant routed-MoE layer and its block.

This module draws random numbers and lays them out in the packed formats; it
holds none of the layer's arithmetic (no dequantisation, no routing, no
products). Both the CUDA path's tests and the fp64 oracle's tests take their
inputs from here, so it depends on numpy alone.

Packed formats (the pages name Q4_K and Q5_K but print no byte layout; this is
the layout the library defines, stated in ``include/qmoe.h``):

* Q4_K super-block, 144 bytes, 256 weights in 8 sub-blocks of 32:
  bytes 0-1 ``d`` (fp16), bytes 2-3 ``dmin`` (fp16), bytes 4-15 sixteen 6-bit
  fields packed little-endian (fields 0-7 are the scales ``s_j``, fields 8-15
  the mins ``m_j``), bytes 16-143 the 4-bit quants (byte ``b`` holds weight
  ``2b`` in its low nibble and weight ``2b+1`` in its high nibble).
* Q5_K super-block, 176 bytes: the same 16-byte header, then 32 bytes holding
  one high bit per weight (weight ``i`` is bit ``i % 8`` of byte ``i // 8``),
  then the 128 bytes of low nibbles laid out as in Q4_K.

Because every 6-bit field, nibble and high bit is drawn uniformly, the scale,
quant and high-bit bytes are plain uniform random bytes; only ``d`` and
``dmin`` are drawn from a range, U[2^-12, 2^-10] rounded to fp16, which keeps
them normal numbers.

Routing skew follows the temperature-scaled reading of the Zipf s=1.1 workload:
hidden column 0 is set to 1 and router row 0 holds the bias
``-s * ln(1 + rank(e))`` for a seeded ranking of the experts, so that the
routing prior over experts is proportional to ``(1 + rank)^-s``.
"""

from __future__ import annotations

import numpy as np

Q4K_BYTES = 144
Q5K_BYTES = 176
QK = 256  # weights per super-block
QTYPE_BYTES = {"q4k": Q4K_BYTES, "q5k": Q5K_BYTES, "q6k": 210, "mxfp4": 136}

# distinct streams per tensor so that changing one shape leaves the others alone
_STREAM = {
    "X": 1, "Wr": 2, "Wg": 3, "Wu": 4, "Wd": 5, "Sg": 6, "Su": 7, "Sd": 8,
    "zipf": 9, "R": 10, "g1": 11, "g2": 12, "Wq": 13, "Wk": 14, "Wv": 15,
    "Wo": 16, "kc": 17, "vc": 18,
}


def generator(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), _STREAM[name]]))


def packed_blocks(rng: np.random.Generator, shape: tuple, qtype: str) -> np.ndarray:
    """Uniform random super-blocks of ``qtype`` with ``shape`` = (..., n_blocks).

    Returns uint8 with a trailing byte axis of 144 (q4k), 176 (q5k), 210 (q6k)
    or 136 (mxfp4). Every byte is uniform except the scales: fp16 d and dmin in
    [2^-12, 2^-10] (q4k, q5k), fp16 d in [2^-14, 2^-12] (q6k, whose signed
    8-bit scales and centred 6-bit quants span about 64 times the range of a
    Q4_K field pair), E8M0 exponents 119..124 (mxfp4: block scales 2^-8..2^-3);
    all four then give weights of similar size."""
    nb = QTYPE_BYTES[qtype]
    count = int(np.prod(shape, dtype=np.int64))
    raw = np.frombuffer(rng.bytes(count * nb), dtype=np.uint8).copy()
    raw = raw.reshape(count, nb)
    if qtype in ("q4k", "q5k"):
        scales = rng.uniform(2.0**-12, 2.0**-10, size=(count, 2)).astype(np.float16)
        raw[:, 0:4] = scales.view(np.uint8).reshape(count, 4)
    elif qtype == "q6k":
        d = rng.uniform(2.0**-14, 2.0**-12, size=(count, 1)).astype(np.float16)
        raw[:, 0:2] = d.view(np.uint8).reshape(count, 2)
    else:
        raw[:, 0:8] = rng.integers(119, 125, size=(count, 8), dtype=np.uint8)
    return raw.reshape(*shape, nb)


def moe_layer(seed: int, H: int, E: int, F: int, shared: bool = True,
              gate_type: str = "q4k", down_type: str = "q5k",
              routing: str = "uniform", zipf_s: float = 1.1) -> dict:
    """Weights of one routed-MoE layer.

    Wr [H, E] fp32 ~ N(0, 0.02); Wg, Wu [E, F, H/256] super-blocks (rows are
    output features, blocks run along the input axis H); Wd [E, H, F/256].
    The shared expert (``Sg``, ``Su``, ``Sd``) has the same per-expert shapes.
    """
    assert H % QK == 0 and F % QK == 0
    Wr = generator(seed, "Wr").normal(0.0, 0.02, size=(H, E)).astype(np.float32)
    if routing == "zipf":
        rank = generator(seed, "zipf").permutation(E)
        Wr[0, :] = (-zipf_s * np.log1p(rank.astype(np.float64))).astype(np.float32)
    elif routing != "uniform":
        raise ValueError(routing)
    out = {
        "H": H, "E": E, "F": F, "gate_type": gate_type, "down_type": down_type,
        "routing": routing, "Wr": Wr,
        "Wg": packed_blocks(generator(seed, "Wg"), (E, F, H // QK), gate_type),
        "Wu": packed_blocks(generator(seed, "Wu"), (E, F, H // QK), gate_type),
        "Wd": packed_blocks(generator(seed, "Wd"), (E, H, F // QK), down_type),
    }
    if shared:
        out["Sg"] = packed_blocks(generator(seed, "Sg"), (F, H // QK), gate_type)
        out["Su"] = packed_blocks(generator(seed, "Su"), (F, H // QK), gate_type)
        out["Sd"] = packed_blocks(generator(seed, "Sd"), (H, F // QK), down_type)
    return out


def hidden(seed: int, T: int, H: int, routing: str = "uniform") -> np.ndarray:
    """Hidden rows X [T, H] fp32 ~ N(0, 1); column 0 is 1 under Zipf routing."""
    X = generator(seed, "X").normal(0.0, 1.0, size=(T, H)).astype(np.float32)
    if routing == "zipf":
        X[:, 0] = 1.0
    return X


def residual(seed: int, T: int, H: int) -> np.ndarray:
    return generator(seed, "R").normal(0.0, 1.0, size=(T, H)).astype(np.float32)


def bf16_from_f32_bits(a: np.ndarray) -> np.ndarray:
    """Keep the top 16 bits of each fp32 draw: a uint16 array of bf16 bit
    patterns. The values are still seeded random draws (truncated, which is
    part of the draw, not a rounding step of the method)."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return (bits >> 16).astype(np.uint16)


def block(seed: int, H: int = 2048, n_heads: int = 16, n_kv: int = 2,
          head_dim: int = 128, ctx: int = 4096, F: int = 512, E: int = 256,
          routing: str = "uniform") -> dict:
    """Weights of one attention + MoE block and a seeded KV cache.

    RMSNorm gains are 1 + N(0, 0.1). Wq [n_heads*head_dim, H/256], Wk and Wv
    [n_kv*head_dim, H/256], Wo [H, n_heads*head_dim/256], all Q4_K. The cache
    holds ``ctx`` positions of ``n_kv`` heads of ``head_dim`` bf16 values drawn
    from N(0, 1) (as uint16 bit patterns); positions a run writes overwrite it.
    """
    q_out, kv_out = n_heads * head_dim, n_kv * head_dim
    out = {
        "H": H, "n_heads": n_heads, "n_kv": n_kv, "head_dim": head_dim, "ctx": ctx,
        "g1": (1.0 + generator(seed, "g1").normal(0.0, 0.1, size=H)).astype(np.float32),
        "g2": (1.0 + generator(seed, "g2").normal(0.0, 0.1, size=H)).astype(np.float32),
        "Wq": packed_blocks(generator(seed, "Wq"), (q_out, H // QK), "q4k"),
        "Wk": packed_blocks(generator(seed, "Wk"), (kv_out, H // QK), "q4k"),
        "Wv": packed_blocks(generator(seed, "Wv"), (kv_out, H // QK), "q4k"),
        "Wo": packed_blocks(generator(seed, "Wo"), (H, q_out // QK), "q4k"),
        "k_cache": bf16_from_f32_bits(
            generator(seed, "kc").normal(0.0, 1.0, size=(ctx, n_kv, head_dim))),
        "v_cache": bf16_from_f32_bits(
            generator(seed, "vc").normal(0.0, 1.0, size=(ctx, n_kv, head_dim))),
        "moe": moe_layer(seed, H, E, F, shared=True, routing=routing),
    }
    return out
