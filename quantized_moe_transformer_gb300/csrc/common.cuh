// Shared device helpers for the k-quant MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmoe.h"

namespace qmoe {

constexpr int QK = 256;          // weights per super-block
constexpr int SUBK = 32;         // weights per sub-block
constexpr int Q4K_BYTES = 144;
constexpr int Q5K_BYTES = 176;

constexpr int Q6K_BYTES = 210;
constexpr int MXFP4_BYTES = 136;

// Bytes of one 256-weight super-block of format ``qt``.
__host__ __device__ constexpr int qtype_size(int qt) {
  return qt == QMOE_Q5K ? Q5K_BYTES : qt == QMOE_Q6K ? Q6K_BYTES : qt == QMOE_MXFP4 ? MXFP4_BYTES : Q4K_BYTES;
}
__host__ __device__ inline int qtype_bytes(int qt) { return qtype_size(qt); }

// One super-block header: d, dmin and the sixteen 6-bit fields. The header is
// the first 16 bytes of both formats, loaded as one 16-byte vector.
struct KHeader {
  float d, dmin;
  uint32_t f0, f1, f2;  // bytes 4..15 as three little-endian words
};

__device__ __forceinline__ KHeader load_header(const uint8_t* blk) {
  uint4 v = __ldg(reinterpret_cast<const uint4*>(blk));
  KHeader h;
  __half2 dd = *reinterpret_cast<const __half2*>(&v.x);
  float2 f = __half22float2(dd);
  h.d = f.x;
  h.dmin = f.y;
  h.f0 = v.y;
  h.f1 = v.z;
  h.f2 = v.w;
  return h;
}

// 6-bit field f (0..15) of the 96-bit little-endian field stream.
__device__ __forceinline__ uint32_t field6(const KHeader& h, int f) {
  const int p = 6 * f;
  const uint32_t lo = p < 32 ? h.f0 : (p < 64 ? h.f1 : h.f2);
  const uint32_t hi = p < 32 ? h.f1 : (p < 64 ? h.f2 : 0u);
  return __funnelshift_r(lo, hi, p & 31) & 63u;
}

// Sub-block j's effective scale d*s_j and offset dmin*m_j.
__device__ __forceinline__ float2 sub_scale(const KHeader& h, int j) {
  return make_float2(h.d * (float)field6(h, j), h.dmin * (float)field6(h, 8 + j));
}

// Byte offset of sub-block j's 16 quant bytes inside a super-block.
__host__ __device__ constexpr int quant_offset(int qt, int j) {
  return (qt == QMOE_Q5K ? 48 : 16) + 16 * j;
}

// Sum over the 32 weights of one sub-block of q_i * x_i, where the quants are
// the 16 bytes ``qv`` (weight 2b low nibble, 2b+1 high nibble of byte b) plus,
// for Q5_K, 16 times bit i of ``hb``.
template <int QT>
__device__ __forceinline__ float dot_sub(const uint4 qv, uint32_t hb, const float* x) {
  const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
  float acc = 0.f;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int i = 8 * n + b;  // weight index within the sub-block
      uint32_t q = (w[n] >> (4 * b)) & 15u;
      if (QT == QMOE_Q5K) q |= ((hb >> i) & 1u) << 4;
      acc = fmaf((float)q, x[i], acc);
    }
  }
  return acc;
}

// Spreads four bits of ``h`` (bits b, b+2, b+4, b+6) to bit 4 of bytes 0..3.
// One multiply places bit 2i at 6i + 2i + 4 = 8i + 4; the other partial
// products land on positions the mask clears, and none of them carry into a
// kept position.
__device__ __forceinline__ uint32_t spread4(uint32_t h, int b) {
  return (((h >> b) & 0x55u) * 0x410410u) & 0x10101010u;
}

// S = sum over the 32 weights of one sub-block of (0.5 + q_i/256) * x_i.
// Each quant byte (0..31) is placed by one byte permute into the mantissa of
// a float whose exponent makes it 0.5 + q/256 exactly, so the unpacking costs
// one integer instruction per weight and no int->float conversion. The caller
// recovers sum q_i x_i = 256 * (S - 0.5 * sum x_i).
template <int QT>
__device__ __forceinline__ float dot_sub_prmt(const uint4 qv, uint32_t hb, const float* x) {
  const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    uint32_t ev = w[n] & 0x0F0F0F0Fu;          // weights 8n + 2k
    uint32_t od = (w[n] >> 4) & 0x0F0F0F0Fu;   // weights 8n + 2k + 1
    if (QT == QMOE_Q5K) {
      ev |= spread4(hb >> (8 * n), 0);
      od |= spread4(hb >> (8 * n), 1);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t sel = 0x7044u | ((uint32_t)k << 8);
      acc0 = fmaf(__uint_as_float(__byte_perm(ev, 0x3F000000u, sel)), x[8 * n + 2 * k], acc0);
      acc1 = fmaf(__uint_as_float(__byte_perm(od, 0x3F000000u, sel)), x[8 * n + 2 * k + 1], acc1);
    }
  }
  return acc0 + acc1;
}

// Two-lane fp32 arithmetic on register pairs (lo, hi): fma.rn.f32x2 rounds
// each lane exactly as fmaf does.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}

__device__ __forceinline__ float2 unpack2(uint64_t v) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

// Contribution of one sub-block: d*s_j * sum q x - dmin*m_j * sum x, from the
// byte-permute sum S of dot_sub_prmt and xs = sum x.
__device__ __forceinline__ float sub_contrib(float S, float xs, float2 sc) {
  return fmaf(256.f * sc.x, S, -(128.f * sc.x + sc.y) * xs);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.f + __expf(-g)) * u;
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace qmoe
