// Grouped dequant-fused GEMV kernels (small T) and the slot-order combine.
//
// "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "What PR #382
// Now Splits": each selected expert runs gate, up, SwiGLU and down on the
// row's hidden state, gate/up weights in Q4_K and down weights in Q5_K.
// "Distributed CPU: Zip Fusion Beyond Tensor Parallelism", "Decode vs Prefill":
// at one row every packed weight byte is read once and used once, so these
// kernels are bound by HBM bandwidth; the packed bytes are unpacked in
// registers straight from 16-byte loads and never written back dequantised.
//
// Formats: Q4_K and Q5_K (the layer's own), and Q6_K and MXFP4 (the other
// formats a Q4_K_M model file and the MXFP4-class models carry); see
// include/qmoe.h for their byte layouts.
//
// Work layout: CTA (a, tile) takes active expert a and a tile of output rows;
// each warp owns RW rows; within a row, G lanes split the row's sub-blocks
// (lane l takes sub-blocks l % G, l % G + G, ...). Each lane keeps the packed
// bytes of all its (row, sub-block) items in registers, then walks the rows
// that selected the expert. Per sub-block it forms
//   d*s_j * sum_i q_i x_i  -  dmin*m_j * sum_i x_i
// and the G lanes of a row are reduced with shuffles.
#include "kernels.cuh"

namespace qmoe {

template <int NSUB>
struct LaneMap {
  static constexpr int G = NSUB < 32 ? NSUB : 32;  // lanes per row
  static constexpr int RPP = 32 / G;               // rows per pass of a warp
  static constexpr int SL = NSUB / G;              // sub-block slots per lane
};

// One sub-block (32 weights) of a packed row, as a lane keeps it in
// registers: ``q`` its 16 quant (or code) bytes, ``hb`` the Q5_K high bits or
// the Q6_K 2-bit high parts (64 bits in hb, hb2), ``sc`` its scales: Q4_K /
// Q5_K (d s_j, dmin m_j); Q6_K (d s of weights 0-15, d s of weights 16-31);
// MXFP4 (2^(e - 127) / 2, unused).
template <int QT>
struct PackedSub {
  uint4 q;
  uint32_t hb, hb2;
  float2 sc;
};

// The 16 bytes at ``p`` as four little-endian 32-bit words, where ``p`` is
// only 2-byte aligned (Q6_K super-blocks are 210 bytes long): loads of the
// alignment each piece has, none of them outside [p, p + 16).
__device__ __forceinline__ uint4 ldg16_align2(const uint8_t* p) {
  if ((reinterpret_cast<uintptr_t>(p) & 3) == 0) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
    return make_uint4(__ldg(w), __ldg(w + 1), __ldg(w + 2), __ldg(w + 3));
  }
  // p = 2 mod 4: a 16-bit piece, three aligned words, a 16-bit piece
  const uint32_t h0 = __ldg(reinterpret_cast<const unsigned short*>(p));
  const uint32_t* w = reinterpret_cast<const uint32_t*>(p + 2);
  const uint32_t a = __ldg(w), b = __ldg(w + 1), c = __ldg(w + 2);
  const uint32_t h1 = __ldg(reinterpret_cast<const unsigned short*>(p + 14));
  return make_uint4(h0 | (a << 16), (a >> 16) | (b << 16), (b >> 16) | (c << 16), (c >> 16) | (h1 << 16));
}

__device__ __forceinline__ uint32_t ldg4_align2(const uint8_t* p) {
  const uint16_t* h = reinterpret_cast<const uint16_t*>(p);
  return (uint32_t)__ldg(h) | ((uint32_t)__ldg(h + 1) << 16);
}

template <int QT>
__device__ __forceinline__ PackedSub<QT> load_sub(const uint8_t* row, int c) {
  constexpr int BYTES = qtype_size(QT);
  const uint8_t* blk = row + (size_t)(c >> 3) * BYTES;
  const int j = c & 7;
  PackedSub<QT> p;
  p.hb = p.hb2 = 0u;
  if (QT == QMOE_Q6K) {
    // d at 0, int8 scales s_0..s_15 at 2, 2-bit high parts at 18 (8 bytes a
    // sub-block), low nibbles at 82 (16 bytes a sub-block)
    const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(blk))));
    const uint32_t s2 = (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(blk + 2 + 2 * j));
    p.sc = make_float2(d * (float)(int8_t)(s2 & 0xFFu), d * (float)(int8_t)(s2 >> 8));
    p.q = ldg16_align2(blk + 82 + 16 * j);
    p.hb = ldg4_align2(blk + 18 + 8 * j);
    p.hb2 = ldg4_align2(blk + 22 + 8 * j);
  } else if (QT == QMOE_MXFP4) {
    // E8M0 scales at 0 (one byte a sub-block), E2M1 codes at 8
    const uint32_t e = blk[j];
    p.sc = make_float2(e == 255u ? __int_as_float(0x7fc00000) : ldexpf(0.5f, (int)e - 127), 0.f);
    // 136-byte super-blocks: the codes are 8-byte aligned
    const uint2 lo = __ldg(reinterpret_cast<const uint2*>(blk + 8 + 16 * j));
    const uint2 hi = __ldg(reinterpret_cast<const uint2*>(blk + 16 + 16 * j));
    p.q = make_uint4(lo.x, lo.y, hi.x, hi.y);
  } else {
    KHeader h = load_header(blk);
    p.sc = sub_scale(h, j);
    p.q = __ldg(reinterpret_cast<const uint4*>(blk + quant_offset(QT, j)));
    p.hb = (QT == QMOE_Q5K) ? __ldg(reinterpret_cast<const uint32_t*>(blk + 16 + 4 * j)) : 0u;
  }
  return p;
}

// Spreads the four 2-bit fields of h at bits 0, 4, 8, 12 to bits 4-5 of
// bytes 0..3 (16 times the field in each byte).
__device__ __forceinline__ uint32_t spread2x4(uint32_t h) {
  uint32_t x = h & 0x3333u;
  x = (x | (x << 8)) & 0x00FF00FFu;
  x = (x | (x << 4)) & 0x0F0F0F0Fu;
  return x << 4;
}

// Q6_K: sum over the sub-block of (q_i - 32) x_i with q_i = nibble + 16 high,
// each half (16 weights) with its own scale: 32-bit word n of the nibbles holds
// weights 8n..8n+7 (byte b: 8n+2b low, 8n+2b+1 high); weight i's high part is
// bits 2(i % 4) of byte i / 4 of the high bytes (hb: bytes 0-3, hb2: 4-7).
// Each quant becomes 0.5 + q/256 by one byte permute (exact, q < 64), so
// sum (q - 32) x = 256 S - 160 sum x.
__device__ __forceinline__ float dot_sub_q6k(const PackedSub<QMOE_Q6K>& p, const float* x) {
  const uint32_t w[4] = {p.q.x, p.q.y, p.q.z, p.q.w};
  float S[2] = {0.f, 0.f}, xs[2] = {0.f, 0.f};
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const uint32_t h16 = ((n < 2 ? p.hb : p.hb2) >> (16 * (n & 1))) & 0xFFFFu;  // weights 8n..8n+7
    const uint32_t ev = (w[n] & 0x0F0F0F0Fu) | spread2x4(h16);
    const uint32_t od = ((w[n] >> 4) & 0x0F0F0F0Fu) | spread2x4(h16 >> 2);
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t sel = 0x7044u | ((uint32_t)b << 8);
      a0 = fmaf(__uint_as_float(__byte_perm(ev, 0x3F000000u, sel)), x[8 * n + 2 * b], a0);
      a1 = fmaf(__uint_as_float(__byte_perm(od, 0x3F000000u, sel)), x[8 * n + 2 * b + 1], a1);
    }
    S[n >> 1] += a0 + a1;
#pragma unroll
    for (int i = 0; i < 8; ++i) xs[n >> 1] += x[8 * n + i];
  }
  return p.sc.x * fmaf(256.f, S[0], -160.f * xs[0]) + p.sc.y * fmaf(256.f, S[1], -160.f * xs[1]);
}

// MXFP4: 2^(e-127) sum E2M1(code_i) x_i. Code = sign bit 3, then 2 exponent
// bits and 1 mantissa bit: the magnitude doubled is one of 0 1 2 3 4 6 8 12,
// taken by a byte permute of that table, made a float by the 2^23 magic
// number, and given the code's sign by one XOR.
__device__ __forceinline__ float dot_sub_mxfp4(const PackedSub<QMOE_MXFP4>& p, const float* x) {
  const uint32_t w[4] = {p.q.x, p.q.y, p.q.z, p.q.w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t c = (w[n] >> (4 * i)) & 0xFu;
      const uint32_t mag2 = __byte_perm(0x03020100u, 0x0C080604u, c & 7u) & 0xFFu;
      const float v = __uint_as_float((__float_as_uint(__uint_as_float(0x4B000000u | mag2) - 8388608.f)) ^ ((c & 8u) << 28));
      if (i & 1) a1 = fmaf(v, x[8 * n + i], a1);
      else a0 = fmaf(v, x[8 * n + i], a0);
    }
  }
  return p.sc.x * (a0 + a1);
}

// d-scaled dot of one sub-block with 32 activations (xs = their sum).
template <int QT>
__device__ __forceinline__ float sub_dot(const PackedSub<QT>& p, const float* x, float xs) {
  if constexpr (QT == QMOE_Q6K) {
    return dot_sub_q6k(p, x);
  } else if constexpr (QT == QMOE_MXFP4) {
    return dot_sub_mxfp4(p, x);
  } else {
    return sub_contrib(dot_sub_prmt<QT>(p.q, p.hb, x), xs, p.sc);
  }
}

// Hides the packed registers' values from the optimiser at the top of each
// row iteration, so the unpacking stays inside the loop instead of being
// hoisted out as 32 live floats per sub-block.
template <int QT>
__device__ __forceinline__ void opaque(PackedSub<QT>& p) {
  asm volatile("" : "+r"(p.q.x), "+r"(p.q.y), "+r"(p.q.z), "+r"(p.q.w), "+r"(p.hb), "+r"(p.hb2));
}

__device__ __forceinline__ void load_x32(const float* x, float* v, float& sum) {
  const float4* p = reinterpret_cast<const float4*>(x);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 a = __ldg(p + i);
    v[4 * i] = a.x;
    v[4 * i + 1] = a.y;
    v[4 * i + 2] = a.z;
    v[4 * i + 3] = a.w;
    s += (a.x + a.y) + (a.z + a.w);
  }
  sum = s;
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ int pair_row(int p, int T, int k) { return p < T * k ? p / k : p - T * k; }

// ---------------------------------------------------------------------------
// gate/up + SwiGLU: h[pos][f] = silu(x_t . Wg_e[f]) * (x_t . Wu_e[f])
// for every perm position pos of expert e (row t of pair perm[pos]).
// ---------------------------------------------------------------------------
template <int NSUB, int QT, int RW>
__global__ void __launch_bounds__(256) gateup_gemv_kernel(GroupedArgs g, const uint8_t* __restrict__ Wu,
                                                          const uint8_t* __restrict__ Su,
                                                          const float* __restrict__ X, int F,
                                                          float* __restrict__ hbuf,
                                                          int tiles_per_expert) {
  using M = LaneMap<NSUB>;
  constexpr int PASSES = RW / M::RPP;
  constexpr int BYTES = qtype_size(QT);
  constexpr int H = NSUB * SUBK;
  const int a = blockIdx.x / tiles_per_expert, tile = blockIdx.x % tiles_per_expert;
  if (a >= g.n_active[0]) return;
  const int e = g.active[a];
  const size_t row_bytes = (size_t)(NSUB / 8) * BYTES;
  const uint8_t* gw = (e < g.E) ? g.W + (size_t)e * F * row_bytes : g.S;
  const uint8_t* uw = (e < g.E) ? Wu + (size_t)e * F * row_bytes : Su;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub_lane = lane % M::G, row_in_pass = lane / M::G;
  const int f_warp = tile * (8 * RW) + warp * RW;

  PackedSub<QT> pg[PASSES][M::SL], pu[PASSES][M::SL];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int f = f_warp + p * M::RPP + row_in_pass;
#pragma unroll
    for (int j = 0; j < M::SL; ++j) {
      const int c = sub_lane + M::G * j;
      pg[p][j] = load_sub<QT>(gw + (size_t)f * row_bytes, c);
      pu[p][j] = load_sub<QT>(uw + (size_t)f * row_bytes, c);
    }
  }

  const int pos0 = g.offsets[e], pos1 = g.offsets[e + 1];
  for (int pos = pos0; pos < pos1; ++pos) {
    const int t = pair_row(g.perm[pos], g.T, g.k);
    const float* x = X + (size_t)t * H;
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
#pragma unroll
      for (int j = 0; j < M::SL; ++j) {
        opaque(pg[p][j]);
        opaque(pu[p][j]);
      }
    float ag[PASSES], au[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) ag[p] = au[p] = 0.f;
#pragma unroll
    for (int j = 0; j < M::SL; ++j) {
      const int c = sub_lane + M::G * j;
      float xv[32], xs;
      load_x32(x + c * SUBK, xv, xs);
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        ag[p] += sub_dot<QT>(pg[p][j], xv, xs);
        au[p] += sub_dot<QT>(pu[p][j], xv, xs);
      }
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      float gs = group_sum<M::G>(ag[p]);
      float us = group_sum<M::G>(au[p]);
      if (sub_lane == 0) {
        const int f = f_warp + p * M::RPP + row_in_pass;
        hbuf[(size_t)pos * F + f] = silu_mul(gs, us);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// down: y[perm[pos]][row] = h[pos] . Wd_e[row]
// ---------------------------------------------------------------------------
template <int NSUB, int QT, int RW>
__global__ void __launch_bounds__(256) down_gemv_kernel(GroupedArgs g, const float* __restrict__ hbuf,
                                                        int H, float* __restrict__ y,
                                                        int tiles_per_expert) {
  using M = LaneMap<NSUB>;
  constexpr int PASSES = RW / M::RPP;
  constexpr int BYTES = qtype_size(QT);
  constexpr int F = NSUB * SUBK;
  const int a = blockIdx.x / tiles_per_expert, tile = blockIdx.x % tiles_per_expert;
  if (a >= g.n_active[0]) return;
  const int e = g.active[a];
  const size_t row_bytes = (size_t)(NSUB / 8) * BYTES;
  const uint8_t* dw = (e < g.E) ? g.W + (size_t)e * H * row_bytes : g.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub_lane = lane % M::G, row_in_pass = lane / M::G;
  const int r_warp = tile * (8 * RW) + warp * RW;

  PackedSub<QT> pd[PASSES][M::SL];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int r = r_warp + p * M::RPP + row_in_pass;
#pragma unroll
    for (int j = 0; j < M::SL; ++j) pd[p][j] = load_sub<QT>(dw + (size_t)r * row_bytes, sub_lane + M::G * j);
  }

  const int pos0 = g.offsets[e], pos1 = g.offsets[e + 1];
  for (int pos = pos0; pos < pos1; ++pos) {
    const int pair = g.perm[pos];
    const float* x = hbuf + (size_t)pos * F;
#pragma unroll
    for (int p = 0; p < PASSES; ++p)
#pragma unroll
      for (int j = 0; j < M::SL; ++j) opaque(pd[p][j]);
    float acc[PASSES];
#pragma unroll
    for (int p = 0; p < PASSES; ++p) acc[p] = 0.f;
#pragma unroll
    for (int j = 0; j < M::SL; ++j) {
      const int c = sub_lane + M::G * j;
      float xv[32], xs;
      load_x32(x + c * SUBK, xv, xs);
#pragma unroll
      for (int p = 0; p < PASSES; ++p)
        acc[p] += sub_dot<QT>(pd[p][j], xv, xs);
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      float s = group_sum<M::G>(acc[p]);
      if (sub_lane == 0) {
        const int r = r_warp + p * M::RPP + row_in_pass;
        y[(size_t)pair * H + r] = s;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// out_t = R_t + y_shared,t + sum_{s=0}^{k-1} w_{t,s} y_{t,s}, in slot order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                      const float* __restrict__ w,
                                                      const float* R, float* out, int T, int H,
                                                      int k, int has_shared) {
  const int H4 = H / 4;
  const size_t n = (size_t)T * H4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H4), c = (int)(i % H4);
    float4 acc = R ? reinterpret_cast<const float4*>(R + (size_t)t * H)[c] : make_float4(0, 0, 0, 0);
    if (has_shared) {
      float4 v = reinterpret_cast<const float4*>(y + ((size_t)T * k + t) * H)[c];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    for (int s = 0; s < k; ++s) {
      const float ws = w[(size_t)t * k + s];
      float4 v = reinterpret_cast<const float4*>(y + ((size_t)t * k + s) * H)[c];
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
    reinterpret_cast<float4*>(out + (size_t)t * H)[c] = acc;
  }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------
template <int NSUB>
constexpr int gemv_rows_per_warp(bool down) {
  return down ? (NSUB >= 32 ? 2 : (LaneMap<NSUB>::RPP > 8 ? LaneMap<NSUB>::RPP : 8))
              : (NSUB >= 128 ? 1 : (LaneMap<NSUB>::RPP > 2 ? LaneMap<NSUB>::RPP : 2));
}

template <int NSUB, int QT>
static cudaError_t gateup_launch_t(const GroupedArgs& g, const uint8_t* Wu, const uint8_t* Su,
                                   const float* X, int F, float* hbuf, cudaStream_t st) {
  constexpr int RW = gemv_rows_per_warp<NSUB>(false);
  const int rows_per_cta = 8 * RW;
  if (F % rows_per_cta) return cudaErrorInvalidValue;
  const int tiles = F / rows_per_cta;
  gateup_gemv_kernel<NSUB, QT, RW><<<g.max_active * tiles, 256, 0, st>>>(g, Wu, Su, X, F, hbuf, tiles);
  return cudaGetLastError();
}

template <int NSUB, int QT>
static cudaError_t down_launch_t(const GroupedArgs& g, const float* hbuf, int H, float* y,
                                 cudaStream_t st) {
  constexpr int RW = gemv_rows_per_warp<NSUB>(true);
  const int rows_per_cta = 8 * RW;
  if (H % rows_per_cta) return cudaErrorInvalidValue;
  const int tiles = H / rows_per_cta;
  down_gemv_kernel<NSUB, QT, RW><<<g.max_active * tiles, 256, 0, st>>>(g, hbuf, H, y, tiles);
  return cudaGetLastError();
}

#define QMOE_QT_SWITCH(NS, QT, CALL)                   \
  switch (QT) {                                        \
    case QMOE_Q4K: return CALL(NS, QMOE_Q4K);          \
    case QMOE_Q5K: return CALL(NS, QMOE_Q5K);          \
    case QMOE_Q6K: return CALL(NS, QMOE_Q6K);          \
    case QMOE_MXFP4: return CALL(NS, QMOE_MXFP4);      \
    default: return cudaErrorInvalidValue;             \
  }
#define QMOE_NSUB_SWITCH(NS, QT, CALL)            \
  switch (NS) {                                   \
    case 8: QMOE_QT_SWITCH(8, QT, CALL)           \
    case 16: QMOE_QT_SWITCH(16, QT, CALL)         \
    case 32: QMOE_QT_SWITCH(32, QT, CALL)         \
    case 64: QMOE_QT_SWITCH(64, QT, CALL)         \
    case 128: QMOE_QT_SWITCH(128, QT, CALL)       \
    default: return cudaErrorInvalidValue;        \
  }

cudaError_t launch_gateup_gemv(const GroupedArgs& g, const uint8_t* Wu, const uint8_t* Su, int qt,
                               const float* X, int H, int F, float* hbuf, cudaStream_t st) {
#define QMOE_GU(NS, Q) gateup_launch_t<NS, Q>(g, Wu, Su, X, F, hbuf, st)
  QMOE_NSUB_SWITCH(H / SUBK, qt, QMOE_GU)
#undef QMOE_GU
}

cudaError_t launch_down_gemv(const GroupedArgs& g, int qt, const float* hbuf, int F, int H,
                             float* y, cudaStream_t st) {
#define QMOE_DN(NS, Q) down_launch_t<NS, Q>(g, hbuf, H, y, st)
  QMOE_NSUB_SWITCH(F / SUBK, qt, QMOE_DN)
#undef QMOE_DN
}

cudaError_t launch_combine(const float* y, const float* w, const float* R, float* out, int T,
                           int H, int k, int has_shared, cudaStream_t st) {
  const size_t n = (size_t)T * (H / 4);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  combine_kernel<<<blocks, 256, 0, st>>>(y, w, R, out, T, H, k, has_shared);
  return cudaGetLastError();
}

}  // namespace qmoe
