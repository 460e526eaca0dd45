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

template <int QT>
struct PackedSub {
  uint4 q;      // 16 quant bytes
  uint32_t hb;  // Q5_K high bits of the sub-block
  float2 sc;    // (d*s_j, dmin*m_j)
};

template <int QT>
__device__ __forceinline__ PackedSub<QT> load_sub(const uint8_t* row, int c) {
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  const uint8_t* blk = row + (size_t)(c >> 3) * BYTES;
  const int j = c & 7;
  PackedSub<QT> p;
  KHeader h = load_header(blk);
  p.sc = sub_scale(h, j);
  p.q = __ldg(reinterpret_cast<const uint4*>(blk + quant_offset(QT, j)));
  p.hb = (QT == QMOE_Q5K) ? __ldg(reinterpret_cast<const uint32_t*>(blk + 16 + 4 * j)) : 0u;
  return p;
}

// Hides the packed registers' values from the optimiser at the top of each
// row iteration, so the unpacking stays inside the loop instead of being
// hoisted out as 32 live floats per sub-block.
template <int QT>
__device__ __forceinline__ void opaque(PackedSub<QT>& p) {
  asm volatile("" : "+r"(p.q.x), "+r"(p.q.y), "+r"(p.q.z), "+r"(p.q.w), "+r"(p.hb));
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
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
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
        ag[p] += sub_contrib(dot_sub_prmt<QT>(pg[p][j].q, pg[p][j].hb, xv), xs, pg[p][j].sc);
        au[p] += sub_contrib(dot_sub_prmt<QT>(pu[p][j].q, pu[p][j].hb, xv), xs, pu[p][j].sc);
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
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
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
        acc[p] += sub_contrib(dot_sub_prmt<QT>(pd[p][j].q, pd[p][j].hb, xv), xs, pd[p][j].sc);
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

#define QMOE_NSUB_SWITCH(NS, QT, CALL)                         \
  switch (NS) {                                                \
    case 8: return QT ? CALL(8, QMOE_Q5K) : CALL(8, QMOE_Q4K);     \
    case 16: return QT ? CALL(16, QMOE_Q5K) : CALL(16, QMOE_Q4K);  \
    case 32: return QT ? CALL(32, QMOE_Q5K) : CALL(32, QMOE_Q4K);  \
    case 64: return QT ? CALL(64, QMOE_Q5K) : CALL(64, QMOE_Q4K);  \
    case 128: return QT ? CALL(128, QMOE_Q5K) : CALL(128, QMOE_Q4K); \
    default: return cudaErrorInvalidValue;                     \
  }

cudaError_t launch_gateup_gemv(const GroupedArgs& g, const uint8_t* Wu, const uint8_t* Su, int qt,
                               const float* X, int H, int F, float* hbuf, cudaStream_t st) {
#define QMOE_GU(NS, Q) gateup_launch_t<NS, Q>(g, Wu, Su, X, F, hbuf, st)
  QMOE_NSUB_SWITCH(H / SUBK, qt == QMOE_Q5K, QMOE_GU)
#undef QMOE_GU
}

cudaError_t launch_down_gemv(const GroupedArgs& g, int qt, const float* hbuf, int F, int H,
                             float* y, cudaStream_t st) {
#define QMOE_DN(NS, Q) down_launch_t<NS, Q>(g, hbuf, H, y, st)
  QMOE_NSUB_SWITCH(F / SUBK, qt == QMOE_Q5K, QMOE_DN)
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
