// Kernels of the attention + MoE block around the routed-MoE layer.
//
// "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "What PR #382
// Now Splits": one Qwen3.5 block with full attention (16 query heads, 2 KV
// heads) and the MoE layer, recombined as attention + residual, routing on the
// whole state, MoE + residual. "Distributed CPU: Zip Fusion Beyond Tensor
// Parallelism", "Two-Dimensional Attention at Long Context": attention over
// context shards merged exactly from each shard's (max, normaliser, weighted
// output) -- used here inside one GPU by the split-context decode kernel.
#include <cmath>

#include "kernels.cuh"

namespace qmoe {

// ---------------------------------------------------------------------------
// RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma, one CTA per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                                      float eps, float* __restrict__ y, int H) {
  __shared__ float red[8];
  const int t = blockIdx.x, tid = threadIdx.x;
  const float* xr = x + (size_t)t * H;
  float s = 0.f;
  for (int i = tid; i < H; i += 256) s = fmaf(xr[i], xr[i], s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if ((tid & 31) == 0) red[tid >> 5] = s;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)H + eps);
  for (int i = tid; i < H; i += 256) y[(size_t)t * H + i] = xr[i] * inv * gamma[i];
}

// RMSNorm fused into the bf16 token operand of a tensor-core projection:
// y = bf16(x / sqrt(mean(x^2) + eps) * gamma), one CTA per row, written in the
// operand's K order (inside every group of 8 values, K offsets 0 4 1 5 2 6 3 7)
// as the bf16 conversion of the projection input would write it. The values
// are the same as RMSNorm then conversion: the fp32 expression is the same.
__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float* __restrict__ x,
                                                           const float* __restrict__ gamma, float eps,
                                                           __nv_bfloat16* __restrict__ y, int H) {
  __shared__ float red[8];
  const int t = blockIdx.x, tid = threadIdx.x;
  const float* xr = x + (size_t)t * H;
  float s = 0.f;
  for (int i = tid; i < H; i += 256) s = fmaf(xr[i], xr[i], s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if ((tid & 31) == 0) red[tid >> 5] = s;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)H + eps);
  for (int g = tid; g < H / 8; g += 256) {
    const float4 a = reinterpret_cast<const float4*>(xr)[2 * g];
    const float4 b = reinterpret_cast<const float4*>(xr)[2 * g + 1];
    const float4 ga = reinterpret_cast<const float4*>(gamma)[2 * g];
    const float4 gb = reinterpret_cast<const float4*>(gamma)[2 * g + 1];
    __nv_bfloat162 o[4];
    o[0] = __floats2bfloat162_rn(a.x * inv * ga.x, b.x * inv * gb.x);
    o[1] = __floats2bfloat162_rn(a.y * inv * ga.y, b.y * inv * gb.y);
    o[2] = __floats2bfloat162_rn(a.z * inv * ga.z, b.z * inv * gb.z);
    o[3] = __floats2bfloat162_rn(a.w * inv * ga.w, b.w * inv * gb.w);
    reinterpret_cast<uint4*>(y + (size_t)t * H)[g] = *reinterpret_cast<const uint4*>(o);
  }
}

cudaError_t launch_rmsnorm_bf16(const float* x, const float* gamma, float eps, __nv_bfloat16* y, int T, int H,
                                cudaStream_t st) {
  if (H % 8 != 0) return cudaErrorInvalidValue;
  rmsnorm_bf16_kernel<<<T, 256, 0, st>>>(x, gamma, eps, y, H);
  return cudaGetLastError();
}

// Routing of a dense projection seen as one expert (index 0) holding all rows;
// with ``offsets2``, also the offsets of a pair of projections of the same rows
// run as one launch (the first as expert 0, the second as the shared expert).
__global__ void dense_route_kernel(int32_t* offsets, int32_t* perm, int32_t* active, int32_t* n_active, int T,
                                   int32_t* offsets2) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T; i += gridDim.x * blockDim.x) perm[i] = i;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    offsets[0] = 0;
    offsets[1] = T;
    offsets[2] = T;
    active[0] = 0;
    n_active[0] = 1;
    if (offsets2 != nullptr) {
      offsets2[0] = 0;
      offsets2[1] = T;
      offsets2[2] = 2 * T;
    }
  }
}

// ---------------------------------------------------------------------------
// Rotate-half RoPE on q [T][nh][hd] (in place) and k [T][nkv][hd]; the rotated
// keys and the values are written to the bf16 caches at positions pos0 + t.
// Angles pos * theta^(-2i/hd) and their sines and cosines are taken in double
// (positions reach thousands of radians).
// ---------------------------------------------------------------------------
// Inverse frequencies theta^(-2i/hd), computed on the host in double.
struct RopeFreq {
  double inv[128];
};

__global__ void __launch_bounds__(256) rope_cache_kernel(float* __restrict__ q, const float* __restrict__ k,
                                                         const float* __restrict__ v, __nv_bfloat16* __restrict__ kc,
                                                         __nv_bfloat16* __restrict__ vc, int pos0, int nh, int nkv,
                                                         int hd, const __grid_constant__ RopeFreq fr) {
  extern __shared__ float cs[];  // [hd/2] cos, [hd/2] sin
  const int t = blockIdx.x, tid = threadIdx.x, half = hd / 2;
  const int pos = pos0 + t;
  for (int i = tid; i < half; i += 256) {
    // the angle pos * inv in double, reduced to [-pi, pi] by n turns with 2 pi
    // split into the double nearest to it and the remainder (two fused
    // multiply-adds), then sine and cosine in single precision
    const double a = (double)pos * fr.inv[i];
    const double n = rint(a * 0.15915494309189535);
    const double r = fma(-n, 2.4492935982947064e-16, fma(-n, 6.283185307179586, a));
    float sn, cn;
    sincosf((float)r, &sn, &cn);
    cs[i] = cn;
    cs[half + i] = sn;
  }
  __syncthreads();
  for (int idx = tid; idx < nh * half; idx += 256) {
    const int h = idx / half, i = idx % half;
    float* r = q + ((size_t)t * nh + h) * hd;
    const float a = r[i], b = r[i + half], c = cs[i], s = cs[half + i];
    r[i] = a * c - b * s;
    r[i + half] = b * c + a * s;
  }
  for (int idx = tid; idx < nkv * half; idx += 256) {
    const int h = idx / half, i = idx % half;
    const float* r = k + ((size_t)t * nkv + h) * hd;
    const float a = r[i], b = r[i + half], c = cs[i], s = cs[half + i];
    __nv_bfloat16* dst = kc + ((size_t)pos * nkv + h) * hd;
    dst[i] = __float2bfloat16_rn(a * c - b * s);
    dst[i + half] = __float2bfloat16_rn(b * c + a * s);
  }
  for (int idx = tid; idx < nkv * hd; idx += 256) {
    const int h = idx / hd, d = idx % hd;
    vc[((size_t)pos * nkv + h) * hd + d] = __float2bfloat16_rn(v[((size_t)t * nkv + h) * hd + d]);
  }
}

// ---------------------------------------------------------------------------
// Split-context attention for few query rows: CTA (row t, head h, chunk c)
// scores the chunk's 256 cache positions (causal: <= pos0 + t), and writes the
// chunk's (max m, normaliser l, weighted sum o[hd]) for the exact merge.
// ---------------------------------------------------------------------------
constexpr int ATT_CHUNK = 256;

__global__ void __launch_bounds__(256) attn_chunk_kernel(const float* __restrict__ q,
                                                         const __nv_bfloat16* __restrict__ kc,
                                                         const __nv_bfloat16* __restrict__ vc,
                                                         float* __restrict__ part, int pos0, int nh, int nkv,
                                                         int hd, int nchunks) {
  extern __shared__ float sm[];
  float* qs = sm;          // [hd]
  float* ps = sm + hd;     // [ATT_CHUNK]
  __shared__ float red[8];
  __shared__ float stat[2];
  const int tid = threadIdx.x;
  const int th = blockIdx.x, c = blockIdx.y;
  const int t = th / nh, h = th % nh, g = h / (nh / nkv);
  const int nvalid = pos0 + t + 1;
  const int j0 = c * ATT_CHUNK;
  float* out = part + ((size_t)th * nchunks + c) * (hd + 2);
  if (j0 >= nvalid) {
    for (int d = tid; d < hd + 2; d += 256) out[d] = (d == 0) ? -INFINITY : 0.f;
    return;
  }
  const float scale = rsqrtf((float)hd);
  for (int d = tid; d < hd; d += 256) qs[d] = q[((size_t)t * nh + h) * hd + d] * scale;
  __syncthreads();
  const int j = j0 + tid;
  float s = -INFINITY;
  if (tid < ATT_CHUNK && j < nvalid) {
    const uint4* kr = reinterpret_cast<const uint4*>(kc + ((size_t)j * nkv + g) * hd);
    float acc = 0.f;
    for (int i = 0; i < hd / 8; ++i) {
      const uint4 u = __ldg(kr + i);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 f = __bfloat1622float2(b2[m]);
        acc = fmaf(qs[8 * i + 2 * m], f.x, acc);
        acc = fmaf(qs[8 * i + 2 * m + 1], f.y, acc);
      }
    }
    s = acc;
  }
  // chunk max
  float mx = s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  if (tid == 0) {
    float m = red[0];
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
    stat[0] = m;
  }
  __syncthreads();
  const float m = stat[0];
  const float p = (s == -INFINITY) ? 0.f : __expf(s - m);
  ps[tid] = p;
  float l = p;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  __syncthreads();
  if ((tid & 31) == 0) red[tid >> 5] = l;
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += red[w];
    stat[1] = tot;
  }
  const int nk = min(ATT_CHUNK, nvalid - j0);
  for (int d = tid; d < hd; d += 256) {
    const __nv_bfloat16* vp = vc + ((size_t)j0 * nkv + g) * hd + d;
    float acc = 0.f;
#pragma unroll 4
    for (int i = 0; i < nk; ++i) acc = fmaf(ps[i], __bfloat162float(vp[(size_t)i * nkv * hd]), acc);
    out[2 + d] = acc;
  }
  __syncthreads();
  if (tid == 0) {
    out[0] = m;
    out[1] = stat[1];
  }
}

// Exact merge of the chunks of one (row, head): rescale every chunk to the
// common maximum, then o = sum(o_c e^(m_c - M)) / sum(l_c e^(m_c - M)).
__global__ void attn_merge_kernel(const float* __restrict__ part, float* __restrict__ o, int nchunks, int hd) {
  const int th = blockIdx.x;
  const float* pc = part + (size_t)th * nchunks * (hd + 2);
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c)
    if (pc[(size_t)c * (hd + 2) + 1] > 0.f) M = fmaxf(M, pc[(size_t)c * (hd + 2)]);
  for (int d = threadIdx.x; d < hd; d += blockDim.x) {
    float L = 0.f, acc = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const float* q = pc + (size_t)c * (hd + 2);
      if (q[1] > 0.f) {
        const float sc = __expf(q[0] - M);
        L = fmaf(q[1], sc, L);
        acc = fmaf(q[2 + d], sc, acc);
      }
    }
    o[(size_t)th * hd + d] = acc / L;
  }
}

__global__ void add_kernel(const float* __restrict__ a, const float* __restrict__ b, float* __restrict__ y, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    y[i] = a[i] + b[i];
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_rmsnorm(const float* x, const float* gamma, float eps, float* y, int T, int H, cudaStream_t st) {
  rmsnorm_kernel<<<T, 256, 0, st>>>(x, gamma, eps, y, H);
  return cudaGetLastError();
}

cudaError_t launch_dense_route(int32_t* offsets, int32_t* perm, int32_t* active, int32_t* n_active, int T,
                               cudaStream_t st, int32_t* offsets2) {
  int blocks = (T + 255) / 256;
  if (blocks > 64) blocks = 64;
  dense_route_kernel<<<blocks, 256, 0, st>>>(offsets, perm, active, n_active, T, offsets2);
  return cudaGetLastError();
}

cudaError_t launch_rope_cache(float* q, const float* k, const float* v, __nv_bfloat16* kc, __nv_bfloat16* vc, int T,
                              int pos0, int nh, int nkv, int hd, double theta, cudaStream_t st) {
  if (hd > 256) return cudaErrorInvalidValue;
  RopeFreq fr{};
  for (int i = 0; i < hd / 2; ++i) fr.inv[i] = std::pow(theta, -2.0 * (double)i / (double)hd);
  rope_cache_kernel<<<T, 256, sizeof(float) * hd, st>>>(q, k, v, kc, vc, pos0, nh, nkv, hd, fr);
  return cudaGetLastError();
}

int attn_nchunks(int T, int pos0) { return (pos0 + T + ATT_CHUNK - 1) / ATT_CHUNK; }

cudaError_t launch_attention(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, float* part, float* o,
                             __nv_bfloat16* ob, int T, int pos0, int nh, int nkv, int hd, bool chunked, int* status,
                             unsigned long long wait_ns, int fault, cudaStream_t st) {
  if (chunked) {
    if (ob != nullptr) return cudaErrorInvalidValue;
    const int nc = attn_nchunks(T, pos0);
    attn_chunk_kernel<<<dim3(T * nh, nc), 256, sizeof(float) * (hd + ATT_CHUNK), st>>>(q, kc, vc, part, pos0, nh,
                                                                                          nkv, hd, nc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attn_merge_kernel<<<T * nh, 128, 0, st>>>(part, o, nc, hd);
    return cudaGetLastError();
  }
  if (hd != 128) return cudaErrorInvalidValue;
  return launch_attention_prefill_tc(q, kc, vc, o, ob, T, pos0, nh, nkv, status, wait_ns, fault, st);
}

cudaError_t launch_add(const float* a, const float* b, float* y, size_t n, cudaStream_t st) {
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  add_kernel<<<blocks, 256, 0, st>>>(a, b, y, n);
  return cudaGetLastError();
}

}  // namespace qmoe
