// Causal attention for many query rows (block prefill), on the tensor cores.
//
// "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "What PR #382
// Now Splits": 16 query heads over 2 KV heads, so query head h attends to the
// keys and values of KV head h / 8, causally, with the 1/sqrt(head_dim) scale.
// "Distributed CPU: Zip Fusion Beyond Tensor Parallelism", "Two-Dimensional
// Attention at Long Context": the softmax over key blocks is carried by its
// running maximum, normaliser and weighted output, which is how this kernel
// walks the keys.
//
// CTA = (64 query rows, one head), 4 warps of 16 rows. Per 64-key tile:
//   S = Q K^T    bf16 mma.sync m16n8k16, fp32 accumulate; Q (scaled by
//                log2(e)/sqrt(hd)) lives in registers as A fragments, K
//                comes from shared memory by ldmatrix;
//   softmax      online in exp2 form: row max over the tile, O and the
//                normaliser rescaled by exp2(m_old - m_new);
//   O += P V     P (bf16) goes from the S accumulator registers straight
//                into A fragments; V by ldmatrix.trans.
// K and V tiles (bf16, from the caches) are double-buffered with cp.async
// into 16-byte-chunk XOR-swizzled rows, so ldmatrix reads no bank twice.
#include "kernels.cuh"

namespace qmoe {

constexpr int FA_BQ = 64, FA_BK = 64, FA_HD = 128;
constexpr int FA_THREADS = 128;
constexpr int FA_TILE_BYTES = FA_BK * FA_HD * 2;  // 16 KB per K or V tile

__device__ __forceinline__ uint32_t fa_smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk c (0..15) of row r in a 256-byte-row tile.
__device__ __forceinline__ uint32_t fa_swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void fa_cp_async16(uint32_t dst, const void* src, bool valid) {
  const uint32_t n = valid ? 16u : 0u;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ void fa_ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void fa_ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void fa_mma(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t fa_pack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// q [T][nh][128] fp32 (rotated), kc/vc [ctx][nkv][128] bf16, o [T][nh][128]
// fp32; query t sits at position pos0 + t and sees keys 0 .. pos0 + t.
__global__ void __launch_bounds__(FA_THREADS) attn_prefill_mma_kernel(const float* __restrict__ q,
                                                                      const __nv_bfloat16* __restrict__ kc,
                                                                      const __nv_bfloat16* __restrict__ vc,
                                                                      float* __restrict__ o, int T, int pos0, int nh,
                                                                      int nkv) {
  extern __shared__ __align__(128) uint8_t fa_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;  // heavy (late) tiles first
  const int h = blockIdx.y, kvh = h / (nh / nkv);
  const int t0 = qt * FA_BQ;
  const int qrow0 = t0 + 16 * warp;  // this warp's first query row
  const uint32_t sbase = fa_smem_u32(fa_smem);
  // stage s: K at s * 2 * TILE, V at s * 2 * TILE + TILE
  auto k_tile = [&](int s) { return sbase + (uint32_t)(s * 2 * FA_TILE_BYTES); };
  auto v_tile = [&](int s) { return sbase + (uint32_t)(s * 2 * FA_TILE_BYTES + FA_TILE_BYTES); };

  const int last_row = min(T - 1, t0 + FA_BQ - 1);
  const int kend = pos0 + last_row + 1;  // keys [0, kend)
  const int ntiles = (kend + FA_BK - 1) / FA_BK;

  // K and V tile loads: 64 rows x 16 chunks each, 16 chunks per thread
  auto load_tile = [&](int kt, int s) {
    const int k0 = kt * FA_BK;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + FA_THREADS * i;  // 0..1023
      const int r = idx >> 4, c = idx & 15;
      const int key = k0 + r;
      const bool valid = key < kend;
      const size_t off = ((size_t)(valid ? key : 0) * nkv + kvh) * FA_HD + 8 * c;
      fa_cp_async16(k_tile(s) + fa_swz(r, c), kc + off, valid);
      fa_cp_async16(v_tile(s) + fa_swz(r, c), vc + off, valid);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  load_tile(0, 0);

  // Q fragments (rows qrow0 + g8, + 8), scaled so that exp2 gives e^(s/sqrt(hd))
  const float qscale = 1.4426950408889634f * rsqrtf((float)FA_HD);
  uint32_t qa[8][4];
  {
    const int ra = qrow0 + g8, rb = ra + 8;
    const float* qa_row = q + ((size_t)(ra < T ? ra : 0) * nh + h) * FA_HD;
    const float* qb_row = q + ((size_t)(rb < T ? rb : 0) * nh + h) * FA_HD;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c = 16 * ks + 2 * t4;
      const float2 x0 = ra < T ? *reinterpret_cast<const float2*>(qa_row + c) : make_float2(0.f, 0.f);
      const float2 x1 = rb < T ? *reinterpret_cast<const float2*>(qb_row + c) : make_float2(0.f, 0.f);
      const float2 x2 = ra < T ? *reinterpret_cast<const float2*>(qa_row + c + 8) : make_float2(0.f, 0.f);
      const float2 x3 = rb < T ? *reinterpret_cast<const float2*>(qb_row + c + 8) : make_float2(0.f, 0.f);
      qa[ks][0] = fa_pack(x0.x * qscale, x0.y * qscale);
      qa[ks][1] = fa_pack(x1.x * qscale, x1.y * qscale);
      qa[ks][2] = fa_pack(x2.x * qscale, x2.y * qscale);
      qa[ks][3] = fa_pack(x3.x * qscale, x3.y * qscale);
    }
  }

  float oacc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) oacc[j][c] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY;  // running max of rows g8, g8 + 8
  float l_a = 0.f, l_b = 0.f;              // this thread's share of the normalisers
  const int pa = pos0 + qrow0 + g8, pb = pa + 8;  // query positions

  for (int kt = 0; kt < ntiles; ++kt) {
    const int s = kt & 1;
    if (kt + 1 < ntiles) {
      load_tile(kt + 1, s ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int k0 = kt * FA_BK;
    // ---- S = Q K^T: 16 rows x 64 keys per warp
    float sacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) sacc[j][c] = 0.f;
    const uint32_t kb = k_tile(s);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {  // key n-tiles 2jp, 2jp+1
        const int m = lane >> 3, rr = lane & 7;
        const int key = 8 * (2 * jp + (m >> 1)) + rr;
        const int chunk = 2 * ks + (m & 1);
        uint32_t b0, b1, b2, b3;
        fa_ldsm_x4(kb + fa_swz(key, chunk), b0, b1, b2, b3);
        fa_mma(sacc[2 * jp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        fa_mma(sacc[2 * jp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    }
    // ---- causal mask and online softmax (rows g8 and g8 + 8)
    const bool diag = k0 + FA_BK - 1 > pos0 + qrow0;  // some key of the tile is past some row's position
    float mx_a = m_a, mx_b = m_b;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int key = k0 + 8 * j + 2 * t4;
      if (diag) {
        if (key > pa) sacc[j][0] = -INFINITY;
        if (key + 1 > pa) sacc[j][1] = -INFINITY;
        if (key > pb) sacc[j][2] = -INFINITY;
        if (key + 1 > pb) sacc[j][3] = -INFINITY;
      }
      mx_a = fmaxf(mx_a, fmaxf(sacc[j][0], sacc[j][1]));
      mx_b = fmaxf(mx_b, fmaxf(sacc[j][2], sacc[j][3]));
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    // rows past T see only masked or zero keys; keep their max finite
    const float ref_a = mx_a == -INFINITY ? 0.f : mx_a;
    const float ref_b = mx_b == -INFINITY ? 0.f : mx_b;
    const float al_a = exp2f(m_a - ref_a), al_b = exp2f(m_b - ref_b);  // 0 on the first tile
    m_a = mx_a;
    m_b = mx_b;
    l_a *= al_a;
    l_b *= al_b;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      oacc[j][0] *= al_a;
      oacc[j][1] *= al_a;
      oacc[j][2] *= al_b;
      oacc[j][3] *= al_b;
    }
    // P = exp2(S - m), as bf16 A fragments of P V (keys 16 ks .. 16 ks + 15)
    uint32_t pfrag[4][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p0 = exp2f(sacc[j][0] - ref_a), p1 = exp2f(sacc[j][1] - ref_a);
      const float p2 = exp2f(sacc[j][2] - ref_b), p3 = exp2f(sacc[j][3] - ref_b);
      l_a += p0 + p1;
      l_b += p2 + p3;
      const int ks = j >> 1, hi = j & 1;
      pfrag[ks][2 * hi + 0] = fa_pack(p0, p1);  // row g8
      pfrag[ks][2 * hi + 1] = fa_pack(p2, p3);  // row g8 + 8
    }
    // ---- O += P V: 16 rows x 128 head dims per warp
    const uint32_t vb = v_tile(s);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int jp = 0; jp < 8; ++jp) {  // head-dim n-tiles 2jp, 2jp+1
        const int m = lane >> 3, rr = lane & 7;
        const int key = 16 * ks + 8 * (m & 1) + rr;
        const int chunk = 2 * jp + (m >> 1);
        uint32_t b0, b1, b2, b3;
        fa_ldsm_x4_t(vb + fa_swz(key, chunk), b0, b1, b2, b3);
        fa_mma(oacc[2 * jp], pfrag[ks][0], pfrag[ks][1], pfrag[ks][2], pfrag[ks][3], b0, b1);
        fa_mma(oacc[2 * jp + 1], pfrag[ks][0], pfrag[ks][1], pfrag[ks][2], pfrag[ks][3], b2, b3);
      }
    }
    __syncthreads();  // the stage is refilled next
  }
  // normalisers: the 4 threads of a row hold parts of it
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const int ra = qrow0 + g8, rb = ra + 8;
  const float ia = 1.f / l_a, ib = 1.f / l_b;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int d = 8 * j + 2 * t4;
    if (ra < T)
      *reinterpret_cast<float2*>(o + ((size_t)ra * nh + h) * FA_HD + d) = make_float2(oacc[j][0] * ia, oacc[j][1] * ia);
    if (rb < T)
      *reinterpret_cast<float2*>(o + ((size_t)rb * nh + h) * FA_HD + d) = make_float2(oacc[j][2] * ib, oacc[j][3] * ib);
  }
}

cudaError_t launch_attention_prefill(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, float* o,
                                     int T, int pos0, int nh, int nkv, cudaStream_t st) {
  const int smem = 2 * 2 * FA_TILE_BYTES;  // two stages of K and V
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(attn_prefill_mma_kernel), smem);
  if (e != cudaSuccess) return e;
  attn_prefill_mma_kernel<<<dim3((T + FA_BQ - 1) / FA_BQ, nh), FA_THREADS, smem, st>>>(q, kc, vc, o, T, pos0, nh,
                                                                                       nkv);
  return cudaGetLastError();
}

}  // namespace qmoe
