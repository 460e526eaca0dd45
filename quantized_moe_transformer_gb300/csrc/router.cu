// Router and token-to-expert permutation.
//
// "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "What The
// First Prototype Split": every row carries its selected top-k expert indices
// and routing weights; "A Separate Decode Result Shows Why Axis Choice
// Matters": the selected routes are independent work items whose outputs are
// merged in slot order. Here the routes are grouped by expert with a histogram
// and an exclusive prefix scan so that each expert's packed weights are read
// once for all the rows that selected it.
#include "kernels.cuh"

namespace qmoe {

// ---------------------------------------------------------------------------
// Router logits, split along H: part[s][t][e] = sum_{h in slice s} X[t][h] Wr[h][e].
// Tile: 32 rows x 64 experts per CTA, 256 threads, each thread 2 rows x 4
// experts, K staged through shared memory in chunks of 32.
// ---------------------------------------------------------------------------
constexpr int RL_BT = 32, RL_BE = 64, RL_BK = 32;

__global__ void __launch_bounds__(256) router_logits_kernel(const float* __restrict__ X,
                                                            const float* __restrict__ Wr,
                                                            float* __restrict__ part, int T, int H,
                                                            int E, int h_per_split) {
  __shared__ float xs[RL_BK][RL_BT + 1];
  __shared__ __align__(16) float ws[RL_BK][RL_BE];
  const int t0 = blockIdx.y * RL_BT, e0 = blockIdx.x * RL_BE;
  const int hs0 = blockIdx.z * h_per_split;
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  float acc[2][4] = {};
  for (int hk = hs0; hk < hs0 + h_per_split; hk += RL_BK) {
    // X tile: 32 rows x 32 h (transposed into xs[h][t])
    for (int i = tid; i < RL_BT * RL_BK; i += 256) {
      int r = i / RL_BK, c = i % RL_BK;
      int t = t0 + r;
      xs[c][r] = (t < T) ? __ldg(&X[(size_t)t * H + hk + c]) : 0.f;
    }
    // Wr tile: 32 h x 64 experts
    for (int i = tid; i < RL_BK * RL_BE; i += 256) {
      int r = i / RL_BE, c = i % RL_BE;
      int e = e0 + c;
      ws[r][c] = (e < E) ? __ldg(&Wr[(size_t)(hk + r) * E + e]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < RL_BK; ++kk) {
      float a0 = xs[kk][ty * 2], a1 = xs[kk][ty * 2 + 1];
      float4 b = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      acc[0][0] = fmaf(a0, b.x, acc[0][0]);
      acc[0][1] = fmaf(a0, b.y, acc[0][1]);
      acc[0][2] = fmaf(a0, b.z, acc[0][2]);
      acc[0][3] = fmaf(a0, b.w, acc[0][3]);
      acc[1][0] = fmaf(a1, b.x, acc[1][0]);
      acc[1][1] = fmaf(a1, b.y, acc[1][1]);
      acc[1][2] = fmaf(a1, b.z, acc[1][2]);
      acc[1][3] = fmaf(a1, b.w, acc[1][3]);
    }
    __syncthreads();
  }
  float* dst = part + (size_t)blockIdx.z * T * E;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    int t = t0 + ty * 2 + r;
    if (t >= T) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int e = e0 + tx * 4 + c;
      if (e < E) dst[(size_t)t * E + e] = acc[r][c];
    }
  }
}

// ---------------------------------------------------------------------------
// Router logits for large T: 128 rows x 128 experts per CTA, 256 threads,
// each thread an 8 x 8 block (two 4-row by two 4-expert sub-blocks, so that
// its shared-memory reads are 16-byte vectors without bank conflicts), K
// staged in slices of 16 through double-buffered shared memory. Same H-split
// partials as above: part[s][t][e].
// ---------------------------------------------------------------------------
constexpr int RG_BT = 128, RG_BE = 128, RG_BK = 16;

__global__ void __launch_bounds__(256) router_gemm_kernel(const float* __restrict__ X, const float* __restrict__ Wr,
                                                          float* __restrict__ part, int T, int H, int E,
                                                          int h_per_split) {
  __shared__ __align__(16) float xs[2][RG_BK][RG_BT + 4];  // X slice, transposed: [h][t]
  __shared__ __align__(16) float ws[2][RG_BK][RG_BE];      // Wr slice: [h][e]
  const int t0 = blockIdx.y * RG_BT, e0 = blockIdx.x * RG_BE;
  const int hs0 = blockIdx.z * h_per_split;
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  // loader mapping: X 128 rows x 16 h = 512 float4 (2 per thread, along h);
  // Wr 16 h x 128 e = 512 float4 (2 per thread, along e)
  float4 xr[2], wr[2];
  auto load = [&](int hk) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int q = tid + 256 * i;
      const int r = q >> 2, c4 = (q & 3) * 4;  // row r, h offset c4
      const int t = t0 + r;
      xr[i] = t < T ? __ldg(reinterpret_cast<const float4*>(X + (size_t)t * H + hk + c4)) : make_float4(0.f, 0.f, 0.f, 0.f);
      const int hr = q >> 5, e4 = (q & 31) * 4;  // h row, expert offset
      const int e = e0 + e4;
      if ((E & 3) == 0 && e + 3 < E) {
        wr[i] = __ldg(reinterpret_cast<const float4*>(Wr + (size_t)(hk + hr) * E + e));
      } else {
        const float* w = Wr + (size_t)(hk + hr) * E;
        wr[i] = make_float4(e < E ? w[e] : 0.f, e + 1 < E ? w[e + 1] : 0.f, e + 2 < E ? w[e + 2] : 0.f,
                            e + 3 < E ? w[e + 3] : 0.f);
      }
    }
  };
  auto store = [&](int b) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int q = tid + 256 * i;
      const int r = q >> 2, c4 = (q & 3) * 4;
      xs[b][c4 + 0][r] = xr[i].x;
      xs[b][c4 + 1][r] = xr[i].y;
      xs[b][c4 + 2][r] = xr[i].z;
      xs[b][c4 + 3][r] = xr[i].w;
      const int hr = q >> 5, e4 = (q & 31) * 4;
      *reinterpret_cast<float4*>(&ws[b][hr][e4]) = wr[i];
    }
  };
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  const int nk = h_per_split / RG_BK;
  load(hs0);
  store(0);
  __syncthreads();
  for (int kb = 0; kb < nk; ++kb) {
    const int b = kb & 1;
    if (kb + 1 < nk) load(hs0 + (kb + 1) * RG_BK);
#pragma unroll
    for (int kk = 0; kk < RG_BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&xs[b][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&xs[b][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&ws[b][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&ws[b][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (kb + 1 < nk) store(b ^ 1);
    __syncthreads();
  }
  float* dst = part + (size_t)blockIdx.z * T * E;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
      if (e < E) dst[(size_t)t * E + e] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// Router logits for moderate T: a CTA (256 threads) covers 8 experts x one
// quarter of H x a block of RR_ROWS rows. Thread t keeps Wr rows h0 + t +
// 256 j of the 8 experts in registers; the block's X slice is staged in
// shared memory with all loads in flight at once; each warp's 8 partial sums
// per row are reduced by recursive halving across the lanes (9 shuffles), the
// 8 warps' through shared memory. part[q][t][e] for the 4 quarters q.
// ---------------------------------------------------------------------------
// rows per CTA: the staged X slice stays within 32 KB
__host__ __device__ constexpr int rr_rows(int rpt) { return rpt >= 4 ? 8 : 16; }

template <int RPT>
__global__ void __launch_bounds__(256) router_rows_kernel(const float* __restrict__ X, const float* __restrict__ Wr,
                                                          float* __restrict__ part, int T, int H, int E) {
  constexpr int HQ = 256 * RPT;  // H / 4
  constexpr int RR_ROWS = rr_rows(RPT);
  __shared__ __align__(16) float xs[RR_ROWS][HQ];
  __shared__ float red[RR_ROWS][8][8];  // [row][warp][expert]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = (blockIdx.x >> 2) * 8, hq = blockIdx.x & 3;
  const int h0 = hq * HQ;
  const int r0 = blockIdx.y * RR_ROWS;
  const int nr = T - r0 < RR_ROWS ? T - r0 : RR_ROWS;
  // X slice: nr rows x HQ floats, 16-byte loads
  for (int i = tid; i < nr * (HQ / 4); i += 256) {
    const int r = i / (HQ / 4), c = i % (HQ / 4);
    reinterpret_cast<float4*>(&xs[r][0])[c] = __ldg(reinterpret_cast<const float4*>(X + (size_t)(r0 + r) * H + h0) + c);
  }
  float w[RPT][8];
#pragma unroll
  for (int j = 0; j < RPT; ++j) {
    const float4* src = reinterpret_cast<const float4*>(Wr + (size_t)(h0 + tid + 256 * j) * E + e0);
    const float4 a = __ldg(src), b = __ldg(src + 1);
    w[j][0] = a.x; w[j][1] = a.y; w[j][2] = a.z; w[j][3] = a.w;
    w[j][4] = b.x; w[j][5] = b.y; w[j][6] = b.z; w[j][7] = b.w;
  }
  __syncthreads();
  const int q_mine = (lane >> 2) & 7;  // expert this lane ends up holding
  for (int r = 0; r < nr; ++r) {
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const float x = xs[r][tid + 256 * j];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = fmaf(x, w[j][q], v[q]);
    }
    // recursive halving: after the xor-16, -8 and -4 steps lane l holds the
    // 4-lane partial of expert (l >> 2) & 7, then two more steps sum those
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool hi = lane & 16;
      const float send = hi ? v[i] : v[i + 4];
      const float keep = hi ? v[i + 4] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const bool hi = lane & 8;
      const float send = hi ? v[i] : v[i + 2];
      const float keep = hi ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    {
      const bool hi = lane & 4;
      const float send = hi ? v[0] : v[1];
      const float keep = hi ? v[1] : v[0];
      v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    if ((lane & 3) == 0) red[r][warp][q_mine] = v[0];
  }
  __syncthreads();
  if (tid < nr * 8) {
    const int r = tid >> 3, q = tid & 7;
    float s2 = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) s2 += red[r][w8][q];
    part[((size_t)hq * T + r0 + r) * E + e0 + q] = s2;
  }
}

// ---------------------------------------------------------------------------
// Top-k of one row by one warp. Lane l holds experts l, l+32, ...; each round
// takes the largest remaining logit, the lower index on ties.
// ---------------------------------------------------------------------------
template <int EPL>
__device__ __forceinline__ void warp_topk_row(const float* part, int nsplit, int T, int E, int k,
                                              int t, int32_t* ids_out, float* w_out,
                                              int32_t* ids_smem) {
  const int lane = threadIdx.x & 31;
  float v[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    float s = 0.f;
    if (e < E) {
      // the split partials are loaded 8 at a time (independent loads in
      // flight) and added in split order
      for (int s0 = 0; s0 < nsplit; s0 += 8) {
        float pv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          pv[q] = (s0 + q < nsplit) ? __ldcg(part + ((size_t)(s0 + q) * T + t) * E + e) : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) s += pv[q];
      }
    }
    v[j] = (e < E) ? s : -INFINITY;
  }
  uint32_t taken = 0;
  float l0 = 0.f, denom = 0.f;
  float sel_l[16];
  int sel_e[16];
  for (int r = 0; r < k; ++r) {
    // local best: highest value, lowest index (j ascending = index ascending)
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      int e = lane + 32 * j;
      bool ok = (e < E) && !((taken >> j) & 1u);
      if (ok && (v[j] > bv || (v[j] == bv && e < be))) {
        bv = v[j];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be >= E) {
      // every remaining logit is NaN or -inf: take the lowest index not yet
      // taken (ties go to the lower index), so that a row never repeats an id
      int lo = 0x7fffffff;
#pragma unroll
      for (int j = EPL - 1; j >= 0; --j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u)) lo = e;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      be = lo;
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    sel_l[r] = bv;
    sel_e[r] = be;
    if (r == 0) l0 = bv;
  }
  if (lane == 0) {
    for (int r = 0; r < k; ++r) denom += expf(sel_l[r] - l0);
    for (int r = 0; r < k; ++r) {
      ids_out[(size_t)t * k + r] = sel_e[r];
      w_out[(size_t)t * k + r] = expf(sel_l[r] - l0) / denom;
      if (ids_smem) ids_smem[(size_t)t * k + r] = sel_e[r];
    }
  }
}

template <int EPL>
__global__ void __launch_bounds__(128) topk_kernel(const float* __restrict__ part, int nsplit,
                                                   int T, int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ w) {
  int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= T) return;
  warp_topk_row<EPL>(part, nsplit, T, E, k, t, ids, w, nullptr);
}

// ---------------------------------------------------------------------------
// Permutation for small T (one CTA): optional top-k, histogram, exclusive scan,
// stable scatter in (t, slot) order, active-expert list, and (with ``chunks``)
// the tensor-core path's token-chunk list. Expert index E is the shared
// expert, which takes every row (pairs T*k + t).
// Workspace outputs: offsets[E+2], perm[T*k+T], active[E+1], n_active[1].
// ---------------------------------------------------------------------------
template <int EPL>
__global__ void __launch_bounds__(1024) route_small_kernel(
    const float* __restrict__ part, int nsplit, const int32_t* __restrict__ ids_in, int T, int E,
    int k, int has_shared, int32_t* __restrict__ ids, float* __restrict__ w,
    int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ active,
    int32_t* __restrict__ n_active, int* status, int cap, int2* __restrict__ chunks,
    int32_t* __restrict__ n_tok_chunks) {
  extern __shared__ int32_t sm[];
  __shared__ int32_t cstart[1025 + 32];
  int32_t* cnt = sm;                 // [E+1]
  int32_t* cur = sm + (E + 1);       // [E+1] running cursor / scan scratch
  int32_t* sid = sm + 2 * (E + 1);   // [T*k] ids of this batch
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = T * k;
  for (int i = tid; i <= E; i += blockDim.x) cnt[i] = 0;
  if (ids_in == nullptr) {
    for (int t = warp; t < T; t += blockDim.x / 32)
      warp_topk_row<EPL>(part, nsplit, T, E, k, t, ids, w, sid);
  } else {
    for (int p = tid; p < P; p += blockDim.x) {
      int e = ids_in[p];
      if (e < 0 || e >= E) {
        record_status(status, QMOE_ERR_DEVICE_ARG);
        e = 0;
      }
      sid[p] = e;
    }
  }
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) atomicAdd(&cnt[sid[p]], 1);
  if (tid == 0) cnt[E] = has_shared ? T : 0;
  __syncthreads();
  // exclusive scan over E+1 counts, and the compacted active list (serial in
  // one warp: E+1 <= 1025 entries, 33 steps of a warp scan)
  if (warp == 0) {
    int run = 0, arun = 0, crun = 0;
    for (int base = 0; base <= E; base += 32) {
      int e = base + lane;
      int c = (e <= E) ? cnt[e] : 0;
      int a = (c > 0) ? 1 : 0;
      int nc = chunks ? (c + cap - 1) / cap : 0;
      int incl = c, aincl = a, cincl = nc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        int oa = __shfl_up_sync(0xffffffffu, aincl, off);
        int oc = __shfl_up_sync(0xffffffffu, cincl, off);
        if (lane >= off) {
          incl += o;
          aincl += oa;
          cincl += oc;
        }
      }
      if (e <= E) {
        offsets[e] = run + incl - c;
        cur[e] = run + incl - c;
        cstart[e] = crun + cincl - nc;
        if (a) active[arun + aincl - 1] = e;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      arun += __shfl_sync(0xffffffffu, aincl, 31);
      crun += __shfl_sync(0xffffffffu, cincl, 31);
    }
    if (lane == 0) {
      offsets[E + 1] = run;
      n_active[0] = arun;
      if (chunks) n_tok_chunks[0] = crun;
    }
  }
  __syncthreads();
  if (chunks) {
    // each expert with rows (the shared expert last) cut into ceil(rows / cap)
    // chunks of near-equal size (first row below 2^24, packed with the count)
    for (int e = tid; e <= E; e += blockDim.x) {
      const int Me = cnt[e];
      if (Me <= 0) continue;
      const int nc = (Me + cap - 1) / cap;
      for (int i = 0; i < nc; ++i) {
        const int c0 = (int)((long long)i * Me / nc);
        const int c1 = (int)((long long)(i + 1) * Me / nc);
        chunks[cstart[e] + i] = make_int2(e, (int)((uint32_t)c0 | ((uint32_t)(c1 - c0 - 1) << 24)));
      }
    }
  }
  // stable scatter: one warp walks the pairs in order, 32 at a time
  if (warp == 0) {
    for (int base = 0; base < P; base += 32) {
      int p = base + lane;
      int e = (p < P) ? sid[p] : -1;
      unsigned mask = __match_any_sync(0xffffffffu, e);
      int rank = __popc(mask & ((1u << lane) - 1u));
      int pos = 0;
      if (p < P) pos = cur[e] + rank;
      __syncwarp();
      if (p < P) {
        perm[pos] = p;
        if ((mask >> lane) == 1u) cur[e] += __popc(mask);  // highest lane of the group
      }
      __syncwarp();
    }
  } else if (has_shared) {
    for (int t = tid - 32; t < T; t += blockDim.x - 32) perm[P + t] = P + t;
  }
}

// ---------------------------------------------------------------------------
// Permutation for large T: per-chunk histogram, one-CTA scan, per-chunk
// stable scatter. Chunks are PERM_CHUNK consecutive pairs handled by one warp.
// chunk_cnt is [n_chunks][E] int32 scratch.
// ---------------------------------------------------------------------------
constexpr int PERM_CHUNK = 512;

__global__ void perm_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                                  int32_t* __restrict__ chunk_cnt, int* status) {
  extern __shared__ int32_t cnt[];
  const int c = blockIdx.x;
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  int p0 = c * PERM_CHUNK, p1 = min(P, p0 + PERM_CHUNK);
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    int e = ids[p];
    if (e < 0 || e >= E) {
      record_status(status, QMOE_ERR_DEVICE_ARG);
      e = 0;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) chunk_cnt[(size_t)c * E + i] = cnt[i];
}

// Also builds the tensor-core path's token-chunk list when ``chunks`` is set:
// every expert with rows (the shared expert last) cut into ceil(rows / cap)
// chunks of near-equal size (first row below 2^24, packed with the row count).
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ chunk_cnt,
                                                         int n_chunks, int T, int E, int k,
                                                         int has_shared, int staged,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ perm,
                                                         int32_t* __restrict__ active,
                                                         int32_t* __restrict__ n_active, int cap,
                                                         int2* __restrict__ chunks,
                                                         int32_t* __restrict__ n_tok_chunks) {
  __shared__ int32_t cstart[1025 + 32];
  extern __shared__ int32_t tot[];  // [E+1], then (staged) [n_chunks][E] counts
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* cs = tot + ((E + 1 + 3) & ~3);
  if (staged) {
    // all counts in one coalesced sweep, the scans in shared memory
    for (int i = tid; i < n_chunks * E; i += blockDim.x) cs[i] = chunk_cnt[i];
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
      int run = 0;
      for (int c = 0; c < n_chunks; ++c) {
        const int v = cs[c * E + e];
        cs[c * E + e] = run;
        run += v;
      }
      tot[e] = run;
    }
  } else {
    // per expert: exclusive running sum over chunks (in place), total; the
    // counts are read 8 chunks at a time so that the loads overlap
    for (int e = tid; e < E; e += blockDim.x) {
      int run = 0;
      for (int c0 = 0; c0 < n_chunks; c0 += 8) {
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = c0 + i < n_chunks ? chunk_cnt[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (c0 + i < n_chunks) chunk_cnt[(size_t)(c0 + i) * E + e] = run;
          run += v[i];
        }
      }
      tot[e] = run;
    }
  }
  if (tid == 0) tot[E] = has_shared ? T : 0;
  __syncthreads();
  if (warp == 0) {
    // offsets, active list and (with a chunk list) each expert's first chunk
    int run = 0, arun = 0, crun = 0;
    for (int base = 0; base <= E; base += 32) {
      int e = base + lane;
      int c = (e <= E) ? tot[e] : 0;
      int a = c > 0;
      int nc = chunks ? (c + cap - 1) / cap : 0;
      int incl = c, aincl = a, cincl = nc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        int oa = __shfl_up_sync(0xffffffffu, aincl, off);
        int oc = __shfl_up_sync(0xffffffffu, cincl, off);
        if (lane >= off) {
          incl += o;
          aincl += oa;
          cincl += oc;
        }
      }
      if (e <= E) {
        offsets[e] = run + incl - c;
        cstart[e] = crun + cincl - nc;
        if (a) active[arun + aincl - 1] = e;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      arun += __shfl_sync(0xffffffffu, aincl, 31);
      crun += __shfl_sync(0xffffffffu, cincl, 31);
    }
    if (lane == 0) {
      offsets[E + 1] = run;
      n_active[0] = arun;
      if (chunks) n_tok_chunks[0] = crun;
    }
  }
  __syncthreads();
  if (staged) {
    // the scatter adds each expert's offset itself
    for (int i = tid; i < n_chunks * E; i += blockDim.x) chunk_cnt[i] = cs[i];
  }
  if (chunks) {
    for (int e = tid; e <= E; e += blockDim.x) {
      const int Me = tot[e];
      if (Me <= 0) continue;
      const int nc = (Me + cap - 1) / cap;
      for (int i = 0; i < nc; ++i) {
        // rows [i Me / nc, (i + 1) Me / nc)
        const int c0 = (int)((long long)i * Me / nc);
        const int c1 = (int)((long long)(i + 1) * Me / nc);
        chunks[cstart[e] + i] = make_int2(e, (int)((uint32_t)c0 | ((uint32_t)(c1 - c0 - 1) << 24)));
      }
    }
  }
  const int P = T * k;
  if (has_shared)
    for (int t = tid; t < T; t += blockDim.x) perm[P + t] = P + t;
}

__global__ void perm_scatter_kernel(const int32_t* __restrict__ ids, int P, int E,
                                    const int32_t* __restrict__ chunk_base,
                                    const int32_t* __restrict__ offsets,
                                    int32_t* __restrict__ perm) {
  extern __shared__ int32_t cur[];
  const int c = blockIdx.x, lane = threadIdx.x;
  for (int i = lane; i < E; i += 32) cur[i] = chunk_base[(size_t)c * E + i] + offsets[i];
  __syncwarp();
  int p0 = c * PERM_CHUNK, p1 = min(P, p0 + PERM_CHUNK);
  // the chunk's expert ids, all loads in flight at once
  int ev[PERM_CHUNK / 32];
#pragma unroll
  for (int i = 0; i < PERM_CHUNK / 32; ++i) {
    const int p = p0 + 32 * i + lane;
    ev[i] = p < p1 ? ids[p] : -1;
  }
#pragma unroll
  for (int i = 0; i < PERM_CHUNK / 32; ++i) {
    const int base = p0 + 32 * i;
    if (base >= p1) break;
    int p = base + lane;
    int e = ev[i];
    if (p < p1 && (e < 0 || e >= E)) e = 0;  // already recorded by the count pass
    unsigned mask = __match_any_sync(0xffffffffu, e);
    int rank = __popc(mask & ((1u << lane) - 1u));
    int pos = (p < p1) ? cur[e] + rank : 0;
    __syncwarp();
    if (p < p1) {
      perm[pos] = p;
      if ((mask >> lane) == 1u) cur[e] += __popc(mask);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------
// Rows from which the 128 x 128 register-tiled kernel is used.
constexpr int kRouterGemmRows = 256;

static bool rows_kernel_fits(int T, int H, int E) {
  return T < kRouterGemmRows && E % 8 == 0 && (H == 1024 || H == 2048 || H == 4096);
}

int router_splits(int T, int H, int E) {
  if (rows_kernel_fits(T, H, E)) return 4;  // one partial per quarter of H
  if (router_tc_eligible(T, H, E)) return router_tc_splits(T, H, E);
  // enough CTAs to fill the GPU, at most 8 partials per logit (the top-k
  // kernels add them up)
  const bool big = T >= kRouterGemmRows;
  const int bt = big ? RG_BT : RL_BT, be = big ? RG_BE : RL_BE, bk = big ? RG_BK : RL_BK;
  const int tiles = ((E + be - 1) / be) * ((T + bt - 1) / bt);
  int s = 1;
  while (s < 8 && tiles * s * 2 <= 304 && (H / (s * 2)) % bk == 0 && H / (s * 2) >= 128) s *= 2;
  return s;
}

int router_launches(int T, int H, int E) { return router_tc_eligible(T, H, E) ? 2 : 1; }

cudaError_t launch_router_logits(const float* X, const float* Wr, float* part, int T, int H, int E,
                                 int nsplit, void* wr3, int* status, cudaStream_t st) {
  if (router_tc_eligible(T, H, E) && wr3 != nullptr && nsplit == router_tc_splits(T, H, E))
    return launch_router_tc(X, Wr, part, T, H, E, nsplit, wr3, status, st);
  if (rows_kernel_fits(T, H, E) && nsplit == 4) {
    const int rpt = H / 1024;
    const dim3 grid((E / 8) * 4, (T + rr_rows(rpt) - 1) / rr_rows(rpt));
    if (H == 1024) router_rows_kernel<1><<<grid, 256, 0, st>>>(X, Wr, part, T, H, E);
    else if (H == 2048) router_rows_kernel<2><<<grid, 256, 0, st>>>(X, Wr, part, T, H, E);
    else router_rows_kernel<4><<<grid, 256, 0, st>>>(X, Wr, part, T, H, E);
  } else if (T >= kRouterGemmRows) {
    dim3 grid((E + RG_BE - 1) / RG_BE, (T + RG_BT - 1) / RG_BT, nsplit);
    router_gemm_kernel<<<grid, 256, 0, st>>>(X, Wr, part, T, H, E, H / nsplit);
  } else {
    dim3 grid((E + RL_BE - 1) / RL_BE, (T + RL_BT - 1) / RL_BT, nsplit);
    router_logits_kernel<<<grid, 256, 0, st>>>(X, Wr, part, T, H, E, H / nsplit);
  }
  return cudaGetLastError();
}

template <int EPL>
static cudaError_t topk_dispatch(const float* part, int nsplit, int T, int E, int k, int32_t* ids,
                                 float* w, cudaStream_t st) {
  topk_kernel<EPL><<<(T + 3) / 4, 128, 0, st>>>(part, nsplit, T, E, k, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* part, int nsplit, int T, int E, int k, int32_t* ids, float* w,
                        cudaStream_t st) {
  if (E <= 32) return topk_dispatch<1>(part, nsplit, T, E, k, ids, w, st);
  if (E <= 64) return topk_dispatch<2>(part, nsplit, T, E, k, ids, w, st);
  if (E <= 128) return topk_dispatch<4>(part, nsplit, T, E, k, ids, w, st);
  if (E <= 256) return topk_dispatch<8>(part, nsplit, T, E, k, ids, w, st);
  if (E <= 512) return topk_dispatch<16>(part, nsplit, T, E, k, ids, w, st);
  return topk_dispatch<32>(part, nsplit, T, E, k, ids, w, st);
}

size_t route_small_smem(int T, int E, int k) { return sizeof(int32_t) * (2 * (E + 1) + T * k); }

template <int EPL>
static cudaError_t route_small_dispatch(const float* part, int nsplit, const int32_t* ids_in, int T,
                                        int E, int k, int has_shared, int32_t* ids, float* w,
                                        int32_t* offsets, int32_t* perm, int32_t* active,
                                        int32_t* n_active, int* status, cudaStream_t st, int cap,
                                        int2* chunks, int32_t* n_tok_chunks) {
  size_t smem = route_small_smem(T, E, k);
  route_small_kernel<EPL><<<1, 1024, smem, st>>>(part, nsplit, ids_in, T, E, k, has_shared, ids, w,
                                                 offsets, perm, active, n_active, status, cap, chunks,
                                                 n_tok_chunks);
  return cudaGetLastError();
}

cudaError_t launch_route_small(const float* part, int nsplit, const int32_t* ids_in, int T, int E,
                               int k, int has_shared, int32_t* ids, float* w, int32_t* offsets,
                               int32_t* perm, int32_t* active, int32_t* n_active, int* status,
                               cudaStream_t st, int cap, int2* chunks, int32_t* n_tok_chunks) {
  if (E > 1024 || (chunks != nullptr && cap != 64 && cap != 128 && cap != 192)) return cudaErrorInvalidValue;
#define QMOE_RS(EPL) \
  route_small_dispatch<EPL>(part, nsplit, ids_in, T, E, k, has_shared, ids, w, offsets, perm, \
                            active, n_active, status, st, cap, chunks, n_tok_chunks)
  if (E <= 32) return QMOE_RS(1);
  if (E <= 64) return QMOE_RS(2);
  if (E <= 128) return QMOE_RS(4);
  if (E <= 256) return QMOE_RS(8);
  if (E <= 512) return QMOE_RS(16);
  return QMOE_RS(32);
#undef QMOE_RS
}

int perm_chunks(int P) { return (P + PERM_CHUNK - 1) / PERM_CHUNK; }

cudaError_t launch_perm_large(const int32_t* ids, int T, int E, int k, int has_shared,
                              int32_t* chunk_cnt, int32_t* offsets, int32_t* perm,
                              int32_t* active, int32_t* n_active, int* status, cudaStream_t st, int cap,
                              int2* chunks, int32_t* n_tok_chunks) {
  if (E > 1024 || (chunks != nullptr && cap != 64 && cap != 128 && cap != 192)) return cudaErrorInvalidValue;
  const int P = T * k, nc = perm_chunks(P);
  perm_count_kernel<<<nc, 256, sizeof(int32_t) * E, st>>>(ids, P, E, chunk_cnt, status);
  // the scan stages every chunk count in shared memory when they fit
  const size_t base_smem = sizeof(int32_t) * (size_t)((E + 1 + 3) & ~3);
  const size_t staged_smem = base_smem + sizeof(int32_t) * (size_t)nc * E;
  const int staged = staged_smem <= 160 * 1024 ? 1 : 0;
  const size_t smem = staged ? staged_smem : base_smem;
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(perm_scan_kernel), smem);
  if (e != cudaSuccess) return e;
  perm_scan_kernel<<<1, 1024, smem, st>>>(chunk_cnt, nc, T, E, k, has_shared, staged, offsets, perm, active,
                                          n_active, cap, chunks, n_tok_chunks);
  perm_scatter_kernel<<<nc, 32, sizeof(int32_t) * E, st>>>(ids, P, E, chunk_cnt, offsets, perm);
  return cudaGetLastError();
}

}  // namespace qmoe
