// Decode path (T <= 4 rows): three kernels chained with programmatic dependent
// launch, no host round trip and no separate permutation or combine kernel.
//
// "Distributed CPU: Zip Fusion Beyond Tensor Parallelism", "Decode vs Prefill":
// at one row every packed weight byte is read once, so the layer is bound by
// HBM bandwidth and the question is how little time the HBM pipe sits idle.
// "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "A Separate
// Decode Result Shows Why Axis Choice Matters": with one row the independent
// work is the eight selected routes, merged in selected-slot order.
//
//   K1 router     one CTA per (8 experts, quarter of H): its threads load
//                 their Wr rows' 32 bytes for those experts before waiting on
//                 the previous grid, then reduce x . Wr over the quarter in a
//                 fixed order and write 4 partial logits per (row, expert);
//                 128 CTAs share the 2 MB read.
//   K1b route     one CTA: sums the partials in a fixed order, takes the top-k
//                 by rank, the weights and the ascending list of distinct
//                 selected experts, once for all later CTAs.
//   K2 gate/up    one CTA per (expert slot, 32 intermediate rows). The shared
//                 expert's CTAs start their weight copies before the routing
//                 is known; the others read the routing record and stream
//                 their expert's rows. Output h per (row, slot) pair.
//   K3 down       one CTA per 8 output rows. It reads the routing record,
//                 streams its 8 rows of every selected expert's down matrix
//                 while K2 is still running, then waits for h, and forms
//                 out = R + y_shared + sum_s w_s y_s in slot order.
// Every CTA reaches the same routing decision from the same partials; every
// wait on a copy is bounded and records QMOE_ERR_TIMEOUT on expiry.
#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

constexpr int DEC_THREADS = 256;
constexpr int RT_EPC = 8;  // router: experts per CTA
constexpr int RT_HQ = 4;   // router: parts of H (CTAs per expert group)
constexpr int DEC_FROWS = 32;   // intermediate rows per gate/up CTA
constexpr int DEC_HROWS = 8;    // output rows per down CTA

struct DecodeArgs {
  const float* X;
  const float* R;
  float* out;
  const float* Wr;
  const uint8_t *Wg, *Wu, *Wd, *Sg, *Su, *Sd;
  int T, H, E, k, F, has_shared;
  float* logits;   // [RT_HQ][T][E] partial logits
  float* hbuf;     // [T*k + T][F], indexed by pair (t*k + s; shared T*k + t)
  float* ybuf;     // [T*k + T][H]
  int32_t* ids;    // [T][k]
  float* w;        // [T][k]
  int32_t* route;  // record: [0] n_distinct, [1..] distinct experts (T*k entries)
  int* status;
};

// ---------------------------------------------------------------------------
// routing shared by K2 and K3: logits from the partials (fixed order), top-k
// per row (lower index on ties), distinct selected experts in ascending order.
// ---------------------------------------------------------------------------
struct RouteSmem {
  int32_t ids[4 * 16];
  float w[4 * 16];
  int32_t distinct[4 * 16];
  int32_t n_distinct;
};

// ---------------------------------------------------------------------------
// K1b: routing, once, in one CTA: logits from the 4 partials (fixed order),
// top-k by rank, weights, the ascending list of distinct selected experts.
// The record (ids and w to the workspace, distinct list to ``route``) is read
// by every CTA of the next two kernels.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(DEC_THREADS) decode_route_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* logits = reinterpret_cast<float*>(smem);                       // [T][E]
  int32_t* mark = reinterpret_cast<int32_t*>(logits + (size_t)a.T * a.E);  // [E]
  __shared__ float sel_l[4 * 16];
  __shared__ int32_t sel_e[4 * 16];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, E = a.E, k = a.k;
  tc::grid_dep_wait();  // the router's partials are complete
  tc::grid_dep_launch();
  for (int i = tid; i < T * E; i += DEC_THREADS) {
    float v[RT_HQ];
#pragma unroll
    for (int q = 0; q < RT_HQ; ++q) v[q] = __ldcg(a.logits + (size_t)q * T * E + i);
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < RT_HQ; ++q) sum += v[q];
    logits[i] = (sum == sum) ? sum : -INFINITY;  // NaN sorts last
  }
  for (int e = tid; e < E; e += DEC_THREADS) mark[e] = 0;
  __syncthreads();
  // top-k by rank: the thread of expert e counts the experts that come before
  // it (larger logit first, lower index on ties), stopping once the count
  // reaches k; a count below k is e's slot
  for (int t = 0; t < T; ++t) {
    const float* L = logits + t * E;
    for (int e = tid; e < E; e += DEC_THREADS) {
      const float v = L[e];
      int cnt = 0;
      for (int j0 = 0; j0 < E && cnt < k; j0 += 4) {
        const float4 q = *reinterpret_cast<const float4*>(L + j0);
        cnt += (q.x > v || (q.x == v && j0 < e)) + (q.y > v || (q.y == v && j0 + 1 < e)) +
               (q.z > v || (q.z == v && j0 + 2 < e)) + (q.w > v || (q.w == v && j0 + 3 < e));
      }
      if (cnt < k) {
        sel_e[t * k + cnt] = e;
        sel_l[t * k + cnt] = v;
      }
    }
  }
  __syncthreads();
  if (tid < T * k) {
    const int t = tid / k;
    const float l0 = sel_l[t * k];
    float den = 0.f;
    for (int r = 0; r < k; ++r) den += expf(sel_l[t * k + r] - l0);
    a.ids[tid] = sel_e[tid];
    a.w[tid] = expf(sel_l[tid] - l0) / den;
    mark[sel_e[tid]] = 1;
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int m = (e < E) ? mark[e] : 0;
      const unsigned bal = __ballot_sync(0xffffffffu, m);
      if (m) a.route[1 + run + __popc(bal & ((1u << lane) - 1u))] = e;
      run += __popc(bal);
    }
    if (lane == 0) a.route[0] = run;
  }
}

// Reads the routing record into shared memory (called after the PDL wait that
// makes the routing grid's writes visible).
__device__ void load_route(const DecodeArgs& a, RouteSmem& rs) {
  const int tid = threadIdx.x;
  const int P = a.T * a.k;
  for (int p = tid; p < P; p += DEC_THREADS) {
    rs.ids[p] = __ldcg(a.ids + p);
    rs.w[p] = __ldcg(a.w + p);
  }
  if (tid == 0) rs.n_distinct = __ldcg(a.route);
  __syncthreads();
  for (int i = tid; i < rs.n_distinct; i += DEC_THREADS) rs.distinct[i] = __ldcg(a.route + 1 + i);
  __syncthreads();
}

__device__ __forceinline__ bool wait_copies(uint64_t* bar, int* status) {
  for (uint32_t i = 0; i < tc::kMaxPolls; ++i)
    if (tc::mbar_try_wait(bar, 0)) return true;
  record_status(status, QMOE_ERR_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------------------
// K1: router partial logits. CTA (g, q) owns experts 8g..8g+7 and rows
// [q H/4, (q+1) H/4); thread i loads rows i + 256j of that quarter (32 bytes
// each) before the dependency wait, multiplies them with x after it, and the
// CTA reduces over its 8 warps in a fixed order.
// ---------------------------------------------------------------------------
template <int RPT>  // Wr rows per thread = H / (256 * RT_HQ)
__global__ void __launch_bounds__(DEC_THREADS) decode_router_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* xs = reinterpret_cast<float*>(smem);  // [T][H]
  __shared__ float red[8][4][RT_EPC];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, E = a.E, T = a.T;
  const int e0 = (blockIdx.x / RT_HQ) * RT_EPC, hq = blockIdx.x % RT_HQ;
  const int h0 = hq * (H / RT_HQ);
  float4 w[RPT][2];
#pragma unroll
  for (int j = 0; j < RPT; ++j) {
    const float4* src = reinterpret_cast<const float4*>(a.Wr + (size_t)(h0 + tid + 256 * j) * E + e0);
    w[j][0] = __ldg(src);
    w[j][1] = __ldg(src + 1);
  }
  tc::grid_dep_wait();    // X may come from the previous grid
  tc::grid_dep_launch();
  for (int i = tid; i < T * H / 4; i += DEC_THREADS)
    reinterpret_cast<float4*>(xs)[i] = __ldcg(reinterpret_cast<const float4*>(a.X) + i);
  __syncthreads();
  for (int t = 0; t < T; ++t) {
    float acc[RT_EPC] = {};
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const float x = xs[t * H + h0 + tid + 256 * j];
      acc[0] = fmaf(x, w[j][0].x, acc[0]);
      acc[1] = fmaf(x, w[j][0].y, acc[1]);
      acc[2] = fmaf(x, w[j][0].z, acc[2]);
      acc[3] = fmaf(x, w[j][0].w, acc[3]);
      acc[4] = fmaf(x, w[j][1].x, acc[4]);
      acc[5] = fmaf(x, w[j][1].y, acc[5]);
      acc[6] = fmaf(x, w[j][1].z, acc[6]);
      acc[7] = fmaf(x, w[j][1].w, acc[7]);
    }
#pragma unroll
    for (int q = 0; q < RT_EPC; ++q) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], off);
    }
    if (lane == 0)
#pragma unroll
      for (int q = 0; q < RT_EPC; ++q) red[warp][t][q] = acc[q];
  }
  __syncthreads();
  if (tid < T * RT_EPC) {
    const int t = tid / RT_EPC, q = tid % RT_EPC;
    float s2 = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) s2 += red[w8][t][q];
    if (e0 + q < E) a.logits[((size_t)hq * T + t) * E + e0 + q] = s2;
  }
}

// ---------------------------------------------------------------------------
// K2: gate/up + SwiGLU for one (expert slot, 32 intermediate rows). The rows
// arrive in 4 stages of 8 gate + 8 up rows, each on its own mbarrier, so the
// warps compute a stage while the next ones stream in. Warp w owns gate row
// 8s+w and up row 8s+w of stage s and produces h for that row itself.
// ---------------------------------------------------------------------------
constexpr int DEC_STAGES = 4;

template <int NSUB, int QT>
__device__ __forceinline__ float row_dot_warp(const uint8_t* row, const float (&xv)[NSUB / 32 > 0 ? NSUB / 32 : 1][32],
                                              const float (&xs)[NSUB / 32 > 0 ? NSUB / 32 : 1], int lane) {
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  constexpr int SL = NSUB / 32;
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < SL; ++j) {
    const int c = lane + 32 * j;
    const uint8_t* blk = row + (size_t)(c >> 3) * BYTES;
    const int sj = c & 7;
    const uint4 hv = *reinterpret_cast<const uint4*>(blk);
    KHeader hd;
    const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
    hd.d = dd.x;
    hd.dmin = dd.y;
    hd.f0 = hv.y;
    hd.f1 = hv.z;
    hd.f2 = hv.w;
    const uint4 qv = *reinterpret_cast<const uint4*>(blk + quant_offset(QT, sj));
    const uint32_t hb = QT == QMOE_Q5K ? *reinterpret_cast<const uint32_t*>(blk + 16 + 4 * sj) : 0u;
    acc += sub_contrib(dot_sub_prmt<QT>(qv, hb, xv[j]), xs[j], sub_scale(hd, sj));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

template <int NSUB, int QT>
__global__ void __launch_bounds__(DEC_THREADS) decode_gateup_kernel(DecodeArgs a) {
  static_assert(NSUB >= 32, "decode gate/up needs H >= 1024");
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar[DEC_STAGES];
  __shared__ RouteSmem rs;
  __shared__ int32_t pairs[4];
  __shared__ int32_t n_pairs;
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  constexpr int H = NSUB * SUBK;
  constexpr int SL = NSUB / 32;
  constexpr int RPS = DEC_FROWS / DEC_STAGES;  // gate rows (and up rows) per stage: 8
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int F = a.F, T = a.T, k = a.k, E = a.E;
  const int FCH = F / DEC_FROWS;
  const int slot = blockIdx.x / FCH, fc = blockIdx.x % FCH;
  constexpr size_t row_bytes = (size_t)(H / QK) * BYTES;
  constexpr uint32_t stage_rows_bytes = (uint32_t)(RPS * row_bytes);
  uint8_t* wgs = smem;                                   // 32 gate rows
  uint8_t* wus = smem + DEC_FROWS * row_bytes;           // 32 up rows
  const bool is_shared = a.has_shared && slot == 0;
  if (tid == 0) {
    for (int i = 0; i < DEC_STAGES; ++i) tc::mbar_init(&bar[i], 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  // warp 0 issues the 8 copies (4 stages x gate/up) from 8 lanes, after lanes
  // 0..3 have set each stage's expected byte count
  auto issue = [&](const uint8_t* gsrc, const uint8_t* usrc) {
    if (lane < DEC_STAGES) tc::mbar_expect_tx(&bar[lane], 2 * stage_rows_bytes);
    __syncwarp();
    if (lane < 2 * DEC_STAGES) {
      const int st = lane >> 1;
      const uint8_t* src = (lane & 1) ? usrc : gsrc;
      uint8_t* dst = (lane & 1) ? wus : wgs;
      tc::bulk_g2s(dst + st * stage_rows_bytes, src + st * stage_rows_bytes, stage_rows_bytes, &bar[st]);
    }
  };
  const size_t chunk_off = (size_t)fc * DEC_FROWS * row_bytes;
  if (is_shared && warp == 0) issue(a.Sg + chunk_off, a.Su + chunk_off);
  tc::grid_dep_wait();     // the routing record (and X) are complete
  tc::grid_dep_launch();
  load_route(a, rs);
  int e = a.E;  // shared
  if (!is_shared) {
    const int ri = slot - a.has_shared;
    if (ri >= rs.n_distinct) return;  // this CTA issued no copies
    e = rs.distinct[ri];
    if (warp == 0) {
      const size_t eoff = (size_t)e * F * row_bytes + chunk_off;
      issue(a.Wg + eoff, a.Wu + eoff);
    }
  }
  if (tid == 0) {
    int n = 0;
    for (int t = 0; t < T; ++t) {
      if (is_shared) {
        pairs[n++] = T * k + t;
      } else {
        for (int s2 = 0; s2 < k; ++s2)
          if (rs.ids[t * k + s2] == e) pairs[n++] = t * k + s2;
      }
    }
    n_pairs = n;
  }
  __syncthreads();
  const int np = n_pairs;
  // one row (pair) at a time: lane l holds the activations of sub-blocks
  // l + 32j; the stages are waited in order (a completed stage stays complete)
  for (int pi = 0; pi < np; ++pi) {
    const int pair = pairs[pi];
    const int t = pair < T * k ? pair / k : pair - T * k;
    float xv[SL][32];
    float xs[SL];
#pragma unroll
    for (int j = 0; j < SL; ++j) {
      const float4* x4 = reinterpret_cast<const float4*>(a.X + (size_t)t * H + (lane + 32 * j) * SUBK);
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(x4 + i);
        xv[j][4 * i] = v.x;
        xv[j][4 * i + 1] = v.y;
        xv[j][4 * i + 2] = v.z;
        xv[j][4 * i + 3] = v.w;
        sum += (v.x + v.y) + (v.z + v.w);
      }
      xs[j] = sum;
    }
    for (int st = 0; st < DEC_STAGES; ++st) {
      if (!wait_copies(&bar[st], a.status)) return;
      const int r = st * RPS + warp;  // row within the 32-row chunk
      const float g = row_dot_warp<NSUB, QT>(wgs + (size_t)r * row_bytes, xv, xs, lane);
      const float u = row_dot_warp<NSUB, QT>(wus + (size_t)r * row_bytes, xv, xs, lane);
      if (lane == 0) a.hbuf[(size_t)pair * F + fc * DEC_FROWS + r] = silu_mul(g, u);
    }
  }
}

// ---------------------------------------------------------------------------
// K3: down projection of 8 output rows for every selected expert and the
// shared expert, then the slot-order combine with the residual. Warp w owns
// output row r0 + w; lanes split a row's sub-blocks (G lanes per pair, 32/G
// pairs per pass).
// ---------------------------------------------------------------------------
template <int NSUBD, int QT>
__global__ void __launch_bounds__(DEC_THREADS) decode_down_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ RouteSmem rs;
  __shared__ int32_t slot_of[4 * 16 + 4];
  __shared__ float ys[(4 * 16 + 4) * DEC_HROWS];
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  constexpr int F = NSUBD * SUBK;
  constexpr int G = NSUBD < 32 ? NSUBD : 32;  // lanes per (pair, row)
  constexpr int PPP = 32 / G;                 // pairs per pass
  constexpr int SL = NSUBD / G;               // sub-blocks per lane
  constexpr size_t row_bytes = (size_t)(F / QK) * BYTES;
  constexpr uint32_t blk_bytes = (uint32_t)(DEC_HROWS * row_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, T = a.T, k = a.k, E = a.E;
  const int r0 = blockIdx.x * DEC_HROWS;
  const int maxx = T * k + 1;  // experts incl. shared
  const int P = T * k + (a.has_shared ? T : 0);
  // h rows are staged with each 32-float sub-block padded to 36 floats, so
  // that the 8 lanes of a quarter-warp reading 8 different sub-blocks of a row
  // hit 8 different bank groups
  constexpr int HSTRIDE = NSUBD * 36;
  uint8_t* wsm = smem;                                                       // [maxx][8 rows]
  float* hs = reinterpret_cast<float*>(smem + (size_t)maxx * blk_bytes);    // [P][NSUBD][36]
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  // the routing grid completed before the gate/up grid let this one launch
  load_route(a, rs);
  const int nd = rs.n_distinct;
  if (warp == 0) {
    // one copy per lane: 8 rows of every selected expert's down matrix, and
    // of the shared expert's
    const int nx = nd + (a.has_shared ? 1 : 0);
    if (lane == 0) tc::mbar_expect_tx(&bar, nx * blk_bytes);
    __syncwarp();
    for (int i = lane; i < nx; i += 32) {
      const uint8_t* src = i < nd ? a.Wd + ((size_t)rs.distinct[i] * H + r0) * row_bytes : a.Sd + (size_t)r0 * row_bytes;
      tc::bulk_g2s(wsm + (size_t)i * blk_bytes, src, blk_bytes, &bar);
    }
  }
  for (int p = tid; p < P; p += DEC_THREADS) {
    int sl = nd;  // shared
    if (p < T * k) {
      const int e = rs.ids[p];
      for (int i = 0; i < nd; ++i)
        if (rs.distinct[i] == e) sl = i;
    }
    slot_of[p] = sl;
  }
  tc::grid_dep_wait();     // h from the gate/up grid is complete
  tc::grid_dep_launch();
  for (int i = tid; i < P * F / 4; i += DEC_THREADS) {
    const int p = i / (F / 4), rem = i % (F / 4);
    reinterpret_cast<float4*>(hs + (size_t)p * HSTRIDE + (rem >> 3) * 36)[rem & 7] =
        __ldcg(reinterpret_cast<const float4*>(a.hbuf) + i);
  }
  __syncthreads();
  if (!wait_copies(&bar, a.status)) return;

  const int row = warp;  // 8 warps, 8 rows
  const int sub_lane = lane % G, pair_lane = lane / G;
  for (int p0 = 0; p0 < P; p0 += PPP) {
    const int p = p0 + pair_lane;
    float acc = 0.f;
    if (p < P) {
      const uint8_t* rowp = wsm + (size_t)slot_of[p] * blk_bytes + (size_t)row * row_bytes;
#pragma unroll
      for (int j = 0; j < SL; ++j) {
        const int c = sub_lane + G * j;
        const uint8_t* blk = rowp + (size_t)(c >> 3) * BYTES;
        const int sj = c & 7;
        const uint4 hv = *reinterpret_cast<const uint4*>(blk);
        KHeader hd;
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
        hd.d = dd.x;
        hd.dmin = dd.y;
        hd.f0 = hv.y;
        hd.f1 = hv.z;
        hd.f2 = hv.w;
        const uint4 qv = *reinterpret_cast<const uint4*>(blk + quant_offset(QT, sj));
        const uint32_t hb = QT == QMOE_Q5K ? *reinterpret_cast<const uint32_t*>(blk + 16 + 4 * sj) : 0u;
        const float4* x4 = reinterpret_cast<const float4*>(hs + (size_t)p * HSTRIDE + c * 36);
        float xv[32], xsum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v = x4[i];
          xv[4 * i] = v.x;
          xv[4 * i + 1] = v.y;
          xv[4 * i + 2] = v.z;
          xv[4 * i + 3] = v.w;
          xsum += (v.x + v.y) + (v.z + v.w);
        }
        acc += sub_contrib(dot_sub_prmt<QT>(qv, hb, xv), xsum, sub_scale(hd, sj));
      }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub_lane == 0 && p < P) {
      ys[p * DEC_HROWS + row] = acc;
      a.ybuf[(size_t)p * H + r0 + row] = acc;
    }
  }
  __syncthreads();
  for (int tr = tid; tr < T * DEC_HROWS; tr += DEC_THREADS) {
    const int t = tr / DEC_HROWS, r = tr % DEC_HROWS;
    float acc = a.R ? a.R[(size_t)t * H + r0 + r] : 0.f;
    if (a.has_shared) acc += ys[(T * k + t) * DEC_HROWS + r];
    for (int s2 = 0; s2 < k; ++s2) acc = fmaf(rs.w[t * k + s2], ys[(t * k + s2) * DEC_HROWS + r], acc);
    a.out[(size_t)t * H + r0 + r] = acc;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t router_smem(int T, int H) { return sizeof(float) * (size_t)T * H; }

static size_t gateup_smem(int T, int H, int E, int qt) {
  const size_t row_bytes = (size_t)(H / QK) * qtype_bytes(qt);
  return 2 * DEC_FROWS * row_bytes;
}

static size_t route_smem(int T, int E) { return sizeof(float) * (size_t)T * E + sizeof(int32_t) * E; }

static size_t down_smem(int T, int E, int F, int k, int qt) {
  const size_t row_bytes = (size_t)(F / QK) * qtype_bytes(qt);
  const int P = T * k + T;
  return (size_t)(T * k + 1) * DEC_HROWS * row_bytes + sizeof(float) * (size_t)P * (F / SUBK) * 36;
}

bool decode_path_supported(int T, int H, int E, int k, int F, int gate_qt, int down_qt) {
  if (T < 1 || T > 4 || k > 8) return false;
  if (H != 1024 && H != 2048 && H != 4096) return false;
  if (F != 256 && F != 512 && F != 1024 && F != 2048) return false;
  if (E % RT_EPC != 0) return false;
  if (router_smem(T, H) > 200 * 1024) return false;
  if (gateup_smem(T, H, E, gate_qt) > 200 * 1024) return false;
  if (down_smem(T, E, F, k, down_qt) > 200 * 1024) return false;
  return true;
}

// The three kernels run concurrently: each asks for the largest shared-memory
// carveout so that CTAs of different kernels can share an SM.
static cudaError_t prepare_kernel(const void* fn, size_t smem) { return ensure_kernel_smem(fn, smem, 100); }

template <typename K>
static cudaError_t launch_pdl(K kernel, int grid, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  cudaError_t pe = prepare_kernel(reinterpret_cast<const void*>(kernel), smem);
  if (pe != cudaSuccess) return pe;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(DEC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int NSUB>
static cudaError_t launch_gateup_t(int qt, int grid, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  return qt == QMOE_Q5K ? launch_pdl(decode_gateup_kernel<NSUB, QMOE_Q5K>, grid, smem, st, a)
                        : launch_pdl(decode_gateup_kernel<NSUB, QMOE_Q4K>, grid, smem, st, a);
}

template <int NSUBD>
static cudaError_t launch_down_t(int qt, int grid, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  return qt == QMOE_Q5K ? launch_pdl(decode_down_kernel<NSUBD, QMOE_Q5K>, grid, smem, st, a)
                        : launch_pdl(decode_down_kernel<NSUBD, QMOE_Q4K>, grid, smem, st, a);
}

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t st) {
  DecodeArgs a{};
  a.X = L.X; a.R = L.R; a.out = L.out; a.Wr = L.Wr;
  a.Wg = L.Wg; a.Wu = L.Wu; a.Wd = L.Wd; a.Sg = L.Sg; a.Su = L.Su; a.Sd = L.Sd;
  a.T = L.T; a.H = L.H; a.E = L.E; a.k = L.k; a.F = L.F; a.has_shared = L.Sg != nullptr;
  a.logits = L.part; a.hbuf = L.hbuf; a.ybuf = L.ybuf; a.ids = L.ids; a.w = L.w; a.route = L.route;
  a.status = L.status;
  const int g1 = (L.E / RT_EPC) * RT_HQ;
  const size_t s1 = router_smem(L.T, L.H);
  cudaError_t e;
  switch (L.H) {
    case 1024: e = launch_pdl(decode_router_kernel<1>, g1, s1, st, a); break;
    case 2048: e = launch_pdl(decode_router_kernel<2>, g1, s1, st, a); break;
    case 4096: e = launch_pdl(decode_router_kernel<4>, g1, s1, st, a); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(decode_route_kernel, 1, route_smem(L.T, L.E), st, a)) != cudaSuccess) return e;
  const int slots = a.has_shared + (L.T * L.k < L.E ? L.T * L.k : L.E);
  const int g2 = slots * (L.F / DEC_FROWS);
  const size_t s2 = gateup_smem(L.T, L.H, L.E, L.gate_qt);
  switch (L.H) {
    case 1024: e = launch_gateup_t<32>(L.gate_qt, g2, s2, st, a); break;
    case 2048: e = launch_gateup_t<64>(L.gate_qt, g2, s2, st, a); break;
    case 4096: e = launch_gateup_t<128>(L.gate_qt, g2, s2, st, a); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  const size_t s3 = down_smem(L.T, L.E, L.F, L.k, L.down_qt);
  const int g3 = L.H / DEC_HROWS;
  switch (L.F) {
    case 256: return launch_down_t<8>(L.down_qt, g3, s3, st, a);
    case 512: return launch_down_t<16>(L.down_qt, g3, s3, st, a);
    case 1024: return launch_down_t<32>(L.down_qt, g3, s3, st, a);
    case 2048: return launch_down_t<64>(L.down_qt, g3, s3, st, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmoe
