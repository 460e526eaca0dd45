// Decode path (T <= 4 rows): a router kernel and one persistent expert
// kernel, chained with programmatic dependent launch.
//
// "Distributed CPU: Zip Fusion Beyond Tensor Parallelism", "Decode vs Prefill:
// Same Weights, Different Bottlenecks": at a few rows every packed weight byte
// is read once and the layer is bound by HBM bandwidth, so the question is how
// little time the HBM pipe sits idle. "CKE Zip: From Splitting Tokens To
// Splitting Qwen3.5 Weights", "A Separate Decode Result Shows Why Axis Choice
// Matters": with one row the independent work is the selected routes, merged
// in selected-slot order.
//
//   K1 router   one CTA per (8 experts, quarter of H): its threads load their
//               Wr rows' 32 bytes for those experts before waiting on the
//               previous grid, then reduce x . Wr over the quarter in a fixed
//               order and write 4 partial logits per (row, expert).
//   K2 experts  one CTA per SM (cooperative launch: every CTA is resident),
//               12 warps. Gate/up work units are (expert slot, intermediate
//               row f), a gate row and an up row each, cut into equal shares
//               of all SMs. The shared expert's units are known before
//               routing, so each CTA starts their copies before it waits for
//               the router; then every CTA takes the top-k itself from the
//               router's partials (the same fixed-order arithmetic everywhere,
//               so every CTA reaches the same decision) and copies its share
//               of the routed experts' rows through a ring of bulk copies
//               (cp.async.bulk + mbarrier), and its block of about H / SMs
//               output rows of every selected expert's down matrix through a
//               second ring. Each warp works through its own units, waiting
//               only on the copies it needs; the last warp done with a ring
//               stage refills it. A unit writes h = silu(x.g) * (x.u) per
//               (row, slot) pair; a CTA done with its units adds their count
//               to a counter. The down phase waits until the counter reaches
//               (slots) F (all of h), stages h, computes y for
//               its output rows and every pair, and forms
//               out = R + y_shared + sum_s w_s y_s for those rows in slot
//               order.
// Every wait (copies, counters) gives up after a bounded time, records
// QMOE_ERR_TIMEOUT and leaves the CTA with no copy in flight.
#include <atomic>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

constexpr int RT_THREADS = 256;
constexpr int RT_EPC = 8;  // router: experts per CTA
constexpr int RT_HQ = 4;   // router: parts of H (CTAs per expert group)

// threads of the expert kernel: 12 warps at one or two rows, 16 above (more
// warps hide more of the longer down phase; at one row the twelve-warp CTA
// starts its routed copies sooner, measured 22.0 against 25.5 us)
constexpr int DX_MAX_THREADS = 512;
__host__ __device__ constexpr int dx_threads(int T) { return T <= 2 ? 384 : 512; }
constexpr int DX_UPS = 8;        // gate/up units per ring stage
constexpr int DX_NSTG = 4;       // gate/up ring stages
constexpr int DD_MAXROWS = 16;   // output rows of a CTA (at most)
constexpr int DD_NST = 12;       // down ring stages (a CTA's rows of one slot each)
constexpr int DX_MAXT = 4;
constexpr int DX_MAXK = 16;
constexpr int DX_MAXSLOT = DX_MAXT * DX_MAXK + 1;

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
  int* sync;       // [1] h rows done (all slots), cleared by the router kernel
  int* status;
  unsigned long long wait_ns;  // a wait gives up after this many nanoseconds
  int fault;                   // test-only: 1 = the first CTA withholds the copy of its last slot's down rows
};

// ---------------------------------------------------------------- waits

__device__ __forceinline__ uint64_t gtime() { return tc::global_ns(); }

// Waits for the phase of ``parity`` of ``bar``; false after ``limit`` ns.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, uint64_t limit) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0 && gtime() - t0 > limit) return false;
  }
}

// ---------------------------------------------------------------- arithmetic

__device__ __forceinline__ float sum2(uint64_t v) {
  const float2 f = unpack2(v);
  return f.x + f.y;
}

// S = sum over the 8 NW weights of ``w`` of (0.5 + q_i/256) * x_i. Word n
// holds weights 8n..8n+7 (byte b: weight 8n+2b in the low nibble, 8n+2b+1 in
// the high one); for Q5_K bit i of ``hb`` is weight i's fifth bit. Each quant
// is placed by one byte permute into the mantissa of a float whose exponent
// makes it 0.5 + q/256 exactly (no int->float conversion); the activation
// pairs x2[4n+b] = (x_{8n+2b}, x_{8n+2b+1}) feed two accumulators (even and
// odd weights), added at the end.
template <int QT, int NW>
__device__ __forceinline__ float dot_words(const uint32_t* w, uint32_t hb, const uint64_t* x2) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int n = 0; n < NW; ++n) {
    uint32_t ev = w[n] & 0x0F0F0F0Fu;
    uint32_t od = (w[n] >> 4) & 0x0F0F0F0Fu;
    if (QT == QMOE_Q5K) {
      ev |= spread4(hb >> (8 * n), 0);
      od |= spread4(hb >> (8 * n), 1);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t sel = 0x7044u | ((uint32_t)b << 8);
      const float2 x = unpack2(x2[4 * n + b]);
      a0 = fmaf(__uint_as_float(__byte_perm(ev, 0x3F000000u, sel)), x.x, a0);
      a1 = fmaf(__uint_as_float(__byte_perm(od, 0x3F000000u, sel)), x.y, a1);
    }
  }
  return a0 + a1;
}

__device__ __forceinline__ KHeader header_of(const uint4 hv) {
  KHeader hd;
  const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
  hd.d = dd.x;
  hd.dmin = dd.y;
  hd.f0 = hv.y;
  hd.f1 = hv.z;
  hd.f2 = hv.w;
  return hd;
}

// x . row for one packed row of H = 1024 SL weights in shared memory: lane l
// takes sub-blocks l + 32 j, whose activations it holds in ``x2`` (pairs) and
// their sums in ``xs``; the warp adds the lanes in a fixed butterfly order.
template <int SL, int QT>
__device__ __forceinline__ float gate_row_dot(const uint8_t* row, const uint64_t (&x2)[SL][16], const float (&xs)[SL],
                                              int lane) {
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < SL; ++j) {
    const int c = lane + 32 * j;
    const uint8_t* blk = row + (size_t)(c >> 3) * BYTES;
    const int sj = c & 7;
    const KHeader hd = header_of(*reinterpret_cast<const uint4*>(blk));
    const uint4 qv = *reinterpret_cast<const uint4*>(blk + quant_offset(QT, sj));
    const uint32_t hb = QT == QMOE_Q5K ? *reinterpret_cast<const uint32_t*>(blk + 16 + 4 * sj) : 0u;
    const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
    acc += sub_contrib(dot_words<QT, 4>(w, hb, x2[j]), xs[j], sub_scale(hd, sj));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

// Shared-memory staging of the activations with 2 floats of padding after
// every sub-block of 32: a lane reading its sub-block's 32 consecutive values
// then sits on banks distinct from its neighbours', so a warp's 8-byte loads
// take two wavefronts instead of 32.
template <int G>
__device__ __forceinline__ int padded(int f) { return f + 2 * (f / G); }

// Down rows: lane l takes sub-block l % FSUB (32 weights) of row l / FSUB of
// the warp's current group of 32 / FSUB rows, so a warp pass covers 2 rows
// (F = 512) or 4 (F = 256). The lane's activations are the same for every row
// it visits, so it holds them in registers (``h2``, pairs, and their sum),
// read from the padded staging of h.
template <int FSUB>
__device__ __forceinline__ float load_down_h(const float* h, int lane, uint64_t (&h2)[16]) {
  const uint64_t* src = reinterpret_cast<const uint64_t*>(h + padded<32>((lane % FSUB) * 32));
  float hs = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    h2[i] = src[i];
    hs += sum2(h2[i]);
  }
  return hs;
}

// h . row for this lane's sub-block of ``row``, reduced over the FSUB lanes of
// the row (the first lane of each row's group holds the sum).
template <int FSUB, int QT>
__device__ __forceinline__ float down_row_dot(const uint8_t* row, const uint64_t (&h2)[16], float hs, int lane) {
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  const int c = lane % FSUB;
  const uint8_t* blk = row + (size_t)(c >> 3) * BYTES;
  const int sj = c & 7;
  const KHeader hd = header_of(*reinterpret_cast<const uint4*>(blk));
  const uint4 qv = *reinterpret_cast<const uint4*>(blk + quant_offset(QT, sj));
  const uint32_t hb = QT == QMOE_Q5K ? *reinterpret_cast<const uint32_t*>(blk + 16 + 4 * sj) : 0u;
  const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
  float acc = sub_contrib(dot_words<QT, 4>(w, hb, h2), hs, sub_scale(hd, sj));
#pragma unroll
  for (int off = FSUB / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

// Selection key of (logit v, expert e): larger logit first, the lower index
// among equal logits; an order-preserving map of the float's bits (v is never
// NaN here; -0 is taken as +0, which it equals) above the complemented index.
__device__ __forceinline__ uint64_t sel_key(float v, int e) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint32_t)(~e);
}

__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Sorts a bitonic sequence of KMAX keys into descending order.
template <int KMAX>
__device__ __forceinline__ void bitonic_desc(uint64_t (&v)[KMAX]) {
#pragma unroll
  for (int d = KMAX / 2; d > 0; d >>= 1)
#pragma unroll
    for (int i = 0; i < KMAX; ++i)
      if ((i & d) == 0) cas_desc(v[i], v[i + d]);
}

// Sorts KMAX keys into descending order (a bitonic sorting network: depth
// log2(KMAX) (log2(KMAX) + 1) / 2, the compare-exchanges of a stage independent).
template <int KMAX>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t (&v)[KMAX]) {
#pragma unroll
  for (int size = 2; size <= KMAX; size <<= 1)
#pragma unroll
    for (int d = size / 2; d > 0; d >>= 1)
#pragma unroll
      for (int i = 0; i < KMAX; ++i) {
        const int j = i ^ d;
        if (j > i) {
          if ((i & size) == 0) cas_desc(v[i], v[j]);  // a descending run
          else cas_desc(v[j], v[i]);                  // an ascending run
        }
      }
}

// The k best experts of one row of E logits (L, shared memory), in selection
// order, into sel_e / sel_l; one warp, KMAX >= k a power of two. Each lane
// sorts groups of KMAX of its experts and keeps the best KMAX seen.
template <int KMAX>
__device__ __forceinline__ void warp_topk(const float* L, int E, int k, int lane, int32_t* sel_e, float* sel_l) {
  uint64_t top[KMAX];
#pragma unroll
  for (int i = 0; i < KMAX; ++i) top[i] = 0;  // below every key
  for (int e0 = 0; e0 < E; e0 += 32 * KMAX) {
    uint64_t g[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) {
      const int e = e0 + lane + 32 * i;
      g[i] = e < E ? sel_key(L[e], e) : 0;
    }
    bitonic_sort_desc<KMAX>(g);
    // the best KMAX of top and g: a bitonic sequence, then sorted
#pragma unroll
    for (int i = 0; i < KMAX; ++i) top[i] = top[i] > g[KMAX - 1 - i] ? top[i] : g[KMAX - 1 - i];
    bitonic_desc<KMAX>(top);
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    uint64_t other[KMAX];
#pragma unroll
    for (int i = 0; i < KMAX; ++i) other[i] = __shfl_xor_sync(0xffffffffu, top[i], m);
#pragma unroll
    for (int i = 0; i < KMAX; ++i) top[i] = top[i] > other[KMAX - 1 - i] ? top[i] : other[KMAX - 1 - i];
    bitonic_desc<KMAX>(top);
  }
  if (lane < k) {
    uint64_t mine = top[0];
#pragma unroll
    for (int i = 1; i < KMAX; ++i)
      if (lane == i) mine = top[i];
    const int e = (int)(~(uint32_t)mine);
    sel_e[lane] = e;
    sel_l[lane] = L[e];
  }
}

// ---------------------------------------------------------------------------
// K1: router partial logits. CTA (g, q) owns experts 8g..8g+7 and rows
// [q H/4, (q+1) H/4); thread i loads rows i + 256j of that quarter (32 bytes
// each) before the dependency wait, multiplies them with x after it, and the
// CTA reduces over its 8 warps in a fixed order. CTA 0 clears the expert
// kernel's counters (after the wait: the previous expert kernel, which used
// them, has completed).
// ---------------------------------------------------------------------------
template <int RPT>  // Wr rows per thread = H / (256 * RT_HQ)
__global__ void __launch_bounds__(RT_THREADS) decode_router_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* xs = reinterpret_cast<float*>(smem);  // [T][H]
  __shared__ float red[8][DX_MAXT][RT_EPC];
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
  if (blockIdx.x == 0 && tid == 0) a.sync[0] = 0;
  for (int i = tid; i < T * H / 4; i += RT_THREADS)
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
// Routing, taken by every CTA of K2 and K3 from the router's partials.
// ---------------------------------------------------------------------------
struct RouteState {
  float sel_l[DX_MAXT * DX_MAXK];
  int32_t sel_e[DX_MAXT * DX_MAXK];
  float wts[DX_MAXT * DX_MAXK];
  int32_t slot_e[DX_MAXSLOT];            // expert of each slot (E = shared)
  int32_t pair_of[DX_MAXSLOT][DX_MAXT];  // pair index of (slot, row), -1 if the row does not use the slot
  int32_t n_slots;
};

// Logits from the 4 partials in a fixed order (NaN is mapped to -inf, so it
// ranks after every number and among equals by index); the top-k of row t in
// warp t (T <= 4 warps); the weights; slots: the shared expert first, then the
// distinct selected experts in ascending order; the pair index of every
// (slot, row). ``lg`` is scratch of T E + E floats. Ends with the block
// synchronised. CTA 0 of K2 writes ids and w to the workspace.
__device__ void decode_route(const DecodeArgs& a, RouteState& S, float* lg, int nthreads, bool write_ids) {
  const int T = a.T, k = a.k, E = a.E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < T * E; i += nthreads) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < RT_HQ; ++q) v += __ldcg(a.logits + (size_t)q * T * E + i);
    lg[i] = (v == v) ? v : -INFINITY;
  }
  __syncthreads();
  // top-k: every expert gets a 64-bit key that orders as the selection does
  // (larger logit first, then the lower index); each lane keeps the best KMAX
  // keys of its experts in a sorted list, and five butterfly steps merge the
  // lanes' lists, each keeping the best KMAX of two
  if (warp < T) {
    if (k <= 8) warp_topk<8>(lg + warp * E, E, k, lane, S.sel_e + warp * k, S.sel_l + warp * k);
    else warp_topk<16>(lg + warp * E, E, k, lane, S.sel_e + warp * k, S.sel_l + warp * k);
  }
  if (T == 1) {
    // one row: the k selected experts are the routed slots; warp 0 takes the
    // weights (the same arithmetic as below), the slot of each expert (its
    // rank by index among the selected) and the pair indices
    if (warp == 0) {
      __syncwarp();
      const bool sel = lane < k;
      const int e = sel ? S.sel_e[lane] : 0x7fffffff;
      float w = 0.f;
      if (lane == 0) {
        const float l0 = S.sel_l[0];
        float den = 0.f;
        for (int r = 0; r < k; ++r) den += expf(S.sel_l[r] - l0);
        w = den;
      }
      const float den = __shfl_sync(0xffffffffu, w, 0);
      int rank = 0;
      for (int j = 0; j < k; ++j) rank += __shfl_sync(0xffffffffu, e, j) < e;
      const int hs = a.has_shared;
      if (sel) {
        const float ws = expf(S.sel_l[lane] - S.sel_l[0]) / den;
        S.wts[lane] = ws;
        if (write_ids) {
          a.ids[lane] = e;
          a.w[lane] = ws;
        }
        S.slot_e[hs + rank] = e;
        S.pair_of[hs + rank][0] = lane;
#pragma unroll
        for (int t = 1; t < DX_MAXT; ++t) S.pair_of[hs + rank][t] = -1;
      }
      if (lane == 0) {
        if (hs) {
          S.slot_e[0] = E;
          S.pair_of[0][0] = k;  // the shared expert's pair of row 0: T k + 0
#pragma unroll
          for (int t = 1; t < DX_MAXT; ++t) S.pair_of[0][t] = -1;
        }
        S.n_slots = k + hs;
      }
    }
    __syncthreads();
    return;
  }
  __syncthreads();
  int* mark = reinterpret_cast<int*>(lg + T * E);  // [E], after the logits
  for (int e = tid; e < E; e += nthreads) mark[e] = 0;
  if (tid < T * k) {
    const int t = tid / k;
    const float l0 = S.sel_l[t * k];
    float den = 0.f;
    for (int r = 0; r < k; ++r) den += expf(S.sel_l[t * k + r] - l0);
    S.wts[tid] = expf(S.sel_l[tid] - l0) / den;
    if (write_ids) {
      a.ids[tid] = S.sel_e[tid];
      a.w[tid] = S.wts[tid];
    }
  }
  __syncthreads();
  if (tid < T * k) mark[S.sel_e[tid]] = 1;
  __syncthreads();
  if (warp == 0) {
    int run = a.has_shared;
    if (a.has_shared && lane == 0) S.slot_e[0] = E;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int m = (e < E) ? mark[e] : 0;
      const unsigned bal = __ballot_sync(0xffffffffu, m);
      if (m) S.slot_e[run + __popc(bal & ((1u << lane) - 1u))] = e;
      run += __popc(bal);
    }
    if (lane == 0) S.n_slots = run;
  }
  __syncthreads();
  const int ns = S.n_slots;
  for (int i = tid; i < ns * DX_MAXT; i += nthreads) {
    const int u = i / DX_MAXT, t = i % DX_MAXT;
    int p = -1;
    if (t < T) {
      const int e = S.slot_e[u];
      if (e == E) {
        p = T * k + t;
      } else {
        for (int s2 = 0; s2 < k; ++s2)
          if (S.sel_e[t * k + s2] == e) p = t * k + s2;
      }
    }
    S.pair_of[u][t] = p;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// K2: the experts. See the top of the file.
// ---------------------------------------------------------------------------
struct DxShared {
  RouteState r;
  uint64_t bar_sh;                 // the shared expert's gate/up rows
  uint64_t bar_g[DX_NSTG];         // gate/up ring
  uint64_t bar_d[DD_NST];          // down ring: this CTA's rows of one slot per stage
  int cons_g[DX_NSTG];             // units of the stage in the slot consumed so far
  int cons_d[DD_NST];              // passes of the slot in the stage done so far
  // the stage (gate/up ring) or slot (down ring) each ring slot was last
  // issued for: a consumer first waits for its own to be issued, so that the
  // barrier phase it then waits on is that copy's, never one two fills back
  int tag_g[DX_NSTG];
  int tag_d[DD_NST];
  int g_issued, d_issued;          // ring stages issued (in order)
  int abort;
};

// Waits until the ring slot's tag names ``want`` (its copy is issued), then
// for the copy's barrier phase; false after ``limit`` ns in either.
__device__ __forceinline__ bool wait_ring(const int* tag, int want, uint64_t* bar, uint32_t parity, uint64_t limit) {
  if (*reinterpret_cast<const volatile int*>(tag) != want) {
    const uint64_t t0 = gtime();
    while (*reinterpret_cast<const volatile int*>(tag) != want) {
      if (gtime() - t0 > limit) return false;
      __nanosleep(20);
    }
  }
  return wait_bar(bar, parity, limit);
}

// Bytes of one gate/up unit (a gate row and an up row) and of one down row.
__host__ __device__ constexpr int dx_unit_bytes(int H, int qt) { return 2 * (H / QK) * (qt == QMOE_Q5K ? 176 : 144); }
__host__ __device__ constexpr int dx_drow_bytes(int F, int qt) { return (F / QK) * (qt == QMOE_Q5K ? 176 : 144); }

// Waits until *p >= target (acquire); false after ``limit`` ns.
__device__ __forceinline__ bool wait_count(const int* p, int target, uint64_t limit) {
  const uint64_t t0 = gtime();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if (gtime() - t0 > limit) return false;
    __nanosleep(32);
  }
}

// (bounds declared for 512 threads, launched with 384: that caps the registers
// at 128 per thread, so that a router CTA fits on the SM beside it)
template <int SL, int FSUB, int GQ, int DQ>
__global__ void __launch_bounds__(DX_MAX_THREADS, 1) decode_experts_kernel(DecodeArgs a) {
  constexpr int H = 1024 * SL;
  constexpr int F = 32 * FSUB;
  constexpr int RB = (H / QK) * (GQ == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES);   // one gate or up row
  constexpr int DRB = (F / QK) * (DQ == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES);  // one down row
  constexpr int STG = 2 * DX_UPS * RB;  // gate/up stage: UPS gate rows, then UPS up rows
  constexpr int DSTG = DD_MAXROWS * DRB;
  constexpr int XP = H + H / 16;        // padded x row (2 floats per 32)
  constexpr int HP = F + F / 16;        // padded h row
  constexpr int RPP = 32 / FSUB;        // down rows per warp pass
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ DxShared S;
  const int T = a.T, k = a.k, E = a.E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const uint64_t lim = a.wait_ns;
  const int P = T * k + T;
  // [shared units | gate/up ring] and later h [P][HP] share the first area
  const size_t area0 = max((size_t)(1 + DX_NSTG) * STG, ((size_t)P * HP * sizeof(float) + 15) & ~(size_t)15);
  uint8_t* sh_rows = smem;                                        // shared expert units [STG]
  uint8_t* ring_g = sh_rows + STG;                                // [DX_NSTG][STG]
  float* hsm = reinterpret_cast<float*>(smem);                    // [P][HP], over the gate/up area once it is dead
  uint8_t* ring_d = smem + area0;                                 // [DD_NST][DSTG]
  float* xsm = reinterpret_cast<float*>(ring_d + DD_NST * DSTG);  // [T][XP]
  float* lg = xsm + T * XP;                                       // routing scratch [T E + E], then y [P][DD_MAXROWS]
  float* ysm = lg;

  // shared expert units of this CTA: rows [fs0, fs1); output rows [o0, o1)
  const int fs0 = a.has_shared ? (int)((long long)cta * F / G) : 0;
  const int fs1 = a.has_shared ? (int)((long long)(cta + 1) * F / G) : 0;
  const int n_sh = fs1 - fs0;
  const int o0 = (int)((long long)cta * H / G), o1 = (int)((long long)(cta + 1) * H / G);
  const int nr = o1 - o0;
  if (tid == 0) {
    tc::mbar_init(&S.bar_sh, 1);
    for (int i = 0; i < DX_NSTG; ++i) tc::mbar_init(&S.bar_g[i], 1);
    for (int i = 0; i < DD_NST; ++i) tc::mbar_init(&S.bar_d[i], 1);
    tc::fence_barrier_init();
    if (n_sh > 0) {
      // the shared expert's weights do not depend on the routing: their copies
      // start before the wait for the router
      const uint32_t n = (uint32_t)(n_sh * RB);
      tc::mbar_expect_tx(&S.bar_sh, 2 * n);
      tc::bulk_g2s(sh_rows, a.Sg + (size_t)fs0 * RB, n, &S.bar_sh);
      tc::bulk_g2s(sh_rows + DX_UPS * RB, a.Su + (size_t)fs0 * RB, n, &S.bar_sh);
    }
    S.abort = 0;
  }
  if (tid < DX_NSTG) {
    S.cons_g[tid] = 0;
    S.tag_g[tid] = -1;
  }
  if (tid < DD_NST) {
    S.cons_d[tid] = 0;
    S.tag_d[tid] = -1;
  }
  tc::grid_dep_wait();  // the router's partials, cleared counters and X are visible
  const int NT = blockDim.x, NW = NT >> 5;
  for (int i = tid; i < T * H / 4; i += NT) {
    const int t = i / (H / 4), f = 4 * (i % (H / 4));
    const float4 v = __ldcg(reinterpret_cast<const float4*>(a.X) + i);
    float2* dst = reinterpret_cast<float2*>(xsm + (size_t)t * XP + padded<32>(f));
    dst[0] = make_float2(v.x, v.y);
    dst[1] = make_float2(v.z, v.w);
  }
  decode_route(a, S.r, lg, NT, cta == 0);
  const int ns = S.r.n_slots;

  // this CTA's routed gate/up units [r0, r1) of U*F (slot has_shared + r / F, row r % F)
  const int U = ns - a.has_shared;
  const int NR = U * F;
  const int r0 = (int)((long long)cta * NR / G), r1 = (int)((long long)(cta + 1) * NR / G);
  const int n_gs = (r1 - r0 + DX_UPS - 1) / DX_UPS;  // routed ring stages

  auto issue_gate_stage = [&](int s) {
    const int slot = s % DX_NSTG;
    const int u0 = r0 + s * DX_UPS, u1 = min(r1, u0 + DX_UPS);
    uint8_t* dst = ring_g + (size_t)slot * STG;
    *reinterpret_cast<volatile int*>(&S.tag_g[slot]) = s;
    tc::mbar_expect_tx(&S.bar_g[slot], (uint32_t)(2 * (u1 - u0) * RB));
    for (int u = u0; u < u1;) {
      const int sl = a.has_shared + u / F, f = u % F;
      const int n = min(u1 - u, F - f);  // rows of this slot in the stage
      const size_t src = ((size_t)S.r.slot_e[sl] * F + f) * RB;
      tc::bulk_g2s(dst + (size_t)(u - u0) * RB, a.Wg + src, (uint32_t)(n * RB), &S.bar_g[slot]);
      tc::bulk_g2s(dst + (size_t)(DX_UPS + u - u0) * RB, a.Wu + src, (uint32_t)(n * RB), &S.bar_g[slot]);
      u += n;
    }
  };
  auto issue_down_slot = [&](int u) {
    const int st = u % DD_NST;
    const int e = S.r.slot_e[u];
    const uint8_t* src = (e == E ? a.Sd : a.Wd + (size_t)e * H * DRB) + (size_t)o0 * DRB;
    *reinterpret_cast<volatile int*>(&S.tag_d[st]) = u;
    tc::mbar_expect_tx(&S.bar_d[st], (uint32_t)(nr * DRB));
    // test-only fault: the first CTA never copies its last slot's down rows,
    // so that wait runs out (nothing else of the CTA is in flight by then)
    if (!(a.fault == 1 && cta == 0 && u == ns - 1))
      tc::bulk_g2s(ring_d + (size_t)st * DSTG, src, (uint32_t)(nr * DRB), &S.bar_d[st]);
  };
  // the first ring fills, one lane per stage: gate/up stages first
  const int g0 = min(n_gs, DX_NSTG), dd0 = min(ns, DD_NST);
  if (warp == 0) {
    if (lane < g0) issue_gate_stage(lane);
    if (lane == 0) {
      S.g_issued = g0;
      S.d_issued = dd0;
    }
  } else if (warp == 1) {
    if (lane < dd0) issue_down_slot(lane);
  }
  // the next layer's router may start loading its weights now
  tc::grid_dep_launch();
  __syncthreads();

  // ---------------------------------------------------------------- gate/up
  // activations of row ``xt`` for the lane's sub-blocks, as fp32 pairs
  bool ok = true;
  {
    uint64_t x2[SL][16];
    float xsum[SL];
    int xt = -1;
    auto load_x = [&](int t) {
#pragma unroll
      for (int j = 0; j < SL; ++j) {
        const uint64_t* src = reinterpret_cast<const uint64_t*>(xsm + (size_t)t * XP + padded<32>((lane + 32 * j) * SUBK));
        float sacc = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x2[j][i] = src[i];
          sacc += sum2(x2[j][i]);
        }
        xsum[j] = sacc;
      }
      xt = t;
    };
    // the CTA's units in order: n_sh shared units, then r1 - r0 routed ones;
    // warp w takes units w, w + NW, ...
    const int n_units = n_sh + (r1 - r0);
    for (int L = warp; L < n_units && ok; L += NW) {
      const uint8_t *grow, *urow;
      int sl, f, s = -1;
      if (L < n_sh) {
        if (!wait_bar(&S.bar_sh, 0, lim)) { ok = false; break; }
        grow = sh_rows + (size_t)L * RB;
        urow = sh_rows + (size_t)(DX_UPS + L) * RB;
        sl = 0;
        f = fs0 + L;
      } else {
        const int r = L - n_sh;
        s = r / DX_UPS;
        const int j = r % DX_UPS, slot = s % DX_NSTG;
        if (!wait_ring(&S.tag_g[slot], s, &S.bar_g[slot], (s / DX_NSTG) & 1, lim)) { ok = false; break; }
        const uint8_t* base = ring_g + (size_t)slot * STG;
        grow = base + (size_t)j * RB;
        urow = base + (size_t)(DX_UPS + j) * RB;
        const int u = r0 + r;
        sl = a.has_shared + u / F;
        f = u % F;
      }
      for (int t = 0; t < T; ++t) {
        const int p = S.r.pair_of[sl][t];
        if (p < 0) continue;
        if (t != xt) load_x(t);
        // gate then up through one copy of the row code (a smaller loop body
        // keeps the warps' instruction fetches in cache)
        float g = 0.f, u = 0.f;
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
          const float v = gate_row_dot<SL, GQ>(m ? urow : grow, x2, xsum, lane);
          if (m) u = v;
          else g = v;
        }
        if (lane == 0) a.hbuf[(size_t)p * F + f] = silu_mul(g, u);
      }
      if (s >= 0 && lane == 0) {
        // the last warp done with a routed stage refills its ring slot. Every
        // read of the stage by a warp fed the products whose warp sum lane 0
        // holds, so those reads have completed when lane 0 counts the unit.
        const int slot = s % DX_NSTG;
        const int in_stage = min(DX_UPS, (r1 - r0) - s * DX_UPS);
        if (atomicAdd(&S.cons_g[slot], 1) == in_stage - 1) {
          S.cons_g[slot] = 0;
          if (s + DX_NSTG < n_gs) {
            issue_gate_stage(s + DX_NSTG);
            atomicAdd(&S.g_issued, 1);
          }
        }
      }
      if (*reinterpret_cast<volatile int*>(&S.abort)) ok = false;
    }
  }
  if (!ok) S.abort = 1;
  if (lane == 0) __threadfence();  // this warp's h stores, before the counters below
  ok = !__syncthreads_or(S.abort);
  // publish: this CTA's h rows, all slots together
  if (ok && tid == 0) atomicAdd(&a.sync[0], n_sh + (r1 - r0));

  // ---------------------------------------------------------------- down
  // all of h: every CTA's gate/up units of every slot are counted
  if (ok && tid == 0 && !wait_count(&a.sync[0], ns * F, lim)) S.abort = 1;
  ok = ok && !__syncthreads_or(S.abort);
  if (ok) {
    // h of every pair, padded rows, over the (now idle) gate/up buffers
    for (int q = tid; q < P * (F / 4); q += NT) {
      const int p = q / (F / 4), c = q % (F / 4);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(a.hbuf + (size_t)p * F) + c);
      float2* dst = reinterpret_cast<float2*>(hsm + (size_t)p * HP + padded<32>(4 * c));
      dst[0] = make_float2(v.x, v.y);
      dst[1] = make_float2(v.z, v.w);
    }
  }
  __syncthreads();
  // passes: slot u, rows RPP q .. RPP q + RPP - 1 of the CTA's rows. When
  // every slot's rows fit the ring at once, warp w takes a contiguous share
  // of the ns * ppu passes (slot-major), so that the lane's sub-block of h for
  // a pair stays in registers while it applies; otherwise the passes go round
  // the warps in order, so that slots are finished (and their ring stages
  // refilled) in order.
  const int ppu = (nr + RPP - 1) / RPP;  // passes per slot
  {
    uint64_t h2[16];
    float hsum = 0.f;
    int hkey = -1;
    int cur_u = -1, cur_passes = 0;
    auto count_passes = [&]() {
      if (cur_u >= 0 && lane == 0) {
        const int st = cur_u % DD_NST;
        if (atomicAdd(&S.cons_d[st], cur_passes) + cur_passes == ppu) {
          S.cons_d[st] = 0;
          if (cur_u + DD_NST < ns) {
            issue_down_slot(cur_u + DD_NST);
            atomicAdd(&S.d_issued, 1);
          }
        }
      }
    };
    const bool contiguous = ns <= DD_NST;
    const int n_it = ns * ppu;
    const int it0 = contiguous ? warp * n_it / NW : warp;
    const int it1 = contiguous ? (warp + 1) * n_it / NW : n_it;
    const int step = contiguous ? 1 : NW;
    for (int it = it0; it < it1 && ok; it += step) {
      const int u = it / ppu, q = it % ppu;
      if (u != cur_u) {
        count_passes();  // the previous slot, before waiting for this one
        cur_u = u;
        cur_passes = 0;
      }
      if (!wait_ring(&S.tag_d[u % DD_NST], u, &S.bar_d[u % DD_NST], (u / DD_NST) & 1, lim)) { ok = false; break; }
      const int r = RPP * q + lane / FSUB;  // this lane's row within the CTA's rows
      const int rr = r < nr ? r : nr - 1;   // lanes past the last row compute a copy, not stored
      const uint8_t* row = ring_d + (size_t)(u % DD_NST) * DSTG + (size_t)rr * DRB;
      for (int t = 0; t < T; ++t) {
        const int p = S.r.pair_of[u][t];
        if (p < 0) continue;
        if (hkey != p) {
          hsum = load_down_h<FSUB>(hsm + (size_t)p * HP, lane, h2);
          hkey = p;
        }
        const float y = down_row_dot<FSUB, DQ>(row, h2, hsum, lane);
        if (lane % FSUB == 0 && r < nr) ysm[p * DD_MAXROWS + r] = y;
      }
      ++cur_passes;
      if (*reinterpret_cast<volatile int*>(&S.abort)) ok = false;
    }
    if (ok) count_passes();
  }
  if (!ok) S.abort = 1;
  if (__syncthreads_or(S.abort)) {
    if (tid == 0) {
      record_status(a.status, QMOE_ERR_TIMEOUT);
      // leave with nothing in flight: wait (bounded) for the phases of every
      // copy this CTA issued (a copy that was never issued just runs out again)
      if (n_sh > 0) wait_bar(&S.bar_sh, 0, lim);
      for (int s = max(0, S.g_issued - DX_NSTG); s < S.g_issued; ++s)
        wait_bar(&S.bar_g[s % DX_NSTG], (s / DX_NSTG) & 1, lim);
      for (int u = max(0, S.d_issued - DD_NST); u < S.d_issued; ++u)
        wait_bar(&S.bar_d[u % DD_NST], (u / DD_NST) & 1, lim);
    }
    return;
  }
  // y of every pair for the CTA's rows (kept for inspection), and the
  // slot-order combine: out = R + y_shared + sum_s w_s y_s
  for (int q = tid; q < P * nr; q += NT) {
    const int p = q / nr, r = q % nr;
    a.ybuf[(size_t)p * H + o0 + r] = ysm[p * DD_MAXROWS + r];
  }
  for (int q = tid; q < T * nr; q += NT) {
    const int t = q / nr, r = q % nr;
    float acc = a.R ? a.R[(size_t)t * H + o0 + r] : 0.f;
    if (a.has_shared) acc += ysm[(T * k + t) * DD_MAXROWS + r];
    for (int s2 = 0; s2 < k; ++s2) acc = fmaf(S.r.wts[t * k + s2], ysm[(t * k + s2) * DD_MAXROWS + r], acc);
    a.out[(size_t)t * H + o0 + r] = acc;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t router_smem(int T, int H) { return sizeof(float) * (size_t)T * H; }

static size_t experts_smem(int T, int H, int E, int k, int F, int gq, int dq) {
  const size_t gu = (size_t)(1 + DX_NSTG) * DX_UPS * dx_unit_bytes(H, gq);
  const size_t P = (size_t)T * k + T;
  const size_t hs = (sizeof(float) * P * (F + F / 16) + 15) & ~(size_t)15;
  const size_t ring = (size_t)DD_NST * DD_MAXROWS * dx_drow_bytes(F, dq);
  const size_t xs = sizeof(float) * (size_t)T * (H + H / 16);
  size_t tail = sizeof(float) * ((size_t)T * E + E);  // routing scratch, then y
  if (sizeof(float) * P * DD_MAXROWS > tail) tail = sizeof(float) * P * DD_MAXROWS;
  return (gu > hs ? gu : hs) + ring + xs + tail;
}

int decode_sync_ints(int H) { return 1; }

bool decode_path_supported(int T, int H, int E, int k, int F, int gate_qt, int down_qt) {
  if (T < 1 || T > DX_MAXT || k > DX_MAXK) return false;
  if (H != 1024 && H != 2048) return false;
  if (F != 256 && F != 512) return false;
  if (E % 32 != 0) return false;  // the router's groups of 8 experts, the top-k's lanes
  const int G = device_sm_count();
  if ((F + G - 1) / G > DX_UPS) return false;      // a CTA's shared-expert units fit one stage
  if ((H + G - 1) / G > DD_MAXROWS) return false;  // a CTA's output rows fit a down stage
  if (experts_smem(T, H, E, k, F, gate_qt, down_qt) > 200 * 1024) return false;
  return true;
}

template <typename K>
static cudaError_t launch_router(K kernel, int grid, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  // both decode kernels ask for the largest shared-memory carveout, so that an
  // SM does not switch its L1 / shared split between them
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(kernel), smem, 100);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(RT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Cooperative launch (every CTA resident at once: the down phase waits on
// counters other CTAs advance), one CTA per SM, programmatically dependent
// on the router.
template <typename K>
static cudaError_t launch_experts(K kernel, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(kernel), smem, 100);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count());
  cfg.blockDim = dim3(dx_threads(a.T));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // if the runtime refuses the programmatic dependency on a cooperative
  // launch, the kernel is launched cooperatively without it (and remembered)
  static std::atomic<int> coop_pdl{0};  // 0 untried, 1 accepted, -1 refused
  const int mode = coop_pdl.load();
  cfg.numAttrs = mode >= 0 ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a);
  if (mode == 0) {
    if (e == cudaSuccess) {
      coop_pdl.store(1);
    } else {
      (void)cudaGetLastError();
      coop_pdl.store(-1);
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, kernel, a);
    }
  }
  return e;
}

template <int SL, int FSUB>
static cudaError_t launch_experts_q(int gq, int dq, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  if (gq == QMOE_Q4K)
    return dq == QMOE_Q5K ? launch_experts(decode_experts_kernel<SL, FSUB, QMOE_Q4K, QMOE_Q5K>, smem, st, a)
                          : launch_experts(decode_experts_kernel<SL, FSUB, QMOE_Q4K, QMOE_Q4K>, smem, st, a);
  return dq == QMOE_Q5K ? launch_experts(decode_experts_kernel<SL, FSUB, QMOE_Q5K, QMOE_Q5K>, smem, st, a)
                        : launch_experts(decode_experts_kernel<SL, FSUB, QMOE_Q5K, QMOE_Q4K>, smem, st, a);
}

cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t st) {
  DecodeArgs a{};
  a.X = L.X; a.R = L.R; a.out = L.out; a.Wr = L.Wr;
  a.Wg = L.Wg; a.Wu = L.Wu; a.Wd = L.Wd; a.Sg = L.Sg; a.Su = L.Su; a.Sd = L.Sd;
  a.T = L.T; a.H = L.H; a.E = L.E; a.k = L.k; a.F = L.F; a.has_shared = L.Sg != nullptr;
  a.logits = L.part; a.hbuf = L.hbuf; a.ybuf = L.ybuf; a.ids = L.ids; a.w = L.w;
  a.sync = L.sync; a.status = L.status;
  a.wait_ns = L.wait_ns;
  a.fault = L.fault;
  const int g1 = (L.E / RT_EPC) * RT_HQ;
  const size_t s1 = router_smem(L.T, L.H);
  cudaError_t e = L.H == 1024 ? launch_router(decode_router_kernel<1>, g1, s1, st, a)
                              : launch_router(decode_router_kernel<2>, g1, s1, st, a);
  if (e != cudaSuccess) return e;
  const size_t s2 = experts_smem(L.T, L.H, L.E, L.k, L.F, L.gate_qt, L.down_qt);
  if (L.H == 1024)
    return L.F == 256 ? launch_experts_q<1, 8>(L.gate_qt, L.down_qt, s2, st, a)
                      : launch_experts_q<1, 16>(L.gate_qt, L.down_qt, s2, st, a);
  return L.F == 256 ? launch_experts_q<2, 8>(L.gate_qt, L.down_qt, s2, st, a)
                    : launch_experts_q<2, 16>(L.gate_qt, L.down_qt, s2, st, a);
}

}  // namespace qmoe
