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
//               order and write 4 partial logits per (row, expert). CTA 0 also
//               clears the expert kernel's counters.
//   K2 experts  one CTA per SM (cooperative launch, so every CTA is resident),
//               16 warps. Work is cut into equal shares of all SMs:
//                 - gate/up units: (expert slot, intermediate row f), a gate
//                   row and an up row each. The shared expert's units are
//                   known before routing, so each CTA starts their copies
//                   before it waits for the router; then every CTA takes the
//                   top-k itself from the router's partials (the same fixed-
//                   order arithmetic everywhere, so every CTA reaches the same
//                   decision) and copies its share of the routed experts' rows
//                   through a ring of bulk copies (cp.async.bulk + mbarrier);
//                 - down units: (expert slot, block of 32 output rows), whose
//                   rows are copied through a second ring as soon as the
//                   routing is known, while the gate/up units still compute.
//               A gate/up unit writes h = silu(x.g) * (x.u) per (row, slot)
//               pair; when a CTA has finished its gate/up units it adds their
//               count to a per-slot counter. A down unit waits for its slot's
//               counter to reach F (all of h), computes y for its 32 rows and
//               every pair of its slot, and takes a ticket of its row block;
//               the CTA that takes the last ticket of a block forms
//               out = R + y_shared + sum_s w_s y_s for those rows, in slot
//               order (no atomics on the data; the result does not depend on
//               which CTA combines).
// Every wait (copies, counters) gives up after a bounded time, records
// QMOE_ERR_TIMEOUT and leaves the CTA with no copy in flight.
#include <atomic>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

constexpr int RT_THREADS = 256;
constexpr int RT_EPC = 8;  // router: experts per CTA
constexpr int RT_HQ = 4;   // router: parts of H (CTAs per expert group)

constexpr int DX_THREADS = 512;
constexpr int DX_WARPS = DX_THREADS / 32;
constexpr int DX_UPS = 8;    // gate/up units per ring stage: one row per warp
constexpr int DX_NSTG = 4;   // gate/up ring stages
constexpr int DX_DR = 32;    // output rows per down unit: two per warp
constexpr int DX_NSTD = 4;   // down ring stages
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
  int* sync;       // [DX_MAXSLOT] h counters per slot, then [H / DX_DR] combine tickets
  int* status;
  unsigned long long wait_ns;  // a wait gives up after this many nanoseconds
  int fault;                   // test-only: 1 = CTA 0 withholds the copy of its last down unit
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

// ---------------------------------------------------------------- arithmetic

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

__device__ __forceinline__ float sum2(uint64_t v) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
  return __uint_as_float(lo) + __uint_as_float(hi);
}

// S = sum over the 8 NW weights of ``w`` of (0.5 + q_i/256) * x_i. Word n
// holds weights 8n..8n+7 (byte b: weight 8n+2b in the low nibble, 8n+2b+1 in
// the high one); for Q5_K bit i of ``hb`` is weight i's fifth bit. Each quant
// is placed by one byte permute into the mantissa of a float whose exponent
// makes it 0.5 + q/256 exactly (no int->float conversion), and the pairs of
// weights (8n+2b, 8n+2b+1) meet their activation pairs x2[4n+b] in one
// two-lane fp32 FMA (each lane rounds as fmaf does).
template <int QT, int NW>
__device__ __forceinline__ float dot_words(const uint32_t* w, uint32_t hb, const uint64_t* x2) {
  uint64_t acc = 0;  // (0.0f, 0.0f)
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
      const uint64_t q2 = pack2(__byte_perm(ev, 0x3F000000u, sel), __byte_perm(od, 0x3F000000u, sel));
      acc = ffma2(q2, x2[4 * n + b], acc);
    }
  }
  return sum2(acc);
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

// h . row for one packed down row of F = 32 FSUB weights: LPS = 32 / FSUB
// lanes per sub-block, each taking 32 / LPS consecutive weights of it.
template <int FSUB, int QT>
__device__ __forceinline__ float down_row_dot(const uint8_t* row, const float* h, int lane) {
  constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  constexpr int LPS = 32 / FSUB;   // 2 (F = 512) or 4 (F = 256)
  constexpr int WPL = 32 / LPS;    // weights per lane: 16 or 8
  constexpr int NW = WPL / 8;      // quant words per lane
  const int c = lane / LPS, p = lane % LPS;
  const uint8_t* blk = row + (size_t)(c >> 3) * BYTES;
  const int sj = c & 7;
  const KHeader hd = header_of(*reinterpret_cast<const uint4*>(blk));
  uint32_t w[NW];
  const uint32_t* qp = reinterpret_cast<const uint32_t*>(blk + quant_offset(QT, sj) + p * (WPL / 2));
#pragma unroll
  for (int n = 0; n < NW; ++n) w[n] = qp[n];
  const uint32_t hb = QT == QMOE_Q5K ? (*reinterpret_cast<const uint32_t*>(blk + 16 + 4 * sj) >> (p * WPL)) : 0u;
  const uint64_t* h2 = reinterpret_cast<const uint64_t*>(h + c * 32 + p * WPL);
  uint64_t x2[WPL / 2];
  float hs = 0.f;
#pragma unroll
  for (int i = 0; i < WPL / 2; ++i) {
    x2[i] = h2[i];
    hs += sum2(x2[i]);
  }
  float acc = sub_contrib(dot_words<QT, NW>(w, hb, x2), hs, sub_scale(hd, sj));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
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
  if (blockIdx.x == 0)
    for (int i = tid; i < DX_MAXSLOT + H / DX_DR; i += RT_THREADS) a.sync[i] = 0;
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
// K2: the experts. See the top of the file.
// ---------------------------------------------------------------------------
struct DxShared {
  uint64_t bar_sh;               // the shared expert's gate/up rows
  uint64_t bar_g[DX_NSTG];       // gate/up ring
  uint64_t bar_d[DX_NSTD];       // down ring
  float sel_l[DX_MAXT * DX_MAXK];
  int32_t sel_e[DX_MAXT * DX_MAXK];
  float wts[DX_MAXT * DX_MAXK];
  int32_t slot_e[DX_MAXSLOT];           // expert of each slot (E = shared)
  int32_t pair_of[DX_MAXSLOT][DX_MAXT]; // pair index of (slot, row), -1 if the row does not use the slot
  float gu[2][DX_UPS][DX_MAXT];         // gate / up dot products of a stage
  float ys[DX_MAXT][DX_DR];             // y of a down unit
  int32_t n_slots;
  int32_t wflag;  // a counter wait succeeded
  int32_t cflag;  // this CTA combines the current row block
};

// Bytes of one gate/up unit (a gate row and an up row) and of one down row.
__host__ __device__ constexpr int dx_unit_bytes(int H, int qt) { return 2 * (H / QK) * (qt == QMOE_Q5K ? 176 : 144); }
__host__ __device__ constexpr int dx_drow_bytes(int F, int qt) { return (F / QK) * (qt == QMOE_Q5K ? 176 : 144); }

template <int SL, int FSUB, int GQ, int DQ>
__global__ void __launch_bounds__(DX_THREADS, 1) decode_experts_kernel(DecodeArgs a) {
  constexpr int H = 1024 * SL;
  constexpr int F = 32 * FSUB;
  constexpr int NBLK = H / DX_DR;
  constexpr int RB = (H / QK) * (GQ == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES);   // one gate or up row
  constexpr int DRB = (F / QK) * (DQ == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES);  // one down row
  constexpr int STG = 2 * DX_UPS * RB;   // gate/up stage: UPS gate rows, then UPS up rows
  constexpr int DSTG = DX_DR * DRB;      // down stage
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ DxShared S;
  const int T = a.T, k = a.k, E = a.E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const uint64_t lim = a.wait_ns;
  uint8_t* sh_rows = smem;                                   // shared expert units [STG]
  uint8_t* ring_g = sh_rows + STG;                           // [DX_NSTG][STG]
  uint8_t* ring_d = ring_g + DX_NSTG * STG;                  // [DX_NSTD][DSTG]
  float* xsm = reinterpret_cast<float*>(ring_d + DX_NSTD * DSTG);  // [T][H]
  float* hsm = xsm + T * H;                                  // [T][F]

  // shared expert units of this CTA: rows [fs0, fs1)
  const int fs0 = a.has_shared ? (int)((long long)cta * F / G) : 0;
  const int fs1 = a.has_shared ? (int)((long long)(cta + 1) * F / G) : 0;
  if (tid == 0) {
    tc::mbar_init(&S.bar_sh, 1);
    for (int i = 0; i < DX_NSTG; ++i) tc::mbar_init(&S.bar_g[i], 1);
    for (int i = 0; i < DX_NSTD; ++i) tc::mbar_init(&S.bar_d[i], 1);
    tc::fence_barrier_init();
    if (fs1 > fs0) {
      // the shared expert's weights do not depend on the routing: their copies
      // start before the wait for the router
      const uint32_t n = (uint32_t)((fs1 - fs0) * RB);
      tc::mbar_expect_tx(&S.bar_sh, 2 * n);
      tc::bulk_g2s(sh_rows, a.Sg + (size_t)fs0 * RB, n, &S.bar_sh);
      tc::bulk_g2s(sh_rows + DX_UPS * RB, a.Su + (size_t)fs0 * RB, n, &S.bar_sh);
    }
  }
  tc::grid_dep_wait();  // the router's partials, cleared counters and X are visible
  __syncthreads();

  // ---------------------------------------------------------------- routing
  // logits from the 4 partials in a fixed order (NaN ranks below -inf's
  // index order: it is mapped to -inf), then the top-k by rank: the thread of
  // (row t, expert e) counts the experts ordered before e (larger logit, or
  // equal logit and lower index) and stops at k; a count below k is e's slot.
  float* lg = hsm;  // [T][E] logits, in the h staging area (not yet in use)
  for (int i = tid; i < T * E; i += DX_THREADS) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < RT_HQ; ++q) v += __ldcg(a.logits + (size_t)q * T * E + i);
    lg[i] = (v == v) ? v : -INFINITY;
  }
  for (int i = tid; i < T * H / 4; i += DX_THREADS)
    reinterpret_cast<float4*>(xsm)[i] = __ldcg(reinterpret_cast<const float4*>(a.X) + i);
  __syncthreads();
  for (int i = tid; i < T * E; i += DX_THREADS) {
    const int t = i / E, e = i % E;
    const float* L = lg + t * E;
    const float v = L[e];
    int cnt = 0;
    for (int j0 = 0; j0 < E && cnt < k; j0 += 4) {
      const float4 q = *reinterpret_cast<const float4*>(L + j0);
      cnt += (q.x > v || (q.x == v && j0 < e)) + (q.y > v || (q.y == v && j0 + 1 < e)) +
             (q.z > v || (q.z == v && j0 + 2 < e)) + (q.w > v || (q.w == v && j0 + 3 < e));
    }
    if (cnt < k) {
      S.sel_e[t * k + cnt] = e;
      S.sel_l[t * k + cnt] = v;
    }
  }
  __syncthreads();
  if (tid < T * k) {
    const int t = tid / k;
    const float l0 = S.sel_l[t * k];
    float den = 0.f;
    for (int r = 0; r < k; ++r) den += expf(S.sel_l[t * k + r] - l0);
    S.wts[tid] = expf(S.sel_l[tid] - l0) / den;
    if (cta == 0) {
      a.ids[tid] = S.sel_e[tid];
      a.w[tid] = S.wts[tid];
    }
  }
  // slots: the shared expert first, then the distinct selected experts in
  // ascending order (warp 0 compacts a mark per expert)
  int* mark = reinterpret_cast<int*>(lg + T * E);  // [E], after the logits
  for (int e = tid; e < E; e += DX_THREADS) mark[e] = 0;
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
  for (int i = tid; i < ns * DX_MAXT; i += DX_THREADS) {
    const int u = i / DX_MAXT, t = i % DX_MAXT;
    int p = -1;
    if (t < T) {
      const int e = S.slot_e[u];
      if (e == E) {
        p = T * k + t;
      } else {
        for (int s = 0; s < k; ++s)
          if (S.sel_e[t * k + s] == e) p = t * k + s;
      }
    }
    S.pair_of[u][t] = p;
  }

  // this CTA's routed gate/up units [r0, r1) of U*F (slot has_shared + r / F,
  // row r % F) and down units [d0, d1) of ns * NBLK (slot d / NBLK, block d % NBLK)
  const int U = ns - a.has_shared;
  const int NR = U * F, ND = ns * NBLK;
  const int r0 = (int)((long long)cta * NR / G), r1 = (int)((long long)(cta + 1) * NR / G);
  const int d0 = (int)((long long)cta * ND / G), d1 = (int)((long long)(cta + 1) * ND / G);
  const int n_gs = (r1 - r0 + DX_UPS - 1) / DX_UPS;  // routed gate/up stages
  const int n_du = d1 - d0;

  auto issue_gate_stage = [&](int s) {
    const int slot = s % DX_NSTG;
    const int u0 = r0 + s * DX_UPS, u1 = min(r1, u0 + DX_UPS);
    uint8_t* dst = ring_g + (size_t)slot * STG;
    tc::mbar_expect_tx(&S.bar_g[slot], (uint32_t)(2 * (u1 - u0) * RB));
    for (int u = u0; u < u1;) {
      const int sl = a.has_shared + u / F, f = u % F;
      const int n = min(u1 - u, F - f);  // rows of this slot in the stage
      const int e = S.slot_e[sl];
      const size_t src = ((size_t)e * F + f) * RB;
      tc::bulk_g2s(dst + (size_t)(u - u0) * RB, a.Wg + src, (uint32_t)(n * RB), &S.bar_g[slot]);
      tc::bulk_g2s(dst + (size_t)(DX_UPS + u - u0) * RB, a.Wu + src, (uint32_t)(n * RB), &S.bar_g[slot]);
      u += n;
    }
  };
  auto issue_down_unit = [&](int i) {
    const int slot = i % DX_NSTD;
    const int d = d0 + i, sl = d / NBLK, b = d % NBLK;
    const int e = S.slot_e[sl];
    const uint8_t* src = (e == E ? a.Sd : a.Wd + (size_t)e * H * DRB) + (size_t)b * DX_DR * DRB;
    tc::mbar_expect_tx(&S.bar_d[slot], (uint32_t)DSTG);
    // test-only fault: the last down unit of CTA 0 is never copied, so its
    // wait runs out (nothing else of this CTA is in flight by then)
    if (!(a.fault == 1 && cta == 0 && i == n_du - 1))
      tc::bulk_g2s(ring_d + (size_t)slot * DSTG, src, (uint32_t)DSTG, &S.bar_d[slot]);
  };
  __syncthreads();
  // ring bookkeeping: stages / units issued (thread 0) and consumed (all)
  int g_iss = 0, d_iss = 0, g_cons = 0, d_cons = 0;
  bool sh_cons = !(fs1 > fs0);
  if (tid == 0) {
    for (; g_iss < min(n_gs, DX_NSTG); ++g_iss) issue_gate_stage(g_iss);
    for (; d_iss < min(n_du, DX_NSTD); ++d_iss) issue_down_unit(d_iss);
  }
  // the next layer's router may start loading its weights now
  tc::grid_dep_launch();

  // ---------------------------------------------------------------- gate/up
  // activations of row ``xt`` for the lane's sub-blocks, as fp32 pairs
  uint64_t x2[SL][16];
  float xsum[SL];
  int xt = -1;
  auto load_x = [&](int t) {
#pragma unroll
    for (int j = 0; j < SL; ++j) {
      const uint64_t* src = reinterpret_cast<const uint64_t*>(xsm + (size_t)t * H + (lane + 32 * j) * SUBK);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x2[j][i] = src[i];
        s += sum2(x2[j][i]);
      }
      xsum[j] = s;
    }
    xt = t;
  };
  bool ok = true;
  // stage -1 is the shared expert's units (rows fs0..fs1), stages 0.. the routed ones
  for (int s = (fs1 > fs0) ? -1 : 0; s < n_gs && ok; ++s) {
    const uint8_t* base;
    int nu, slot_first, f_first;
    if (s < 0) {
      ok = __syncthreads_and(wait_bar(&S.bar_sh, 0, lim));
      sh_cons = ok;
      base = sh_rows;
      nu = fs1 - fs0;
      slot_first = 0;
      f_first = fs0;
    } else {
      ok = __syncthreads_and(wait_bar(&S.bar_g[s % DX_NSTG], (s / DX_NSTG) & 1, lim));
      if (ok) g_cons = s + 1;
      base = ring_g + (size_t)(s % DX_NSTG) * STG;
      const int u0 = r0 + s * DX_UPS;
      nu = min(r1 - u0, DX_UPS);
      slot_first = a.has_shared + u0 / F;
      f_first = u0 % F;
    }
    if (!ok) break;
    // warp w: unit w % UPS, matrix w / UPS (0 gate, 1 up)
    const int j = warp % DX_UPS, mat = warp / DX_UPS;
    if (j < nu) {
      // a stage holds at most two slots (UPS <= F)
      const int f = f_first + j;
      const int sl = f < F ? slot_first : slot_first + 1;
      const uint8_t* row = base + (size_t)(mat * DX_UPS + j) * RB;
      for (int t = 0; t < T; ++t) {
        if (S.pair_of[sl][t] < 0) continue;
        if (t != xt) load_x(t);
        const float v = gate_row_dot<SL, GQ>(row, x2, xsum, lane);
        if (lane == 0) S.gu[mat][j][t] = v;
      }
    }
    __syncthreads();
    if (tid < DX_UPS * T) {
      const int jj = tid / T, t = tid % T;
      if (jj < nu) {
        const int f = f_first + jj;
        const int sl = f < F ? slot_first : slot_first + 1;
        const int p = S.pair_of[sl][t];
        if (p >= 0) a.hbuf[(size_t)p * F + (f < F ? f : f - F)] = silu_mul(S.gu[0][jj][t], S.gu[1][jj][t]);
      }
    }
    if (tid == 0 && s >= 0 && s + DX_NSTG < n_gs) {
      // every read of this ring stage is done (barrier above)
      tc::fence_proxy_async_smem();
      issue_gate_stage(g_iss++);
    }
    __syncthreads();
  }
  // publish this CTA's h rows per slot
  __threadfence();
  __syncthreads();
  if (ok && tid == 0) {
    if (fs1 > fs0) atomicAdd(&a.sync[0], fs1 - fs0);
    for (int u = r0; u < r1;) {
      const int sl = a.has_shared + u / F, n = min(r1 - u, F - u % F);
      atomicAdd(&a.sync[sl], n);
      u += n;
    }
  }

  // ---------------------------------------------------------------- down
  int cur = -1;
  for (int i = 0; i < n_du && ok; ++i) {
    const int d = d0 + i, sl = d / NBLK, b = d % NBLK;
    if (sl != cur) {
      // all of h for this slot: every CTA's gate/up units of it are counted
      if (tid == 0) S.wflag = wait_count(&a.sync[sl], F, lim) ? 1 : 0;
      __syncthreads();
      if (!S.wflag) {
        ok = false;
        break;
      }
      for (int q = tid; q < T * F / 4; q += DX_THREADS) {
        const int t = q / (F / 4), c = q % (F / 4);
        const int p = S.pair_of[sl][t];
        if (p >= 0)
          reinterpret_cast<float4*>(hsm + (size_t)t * F)[c] = __ldcg(reinterpret_cast<const float4*>(a.hbuf + (size_t)p * F) + c);
      }
      cur = sl;
    }
    ok = __syncthreads_and(wait_bar(&S.bar_d[i % DX_NSTD], (i / DX_NSTD) & 1, lim));
    if (!ok) break;
    d_cons = i + 1;
    const uint8_t* base = ring_d + (size_t)(i % DX_NSTD) * DSTG;
#pragma unroll
    for (int rr = 0; rr < DX_DR / DX_WARPS; ++rr) {
      const int r = warp * (DX_DR / DX_WARPS) + rr;
      for (int t = 0; t < T; ++t) {
        if (S.pair_of[sl][t] < 0) continue;
        const float v = down_row_dot<FSUB, DQ>(base + (size_t)r * DRB, hsm + (size_t)t * F, lane);
        if (lane == 0) S.ys[t][r] = v;
      }
    }
    __syncthreads();
    if (tid < T * DX_DR) {
      const int t = tid / DX_DR, r = tid % DX_DR;
      const int p = S.pair_of[sl][t];
      if (p >= 0) {
        a.ybuf[(size_t)p * H + b * DX_DR + r] = S.ys[t][r];
        __threadfence();
      }
    }
    if (tid == 0 && i + DX_NSTD < n_du) {
      tc::fence_proxy_async_smem();
      issue_down_unit(d_iss++);
    }
    __syncthreads();
    // one ticket per (slot, block); the CTA with the last one of the block combines
    if (tid == 0) {
      const int old = atomicAdd(&a.sync[DX_MAXSLOT + b], 1);
      S.cflag = (old == ns - 1) ? 1 : 0;
      if (S.cflag) __threadfence();
    }
    __syncthreads();
    if (S.cflag && tid < T * DX_DR) {
      const int t = tid / DX_DR, r = b * DX_DR + tid % DX_DR;
      float acc = a.R ? a.R[(size_t)t * H + r] : 0.f;
      if (a.has_shared) acc += __ldcg(a.ybuf + (size_t)(T * k + t) * H + r);
      for (int s2 = 0; s2 < k; ++s2) acc = fmaf(S.wts[t * k + s2], __ldcg(a.ybuf + (size_t)(t * k + s2) * H + r), acc);
      a.out[(size_t)t * H + r] = acc;
    }
  }
  if (!ok && tid == 0) {
    record_status(a.status, QMOE_ERR_TIMEOUT);
    // leave with nothing in flight: wait (bounded) for every copy this CTA
    // issued and did not consume (a copy that was never issued just runs
    // out again)
    if (!sh_cons) wait_bar(&S.bar_sh, 0, lim);
    for (int s = g_cons; s < g_iss; ++s) wait_bar(&S.bar_g[s % DX_NSTG], (s / DX_NSTG) & 1, lim);
    for (int i = d_cons; i < d_iss; ++i) wait_bar(&S.bar_d[i % DX_NSTD], (i / DX_NSTD) & 1, lim);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t router_smem(int T, int H) { return sizeof(float) * (size_t)T * H; }

static size_t experts_smem(int T, int H, int E, int F, int gq, int dq) {
  const size_t stg = (size_t)DX_UPS * dx_unit_bytes(H, gq);
  const size_t dstg = (size_t)DX_DR * dx_drow_bytes(F, dq);
  const size_t xs = sizeof(float) * (size_t)T * H;
  // the h staging area also holds the routing's logits and expert marks
  size_t hs = sizeof(float) * (size_t)T * F;
  const size_t route = sizeof(float) * (size_t)T * E + sizeof(int) * (size_t)E;
  if (route > hs) hs = route;
  return stg + DX_NSTG * stg + DX_NSTD * dstg + xs + hs;
}

int decode_sync_ints(int H) { return DX_MAXSLOT + H / DX_DR; }

bool decode_path_supported(int T, int H, int E, int k, int F, int gate_qt, int down_qt) {
  if (T < 1 || T > DX_MAXT || k > DX_MAXK) return false;
  if (H != 1024 && H != 2048) return false;
  if (F != 256 && F != 512) return false;
  if (E % RT_EPC != 0) return false;
  const int G = device_sm_count();
  if ((F + G - 1) / G > DX_UPS) return false;  // the shared expert's units of a CTA fit one stage
  if (experts_smem(T, H, E, F, gate_qt, down_qt) > 200 * 1024) return false;
  return true;
}

template <typename K>
static cudaError_t launch_router(K kernel, int grid, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(kernel), smem);
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

// Cooperative launch (every CTA resident at once: the down units wait on
// counters other CTAs advance), one CTA per SM, programmatically dependent
// on the router.
template <typename K>
static cudaError_t launch_experts(K kernel, size_t smem, cudaStream_t st, const DecodeArgs& a) {
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count());
  cfg.blockDim = dim3(DX_THREADS);
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
  const size_t s2 = experts_smem(L.T, L.H, L.E, L.F, L.gate_qt, L.down_qt);
  if (L.H == 1024)
    return L.F == 256 ? launch_experts_q<1, 8>(L.gate_qt, L.down_qt, s2, st, a)
                      : launch_experts_q<1, 16>(L.gate_qt, L.down_qt, s2, st, a);
  return L.F == 256 ? launch_experts_q<2, 8>(L.gate_qt, L.down_qt, s2, st, a)
                    : launch_experts_q<2, 16>(L.gate_qt, L.down_qt, s2, st, a);
}

}  // namespace qmoe
