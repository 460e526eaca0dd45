// Grouped dequant + bf16 tcgen05 GEMM for large T (prefill).
//
// "Distributed CPU: Zip Fusion Beyond Tensor Parallelism", "Prefill First, Then
// One Matrix-Work Scheduler": with many rows per weight region each packed
// weight is reused across the rows and the region becomes GEMM-bound. Here the
// rows routed to one expert (contiguous in permutation order) form the M side
// of a tile; the expert's packed Q4_K/Q5_K rows are dequantised to bf16 in
// shared memory and fed to tcgen05.mma with the fp32 accumulator in tensor
// memory ("What PR #382 Now Splits" in "CKE Zip: From Splitting Tokens To
// Splitting Qwen3.5 Weights": gate, up, SwiGLU and down per expert).
//
// One persistent CTA per SM walks work items (m-tile of 128 rows of one expert,
// n-tile of 256 output columns). Warp roles (416 threads):
//   warps 0-3   epilogue: TMEM -> registers (warp w reads lanes 32w..32w+31),
//               fused SwiGLU (gate/up) or bf16 store (down);
//   warps 4-11  producers: thread p owns weight row p of the n-tile; it keeps
//               the packed super-block of its row in registers, prefetching
//               the next super-blocks in a bulk-copy ring while it
//               dequantises the current one to bf16, written in the
//               128-byte-swizzled K-major layout the MMA descriptors describe;
//   warp 12     allocates 512 TMEM columns (two 256-column accumulators) and
//               issues the MMAs from one lane;
//   warp 13     gathers the activation tile of each k-tile (the rows of an
//               m-tile, through the permutation) with cp.async, up to BS
//               k-tiles ahead of the MMAs.
// A 4-stage shared-memory ring (48 KB per stage) decouples producers and the
// MMA issuer; the two accumulators let the epilogue of one tile overlap the
// main loop of the next. Every wait is bounded: on time-out the CTA records
// QMOE_ERR_TIMEOUT, drains its MMAs, frees its TMEM and returns.
#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64;
constexpr int TC_THREADS = 448;
constexpr int TC_MMA_WARP = 12;
constexpr int TC_LOAD_WARP = 13;
constexpr int TC_PRODUCERS = 256;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 32 KB
// Per weight format: RS stages of packed super-blocks (256 rows each, filled by
// bulk copies) and BS stages of bf16 operand tiles, within 227 KB.
template <int QT>
struct TcCfg {
  static constexpr int BYTES = QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES;
  static constexpr int RS = 2;
  static constexpr int BS = QT == QMOE_Q5K ? 2 : 3;
  static constexpr int RAW_STAGE = TC_PRODUCERS * BYTES;
  static constexpr int SMEM = BS * (TC_A_BYTES + TC_B_BYTES) + RS * RAW_STAGE + 1024 /*align*/ + 256 /*barriers*/;
};

struct TcArgs {
  const uint8_t* W;   // gate (gate/up pass) or down weights of the routed experts
  const uint8_t* W2;  // up weights (gate/up pass)
  const uint8_t* S;   // shared expert counterpart of W
  const uint8_t* S2;  // shared expert counterpart of W2
  const int32_t* offsets;
  const int32_t* perm;
  const int2* mtiles;  // (expert, first row) per m-tile
  const int32_t* n_mtiles;
  const float* X;               // gate/up A source, [T][H] fp32
  const __nv_bfloat16* xb;      // gate/up A source, [T][H] bf16 (converted X)
  const __nv_bfloat16* hin;     // down A source, [P+T][F] bf16
  __nv_bfloat16* hout;          // gate/up output, [P+T][F] bf16
  __nv_bfloat16* yout;          // down output, [P+T][H] bf16
  float* yout_f32;              // down output in fp32 instead, when not null
  int a_rows;                   // rows of the activation tensor the TMA map covers
  int T, k, E, H, F;
  int* status;
};

__device__ __forceinline__ int tc_pair_row(int p, int T, int k) { return p < T * k ? p / k : p - T * k; }

// Packed super-block of one weight row held in registers (16-byte chunks).
template <int QT>
struct RawBlock {
  static constexpr int N = (QT == QMOE_Q5K ? Q5K_BYTES : Q4K_BYTES) / 16;
  uint4 c[N];
};

template <int QT>
__device__ __forceinline__ void load_raw(RawBlock<QT>& r, const uint8_t* blk) {
  const uint4* p = reinterpret_cast<const uint4*>(blk);
#pragma unroll
  for (int i = 0; i < RawBlock<QT>::N; ++i) r.c[i] = __ldg(p + i);
}

// K order inside every group of 8 consecutive K values of the tensor-core
// operands: element e of a 16-byte chunk holds K offset kPerm8[e]. The weight
// dequantisation below produces this order directly (a bf16x2 word takes the
// quants of weights i and i+4 from one 32-bit quant word), and the activation
// producers (the bf16 conversion of X and the gate/up epilogue writing h)
// store their rows in the same order, so the dot products are unchanged.
__device__ constexpr int kPerm8[8] = {0, 4, 1, 5, 2, 6, 3, 7};

// Dequantises sub-blocks j0, j0+1 (64 weights) of a register-held super-block
// into 8 swizzled 16-byte bf16 chunks of row ``r`` of a B stage, in bf16x2
// arithmetic: q is exact (the quant bits under the exponent of 128.0, minus
// 128), then w = q * (d*s_j) - dmin*m_j in one bf16x2 FMA with the two scales
// rounded to bf16.
template <int QT, int J0>
__device__ __forceinline__ void dequant_store(const RawBlock<QT>& raw, uint8_t* stage, int r) {
  KHeader h;
  const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&raw.c[0].x));
  h.d = dd.x;
  h.dmin = dd.y;
  h.f0 = raw.c[0].y;
  h.f1 = raw.c[0].z;
  h.f2 = raw.c[0].w;
  const __nv_bfloat162 m128 = __float2bfloat162_rn(-128.f);
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int j = J0 + s;
    const float2 sc = sub_scale(h, j);
    const __nv_bfloat162 ds2 = __float2bfloat162_rn(sc.x);
    const __nv_bfloat162 ndm2 = __float2bfloat162_rn(-sc.y);
    const uint4 q = QT == QMOE_Q5K ? raw.c[3 + j] : raw.c[1 + j];
    uint32_t hb = 0;
    if (QT == QMOE_Q5K) {
      const uint4 hq = raw.c[1 + (j >> 2)];
      const uint32_t hw[4] = {hq.x, hq.y, hq.z, hq.w};
      hb = hw[j & 3];
    }
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // quants of weights 8n+i and 8n+i+4 as bf16 128+q in the two halves
        uint32_t x = ((w[n] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
        if (QT == QMOE_Q5K) x |= (((hb >> (8 * n + i)) & 0x11u) * 0x10010u) & 0x00100010u;
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&x);
        v = __hadd2(v, m128);             // q, exact
        v = __hfma2(v, ds2, ndm2);        // q*d*s - dmin*m, one rounding
        o[i] = *reinterpret_cast<uint32_t*>(&v);
      }
      *reinterpret_cast<uint4*>(stage + tc::sw128_offset(r, 4 * s + n)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <bool GATEUP, int QT>
__global__ void __launch_bounds__(TC_THREADS, 1) moe_tc_kernel(TcArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Cfg = TcCfg<QT>;
  constexpr int BS = Cfg::BS, RS = Cfg::RS;
  uint8_t* sA = smem;
  uint8_t* sB = smem + BS * TC_A_BYTES;
  uint8_t* sRaw = sB + BS * TC_B_BYTES;              // [RS][256 rows][BYTES]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + RS * Cfg::RAW_STAGE);
  uint64_t* full = bars;                     // [BS]
  uint64_t* empty = bars + BS;               // [BS]
  uint64_t* raw_full = bars + 2 * BS;        // [RS]
  uint64_t* acc_full = raw_full + RS;        // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint64_t* drain = acc_empty + 2;           // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = GATEUP ? g.F / 128 : g.H / TC_BN;      // n-tiles per m-tile
  const int KT = GATEUP ? g.H / TC_BK : g.F / TC_BK;    // k-tiles
  const int total = g.n_mtiles[0] * NT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < BS; ++i) {
      tc::mbar_init(&full[i], TC_PRODUCERS + 32);  // + one cp.async completion per loader lane
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < RS; ++i) tc::mbar_init(&raw_full[i], TC_PRODUCERS);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], 128);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == TC_MMA_WARP) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    int it = 0;
    for (int wi = blockIdx.x; wi < total; wi += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!tc::mbar_wait(&acc_full[acc], ph, abort_flag)) break;
      tc::tc_fence_after();
      const int2 mt = g.mtiles[wi / NT];
      const int nt = wi % NT;
      const int e = mt.x, m0 = mt.y;
      const int row = 32 * warp + lane;
      const int base = g.offsets[e];
      const int Me = g.offsets[e + 1] - base;
      const bool valid = m0 + row < Me;
      const int pos = base + m0 + row;
      const uint32_t tq = tmem + (uint32_t)(acc * 256) + ((uint32_t)(32 * warp) << 16);
      if (GATEUP) {
        __nv_bfloat16* dst = g.hout + (size_t)pos * g.F + nt * 128;
#pragma unroll 1
        for (int c = 0; c < 128; c += 16) {
          uint32_t gr[16], ur[16];
          tc::tmem_ld16x2(tq + c, tq + 128 + c, gr, ur);
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[i] = silu_mul(__uint_as_float(gr[i]), __uint_as_float(ur[i]));
          // stored in the operand K order (kPerm8 inside each group of 8)
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int g8 = (i >> 2) * 8, e = 2 * (i & 3);
            o[i] = tc::pack_bf16x2(hv[g8 + kPerm8[e]], hv[g8 + kPerm8[e + 1]]);
          }
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
            d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
            d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
      } else {
        const int pair = valid ? g.perm[pos] : 0;
        __nv_bfloat16* dst = g.yout + (size_t)pair * g.H + nt * TC_BN;
        float* dst32 = g.yout_f32 ? g.yout_f32 + (size_t)pair * g.H + nt * TC_BN : nullptr;
#pragma unroll 1
        for (int c = 0; c < TC_BN; c += 32) {
          uint32_t a[16], b[16];
          tc::tmem_ld16x2(tq + c, tq + c + 16, a, b);
          if (g.yout_f32 != nullptr) {
            if (valid) {
              float4* d4 = reinterpret_cast<float4*>(dst32 + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d4[i] = make_float4(__uint_as_float(a[4 * i]), __uint_as_float(a[4 * i + 1]),
                                    __uint_as_float(a[4 * i + 2]), __uint_as_float(a[4 * i + 3]));
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d4[4 + i] = make_float4(__uint_as_float(b[4 * i]), __uint_as_float(b[4 * i + 1]),
                                        __uint_as_float(b[4 * i + 2]), __uint_as_float(b[4 * i + 3]));
            }
            continue;
          }
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i] = tc::pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
            o[8 + i] = tc::pack_bf16x2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
          }
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
            d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
            d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
            d4[2] = make_uint4(o[8], o[9], o[10], o[11]);
            d4[3] = make_uint4(o[12], o[13], o[14], o[15]);
          }
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acc_empty[acc]);
    }
  } else if (warp < 4 + TC_PRODUCERS / 32) {
    // ------------------------------------------------------------ producers
    // Thread p owns weight row p of the n-tile (and, p < 128, activation row
    // p). Packed super-blocks of its row arrive by bulk copy into a ring of RS
    // stages, RS super-blocks ahead of use; the activation row of the next
    // k-tile is gathered with cp.async while the current k-tile is
    // dequantised; each k-tile's operand stage is released with one arrive.
    constexpr int BYTES = Cfg::BYTES;
    const int p = threadIdx.x - 128;
    const int KB = KT / 4;  // super-blocks along K
    const size_t rb = GATEUP ? (size_t)(g.H / QK) * BYTES : (size_t)(g.F / QK) * BYTES;
    const int n_mine = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto item = [&](int j) { return (int)blockIdx.x + j * (int)gridDim.x; };
    auto row_of = [&](int wi) -> const uint8_t* {
      const int2 mt = g.mtiles[wi / NT];
      const int nt = wi % NT, e = mt.x;
      if (GATEUP) {
        const bool up = p >= 128;
        const uint8_t* base = e < g.E ? (up ? g.W2 : g.W) + (size_t)e * g.F * rb : (up ? g.S2 : g.S);
        return base + (size_t)(nt * 128 + (p & 127)) * rb;
      }
      const uint8_t* base = e < g.E ? g.W + (size_t)e * g.H * rb : g.S;
      return base + (size_t)(nt * TC_BN + p) * rb;
    };
    auto issue_raw = [&](int u) {
      const int j = u / KB;
      if (j >= n_mine) return;
      uint64_t* bar = &raw_full[u % RS];
      tc::mbar_expect_tx(bar, BYTES);
      tc::bulk_g2s(sRaw + (size_t)(u % RS) * Cfg::RAW_STAGE + (size_t)p * BYTES,
                   row_of(item(j)) + (size_t)(u % KB) * BYTES, BYTES, bar);
    };
    for (int u = 0; u < RS; ++u) issue_raw(u);
    bool ok = true;
    int kg = 0;
    for (int u = 0; u < n_mine * KB && ok; ++u) {
      if (!tc::mbar_wait(&raw_full[u % RS], (u / RS) & 1, abort_flag)) {
        ok = false;
        break;
      }
      RawBlock<QT> cur;
      const uint4* rp = reinterpret_cast<const uint4*>(sRaw + (size_t)(u % RS) * Cfg::RAW_STAGE + (size_t)p * BYTES);
#pragma unroll
      for (int i = 0; i < RawBlock<QT>::N; ++i) cur.c[i] = rp[i];
      tc::fence_proxy_async_smem();  // these reads come before the copy that refills the slot
      issue_raw(u + RS);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (!tc::mbar_wait(&empty[kg % BS], ((kg / BS) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* b_st = sB + (kg % BS) * TC_B_BYTES;
        if (kk == 0) dequant_store<QT, 0>(cur, b_st, p);
        else if (kk == 1) dequant_store<QT, 2>(cur, b_st, p);
        else if (kk == 2) dequant_store<QT, 4>(cur, b_st, p);
        else dequant_store<QT, 6>(cur, b_st, p);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&full[kg % BS]);
        ++kg;
      }
    }
  } else if (warp == TC_LOAD_WARP) {
    // ------------------------------------------------------------ activation loader
    // Lane l gathers rows l, l+32, l+64, l+96 of the m-tile (16-byte cp.async
    // into the swizzled positions; rows past the expert's count are zero
    // filled) up to BS k-tiles ahead; each lane's completion arrives on the
    // stage's barrier (cp.async.mbarrier.arrive.noinc).
    int kg = 0;
    bool ok = true;
    for (int wi = blockIdx.x; wi < total && ok; wi += gridDim.x) {
      const int2 mt = g.mtiles[wi / NT];
      const int e = mt.x, m0 = mt.y;
      const int base = g.offsets[e];
      const int Me = g.offsets[e + 1] - base;
      const __nv_bfloat16* src[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = lane + 32 * q;
        src[q] = nullptr;
        if (m0 + r < Me) {
          const int pos = base + m0 + r;
          src[q] = GATEUP ? g.xb + (size_t)tc_pair_row(g.perm[pos], g.T, g.k) * g.H : g.hin + (size_t)pos * g.F;
        }
      }
      const __nv_bfloat16* zsrc = GATEUP ? g.xb : g.hin;  // any valid address: nothing is read
      for (int kt = 0; kt < KT; ++kt, ++kg) {
        const int stage = kg % BS;
        if (!tc::mbar_wait(&empty[stage], ((kg / BS) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* a_st = sA + stage * TC_A_BYTES;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = lane + 32 * q;
          const bool valid = src[q] != nullptr;
          const __nv_bfloat16* s0 = valid ? src[q] + kt * TC_BK : zsrc;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            tc::cp_async16(a_st + tc::sw128_offset(r, c), s0 + (valid ? 8 * c : 0), valid);
        }
        tc::cp_async_arrive_noinc(&full[stage]);
      }
    }
    tc::cp_async_wait_all();
  } else {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = tc::idesc_bf16_f32(TC_BM, TC_BN);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int wi = blockIdx.x; wi < total && ok; wi += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!tc::mbar_wait(&acc_empty[acc], ph ^ 1, abort_flag)) break;
      tc::tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(acc * 256);
      for (int kt = 0; kt < KT; ++kt) {
        if (!tc::mbar_wait(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        // the activation tile was written by cp.async (generic proxy): order it
        // before the tensor core's reads
        tc::fence_proxy_async_smem();
        tc::tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = tc::smem_u32(sA + stage * TC_A_BYTES);
          const uint32_t b_addr = tc::smem_u32(sB + stage * TC_B_BYTES);
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            tc::mma_bf16(d_tmem, tc::sw128_desc(a_addr + 32 * kk), tc::sw128_desc(b_addr + 32 * kk), idesc,
                         (kt | kk) != 0);
          }
          tc::mma_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == BS) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (ok && lane == 0) tc::mma_commit(&acc_full[acc]);
      __syncwarp();
    }
    // drain: every MMA this thread issued has completed before TMEM is freed
    if (lane == 0) {
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never);
    }
    __syncwarp();
  }

  if (*abort_flag && threadIdx.x == 0) record_status(g.status, QMOE_ERR_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == TC_MMA_WARP) tc::tmem_dealloc(tmem, 512);
}

// Builds the m-tile list: for every expert with rows (the shared expert last),
// one entry per 128 rows. One CTA; the scan runs in warp 0.
__global__ void __launch_bounds__(1024) build_mtiles_kernel(const int32_t* __restrict__ offsets, int E,
                                                            int2* __restrict__ mtiles,
                                                            int32_t* __restrict__ n_mtiles) {
  extern __shared__ int32_t start[];  // [E+1] exclusive scan of tile counts
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int run = 0;
    for (int b = 0; b <= E; b += 32) {
      const int e = b + lane;
      const int c = e <= E ? (offsets[e + 1] - offsets[e] + TC_BM - 1) / TC_BM : 0;
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e <= E) start[e] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) n_mtiles[0] = run;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    const int Me = offsets[e + 1] - offsets[e];
    int s = start[e];
    for (int m0 = 0; m0 < Me; m0 += TC_BM) mtiles[s++] = make_int2(e, m0);
  }
}

// out_t = R_t + y_shared,t + sum_s w_{t,s} y_{t,s} with bf16 y, in slot order.
__global__ void __launch_bounds__(256) combine_bf16_kernel(const __nv_bfloat16* __restrict__ y,
                                                           const float* __restrict__ w, const float* R,
                                                           float* out, int T, int H, int k,
                                                           int has_shared) {
  const int H8 = H / 8;
  const size_t n = (size_t)T * H8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H8), c = (int)(i % H8);
    float acc[8];
    if (R) {
      const float4* r4 = reinterpret_cast<const float4*>(R + (size_t)t * H) + 2 * c;
      float4 a = r4[0], b = r4[1];
      acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
      acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    }
    if (has_shared) {
      uint4 v = reinterpret_cast<const uint4*>(y + ((size_t)T * k + t) * H)[c];
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 f = __bfloat1622float2(h2[j]);
        acc[2 * j] += f.x;
        acc[2 * j + 1] += f.y;
      }
    }
    for (int s = 0; s < k; ++s) {
      const float ws = w[(size_t)t * k + s];
      uint4 v = reinterpret_cast<const uint4*>(y + ((size_t)t * k + s) * H)[c];
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 f = __bfloat1622float2(h2[j]);
        acc[2 * j] = fmaf(ws, f.x, acc[2 * j]);
        acc[2 * j + 1] = fmaf(ws, f.y, acc[2 * j + 1]);
      }
    }
    float4* o4 = reinterpret_cast<float4*>(out + (size_t)t * H) + 2 * c;
    o4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// X [T][H] fp32 -> bf16 (round to nearest even) in the operand K order
// (kPerm8 inside each group of 8), the A operand of the tensor-core path.
__global__ void __launch_bounds__(256) to_bf16_kernel(const float* __restrict__ x, __nv_bfloat16* __restrict__ y,
                                                      size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(x)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(x)[2 * i + 1];
    // group (0..7) = a.x a.y a.z a.w b.x b.y b.z b.w -> order 0,4,1,5,2,6,3,7
    uint4 o;
    o.x = tc::pack_bf16x2(a.x, b.x);
    o.y = tc::pack_bf16x2(a.y, b.y);
    o.z = tc::pack_bf16x2(a.z, b.z);
    o.w = tc::pack_bf16x2(a.w, b.w);
    reinterpret_cast<uint4*>(y)[i] = o;
  }
}

cudaError_t launch_to_bf16(const float* x, __nv_bfloat16* y, size_t n, cudaStream_t st) {
  const size_t n8 = n / 8;
  int blocks = (int)((n8 + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  to_bf16_kernel<<<blocks, 256, 0, st>>>(x, y, n8);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
int tc_num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n = v > 0 ? v : 1;
  }
  return n;
}

int tc_max_mtiles(int T, int k, int E, int has_shared) {
  const int P = T * k;
  return (P + (has_shared ? T : 0)) / TC_BM + E + 1;
}

cudaError_t launch_build_mtiles(const int32_t* offsets, int E, int2* mtiles, int32_t* n_mtiles,
                                cudaStream_t st) {
  build_mtiles_kernel<<<1, 1024, sizeof(int32_t) * (E + 1), st>>>(offsets, E, mtiles, n_mtiles);
  return cudaGetLastError();
}

template <bool GATEUP, int QT>
static cudaError_t tc_launch_t(const TcArgs& a, int max_items, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(moe_tc_kernel<GATEUP, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcCfg<QT>::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  int grid = tc_num_sms();
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  moe_tc_kernel<GATEUP, QT><<<grid, TC_THREADS, TcCfg<QT>::SMEM, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gateup_tc(const GroupedTcArgs& p, cudaStream_t st) {
  TcArgs a{};
  a.W = p.W; a.W2 = p.W2; a.S = p.S; a.S2 = p.S2;
  a.offsets = p.offsets; a.perm = p.perm; a.mtiles = p.mtiles; a.n_mtiles = p.n_mtiles;
  a.X = p.X; a.xb = p.xb; a.hout = p.hout; a.a_rows = p.a_rows;
  a.T = p.T; a.k = p.k; a.E = p.E; a.H = p.H; a.F = p.F; a.status = p.status;
  const int items = p.max_mtiles * (p.F / 128);
  return p.qt == QMOE_Q5K ? tc_launch_t<true, QMOE_Q5K>(a, items, st) : tc_launch_t<true, QMOE_Q4K>(a, items, st);
}

cudaError_t launch_down_tc(const GroupedTcArgs& p, cudaStream_t st) {
  TcArgs a{};
  a.W = p.W; a.S = p.S;
  a.offsets = p.offsets; a.perm = p.perm; a.mtiles = p.mtiles; a.n_mtiles = p.n_mtiles;
  a.hin = p.hin; a.yout = p.yout; a.yout_f32 = p.yout_f32; a.a_rows = p.a_rows;
  a.T = p.T; a.k = p.k; a.E = p.E; a.H = p.H; a.F = p.F; a.status = p.status;
  const int items = p.max_mtiles * (p.H / TC_BN);
  return p.qt == QMOE_Q5K ? tc_launch_t<false, QMOE_Q5K>(a, items, st) : tc_launch_t<false, QMOE_Q4K>(a, items, st);
}

cudaError_t launch_combine_bf16(const __nv_bfloat16* y, const float* w, const float* R, float* out, int T, int H,
                                int k, int has_shared, cudaStream_t st) {
  const size_t n = (size_t)T * (H / 8);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  combine_bf16_kernel<<<blocks, 256, 0, st>>>(y, w, R, out, T, H, k, has_shared);
  return cudaGetLastError();
}

}  // namespace qmoe
