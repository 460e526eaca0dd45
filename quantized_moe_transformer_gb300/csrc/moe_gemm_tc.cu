// Grouped dequant + bf16 tcgen05 GEMM for large T (prefill).
//
// "Distributed CPU: Zip Fusion Beyond Tensor Parallelism", "Prefill First, Then
// One Matrix-Work Scheduler": with many rows per weight region each packed
// weight is reused across the rows and the region becomes GEMM-bound. Here the
// rows routed to one expert (contiguous in permutation order) are cut into
// chunks of at most 64, 128 or 192 tokens; per work item one expert's packed
// rows are dequantised to bf16 and multiplied with the chunk's activations on
// the tensor cores, fp32 accumulation in tensor memory ("What PR #382 Now
// Splits" in "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights":
// gate, up, SwiGLU and down per expert).
//
// The weights are the MMA's M side and the tokens its N side: the
// dequantised weights go from registers straight into tensor memory
// (tcgen05.st) and are read there as the A operand, so they never pass through
// shared memory; only the token tile is staged in shared memory (128-byte
// swizzled, K-major). N is the chunk's token count rounded up to 16, so a
// chunk of 20 tokens costs the tensor core 32 columns, not 128 rows.
//
// A work item is (token chunk, weight block). A weight block is two 128-row
// matrices A0, A1 with accumulators D0, D1 (TMEM columns [0, NMAX) and
// [NMAX, 2 NMAX), NMAX = the chunk cap, 64, 128 or 192):
// gate rows and the matching up rows (gate/up pass: SwiGLU pairs lane f of D0
// with lane f of D1 in one thread), or two consecutive 128-row blocks of the
// down matrix. One persistent CTA per SM walks the items; warp roles (896
// threads):
//   warps 0-3, 24-27  epilogue: TMEM -> registers (warp w reads lanes
//               32 (w % 4) .. + 31; the two warps of a lane quarter take
//               alternate groups of 16 tokens), SwiGLU to bf16 h (gate/up) or
//               the y store (down), leaving through a small shared-memory
//               transpose in 16-byte stores;
//   warps 4-19  producers: warp 4 + pw covers lane quarter pw % 4 of A0
//               (pw / 4 even) or A1, and half of each k-tile's sub-blocks
//               (k-tile = K 128, half a super-block, or K 64 at NMAX 192); a
//               thread dequantises 64 (or 32) weights of its row per k-tile
//               from the packed super-block ring and stores them into the
//               k-tile's A stage in TMEM (columns 2 NMAX + BK s ..);
//   warps 20,23 issue the MMAs of D0 and D1 (one lane each); warp 20 also
//               allocates the 512 TMEM columns;
//   warp 21     copies each k-tile's token rows into the stage's
//               shared-memory tile (one lane, 2-D tensor copies);
//   warp 22     copies the packed weight rows into the super-block ring (one
//               lane, 2-D tensor copies).
// Two A stages in TMEM (three when NMAX is 64), three to five token stages
// and two or three packed super-block stages in shared memory, each ring with
// its own full/empty barriers, decouple the roles.
// Every wait is bounded: on time-out the CTA records QMOE_ERR_TIMEOUT, drains
// its MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>
#include <type_traits>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

constexpr int TC_PRODUCER_WARPS = 16;
constexpr int TC_MMA_WARP = 4 + TC_PRODUCER_WARPS;  // 20
constexpr int TC_LOAD_WARP = TC_MMA_WARP + 1;       // 21: token tiles
constexpr int TC_RAW_WARP = TC_MMA_WARP + 2;        // 22: packed weights
constexpr int TC_MMA_WARP2 = TC_MMA_WARP + 3;       // 23: MMAs of the second accumulator
constexpr int TC_EPI_WARP2 = TC_MMA_WARP2 + 1;      // 24-27: second epilogue warp per lane quarter
constexpr int TC_EPI_WARPS = 8;
constexpr int TC_THREADS = 32 * (TC_EPI_WARP2 + 4); // 896
constexpr int TC_EPI_BYTES = 2048;            // per epilogue warp: 16 tokens x 32 values x 4 B
constexpr int TC_N_MIN = 64;                  // the smallest chunk cap (bounds the chunk count)
// experts' mean rows (T k / E) above which the chunk cap is 192
#ifndef TC_CAP192_MIN_ROWS
#define TC_CAP192_MIN_ROWS 120
#endif

// Packed weights are staged per super-block: RS ring stages of 256 rows (A0
// rows, then A1 rows), each filled by one or two 2-D tensor copies.
// Token tiles have their own ring of TS stages (deeper than the TMEM A ring)
// so that their loads run ahead of the MMAs instead of inside the A ring's
// round trip.
// NMAX is the chunk cap (largest MMA N): the two accumulators take 2 NMAX of
// the 512 TMEM columns and the A stages (BK columns each: K = BK for both
// matrices) the rest. A cap of 64 rows buys 3 A stages of K 128 (chosen when
// experts get few rows, T * k / E <= 32); a cap of 192 leaves 128 columns,
// two A stages of K 64 (chosen when experts get many rows: an expert's rows
// are then one chunk, its weights dequantised once, where a cap of 128 cuts
// about half of them in two).
// Q6_K and MXFP4 weights (down pass only): a 210- or 136-byte super-block is
// only 2- or 8-byte aligned, so neither a tensor-map box nor a bulk copy can
// take one super-block column. An item's 256 rows of the down matrix are
// contiguous and 16-byte aligned instead (256 x 210 and 256 x 136 bytes are
// multiples of 16): the weight loader copies all of them (every super-block
// for K <= 512) into the one raw stage with four bulk copies.
template <int QT>
__host__ __device__ constexpr bool tc_rowcopy() { return QT == QMOE_Q6K || QT == QMOE_MXFP4; }
constexpr int TC_ROWCOPY_KB = 2;  // super-blocks along K that the raw stage holds

template <int QT, int NMAX>
struct TcCfg {
  static constexpr int BYTES = qtype_size(QT);
  static constexpr int BK = NMAX > 128 ? 64 : 128;                  // K per stage (k-tile)
  static constexpr uint32_t A_STAGE_COLS = BK;                      // two matrices x BK / 2 columns
  static constexpr int S = (512 - 2 * NMAX) / BK;                   // A stages in TMEM
  static constexpr uint32_t D1_COL = NMAX;                          // D0 at column 0
  static constexpr uint32_t A_COL = 2 * NMAX;                       // A stage s at A_COL + BK s
  static constexpr int B_HALF = NMAX * 128;                         // K 64 x NMAX rows, one swizzle atom row each
  static constexpr int B_BYTES = (BK / 64) * B_HALF;                // token tile per stage: one or two K halves
  static constexpr int RS = tc_rowcopy<QT>() ? 1 : ((QT == QMOE_Q5K && NMAX >= 128) ? 2 : 3);
  static constexpr int TS = NMAX == 64 ? (QT == QMOE_Q5K ? 4 : 5)
                          : NMAX == 128 ? 3
                                        : ((QT == QMOE_Q4K || QT == QMOE_Q6K) ? 4 : 5);
  static constexpr int RAW_STAGE = tc_rowcopy<QT>() ? 256 * TC_ROWCOPY_KB * BYTES : 256 * BYTES;
  static constexpr int SMEM = TS * B_BYTES + RS * RAW_STAGE + TC_EPI_WARPS * TC_EPI_BYTES + 1024 /*align*/ +
                              512 /*barriers*/;
};

struct TcArgs {
  const uint8_t* W;   // gate (gate/up pass) or down weights of the routed experts
  const uint8_t* W2;  // up weights (gate/up pass)
  const uint8_t* S;   // shared expert counterpart of W
  const uint8_t* S2;  // shared expert counterpart of W2
  const int32_t* offsets;
  const int32_t* perm;
  const int2* chunks;  // (expert, first row | (rows - 1) << 24) per token chunk
  const int32_t* n_chunks;
  const __nv_bfloat16* xb;      // gate/up token source, [P+T][H] bf16: X rows in permutation order
  const __nv_bfloat16* hin;     // down token source, [P+T][F] bf16
  __nv_bfloat16* hout;          // gate/up output, [P+T][F] bf16
  __nv_bfloat16* yout;          // down output, [P+T][H] bf16, rows in permutation order
  float* yout_f32;              // down output in fp32 instead, when not null
  int tok_shift;                // the shared expert's token rows start this many rows before its output rows
  int T, k, E, H, F;
  int* status;
  unsigned long long wait_ns;   // a bounded wait gives up after this long
  int fault;                    // test-only: 1 = CTA 0's producer warp 4 withholds its last full arrival
};

// Tensor maps of the packed weights as 2-D byte arrays [rows][row bytes]:
// w/w2 the routed experts' gate/up (or down in w), s/s2 the shared expert's.
struct TcMaps {
  CUtensorMap w, w2, s, s2;
  CUtensorMap tok;  // token rows [rows][K] bf16, 128-byte swizzled boxes of 32 rows x 64
};

__device__ __forceinline__ int tc_pair_row(int p, int T, int k) { return p < T * k ? p / k : p - T * k; }

struct Chunk {
  int e, c0, n;
};
__device__ __forceinline__ Chunk chunk_at(const int2* chunks, int i) {
  const int2 c = chunks[i];
  return {c.x, c.y & 0xFFFFFF, (int)((uint32_t)c.y >> 24) + 1};
}

// K order inside every group of 8 consecutive K values of the tensor-core
// operands: element e of a group holds K offset kPerm8[e],
//   kPerm8 = {0, 4, 1, 5, 2, 6, 3, 7}.
// The weight dequantisation below produces this order directly (a bf16x2
// word takes the quants of weights i and i+4 from one 32-bit quant word), and
// the activation producers (the bf16 conversion of X and the gate/up epilogue
// writing h) store their rows in the same order, so the dot products are
// unchanged.
// Position within its group of 8 at which K offset f % 8 is stored (the
// inverse of kPerm8), as an index into the row.
__device__ __forceinline__ int kperm_slot(int f) { return (f & ~7) | ((f & 3) << 1) | ((f >> 2) & 1); }

// Dequantises sub-block j (32 weights) into 16 bf16x2 words in kPerm8 order:
// each weight d*s_j*q - dmin*m_j is formed in fp32 and rounded once to bf16
// (nearest even). The quant enters as f = 0.5 + q/256, placed by one byte
// permute into the mantissa of a float whose exponent makes it exact, and
// w = f * (256 d s_j) - (128 d s_j + dmin m_j) is one fp32 FMA (two weights per
// two-lane FMA): 256 d s_j is exact, and the fp32 rounding of the constant
// term is about 2^-24 of 128 d s_j, far below the bf16 step of the weight.
// ``hdr`` is the super-block's first 16 bytes, ``qv`` the sub-block's 16
// quant bytes, ``hb`` (Q5_K) its 32 high bits. Word 4n+i of the output holds
// weights 8n+i (low half) and 8n+i+4 (high half).
template <int QT>
__device__ __forceinline__ void dequant_sub(const uint4 hdr, const uint4 qv, uint32_t hb, int j, uint32_t* o) {
  KHeader h;
  const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));
  h.d = dd.x;
  h.dmin = dd.y;
  h.f0 = hdr.y;
  h.f1 = hdr.z;
  h.f2 = hdr.w;
  const float2 sc = sub_scale(h, j);
  const uint32_t av = __float_as_uint(256.f * sc.x);
  const uint32_t cv = __float_as_uint(-fmaf(128.f, sc.x, sc.y));
  const uint64_t a2 = pack2(av, av), c2 = pack2(cv, cv);
  const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    // ev: quants of weights 8n, 8n+2, 8n+4, 8n+6 in bytes 0..3; od: 8n+1, ...
    uint32_t ev = w[n] & 0x0F0F0F0Fu;
    uint32_t od = (w[n] >> 4) & 0x0F0F0F0Fu;
    if (QT == QMOE_Q5K) {
      ev |= spread4(hb >> (8 * n), 0);
      od |= spread4(hb >> (8 * n), 1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t src = (i & 1) ? od : ev;
      const uint32_t blo = (uint32_t)(i >> 1), bhi = blo + 2;  // weights 8n+i, 8n+i+4
      const uint64_t f2 = pack2(__byte_perm(src, 0x3F000000u, 0x7044u | (blo << 8)),
                                __byte_perm(src, 0x3F000000u, 0x7044u | (bhi << 8)));
      const float2 wv = unpack2(ffma2(f2, a2, c2));
      o[4 * n + i] = tc::pack_bf16x2(wv.x, wv.y);
    }
  }
}

// Q6_K: 32 weights (group g of a 210-byte super-block at ``blk``, 2-byte
// aligned in shared memory) into 16 bf16x2 words in kPerm8 order. Weight i
// of the super-block is d * s_{i/16} * (q_i - 32), q_i = its low nibble
// (byte 82 + i/2, the high nibble for odd i) + 16 * its 2-bit high part
// (byte 18 + i/4, bits 2 (i % 4)); the s are signed bytes at 2. As in
// dequant_sub the quant enters as f = 0.5 + q/256 (a byte permute into a
// float's mantissa; q < 64) and w = f * (256 d s) - 160 d s is one fp32 FMA
// (both constants exact: d s has at most 19 significant bits), rounded once
// to bf16.
__device__ __forceinline__ uint32_t lds_u32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// The 16 bytes at ``p`` (2-byte aligned, shared memory) as four words.
__device__ __forceinline__ uint4 lds16_align2(const uint8_t* p) {
  const uint32_t off = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u);
  const uint8_t* a = p - off;
  const uint32_t w0 = lds_u32(a), w1 = lds_u32(a + 4), w2 = lds_u32(a + 8), w3 = lds_u32(a + 12);
  if (off == 0) return make_uint4(w0, w1, w2, w3);
  const uint32_t w4 = lds_u32(a + 16);  // off == 2: the piece ends 2 bytes into this word
  return make_uint4(__funnelshift_r(w0, w1, 16), __funnelshift_r(w1, w2, 16), __funnelshift_r(w2, w3, 16),
                    __funnelshift_r(w3, w4, 16));
}

__device__ __forceinline__ uint2 lds8_align2(const uint8_t* p) {
  const uint32_t off = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u);
  const uint8_t* a = p - off;
  const uint32_t w0 = lds_u32(a), w1 = lds_u32(a + 4);
  if (off == 0) return make_uint2(w0, w1);
  const uint32_t w2 = lds_u32(a + 8);
  return make_uint2(__funnelshift_r(w0, w1, 16), __funnelshift_r(w1, w2, 16));
}

__device__ __forceinline__ void dequant_q6k_group(const uint8_t* blk, int g, uint32_t* o) {
  const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk)));
  const uint32_t s2 = (uint32_t)*reinterpret_cast<const unsigned short*>(blk + 2 + 2 * g);
  const float ds0 = d * (float)(int8_t)(s2 & 0xFFu), ds1 = d * (float)(int8_t)(s2 >> 8);
  const uint32_t a0 = __float_as_uint(256.f * ds0), c0 = __float_as_uint(-160.f * ds0);
  const uint32_t a1 = __float_as_uint(256.f * ds1), c1 = __float_as_uint(-160.f * ds1);
  const uint4 qv = lds16_align2(blk + 82 + 16 * g);
  const uint2 hv = lds8_align2(blk + 18 + 8 * g);  // 2-bit high parts of the group's 32 weights
  const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    // the high parts of weights 8n .. 8n + 7 (2 bits each), bytes duplicated:
    // a = [b0, b0, b1, b1] with b0 = weights 8n..8n+3, b1 = 8n+4..8n+7
    const uint32_t hh = ((n < 2 ? hv.x : hv.y) >> (16 * (n & 1))) & 0xFFFFu;
    const uint32_t a = __byte_perm(hh, 0u, 0x1100u);
    // weights 8n + 2k (byte k of ev) and 8n + 2k + 1 (byte k of od): their
    // high parts moved to bits 4-5 of byte k
    const uint32_t ev_hi = ((a << 4) & 0x00300030u) | (a & 0x30003000u);
    const uint32_t od_hi = ((a << 2) & 0x00300030u) | ((a >> 2) & 0x30003000u);
    const uint32_t ev = (w[n] & 0x0F0F0F0Fu) | ev_hi;
    const uint32_t od = ((w[n] >> 4) & 0x0F0F0F0Fu) | od_hi;
    const uint64_t a2 = n < 2 ? pack2(a0, a0) : pack2(a1, a1);  // 16 weights per scale
    const uint64_t c2 = n < 2 ? pack2(c0, c0) : pack2(c1, c1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t src = (i & 1) ? od : ev;
      const uint32_t blo = (uint32_t)(i >> 1), bhi = blo + 2;  // weights 8n+i, 8n+i+4
      const uint64_t f2 = pack2(__byte_perm(src, 0x3F000000u, 0x7044u | (blo << 8)),
                                __byte_perm(src, 0x3F000000u, 0x7044u | (bhi << 8)));
      const float2 wv = unpack2(ffma2(f2, a2, c2));
      o[4 * n + i] = tc::pack_bf16x2(wv.x, wv.y);
    }
  }
}

// MXFP4: 32 weights (group g of a 136-byte super-block at ``blk``, 8-byte
// aligned in shared memory) into 16 bf16x2 words in kPerm8 order. Weight i is
// E2M1(code_i) * 2^(e_{i/32} - 127): the codes' magnitudes 0, 0.5, 1, 1.5, 2,
// 3, 4, 6 as q = 2 |v| (one byte permute from an 8-entry table picks four),
// f = 0.5 + q/256 (a byte permute into a float's mantissa), w = f * 128 s -
// 64 s = |v| s in one fp32 FMA, exact, and the code's sign bit moved into
// each bf16 half by a shift and an exclusive or. The products of E2M1 values
// and powers of two are exact in bf16 (up to overflow and the flush of fp32
// subnormals to zero).
__device__ __forceinline__ void dequant_mxfp4_group(const uint8_t* blk, int g, uint32_t* o) {
  const uint32_t e = blk[g];
  const float sc = __uint_as_float(e == 0u ? 0x00400000u : (e == 255u ? 0x7FC00000u : e << 23));
  const uint64_t a2 = pack2(__float_as_uint(128.f * sc), __float_as_uint(128.f * sc));
  const uint64_t c2 = pack2(__float_as_uint(-64.f * sc), __float_as_uint(-64.f * sc));
  const uint2 c01 = *reinterpret_cast<const uint2*>(blk + 8 + 16 * g);
  const uint2 c23 = *reinterpret_cast<const uint2*>(blk + 16 + 16 * g);
  const uint32_t w[4] = {c01.x, c01.y, c23.x, c23.y};
  constexpr uint32_t LUT0 = 0x03020100u, LUT1 = 0x0C080604u;  // q = 2 |v| of magnitude codes 0..7
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const uint32_t sel = w[n] & 0x77777777u;       // the magnitude of code m (weight 8n + m) in nibble m
    const uint32_t mlo = __byte_perm(LUT0, LUT1, sel);        // q of weights 8n .. 8n + 3
    const uint32_t mhi = __byte_perm(LUT0, LUT1, sel >> 16);  // q of weights 8n + 4 .. 8n + 7
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t pi = 0x7044u | ((uint32_t)i << 8);
      const float2 wv = unpack2(ffma2(pack2(__byte_perm(mlo, 0x3F000000u, pi), __byte_perm(mhi, 0x3F000000u, pi)), a2, c2));
      // sign bits of weights 8n + i (bit 4i + 3) and 8n + i + 4 (bit 4i + 19) to bits 15 and 31
      o[4 * n + i] = tc::pack_bf16x2(wv.x, wv.y) ^ ((w[n] << (12 - 4 * i)) & 0x80008000u);
    }
  }
}

// silu(g) * u with silu(g) = g * sigmoid(g) = g/2 + (g/2) tanh(g/2): one
// hardware tanh approximation (tanh.approx.f32, maximum relative error about
// 2^-11) instead of an exponential and a reciprocal; the result is rounded to
// bf16 (relative step 2^-8) right after.
__device__ __forceinline__ float silu_mul_tanh(float g, float u) {
  const float hg = 0.5f * g;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hg));
  return fmaf(hg, t, hg) * u;
}

__device__ __forceinline__ uint32_t pick_word(const uint4 v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

template <bool GATEUP, int QT, int NMAX>
__global__ void __launch_bounds__(TC_THREADS, 1) moe_tc_kernel(const TcArgs g, const __grid_constant__ TcMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned start, reached by pointer arithmetic on the shared
  // array so that accesses stay shared-memory instructions
  const uint32_t s0 = tc::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((s0 + 1023u) & ~1023u) - s0);
  using Cfg = TcCfg<QT, NMAX>;
  constexpr int S = Cfg::S, RS = Cfg::RS, TS = Cfg::TS, BYTES = Cfg::BYTES, BK = Cfg::BK;
  constexpr int TC_B_BYTES = Cfg::B_BYTES, TC_B_HALF = Cfg::B_HALF;
  constexpr uint32_t TC_D1_COL = Cfg::D1_COL, TC_A_COL = Cfg::A_COL;
  uint8_t* sB = smem;                                         // [TS][NMAX][128 B] token tiles
  uint8_t* sRaw = smem + TS * TC_B_BYTES;                     // [RS][256][BYTES] packed rows
  uint8_t* sEpi = sRaw + RS * Cfg::RAW_STAGE;                 // [TC_EPI_WARPS][TC_EPI_BYTES]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + TC_EPI_WARPS * TC_EPI_BYTES);
  uint64_t* full = bars;                // [S]  A stage stored
  uint64_t* empty = bars + S;           // [S]  MMAs of the stage done
  uint64_t* tok_full = bars + 2 * S;    // [TS] token tile landed
  uint64_t* tok_empty = tok_full + TS;  // [TS] MMAs reading the token tile done
  uint64_t* raw_full = tok_empty + TS;  // [RS] packed rows landed
  uint64_t* raw_empty = raw_full + RS;  // [RS] packed rows consumed
  uint64_t* acc_full = raw_empty + RS;  // [1]
  uint64_t* acc_empty = acc_full + 1;   // [1]
  uint64_t* drain = acc_empty + 1;      // [2] one per MMA warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = g.wait_ns;
  const int NB = GATEUP ? g.F / 128 : g.H / 256;      // weight blocks per chunk
  const int KT = GATEUP ? g.H / BK : g.F / BK;        // k-tiles
  const int KB = KT / (256 / BK);                     // super-blocks along K
  const int total = g.n_chunks[0] * NB;
  const int n_mine = (int)blockIdx.x < total ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], TC_PRODUCER_WARPS);
      tc::mbar_init(&empty[i], 2);  // one commit per MMA warp
    }
    for (int i = 0; i < TS; ++i) {
      tc::mbar_init(&tok_full[i], 1);   // the token loader's arrive, with its bytes
      tc::mbar_init(&tok_empty[i], 1);  // forwarded by producer warp 4, see below
    }
    for (int i = 0; i < RS; ++i) {
      tc::mbar_init(&raw_full[i], 1);
      tc::mbar_init(&raw_empty[i], TC_PRODUCER_WARPS);
    }
    tc::mbar_init(acc_full, 2);
    tc::mbar_init(acc_empty, TC_EPI_WARPS);
    tc::mbar_init(&drain[0], 1);
    tc::mbar_init(&drain[1], 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == TC_MMA_WARP) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4 || warp >= TC_EPI_WARP2) {
    // ------------------------------------------------------------ epilogue
    // Per 16 tokens: TMEM -> registers, the values of the warp's 32 rows are
    // transposed through shared memory so that each token's 32 outputs leave
    // in 16-byte stores.
    // Two warps per TMEM lane quarter lq (warps lq and TC_EPI_WARP2 + lq)
    // take alternate groups of 16 tokens.
    const int lq = warp & 3, par = warp < 4 ? 0 : 1;
    const uint32_t tq = tmem + ((uint32_t)(32 * lq) << 16);
    uint8_t* stg = sEpi + (4 * par + lq) * TC_EPI_BYTES;
    int it = 0;
    for (int wi = blockIdx.x; wi < total; wi += gridDim.x, ++it) {
      // warp-uniform outcome: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, tc::mbar_wait(acc_full, it & 1, abort_flag, lim))) break;
      tc::tc_fence_after();
      const Chunk ch = chunk_at(g.chunks, wi / NB);
      const int blk = wi % NB;
      const int pos0 = g.offsets[ch.e] + ch.c0;
#pragma unroll 1
      for (int c = 16 * par; c < ch.n; c += 32) {
        uint32_t a[16], b[16];
        tc::tmem_ld16x2(tq + c, tq + TC_D1_COL + c, a, b);
        if (GATEUP) {
          // h[pos][f] = silu(gate) * up, in the operand K order
          __nv_bfloat16* st16 = reinterpret_cast<__nv_bfloat16*>(stg);
          const int col = kperm_slot(lane);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st16[i * 32 + col] = __float2bfloat16_rn(silu_mul_tanh(__uint_as_float(a[i]), __uint_as_float(b[i])));
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int id = lane + 32 * j, i = id >> 2, part = id & 3;
            if (c + i < ch.n)
              *reinterpret_cast<uint4*>(g.hout + (size_t)(pos0 + c + i) * g.F + blk * 128 + 32 * lq + 8 * part) =
                  reinterpret_cast<const uint4*>(stg)[id];
          }
          __syncwarp();
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* v = half ? b : a;
            const int col0 = blk * 256 + half * 128 + 32 * lq;
            if (g.yout_f32 != nullptr) {
              float* s32 = reinterpret_cast<float*>(stg);
#pragma unroll
              for (int i = 0; i < 16; ++i) s32[i * 32 + lane] = __uint_as_float(v[i]);
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int id = lane + 32 * j, i = id >> 3, part = id & 7;
                const int t = c + i;
                if (t < ch.n)
                  *reinterpret_cast<uint4*>(g.yout_f32 + (size_t)(pos0 + t) * g.H + col0 + 4 * part) =
                      reinterpret_cast<const uint4*>(stg)[id];
              }
            } else {
              __nv_bfloat16* s16 = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
              for (int i = 0; i < 16; ++i) s16[i * 32 + lane] = __float2bfloat16_rn(__uint_as_float(v[i]));
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int id = lane + 32 * j, i = id >> 2, part = id & 3;
                const int t = c + i;
                if (t < ch.n)
                  *reinterpret_cast<uint4*>(g.yout + (size_t)(pos0 + t) * g.H + col0 + 8 * part) =
                      reinterpret_cast<const uint4*>(stg)[id];
              }
            }
            __syncwarp();
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty);
    }
  } else if (warp < 4 + TC_PRODUCER_WARPS) {
    // ------------------------------------------------------------ producers
    // Warp 4 + pw covers TMEM lane quarter pw % 4 of matrix (pw / 4) % 2 and
    // sub-blocks 2 sp, 2 sp + 1 (sp = pw / 8) of each k-tile's four (BK 128),
    // or sub-block sp of its two (BK 64): thread = one weight row, 64 or 32
    // weights per k-tile. A k-tile is stored and its stage
    // released before the next one is dequantised, so that the stage round
    // trip (MMA commit -> producers -> MMA) stays short.
    // (sp is a compile-time constant in each of the two copies of the body, so
    // that the sub-block indices, and with them the scale-field extraction,
    // fold into constants)
    const int pw = warp - 4;
    auto producer = [&](auto sp_c) {
      constexpr int sp = decltype(sp_c)::value;
      const int mat = (pw >> 2) & 1;
      const int r = 32 * (pw & 3) + lane;
      constexpr int HPS = 256 / BK;  // k-tiles per super-block
      constexpr int SUBS = BK / 64;  // sub-blocks per thread and k-tile
      const uint32_t ta0 =
          tmem + ((uint32_t)(32 * (pw & 3)) << 16) + TC_A_COL + (uint32_t)(mat * (BK / 2) + sp * (BK / 4));
      // (whole rows: the item's rows, every super-block, in one stage)
      constexpr bool ROWCOPY = tc_rowcopy<QT>();
      const size_t row_pitch = ROWCOPY ? (size_t)KB * BYTES : (size_t)BYTES;
      const uint8_t* my_row = sRaw + (size_t)(mat * 128 + r) * row_pitch;
      const int NU = n_mine * KB;
      uint32_t wa[16], wb[16];
      uint4 hdr = make_uint4(0, 0, 0, 0), hq0 = hdr, hq1 = hdr;
      // loads the super-block header (and Q5_K high bits) of ring slot u % RS
      auto open_sb = [&](int u) -> bool {
        if constexpr (ROWCOPY) {
          // the stage holds item u / KB; its first super-block waits for it
          return u % KB != 0 ||
                 __all_sync(0xffffffffu, tc::mbar_wait(&raw_full[0], (u / KB) & 1, abort_flag, lim));
        }
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&raw_full[u % RS], (u / RS) & 1, abort_flag, lim))) return false;
        const uint4* rp = reinterpret_cast<const uint4*>(my_row + (size_t)(u % RS) * Cfg::RAW_STAGE);
        hdr = rp[0];
        if (QT == QMOE_Q5K) {
          hq0 = rp[1];
          hq1 = rp[2];
        }
        return true;
    };
    // sub-blocks j0 .. j0 + SUBS - 1 of super-block u, k-tile hh, into o0 (and o1)
    auto deq = [&](int u, int hh, uint32_t* o0, uint32_t* o1) {
      const int j0 = (BK / 32) * hh + SUBS * sp;
      if constexpr (ROWCOPY) {
        const uint8_t* blk = my_row + (size_t)(u % KB) * BYTES;
        if constexpr (QT == QMOE_Q6K) {
          dequant_q6k_group(blk, j0, o0);
          if (SUBS == 2) dequant_q6k_group(blk, j0 + 1, o1);
        } else {
          dequant_mxfp4_group(blk, j0, o0);
          if (SUBS == 2) dequant_mxfp4_group(blk, j0 + 1, o1);
        }
        return;
      }
      const uint4* rp = reinterpret_cast<const uint4*>(my_row + (size_t)(u % RS) * Cfg::RAW_STAGE);
      const uint4 hq = (j0 >> 2) ? hq1 : hq0;  // high bits of sub-blocks 4 (j0 / 4) .. + 3
      const uint4 q0 = rp[(QT == QMOE_Q5K ? 3 : 1) + j0];
      dequant_sub<QT>(hdr, q0, QT == QMOE_Q5K ? pick_word(hq, j0 & 3) : 0u, j0, o0);
      if (SUBS == 2) {
        const uint4 q1 = rp[(QT == QMOE_Q5K ? 3 : 1) + j0 + 1];
        dequant_sub<QT>(hdr, q1, QT == QMOE_Q5K ? pick_word(hq, (j0 + 1) & 3) : 0u, j0 + 1, o1);
      }
    };
    bool ok = NU > 0 && open_sb(0);
    if (ok) deq(0, 0, wa, wb);
    int kg = 0;
    for (int u = 0; u < NU && ok; ++u) {
#pragma unroll
      for (int hh = 0; hh < HPS; ++hh) {
        const int stage = kg % S;
        // warp-uniform outcome: the TMEM stores below are warp-collective
        if (!__all_sync(0xffffffffu, tc::mbar_wait(&empty[stage], ((kg / S) & 1) ^ 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        // The empty phase just seen certifies that the MMAs of k-tile kg - S
        // have completed: warp 4 forwards that to the token ring, which saves
        // the MMA warps a second commit per k-tile.
        if (pw == 0 && lane == 0 && kg >= S) tc::mbar_arrive(&tok_empty[(kg - S) % TS]);
        // store and release the stage first: this is the path the MMAs wait on
        tc::tc_fence_after();
        const uint32_t ta = ta0 + (uint32_t)stage * Cfg::A_STAGE_COLS;
        tc::tmem_st16(ta, wa);
        if (SUBS == 2) tc::tmem_st16(ta + 16, wb);
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        // test-only fault: the first CTA's first producer warp never marks the
        // last k-tile of its last item stored, so the MMA warps' wait on it
        // runs out (every copy of the CTA has landed by then)
        const bool withhold = GATEUP && g.fault == 1 && blockIdx.x == 0 && pw == 0 && u == NU - 1 && hh == HPS - 1;
        if (lane == 0 && !withhold) tc::mbar_arrive(&full[stage]);
        ++kg;
        // then dequantise the next k-tile while the MMAs run
        if (hh < HPS - 1) {
          deq(u, hh + 1, wa, wb);
        } else {
          // every read of slot u is done: release it to the weight loader
          // (whole rows: after the item's last super-block)
          if (!ROWCOPY || u % KB == KB - 1) {
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&raw_empty[ROWCOPY ? 0 : u % RS]);
          }
          if (u + 1 < NU) {
            if (!open_sb(u + 1)) ok = false;
            else deq(u + 1, 0, wa, wb);
          }
        }
        if (!ok) break;
      }
    }
    };
    if ((pw >> 3) == 0)
      producer(std::integral_constant<int, 0>{});
    else
      producer(std::integral_constant<int, 1>{});
  } else if (warp == TC_RAW_WARP) {
    // ------------------------------------------------------------ weight loader
    // One lane: super-block u of the CTA's item sequence goes to ring slot
    // u % RS as 2-D tensor copies of 128 (gate/up: A0 from the gate matrix, A1
    // from the up matrix) or 256 (down) rows x one super-block column. (An L2
    // prefetch of the next item's rows, tried here, cost more in tensor-copy
    // queue time than it saved.)
    if (lane == 0) {
      const int NU = n_mine * KB;
      auto block_of = [&](int j, int& e, int& y0) {
        const int wi = (int)blockIdx.x + j * (int)gridDim.x;
        const Chunk ch = chunk_at(g.chunks, wi / NB);
        const int blk = wi % NB;
        e = ch.e;
        y0 = GATEUP ? (e < g.E ? e * g.F : 0) + blk * 128 : (e < g.E ? e * g.H : 0) + blk * 256;
      };
      if constexpr (tc_rowcopy<QT>()) {
        // item j: its 256 rows (every super-block) as four bulk copies of 64
        // rows, each 16-byte aligned (64 x 210 x KB bytes)
        const size_t pitch = (size_t)KB * BYTES;
        for (int j = 0; j < n_mine; ++j) {
          if (!tc::mbar_wait(&raw_empty[0], (j & 1) ^ 1, abort_flag, lim)) break;
          int e, y0;
          block_of(j, e, y0);
          const uint8_t* src = (e < g.E ? g.W : g.S) + (size_t)y0 * pitch;
          tc::mbar_expect_tx(&raw_full[0], (uint32_t)(256 * pitch));
          for (int q = 0; q < 4; ++q)
            tc::bulk_g2s(sRaw + (size_t)q * 64 * pitch, src + (size_t)q * 64 * pitch, (uint32_t)(64 * pitch),
                         &raw_full[0]);
        }
      }
      for (int u = 0; u < NU && !tc_rowcopy<QT>(); ++u) {
        const int slot = u % RS;
        if (!tc::mbar_wait(&raw_empty[slot], ((u / RS) & 1) ^ 1, abort_flag, lim)) break;
        const int j = u / KB, sb = u % KB;
        int e, y0;
        block_of(j, e, y0);
        uint8_t* dst = sRaw + (size_t)slot * Cfg::RAW_STAGE;
        tc::mbar_expect_tx(&raw_full[slot], 256 * BYTES);
        const int x = sb * BYTES;
        if (GATEUP) {
          tc::tma_load_2d(dst, e < g.E ? &maps.w : &maps.s, x, y0, &raw_full[slot]);
          tc::tma_load_2d(dst + 128 * BYTES, e < g.E ? &maps.w2 : &maps.s2, x, y0, &raw_full[slot]);
        } else {
          tc::tma_load_2d(dst, e < g.E ? &maps.w : &maps.s, x, y0, &raw_full[slot]);
        }
      }
    }
    __syncwarp();
  } else if (warp == TC_LOAD_WARP) {
    // ------------------------------------------------------------ token loader
    // The chunk's rows are consecutive rows of the token matrix (X in
    // permutation order, or h): per k-tile one lane copies them as boxes of
    // 32 rows x 64 values with 128-byte swizzle, which is the layout the MMA's
    // operand descriptor describes. Rows past the chunk (up to the MMA N, or
    // to the next multiple of 32) are the next rows of the matrix or zero fill
    // past its end; their outputs are never stored. (Boxes of 16 rows took
    // twice the copy instructions and queued behind the weight copies.)
    if (lane == 0) {
      int kg = 0;
      bool ok = true;
      for (int wi = blockIdx.x; wi < total && ok; wi += gridDim.x) {
        const Chunk ch = chunk_at(g.chunks, wi / NB);
        const int n32 = (ch.n + 31) >> 5;  // NMAX is a multiple of 32
        const int pos0 = g.offsets[ch.e] + ch.c0 - (ch.e == g.E ? g.tok_shift : 0);
        for (int kt = 0; kt < KT; ++kt, ++kg) {
          const int stage = kg % TS;
          if (!tc::mbar_wait(&tok_empty[stage], ((kg / TS) & 1) ^ 1, abort_flag, lim)) {
            ok = false;
            break;
          }
          uint8_t* b_st = sB + stage * TC_B_BYTES;
          tc::mbar_expect_tx(&tok_full[stage], (uint32_t)n32 * (BK / 64) * 32 * 128);
          for (int half = 0; half < BK / 64; ++half)
            for (int i = 0; i < n32; ++i)
              tc::tma_load_2d(b_st + half * TC_B_HALF + i * 4096, &maps.tok, kt * BK + 64 * half, pos0 + 32 * i,
                              &tok_full[stage]);
        }
      }
    }
    __syncwarp();
  } else if (warp == TC_MMA_WARP || warp == TC_MMA_WARP2) {
    // ------------------------------------------------------------ MMA issuers
    // Two warps, one per accumulator (D0 from A0, D1 from A1), each issuing
    // from its lane 0 and committing its own MMAs: a commit holds up the
    // issuing thread for a while, and the other warp's MMAs fill that gap.
    // The other lanes wait at the end; operand descriptors are precomputed.
    const int which = warp == TC_MMA_WARP ? 0 : 1;
    if (lane == 0) {
      const uint32_t d_tmem = tmem + (uint32_t)which * TC_D1_COL;
      // descriptor of token stage 0; stage t starts t * TC_B_BYTES / 16 units later
      const uint64_t bdesc0 = tc::sw128_desc(tc::smem_u32(sB));
      int kg = 0;
      int it = 0;
      bool ok = true;
      for (int wi = blockIdx.x; wi < total && ok; wi += gridDim.x, ++it) {
        const Chunk ch = chunk_at(g.chunks, wi / NB);
        const uint32_t idesc = tc::idesc_bf16_f32(128, (ch.n + 15) & ~15);
        if (!tc::mbar_wait(acc_empty, (it & 1) ^ 1, abort_flag, lim)) break;
        tc::tc_fence_after();
        int stage = kg % S, ts = kg % TS;
        for (int kt = 0; kt < KT; ++kt, ++kg) {
          if (!tc::mbar_wait_spin(&tok_full[ts], (kg / TS) & 1, abort_flag, lim) ||
              !tc::mbar_wait_spin(&full[stage], (kg / S) & 1, abort_flag, lim)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a = tmem + TC_A_COL + (uint32_t)stage * Cfg::A_STAGE_COLS + (uint32_t)which * (BK / 2);
          // the descriptor's start address (16-byte units, low bits) advances by
          // 32 bytes per K step of 16 within a K half, by TC_B_HALF per half
          const uint64_t bd = bdesc0 + (uint64_t)(ts * (TC_B_BYTES >> 4));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_bf16_ts(d_tmem, a + 8 * kk, bd + (uint64_t)((kk >> 2) * (TC_B_HALF >> 4) + 2 * (kk & 3)), idesc,
                            (kt | kk) != 0);
          tc::mma_commit(&empty[stage]);
          if (++stage == S) stage = 0;
          if (++ts == TS) ts = 0;
        }
        if (ok) tc::mma_commit(acc_full);
      }
      // drain: every MMA this thread issued has completed before TMEM is freed
      tc::mma_commit(&drain[which]);
      volatile int never = 0;
      tc::mbar_wait(&drain[which], 0, &never, lim);
    }
    __syncwarp();
  }

  if (*abort_flag && threadIdx.x == 0) record_status(g.status, QMOE_ERR_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == TC_MMA_WARP) tc::tmem_dealloc(tmem, 512);
}

// Builds the token-chunk list: every expert with rows (the shared expert
// last) is cut into ceil(rows / cap) chunks of near-equal size (first row
// below 2^24, packed with the row count - 1 in the top 8 bits). One CTA; the scan of chunk counts
// runs in warp 0.
__global__ void __launch_bounds__(1024) build_chunks_kernel(const int32_t* __restrict__ offsets, int E, int cap,
                                                            int2* __restrict__ chunks,
                                                            int32_t* __restrict__ n_chunks) {
  extern __shared__ int32_t start[];  // [E+1] chunk counts, then their exclusive scan
  const int lane = threadIdx.x & 31;
  // the counts first, all loads in flight at once
  for (int e = threadIdx.x; e <= E; e += blockDim.x) start[e] = (offsets[e + 1] - offsets[e] + cap - 1) / cap;
  __syncthreads();
  if (threadIdx.x < 32) {
    int run = 0;
    for (int b = 0; b <= E; b += 32) {
      const int e = b + lane;
      const int c = e <= E ? start[e] : 0;
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e <= E) start[e] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) n_chunks[0] = run;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    const int Me = offsets[e + 1] - offsets[e];
    if (Me <= 0) continue;
    const int nc = (Me + cap - 1) / cap;
    for (int i = 0; i < nc; ++i) {
      // rows [i*Me/nc, (i+1)*Me/nc): between 1 and cap of them
      const int c0 = (int)((long long)i * Me / nc);
      const int c1 = (int)((long long)(i + 1) * Me / nc);
      chunks[start[e] + i] = make_int2(e, (int)((uint32_t)c0 | ((uint32_t)(c1 - c0 - 1) << 24)));
    }
  }
}

// out_t = R_t + y_shared,t + sum_s w_{t,s} y_{t,s} with bf16 y, in slot order;
// y's rows are in permutation order, inv[pair] is the row of a pair.
__global__ void __launch_bounds__(256) combine_bf16_kernel(const __nv_bfloat16* __restrict__ y,
                                                           const int32_t* __restrict__ inv,
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
      uint4 v = reinterpret_cast<const uint4*>(y + (size_t)inv[T * k + t] * H)[c];
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
      uint4 v = reinterpret_cast<const uint4*>(y + (size_t)inv[t * k + s] * H)[c];
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

// y[i] = bf16(x[row(i)]) (round to nearest even) for the rows i of y, in the
// operand K order (kPerm8 inside each group of 8): the token operand of the
// tensor-core path. row(i) = i, or with ``perm`` the token of permutation
// position i (pairs t*k + s, then the shared expert's rows t); then also
// inv[perm[i]] = i, the position of each pair. One warp per row: the row's
// source is looked up once, and each lane has K/256 groups of 8 values (two
// 16-byte loads each) in flight at once.
__global__ void __launch_bounds__(256) to_bf16_kernel(const float* __restrict__ x, __nv_bfloat16* __restrict__ y,
                                                      int rows, int K, const int32_t* __restrict__ perm, int T,
                                                      int k, int32_t* __restrict__ inv) {
  const int lane = threadIdx.x & 31;
  const int K8 = K / 8;
  const int wpb = blockDim.x >> 5;
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpb) {
    const int pr = perm ? perm[r] : r;
    const int src = perm ? tc_pair_row(pr, T, k) : r;
    if (inv != nullptr && lane == 0) inv[pr] = r;
    const float4* x4 = reinterpret_cast<const float4*>(x + (size_t)src * K);
    uint4* y4 = reinterpret_cast<uint4*>(y + (size_t)r * K);
    constexpr int G = 8;  // groups a lane converts per pass (K = 2048: the whole row)
    for (int c0 = 0; c0 < K8; c0 += 32 * G) {
      float4 a[G], b[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int c = c0 + 32 * j + lane;
        if (c < K8) {
          a[j] = __ldg(x4 + 2 * c);
          b[j] = __ldg(x4 + 2 * c + 1);
        }
      }
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int c = c0 + 32 * j + lane;
        if (c < K8) {
          // group (0..7) = a.x a.y a.z a.w b.x b.y b.z b.w -> order 0,4,1,5,2,6,3,7
          uint4 o;
          o.x = tc::pack_bf16x2(a[j].x, b[j].x);
          o.y = tc::pack_bf16x2(a[j].y, b[j].y);
          o.z = tc::pack_bf16x2(a[j].z, b[j].z);
          o.w = tc::pack_bf16x2(a[j].w, b[j].w);
          y4[c] = o;
        }
      }
    }
  }
}

cudaError_t launch_to_bf16(const float* x, __nv_bfloat16* y, int rows, int K, const int32_t* perm, int T, int k,
                           int32_t* inv, cudaStream_t st) {
  // 8 rows (warps) a block, up to 8 blocks per SM
  int blocks = (rows + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  to_bf16_kernel<<<blocks, 256, 0, st>>>(x, y, rows, K, perm, T, k, inv);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
int tc_max_chunks(int T, int k, int E, int has_shared) {
  const int P = T * k;
  return (P + (has_shared ? T : 0)) / TC_N_MIN + E + 1;
}

int tc_chunk_cap(int T, int k, int E) {
  const long long P = (long long)T * k;
  return P <= 32LL * E ? 64 : (P <= (long long)TC_CAP192_MIN_ROWS * E ? 128 : 192);
}

cudaError_t launch_build_chunks(const int32_t* offsets, int E, int cap, int2* chunks, int32_t* n_chunks,
                                cudaStream_t st) {
  if (cap != 64 && cap != 128 && cap != 192) return cudaErrorInvalidValue;
  build_chunks_kernel<<<1, 1024, sizeof(int32_t) * (E + 1), st>>>(offsets, E, cap, chunks, n_chunks);
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled, taken from the driver through the runtime once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a packed matrix seen as bytes [rows][row_bytes], box = one
// super-block column (``bytes``) x ``box_rows`` rows, no swizzle. Encoded maps
// are kept in a small cache keyed by their arguments (a map is 128 bytes and
// holds no device state).
static bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t bytes,
                        uint32_t box_rows) {
  if (base == nullptr) {
    memset(m, 0, sizeof(*m));
    return true;
  }
  struct Entry {
    const void* base;
    uint64_t rows, row_bytes;
    uint32_t bytes, box_rows;
    CUtensorMap map;
  };
  static Entry cache[32];
  static int n = 0, next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i) {
    const Entry& c = cache[i];
    if (c.base == base && c.rows == rows && c.row_bytes == row_bytes && c.bytes == bytes && c.box_rows == box_rows) {
      *m = c.map;
      return true;
    }
  }
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& c = cache[next];
  c = Entry{base, rows, row_bytes, bytes, box_rows, *m};
  next = (next + 1) % 32;
  if (n < 32) ++n;
  return true;
}

template <bool GATEUP, int QT, int NMAX>
static cudaError_t tc_launch_n(const TcArgs& a, const TcMaps& maps, int max_items, cudaStream_t st) {
  static_assert(TcCfg<QT, NMAX>::SMEM <= 227 * 1024, "shared memory per CTA");
  static_assert(TcCfg<QT, NMAX>::S >= 2 && TcCfg<QT, NMAX>::TS >= TcCfg<QT, NMAX>::S, "ring depths");
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(moe_tc_kernel<GATEUP, QT, NMAX>),
                                     TcCfg<QT, NMAX>::SMEM);
  if (e != cudaSuccess) return e;
  int grid = device_sm_count();
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  moe_tc_kernel<GATEUP, QT, NMAX><<<grid, TC_THREADS, TcCfg<QT, NMAX>::SMEM, st>>>(a, maps);
  return cudaGetLastError();
}

template <bool GATEUP, int QT>
static cudaError_t tc_launch_t(const TcArgs& a, const TcMaps& maps, int max_items, int nmax, cudaStream_t st) {
  return nmax == 64    ? tc_launch_n<GATEUP, QT, 64>(a, maps, max_items, st)
         : nmax == 128 ? tc_launch_n<GATEUP, QT, 128>(a, maps, max_items, st)
                       : tc_launch_n<GATEUP, QT, 192>(a, maps, max_items, st);
}

static TcArgs tc_args(const GroupedTcArgs& p) {
  TcArgs a{};
  a.W = p.W; a.W2 = p.W2; a.S = p.S; a.S2 = p.S2;
  a.offsets = p.offsets; a.perm = p.perm; a.chunks = p.chunks; a.n_chunks = p.n_chunks;
  a.xb = p.xb; a.hin = p.hin; a.hout = p.hout; a.yout = p.yout; a.yout_f32 = p.yout_f32;
  a.tok_shift = p.tok_shift;
  a.T = p.T; a.k = p.k; a.E = p.E; a.H = p.H; a.F = p.F; a.status = p.status;
  a.wait_ns = p.wait_ns ? p.wait_ns : tc::kWaitLimitNs;
  a.fault = p.fault;
  return a;
}

// Token matrix [rows][K] bf16 as boxes of 32 rows x 64 values, 128-byte swizzle.
static bool encode_tokens(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K) {
  struct Entry {
    const void* base;
    uint64_t rows, K;
    CUtensorMap map;
  };
  static Entry cache[16];
  static int n = 0, next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].base == base && cache[i].rows == rows && cache[i].K == K) {
      *m = cache[i].map;
      return true;
    }
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {64, 32};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next] = Entry{base, rows, K, *m};
  next = (next + 1) % 16;
  if (n < 16) ++n;
  return true;
}

cudaError_t launch_gateup_tc(const GroupedTcArgs& p, cudaStream_t st) {
  const TcArgs a = tc_args(p);
  const uint32_t bytes = (uint32_t)qtype_bytes(p.qt);
  const uint64_t rb = (uint64_t)(p.H / QK) * bytes;
  TcMaps m;
  if (!encode_rows(&m.w, p.W, (uint64_t)p.E * p.F, rb, bytes, 128) ||
      !encode_rows(&m.w2, p.W2, (uint64_t)p.E * p.F, rb, bytes, 128) ||
      !encode_rows(&m.s, p.S, (uint64_t)p.F, rb, bytes, 128) || !encode_rows(&m.s2, p.S2, (uint64_t)p.F, rb, bytes, 128) ||
      !encode_tokens(&m.tok, p.xb, (uint64_t)p.tok_rows, (uint64_t)p.H))
    return cudaErrorInvalidValue;
  const int items = p.max_chunks * (p.F / 128);
  return p.qt == QMOE_Q5K ? tc_launch_t<true, QMOE_Q5K>(a, m, items, p.nmax, st)
                          : tc_launch_t<true, QMOE_Q4K>(a, m, items, p.nmax, st);
}

cudaError_t launch_down_tc(const GroupedTcArgs& p, cudaStream_t st) {
  const TcArgs a = tc_args(p);
  const uint32_t bytes = (uint32_t)qtype_bytes(p.qt);
  const uint64_t rb = (uint64_t)(p.F / QK) * bytes;
  TcMaps m;
  if (p.qt == QMOE_Q6K || p.qt == QMOE_MXFP4) {
    // whole rows by bulk copies (no weight tensor maps)
    if (p.F / QK > TC_ROWCOPY_KB || !encode_tokens(&m.tok, p.hin, (uint64_t)p.tok_rows, (uint64_t)p.F))
      return cudaErrorInvalidValue;
    memset(&m.w, 0, sizeof(m.w));
    memset(&m.s, 0, sizeof(m.s));
    memset(&m.w2, 0, sizeof(m.w2));
    memset(&m.s2, 0, sizeof(m.s2));
    return p.qt == QMOE_Q6K ? tc_launch_t<false, QMOE_Q6K>(a, m, p.max_chunks * (p.H / 256), p.nmax, st)
                            : tc_launch_t<false, QMOE_MXFP4>(a, m, p.max_chunks * (p.H / 256), p.nmax, st);
  }
  if (!encode_rows(&m.w, p.W, (uint64_t)p.E * p.H, rb, bytes, 256) ||
      !encode_rows(&m.s, p.S, (uint64_t)p.H, rb, bytes, 256) ||
      !encode_tokens(&m.tok, p.hin, (uint64_t)p.tok_rows, (uint64_t)p.F))
    return cudaErrorInvalidValue;
  memset(&m.w2, 0, sizeof(m.w2));
  memset(&m.s2, 0, sizeof(m.s2));
  const int items = p.max_chunks * (p.H / 256);
  return p.qt == QMOE_Q5K ? tc_launch_t<false, QMOE_Q5K>(a, m, items, p.nmax, st)
                          : tc_launch_t<false, QMOE_Q4K>(a, m, items, p.nmax, st);
}

cudaError_t launch_combine_bf16(const __nv_bfloat16* y, const int32_t* inv, const float* w, const float* R, float* out,
                                int T, int H, int k, int has_shared, cudaStream_t st) {
  const size_t n = (size_t)T * (H / 8);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  combine_bf16_kernel<<<blocks, 256, 0, st>>>(y, inv, w, R, out, T, H, k, has_shared);
  return cudaGetLastError();
}

}  // namespace qmoe
