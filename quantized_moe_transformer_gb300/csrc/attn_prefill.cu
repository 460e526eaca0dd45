// Causal attention for many query rows (block prefill), on the tensor cores.
//
// "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "What PR #382
// Now Splits": 16 query heads over 2 KV heads, so query head h attends to the
// keys and values of KV head h / 8, causally, with the 1/sqrt(head_dim) scale.
// "Distributed CPU: Zip Fusion Beyond Tensor Parallelism", "Two-Dimensional
// Attention at Long Context": the softmax over key blocks is carried by its
// running maximum, normaliser and weighted output, which is how this kernel
// walks the keys.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

// CTA = (128 query rows, one head); key blocks of 128.
//   S_j = Q K_j^T   Q scaled by log2(e)/sqrt(hd) and split into two bf16
//                   parts (hi = bf16(q), lo = bf16(q - hi)), two MMAs per K
//                   step, so that S carries about 16 bits of q (with scores
//                   of a few thousand, which random weights give, the 2^-9
//                   step of a bf16 q alone would move the softmax argument by
//                   several units); K is exact (the cache is bf16); Q and K_j
//                   in shared memory
//                   (128-byte swizzled, K-major), fp32 S in TMEM, two S
//                   buffers so that S_{j+1} is computed while the softmax
//                   reads S_j;
//   softmax         warps 0-7: warps w and w + 4 share TMEM lane quarter
//                   w % 4 (query rows 32 (w % 4) ..), and each takes half of
//                   every row's 128 scores; the two halves' maxima meet in
//                   shared memory (an mbarrier per warp pair and block
//                   parity, every lane of both warps arriving) so both use
//                   the same reference; p = exp2(s - m) written back to
//                   TMEM as bf16 P_j (two buffers), the normaliser l summed
//                   in fp32 per half and added at the end;
//   O += P_j V_j    P_j from TMEM as the A operand, V_j from shared memory as
//                   an MN-major B operand (its rows are keys, head dims
//                   contiguous), fp32 O in TMEM.
// The running max m is a reference, not the exact maximum: O and l are
// rescaled by exp2(m_old - m_new) only when a row's maximum exceeds m by more
// than 2^8 (so p <= 256), which leaves out(t) = O / l unchanged in exact
// arithmetic; the rescale waits for the previous P V to complete.
// Warps 8 and 10 copy K_j and V_j (2-D boxes of 64 head dims x 128 keys of
// one KV head, by a 3-D tensor map [position][kv head][head dim]) into two
// rings of two stages each: a K stage is refilled as soon as S_j is computed,
// a V stage once P_j V_j is, each by its own thread so that neither waits on
// the other. Warp 9 allocates TMEM and issues the S MMAs, warp 11 the P V
// MMAs, each from one lane (a thread issues an MMA in about 80 cycles, so a
// single issuer would add up to about a microsecond a block). Every wait is bounded: on time-out the CTA records
// QMOE_ERR_TIMEOUT, drains its MMAs, frees its TMEM and returns.
constexpr int AT_BQ = 128, AT_BK = 128, AT_HD = 128;
constexpr int AT_SOFT_WARPS = 8;
constexpr int AT_THREADS = 32 * (AT_SOFT_WARPS + 4);
constexpr int AT_KLOAD_WARP = AT_SOFT_WARPS, AT_MMA_WARP = AT_SOFT_WARPS + 1;
constexpr int AT_VLOAD_WARP = AT_SOFT_WARPS + 2, AT_PV_WARP = AT_SOFT_WARPS + 3;
constexpr int AT_HALF = 128 * 128;               // 128 rows x 64 bf16 (one K half of a tile)
constexpr int AT_Q_BYTES = 4 * AT_HALF;          // 64 KB: hi part (two K halves), then lo part
constexpr int AT_TILE = 2 * AT_HALF;             // K_j or V_j: 32 KB
constexpr int AT_STAGES = 2;                     // per ring (K, V)
constexpr int AT_XCH_BYTES = 2 * 2 * AT_BQ * 4;  // row maxima of both halves, two blocks deep
constexpr int AT_SMEM = 1024 + AT_Q_BYTES + 2 * AT_STAGES * AT_TILE + AT_XCH_BYTES + 512;
constexpr uint32_t AT_S_COL = 0;                 // S buffer b at 128 b
constexpr uint32_t AT_O_COL = 256;
constexpr uint32_t AT_P_COL = 384;               // P buffer b at 384 + 64 b
constexpr float AT_RESCALE_LOG2 = 8.f;

__device__ __forceinline__ void at_tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                               uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit TMEM columns at ``ta``, then the wait.
__device__ __forceinline__ void at_tmem_ld32(uint32_t ta, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(ta)
      : "memory");
}

// 32 lanes x 64 consecutive 32-bit TMEM columns at ``ta`` (two loads of 32
// columns in flight at once), then the wait, in one statement so that no use
// of the registers is scheduled before the data has arrived.
__device__ __forceinline__ void at_tmem_ld64(uint32_t ta, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
      : "r"(ta), "r"(ta + 32)
      : "memory");
}

// Descriptor of an MN-major operand with 128-byte swizzle: rows of 128 bytes
// (64 values along N) for consecutive K, 8-row atoms of 1024 bytes; the
// leading byte offset steps to the next 64 values along N, the stride byte
// offset to the next 8 rows along K.
__device__ __forceinline__ uint64_t at_mn_sw128_desc(uint32_t smem_addr, uint32_t lbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// q [T][nh][128] fp32 (rotated), the caches through the tensor maps
// (positions [0, pos0 + T)), o [T][nh][128] fp32; query t sits at position
// pos0 + t and sees keys 0 .. pos0 + t.
__global__ void __launch_bounds__(AT_THREADS, 1)
    attn_prefill_tc_kernel(const float* __restrict__ q, float* __restrict__ o, __nv_bfloat16* __restrict__ ob,
                           int T, int pos0, int nh, int nkv,
                           int* status, unsigned long long wait_ns, int fault,
                           const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t at_smem_raw[];
  const uint32_t s0 = tc::smem_u32(at_smem_raw);
  uint8_t* smem = at_smem_raw + (((s0 + 1023u) & ~1023u) - s0);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + AT_Q_BYTES;              // [2] K stages
  uint8_t* sV = sK + AT_STAGES * AT_TILE;       // [2] V stages
  float* xch = reinterpret_cast<float*>(sV + AT_STAGES * AT_TILE);  // [2 blocks][2 halves][128 rows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + AT_STAGES * AT_TILE + AT_XCH_BYTES);
  uint64_t* k_full = bars;        // [2] K_j landed
  uint64_t* k_empty = bars + 2;   // [2] S_j done (the K stage may be refilled)
  uint64_t* v_full = bars + 4;    // [2] V_j landed
  uint64_t* v_empty = bars + 6;   // [2] P_j V_j done (the V stage may be refilled)
  uint64_t* s_full = bars + 8;    // [2] S_j computed
  uint64_t* s_free = bars + 10;   // [2] S buffer read by the softmax
  uint64_t* p_full = bars + 12;   // [2] P_j stored
  uint64_t* p_free = bars + 14;   // [2] P_j V_j done (P buffer reusable, O current)
  uint64_t* q_ready = bars + 16;
  uint64_t* o_final = bars + 17;
  uint64_t* drain = bars + 18;    // [2] one per MMA issuer
  uint64_t* x_bar = bars + 20;    // [2 block parities][4 lane quarters] both halves' maxima written
  uint64_t* l_bar = bars + 28;    // [4 lane quarters] both halves' normalisers written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;  // late (long) query tiles first
  const int h = blockIdx.y, kvh = h / (nh / nkv);
  const int q0 = qt * AT_BQ;
  const int last_row = min(T - 1, q0 + AT_BQ - 1);
  const int nb = (pos0 + last_row + 1 + AT_BK - 1) / AT_BK;  // key blocks
  const uint64_t lim = wait_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&k_full[i], 1);
      tc::mbar_init(&k_empty[i], 1);
      tc::mbar_init(&v_full[i], 1);
      tc::mbar_init(&v_empty[i], 1);
      tc::mbar_init(&s_full[i], 1);
      tc::mbar_init(&s_free[i], AT_SOFT_WARPS);
      tc::mbar_init(&p_full[i], AT_SOFT_WARPS);
      tc::mbar_init(&p_free[i], 1);
    }
    tc::mbar_init(q_ready, AT_SOFT_WARPS);
    for (int i = 0; i < 8; ++i) tc::mbar_init(&x_bar[i], 64);
    for (int i = 0; i < 4; ++i) tc::mbar_init(&l_bar[i], 64);
    tc::mbar_init(o_final, 1);
    tc::mbar_init(&drain[0], 1);
    tc::mbar_init(&drain[1], 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == AT_MMA_WARP) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < AT_SOFT_WARPS) {
    // ------------------------------------------------------------ softmax
    const int lq = warp & 3, half = warp >> 2;  // TMEM lane quarter, half of the row's columns
    const int r = 32 * lq + lane, t = q0 + r;
    const int pr = pos0 + t;  // this row's position
    // Q row (this thread's half) -> bf16 hi and lo parts, scaled, into the
    // swizzled K-major tiles
    {
      const float qscale = 1.4426950408889634f * rsqrtf((float)AT_HD);
      const float* qr = q + ((size_t)(t < T ? t : 0) * nh + h) * AT_HD;
#pragma unroll 4
      for (int c = 8 * half; c < 8 * half + 8; ++c) {
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (t < T) {
          const float4 a = *reinterpret_cast<const float4*>(qr + 8 * c);
          const float4 b = *reinterpret_cast<const float4*>(qr + 8 * c + 4);
          x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
          x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = x[2 * i] * qscale, x1 = x[2 * i + 1] * qscale;
          hi[i] = tc::pack_bf16x2(x0, x1);
          lo[i] = tc::pack_bf16x2(x0 - __uint_as_float(hi[i] << 16), x1 - __uint_as_float(hi[i] & 0xFFFF0000u));
        }
        const uint32_t off = (uint32_t)(c >> 3) * AT_HALF + tc::sw128_offset(r, c & 7);
        *reinterpret_cast<uint4*>(sQ + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(sQ + 2 * AT_HALF + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(q_ready);
    }
    const uint32_t tq = tmem + ((uint32_t)(32 * lq) << 16);
    const uint32_t col = 64u * half;  // this warp's score columns (keys) and O columns (head dims)
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nb && ok; ++j) {
      const int b = j & 1;
      // (polling waits: the softmax is on the critical path, and a suspended
      // thread wakes up late)
      if (!__all_sync(0xffffffffu, tc::mbar_wait_poll(&s_full[b], (j >> 1) & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const int k0 = j * AT_BK + (int)col;
      const bool diag = k0 + 63 > pos0 + q0;
      // this half's 64 scores of the row, masked past the row's position
      uint32_t v[64];
      at_tmem_ld64(tq + AT_S_COL + 128u * b + col, v);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&s_free[b]);  // the S buffer may be overwritten
      if (diag) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (k0 + i > pr) v[i] = __float_as_uint(-INFINITY);
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 64; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(v[i]));
      float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // the row's maximum over both halves (every lane arrives after its own
      // store, which the arrival releases)
      float* xb = xch + (size_t)b * 2 * AT_BQ;
      xb[half * AT_BQ + r] = mx;
      tc::mbar_arrive(&x_bar[4 * b + lq]);
      if (!__all_sync(0xffffffffu, tc::mbar_wait_poll(&x_bar[4 * b + lq], (j >> 1) & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, xb[(half ^ 1) * AT_BQ + r]);
      // a new reference where the row maximum outgrew the old one; O is
      // rescaled below, after the exponentials, when P_{j-1} V_{j-1} is done
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m = mx;
      } else {
        const bool need = mx > m + AT_RESCALE_LOG2;
        rescale = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = exp2f(m - mx);
          m = mx;
          l *= alpha;
        }
      }
      // p = exp2(s - m) as bf16 P (masked scores give 0), the normaliser in fp32
      const float mref = m == -INFINITY ? 0.f : m;
      const uint64_t one2 = pack2(__float_as_uint(1.f), __float_as_uint(1.f));
      const uint64_t negm2 = pack2(__float_as_uint(-mref), __float_as_uint(-mref));
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 d = unpack2(ffma2(pack2(v[2 * i], v[2 * i + 1]), one2, negm2));
        const float p0 = exp2f(d.x), p1 = exp2f(d.y);
        l4[i & 3] += p0 + p1;
        v[i] = tc::pack_bf16x2(p0, p1);  // packed in place: v[i] is no longer needed as a score
      }
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      if (rescale) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled (this warp's 64 columns)
        if (!__all_sync(0xffffffffu, tc::mbar_wait_poll(&p_free[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        uint32_t ov[32];
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          at_tmem_ld32(tq + AT_O_COL + col + 32 * c, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tc::tmem_st16(tq + AT_O_COL + col + 32 * c, ov);
          tc::tmem_st16(tq + AT_O_COL + col + 32 * c + 16, ov + 16);
        }
        tc::tmem_wait_st();
      }
      // P buffer b is reusable once P_{j-2} V_{j-2} is done
      if (j >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait_poll(&p_free[b], ((j - 2) >> 1) & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint32_t tp = tq + AT_P_COL + 64u * b + 32u * half;
      tc::tmem_st16(tp, v);
      tc::tmem_st16(tp + 16, v + 16);
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&p_full[b]);
    }
    // out = O / l, l over both halves; each warp stores its 64 head dims
    if (ok) {
      // the exchange slots of the block parity the last block did not use
      float* xb = xch + (size_t)(nb & 1) * 2 * AT_BQ;
      xb[half * AT_BQ + r] = l;
      tc::mbar_arrive(&l_bar[lq]);
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&l_bar[lq], 0, abort_flag, lim));
      if (ok) l += xb[(half ^ 1) * AT_BQ + r];
    }
    if (ok && __all_sync(0xffffffffu, tc::mbar_wait(o_final, 0, abort_flag, lim))) {
      tc::tc_fence_after();
      const float il = 1.f / l;
      const size_t row0 = ((size_t)(t < T ? t : 0) * nh + h) * AT_HD + col;
      uint32_t v[32];
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        at_tmem_ld32(tq + AT_O_COL + col + 32 * c, v);
        if (t < T && ob != nullptr) {
          // bf16 (nearest even) in the tensor-core operand order: word i of
          // a group of 8 head dims holds dims i and i + 4
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            uint4 w;
            w.x = tc::pack_bf16x2(__uint_as_float(v[8 * m + 0]) * il, __uint_as_float(v[8 * m + 4]) * il);
            w.y = tc::pack_bf16x2(__uint_as_float(v[8 * m + 1]) * il, __uint_as_float(v[8 * m + 5]) * il);
            w.z = tc::pack_bf16x2(__uint_as_float(v[8 * m + 2]) * il, __uint_as_float(v[8 * m + 6]) * il);
            w.w = tc::pack_bf16x2(__uint_as_float(v[8 * m + 3]) * il, __uint_as_float(v[8 * m + 7]) * il);
            *reinterpret_cast<uint4*>(ob + row0 + 32 * c + 8 * m) = w;
          }
        } else if (t < T) {
          float* orow = o + row0;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(orow + 32 * c + 4 * i) =
                make_float4(__uint_as_float(v[4 * i]) * il, __uint_as_float(v[4 * i + 1]) * il,
                            __uint_as_float(v[4 * i + 2]) * il, __uint_as_float(v[4 * i + 3]) * il);
        }
      }
    }
  } else if (warp == AT_KLOAD_WARP || warp == AT_VLOAD_WARP) {
    // ------------------------------------------------------------ K or V copies
    // K_j as soon as S_{j-2} is done, V_j as soon as P_{j-2} V_{j-2} is
    if (lane == 0) {
      const bool is_k = warp == AT_KLOAD_WARP;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = is_k ? sK : sV;
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      for (int j = 0; j < nb; ++j) {
        const int st = j & 1;
        if (!tc::mbar_wait(&empty[st], ((j >> 1) & 1) ^ 1, abort_flag, lim)) break;
        const uint32_t dst = tc::smem_u32(ring + st * AT_TILE);
        const uint32_t bar = tc::smem_u32(&full[st]);
        tc::mbar_expect_tx(&full[st], AT_TILE);
        at_tma_load_3d(dst, map, 0, kvh, j * AT_BK, bar);
        at_tma_load_3d(dst + AT_HALF, map, 64, kvh, j * AT_BK, bar);
      }
    }
    __syncwarp();
  } else if (warp == AT_MMA_WARP) {
    // ------------------------------------------------------------ S = Q K^T
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(AT_BQ, AT_BK);
      const uint64_t qd = tc::sw128_desc(tc::smem_u32(sQ));                  // hi part
      const uint64_t qld = tc::sw128_desc(tc::smem_u32(sQ + 2 * AT_HALF));   // lo part
      bool ok = tc::mbar_wait(q_ready, 0, abort_flag, lim);
      for (int j = 0; j < nb && ok; ++j) {
        const int st = j & 1;
        if (!tc::mbar_wait_poll(&k_full[st], (j >> 1) & 1, abort_flag, lim) ||
            (j >= 2 && !tc::mbar_wait_poll(&s_free[st], ((j - 2) >> 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint64_t kd = tc::sw128_desc(tc::smem_u32(sK + st * AT_TILE));
        const uint32_t d = tmem + AT_S_COL + 128u * st;
#pragma unroll
        for (int kk = 0; kk < AT_HD / 16; ++kk) {
          const uint64_t off = (uint64_t)((kk >> 2) * (AT_HALF >> 4) + 2 * (kk & 3));
          tc::mma_bf16(d, qd + off, kd + off, idesc_s, kk != 0);
          tc::mma_bf16(d, qld + off, kd + off, idesc_s, 1u);
        }
        tc::mma_commit(&s_full[st]);
        tc::mma_commit(&k_empty[st]);
      }
      // drain: every MMA issued here has completed before TMEM is freed
      tc::mma_commit(&drain[0]);
      volatile int never = 0;
      tc::mbar_wait(&drain[0], 0, &never, lim);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ O += P V
    if (lane == 0) {
      const uint32_t idesc_o = tc::idesc_bf16_f32(AT_BQ, AT_HD) | (1u << 16);  // B (V) MN-major
      bool ok = true;
      for (int j = 0; j < nb && ok; ++j) {
        const int b = j & 1;
        // (polling waits: a suspended issuer wakes up late, and each block's
        // P V is on the critical path)
        if (!tc::mbar_wait_poll(&v_full[b], (j >> 1) & 1, abort_flag, lim) ||
            !tc::mbar_wait_poll(&p_full[b], (j >> 1) & 1, abort_flag, lim)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t vs = tc::smem_u32(sV + b * AT_TILE);
#pragma unroll
        for (int kk = 0; kk < AT_BK / 16; ++kk)
          tc::mma_bf16_ts(tmem + AT_O_COL, tmem + AT_P_COL + 64u * b + 8u * kk, at_mn_sw128_desc(vs + 2048u * kk, AT_HALF),
                          idesc_o, (j | kk) != 0);
        tc::mma_commit(&p_free[b]);
        tc::mma_commit(&v_empty[b]);
      }
      // test-only fault: the first CTA never marks O final, so the softmax
      // warps' wait for it runs out (every MMA of the CTA has been issued and
      // is drained below)
      if (ok && !(fault == 1 && blockIdx.x == 0 && blockIdx.y == 0)) tc::mma_commit(o_final);
      tc::mma_commit(&drain[1]);
      volatile int never = 0;
      tc::mbar_wait(&drain[1], 0, &never, lim);
    }
    __syncwarp();
  }

  if (*abort_flag && threadIdx.x == 0) record_status(status, QMOE_ERR_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == AT_MMA_WARP) tc::tmem_dealloc(tmem, 512);
}

// A cache [positions][nkv][128] bf16 as a 3-D tensor map over positions
// [0, rows): boxes of 64 head dims x 1 KV head x 128 positions, 128-byte
// swizzle; positions from ``rows`` on read as zero.
static bool at_encode_cache(CUtensorMap* m, const void* base, int nkv, int rows) {
  struct Entry {
    const void* base;
    int nkv, rows;
    CUtensorMap map;
  };
  static Entry cache[8];
  static int n = 0, next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].base == base && cache[i].nkv == nkv && cache[i].rows == rows) {
      *m = cache[i].map;
      return true;
    }
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)AT_HD, (cuuint64_t)nkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)AT_HD * 2, (cuuint64_t)nkv * AT_HD * 2};
  const cuuint32_t box[3] = {64, 1, AT_BK};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache[next] = Entry{base, nkv, rows, *m};
  next = (next + 1) % 8;
  if (n < 8) ++n;
  return true;
}

cudaError_t launch_attention_prefill_tc(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, float* o,
                                        __nv_bfloat16* ob, int T, int pos0, int nh, int nkv, int* status,
                                        unsigned long long wait_ns, int fault, cudaStream_t st) {
  if (T < 1 || nkv < 1 || nh % nkv != 0) return cudaErrorInvalidValue;
  CUtensorMap km, vm;
  if (!at_encode_cache(&km, kc, nkv, pos0 + T) || !at_encode_cache(&vm, vc, nkv, pos0 + T))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_kernel_smem(reinterpret_cast<const void*>(attn_prefill_tc_kernel), AT_SMEM);
  if (e != cudaSuccess) return e;
  attn_prefill_tc_kernel<<<dim3((T + AT_BQ - 1) / AT_BQ, nh), AT_THREADS, AT_SMEM, st>>>(
      q, o, ob, T, pos0, nh, nkv, status, wait_ns ? wait_ns : tc::kWaitLimitNs, fault, km, vm);
  return cudaGetLastError();
}

}  // namespace qmoe
