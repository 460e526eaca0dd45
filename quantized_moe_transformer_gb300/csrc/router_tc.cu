// Router logits on the tensor cores, at fp32 accuracy, for T >= 256 rows.
//
// "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights", "What The
// First Prototype Split": every row's top-k experts and weights come from its
// router logits L = X Wr (X [T][H], Wr [H][E], fp32). At prefill sizes this
// is a dense fp32 GEMM (4.3 GFLOP at T = 4096), which the CUDA cores run at
// their fp32 rate; here it runs on the bf16 tensor cores without giving up
// fp32 accuracy, because the top-k decisions depend on the low bits.
//
// Every fp32 value v is split exactly into three bf16 parts,
//   v = v1 + v2 + v3 + e,  v1 = bf16(v), v2 = bf16(v - v1), v3 = bf16(v - v1 - v2),
// each a round-to-nearest bf16 (8 significant bits) of what the earlier parts
// leave, with the subtractions exact in fp32, so |e| <= 2^-24 |v|. Of the nine
// products of the parts, the six whose scales are at least 2^-16 of x w,
//   x1 w1 + x1 w2 + x2 w1 + x1 w3 + x3 w1 + x2 w2,
// are accumulated in fp32 in tensor memory; the three dropped ones and the
// split errors stay below about 2^-22 |x w|, the size of fp32 rounding over a
// few operations. The tensor core's fp32 accumulation does not round to
// nearest (measured: with all six products in one accumulator over 1024 K,
// logits drifted by up to 1.5e-5, one sided), so x1 w1 has an accumulator of
// its own and the five smaller products another (2^-8 of the size, so 2^-8 of
// the drift), H is cut into at least 4 slices (at most 32 accumulation steps
// per slice), and the epilogue and the top-k kernels add the pieces in fp32.
//
// One CTA per (128 rows, 128 experts, slice of H): rows are the MMA's M side,
// experts its N side, K = H in stages of 64. Tensor memory: the two
// accumulators in columns [0, 256), two A stages of 96 columns after them.
//   warps 0-7  producers: warp w covers TMEM lane quarter w % 4 (its 32 rows)
//              and K half w / 4 of each stage; a thread loads its row's 32
//              fp32 values (prefetched one stage ahead), splits them and stores
//              the three parts as bf16x2 words into the stage's A columns
//              (tcgen05.st); warps 0-3 then read the accumulator out;
//   warp 8     issues the MMAs (one lane): 4 K steps x 6 part products per
//              stage, A from tensor memory (2-stage ring), B from shared
//              memory (3-stage ring);
//   warp 9     copies the three parts of Wr^T for the CTA's 128 experts
//              (prepared once per call by router_split_wr_kernel, [3][E][H]
//              bf16) into the stage's 128-byte-swizzled tiles (one lane,
//              2-D tensor copies).
// The output is one partial logit per (slice, row, expert), part[s][t][e], as
// for the CUDA-core router; the top-k kernels add the slices in order.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

constexpr int RT_BM = 128;                             // rows per tile (MMA M)
constexpr int RT_BN = 128;                             // experts per tile (MMA N)
constexpr int RT_BK = 64;                              // K per stage: one 128-byte bf16 row
constexpr int RT_STAGES = 3;                           // B ring (shared memory)
constexpr int RT_ASTAGES = 2;                          // A ring (tensor memory)
constexpr int RT_PROD_WARPS = 8;
constexpr int RT_MMA_WARP = RT_PROD_WARPS;             // 8
constexpr int RT_LOAD_WARP = RT_PROD_WARPS + 1;        // 9
constexpr int RT_THREADS = 32 * (RT_PROD_WARPS + 2);   // 320
constexpr int RT_PIECE = RT_BN * 128;                  // one part of Wr^T per stage: 16 KB
constexpr int RT_STAGE_B = 3 * RT_PIECE;               // 48 KB
constexpr uint32_t RT_A_COLS = 3 * (RT_BK / 2);        // three parts x 32 bf16x2 columns
constexpr uint32_t RT_DC_COL = RT_BN;                  // x1 w1 in [0, 128), the rest in [128, 256)
constexpr uint32_t RT_A_COL0 = 2 * RT_BN;
constexpr int RT_SMEM = RT_STAGES * RT_STAGE_B + 1024 /*align*/ + 256 /*barriers*/;

bool router_tc_eligible(int T, int H, int E) {
  return T >= 256 && E % RT_BN == 0 && E <= 1024 && H % (4 * RT_BK) == 0;
}

// At least 4 slices (accuracy, see above), up to 8 while the grid is below
// one CTA per SM.
int router_tc_splits(int T, int H, int E) {
  const int tiles = (E / RT_BN) * ((T + RT_BM - 1) / RT_BM);
  int s = 4;
  while (s < 8 && tiles * s * 2 <= 152 && (H / (s * 2)) % RT_BK == 0 && H / (s * 2) >= 2 * RT_BK) s *= 2;
  return s;
}

size_t router_tc_ws_bytes(int T, int H, int E) {
  return router_tc_eligible(T, H, E) ? (size_t)3 * E * H * sizeof(__nv_bfloat16) : 0;
}

// v = p1 + p2 + p3 (+ below 2^-24 |v|), each part bf16 round-to-nearest of
// the remainder; two values at once, as bf16x2 words (low half = a).
__device__ __forceinline__ void split3(float a, float b, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(a, b);
  const float2 f1 = __bfloat1622float2(h1);
  const float ra = a - f1.x, rb = b - f1.y;
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(ra, rb);
  const float2 f2 = __bfloat1622float2(h2);
  const __nv_bfloat162 h3 = __floats2bfloat162_rn(ra - f2.x, rb - f2.y);
  p1 = *reinterpret_cast<const uint32_t*>(&h1);
  p2 = *reinterpret_cast<const uint32_t*>(&h2);
  p3 = *reinterpret_cast<const uint32_t*>(&h3);
}

// WR3[p][e][h] = part p of Wr[h][e]: the B operand, K-major, for every call
// (Wr is an argument of each call). 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) router_split_wr_kernel(const float* __restrict__ Wr,
                                                              __nv_bfloat16* __restrict__ wr3, int H, int E) {
  __shared__ float tile[32][33];
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int r = ty; r < 32; r += 8) tile[r][tx] = Wr[(size_t)(h0 + r) * E + e0 + tx];
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const float v = tile[tx][r];  // Wr[h0 + tx][e0 + r]
    uint32_t p1, p2, p3;
    split3(v, 0.f, p1, p2, p3);
    const size_t o = (size_t)(e0 + r) * H + h0 + tx;
    const size_t plane = (size_t)E * H;
    wr3[o] = __ushort_as_bfloat16((unsigned short)(p1 & 0xFFFFu));
    wr3[plane + o] = __ushort_as_bfloat16((unsigned short)(p2 & 0xFFFFu));
    wr3[2 * plane + o] = __ushort_as_bfloat16((unsigned short)(p3 & 0xFFFFu));
  }
}

__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const float* __restrict__ X, float* __restrict__ part, int T, int H, int E, int k_per_split,
                     int* status, const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t s0 = tc::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((s0 + 1023u) & ~1023u) - s0);
  uint8_t* sB = smem;  // [RT_STAGES][3 parts][128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RT_STAGES * RT_STAGE_B);
  uint64_t* bfull = bars;                    // [RT_STAGES] B parts landed
  uint64_t* bempty = bars + RT_STAGES;       // [RT_STAGES] MMAs reading them done
  uint64_t* afull = bars + 2 * RT_STAGES;    // [RT_ASTAGES] A parts stored
  uint64_t* aempty = afull + RT_ASTAGES;     // [RT_ASTAGES] MMAs reading them done
  uint64_t* acc_full = aempty + RT_ASTAGES;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * RT_BN, m0 = blockIdx.y * RT_BM, sl = blockIdx.z;
  const int kb = sl * k_per_split;       // first K of this slice
  const int KT = k_per_split / RT_BK;    // stages

  if (threadIdx.x == 0) {
    for (int i = 0; i < RT_STAGES; ++i) {
      tc::mbar_init(&bfull[i], 1);  // the loader's arrive, with its bytes
      tc::mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < RT_ASTAGES; ++i) {
      tc::mbar_init(&afull[i], RT_PROD_WARPS);
      tc::mbar_init(&aempty[i], 1);
    }
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == RT_MMA_WARP) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < RT_PROD_WARPS) {
    // ------------------------------------------------------------ producers
    const int q = warp & 3, hh = warp >> 2;
    const int m = m0 + 32 * q + lane;
    const bool valid = m < T;
    const float4* xrow = reinterpret_cast<const float4*>(X + (size_t)(valid ? m : 0) * H + kb + 32 * hh);
    const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + RT_A_COL0 + (uint32_t)(16 * hh);
    float4 cur[8], nxt[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = valid ? __ldg(xrow + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    bool ok = true;
    for (int kt = 0; kt < KT && ok; ++kt) {
      const int st = kt % RT_ASTAGES;
      if (kt + 1 < KT) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          nxt[i] = valid ? __ldg(xrow + (kt + 1) * (RT_BK / 4) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      uint32_t w1[16], w2[16], w3[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        split3(cur[i].x, cur[i].y, w1[2 * i], w2[2 * i], w3[2 * i]);
        split3(cur[i].z, cur[i].w, w1[2 * i + 1], w2[2 * i + 1], w3[2 * i + 1]);
      }
      // warp-uniform outcome: the TMEM stores below are warp-collective
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&aempty[st], ((kt / RT_ASTAGES) & 1) ^ 1, abort_flag))) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const uint32_t a = ta + (uint32_t)st * RT_A_COLS;
      tc::tmem_st16(a, w1);
      tc::tmem_st16(a + 32, w2);
      tc::tmem_st16(a + 64, w3);
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&afull[st]);
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
    }
    // ------------------------------------------------------------ epilogue
    if (warp < 4) {
      if (__all_sync(0xffffffffu, ok && tc::mbar_wait(acc_full, 0, abort_flag))) {
        tc::tc_fence_after();
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        float* dst = part + ((size_t)sl * T + (valid ? m : 0)) * E + n0;
#pragma unroll 1
        for (int c = 0; c < RT_BN; c += 16) {
          uint32_t v0[16], v1[16];  // x1 w1, and the five smaller products
          tc::tmem_ld16x2(tq + c, tq + RT_DC_COL + c, v0, v1);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<float4*>(dst + c)[i] =
                  make_float4(__uint_as_float(v0[4 * i]) + __uint_as_float(v1[4 * i]),
                              __uint_as_float(v0[4 * i + 1]) + __uint_as_float(v1[4 * i + 1]),
                              __uint_as_float(v0[4 * i + 2]) + __uint_as_float(v1[4 * i + 2]),
                              __uint_as_float(v0[4 * i + 3]) + __uint_as_float(v1[4 * i + 3]));
          }
        }
      }
    }
  } else if (warp == RT_LOAD_WARP) {
    // ------------------------------------------------------------ Wr^T parts
    if (lane == 0) {
      for (int kt = 0; kt < KT; ++kt) {
        const int st = kt % RT_STAGES;
        if (!tc::mbar_wait(&bempty[st], ((kt / RT_STAGES) & 1) ^ 1, abort_flag)) break;
        uint8_t* b = sB + st * RT_STAGE_B;
        tc::mbar_expect_tx(&bfull[st], RT_STAGE_B);
#pragma unroll
        for (int p = 0; p < 3; ++p) tc::tma_load_2d(b + p * RT_PIECE, &wmap, kb + kt * RT_BK, p * E + n0, &bfull[st]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(RT_BM, RT_BN);
      const uint64_t bdesc0 = tc::sw128_desc(tc::smem_u32(sB));
      // (A part, B part) of the six products; product 0 into the first
      // accumulator, the others into the second
      const int pa[6] = {0, 0, 1, 0, 2, 1}, pb[6] = {0, 1, 0, 2, 0, 1};
      bool ok = true;
      for (int kt = 0; kt < KT; ++kt) {
        const int st = kt % RT_STAGES, as = kt % RT_ASTAGES;
        if (!tc::mbar_wait_spin(&bfull[st], (kt / RT_STAGES) & 1, abort_flag) ||
            !tc::mbar_wait_spin(&afull[as], (kt / RT_ASTAGES) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t a = tmem + RT_A_COL0 + (uint32_t)as * RT_A_COLS;
        const uint64_t bd = bdesc0 + (uint64_t)(st * (RT_STAGE_B >> 4));
#pragma unroll
        for (int kk = 0; kk < RT_BK / 16; ++kk)
#pragma unroll
          for (int j = 0; j < 6; ++j)
            tc::mma_bf16_ts(tmem + (j == 0 ? 0u : RT_DC_COL), a + 32 * pa[j] + 8 * kk,
                            bd + (uint64_t)(pb[j] * (RT_PIECE >> 4) + 2 * kk), idesc,
                            j == 0 ? (kt | kk) != 0 : (kt | kk | (j - 1)) != 0);
        tc::mma_commit(&aempty[as]);
        tc::mma_commit(&bempty[st]);
      }
      if (ok) tc::mma_commit(acc_full);
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never);
    }
    __syncwarp();
  }

  if (*abort_flag && threadIdx.x == 0) record_status(status, QMOE_ERR_TIMEOUT);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == RT_MMA_WARP) tc::tmem_dealloc(tmem, 512);
}

// bf16 [rows][K] as boxes of 128 rows x 64 values, 128-byte swizzle; the
// last map is kept (the workspace, and so the map, usually repeats).
static bool encode_wr3(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K) {
  static std::mutex mu;
  static const void* last_base = nullptr;
  static uint64_t last_rows = 0, last_K = 0;
  static CUtensorMap last;
  std::lock_guard<std::mutex> lock(mu);
  if (base == last_base && rows == last_rows && K == last_K) {
    *m = last;
    return true;
  }
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {RT_BK, RT_BN};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  last_base = base;
  last_rows = rows;
  last_K = K;
  last = *m;
  return true;
}

cudaError_t launch_router_tc(const float* X, const float* Wr, float* part, int T, int H, int E, int nsplit,
                             void* wr3, int* status, cudaStream_t st) {
  if (!router_tc_eligible(T, H, E) || wr3 == nullptr || H % (nsplit * RT_BK) != 0) return cudaErrorInvalidValue;
  __nv_bfloat16* w3 = static_cast<__nv_bfloat16*>(wr3);
  router_split_wr_kernel<<<dim3(H / 32, E / 32), 256, 0, st>>>(Wr, w3, H, E);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap m;
  if (!encode_wr3(&m, w3, (uint64_t)3 * E, (uint64_t)H)) return cudaErrorInvalidValue;
  e = ensure_kernel_smem(reinterpret_cast<const void*>(router_tc_kernel), RT_SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid(E / RT_BN, (T + RT_BM - 1) / RT_BM, nsplit);
  router_tc_kernel<<<grid, RT_THREADS, RT_SMEM, st>>>(X, part, T, H, E, H / nsplit, status, m);
  return cudaGetLastError();
}

}  // namespace qmoe
