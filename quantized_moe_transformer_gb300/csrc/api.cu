// C ABI of libqmoe.so: argument checks, workspace carving and launch order.
// The operations are defined in include/qmoe.h.
#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>
#include <cstdio>

#include "kernels.cuh"

using namespace qmoe;

namespace {

__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::atomic<int> g_arch_ok[kMaxDevices];     // 0 unknown, 1 sm_103, -1 other
std::atomic<int*> g_status_ptr[kMaxDevices];
constexpr int kDefaultGemmThreshold = 4;
std::atomic<int> g_gemm_threshold{kDefaultGemmThreshold};
constexpr int kDefaultDecodeRows = 4;
std::atomic<int> g_decode_max_rows{kDefaultDecodeRows};
thread_local int g_last_path = QMOE_PATH_NONE;
thread_local int g_last_cuda_error = 0;
std::atomic<long long> g_launches{0};
// test-only fault injection (qmoe_test_inject) and the bound on device waits
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
std::atomic<int> g_fault_site{0};
std::atomic<int> g_fault_wait_us{0};

unsigned long long wait_limit_ns() {
  const int us = g_fault_wait_us.load();
  return (g_fault_site.load() != 0 && us > 0) ? 1000ull * (unsigned long long)us : kWaitLimitNs;
}

// Opt-in per-stage timing: events recorded around every launch of one stage.
constexpr int kProfCap = 4096;
struct StageProfile {
  int stage = 0;
  int n = 0;
  cudaEvent_t start[kProfCap];
  cudaEvent_t stop[kProfCap];
  int created = 0;
};
thread_local StageProfile g_prof;

// Records ``ev`` on ``st``; while ``st`` is capturing a graph the record becomes
// an event-record node of the graph (cudaEventRecordExternal), so that the
// event's time is that of the node in each replay.
void record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}

// Runs ``launch`` (a kernel launch on ``st``), counting it and, when its stage
// is being profiled, bracketing it with a pair of events.
template <typename F>
cudaError_t staged(int stage, int n_kernels, cudaStream_t st, F&& launch) {
  const bool prof = g_prof.stage == stage && g_prof.n < kProfCap;
  if (prof) {
    if (g_prof.n >= g_prof.created) {
      if (cudaEventCreate(&g_prof.start[g_prof.n]) != cudaSuccess ||
          cudaEventCreate(&g_prof.stop[g_prof.n]) != cudaSuccess)
        return cudaErrorMemoryAllocation;
      g_prof.created = g_prof.n + 1;
    }
    record_event(g_prof.start[g_prof.n], st);
  }
  cudaError_t e = launch();
  g_launches.fetch_add(n_kernels);
  if (e != cudaSuccess) g_last_cuda_error = (int)e;
  if (prof) {
    record_event(g_prof.stop[g_prof.n], st);
    ++g_prof.n;
  }
  return e;
}

// Checks the current device once (sm_103) and finds the status word's address.
int device_ready(int** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMOE_ERR_CUDA;
  int ok = g_arch_ok[dev].load();
  if (ok == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return QMOE_ERR_CUDA;
    ok = (major == 10 && minor == 3) ? 1 : -1;
    g_arch_ok[dev].store(ok);
  }
  if (ok != 1) return QMOE_ERR_ARCH;
  int* p = g_status_ptr[dev].load();
  if (p == nullptr) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_status_word) != cudaSuccess)
      return QMOE_ERR_CUDA;
    g_status_ptr[dev].store(p);
  }
  *status = p;
  return QMOE_OK;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace carve-up (every piece 256-byte aligned).
struct MoeWs {
  size_t part, wr3, ids, w, sync, offsets, perm, inv, active, n_active, chunk, chunks, n_chunks, xb, h, y, total;
  int nsplit;
};

MoeWs moe_ws_layout(int T, int H, int E, int k, int F) {
  MoeWs L{};
  const size_t P = (size_t)T * k, rows = P + T;
  L.nsplit = router_splits(T, H, E);
  size_t o = 0;
  const int parts = L.nsplit > 4 ? L.nsplit : 4;  // the decode router writes 4 partials
  L.part = o;     o += up256(sizeof(float) * (size_t)parts * T * E);
  L.wr3 = o;      o += up256(router_tc_ws_bytes(T, H, E));  // tensor-core router's Wr parts
  L.ids = o;      o += up256(sizeof(int32_t) * P);
  L.w = o;        o += up256(sizeof(float) * P);
  L.sync = o;     o += up256(sizeof(int32_t) * (size_t)decode_sync_ints(H));  // decode path counters
  L.offsets = o;  o += up256(sizeof(int32_t) * (E + 2));
  L.perm = o;     o += up256(sizeof(int32_t) * rows);
  L.inv = o;      o += up256(sizeof(int32_t) * rows);
  L.active = o;   o += up256(sizeof(int32_t) * (E + 1));
  L.n_active = o; o += 256;
  L.chunk = o;    o += up256(sizeof(int32_t) * (size_t)perm_chunks((int)P) * E);
  L.chunks = o;   o += up256(sizeof(int2) * (size_t)tc_max_chunks(T, k, E, 1));
  L.n_chunks = o; o += 256;
  L.h = o;        o += up256(sizeof(float) * rows * F);
  L.y = o;        o += up256(sizeof(float) * rows * H);
  // the tensor-core path's bf16 tokens [rows][H] live in y's space: they are
  // dead once the gate/up kernel has run, before the down kernel writes y
  L.xb = L.y;
  L.total = o;
  return L;
}

bool supported_width(int n) { return n == 256 || n == 512 || n == 1024 || n == 2048 || n == 4096; }

int check_desc(const qmoe_moe_desc* d) {
  if (!d) return QMOE_ERR_NULL;
  if (!supported_width(d->H) || !supported_width(d->F)) return QMOE_ERR_ARG;
  if (d->E < 1 || d->E > 1024 || d->k < 1 || d->k > 16 || d->k > d->E) return QMOE_ERR_ARG;
  if (d->gate_type < QMOE_Q4K || d->gate_type > QMOE_MXFP4 || d->down_type < QMOE_Q4K || d->down_type > QMOE_MXFP4)
    return QMOE_ERR_ARG;
  if (!d->Wr || !d->Wg || !d->Wu || !d->Wd) return QMOE_ERR_NULL;
  const bool any_shared = d->Sg || d->Su || d->Sd;
  const bool all_shared = d->Sg && d->Su && d->Sd;
  if (any_shared && !all_shared) return QMOE_ERR_NULL;
  const void* ptrs[] = {d->Wr, d->Wg, d->Wu, d->Wd, d->Sg, d->Su, d->Sd};
  for (const void* p : ptrs)
    if (p && !aligned(p, 16)) return QMOE_ERR_ALIGN;
  return QMOE_OK;
}

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return QMOE_OK;
  g_last_cuda_error = (int)e;
  return QMOE_ERR_LAUNCH;
}

// ---------------------------------------------------------------- block
struct AttnWs {
  size_t r, q, k, v, o, part, offsets, perm, active, n_active, chunks, n_chunks, xb, offsets2, chunks2, n_chunks2,
      total;
  bool chunked;
};

constexpr int kChunkedAttnRows = 16;

AttnWs attn_ws_layout(const qmoe_block_desc* b, int T, int pos0) {
  AttnWs L{};
  const int H = b->H, nh = b->n_heads, nkv = b->n_kv, hd = b->head_dim;
  const size_t Q = (size_t)nh * hd, KV = (size_t)nkv * hd;
  L.chunked = T <= kChunkedAttnRows;
  size_t o = 0;
  L.r = o;        o += up256(sizeof(float) * T * (size_t)H);
  L.q = o;        o += up256(sizeof(float) * T * Q);
  L.k = o;        o += up256(sizeof(float) * T * KV);
  L.v = o;        o += up256(sizeof(float) * T * KV);
  L.o = o;        o += up256(sizeof(float) * T * Q);
  L.part = o;     o += L.chunked ? up256(sizeof(float) * T * (size_t)nh * attn_nchunks(T, pos0) * (hd + 2)) : 0;
  L.offsets = o;  o += 256;
  L.perm = o;     o += up256(sizeof(int32_t) * T);
  L.active = o;   o += 256;
  L.n_active = o; o += 256;
  L.chunks = o;   o += up256(sizeof(int2) * (size_t)tc_max_chunks(T, 1, 1, 0));
  L.n_chunks = o; o += 256;
  L.xb = o;       o += up256(sizeof(uint16_t) * T * (Q > (size_t)H ? Q : (size_t)H));
  // the K and V projections as one launch (V as the shared expert of a
  // two-expert chunk list; its output rows follow K's, L.v == L.k + T KV)
  L.offsets2 = o; o += 256;
  L.chunks2 = o;  o += up256(sizeof(int2) * (size_t)tc_max_chunks(T, 1, 1, 1));
  L.n_chunks2 = o; o += 256;
  L.total = o;
  return L;
}

int check_block(const qmoe_block_desc* b) {
  if (!b) return QMOE_ERR_NULL;
  const int H = b->H, nh = b->n_heads, nkv = b->n_kv, hd = b->head_dim;
  if (!supported_width(H) || nh < 1 || nkv < 1 || nh % nkv != 0) return QMOE_ERR_ARG;
  if (hd < 8 || hd > 256 || hd % 8 != 0) return QMOE_ERR_ARG;
  if (!supported_width(nh * hd) || (nkv * hd) % 16 != 0) return QMOE_ERR_ARG;
  if (!(b->eps >= 0.f) || !(b->rope_theta > 0.f)) return QMOE_ERR_ARG;
  if (!b->g1 || !b->g2 || !b->Wq || !b->Wk || !b->Wv || !b->Wo) return QMOE_ERR_NULL;
  const void* ptrs[] = {b->g1, b->g2, b->Wq, b->Wk, b->Wv, b->Wo};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return QMOE_ERR_ALIGN;
  return QMOE_OK;
}

// y [T][N] fp32 = x [T][K] fp32 . W^T for packed Q4_K/Q5_K matrices W [N][K/256]:
// the grouped kernels with one "expert" holding all rows. dense_prep sets up
// the routing of that expert (and, on the tensor-core path, the chunk list and
// the bf16 copy of x) once for every projection of the same x.
bool dense_uses_tc(int T) { return T > g_gemm_threshold.load(); }

// dense_prep of RMSNorm(x; gamma) on the tensor-core path: the norm is written
// straight into the bf16 token operand (no fp32 normed copy).
// (``kv_pair``: also the two-expert chunk list of the fused K and V launch)
cudaError_t dense_prep_norm(const float* x, const float* gamma, float eps, int T, int K, char* base,
                            const AttnWs& L, bool kv_pair, cudaStream_t st) {
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
  int32_t* active = reinterpret_cast<int32_t*>(base + L.active);
  int32_t* n_active = reinterpret_cast<int32_t*>(base + L.n_active);
  int32_t* offsets2 = reinterpret_cast<int32_t*>(base + L.offsets2);
  cudaError_t e = launch_dense_route(offsets, perm, active, n_active, T, st, kv_pair ? offsets2 : nullptr);
  if (e != cudaSuccess) return e;
  int2* chunks = reinterpret_cast<int2*>(base + L.chunks);
  int32_t* n_chunks = reinterpret_cast<int32_t*>(base + L.n_chunks);
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(base + L.xb);
  if ((e = launch_build_chunks(offsets, 1, 128, chunks, n_chunks, st)) != cudaSuccess) return e;
  if (kv_pair) {
    e = launch_build_chunks(offsets2, 1, 128, reinterpret_cast<int2*>(base + L.chunks2),
                            reinterpret_cast<int32_t*>(base + L.n_chunks2), st);
    if (e != cudaSuccess) return e;
    g_launches.fetch_add(1);
  }
  g_launches.fetch_add(3);
  return launch_rmsnorm_bf16(x, gamma, eps, xb, T, K, st);
}

// The K and V projections of the bf16 normed rows as one tensor-core launch:
// K is expert 0 and V the shared expert of the two-expert chunk list, so V's
// output rows land right after K's (kv = [K rows; V rows]) and its token rows
// are read T rows back.
cudaError_t dense_proj_kv(int T, int K, const void* Wk, const void* Wv, int N, float* kv, char* base,
                          const AttnWs& L, int* status, cudaStream_t st) {
  GroupedTcArgs p{};
  p.W = static_cast<const uint8_t*>(Wk);
  p.S = static_cast<const uint8_t*>(Wv);
  p.qt = QMOE_Q4K;
  p.offsets = reinterpret_cast<int32_t*>(base + L.offsets2);
  p.perm = reinterpret_cast<int32_t*>(base + L.perm);
  p.chunks = reinterpret_cast<int2*>(base + L.chunks2);
  p.n_chunks = reinterpret_cast<int32_t*>(base + L.n_chunks2);
  p.max_chunks = tc_max_chunks(T, 1, 1, 1);
  p.hin = reinterpret_cast<__nv_bfloat16*>(base + L.xb);
  p.tok_rows = T;
  p.tok_shift = T;
  p.nmax = 128;
  p.yout_f32 = kv;
  p.T = T;
  p.k = 1;
  p.E = 1;
  p.H = N;
  p.F = K;
  p.status = status;
  g_launches.fetch_add(1);
  return launch_down_tc(p, st);
}

cudaError_t dense_prep(const float* x, int T, int K, char* base, const AttnWs& L, cudaStream_t st) {
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
  int32_t* active = reinterpret_cast<int32_t*>(base + L.active);
  int32_t* n_active = reinterpret_cast<int32_t*>(base + L.n_active);
  cudaError_t e = launch_dense_route(offsets, perm, active, n_active, T, st);
  g_launches.fetch_add(1);
  if (e != cudaSuccess || !dense_uses_tc(T)) return e;
  int2* chunks = reinterpret_cast<int2*>(base + L.chunks);
  int32_t* n_chunks = reinterpret_cast<int32_t*>(base + L.n_chunks);
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(base + L.xb);
  if ((e = launch_build_chunks(offsets, 1, 128, chunks, n_chunks, st)) != cudaSuccess) return e;
  g_launches.fetch_add(2);
  return launch_to_bf16(x, xb, T, K, nullptr, T, 1, nullptr, st);
}

// The projection runs on the tensor cores when T is above the threshold and N
// is a multiple of 256 (the grouped kernel's 256-row weight blocks), else on
// the fp32 GEMV, which reads x itself.
bool dense_tc(int T, int N) { return dense_uses_tc(T) && N % 256 == 0; }

cudaError_t dense_proj(const float* x, int T, int K, const void* W, int qt, int N, float* y, char* base,
                       const AttnWs& L, int* status, cudaStream_t st) {
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
  if (dense_tc(T, N)) {
    GroupedTcArgs p{};
    p.W = static_cast<const uint8_t*>(W);
    p.qt = qt;
    p.offsets = offsets;
    p.perm = perm;
    p.chunks = reinterpret_cast<int2*>(base + L.chunks);
    p.n_chunks = reinterpret_cast<int32_t*>(base + L.n_chunks);
    p.max_chunks = tc_max_chunks(T, 1, 1, 0);
    p.hin = reinterpret_cast<__nv_bfloat16*>(base + L.xb);
    p.tok_rows = T;
    p.nmax = 128;
    p.yout_f32 = y;
    p.T = T;
    p.k = 1;
    p.E = 1;
    p.H = N;
    p.F = K;
    p.status = status;
    g_launches.fetch_add(1);
    return launch_down_tc(p, st);
  }
  GroupedArgs g{};
  g.W = static_cast<const uint8_t*>(W);
  g.S = nullptr;
  g.offsets = offsets;
  g.perm = perm;
  g.active = reinterpret_cast<int32_t*>(base + L.active);
  g.n_active = reinterpret_cast<int32_t*>(base + L.n_active);
  g.T = T;
  g.k = 1;
  g.E = 1;
  g.max_active = 1;
  g_launches.fetch_add(1);
  return launch_down_gemv(g, qt, x, K, N, y, st);
}

int attn_impl(const qmoe_block_desc* b, const float* X, const float* R, float* out, int T, uint16_t* kc, uint16_t* vc,
              int pos0, int ctx_cap, void* ws, size_t ws_bytes, cudaStream_t st) {
  int r = check_block(b);
  if (r != QMOE_OK) return r;
  if (T < 0 || pos0 < 0) return QMOE_ERR_ARG;
  if (T == 0) return QMOE_OK;
  if ((long long)pos0 + T > ctx_cap) return QMOE_ERR_ARG;
  if (!X || !out || !kc || !vc || !ws) return QMOE_ERR_NULL;
  if (!aligned(X, 16) || !aligned(out, 16) || (R && !aligned(R, 16)) || !aligned(kc, 16) || !aligned(vc, 16) ||
      !aligned(ws, 256))
    return QMOE_ERR_ALIGN;
  if (T > kChunkedAttnRows && b->head_dim != 128) return QMOE_ERR_ARG;
  const AttnWs L = attn_ws_layout(b, T, pos0);
  if (ws_bytes < L.total) return QMOE_ERR_WORKSPACE;
  int* status = nullptr;
  r = device_ready(&status);
  if (r != QMOE_OK) return r;
  char* base = static_cast<char*>(ws);
  float* rr = reinterpret_cast<float*>(base + L.r);
  float* q = reinterpret_cast<float*>(base + L.q);
  float* k = reinterpret_cast<float*>(base + L.k);
  float* v = reinterpret_cast<float*>(base + L.v);
  float* o = reinterpret_cast<float*>(base + L.o);
  float* part = reinterpret_cast<float*>(base + L.part);
  const int H = b->H, nh = b->n_heads, nkv = b->n_kv, hd = b->head_dim;
  __nv_bfloat16* kcb = reinterpret_cast<__nv_bfloat16*>(kc);
  __nv_bfloat16* vcb = reinterpret_cast<__nv_bfloat16*>(vc);
  cudaError_t e;
  // RMSNorm fused into the bf16 token operand when every one of the Q, K, V
  // projections runs on the tensor cores (a GEMV projection reads the fp32
  // normed rows); then the K and V projections run as one launch (V's rows
  // follow K's in the workspace)
  const bool qkv_tc = dense_tc(T, nh * hd) && dense_tc(T, nkv * hd);
  const bool kv_pair = qkv_tc && L.v == L.k + sizeof(float) * (size_t)T * nkv * hd;
  if (qkv_tc) {
    e = dense_prep_norm(X, b->g1, b->eps, T, H, base, L, kv_pair, st);
  } else {
    e = launch_rmsnorm(X, b->g1, b->eps, rr, T, H, st);
    g_launches.fetch_add(1);
    if (e == cudaSuccess) e = dense_prep(rr, T, H, base, L, st);
  }
  if (e == cudaSuccess) e = dense_proj(rr, T, H, b->Wq, QMOE_Q4K, nh * hd, q, base, L, status, st);
  if (kv_pair) {
    if (e == cudaSuccess) e = dense_proj_kv(T, H, b->Wk, b->Wv, nkv * hd, k, base, L, status, st);
  } else {
    if (e == cudaSuccess) e = dense_proj(rr, T, H, b->Wk, QMOE_Q4K, nkv * hd, k, base, L, status, st);
    if (e == cudaSuccess) e = dense_proj(rr, T, H, b->Wv, QMOE_Q4K, nkv * hd, v, base, L, status, st);
  }
  if (e == cudaSuccess) {
    e = launch_rope_cache(q, k, v, kcb, vcb, T, pos0, nh, nkv, hd, (double)b->rope_theta, st);
    g_launches.fetch_add(1);
  }
  // O projection on the tensor cores: the prefill attention writes its bf16
  // token operand itself
  // (with the route and chunk list of these rows from the Q, K, V projections)
  const bool o_tc = dense_tc(T, H) && qkv_tc;
  __nv_bfloat16* ob = (o_tc && !L.chunked) ? reinterpret_cast<__nv_bfloat16*>(base + L.xb) : nullptr;
  if (e == cudaSuccess) {
    e = launch_attention(q, kcb, vcb, part, o, ob, T, pos0, nh, nkv, hd, L.chunked, status, wait_limit_ns(),
                         g_fault_site.load() == QMOE_FAULT_ATTN_FINAL ? 1 : 0, st);
    g_launches.fetch_add(L.chunked ? 2 : 1);
  }
  if (o_tc) {
    // the dense route and chunk list are the Q, K, V projections' (the same rows)
    if (e == cudaSuccess && ob == nullptr) {
      e = launch_to_bf16(o, reinterpret_cast<__nv_bfloat16*>(base + L.xb), T, nh * hd, nullptr, T, 1, nullptr, st);
      g_launches.fetch_add(1);
    }
  } else if (e == cudaSuccess) {
    e = dense_prep(o, T, nh * hd, base, L, st);
  }
  // (the residual as its own pass: added in the projection's epilogue, the
  // loads of R held up each 16-token group, 75 against 42 + 20 us at T=4096)
  float* proj_out = R ? rr : out;  // rr is free once Q, K, V exist
  if (e == cudaSuccess) e = dense_proj(o, T, nh * hd, b->Wo, QMOE_Q4K, H, proj_out, base, L, status, st);
  if (e == cudaSuccess && R) {
    e = launch_add(R, proj_out, out, (size_t)T * H, st);
    g_launches.fetch_add(1);
  }
  return launch_status(e);
}

}  // namespace

extern "C" {

int qmoe_rmsnorm(const float* X, const float* gamma, float eps, float* y, int T, int H, qmoe_stream_t stream) {
  if (T < 0 || H < 1 || !(eps >= 0.f)) return QMOE_ERR_ARG;
  if (T == 0) return QMOE_OK;
  if (!X || !gamma || !y) return QMOE_ERR_NULL;
  int* status = nullptr;
  int r = device_ready(&status);
  if (r != QMOE_OK) return r;
  g_launches.fetch_add(1);
  return launch_status(launch_rmsnorm(X, gamma, eps, y, T, H, reinterpret_cast<cudaStream_t>(stream)));
}

size_t qmoe_attn_workspace_bytes(const qmoe_block_desc* b, int T, int pos0) {
  if (check_block(b) != QMOE_OK || T <= 0 || pos0 < 0) return 0;
  return attn_ws_layout(b, T, pos0).total;
}

int qmoe_attn_forward(const qmoe_block_desc* b, const float* X, const float* R, float* out, int T,
                      uint16_t* k_cache, uint16_t* v_cache, int pos0, int ctx_cap, void* ws, size_t ws_bytes,
                      qmoe_stream_t stream) {
  return attn_impl(b, X, R, out, T, k_cache, v_cache, pos0, ctx_cap, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream));
}

size_t qmoe_block_workspace_bytes(const qmoe_block_desc* b, int T, int pos0) {
  if (check_block(b) != QMOE_OK || T <= 0 || pos0 < 0) return 0;
  const size_t moe = qmoe_moe_workspace_bytes(&b->moe, T);
  if (moe == 0) return 0;
  return attn_ws_layout(b, T, pos0).total + 2 * up256(sizeof(float) * (size_t)T * b->H) + moe;
}

int qmoe_block_forward(const qmoe_block_desc* b, const float* X, float* out, int T, uint16_t* k_cache,
                       uint16_t* v_cache, int pos0, int ctx_cap, void* ws, size_t ws_bytes, qmoe_stream_t stream) {
  int r = check_block(b);
  if (r != QMOE_OK) return r;
  r = check_desc(&b->moe);
  if (r != QMOE_OK) return r;
  if (b->moe.H != b->H) return QMOE_ERR_ARG;
  if (T < 0 || pos0 < 0) return QMOE_ERR_ARG;
  if (T == 0) return QMOE_OK;
  if (X == out) return QMOE_ERR_ARG;
  if (!ws) return QMOE_ERR_NULL;
  if (!aligned(ws, 256)) return QMOE_ERR_ALIGN;
  const size_t need = qmoe_block_workspace_bytes(b, T, pos0);
  if (ws_bytes < need) return QMOE_ERR_WORKSPACE;
  const size_t a_bytes = attn_ws_layout(b, T, pos0).total;
  const size_t row_bytes = up256(sizeof(float) * (size_t)T * b->H);
  char* base = static_cast<char*>(ws);
  float* h1 = reinterpret_cast<float*>(base + a_bytes);
  float* r2 = reinterpret_cast<float*>(base + a_bytes + row_bytes);
  char* moe_ws = base + a_bytes + 2 * row_bytes;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  r = attn_impl(b, X, X, h1, T, k_cache, v_cache, pos0, ctx_cap, base, a_bytes, st);
  if (r != QMOE_OK) return r;
  g_launches.fetch_add(1);
  if (launch_rmsnorm(h1, b->g2, b->eps, r2, T, b->H, st) != cudaSuccess) return QMOE_ERR_LAUNCH;
  return qmoe_moe_forward(&b->moe, r2, h1, nullptr, nullptr, out, T, moe_ws, ws_bytes - a_bytes - 2 * row_bytes,
                          stream);
}


const char* qmoe_status_str(int s) {
  switch (s) {
    case QMOE_OK: return "ok";
    case QMOE_ERR_ARG: return "argument out of range";
    case QMOE_ERR_NULL: return "required pointer is NULL";
    case QMOE_ERR_ALIGN: return "pointer not aligned (16 B; workspace 256 B)";
    case QMOE_ERR_WORKSPACE: return "workspace too small";
    case QMOE_ERR_ARCH: return "current device is not sm_103 (GB300)";
    case QMOE_ERR_LAUNCH: return "kernel launch failed";
    case QMOE_ERR_TIMEOUT: return "device wait timed out";
    case QMOE_ERR_DEVICE_ARG: return "device: route id out of range";
    case QMOE_ERR_CUDA: return "CUDA runtime error";
    case QMOE_ERR_TOO_LARGE: return "problem exceeds the library's fixed scratch (use a workspace)";
    default: return "unknown status";
  }
}

int qmoe_query_status(qmoe_stream_t stream) {
  int* p = nullptr;
  int r = device_ready(&p);
  if (r != QMOE_OK) return r;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return QMOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QMOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return QMOE_ERR_CUDA;
  return v;
}

int qmoe_get_gemm_threshold(void) { return g_gemm_threshold.load(); }
void qmoe_set_gemm_threshold(int rows) { g_gemm_threshold.store(rows < 0 ? kDefaultGemmThreshold : rows); }
int qmoe_last_path(void) { return g_last_path; }
int qmoe_last_cuda_error(void) { return g_last_cuda_error; }
int qmoe_get_decode_max_rows(void) { return g_decode_max_rows.load(); }
void qmoe_set_decode_max_rows(int rows) {
  g_decode_max_rows.store(rows < 0 ? kDefaultDecodeRows : (rows > kDefaultDecodeRows ? kDefaultDecodeRows : rows));
}

size_t qmoe_moe_route_workspace_bytes(int T, int H, int E, int k) {
  (void)k;
  if (T <= 0 || H <= 0 || E <= 0) return 0;
  return up256(sizeof(float) * (size_t)router_splits(T, H, E) * T * E) + up256(router_tc_ws_bytes(T, H, E));
}

int qmoe_moe_route(const float* X, const float* Wr, int T, int H, int E, int k, int32_t* ids,
                   float* w, void* ws, size_t ws_bytes, qmoe_stream_t stream) {
  if (T < 0 || !supported_width(H) || E < 1 || E > 1024 || k < 1 || k > 16 || k > E)
    return QMOE_ERR_ARG;
  if (T == 0) return QMOE_OK;
  if (!X || !Wr || !ids || !w || !ws) return QMOE_ERR_NULL;
  if (!aligned(X, 16) || !aligned(Wr, 16) || !aligned(ws, 256)) return QMOE_ERR_ALIGN;
  if (ws_bytes < qmoe_moe_route_workspace_bytes(T, H, E, k)) return QMOE_ERR_WORKSPACE;
  int* status = nullptr;
  int r = device_ready(&status);
  if (r != QMOE_OK) return r;
  const int ns = router_splits(T, H, E);
  float* part = static_cast<float*>(ws);
  void* wr3 = static_cast<char*>(ws) + up256(sizeof(float) * (size_t)ns * T * E);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = staged(QMOE_STAGE_ROUTER, router_launches(T, H, E), st,
                         [&] { return launch_router_logits(X, Wr, part, T, H, E, ns, wr3, status, st); });
  if (e == cudaSuccess)
    e = staged(QMOE_STAGE_ROUTE, 1, st, [&] { return launch_topk(part, ns, T, E, k, ids, w, st); });
  return launch_status(e);
}

size_t qmoe_moe_workspace_bytes(const qmoe_moe_desc* d, int T) {
  if (check_desc(d) != QMOE_OK || T < 0) return 0;
  if (T == 0) return 0;
  return moe_ws_layout(T, d->H, d->E, d->k, d->F).total;
}

int qmoe_moe_workspace_layout(const qmoe_moe_desc* d, int T, qmoe_moe_ws_layout* out) {
  int r = check_desc(d);
  if (r != QMOE_OK) return r;
  if (!out) return QMOE_ERR_NULL;
  if (T < 0) return QMOE_ERR_ARG;
  MoeWs L = moe_ws_layout(T, d->H, d->E, d->k, d->F);
  out->ids = L.ids;
  out->w = L.w;
  out->offsets = L.offsets;
  out->perm = L.perm;
  out->y = L.y;
  return QMOE_OK;
}

int qmoe_moe_forward(const qmoe_moe_desc* d, const float* X, const float* R, const int32_t* ids,
                     const float* w, float* out, int T, void* ws, size_t ws_bytes,
                     qmoe_stream_t stream) {
  int r = check_desc(d);
  if (r != QMOE_OK) return r;
  if (T < 0 || (long long)T * (d->k + 1) >= (1LL << 24)) return QMOE_ERR_ARG;
  if ((ids == nullptr) != (w == nullptr)) return QMOE_ERR_NULL;
  if (T == 0) {
    g_last_path = QMOE_PATH_NONE;
    return QMOE_OK;
  }
  if (!X || !out || !ws) return QMOE_ERR_NULL;
  if (!aligned(X, 16) || !aligned(out, 16) || (R && !aligned(R, 16)) || !aligned(ws, 256) ||
      (ids && !aligned(ids, 4)) || (w && !aligned(w, 4)))
    return QMOE_ERR_ALIGN;
  if (X == out) return QMOE_ERR_ARG;
  const int H = d->H, E = d->E, k = d->k, F = d->F;
  const MoeWs L = moe_ws_layout(T, H, E, k, F);
  if (ws_bytes < L.total) return QMOE_ERR_WORKSPACE;
  int* status = nullptr;
  r = device_ready(&status);
  if (r != QMOE_OK) return r;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  float* part = reinterpret_cast<float*>(base + L.part);
  int32_t* ws_ids = reinterpret_cast<int32_t*>(base + L.ids);
  float* ws_w = reinterpret_cast<float*>(base + L.w);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(base + L.inv);
  int32_t* active = reinterpret_cast<int32_t*>(base + L.active);
  int32_t* n_active = reinterpret_cast<int32_t*>(base + L.n_active);
  int32_t* chunk = reinterpret_cast<int32_t*>(base + L.chunk);
  float* hbuf = reinterpret_cast<float*>(base + L.h);
  float* y = reinterpret_cast<float*>(base + L.y);
  const int has_shared = d->Sg != nullptr;
  const int P = T * k;

  cudaError_t e = cudaSuccess;
  // the decode and tensor-core paths take the k-quant formats; Q6_K and MXFP4
  // layers take the grouped GEMV path at every row count
  const bool kquant = d->gate_type <= QMOE_Q5K && d->down_type <= QMOE_Q5K;
  if (kquant && ids == nullptr && T <= g_decode_max_rows.load() &&
      decode_path_supported(T, H, E, k, F, d->gate_type, d->down_type)) {
    DecodeLaunch D{};
    D.X = X;
    D.R = R;
    D.out = out;
    D.Wr = d->Wr;
    D.Wg = static_cast<const uint8_t*>(d->Wg);
    D.Wu = static_cast<const uint8_t*>(d->Wu);
    D.Wd = static_cast<const uint8_t*>(d->Wd);
    D.Sg = static_cast<const uint8_t*>(d->Sg);
    D.Su = static_cast<const uint8_t*>(d->Su);
    D.Sd = static_cast<const uint8_t*>(d->Sd);
    D.T = T;
    D.H = H;
    D.E = E;
    D.k = k;
    D.F = F;
    D.gate_qt = d->gate_type;
    D.down_qt = d->down_type;
    D.part = part;
    D.hbuf = hbuf;
    D.ybuf = y;
    D.ids = ws_ids;
    D.w = ws_w;
    D.sync = reinterpret_cast<int*>(base + L.sync);
    D.status = status;
    D.wait_ns = wait_limit_ns();
    D.fault = g_fault_site.load() == QMOE_FAULT_DECODE_COPY ? 1 : 0;
    // router, experts
    e = staged(QMOE_STAGE_DECODE, 2, st, [&] { return launch_decode(D, st); });
    if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
    g_last_path = QMOE_PATH_DECODE;
    return QMOE_OK;
  }
  const bool small = P <= 2048;
  // the tensor-core kernels take Q4_K/Q5_K weights, and Q6_K or MXFP4 down
  // weights (whole rows by bulk copies) with F up to 512
  const bool tc_formats = d->gate_type <= QMOE_Q5K &&
                          (d->down_type <= QMOE_Q5K ||
                           ((d->down_type == QMOE_Q6K || d->down_type == QMOE_MXFP4) && F <= 512));
  const bool use_tc = tc_formats && T > g_gemm_threshold.load();
  // on the tensor-core path at large T the permutation scan also builds the
  // token-chunk list
  // (the permutation kernels also build the tensor-core path's token-chunk list)
  const bool chunks_in_scan = use_tc;
  int2* tc_chunks = reinterpret_cast<int2*>(base + L.chunks);
  int32_t* tc_n_chunks = reinterpret_cast<int32_t*>(base + L.n_chunks);
  const int tc_cap = tc_chunk_cap(T, k, E);
  if (ids == nullptr) {
    e = staged(QMOE_STAGE_ROUTER, router_launches(T, H, E), st, [&] {
      return launch_router_logits(X, d->Wr, part, T, H, E, L.nsplit, base + L.wr3, status, st);
    });
    if (e == cudaSuccess) {
      if (small) {
        // top-k over many CTAs, then the permutation in one
        e = staged(QMOE_STAGE_ROUTE, 2, st, [&] {
          cudaError_t e2 = launch_topk(part, L.nsplit, T, E, k, ws_ids, ws_w, st);
          if (e2 != cudaSuccess) return e2;
          return launch_route_small(nullptr, 0, ws_ids, T, E, k, has_shared, ws_ids, ws_w, offsets, perm,
                                    active, n_active, status, st, tc_cap, chunks_in_scan ? tc_chunks : nullptr,
                                    tc_n_chunks);
        });
      } else {
        e = staged(QMOE_STAGE_ROUTE, 4, st, [&] {
          cudaError_t e2 = launch_topk(part, L.nsplit, T, E, k, ws_ids, ws_w, st);
          if (e2 != cudaSuccess) return e2;
          return launch_perm_large(ws_ids, T, E, k, has_shared, chunk, offsets, perm, active,
                                   n_active, status, st, tc_cap, chunks_in_scan ? tc_chunks : nullptr,
                                   tc_n_chunks);
        });
      }
    }
  } else {
    if (small)
      e = staged(QMOE_STAGE_ROUTE, 1, st, [&] {
        return launch_route_small(nullptr, 0, ids, T, E, k, has_shared, ws_ids, ws_w, offsets,
                                  perm, active, n_active, status, st, tc_cap,
                                  chunks_in_scan ? tc_chunks : nullptr, tc_n_chunks);
      });
    else
      e = staged(QMOE_STAGE_ROUTE, 3, st, [&] {
        return launch_perm_large(ids, T, E, k, has_shared, chunk, offsets, perm, active,
                                 n_active, status, st, tc_cap, chunks_in_scan ? tc_chunks : nullptr,
                                 tc_n_chunks);
      });
  }
  if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
  const float* w_use = ids ? w : ws_w;

  if (use_tc) {
    // grouped dequant + bf16 tcgen05 GEMM path: h and y are bf16
    int2* chunks = tc_chunks;
    int32_t* n_chunks = tc_n_chunks;
    __nv_bfloat16* h16 = reinterpret_cast<__nv_bfloat16*>(hbuf);
    __nv_bfloat16* y16 = reinterpret_cast<__nv_bfloat16*>(y);
    __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(base + L.xb);
    e = staged(QMOE_STAGE_ROUTE, chunks_in_scan ? 1 : 2, st, [&] {
      if (!chunks_in_scan) {
        cudaError_t e2 = launch_build_chunks(offsets, E, tc_cap, chunks, n_chunks, st);
        if (e2 != cudaSuccess) return e2;
      }
      return launch_to_bf16(X, xb, (int)(P + (has_shared ? T : 0)), H, perm, T, k, inv, st);
    });
    if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
    GroupedTcArgs p{};
    p.offsets = offsets;
    p.perm = perm;
    p.chunks = chunks;
    p.n_chunks = n_chunks;
    p.max_chunks = tc_max_chunks(T, k, E, has_shared);
    p.nmax = tc_cap;
    p.T = T;
    p.k = k;
    p.E = E;
    p.H = H;
    p.F = F;
    p.status = status;
    p.W = static_cast<const uint8_t*>(d->Wg);
    p.W2 = static_cast<const uint8_t*>(d->Wu);
    p.S = static_cast<const uint8_t*>(d->Sg);
    p.S2 = static_cast<const uint8_t*>(d->Su);
    p.qt = d->gate_type;
    p.xb = xb;
    p.tok_rows = (int)(P + (has_shared ? T : 0));
    p.hout = h16;
    p.wait_ns = wait_limit_ns();
    p.fault = g_fault_site.load() == QMOE_FAULT_TC_ARRIVE ? 1 : 0;
    e = staged(QMOE_STAGE_GATEUP, 1, st, [&] { return launch_gateup_tc(p, st); });
    p.fault = 0;
    if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
    p.W = static_cast<const uint8_t*>(d->Wd);
    p.W2 = nullptr;
    p.S = static_cast<const uint8_t*>(d->Sd);
    p.S2 = nullptr;
    p.qt = d->down_type;
    p.hin = h16;
    p.tok_rows = (int)(P + (has_shared ? T : 0));
    p.yout = y16;
    e = staged(QMOE_STAGE_DOWN, 1, st, [&] { return launch_down_tc(p, st); });
    if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
    e = staged(QMOE_STAGE_COMBINE, 1, st,
               [&] { return launch_combine_bf16(y16, inv, w_use, R, out, T, H, k, has_shared, st); });
    if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
    g_last_path = QMOE_PATH_GEMM_TC;
    return QMOE_OK;
  }

  GroupedArgs g;
  g.offsets = offsets;
  g.perm = perm;
  g.active = active;
  g.n_active = n_active;
  g.T = T;
  g.k = k;
  g.E = E;
  g.max_active = (P < E ? P : E) + has_shared;

  g.W = static_cast<const uint8_t*>(d->Wg);
  g.S = static_cast<const uint8_t*>(d->Sg);
  e = staged(QMOE_STAGE_GATEUP, 1, st, [&] {
    return launch_gateup_gemv(g, static_cast<const uint8_t*>(d->Wu),
                              static_cast<const uint8_t*>(d->Su), d->gate_type, X, H, F, hbuf, st);
  });
  if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
  g.W = static_cast<const uint8_t*>(d->Wd);
  g.S = static_cast<const uint8_t*>(d->Sd);
  e = staged(QMOE_STAGE_DOWN, 1, st,
             [&] { return launch_down_gemv(g, d->down_type, hbuf, F, H, y, st); });
  if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
  e = staged(QMOE_STAGE_COMBINE, 1, st,
             [&] { return launch_combine(y, w_use, R, out, T, H, k, has_shared, st); });
  if (e != cudaSuccess) return QMOE_ERR_LAUNCH;
  g_last_path = QMOE_PATH_GEMV;
  return QMOE_OK;
}

size_t qmoe_moe_forward_host_workspace_bytes(const qmoe_moe_desc* d, int T) {
  const size_t base = qmoe_moe_workspace_bytes(d, T);
  if (base == 0) return 0;
  return base + 3 * up256(sizeof(float) * (size_t)T * d->H);
}

}  // extern "C"

namespace {

// The device-accessible address of pinned, mapped host memory ``p`` (nullptr
// when it has none: pageable memory).
const void* host_mapped(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Outputs up to this size are written by the layer's last kernel straight into
// mapped host memory (and a residual of the same size is read from there): no
// copy node; larger ones go through the workspace and one copy (at 32 MiB the
// copy is faster: 4096 rows of 2048 took 5.19 M tokens/s end to end with the
// copy, 5.02 M written in place; at 512 rows 1.63 M against 1.66 M).
constexpr size_t kDirectHostBytes = (size_t)4 << 20;

// Copies in, the layer, copies out: the work of one host-buffer call, enqueued
// on ``st`` (no wait).
int host_forward_enqueue(const qmoe_moe_desc* d, const float* X_host, const float* R_host, float* out_host, int T,
                         void* ws, cudaStream_t st) {
  const size_t base = qmoe_moe_workspace_bytes(d, T);
  const size_t rows = up256(sizeof(float) * (size_t)T * d->H);
  char* p = static_cast<char*>(ws);
  float* Xd = reinterpret_cast<float*>(p + base);
  float* Rd = R_host ? reinterpret_cast<float*>(p + base + rows) : nullptr;
  float* Od = reinterpret_cast<float*>(p + base + 2 * rows);
  const size_t nbytes = sizeof(float) * (size_t)T * d->H;
  float* out_dev = nullptr;
  const float* res_dev = nullptr;
  if (nbytes <= kDirectHostBytes) {
    out_dev = static_cast<float*>(const_cast<void*>(host_mapped(out_host)));
    if (R_host) res_dev = static_cast<const float*>(host_mapped(R_host));
  }
  if (cudaMemcpyAsync(Xd, X_host, nbytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return QMOE_ERR_CUDA;
  if (R_host && !res_dev && cudaMemcpyAsync(Rd, R_host, nbytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return QMOE_ERR_CUDA;
  int r = qmoe_moe_forward(d, Xd, res_dev ? res_dev : Rd, nullptr, nullptr, out_dev ? out_dev : Od, T, ws, base,
                           reinterpret_cast<qmoe_stream_t>(st));
  if (r != QMOE_OK) return r;
  if (!out_dev && cudaMemcpyAsync(out_host, Od, nbytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return QMOE_ERR_CUDA;
  return QMOE_OK;
}

// Host-buffer calls that repeat their arguments replay a CUDA graph of the
// copies and the layer's kernels (one launch instead of one per copy and
// kernel). A key is the descriptor, the buffers, T, the stream, the device and
// the path threshold; its first call runs directly (every lazy setup happens
// then), its second captures and replays, later ones replay. Calls made while
// a test fault site or stage profiling is set, on a stream that is already
// capturing, or with pageable host buffers always run directly.
struct HostGraph {
  qmoe_moe_desc d;
  const float *x, *r;
  float* out;
  int T, device, threshold, decode_rows;
  void* ws;
  cudaStream_t st;
  int calls;       // calls seen with this key
  bool direct;     // never replayed (capture failed or pageable buffers)
  cudaGraphExec_t exec;
  long long launches;
  int path;
};
constexpr int kHostGraphs = 64;
std::mutex g_hg_mu;
HostGraph g_hg[kHostGraphs];
int g_hg_n = 0, g_hg_next = 0;

bool host_pinned(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

bool same_key(const HostGraph& g, const qmoe_moe_desc* d, const float* x, const float* r, float* out, int T,
              void* ws, cudaStream_t st, int device, int threshold, int decode_rows) {
  return g.x == x && g.r == r && g.out == out && g.T == T && g.ws == ws && g.st == st && g.device == device &&
         g.threshold == threshold && g.decode_rows == decode_rows && memcmp(&g.d, d, sizeof(*d)) == 0;
}

}  // namespace

extern "C" {

int qmoe_moe_forward_host(const qmoe_moe_desc* d, const float* X_host, const float* R_host,
                          float* out_host, int T, void* ws, size_t ws_bytes,
                          qmoe_stream_t stream) {
  int r = check_desc(d);
  if (r != QMOE_OK) return r;
  if (T < 0) return QMOE_ERR_ARG;
  if (T == 0) return QMOE_OK;
  if (!X_host || !out_host || !ws) return QMOE_ERR_NULL;
  if (!aligned(ws, 256)) return QMOE_ERR_ALIGN;
  const size_t base = qmoe_moe_workspace_bytes(d, T);
  const size_t rows = up256(sizeof(float) * (size_t)T * d->H);
  if (ws_bytes < base + 3 * rows) return QMOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  int device = 0;
  const bool graphs_ok = g_fault_site.load() == 0 && g_prof.stage == 0 &&
                         cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone &&
                         cudaGetDevice(&device) == cudaSuccess;
  if (graphs_ok) {
    std::lock_guard<std::mutex> lock(g_hg_mu);
    const int threshold = g_gemm_threshold.load(), decode_rows = g_decode_max_rows.load();
    HostGraph* g = nullptr;
    for (int i = 0; i < g_hg_n && !g; ++i)
      if (same_key(g_hg[i], d, X_host, R_host, out_host, T, ws, st, device, threshold, decode_rows)) g = &g_hg[i];
    if (g == nullptr) {
      // a new key (replacing the oldest when the table is full): this call runs directly
      g = &g_hg[g_hg_next];
      if (g_hg_n < kHostGraphs) ++g_hg_n;
      g_hg_next = (g_hg_next + 1) % kHostGraphs;
      if (g->exec) cudaGraphExecDestroy(g->exec);
      *g = HostGraph{};
      g->d = *d;
      g->x = X_host;
      g->r = R_host;
      g->out = out_host;
      g->T = T;
      g->device = device;
      g->threshold = threshold;
      g->decode_rows = decode_rows;
      g->ws = ws;
      g->st = st;
      g->direct = !host_pinned(X_host) || !host_pinned(out_host) || (R_host && !host_pinned(R_host));
    } else if (!g->direct) {
      if (g->exec == nullptr) {
        // second call: capture the copies and kernels once
        cudaGraph_t graph = nullptr;
        const long long l0 = g_launches.load();
        bool ok = cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed) == cudaSuccess;
        int rr = ok ? host_forward_enqueue(d, X_host, R_host, out_host, T, ws, st) : QMOE_ERR_CUDA;
        if (ok) ok = cudaStreamEndCapture(st, &graph) == cudaSuccess && rr == QMOE_OK;
        if (ok) ok = cudaGraphInstantiate(&g->exec, graph, 0) == cudaSuccess;
        if (graph) cudaGraphDestroy(graph);
        if (!ok) {
          cudaGetLastError();
          if (g->exec) cudaGraphExecDestroy(g->exec);
          g->exec = nullptr;
          g->direct = true;
          if (rr != QMOE_OK && rr != QMOE_ERR_CUDA) return rr;
        } else {
          g->launches = g_launches.load() - l0;
          g->path = g_last_path;
        }
      }
      if (g->exec) {
        if (cudaGraphLaunch(g->exec, st) != cudaSuccess) return QMOE_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return QMOE_ERR_CUDA;
        g_launches.fetch_add(g->launches);
        g_last_path = g->path;
        ++g->calls;
        return QMOE_OK;
      }
    }
    ++g->calls;
  }
  r = host_forward_enqueue(d, X_host, R_host, out_host, T, ws, st);
  if (r != QMOE_OK) return r;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QMOE_ERR_CUDA;
  return QMOE_OK;
}

long long qmoe_launch_count(void) { return g_launches.load(); }

int qmoe_test_inject(int site, int wait_us) {
  if (site < 0 || site > QMOE_FAULT_ATTN_FINAL || wait_us < 0) return QMOE_ERR_ARG;
  g_fault_wait_us.store(wait_us);
  g_fault_site.store(site);
  return QMOE_OK;
}

int qmoe_profile_start(int stage) {
  if (stage < 0 || stage > QMOE_STAGE_DECODE) return QMOE_ERR_ARG;
  g_prof.stage = stage;
  g_prof.n = 0;
  return QMOE_OK;
}

int qmoe_profile_read(double* total_ms, int* launches) {
  if (!total_ms || !launches) return QMOE_ERR_NULL;
  double tot = 0.0;
  for (int i = 0; i < g_prof.n; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.stop[i]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.start[i], g_prof.stop[i]) != cudaSuccess)
      return QMOE_ERR_CUDA;
    tot += ms;
  }
  *total_ms = tot;
  *launches = g_prof.n;
  return QMOE_OK;
}

int qmoe_profile_stop(double* total_ms, int* launches) {
  if (!total_ms || !launches) return QMOE_ERR_NULL;
  double tot = 0.0;
  for (int i = 0; i < g_prof.n; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.stop[i]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.start[i], g_prof.stop[i]) != cudaSuccess)
      return QMOE_ERR_CUDA;
    tot += ms;
  }
  *total_ms = tot;
  *launches = g_prof.n;
  g_prof.stage = 0;
  g_prof.n = 0;
  return QMOE_OK;
}

}  // extern "C"
