// Launchers of the library's kernels (host side), one translation unit each.
#pragma once

#include "common.cuh"

namespace qmoe {

// device_cache.cu: per-device launch bookkeeping. ensure_kernel_smem raises
// ``fn``'s dynamic shared-memory limit to at least ``smem`` bytes on the
// current device (and sets the preferred carveout when ``carveout`` >= 0),
// once per (device, kernel, size); device_sm_count is the current device's SM
// count.
cudaError_t ensure_kernel_smem(const void* fn, size_t smem, int carveout = -1);
int device_sm_count();

// router.cu
int router_splits(int T, int H, int E);
// ``wr3``: scratch of router_tc_ws_bytes(T, H, E) bytes, used (with ``status``)
// by the tensor-core router when router_tc_eligible(T, H, E)
cudaError_t launch_router_logits(const float* X, const float* Wr, float* part, int T, int H, int E,
                                 int nsplit, void* wr3, int* status, cudaStream_t st);
int router_launches(int T, int H, int E);
// router_tc.cu
bool router_tc_eligible(int T, int H, int E);
int router_tc_splits(int T, int H, int E);
size_t router_tc_ws_bytes(int T, int H, int E);
cudaError_t launch_router_tc(const float* X, const float* Wr, float* part, int T, int H, int E, int nsplit,
                             void* wr3, int* status, cudaStream_t st);
cudaError_t launch_topk(const float* part, int nsplit, int T, int E, int k, int32_t* ids, float* w,
                        cudaStream_t st);
size_t route_small_smem(int T, int E, int k);
// with ``chunks`` set, also the tensor-core path's token-chunk list (cap 64,
// 128 or 192 rows)
cudaError_t launch_route_small(const float* part, int nsplit, const int32_t* ids_in, int T, int E,
                               int k, int has_shared, int32_t* ids, float* w, int32_t* offsets,
                               int32_t* perm, int32_t* active, int32_t* n_active, int* status,
                               cudaStream_t st, int cap = 0, int2* chunks = nullptr,
                               int32_t* n_tok_chunks = nullptr);
int perm_chunks(int P);
// with ``chunks`` set, also the tensor-core path's token-chunk list (cap 64,
// 128 or 192 rows), as launch_build_chunks would build it
cudaError_t launch_perm_large(const int32_t* ids, int T, int E, int k, int has_shared,
                              int32_t* chunk_cnt, int32_t* offsets, int32_t* perm,
                              int32_t* active, int32_t* n_active, int* status, cudaStream_t st,
                              int cap = 0, int2* chunks = nullptr, int32_t* n_tok_chunks = nullptr);

// moe_gemv.cu: grouped dequant-fused GEMV kernels and the combine.
struct GroupedArgs {
  const uint8_t* W;        // routed experts, [E][rows][cols/256] super-blocks
  const uint8_t* S;        // shared expert (expert index E) or nullptr
  const int32_t* offsets;  // [E+2]
  const int32_t* perm;     // [T*k + T]
  const int32_t* active;   // [E+1]
  const int32_t* n_active; // [1]
  int T, k, E;
  int max_active;          // grid bound on the active-expert count
};
cudaError_t launch_gateup_gemv(const GroupedArgs& g, const uint8_t* Wu, const uint8_t* Su, int qt,
                               const float* X, int H, int F, float* hbuf, cudaStream_t st);
cudaError_t launch_down_gemv(const GroupedArgs& g, int qt, const float* hbuf, int F, int H,
                             float* y, cudaStream_t st);
cudaError_t launch_combine(const float* y, const float* w, const float* R, float* out, int T,
                           int H, int k, int has_shared, cudaStream_t st);

// moe_gemm_tc.cu: grouped dequant + bf16 tcgen05 GEMM path.
struct GroupedTcArgs {
  const uint8_t *W, *W2, *S, *S2;  // (gate, up, shared gate, shared up) or (down, -, shared down, -)
  int qt;
  const int32_t* offsets;
  const int32_t* perm;
  const int2* chunks;       // token chunks of at most 128 rows, built on the device
  const int32_t* n_chunks;
  int max_chunks;           // grid bound on the chunk count
  const __nv_bfloat16* xb;
  const __nv_bfloat16* hin;
  __nv_bfloat16* hout;
  __nv_bfloat16* yout;
  float* yout_f32;    // down pass: write fp32 instead of bf16 when not null
  int tok_shift;      // down pass: the shared expert's token rows start this many rows before its output rows
  int tok_rows;     // rows of the token matrix (xb for gate/up, hin for down)
  int nmax;         // chunk cap the chunk list was built with (64, 128 or 192)
  int T, k, E, H, F;
  int* status;
  unsigned long long wait_ns;  // bound on a device wait (0: the default 2 s)
  int fault;                   // test-only fault site of the gate/up kernel (0 = none)
};
int tc_max_chunks(int T, int k, int E, int has_shared);
int tc_chunk_cap(int T, int k, int E);
cudaError_t launch_build_chunks(const int32_t* offsets, int E, int cap, int2* chunks, int32_t* n_chunks,
                                cudaStream_t st);
cudaError_t launch_gateup_tc(const GroupedTcArgs& p, cudaStream_t st);
cudaError_t launch_down_tc(const GroupedTcArgs& p, cudaStream_t st);
cudaError_t launch_to_bf16(const float* x, __nv_bfloat16* y, int rows, int K, const int32_t* perm, int T, int k,
                           int32_t* inv, cudaStream_t st);
cudaError_t launch_combine_bf16(const __nv_bfloat16* y, const int32_t* inv, const float* w, const float* R,
                                float* out, int T, int H, int k, int has_shared, cudaStream_t st);

// block.cu: the attention + MoE block's other kernels.
cudaError_t launch_rmsnorm(const float* x, const float* gamma, float eps, float* y, int T, int H, cudaStream_t st);
// RMSNorm straight into the bf16 token operand of a tensor-core projection.
cudaError_t launch_rmsnorm_bf16(const float* x, const float* gamma, float eps, __nv_bfloat16* y, int T, int H,
                                cudaStream_t st);
cudaError_t launch_dense_route(int32_t* offsets, int32_t* perm, int32_t* active, int32_t* n_active, int T,
                               cudaStream_t st, int32_t* offsets2 = nullptr);
cudaError_t launch_rope_cache(float* q, const float* k, const float* v, __nv_bfloat16* kc, __nv_bfloat16* vc, int T,
                              int pos0, int nh, int nkv, int hd, double theta, cudaStream_t st);
int attn_nchunks(int T, int pos0);
// With ``ob`` (prefill only), the output rows go there as bf16 in the
// tensor-core operand order (kPerm8 inside each group of 8) instead of to ``o``.
cudaError_t launch_attention(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, float* part, float* o,
                             __nv_bfloat16* ob, int T, int pos0, int nh, int nkv, int hd, bool chunked, int* status,
                             unsigned long long wait_ns, int fault, cudaStream_t st);
cudaError_t launch_add(const float* a, const float* b, float* y, size_t n, cudaStream_t st);

// attn_prefill.cu: causal attention for many query rows (head_dim 128) on the
// tcgen05 tensor cores (S and O in tensor memory); bounded waits record
// QMOE_ERR_TIMEOUT in *status.
// ``fault`` (test-only): 1 = CTA 0's P V issuer never marks its output final.
cudaError_t launch_attention_prefill_tc(const float* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, float* o,
                                        __nv_bfloat16* ob, int T, int pos0, int nh, int nkv, int* status,
                                        unsigned long long wait_ns, int fault, cudaStream_t st);

// moe_decode.cu: the decode path for T <= 4 (router kernel + one persistent
// expert kernel, programmatic dependent launch).
struct DecodeLaunch {
  const float* X;
  const float* R;
  float* out;
  const float* Wr;
  const uint8_t *Wg, *Wu, *Wd, *Sg, *Su, *Sd;
  int T, H, E, k, F, gate_qt, down_qt;
  float* part;
  float* hbuf;
  float* ybuf;
  int32_t* ids;
  float* w;
  int* sync;                   // decode_sync_ints(H) ints, cleared by the router kernel
  int* status;
  unsigned long long wait_ns;  // a bounded wait gives up after this long
  int fault;                   // test-only fault site (0 = none)
};
int decode_sync_ints(int H);
bool decode_path_supported(int T, int H, int E, int k, int F, int gate_qt, int down_qt);
cudaError_t launch_decode(const DecodeLaunch& L, cudaStream_t st);

}  // namespace qmoe
