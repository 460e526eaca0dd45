/*
 * qmoe.h -- C ABI of libqmoe.so, a GB300 (sm_103a) library for the k-quant
 * weight-quantized routed-MoE layer of a Qwen3.5-35B-A3B-shaped transformer
 * block and for that block.
 *
 * Sources (the operations; the pages describe no API):
 *   [CKE-Zip]  "CKE Zip: From Splitting Tokens To Splitting Qwen3.5 Weights",
 *              sections "What The First Prototype Split" (hidden rows X [T, H],
 *              selected top-k expert indices and routing weights, routed and
 *              shared SwiGLU branches), "What PR #382 Now Splits" (256 routed
 *              experts, eight per token, Q4_K gate/up and Q5_K down weights,
 *              the 256/256 intermediate split, 16 query / 2 KV heads, the
 *              block recombination order) and "A Separate Decode Result Shows
 *              Why Axis Choice Matters" (routes merged in selected-slot order).
 *   [CKE-Dist] "Distributed CPU: Zip Fusion Beyond Tensor Parallelism",
 *              "The Reduction Algebra" and "Streaming reductions" (partials are
 *              summed in a fixed, declared order).
 *
 * Conventions for every entry point:
 *   - Every pointer argument except the descriptors is a DEVICE pointer on the
 *     current CUDA device, owned by the caller. The library allocates nothing
 *     and frees nothing; scratch lives in the caller's workspace ``ws``.
 *   - All work is enqueued on ``stream`` (a cudaStream_t; NULL = the legacy
 *     default stream) with no host synchronisation. Buffers must stay valid
 *     until that work completes.
 *   - Row-major, contiguous tensors. fp32 tensors, packed weights and the
 *     workspace must be 16-byte aligned (the workspace 256-byte aligned).
 *   - Return value: QMOE_OK or a negative qmoe_status; nothing is enqueued
 *     when an argument check fails. Errors detected on the device (an expert
 *     id out of range in caller-supplied routes, a bounded wait that ran out)
 *     are recorded in a per-device status word read by qmoe_query_status().
 *   - T = 0 is valid and enqueues nothing.
 *
 * Packed super-block formats (256 weights, 8 sub-blocks of 32; the pages name
 * Q4_K and Q5_K only, so this byte layout is the library's own):
 *   Q4_K, 144 bytes: [0,2) d fp16; [2,4) dmin fp16; [4,16) sixteen 6-bit
 *     fields packed little-endian, fields 0..7 the scales s_j, 8..15 the mins
 *     m_j; [16,144) quants, byte b = weight 2b (low nibble), 2b+1 (high).
 *   Q5_K, 176 bytes: the same 16-byte header; [16,48) high bits, weight i is
 *     bit i%8 of byte 16 + i/8; [48,176) low nibbles as in Q4_K.
 *   Weight i (sub-block j = i/32): w_i = d*s_j*q_i - dmin*m_j, q_i the 4-bit
 *   quant (Q4_K) or quant + 16*high bit (Q5_K).
 *   Q6_K, 210 bytes ("CKE Zip: From Splitting Tokens To Splitting Qwen3.5
 *     Weights", opening paragraphs: a Q4_K_M model file keeps some tensors in
 *     Q6_K; the layout is the library's own): [0,2) d fp16; [2,18) sixteen
 *     signed 8-bit scales s_0..s_15, one per 16 weights; [18,82) 2-bit high
 *     parts, weight i in bits 2(i%4)..2(i%4)+1 of byte 18 + i/4; [82,210) low
 *     nibbles as in Q4_K. w_i = d*s_{i/16}*(q_i - 32), q_i = nibble + 16*high.
 *   MXFP4, 136 bytes ("Distributed CPU: Zip Fusion Beyond Tensor
 *     Parallelism", "Decode vs Prefill: Same Weights, Different
 *     Bottlenecks": an MXFP4-class format; element and scale types of the OCP
 *     microscaling format, the 256-weight grouping the library's own): [0,8)
 *     E8M0 scales e_0..e_7, one per 32 weights (2^(e-127), 255 = NaN);
 *     [8,136) FP4 E2M1 codes (sign, 2 exponent bits, 1 mantissa bit), byte b
 *     = weight 2b (low nibble), 2b+1 (high). w_i = 2^(e_{i/32}-127)*E2M1(code).
 *   Q6_K and MXFP4 are taken by the grouped GEMV path at every row count
 *   (qmoe_last_path() reports it); the decode and tensor-core paths take
 *   Q4_K and Q5_K.
 *   Matrices are stored one output feature per row, super-blocks running
 *   along the input (reduction) axis: a [rows][cols] matrix with cols % 256
 *   == 0 is rows * (cols/256) consecutive super-blocks.
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qmoe_stream_t; /* same type as cudaStream_t */

typedef enum {
  QMOE_OK = 0,
  QMOE_ERR_ARG = -1,         /* a size or type argument is out of range      */
  QMOE_ERR_NULL = -2,        /* a required pointer is NULL                   */
  QMOE_ERR_ALIGN = -3,       /* a pointer is not 16-byte (workspace 256) aligned */
  QMOE_ERR_WORKSPACE = -4,   /* ws_bytes is below the queried requirement    */
  QMOE_ERR_ARCH = -5,        /* the current device is not sm_103             */
  QMOE_ERR_LAUNCH = -6,      /* a kernel launch failed (cudaGetLastError)    */
  QMOE_ERR_TIMEOUT = -7,     /* device: a bounded wait ran out               */
  QMOE_ERR_DEVICE_ARG = -8,  /* device: caller-supplied route out of range   */
  QMOE_ERR_CUDA = -9,        /* another CUDA runtime error                   */
  QMOE_ERR_TOO_LARGE = -10   /* the problem needs more than the library's fixed scratch */
} qmoe_status;

typedef enum { QMOE_Q4K = 0, QMOE_Q5K = 1, QMOE_Q6K = 2, QMOE_MXFP4 = 3 } qmoe_qtype;

/* Execution path the last successful qmoe_moe_forward took on this thread. */
typedef enum {
  QMOE_PATH_NONE = 0,
  QMOE_PATH_GEMV = 1,     /* grouped dequant-fused GEMV kernels        */
  QMOE_PATH_GEMM_TC = 2,  /* grouped dequant + bf16 tcgen05 GEMM       */
  QMOE_PATH_DECODE = 3    /* T <= 4: router + persistent expert kernel */
} qmoe_path;

/*
 * One routed-MoE layer ([CKE-Zip] "What PR #382 Now Splits").
 *   H  hidden width, multiple of 256;  E routed experts, 1..1024;
 *   k  experts per row, 1..min(E, 16); F expert intermediate, multiple of 256.
 *   Wr       fp32 [H][E] router weights (logits = x . Wr).
 *   Wg, Wu   gate / up, gate_type, [E][F rows][H/256 blocks].
 *   Wd       down, down_type, [E][H rows][F/256 blocks].
 *   Sg,Su,Sd the shared expert, same per-expert shapes and types, or all NULL.
 */
typedef struct {
  int H, E, k, F;
  int gate_type, down_type; /* qmoe_qtype */
  const float *Wr;
  const void *Wg, *Wu, *Wd;
  const void *Sg, *Su, *Sd;
} qmoe_moe_desc;

/*
 * Router: logits = X . Wr (fp32), then per row the k largest logits (equal
 * logits: the lower expert index first), in descending-logit slot order, with
 * weights w_s = exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0), which is the
 * softmax over all E renormalised over the selected k.
 * The logits are fp32-accurate: summed on the CUDA cores, or, from T = 256
 * rows when E is a multiple of 128 and H of 256, on the bf16 tensor cores with
 * every fp32 value of X and Wr split exactly into three bf16 parts (six part
 * products accumulated in fp32, over at least 4 slices of H); the workspace
 * then also holds Wr's parts, 3 * E * H * 2 bytes.
 * ([CKE-Zip] "What The First Prototype Split": selected top-k indices and
 * routing weights; "What PR #382 Now Splits": one synchronised router decision.)
 *   X [T][H] fp32, Wr [H][E] fp32 -> ids [T][k] int32, w [T][k] fp32.
 *   ws: qmoe_moe_route_workspace_bytes(T, H, E, k) bytes.
 */
size_t qmoe_moe_route_workspace_bytes(int T, int H, int E, int k);
int qmoe_moe_route(const float *X, const float *Wr, int T, int H, int E, int k,
                   int32_t *ids, float *w, void *ws, size_t ws_bytes,
                   qmoe_stream_t stream);

/*
 * The routed-MoE layer on rows X [T][H] fp32:
 *   out_t = R_t + y_shared,t + sum_{s=0}^{k-1} w_{t,s} * y_{t,s}
 * with y = down(silu(gate(x)) * up(x)) per selected expert and for the shared
 * expert (weight 1, no gate), the slot sum taken in slot order s = 0..k-1
 * without atomics, so the result is run-to-run bit-identical.
 * ([CKE-Zip] "What The First Prototype Split", "What PR #382 Now Splits",
 * "A Separate Decode Result Shows Why Axis Choice Matters".)
 *   R    [T][H] fp32 residual, or NULL for none (R may equal out).
 *   ids, w  [T][k] int32 / fp32 precomputed routes (e.g. one synchronised
 *        decision shared by two rank partials), or both NULL to route X here.
 *   out  [T][H] fp32; may alias R but not X.
 *   ws   qmoe_moe_workspace_bytes(d, T) bytes, 256-byte aligned.
 * T <= 4 (internal routing) takes the decode path, other small T the
 * dequant-fused grouped GEMV path (both fp32 accumulation); large T the
 * grouped dequant + bf16 tcgen05 GEMM path (fp32 accumulation in tensor
 * memory); qmoe_last_path() tells which ran.
 * A rank partial of the intermediate split is computed by passing that
 * rank's slices of the packed tensors with F halved.
 * T * (k + 1) must stay below 2^24 (QMOE_ERR_ARG otherwise).
 */
size_t qmoe_moe_workspace_bytes(const qmoe_moe_desc *d, int T);
int qmoe_moe_forward(const qmoe_moe_desc *d, const float *X, const float *R,
                     const int32_t *ids, const float *w, float *out, int T,
                     void *ws, size_t ws_bytes, qmoe_stream_t stream);

/* Path selection threshold: T above it takes the tensor-core path (built-in
 * value 4 rows: from 5 rows on, one pass over each expert's weights on the
 * tensor cores beats the grouped GEMV). qmoe_set_gemm_threshold(-1) restores
 * the built-in value. */
int qmoe_get_gemm_threshold(void);
void qmoe_set_gemm_threshold(int rows);
int qmoe_last_path(void);

/* Rows up to this count (at most 4, the built-in value) take the decode path
 * when the layer's routes are computed internally and the shape allows it
 * (H 1024 or 2048, F 256 or 512, E a multiple of 8): a router kernel and one
 * persistent expert kernel (one CTA per SM, cooperative launch) chained with
 * programmatic dependent launch, every CTA taking the top-k itself; the
 * expert kernel's CTAs form the slot-order combine. 0 turns it off; -1
 * restores the built-in value. */
int qmoe_get_decode_max_rows(void);
void qmoe_set_decode_max_rows(int rows);

/*
 * Byte offsets of the intermediates inside a moe_forward workspace, for
 * stagewise checks: ids [T][k] int32, w [T][k] fp32, offsets [E+2] int32
 * (row ranges per expert, the shared expert last), perm [T*k + T] int32 (pair
 * index t*k+s grouped by expert, stable), y [T*k + T][H] (fp32 per pair,
 * shared rows last, on the GEMV path; bf16 in permutation order, row i for
 * pair perm[i], on the tensor-core path). Valid after the forward has
 * completed.
 */
typedef struct {
  size_t ids, w, offsets, perm, y;
} qmoe_moe_ws_layout;
int qmoe_moe_workspace_layout(const qmoe_moe_desc *d, int T, qmoe_moe_ws_layout *out);

/*
 * End-to-end variant of qmoe_moe_forward on HOST buffers: copies X_host (and
 * R_host, if not NULL) into the workspace, runs the layer on ``stream``,
 * copies the result to out_host and waits for the stream. X_host, R_host and
 * out_host are [T][H] fp32 host arrays (pinned memory makes the copies
 * asynchronous DMA; pageable memory works too). ws is a DEVICE workspace of
 * qmoe_moe_forward_host_workspace_bytes(d, T) bytes. Routing is internal.
 * A call that repeats the arguments (descriptor contents, buffers, T, ws,
 * stream, device, path thresholds) of an earlier one replays a CUDA graph of
 * the copies and the kernels, captured on its second occurrence (the first
 * runs directly); calls with pageable buffers, on a stream that is already
 * capturing, or while a test fault site or stage profiling is set always run
 * directly. Same results either way. With pinned (mapped) host buffers of at
 * most 4 MiB, the layer's last kernel writes out_host itself and reads R_host
 * itself (no copy for them); X_host is always copied in.
 */
size_t qmoe_moe_forward_host_workspace_bytes(const qmoe_moe_desc *d, int T);
int qmoe_moe_forward_host(const qmoe_moe_desc *d, const float *X_host, const float *R_host,
                          float *out_host, int T, void *ws, size_t ws_bytes,
                          qmoe_stream_t stream);

/*
 * qmoe_moe_forward for callers that cannot allocate device memory (the paper
 * has no counterpart; it is an interface convenience). Some callers have no
 * way to hand over a workspace: plugin interfaces that give an operator only
 * its input and output buffers, or threads that must not call cudaMalloc
 * because it may synchronise the whole device. This entry point allocates
 * nothing and calls no allocating routine; its scratch is a fixed array of
 * QMOE_NOALLOC_SCRATCH_BYTES (8 MiB) in device memory that the library
 * declares, which every GPU that loads the library holds until the process
 * exits.
 *   Same arguments and result as qmoe_moe_forward with internal routing
 *   (no ids/w): X [T][H] fp32, R [T][H] fp32 or NULL, out [T][H] fp32.
 *   Returns QMOE_ERR_TOO_LARGE, enqueuing nothing and leaving ``out``
 *   untouched, when qmoe_moe_workspace_bytes(d, T) exceeds the scratch size;
 *   the largest row count that fits is therefore the largest T whose
 *   workspace is at most QMOE_NOALLOC_SCRATCH_BYTES (86 rows at the
 *   Qwen3.5-35B-A3B layer shape: H=2048, E=256, k=8, F=512, shared expert).
 *   The first call on each device looks up the scratch array's device
 *   address with that device current; make that first call before any
 *   stream capture. Every call on a device shares the one array and leaves
 *   its contents behind; nothing in it needs to start at zero, because every
 *   byte a call reads is written earlier in the same call. Calls whose work
 *   overlaps on the GPU (other streams, other host threads) race on the
 *   array: serialise them.
 */
#define QMOE_NOALLOC_SCRATCH_BYTES (8u << 20)
int qmoe_moe_forward_noalloc(const qmoe_moe_desc *d, const float *X, const float *R,
                             float *out, int T, qmoe_stream_t stream);

/*
 * Test-only fault injection (the pages have no counterpart: this exists so
 * that the library's bounded device waits can be exercised without faulting
 * a GPU). While a site is set, every call that reaches that site
 * withholds one copy or arrival, so that one wait can never complete; the
 * waiting CTA gives up after ``wait_us`` microseconds (0: the normal limit of
 * 2 s), records QMOE_ERR_TIMEOUT in the status word and returns with nothing
 * of its own in flight. The call's ``out`` is then incomplete. Sites:
 *   QMOE_FAULT_NONE        off (the default);
 *   QMOE_FAULT_DECODE_COPY decode path: the first CTA never copies the down
 *                          weights of its last down unit;
 *   QMOE_FAULT_TC_ARRIVE   tensor-core path, gate/up kernel: the first CTA's
 *                          producers never mark the last stage of their last
 *                          work item stored;
 *   QMOE_FAULT_ATTN_FINAL  block prefill attention (T > 16): the first CTA's
 *                          P V issuer never marks its output final, so its
 *                          softmax warps' last wait runs out.
 * Returns QMOE_ERR_ARG for an unknown site or a negative wait. Not for use
 * outside tests; set QMOE_FAULT_NONE afterwards.
 */
enum { QMOE_FAULT_NONE = 0, QMOE_FAULT_DECODE_COPY = 1, QMOE_FAULT_TC_ARRIVE = 2, QMOE_FAULT_ATTN_FINAL = 3 };
int qmoe_test_inject(int site, int wait_us);

/* Number of kernels this library has enqueued since it was loaded (a CUDA
 * graph replay of captured launches does not add to it). */
long long qmoe_launch_count(void);

/*
 * Stage timing. After qmoe_profile_start(stage), every launch of that stage
 * by this thread is bracketed with a pair of CUDA events on its stream, up to
 * 4096 launches; qmoe_profile_stop waits for them and returns the summed
 * kernel time in milliseconds and the launch count, and turns profiling off.
 * stage 0 turns profiling off. While the stream is capturing a graph the
 * events are recorded as event-record nodes of that graph
 * (cudaEventRecordExternal): after each replay of the graph,
 * qmoe_profile_read returns the summed times of that replay's bracketed
 * launches without turning profiling off (call qmoe_profile_stop once done).
 */
typedef enum {
  QMOE_STAGE_ROUTER = 1,  /* router logits                          */
  QMOE_STAGE_ROUTE = 2,   /* top-k, histogram, scan, permutation    */
  QMOE_STAGE_GATEUP = 3,  /* grouped gate/up + SwiGLU               */
  QMOE_STAGE_DOWN = 4,    /* grouped down projection                */
  QMOE_STAGE_COMBINE = 5, /* slot-order combine + shared + residual */
  QMOE_STAGE_DECODE = 6   /* the decode path's two chained kernels, as one unit */
} qmoe_stage;
int qmoe_profile_start(int stage);
int qmoe_profile_stop(double *total_ms, int *launches);
int qmoe_profile_read(double *total_ms, int *launches);

/*
 * One transformer block around the MoE layer ([CKE-Zip] "What PR #382 Now
 * Splits": full attention with 16 query heads and 2 KV heads, then the MoE
 * layer, each with its residual):
 *   h1  = X + O( attention( RoPE(Q(r1)), RoPE(K(r1)), V(r1) ) ),  r1 = RMSNorm(X; g1)
 *   out = h1 + moe( RMSNorm(h1; g2) )
 * RMSNorm(x; g) = x / sqrt(mean(x^2) + eps) * g. RoPE rotates pairs (i, i+hd/2)
 * by pos * theta^(-2i/hd). Query head h reads KV head h / (n_heads/n_kv);
 * scores are scaled by 1/sqrt(hd), causal. Keys and values are rounded to
 * bf16 (nearest even) when written to the cache. No biases, no QK-norm.
 *   Wq [n_heads*hd][H/256], Wk, Wv [n_kv*hd][H/256], Wo [H][n_heads*hd/256]:
 *   Q4_K super-blocks (formats above). g1, g2: fp32 [H].
 *   moe: the MoE layer (moe.H == H).
 */
typedef struct {
  int H, n_heads, n_kv, head_dim;
  float rope_theta, eps;
  const float *g1, *g2;
  const void *Wq, *Wk, *Wv, *Wo;
  qmoe_moe_desc moe;
} qmoe_block_desc;

/* y = RMSNorm(X; gamma) for X, y [T][H] fp32 (y may equal X). */
int qmoe_rmsnorm(const float *X, const float *gamma, float eps, float *y, int T, int H,
                 qmoe_stream_t stream);

/*
 * The attention branch: out = R + O(attention(...)) for rows X [T][H] at
 * positions pos0 .. pos0+T-1 (R [T][H] or NULL). k_cache, v_cache: bf16 bit
 * patterns [ctx_cap][n_kv][hd]; positions 0..pos0-1 must hold earlier keys and
 * values, positions pos0..pos0+T-1 are written. pos0 + T <= ctx_cap.
 * A rank partial of the head split is this call with that rank's query heads,
 * KV head(s), cache and O-projection input columns, and R = NULL.
 */
size_t qmoe_attn_workspace_bytes(const qmoe_block_desc *b, int T, int pos0);
int qmoe_attn_forward(const qmoe_block_desc *b, const float *X, const float *R, float *out, int T,
                      uint16_t *k_cache, uint16_t *v_cache, int pos0, int ctx_cap, void *ws,
                      size_t ws_bytes, qmoe_stream_t stream);

/* The whole block (out [T][H] fp32, may not alias X). */
size_t qmoe_block_workspace_bytes(const qmoe_block_desc *b, int T, int pos0);
int qmoe_block_forward(const qmoe_block_desc *b, const float *X, float *out, int T,
                       uint16_t *k_cache, uint16_t *v_cache, int pos0, int ctx_cap, void *ws,
                       size_t ws_bytes, qmoe_stream_t stream);

/* The CUDA runtime error code (cudaError_t) behind the last QMOE_ERR_LAUNCH
 * returned on this thread, 0 if none. */
int qmoe_last_cuda_error(void);

/* Human-readable text of a status code (static storage). */
const char *qmoe_status_str(int status);

/* Waits for ``stream``, then returns and clears the device status word of the
 * current device (QMOE_OK if no kernel recorded an error). */
int qmoe_query_status(qmoe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QMOE_H */
