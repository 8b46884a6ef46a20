/*
 * lmoe.h -- C ABI of the GB300 (sm_103a) latent mixture-of-experts layer.
 *
 * The layer ("Muse Spark Open on Gaudi 2", section "The latent MoE: A' with a
 * per-expert norm"; "Soporte de dia 0 para Muse Spark Open en vLLM", section
 * "MoE latente"):
 *
 *   logits = fp32(x) . Wr^T (+ bias)        fp32 router, E experts, top k
 *   idx, w = top-k(logits), softmax over all E renormalised over the k picks
 *   x_lat  = bf16(x . P^T)                   pooler   H -> L
 *   per (token t, route j) row r = t*k + j, expert e = idx[t][j]:
 *     h_r  = bf16(silu(x_lat[t] . Wg_e^T) * (x_lat[t] . Wu_e^T))   MXFP4 W4A16
 *     y_r  = h_r . Wd_e^T                                          fp32, kept per row
 *     yh_r = y_r * rsqrt(mean(y_r^2) + eps) * g_e                  post_expert_norm
 *   z_t    = sum_j w[t][j] * yh_{t*k+j}      fp32, in route order j
 *   out    = bf16(bf16(z) . U^T)             unpooler L -> H
 *
 * Conventions
 *  - Every pointer argument is a DEVICE pointer owned by the caller unless a
 *    comment says otherwise.  The library never allocates, frees or keeps a
 *    pointer after a call returns.
 *  - Matrices are row-major [N_out][K_in] (K contiguous).  bf16 tensors are
 *    passed as uint16_t bit patterns.
 *  - MXFP4 (OCP MX v1.0): codes [N][K/2] bytes, element 2m in the low nibble
 *    of byte m, element 2m+1 in the high nibble; one E8M0 scale byte per 32
 *    consecutive K elements, [N][K/32].  Weights are read as stored; there is
 *    no repacking ("Muse Spark Open on Gaudi 2", "At a glance", "Why it
 *    needed a port").
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous.  Host-detectable errors are returned
 *    directly; errors found on the device (a wait that ran out, a routing
 *    table entry out of range) are written to the status word inside the
 *    workspace and read back with lmoe_status_check().
 *  - Calls sharing one workspace must not overlap in time.
 *  - Constraints checked on the host: hidden, latent, inter multiples of 128;
 *    1 <= top_k <= 8; top_k <= n_experts <= 256; 1 <= T <= 65536; every
 *    pointer 16-byte aligned; a compute-capability 10.3 device (else
 *    LMOE_EINVAL / LMOE_EUNSUPPORTED).  Supported shapes (else
 *    LMOE_EUNSUPPORTED): hidden, latent, inter multiples of 256; latent and
 *    inter at most 8192, and multiples of 2048 when above 2048.
 */
#ifndef LMOE_H
#define LMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LMOE_API __attribute__((visibility("default")))
#else
#define LMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lmoe_stream_t; /* identical to cudaStream_t */

enum {
  LMOE_OK = 0,
  LMOE_EINVAL = -1,        /* bad argument: null/misaligned pointer, bad dims */
  LMOE_EUNSUPPORTED = -2,  /* dims or device outside what the kernels support */
  LMOE_ECUDA = -3,         /* a CUDA runtime call failed */
  LMOE_ETIMEOUT = -4,      /* a bounded device-side wait ran out */
  LMOE_EDEVICE_CHECK = -5, /* a device-side input check failed (e.g. expert id) */
  LMOE_EWORKSPACE = -6,    /* workspace too small */
  LMOE_ENOSCRATCH = -7     /* larger than the fixed scratch of lmoe_route_noalloc */
};

typedef struct {
  int32_t T;         /* tokens in this call */
  int32_t hidden;    /* H, e.g. 8192 */
  int32_t latent;    /* L, e.g. 4096 */
  int32_t inter;     /* I, expert intermediate width, e.g. 4096 */
  int32_t n_experts; /* E, e.g. 256 */
  int32_t top_k;     /* k, e.g. 8 */
  float eps;         /* post_expert_norm epsilon, e.g. 1e-6 */
} lmoe_dims;

typedef struct {
  const float* router_w;      /* fp32 [E][H] */
  const float* router_bias;   /* fp32 [E], or NULL for none */
  const uint16_t* pooler_w;   /* bf16 [L][H] */
  const uint8_t* w13_q;       /* MXFP4 codes [E][2I][L/2]; rows 0..I-1 gate, I..2I-1 up */
  const uint8_t* w13_s;       /* E8M0 scales [E][2I][L/32] */
  const uint8_t* w2_q;        /* MXFP4 codes [E][L][I/2] (down projection) */
  const uint8_t* w2_s;        /* E8M0 scales [E][L][I/32] */
  const uint16_t* norm_g;     /* bf16 [E][L], per-expert post_expert_norm gain */
  const uint16_t* unpooler_w; /* bf16 [H][L] */
} lmoe_weights;

/* Byte offsets of the intermediates that lmoe_forward leaves in the workspace
 * (for inspection and tests; valid after the stream has reached the end of
 * the call).  Offsets are from the workspace base. */
typedef struct {
  size_t status;         /* int32[2]: code, location */
  size_t topk_idx;       /* int32 [T][k] */
  size_t topk_w;         /* fp32 [T][k] */
  size_t expert_offsets; /* int32 [E+1] */
  size_t sorted_rows;    /* int32 [T*k] */
  size_t row_pos;        /* int32 [T*k] */
  size_t x_lat;          /* bf16 [T][L] */
  size_t y;              /* fp32 [T*k][L], row t*k+j */
  size_t z;              /* bf16 [T][L], bf16(z) as fed to the unpooler */
  size_t total;          /* = lmoe_workspace_bytes() */
} lmoe_ws_layout;

/* Workspace size in bytes for `dims` (0 if dims are invalid).  The workspace
 * must be 256-byte aligned device memory; its contents need no
 * initialisation and are overwritten by every call. */
LMOE_API size_t lmoe_workspace_bytes(const lmoe_dims* dims);

/* Fills `layout` for `dims`.  Returns LMOE_OK or LMOE_EINVAL. */
LMOE_API int lmoe_workspace_layout(const lmoe_dims* dims, lmoe_ws_layout* layout);

/* Router, top-k and routing table ("Muse Spark Open on Gaudi 2", "What was
 * built": fp32 router, 256 experts, top 8; "The latent MoE: A' with a
 * per-expert norm": one row per (token, route)).
 *   x              bf16 [T][H], the layer input
 *   router_w       fp32 [E][H];  router_bias fp32 [E] or NULL
 *   topk_idx       out int32 [T][k], descending logit, ties to the lower index
 *   topk_w         out fp32 [T][k], softmax over all E renormalised over the k
 *   expert_offsets out int32 [E+1], exclusive scan of per-expert row counts
 *   sorted_rows    out int32 [T*k], row ids r = t*k+j grouped by expert,
 *                  ascending r within an expert
 *   row_pos        out int32 [T*k], inverse of sorted_rows
 * Logits are fp32 sums of fp32 products (not TF32). */
LMOE_API int lmoe_route(const lmoe_dims* dims, const uint16_t* x, const float* router_w, const float* router_bias,
               int32_t* topk_idx, float* topk_w, int32_t* expert_offsets, int32_t* sorted_rows,
               int32_t* row_pos, void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* Pooler ("Soporte de dia 0 ...", "MoE latente": 8192 -> 4096 learned
 * projection shared by all experts).
 *   x        bf16 [T][H];  pooler_w bf16 [L][H]
 *   x_lat    out bf16 [T][L] = bf16_rne(sum_h x*P), fp32 accumulation.
 *   ws, ws_bytes  optional (ws may be NULL): the projection needs no
 *            scratch.  When a workspace is given, the call zeroes its status
 *            word and a bounded device wait that runs out is reported there
 *            (lmoe_status_check), as for every other layer call; with NULL
 *            nothing is recorded.  This optional pair is the only difference
 *            from a plain (dims, x, pooler_w, x_lat, stream) signature. */
LMOE_API int lmoe_pool(const lmoe_dims* dims, const uint16_t* x, const uint16_t* pooler_w, uint16_t* x_lat,
              void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* Routed experts, MXFP4 W4A16 SwiGLU, one output row per (token, route)
 * ("Muse Spark Open on Gaudi 2", "What was built": W4A16; "The latent MoE
 * ...": per-route rows, cost per touched expert slice).
 *   x_lat          bf16 [T][L]
 *   expert_offsets int32 [E+1] and sorted_rows int32 [T*k] as from lmoe_route
 *   w13_q/w13_s, w2_q/w2_s as in lmoe_weights
 *   y              out fp32 [T*k][L]; row r = t*k+j holds expert idx[t][j]'s
 *                  output for token t (before the norm)
 * Each touched expert slice is streamed from HBM once per group of up to 8
 * of its rows.  A row id outside [0, T*k) or offsets that are not monotone
 * are reported as LMOE_EDEVICE_CHECK in the status word. */
LMOE_API int lmoe_experts_mxfp4(const lmoe_dims* dims, const uint16_t* x_lat, const int32_t* expert_offsets,
                       const int32_t* sorted_rows, const uint8_t* w13_q, const uint8_t* w13_s,
                       const uint8_t* w2_q, const uint8_t* w2_s, float* y, void* ws, size_t ws_bytes,
                       lmoe_stream_t stream);

/* post_expert_norm on every route row, fp32 router-weighted sum, unpooler
 * ("Muse Spark Open on Gaudi 2", "The latent MoE ...": norm per row, then
 * x router weight, fp32 sum, unpool 4096 -> 8192; "Why it needed a port":
 * the norm applies to each expert's output before the weighted sum).
 *   y        fp32 [T*k][L];  topk_idx int32 [T][k];  topk_w fp32 [T][k]
 *   norm_g   bf16 [E][L];    unpooler_w bf16 [H][L]
 *   out      out bf16 [T][H] */
LMOE_API int lmoe_norm_combine_unpool(const lmoe_dims* dims, const float* y, const int32_t* topk_idx,
                             const float* topk_w, const uint16_t* norm_g, const uint16_t* unpooler_w,
                             uint16_t* out, void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* The whole layer: route, pool, experts, norm + combine + unpool.
 *   x   bf16 [T][H];  out bf16 [T][H]
 * Intermediates stay in the workspace (see lmoe_workspace_layout). */
LMOE_API int lmoe_forward(const lmoe_dims* dims, const lmoe_weights* weights, const uint16_t* x, uint16_t* out,
                 void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* The whole layer with its input and output in pinned host memory, for a
 * caller that holds the tokens on the host (a serving loop at decode sizes).
 * No counterpart in the pages: up to 256 KB each way (16 tokens at hidden
 * 8192) it moves the T x H bf16 tokens in and the output back with two small
 * kernels that read and write the host buffers over the host link, in place
 * of two copy-engine transfers; above that, with the copy engines.
 *   x_host    bf16 [T][H], page-locked host memory (cudaMallocHost /
 *             cudaHostAlloc, or cudaHostRegister'ed), 16-byte aligned
 *   out_host  out bf16 [T][H], page-locked host memory, 16-byte aligned;
 *             complete once the stream has reached the end of the call
 *   ws        at least lmoe_host_workspace_bytes(dims) bytes: the layer's
 *             workspace followed by a device staging buffer for the tokens
 *             and one for the output
 * The upload kernel also zeroes the workspace's status and counter words (the
 * other entry points launch a small kernel for that).  The result is
 * bit-identical to lmoe_forward on the same tokens.  Device, managed or
 * pageable pointers for x_host or out_host return LMOE_EINVAL; a short
 * workspace returns LMOE_EWORKSPACE. */
LMOE_API size_t lmoe_host_workspace_bytes(const lmoe_dims* dims);
LMOE_API int lmoe_forward_host(const lmoe_dims* dims, const lmoe_weights* weights, const uint16_t* x_host,
                               uint16_t* out_host, void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* The whole layer with caller-supplied routing ("Muse Spark Open on Gaudi 2",
 * "The latent MoE: A' with a per-expert norm": the experts, the per-route
 * post_expert_norm, the fp32 weighted sum and the unpooler all take the
 * routing as given).  The router is not run: the routing table is built from
 * topk_idx, the weighted sum uses topk_w as they are.  For replaying a
 * recorded routing, or forcing an expert choice.
 *   topk_idx in  int32 [T][k], device; expert ids in [0, E) (a token may name
 *                an expert more than once: each route row stays separate)
 *   topk_w   in  fp32 [T][k], device; the weights of the sum, used as given
 *   out      out bf16 [T][H]
 * weights->router_w and router_bias are ignored.  An id outside [0, E) is
 * reported on the device (LMOE_EDEVICE_CHECK through lmoe_status_check) and
 * counted as expert 0.  Workspace, streams and errors as for lmoe_forward. */
LMOE_API int lmoe_forward_routed(const lmoe_dims* dims, const lmoe_weights* weights, const uint16_t* x,
                                 const int32_t* topk_idx, const float* topk_w, uint16_t* out, void* ws,
                                 size_t ws_bytes, lmoe_stream_t stream);

/* NVFP4 expert weights (the pages' checkpoint format, "Muse Spark Open on
 * Gaudi 2" and the vLLM page; they give no layout, so this follows NVIDIA's
 * public NVFP4 description): the same E2M1 codes as MXFP4 (two per byte, low
 * nibble = even element), one FP8 E4M3 scale byte per 16 elements along K
 * (OCP FP8 E4M3: bias 7, no infinity, S.1111.111 = NaN), and an fp32 global
 * scale per expert matrix:  w[n][c] = E2M1 * E4M3(s[n][c/16]) * global[e].
 * With NVFP4, lmoe_weights.w13_s is E4M3 [E][2I][L/16] and w2_s [E][L][I/16]. */
typedef struct {
  const float* w13_gs; /* fp32 [E], global scale of each expert's W13 (gate and up) */
  const float* w2_gs;  /* fp32 [E], global scale of each expert's W2 */
} lmoe_nvfp4_scales;

/* lmoe_experts_mxfp4 on NVFP4 weights (see above); same arguments otherwise.
 *   w13_s E4M3 [E][2I][L/16];  w2_s E4M3 [E][L][I/16];  w13_gs, w2_gs fp32 [E] */
LMOE_API int lmoe_experts_nvfp4(const lmoe_dims* dims, const uint16_t* x_lat, const int32_t* expert_offsets,
                                const int32_t* sorted_rows, const uint8_t* w13_q, const uint8_t* w13_s,
                                const float* w13_gs, const uint8_t* w2_q, const uint8_t* w2_s, const float* w2_gs,
                                float* y, void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* lmoe_forward with NVFP4 experts: weights->w13_s and w2_s hold the E4M3
 * scales, `nv` the global scales.  Workspace, streams and errors as for
 * lmoe_forward (LMOE_EINVAL if nv or one of its arrays is NULL). */
LMOE_API int lmoe_forward_nvfp4(const lmoe_dims* dims, const lmoe_weights* weights, const lmoe_nvfp4_scales* nv,
                                const uint16_t* x, uint16_t* out, void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* The transformer block around the layer, with sandwich normalisation
 * ("Soporte de dia 0 para Muse Spark Open en vLLM", section "Normalizacion en
 * sandwich": y = x + post_norm(F(pre_norm(x)))), and the router fed by the
 * pre-norm's fp32 output (same page, section "Nvidia").
 *   pre_norm, post_norm: RMSNorm over H, n = (x * rinv) * g with
 *     rinv = 1/sqrt(sum(x^2)/H + eps) and a bf16 gain g per column
 *   F: the layer of lmoe_forward; its router takes the pre-norm output in
 *     fp32, its pooler that output rounded to bf16
 *   y = bf16(x + post_norm(F(...))), the residual sum in fp32
 * Each norm gain is a bf16 [H] device array; eps applies to both norms. */
typedef struct {
  const uint16_t* pre_g;  /* bf16 [H], gain of the norm before the layer */
  const uint16_t* post_g; /* bf16 [H], gain of the norm after the layer */
  float eps;              /* both norms' epsilon (inside the square root), >= 0 */
} lmoe_block_norms;

/* Workspace size in bytes for lmoe_block_forward (0 if dims are invalid):
 * lmoe_workspace_bytes plus the pre-norm output, its per-token scale, the
 * router's split input and the layer's output.  Same alignment rule. */
LMOE_API size_t lmoe_block_workspace_bytes(const lmoe_dims* dims);

/* The block above.
 *   x   bf16 [T][H], the residual stream;  y out bf16 [T][H] (may be x itself,
 *       for an in-place update)
 * The layer's intermediates stay in the workspace at the offsets of
 * lmoe_workspace_layout.  Streams and errors as for lmoe_forward; the
 * workspace must hold lmoe_block_workspace_bytes (LMOE_EWORKSPACE if not). */
LMOE_API int lmoe_block_forward(const lmoe_dims* dims, const lmoe_weights* weights, const lmoe_block_norms* norms,
                                const uint16_t* x, uint16_t* y, void* ws, size_t ws_bytes, lmoe_stream_t stream);

/* Synchronises `stream`, reads the device status word of `ws` and returns it
 * (LMOE_OK, LMOE_ETIMEOUT or LMOE_EDEVICE_CHECK), or LMOE_ECUDA if the
 * stream itself reports an error.  `ws` is a device pointer. */
LMOE_API int lmoe_status_check(const void* ws, lmoe_stream_t stream);

/* Static description of an error code (never NULL). */
LMOE_API const char* lmoe_error_string(int code);

/* Number of kernel launches the last lmoe_* call on this thread enqueued. */
LMOE_API int lmoe_last_launch_count(void);

/* Name of kernel launch i (0-based) of the last lmoe_* call on this host
 * thread, e.g. "expert_gateup" or "pool_tc_gemm": a static string owned by
 * the library, or NULL when i is out of range. */
LMOE_API const char* lmoe_last_launch_name(int i);

/* Routing without a workspace, for callers that cannot allocate device
 * memory where they run the layer (for example a plugin called from another
 * runtime's enqueue path, where that runtime owns every device allocation, or
 * an embedded runtime with a memory budget fixed at start-up).  The pages
 * have no counterpart: this is a deployment variant of lmoe_route.
 *   Same arguments and outputs as lmoe_route, minus ws/ws_bytes, and the same
 *   dimension rules (LMOE_EINVAL, LMOE_EUNSUPPORTED).  It runs lmoe_route's
 *   CUDA-core routers (fp32 FMA: the one-launch routing up to 16 tokens, the
 *   split-K partials above), so its results are bit-identical to lmoe_route's
 *   wherever lmoe_route runs those too: below 64 tokens, or when n_experts is
 *   not a multiple of 32.  From 64 tokens with n_experts % 32 == 0, lmoe_route
 *   computes the logits on the tensor cores, which sums the same exact fp32
 *   products in another order; the picks then agree except where two logits
 *   lie within that rounding of each other, and the weights agree to fp32
 *   rounding.
 *   Its scratch is a fixed array inside the library (about 1.1 MB, held on
 *   every GPU that loads the library until the process exits), so it accepts
 *   at most T = 64 tokens and n_experts <= 256, and returns LMOE_ENOSCRATCH
 *   beyond that.  It never allocates or frees device memory.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture on the device.
 *   Every call shares the one array and its contents persist between calls:
 *   calls that overlap on the GPU race and must be serialised by the caller.
 *   Device-side check results are not reported (there is no workspace for
 *   lmoe_status_check to read). */
LMOE_API int lmoe_route_noalloc(const lmoe_dims* dims, const uint16_t* x, const float* router_w,
                                const float* router_bias, int32_t* topk_idx, float* topk_w,
                                int32_t* expert_offsets, int32_t* sorted_rows, int32_t* row_pos,
                                lmoe_stream_t stream);

/* Optional per-launch timing: while set, every kernel launch i of the
 * following lmoe_* calls on this host thread is bracketed by
 * cudaEventRecord(events[2i]) before it and cudaEventRecord(events[2i + 1])
 * after it, both on the stream that launch runs on (as far as n allows), so
 * the device time of launch i is the time between events 2i and 2i + 1.
 * Above 16 tokens a call runs its routing launches on a second stream beside
 * the pooler, so events of different launches need not be ordered.
 * `events` holds cudaEvent_t handles owned by the caller; pass n = 0 to switch
 * off.  Recording events between launches serialises the kernels of one
 * stream, so use it only to time kernels. */
LMOE_API int lmoe_profile_events(void* const* events, int n);

/* Regime switches (process-wide; they apply to calls issued after the
 * setter returns).  No counterpart in the pages: they exist so that both
 * implementations of a stage can be run and tested on the same input.
 *
 *  LMOE_OPT_DENSE_MIN_TOKENS: from this many tokens on, the pooler (H -> L)
 *    and the unpooler (L -> H) run as tensor-core GEMMs (tcgen05, 128 x 256
 *    output tiles accumulated in tensor memory); below it, as a
 *    weight-streaming kernel tuned for a few tokens.  Default 64.
 *  LMOE_OPT_EXPERT_TC_MIN_TOKENS: from this many tokens on, the experts run
 *    as grouped tensor-core GEMMs (weights dequantised to bf16 into tensor
 *    memory, up to 160 rows of one expert per group); below it, as the
 *    weight-streaming kernels.  Default 352.
 *  LMOE_OPT_FUSED_MAX_TOKENS: up to this many tokens (at most 8, and at most
 *    64 route rows) the MXFP4 experts run as one persistent launch: gate/up +
 *    SwiGLU, a device-wide hand-off, then down, with the weight stream kept
 *    going across the hand-off; above it (or with value 0), as two
 *    weight-streaming launches.  Default 0 (off: measured no faster).
 *  LMOE_OPT_DOWN_Z_MAX_TOKENS: up to this many tokens (and at most 64 route
 *    rows) the streaming down launch also applies the post-expert norm and
 *    forms the weighted sum z, after a device-wide count of its CTAs; above
 *    it (or with value 0), a separate combine launch does.  The two give
 *    bit-identical z (same arithmetic, same order).  Default 0 (off:
 *    measured no faster than the combine launch).
 *
 * Both implementations of a stage give bf16 (or fp32) of an fp32 sum per
 * output and differ only in the order of that sum.  value <= 0 restores the
 * default (for LMOE_OPT_FUSED_MAX_TOKENS and LMOE_OPT_DOWN_Z_MAX_TOKENS,
 * value < 0 does and 0 switches the in-launch form off).  Returns the
 * previous value, or LMOE_EINVAL for an unknown key. */
enum {
  LMOE_OPT_DENSE_MIN_TOKENS = 1,
  LMOE_OPT_EXPERT_TC_MIN_TOKENS = 2,
  LMOE_OPT_FUSED_MAX_TOKENS = 3,
  LMOE_OPT_DOWN_Z_MAX_TOKENS = 4
};
LMOE_API int lmoe_set_option(int key, int value);

/* Failure-detection self-check: enqueues one kernel whose single thread waits
 * on a barrier that nothing completes, bounded by limit_us microseconds
 * (1 .. 1e6) and an iteration cap, as every device-side wait of the library
 * is; when the wait runs out it records LMOE_ETIMEOUT in the status word of
 * `ws` (which it zeroes first) and returns.  lmoe_status_check(ws) then reports
 * LMOE_ETIMEOUT, and the context stays usable.  ws: device memory of at least
 * 8 bytes, 256-byte aligned. */
LMOE_API int lmoe_selftest_timeout(void* ws, size_t ws_bytes, unsigned limit_us, lmoe_stream_t stream);

/* Format self-check: converts every byte value b (two E2M1 codes, low nibble
 * first) with the same in-register conversion the expert kernels use and
 * writes the two values as fp32 to out[2*b], out[2*b+1] (device pointer,
 * 512 floats).  Synchronous. */
LMOE_API int lmoe_selftest_e2m1(float* out);

/* Format self-check of the grouped tensor-core experts: dequantises block b
 * of 32 E2M1 codes (codes[16b .. 16b+15], low nibble first) with E8M0 scale
 * byte scales[b] exactly as those kernels do and writes the 32 bf16 values to
 * out[32b .. 32b+31].  E2M1 times 2^(s-127) is exact in bf16 for every finite
 * result (OCP MX v1.0; s = 255 gives NaN).  Device pointers; codes and out
 * 16-byte aligned.  Synchronous. */
LMOE_API int lmoe_selftest_dequant_bf16(const uint8_t* codes, const uint8_t* scales, int nblocks, uint16_t* out);

#ifdef __cplusplus
}
#endif

#endif /* LMOE_H */
