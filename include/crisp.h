/*
 * crisp.h -- C ABI of the GB300 (sm_103a) CRISP sparse-prefill attention library.
 *
 * CRISP is described on the analysis page "CRISP: Cliff-awaRe Input-adaptive Sparse
 * Prefilling with Structural-Mass-Motivated Routing" (paper.rainbus.top/paper/2609.01925).
 * Section names below are that page's:
 *   "Method step details"  -- Algorithm 1: PatSearch -> VSIndex | PEIndex -> A(Q,K,V,S),
 *                             with tau_proxy=0.2, gamma=0.95, alpha in {1.0,1.25}, B=128,
 *                             k_min=1024 tokens per direction.
 *   "Core method"          -- step 1 PatSearch and C_struct routing; the noise floor.
 *   "Prerequisites"        -- A(Q,K,V,S) = Softmax(QK^T/sqrt(d) + M_S) V.
 *   "Figures and tables"   -- descriptions of Algorithms 2 (PatSearch), 3 (VSIndex) and
 *                             4 (PEIndex).
 *
 * Conventions for every entry point:
 *   - Q is [batch, hq, n, d], K and V are [batch, hkv, n, d], O is [batch, hq, n, d]; all
 *     bf16, contiguous, head-major, in device memory owned by the caller.  Query head h
 *     uses key/value head h / (hq/hkv) of the same batch entry (GQA).
 *   - Supported shapes: d == 128, n a multiple of 128 with 128 <= n <= 1048576,
 *     hq % hkv == 0, batch*hq <= 65535.  Parameters: B == b == 128,
 *     1 <= w_sink, w_local <= 128, 0 < gamma <= 1, alpha >= 0, k_min_tokens >= 0;
 *     CRISP_FLAG_FORCE_VS and CRISP_FLAG_FORCE_PE are exclusive, and so are
 *     CRISP_FLAG_MEDIAN_FLOOR and CRISP_FLAG_VS_GAMMA_CUMSUM.
 *     Anything else returns CRISP_ERR_INVALID_ARG or CRISP_ERR_UNSUPPORTED before any
 *     work is queued.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Compute entry points
 *     only enqueue work on it and return; they never synchronise.  The *_get, *_set,
 *     *_stats and crisp_sync_status calls synchronise `stream`.
 *   - The context owns every device buffer the path needs (allocated once by
 *     crisp_create for the largest dims it will see) and the current selection.  A
 *     context must not be used from two host threads at once, and work queued with one
 *     context must not overlap on two streams.
 *   - No call aborts, traps or throws.  Argument errors come back synchronously.  Errors
 *     met on the device (a bounded wait that ran out, an index out of range) are latched
 *     in a device error word and reported by the next crisp_sync_status.
 */
#ifndef CRISP_H
#define CRISP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CRISP_OK = 0,
  CRISP_ERR_INVALID_ARG = 1,   /* null pointer, bad shape or parameter             */
  CRISP_ERR_UNSUPPORTED = 2,   /* valid but not implemented (d != 128, B != 128...) */
  CRISP_ERR_NO_MEMORY = 3,     /* device allocation failed                          */
  CRISP_ERR_CUDA = 4,          /* a CUDA runtime call failed (see crisp_last_error)  */
  CRISP_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out                    */
  CRISP_ERR_DEVICE_ASSERT = 6, /* a kernel's range check failed                      */
  CRISP_ERR_NO_SELECTION = 7   /* crisp_attend / *_get before any selection exists  */
} crisp_status;

typedef struct {
  int32_t batch; /* batch entries                        */
  int32_t n;     /* tokens per sequence                  */
  int32_t hq;    /* query heads                          */
  int32_t hkv;   /* key/value heads                      */
  int32_t d;     /* head dimension (128)                 */
} crisp_dims;

/* Method parameters ("Method step details"). */
typedef struct {
  int32_t B;            /* key/query block size (128)                                 */
  int32_t b;            /* proxy queries: the last b rows of Q (128)                   */
  int32_t w_sink;       /* anchor: first w_sink keys (128)                             */
  int32_t w_local;      /* anchor: last w_local keys (128)                             */
  int32_t k_min_tokens; /* minimum VS budget per direction, tokens (1024 = 8 blocks)   */
  float tau_proxy;      /* route VS iff C_struct >= tau_proxy (0.2)                    */
  float alpha;          /* VS: keep blocks with p_d > alpha * mu_d (1.0)               */
  float gamma;          /* PE: cumulative coverage target (0.95)                      */
  uint32_t flags;       /* CRISP_FLAG_*                                                */
} crisp_cfg;

#define CRISP_FLAG_FORCE_VS 0x1u /* route every head VS (C_struct still computed) */
#define CRISP_FLAG_FORCE_PE 0x2u /* route every head PE                          */
/* VS variants ("Limitations" item 6, "Weaknesses" item 4; Table 5 ablation Abl.1): */
#define CRISP_FLAG_MEDIAN_FLOOR 0x4u     /* mu_d = median of p_d[1..N_b-2] instead of the mean */
#define CRISP_FLAG_VS_GAMMA_CUMSUM 0x8u  /* VS blocks by cumulative coverage >= gamma (largest
                                            first, padded to k_min) instead of p_d > alpha*mu_d;
                                            FlexPrefill's budget rule                          */

/* crisp_prefill only: capture the call's launches once as a CUDA graph (on a stream the
 * context owns) and replay it on the caller's stream while the dims, the cfg, Q, K, V, O,
 * the timeout and the debug flags stay the same; any change captures again.  Same kernels
 * and results as the eager call; saves the launch gaps of the ~30 launches (about 0.05 ms
 * per call), which matters at short lengths.  One graph per context. */
#define CRISP_FLAG_GRAPH_REPLAY 0x10u

/* Debug flags for crisp_set_debug. */
#define CRISP_DEBUG_DROP_ARRIVE 0x1u /* attention: skip one barrier arrive in the first
                                        work item so a bounded wait runs out (tests the
                                        timeout path; the kernel still exits cleanly)   */

typedef struct crisp_ctx_s* crisp_ctx;

/* The page's defaults: B=b=128, w_sink=w_local=128, k_min=1024, tau=0.2, alpha=1, gamma=0.95. */
crisp_cfg crisp_cfg_default(void);

/* Allocate a context and all device workspace for problems up to `max_dims` on the
 * current CUDA device.  Returns CRISP_ERR_NO_MEMORY if the workspace does not fit. */
crisp_status crisp_create(const crisp_dims* max_dims, crisp_ctx* out);

/* Free the context and its workspace (synchronises the device first). NULL is a no-op. */
void crisp_destroy(crisp_ctx ctx);

/* Steps 1-3 of Algorithm 1 ("Method step details"; Algorithms 2, 3, 4 under "Figures and
 * tables"): per query head, the proxy attention of the last b queries, C_struct and the
 * VS/PE route; then the VS sink-aware noise-floor selection or the PE pooled
 * gamma-cumsum selection; then the per-query-block key-block lists (CSR, sorted).
 * Reads Q and K; writes only context buffers.  The selection stays in the context. */
crisp_status crisp_select(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                          const crisp_cfg* cfg, void* stream);

/* Step 4 ("Method step details"; "Prerequisites" A(Q,K,V,S)): exact causal softmax
 * attention of every query block over its selected key blocks (token-causal inside the
 * diagonal block), using the context's current selection (from crisp_select or
 * crisp_selection_set with the same dims).  Writes O. */
crisp_status crisp_attend(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                          const void* V, void* O, void* stream);

/* crisp_select followed by crisp_attend: CRISP(Q,K,V) -> O (Algorithm 1). */
crisp_status crisp_prefill(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                           const void* V, const crisp_cfg* cfg, void* O, void* stream);

/* crisp_prefill from host memory, overlapping the copies with the work: the heads are
 * independent ("Method step details" runs steps 1-4 per head), so the call splits them
 * into chunks of whole KV-head groups (at long lengths the first and the last group go
 * one query head per chunk, so that only one head's upload precedes the first
 * computation and one head's download follows the last) and, per chunk, uploads Q, K, V
 * (host -> the caller's device buffers Q, K, V), selects and attends on `stream`, and
 * downloads O (-> O_host) while the next chunk is uploaded and computed.  Two copy streams owned by
 * the context carry the copies; events order them against `stream`, so synchronising
 * `stream` waits for everything, O_host included.  Host buffers should be page-locked
 * (cudaHostAlloc / cudaHostRegister) for the copies to overlap.  All eight buffers are
 * caller-owned and hold the full [batch*heads][n][128] tensors; the call allocates
 * nothing.  Leaves the context without a selection (crisp_attend then returns
 * CRISP_ERR_NO_SELECTION until the next crisp_select); crisp_attend_info reports the
 * last chunk. */
crisp_status crisp_prefill_host(crisp_ctx ctx, const crisp_dims* dims, const void* Q_host,
                                const void* K_host, const void* V_host, const crisp_cfg* cfg,
                                void* O_host, void* Q, void* K, void* V, void* O, void* stream);

/* Dense causal attention with the same kernel and every key block K <= I: the in-library
 * denominator of the speedup ("Prerequisites", FlashAttention).  Writes O; does not touch
 * the selection. */
crisp_status crisp_dense(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                         const void* V, void* O, void* stream);

/* Host copy of the current selection.  Every pointer is caller-owned host memory and may
 * be NULL to skip that field.  H = batch*hq, N_b = n/128. */
typedef struct {
  uint8_t* route_vs;    /* [H]        1 = VS, 0 = PE                                  */
  float* c_struct;      /* [H]        C_struct                                       */
  float* mu;            /* [H][2]     mu_v, mu_s (VS heads; 0 for PE)                 */
  int32_t* counts;      /* [H][4]     VS: c_v, c_s, k_v, k_s (c_d = blocks above the floor,
                                      or the gamma-cumsum cut size with CRISP_FLAG_VS_GAMMA_CUMSUM).
                                      PE: pairs kept by the gamma cut, rescued rows, 0, 0 */
  float* p_v;           /* [H][N_b]   pooled vertical score (all heads)               */
  float* p_s;           /* [H][N_b]   pooled slash score (all heads)                  */
  uint8_t* sel_v;       /* [H][N_b]   S_v membership (VS heads)                        */
  uint8_t* sel_s;       /* [H][N_b]   S_s membership (VS heads)                        */
  int64_t* row_ptr;     /* [H*N_b+1]  CSR row offsets, row = h*N_b + I                 */
  int32_t* col;         /* [col_capacity] key blocks, ascending within a row           */
  int64_t col_capacity; /* in: size of `col` (entries)                                 */
  int64_t nnz;          /* out: number of selected (query block, key block) pairs      */
} crisp_selection_host;

crisp_status crisp_selection_get(crisp_ctx ctx, const crisp_dims* dims, void* stream,
                                 crisp_selection_host* out);

/* Replace the context's selection by a caller-supplied CSR (host arrays, H*N_b+1 row
 * offsets and nnz key blocks).  Each row must be strictly ascending with entries in
 * [0, I]; rows must be non-empty.  Checked on the host: CRISP_ERR_INVALID_ARG otherwise. */
crisp_status crisp_selection_set(crisp_ctx ctx, const crisp_dims* dims, void* stream,
                                 const int64_t* row_ptr, const int32_t* col, int64_t nnz);

typedef struct {
  int64_t nnz;         /* selected block pairs over all heads                          */
  int64_t rows;        /* query-block rows (H*N_b)                                      */
  int64_t max_row;     /* longest row                                                    */
  int64_t pe_rescued;  /* PE rows whose only block is the forced diagonal               */
  int32_t n_vs;        /* heads routed VS                                                */
  int32_t n_pe;        /* heads routed PE                                                */
  /* Near-threshold items, counted on the device: decisions that a relative change of
   * 1e-3 in the deciding score could flip.  Routes: |C_struct - tau| <= 1e-3 tau.  VS
   * blocks (both directions of every VS head): |p_d[J] - alpha mu_d| <= 1e-3 alpha mu_d,
   * or, when the k_min padding applies (or CRISP_FLAG_VS_GAMMA_CUMSUM), within 1e-3 of
   * the smallest kept score.  PE pairs: |v - v*| <= 1e-3 v*, v* the gamma cut's value
   * (0 for a head whose scores sum to less than gamma: the cut then keeps everything).  They describe the last
   * crisp_select (or crisp_prefill); crisp_selection_set leaves them as they were. */
  int32_t near_routes;
  int64_t near_vs_blocks;
  int64_t near_pe_pairs;
} crisp_stats;

crisp_status crisp_selection_stats(crisp_ctx ctx, const crisp_dims* dims, void* stream,
                                   crisp_stats* out);

/* Diagnostic: FlexPrefill's JSD routing signal, which CRISP's C_struct replaces
 * ("Prerequisites", JSD; "Motivation").  For each query head, D_JS = 1/2 KL(a_hat || m) +
 * 1/2 KL(a_bar || m), m = (a_hat + a_bar)/2, where a_hat is the pooled proxy attention
 * p_v of the preceding crisp_select on the same Q/K (the "softmax, then average"
 * distribution over key blocks) and a_bar is the softmax over key blocks of
 * (mean of the last 128 queries) . (block mean of the keys) / sqrt(d) ("pool, then
 * softmax").  Writes, in caller-owned device memory, d_js[H] (float, nats) and
 * route_vs[H] (1 iff D_JS >= tau_jsd; the pages give no value for tau_jsd).  Returns
 * CRISP_ERR_NO_SELECTION unless the context's last call was crisp_select / crisp_prefill
 * with these dims.  Enqueues work on `stream` only. */
crisp_status crisp_jsd(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                       float tau_jsd, float* d_js, uint8_t* route_vs, void* stream);

/* Synchronise `stream`, then write to *rows the number of query-block rows the last
 * crisp_attend / crisp_dense on this context recomputed in its rescue pass.  The attention
 * kernel exponentiates every row against one reference (the larger of two first-block row
 * maxima); a row with a logit more than 64 log2-units above it is recomputed with running
 * maxima ("Prerequisites": exact softmax attention either way).  Normally 0. */
crisp_status crisp_attend_info(crisp_ctx ctx, void* stream, int64_t* rows);

/* Number of kernel launches one crisp_prefill enqueues for `dims` on a GPU with `num_sms`
 * SMs: selection 7 for N_b = n/128 <= 256, else 20 or 21 (PatSearch and the route 2 or
 * 4; PEIndex: block means 1, pooled softmax 1, the gamma cut 1 or 12; CSR 2 for at most
 * 32768 query-block rows over all heads, else 3), the attention work order (1 for at most
 * 16384 query-block rows, else 3), the fast attention kernel once per group of KV heads,
 * and the rescue pass once.  Host-only arithmetic (no context, no CUDA call); 0 for dims
 * the library does not support. */
int32_t crisp_prefill_launches(const crisp_dims* dims, int32_t num_sms);

/* Synchronise `stream`, then report and clear the device error word: CRISP_OK,
 * CRISP_ERR_TIMEOUT or CRISP_ERR_DEVICE_ASSERT, or CRISP_ERR_CUDA if the stream itself
 * reports a CUDA error. */
crisp_status crisp_sync_status(crisp_ctx ctx, void* stream);

/* Debug controls: CRISP_DEBUG_* flags and the bounded-wait limit in nanoseconds
 * (0 = default, one second). */
crisp_status crisp_set_debug(crisp_ctx ctx, uint32_t flags, uint64_t timeout_ns);

const char* crisp_status_string(crisp_status s);

/* Routing with no device allocation.  The CRISP paper has no counterpart to this call:
 * it exists for callers that cannot call cudaMalloc -- for example a plug-in inside an
 * engine that owns all device memory through its own pool, or a latency-critical loop
 * that cannot afford the device synchronisation an allocation implies.
 *
 * Computes what the routing part of crisp_select computes (the proxy attention of the
 * last 128 queries, C_struct and the VS/PE decision) and writes, in caller-owned device
 * memory: route_vs[H] (1 = VS, 0 = PE), c_struct[H] (float) and status[0] (a uint32
 * word: 0 on success, nonzero when a bounded wait ran out or a range check failed),
 * with H = batch*hq.  Only enqueues work on `stream`; read the outputs after
 * synchronising it.
 *
 * Scratch is a fixed array in the library's device memory (about 15 MB on every GPU
 * that loads the library, held until the process exits).  Limits: batch*hq <= 128 and
 * batch*hq*(n/128) <= 8192; larger problems return CRISP_ERR_UNSUPPORTED before any work
 * is queued.  Other shape and parameter rules are those of crisp_select.  The first call
 * on a device resolves the array's device address and sets kernel attributes; make
 * that first call before any stream capture.  Every call shares the one array, so calls
 * whose work overlaps on the GPU (two streams, or two host threads) race and give
 * undefined results: serialise them. */
crisp_status crisp_route_static(const crisp_dims* dims, const void* Q, const void* K,
                                const crisp_cfg* cfg, uint8_t* route_vs, float* c_struct,
                                uint32_t* status, void* stream);

/* Text of the last CUDA error seen by this context ("" if none). */
const char* crisp_last_error(crisp_ctx ctx);

#ifdef __cplusplus
}
#endif
#endif /* CRISP_H */
