// internal.h -- context layout and kernel launchers shared by the library's translation
// units.  Not part of the public ABI (include/crisp.h is).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "crisp.h"

#include <nvtx3/nvToolsExt.h>

namespace crisp {

constexpr int kD = 128;        // head dimension
constexpr int kBlk = 128;      // block size B = proxy rows b
constexpr int kTileBytes = kBlk * kD * 2;  // one 128 x 128 bf16 tile

// Masses of the PE gamma cut (bin masses, running sums, the target) are fixed point in
// units of 2^-56: the probabilities v are >= 0 and a head's triangle sums to 1 (each row of
// the pooled softmax sums to 1, scaled by 1/N_b), so every sum fits in 64 bits and adds
// exactly, and the digit picks run on integer adds instead of fp64 (slow on this GPU).
// An fp32 partial sum of v is rounded once, to 2^-56, when it enters the histogram.

// Radix-select state of one PE head's gamma cut (device).
struct PeState {
  uint32_t prefix;          // decided high bits of the threshold
  uint32_t decided;         // mask of decided bits
  unsigned long long above;  // mass of items strictly above the decided range (fixed point)
  uint32_t thresh;          // threshold bit pattern (after the last pass)
  uint32_t select_all;      // 1: the whole triangle is taken
  unsigned long long need_eq;   // items equal to thresh to take, in flat order
  unsigned long long count_eq;  // items equal to thresh
};

// CTAs per head that merge PatSearch's per-tile row statistics (patsearch.cu).
constexpr int kRowSplit = 16;
// Work-order bins of the attention's short rows per launch (length classes x query-block
// bands, attention.cu); the workspace sizes the order histogram with them.
constexpr int kOrderShortBins = 256;
struct Workspace {
  // PatSearch per-tile statistics, [H][nb][128] each (log2 domain max, sums under it)
  float* st_m = nullptr;
  float* st_u = nullptr;   // keys on or left of the row's diagonal offset (slash block N_b-1-t)
  float* st_w = nullptr;   // keys right of it (slash block N_b-2-t)
  float* anc = nullptr;    // [H][2][128] anchor partial sums (tile 0, tile N_b-1)
  float* rowM = nullptr;   // [H][128]
  float* rowZ = nullptr;   // [H][128]
  float2* row_part = nullptr;  // [H][kRowSplit][128] per-CTA (max, sum) partials of the row statistics
  int* row_ticket = nullptr;   // [H] CTAs done per head (zero between launches)
  float* pv = nullptr;     // [H][nb] pooled vertical score
  float* pshi = nullptr;   // [H][nb] slash contribution of tile t to block N_b-1-t
  float* pslo = nullptr;   // [H][nb] slash contribution of tile t to block N_b-2-t
  float* ps = nullptr;     // [H][nb] pooled slash score
  float* cstruct = nullptr;  // [H]
  uint8_t* route = nullptr;  // [H] 1 = VS
  float* mu = nullptr;       // [H][2]
  int32_t* counts = nullptr; // [H][4]
  int32_t* near = nullptr;   // [H][3] near-threshold route, VS blocks, PE pairs (crisp_stats)
  uint8_t* selv = nullptr;   // [H][nb]
  uint8_t* sels = nullptr;   // [H][nb]
  // VS heads: S_v as bits (bit x of word x/32 = block x), then S_s reversed as bits
  // (bit x = slash block N_b-1-x, one spare word), [H][2*nbw+1] (patsearch.cu -> csr.cu)
  uint32_t* selbits = nullptr;
  // PEIndex
  uint16_t* qs = nullptr;    // [2][H*nb][128] bf16: Qbar * log2(e)/sqrt(d) as hi rows, then lo rows
  uint16_t* ks = nullptr;    // [2][Hkv*nb][128] bf16: Kbar as hi rows, then lo rows
  float* kbar = nullptr;     // [Hkv][nb][128] fp32 (JSD routing)
  float* pev = nullptr;      // [H][nb][nb] v = A_bar / N_b (lower triangle)
  unsigned long long* hist_cnt = nullptr;  // [H][256]
  unsigned long long* hist_mass = nullptr; // [H][256], fixed point (2^-56 units)
  PeState* pe = nullptr;                   // [H]
  int* pe_list = nullptr;                  // [H + 1]: count of PE heads, then the heads
  int64_t* eq_off = nullptr;               // [H][nb+1]
  // per-row block masks and CSR
  uint32_t* rowmask = nullptr;  // [H][nb][nbw]
  int64_t* scan_blk = nullptr;  // [ceil(H*nb/1024)] per-1024-row totals, then offsets
  int64_t* row_ptr = nullptr;   // [H*nb+1]
  int32_t* col = nullptr;       // [col_cap]
  int64_t col_cap = 0;
  // attention work order: rows sorted by descending length (counting sort)
  int32_t* order = nullptr;     // [H*nb]
  int32_t* len_hist = nullptr;  // [Hkv*(nb+1+kOrderShortBins)] histogram of the work-order keys, then cursors
  // rows the fast attention pass hands to the rescue pass (see attention.cu)
  int32_t* redo = nullptr;      // [H*nb]
  int* redo_count = nullptr;
  int* work_ctr = nullptr;      // [Hkv] per-launch item counters of the fast attention pass
  uint32_t* err = nullptr;      // device error word
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// What a captured crisp_prefill graph depends on (compared bytewise; zero-filled first).
struct GraphKey {
  crisp_dims dims;
  crisp_cfg cfg;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  uint64_t timeout_ns;
  uint32_t debug_flags;
};

// Shapes of one call, flattened: H = batch*hq query heads, Hkv = batch*hkv.
struct Shape {
  int n, nb, nbw, H, Hkv, hq, hkv, group;
};

}  // namespace crisp

struct crisp_ctx_s {
  int device = 0;
  int num_sms = 0;
  crisp_dims maxd{};
  int64_t max_H = 0, max_Hkv = 0, max_nb = 0, max_nbw = 0;
  crisp::Workspace ws;
  crisp::EncodeTiledFn encode = nullptr;
  bool has_sel = false;
  bool has_patsearch = false;  // workspace p_v belongs to the current selection
  crisp_dims sel_dims{};
  uint32_t debug_flags = 0;
  uint64_t timeout_ns = 1000000000ull;
  // crisp_prefill_host: copy streams and the events that order them against the caller's
  // stream (created with the context).
  static constexpr int kMaxChunks = 64;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_entry = nullptr, ev_done = nullptr;
  cudaEvent_t ev_in[kMaxChunks] = {}, ev_out[kMaxChunks] = {};
  // crisp_prefill with CRISP_FLAG_GRAPH_REPLAY: capture stream and the last call's graph.
  cudaStream_t cap = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  crisp::GraphKey graph_key{};
  char last_err[256] = {0};
};

namespace crisp {

Shape make_shape(const crisp_dims& d);

// An NVTX range in the library's "crisp" domain for the launches of one phase (PatSearch,
// VS, PE, CSR, work order, attention); costs nothing unless a profiler is attached.
class PhaseRange {
 public:
  explicit PhaseRange(const char* name) {
    nvtxEventAttributes_t ev = {};
    ev.version = NVTX_VERSION;
    ev.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    ev.messageType = NVTX_MESSAGE_TYPE_ASCII;
    ev.message.ascii = name;
    nvtxDomainRangePushEx(domain(), &ev);
  }
  ~PhaseRange() { nvtxDomainRangePop(domain()); }
  PhaseRange(const PhaseRange&) = delete;
  PhaseRange& operator=(const PhaseRange&) = delete;

 private:
  static nvtxDomainHandle_t domain() {
    static nvtxDomainHandle_t d = nvtxDomainCreateA("crisp");
    return d;
  }
};
// The shape and parameter rules of include/crisp.h (CRISP_OK, CRISP_ERR_INVALID_ARG or
// CRISP_ERR_UNSUPPORTED); host only.
crisp_status check_dims(const crisp_dims* d);
crisp_status check_cfg(const crisp_cfg* c);

// Each launcher only enqueues work on `st` and returns the launch status.
cudaError_t launch_patsearch(crisp_ctx ctx, const Shape& s, const crisp_cfg& cfg,
                             const CUtensorMap& tmQ, const CUtensorMap& tmK, cudaStream_t st);
// tmQs/tmKs: 3-D maps (see make_map3) of ws.qs and ws.ks with 2*H*nb and 2*Hkv*nb rows;
// tmO: fp32 map of ws.pev, dims {nb, nb, H}, box {16, 32, 1}, 64-byte swizzle, valid when
// tma_out (nb % 4 == 0).
cudaError_t launch_pe_index(crisp_ctx ctx, const Shape& s, const crisp_cfg& cfg, const void* Q,
                            const void* K, const CUtensorMap& tmQs, const CUtensorMap& tmKs,
                            const CUtensorMap& tmO, bool tma_out, cudaStream_t st);
cudaError_t launch_build_csr(crisp_ctx ctx, const Shape& s, cudaStream_t st);
// Launches of PatSearch and the route (2 for short sequences, else 4).
int patsearch_launches(int nb);
// Launches of the PE gamma cut after the pooled softmax (1 for short sequences, else 12).
int pe_select_launches(int nb);
// KV heads per launch of the fast attention kernel (launch_attention splits the heads).
int attention_kv_heads_per_launch(const Shape& s, int num_sms);
// Launches of the attention work order (1 for short sequences, else 3).
int order_launches(const Shape& s, int num_sms);
int csr_launches(int64_t rows);
// tmQ/tmK/tmV: 3-D maps of Q, K, V (dims {64, rows, 2}, box {64, 128, 2}; see make_map3).
cudaError_t launch_attention(crisp_ctx ctx, const Shape& s, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, void* O, bool dense,
                             cudaStream_t st);
cudaError_t launch_jsd(crisp_ctx ctx, const Shape& s, const void* Q, const void* K, float tau,
                       float* d_js, uint8_t* route, cudaStream_t st);

}  // namespace crisp
