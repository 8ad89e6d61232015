// api.cu -- the C ABI (include/crisp.h): context and workspace, argument validation,
// TMA tensor maps, and the launch sequence of the CRISP path.  Host code only; every
// step of the path runs in the library's kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <vector>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace crisp {
cudaError_t init_patsearch_attributes();
cudaError_t init_attention_attributes();
cudaError_t init_pe_attributes();
}  // namespace crisp

using namespace crisp;

namespace {

void set_err(crisp_ctx ctx, const char* what, cudaError_t e) {
  if (ctx) snprintf(ctx->last_err, sizeof(ctx->last_err), "%s: %s", what, cudaGetErrorString(e));
}

bool dims_valid(const crisp_dims* d) {
  return d && d->batch >= 1 && d->n >= 1 && d->hq >= 1 && d->hkv >= 1 && d->d >= 1 &&
         d->hq % d->hkv == 0;
}

}  // namespace

namespace crisp {

crisp_status check_dims(const crisp_dims* d) {
  if (!dims_valid(d)) return CRISP_ERR_INVALID_ARG;
  if (d->d != kD) return CRISP_ERR_UNSUPPORTED;
  if (d->n % kBlk != 0 || d->n < kBlk || d->n > (1 << 20)) return CRISP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->batch) * d->hq > 65535) return CRISP_ERR_UNSUPPORTED;
  return CRISP_OK;
}

crisp_status check_cfg(const crisp_cfg* c) {
  if (!c) return CRISP_ERR_INVALID_ARG;
  if (c->B != kBlk || c->b != kBlk) return CRISP_ERR_UNSUPPORTED;
  if (c->w_sink < 1 || c->w_sink > kBlk || c->w_local < 1 || c->w_local > kBlk)
    return CRISP_ERR_UNSUPPORTED;
  if (!(c->gamma > 0.f && c->gamma <= 1.f)) return CRISP_ERR_INVALID_ARG;
  if (!(c->alpha >= 0.f) || c->k_min_tokens < 0) return CRISP_ERR_INVALID_ARG;
  if (!(c->tau_proxy == c->tau_proxy)) return CRISP_ERR_INVALID_ARG;
  if ((c->flags & CRISP_FLAG_FORCE_VS) && (c->flags & CRISP_FLAG_FORCE_PE))
    return CRISP_ERR_INVALID_ARG;
  if ((c->flags & CRISP_FLAG_MEDIAN_FLOOR) && (c->flags & CRISP_FLAG_VS_GAMMA_CUMSUM))
    return CRISP_ERR_INVALID_ARG;
  return CRISP_OK;
}

}  // namespace crisp

namespace {

bool fits(const crisp_ctx ctx, const crisp_dims* d) {
  const int64_t H = static_cast<int64_t>(d->batch) * d->hq;
  const int64_t Hkv = static_cast<int64_t>(d->batch) * d->hkv;
  return H <= ctx->max_H && Hkv <= ctx->max_Hkv && d->n / kBlk <= ctx->max_nb &&
         H * (d->n / kBlk) <= ctx->max_H * ctx->max_nb;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

crisp_status make_map(crisp_ctx ctx, CUtensorMap* map, const void* base, int64_t rows) {
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(kD) * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                           gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(ctx->last_err, sizeof(ctx->last_err), "cuTensorMapEncodeTiled failed (%d)",
             static_cast<int>(r));
    return CRISP_ERR_CUDA;
  }
  return CRISP_OK;
}

// The attention kernels' map: the same [rows][128] bf16 tensor seen as {64 columns, rows,
// 2 column halves} (strides 256 B and 128 B), box {64, 128, 2}: one copy per 128 x 128
// tile, landing in the two-region swizzled layout (see ptx.cuh).
crisp_status make_map3(crisp_ctx ctx, CUtensorMap* map, const void* base, int64_t rows) {
  cuuint64_t gdim[3] = {64, static_cast<cuuint64_t>(rows), 2};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(kD) * 2, 128};
  cuuint32_t box[3] = {64, 128, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                           gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(ctx->last_err, sizeof(ctx->last_err), "cuTensorMapEncodeTiled (3-D) failed (%d)",
             static_cast<int>(r));
    return CRISP_ERR_CUDA;
  }
  return CRISP_OK;
}

// The PE probability triangle v as an fp32 tensor {nb keys, nb rows, H heads} (row pitch
// nb * 4 bytes, a multiple of 16 when nb % 4 == 0), stored in boxes of 16 keys x 32 rows
// from a 64-byte swizzled shared-memory tile.
crisp_status make_prob_map(crisp_ctx ctx, CUtensorMap* map, const void* base, int64_t nb,
                           int64_t heads) {
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(nb),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(nb) * 4, static_cast<cuuint64_t>(nb * nb) * 4};
  cuuint32_t box[3] = {16, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
                           gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(ctx->last_err, sizeof(ctx->last_err), "cuTensorMapEncodeTiled (fp32) failed (%d)",
             static_cast<int>(r));
    return CRISP_ERR_CUDA;
  }
  return CRISP_OK;
}

crisp_status launched(crisp_ctx ctx, cudaError_t e, const char* what) {
  if (e == cudaSuccess) return CRISP_OK;
  set_err(ctx, what, e);
  return CRISP_ERR_CUDA;
}

crisp_status check_common(crisp_ctx ctx, const crisp_dims* dims) {
  if (!ctx) return CRISP_ERR_INVALID_ARG;
  crisp_status st = check_dims(dims);
  if (st != CRISP_OK) return st;
  if (!fits(ctx, dims)) return CRISP_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != ctx->device) return CRISP_ERR_INVALID_ARG;
  return CRISP_OK;
}

bool create_copy_streams(crisp_ctx ctx) {
  const unsigned f = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&ctx->h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->d2h, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->cap, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->ev_entry, f) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->ev_done, f) != cudaSuccess)
    return false;
  for (int c = 0; c < crisp_ctx_s::kMaxChunks; ++c)
    if (cudaEventCreateWithFlags(&ctx->ev_in[c], f) != cudaSuccess ||
        cudaEventCreateWithFlags(&ctx->ev_out[c], f) != cudaSuccess)
      return false;
  return true;
}

void destroy_copy_streams(crisp_ctx ctx) {
  for (int c = 0; c < crisp_ctx_s::kMaxChunks; ++c) {
    if (ctx->ev_in[c]) cudaEventDestroy(ctx->ev_in[c]);
    if (ctx->ev_out[c]) cudaEventDestroy(ctx->ev_out[c]);
  }
  if (ctx->ev_entry) cudaEventDestroy(ctx->ev_entry);
  if (ctx->ev_done) cudaEventDestroy(ctx->ev_done);
  if (ctx->h2d) cudaStreamDestroy(ctx->h2d);
  if (ctx->d2h) cudaStreamDestroy(ctx->d2h);
  if (ctx->graph_exec) cudaGraphExecDestroy(ctx->graph_exec);
  if (ctx->cap) cudaStreamDestroy(ctx->cap);
  cudaGetLastError();
}

}  // namespace

namespace crisp {
Shape make_shape(const crisp_dims& d) {
  Shape s;
  s.n = d.n;
  s.nb = d.n / kBlk;
  s.nbw = (s.nb + 31) / 32;
  s.H = d.batch * d.hq;
  s.Hkv = d.batch * d.hkv;
  s.hq = d.hq;
  s.hkv = d.hkv;
  s.group = d.hq / d.hkv;
  return s;
}
}  // namespace crisp

extern "C" {

crisp_cfg crisp_cfg_default(void) {
  crisp_cfg c;
  c.B = 128;
  c.b = 128;
  c.w_sink = 128;
  c.w_local = 128;
  c.k_min_tokens = 1024;
  c.tau_proxy = 0.2f;
  c.alpha = 1.0f;
  c.gamma = 0.95f;
  c.flags = 0;
  return c;
}

const char* crisp_status_string(crisp_status s) {
  switch (s) {
    case CRISP_OK: return "ok";
    case CRISP_ERR_INVALID_ARG: return "invalid argument";
    case CRISP_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case CRISP_ERR_NO_MEMORY: return "device allocation failed";
    case CRISP_ERR_CUDA: return "CUDA error";
    case CRISP_ERR_TIMEOUT: return "device wait timed out";
    case CRISP_ERR_DEVICE_ASSERT: return "device range check failed";
    case CRISP_ERR_NO_SELECTION: return "no selection for these dims";
  }
  return "unknown status";
}

crisp_status crisp_create(const crisp_dims* max_dims, crisp_ctx* out) {
  if (!out) return CRISP_ERR_INVALID_ARG;
  *out = nullptr;
  crisp_status st = check_dims(max_dims);
  if (st != CRISP_OK) return st;
  crisp_ctx ctx = new (std::nothrow) crisp_ctx_s();
  if (!ctx) return CRISP_ERR_NO_MEMORY;
  if (cudaGetDevice(&ctx->device) != cudaSuccess) {
    delete ctx;
    return CRISP_ERR_CUDA;
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, ctx->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, ctx->device);
  cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
  if (major != 10 || minor != 3) {  // the kernels are built for sm_103a only
    delete ctx;
    return CRISP_ERR_UNSUPPORTED;
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    delete ctx;
    return CRISP_ERR_CUDA;
  }
  ctx->encode = reinterpret_cast<EncodeTiledFn>(fn);
  if (init_patsearch_attributes() != cudaSuccess || init_attention_attributes() != cudaSuccess ||
      init_pe_attributes() != cudaSuccess) {
    delete ctx;
    return CRISP_ERR_CUDA;
  }
  ctx->maxd = *max_dims;
  const int64_t H = static_cast<int64_t>(max_dims->batch) * max_dims->hq;
  const int64_t Hkv = static_cast<int64_t>(max_dims->batch) * max_dims->hkv;
  const int64_t nb = max_dims->n / kBlk;
  const int64_t nbw = (nb + 31) / 32;
  ctx->max_H = H;
  ctx->max_Hkv = Hkv;
  ctx->max_nb = nb;
  ctx->max_nbw = nbw;

  // One allocation, carved into 256-byte aligned pieces.
  struct Piece {
    void** p;
    size_t bytes;
  };
  Workspace& w = ctx->ws;
  w.col_cap = H * nb * (nb + 1) / 2;
  std::vector<Piece> pieces = {
      {reinterpret_cast<void**>(&w.st_m), sizeof(float) * H * nb * kBlk},
      {reinterpret_cast<void**>(&w.st_u), sizeof(float) * H * nb * kBlk},
      {reinterpret_cast<void**>(&w.st_w), sizeof(float) * H * nb * kBlk},
      {reinterpret_cast<void**>(&w.anc), sizeof(float) * H * 2 * kBlk},
      {reinterpret_cast<void**>(&w.rowM), sizeof(float) * H * kBlk},
      {reinterpret_cast<void**>(&w.rowZ), sizeof(float) * H * kBlk},
      {reinterpret_cast<void**>(&w.row_part), sizeof(float2) * H * kRowSplit * kBlk},
      {reinterpret_cast<void**>(&w.row_ticket), sizeof(int) * H},
      {reinterpret_cast<void**>(&w.pv), sizeof(float) * H * nb},
      {reinterpret_cast<void**>(&w.pshi), sizeof(float) * H * nb},
      {reinterpret_cast<void**>(&w.pslo), sizeof(float) * H * nb},
      {reinterpret_cast<void**>(&w.ps), sizeof(float) * H * nb},
      {reinterpret_cast<void**>(&w.cstruct), sizeof(float) * H},
      {reinterpret_cast<void**>(&w.route), static_cast<size_t>(H)},
      {reinterpret_cast<void**>(&w.mu), sizeof(float) * H * 2},
      {reinterpret_cast<void**>(&w.counts), sizeof(int32_t) * H * 4},
      {reinterpret_cast<void**>(&w.near), sizeof(int32_t) * H * 3},
      {reinterpret_cast<void**>(&w.selv), static_cast<size_t>(H * nb)},
      {reinterpret_cast<void**>(&w.sels), static_cast<size_t>(H * nb)},
      {reinterpret_cast<void**>(&w.selbits), sizeof(uint32_t) * H * (2 * nbw + 1)},
      {reinterpret_cast<void**>(&w.qs), sizeof(uint16_t) * 2 * H * nb * kD},
      {reinterpret_cast<void**>(&w.ks), sizeof(uint16_t) * 2 * Hkv * nb * kD},
      {reinterpret_cast<void**>(&w.kbar), sizeof(float) * Hkv * nb * kD},
      {reinterpret_cast<void**>(&w.pev), sizeof(float) * H * nb * nb},
      {reinterpret_cast<void**>(&w.hist_cnt), sizeof(unsigned long long) * H * 256},
      {reinterpret_cast<void**>(&w.hist_mass), sizeof(unsigned long long) * H * 256},
      {reinterpret_cast<void**>(&w.pe), sizeof(PeState) * H},
      {reinterpret_cast<void**>(&w.pe_list), sizeof(int) * (H + 1)},
      {reinterpret_cast<void**>(&w.eq_off), sizeof(int64_t) * H * (nb + 1)},
      {reinterpret_cast<void**>(&w.rowmask), sizeof(uint32_t) * H * nb * nbw},
      {reinterpret_cast<void**>(&w.scan_blk), sizeof(int64_t) * ((H * nb + 1023) / 1024 + 1)},
      {reinterpret_cast<void**>(&w.row_ptr), sizeof(int64_t) * (H * nb + 1)},
      {reinterpret_cast<void**>(&w.col), sizeof(int32_t) * w.col_cap},
      {reinterpret_cast<void**>(&w.order), sizeof(int32_t) * H * nb},
      {reinterpret_cast<void**>(&w.len_hist), sizeof(int32_t) * (Hkv * (nb + 1 + kOrderShortBins) + 2)},
      {reinterpret_cast<void**>(&w.redo), sizeof(int32_t) * H * nb},
      {reinterpret_cast<void**>(&w.redo_count), sizeof(int)},
      {reinterpret_cast<void**>(&w.work_ctr), sizeof(int) * Hkv},
      {reinterpret_cast<void**>(&w.err), sizeof(uint32_t)},
  };
  size_t total = 0;
  for (auto& pc : pieces) total += (pc.bytes + 255) & ~static_cast<size_t>(255);
  void* base = nullptr;
  if (cudaMalloc(&base, total) != cudaSuccess) {
    cudaGetLastError();
    delete ctx;
    return CRISP_ERR_NO_MEMORY;
  }
  size_t off = 0;
  for (auto& pc : pieces) {
    *pc.p = static_cast<char*>(base) + off;
    off += (pc.bytes + 255) & ~static_cast<size_t>(255);
  }
  if (cudaMemset(w.err, 0, sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(w.redo_count, 0, sizeof(int)) != cudaSuccess ||
      cudaMemset(w.row_ticket, 0, sizeof(int) * H) != cudaSuccess || !create_copy_streams(ctx)) {
    destroy_copy_streams(ctx);
    cudaFree(base);
    delete ctx;
    return CRISP_ERR_CUDA;
  }
  *out = ctx;
  return CRISP_OK;
}

void crisp_destroy(crisp_ctx ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  destroy_copy_streams(ctx);
  cudaFree(ctx->ws.st_m);  // the first piece is the allocation's base
  delete ctx;
}

crisp_status crisp_select(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                          const crisp_cfg* cfg, void* stream) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if ((st = check_cfg(cfg)) != CRISP_OK) return st;
  if (!Q || !K || !aligned16(Q) || !aligned16(K)) return CRISP_ERR_INVALID_ARG;
  const Shape s = make_shape(*dims);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  CUtensorMap tmQ, tmK;
  if ((st = make_map(ctx, &tmQ, Q, static_cast<int64_t>(s.H) * s.n)) != CRISP_OK) return st;
  if ((st = make_map(ctx, &tmK, K, static_cast<int64_t>(s.Hkv) * s.n)) != CRISP_OK) return st;
  ctx->has_sel = false;
  ctx->has_patsearch = false;
  if ((st = launched(ctx, launch_patsearch(ctx, s, *cfg, tmQ, tmK, cs), "patsearch")) != CRISP_OK)
    return st;
  CUtensorMap tmQs, tmKs;
  if ((st = make_map3(ctx, &tmQs, ctx->ws.qs, 2 * static_cast<int64_t>(s.H) * s.nb)) != CRISP_OK ||
      (st = make_map3(ctx, &tmKs, ctx->ws.ks, 2 * static_cast<int64_t>(s.Hkv) * s.nb)) != CRISP_OK)
    return st;
  CUtensorMap tmO;
  memset(&tmO, 0, sizeof(tmO));
  const bool tma_out = (s.nb % 4) == 0;
  if (tma_out && (st = make_prob_map(ctx, &tmO, ctx->ws.pev, s.nb, s.H)) != CRISP_OK) return st;
  {
    PhaseRange r("PE");
    if ((st = launched(ctx, launch_pe_index(ctx, s, *cfg, Q, K, tmQs, tmKs, tmO, tma_out, cs),
                       "pe_index")) != CRISP_OK)
      return st;
  }
  {
    PhaseRange r("CSR");
    if ((st = launched(ctx, launch_build_csr(ctx, s, cs), "build_csr")) != CRISP_OK) return st;
  }
  ctx->has_sel = true;
  ctx->has_patsearch = true;
  ctx->sel_dims = *dims;
  return CRISP_OK;
}

static bool same_dims(const crisp_dims& a, const crisp_dims& b) {
  return a.batch == b.batch && a.n == b.n && a.hq == b.hq && a.hkv == b.hkv && a.d == b.d;
}

static crisp_status run_attention(crisp_ctx ctx, const crisp_dims* dims, const void* Q,
                                  const void* K, const void* V, void* O, bool dense,
                                  void* stream) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if (!Q || !K || !V || !O || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
    return CRISP_ERR_INVALID_ARG;
  if (!dense && (!ctx->has_sel || !same_dims(ctx->sel_dims, *dims))) return CRISP_ERR_NO_SELECTION;
  const Shape s = make_shape(*dims);
  CUtensorMap tmQ, tmK, tmV;
  if ((st = make_map3(ctx, &tmQ, Q, static_cast<int64_t>(s.H) * s.n)) != CRISP_OK) return st;
  if ((st = make_map3(ctx, &tmK, K, static_cast<int64_t>(s.Hkv) * s.n)) != CRISP_OK) return st;
  if ((st = make_map3(ctx, &tmV, V, static_cast<int64_t>(s.Hkv) * s.n)) != CRISP_OK) return st;
  return launched(ctx,
                  launch_attention(ctx, s, tmQ, tmK, tmV, O, dense, static_cast<cudaStream_t>(stream)),
                  "attention");
}

crisp_status crisp_attend(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                          const void* V, void* O, void* stream) {
  return run_attention(ctx, dims, Q, K, V, O, false, stream);
}

crisp_status crisp_dense(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                         const void* V, void* O, void* stream) {
  return run_attention(ctx, dims, Q, K, V, O, true, stream);
}

// crisp_prefill with CRISP_FLAG_GRAPH_REPLAY: capture select + attend on the context's own
// stream (the caller's may be the legacy default stream, which cannot be captured), keep
// the executable graph, and launch it on the caller's stream.
static crisp_status prefill_replay(crisp_ctx ctx, const crisp_dims* dims, const void* Q,
                                   const void* K, const void* V, const crisp_cfg* cfg, void* O,
                                   void* stream) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if ((st = check_cfg(cfg)) != CRISP_OK) return st;
  GraphKey key;
  memset(&key, 0, sizeof(key));
  key.dims = *dims;
  key.cfg = *cfg;
  key.q = Q;
  key.k = K;
  key.v = V;
  key.o = O;
  key.timeout_ns = ctx->timeout_ns;
  key.debug_flags = ctx->debug_flags;
  if (!ctx->graph_exec || memcmp(&key, &ctx->graph_key, sizeof(key)) != 0) {
    if (ctx->graph_exec) {
      cudaGraphExecDestroy(ctx->graph_exec);
      ctx->graph_exec = nullptr;
    }
    crisp_cfg eager = *cfg;
    eager.flags &= ~CRISP_FLAG_GRAPH_REPLAY;
    cudaError_t e = cudaStreamBeginCapture(ctx->cap, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
      set_err(ctx, "cudaStreamBeginCapture", e);
      return CRISP_ERR_CUDA;
    }
    st = crisp_select(ctx, dims, Q, K, &eager, ctx->cap);
    if (st == CRISP_OK) st = crisp_attend(ctx, dims, Q, K, V, O, ctx->cap);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(ctx->cap, &g);
    if (st == CRISP_OK && (e != cudaSuccess || !g)) {
      set_err(ctx, "cudaStreamEndCapture", e);
      st = CRISP_ERR_CUDA;
    }
    if (st == CRISP_OK) {
      e = cudaGraphInstantiate(&ctx->graph_exec, g, 0);
      if (e != cudaSuccess) {
        ctx->graph_exec = nullptr;
        set_err(ctx, "cudaGraphInstantiate", e);
        st = CRISP_ERR_CUDA;
      }
    }
    if (g) cudaGraphDestroy(g);
    if (st != CRISP_OK) {
      cudaGetLastError();
      ctx->has_sel = false;
      ctx->has_patsearch = false;
      return st;
    }
    ctx->graph_key = key;
  }
  const cudaError_t e = cudaGraphLaunch(ctx->graph_exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_err(ctx, "cudaGraphLaunch", e);
    return CRISP_ERR_CUDA;
  }
  ctx->has_sel = true;
  ctx->has_patsearch = true;
  ctx->sel_dims = *dims;
  return CRISP_OK;
}

crisp_status crisp_prefill(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                           const void* V, const crisp_cfg* cfg, void* O, void* stream) {
  if (!V || !O) return CRISP_ERR_INVALID_ARG;
  if (cfg && (cfg->flags & CRISP_FLAG_GRAPH_REPLAY))
    return prefill_replay(ctx, dims, Q, K, V, cfg, O, stream);
  crisp_status st = crisp_select(ctx, dims, Q, K, cfg, stream);
  if (st != CRISP_OK) return st;
  return crisp_attend(ctx, dims, Q, K, V, O, stream);
}

int32_t crisp_prefill_launches(const crisp_dims* dims, int32_t num_sms) {
  if (!dims || num_sms < 1 || check_dims(dims) != CRISP_OK) return 0;
  const Shape s = make_shape(*dims);
  const int per = attention_kv_heads_per_launch(s, num_sms);
  // selection: PatSearch and route, PE block means 1, pooled softmax 1, the gamma cut, CSR
  return patsearch_launches(s.nb) + 1 + 1 + pe_select_launches(s.nb) +
         csr_launches(static_cast<int64_t>(s.H) * s.nb) +
         order_launches(s, num_sms) + (s.Hkv + per - 1) / per + 1;
}

crisp_status crisp_prefill_host(crisp_ctx ctx, const crisp_dims* dims, const void* Q_host,
                                const void* K_host, const void* V_host, const crisp_cfg* cfg,
                                void* O_host, void* Q, void* K, void* V, void* O, void* stream) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if ((st = check_cfg(cfg)) != CRISP_OK) return st;
  if (!Q_host || !K_host || !V_host || !O_host || !Q || !K || !V || !O || !aligned16(Q) ||
      !aligned16(K) || !aligned16(V) || !aligned16(O))
    return CRISP_ERR_INVALID_ARG;
  const Shape s = make_shape(*dims);
  const int group = s.group;
  // KV heads per chunk: at least 8 query-block rows per SM in every chunk, and no more
  // than kMaxChunks chunks.
  const int rows_per_kv = group * s.nb;
  int per = (8 * ctx->num_sms + rows_per_kv - 1) / rows_per_kv;
  per = std::max(per, (s.Hkv + crisp_ctx_s::kMaxChunks - 1) / crisp_ctx_s::kMaxChunks);
  per = std::max(1, std::min(per, s.Hkv));
  // Chunks (first KV head, KV heads, first query head, query heads, upload K/V).  With one
  // KV head per chunk, the first and the last KV groups are split into one query head per
  // chunk, so the upload before the first computation and the download after the last are
  // one head's worth (the group's K/V travel with its first head).
  struct Chunk {
    int g0, m, h0, hn;
    bool kv;
  };
  Chunk chunks[crisp_ctx_s::kMaxChunks];
  int nchunks = 0;
  const bool split_ends = per == 1 && group > 1 && s.Hkv >= 2 &&
                          s.Hkv + 2 * (group - 1) <= crisp_ctx_s::kMaxChunks;
  for (int g0 = 0; g0 < s.Hkv; g0 += per) {
    const int m = std::min(per, s.Hkv - g0);
    if (split_ends && (g0 == 0 || g0 == s.Hkv - 1)) {
      for (int i = 0; i < group; ++i) chunks[nchunks++] = Chunk{g0, 1, g0 * group + i, 1, i == 0};
    } else {
      chunks[nchunks++] = Chunk{g0, m, g0 * group, m * group, true};
    }
  }
  const size_t head_bytes = static_cast<size_t>(s.n) * kD * 2;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  auto ok = [&](cudaError_t e, const char* what) { return launched(ctx, e, what) == CRISP_OK; };
  // Work already queued on the caller's stream (earlier use of Q/K/V/O) comes first.
  if (!ok(cudaEventRecord(ctx->ev_entry, cs), "record") ||
      !ok(cudaStreamWaitEvent(ctx->h2d, ctx->ev_entry, 0), "wait") ||
      !ok(cudaStreamWaitEvent(ctx->d2h, ctx->ev_entry, 0), "wait"))
    return CRISP_ERR_CUDA;
  for (int c = 0; c < nchunks; ++c) {
    const Chunk& ch = chunks[c];
    const size_t qoff = static_cast<size_t>(ch.h0) * head_bytes;
    const size_t kvoff = static_cast<size_t>(ch.g0) * head_bytes;
    const size_t qbytes = static_cast<size_t>(ch.hn) * head_bytes;
    const size_t kvbytes = static_cast<size_t>(ch.m) * head_bytes;
    // upload chunk c (the copy stream runs ahead of the compute stream)
    if (!ok(cudaMemcpyAsync(static_cast<char*>(Q) + qoff, static_cast<const char*>(Q_host) + qoff,
                            qbytes, cudaMemcpyHostToDevice, ctx->h2d), "upload Q") ||
        (ch.kv &&
         (!ok(cudaMemcpyAsync(static_cast<char*>(K) + kvoff, static_cast<const char*>(K_host) + kvoff,
                              kvbytes, cudaMemcpyHostToDevice, ctx->h2d), "upload K") ||
          !ok(cudaMemcpyAsync(static_cast<char*>(V) + kvoff, static_cast<const char*>(V_host) + kvoff,
                              kvbytes, cudaMemcpyHostToDevice, ctx->h2d), "upload V"))) ||
        !ok(cudaEventRecord(ctx->ev_in[c], ctx->h2d), "record") ||
        !ok(cudaStreamWaitEvent(cs, ctx->ev_in[c], 0), "wait"))
      return CRISP_ERR_CUDA;
    // select and attend chunk c: an independent problem of ch.hn query heads over ch.m KV
    // heads
    const crisp_dims sub{1, s.n, ch.hn, ch.m, kD};
    if ((st = crisp_select(ctx, &sub, static_cast<char*>(Q) + qoff, static_cast<char*>(K) + kvoff,
                           cfg, stream)) != CRISP_OK ||
        (st = crisp_attend(ctx, &sub, static_cast<char*>(Q) + qoff, static_cast<char*>(K) + kvoff,
                           static_cast<char*>(V) + kvoff, static_cast<char*>(O) + qoff, stream)) !=
            CRISP_OK)
      return st;
    // download chunk c's output once it is written
    if (!ok(cudaEventRecord(ctx->ev_out[c], cs), "record") ||
        !ok(cudaStreamWaitEvent(ctx->d2h, ctx->ev_out[c], 0), "wait") ||
        !ok(cudaMemcpyAsync(static_cast<char*>(O_host) + qoff, static_cast<char*>(O) + qoff, qbytes,
                            cudaMemcpyDeviceToHost, ctx->d2h), "download O"))
      return CRISP_ERR_CUDA;
  }
  if (!ok(cudaEventRecord(ctx->ev_done, ctx->d2h), "record") ||
      !ok(cudaStreamWaitEvent(cs, ctx->ev_done, 0), "wait"))
    return CRISP_ERR_CUDA;
  ctx->has_sel = false;  // the context held one chunk's selection at a time
  ctx->has_patsearch = false;
  return CRISP_OK;
}

static crisp_status copy_out(crisp_ctx ctx, void* dst, const void* src, size_t bytes) {
  if (!dst || !bytes) return CRISP_OK;
  cudaError_t e = cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost);
  return launched(ctx, e, "copy selection");
}

crisp_status crisp_selection_get(crisp_ctx ctx, const crisp_dims* dims, void* stream,
                                 crisp_selection_host* out) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if (!out) return CRISP_ERR_INVALID_ARG;
  if (!ctx->has_sel || !same_dims(ctx->sel_dims, *dims)) return CRISP_ERR_NO_SELECTION;
  if ((st = launched(ctx, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "sync")) != CRISP_OK)
    return st;
  const Shape s = make_shape(*dims);
  const size_t H = s.H, nb = s.nb, rows = H * nb;
  const Workspace& w = ctx->ws;
  if ((st = copy_out(ctx, out->route_vs, w.route, H)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, out->c_struct, w.cstruct, H * 4)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, out->mu, w.mu, H * 8)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, out->counts, w.counts, H * 16)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, out->p_v, w.pv, H * nb * 4)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, out->p_s, w.ps, H * nb * 4)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, out->sel_v, w.selv, H * nb)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, out->sel_s, w.sels, H * nb)) != CRISP_OK) return st;
  int64_t nnz = 0;
  if ((st = copy_out(ctx, &nnz, w.row_ptr + rows, sizeof(int64_t))) != CRISP_OK) return st;
  out->nnz = nnz;
  if ((st = copy_out(ctx, out->row_ptr, w.row_ptr, (rows + 1) * 8)) != CRISP_OK) return st;
  if (out->col) {
    if (out->col_capacity < nnz) return CRISP_ERR_INVALID_ARG;
    if ((st = copy_out(ctx, out->col, w.col, static_cast<size_t>(nnz) * 4)) != CRISP_OK) return st;
  }
  return CRISP_OK;
}

crisp_status crisp_selection_set(crisp_ctx ctx, const crisp_dims* dims, void* stream,
                                 const int64_t* row_ptr, const int32_t* col, int64_t nnz) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if (!row_ptr || !col || nnz <= 0) return CRISP_ERR_INVALID_ARG;
  const Shape s = make_shape(*dims);
  const int64_t rows = static_cast<int64_t>(s.H) * s.nb;
  if (row_ptr[0] != 0 || row_ptr[rows] != nnz || nnz > ctx->ws.col_cap) return CRISP_ERR_INVALID_ARG;
  for (int64_t r = 0; r < rows; ++r) {
    const int64_t b = row_ptr[r], e = row_ptr[r + 1];
    if (e <= b) return CRISP_ERR_INVALID_ARG;
    const int I = static_cast<int>(r % s.nb);
    for (int64_t k = b; k < e; ++k) {
      if (col[k] < 0 || col[k] > I) return CRISP_ERR_INVALID_ARG;
      if (k > b && col[k] <= col[k - 1]) return CRISP_ERR_INVALID_ARG;
    }
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if ((st = launched(ctx, cudaStreamSynchronize(cs), "sync")) != CRISP_OK) return st;
  if ((st = launched(ctx, cudaMemcpy(ctx->ws.row_ptr, row_ptr, (rows + 1) * 8, cudaMemcpyHostToDevice),
                     "upload row_ptr")) != CRISP_OK)
    return st;
  if ((st = launched(ctx, cudaMemcpy(ctx->ws.col, col, nnz * 4, cudaMemcpyHostToDevice),
                     "upload col")) != CRISP_OK)
    return st;
  ctx->has_sel = true;
  ctx->has_patsearch = false;
  ctx->sel_dims = *dims;
  return CRISP_OK;
}

crisp_status crisp_jsd(crisp_ctx ctx, const crisp_dims* dims, const void* Q, const void* K,
                       float tau_jsd, float* d_js, uint8_t* route_vs, void* stream) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if (!Q || !K || !d_js || !route_vs || !aligned16(Q) || !aligned16(K) || !(tau_jsd == tau_jsd))
    return CRISP_ERR_INVALID_ARG;
  if (!ctx->has_sel || !ctx->has_patsearch || !same_dims(ctx->sel_dims, *dims))
    return CRISP_ERR_NO_SELECTION;
  const Shape s = make_shape(*dims);
  return launched(ctx,
                  launch_jsd(ctx, s, Q, K, tau_jsd, d_js, route_vs, static_cast<cudaStream_t>(stream)),
                  "jsd");
}

crisp_status crisp_selection_stats(crisp_ctx ctx, const crisp_dims* dims, void* stream,
                                   crisp_stats* out) {
  crisp_status st = check_common(ctx, dims);
  if (st != CRISP_OK) return st;
  if (!out) return CRISP_ERR_INVALID_ARG;
  if (!ctx->has_sel || !same_dims(ctx->sel_dims, *dims)) return CRISP_ERR_NO_SELECTION;
  if ((st = launched(ctx, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "sync")) != CRISP_OK)
    return st;
  const Shape s = make_shape(*dims);
  const int64_t rows = static_cast<int64_t>(s.H) * s.nb;
  std::vector<int64_t> rp(rows + 1);
  std::vector<uint8_t> route(s.H);
  std::vector<int32_t> counts(4 * s.H), near(3 * s.H);
  if ((st = copy_out(ctx, rp.data(), ctx->ws.row_ptr, (rows + 1) * 8)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, route.data(), ctx->ws.route, s.H)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, counts.data(), ctx->ws.counts, 16 * s.H)) != CRISP_OK) return st;
  if ((st = copy_out(ctx, near.data(), ctx->ws.near, 12 * s.H)) != CRISP_OK) return st;
  out->nnz = rp[rows];
  out->rows = rows;
  out->max_row = 0;
  for (int64_t r = 0; r < rows; ++r)
    if (rp[r + 1] - rp[r] > out->max_row) out->max_row = rp[r + 1] - rp[r];
  out->n_vs = 0;
  out->n_pe = 0;
  out->pe_rescued = 0;
  out->near_routes = 0;
  out->near_vs_blocks = 0;
  out->near_pe_pairs = 0;
  for (int h = 0; h < s.H; ++h) {
    out->near_routes += near[3 * h];
    out->near_vs_blocks += near[3 * h + 1];
    out->near_pe_pairs += near[3 * h + 2];
    if (route[h]) {
      ++out->n_vs;
    } else {
      ++out->n_pe;
      out->pe_rescued += counts[4 * h + 1];
    }
  }
  return CRISP_OK;
}

crisp_status crisp_attend_info(crisp_ctx ctx, void* stream, int64_t* rows) {
  if (!ctx || !rows) return CRISP_ERR_INVALID_ARG;
  crisp_status st = launched(ctx, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "sync");
  if (st != CRISP_OK) return st;
  int count = 0;
  if ((st = copy_out(ctx, &count, ctx->ws.redo_count, sizeof(int))) != CRISP_OK) return st;
  *rows = count;
  return CRISP_OK;
}

crisp_status crisp_sync_status(crisp_ctx ctx, void* stream) {
  if (!ctx) return CRISP_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_err(ctx, "stream", e);
    return CRISP_ERR_CUDA;
  }
  uint32_t word = 0;
  if ((e = cudaMemcpy(&word, ctx->ws.err, 4, cudaMemcpyDeviceToHost)) != cudaSuccess) {
    set_err(ctx, "read error word", e);
    return CRISP_ERR_CUDA;
  }
  if (word) cudaMemset(ctx->ws.err, 0, 4);
  if (word & kErrTimeout) return CRISP_ERR_TIMEOUT;
  if (word & kErrRange) return CRISP_ERR_DEVICE_ASSERT;
  return CRISP_OK;
}

crisp_status crisp_set_debug(crisp_ctx ctx, uint32_t flags, uint64_t timeout_ns) {
  if (!ctx) return CRISP_ERR_INVALID_ARG;
  ctx->debug_flags = flags;
  ctx->timeout_ns = timeout_ns ? timeout_ns : 1000000000ull;
  return CRISP_OK;
}

const char* crisp_last_error(crisp_ctx ctx) { return ctx ? ctx->last_err : ""; }

}  // extern "C"
