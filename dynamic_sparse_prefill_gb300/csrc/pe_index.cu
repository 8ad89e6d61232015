// pe_index.cu -- PEIndex (GlobalAdaptive) selection for heads routed PE.
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top), "Method step details" step 3 and Algorithm 4
// (PEIndex) under "Figures and tables": pool all queries and keys by block, softmax the
// pooled scores, normalise and flatten, sort, and keep the top pairs until their
// cumulative mass reaches gamma ("Prerequisites", the cumulative coverage rule).
//
// The sort is a radix select on the fp32 bit patterns of the (positive) flattened scores
// with fp64 mass per digit: four 8-bit passes find the threshold value T with
// mass(v > T) < gamma <= mass(v >= T); items equal to T are then taken in flat-index
// order (I*N_b + K) until the running mass reaches gamma.  Every PE row also gets its
// diagonal pair, so that no query block is left without keys.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace crisp {
namespace {

// ---------------------------------------------------------------- block means
// Qbar[h][I][:] = mean of the 128 rows of query block I (PE heads only).
__global__ void __launch_bounds__(128) pe_pool_q_kernel(const uint16_t* __restrict__ Q,
                                                        const uint8_t* __restrict__ route,
                                                        int n, int nb, float* qbar) {
  const int h = blockIdx.y, I = blockIdx.x;
  if (route[h]) return;
  __shared__ float part[8][kD];
  const int rg = threadIdx.x >> 4;          // row group 0..7
  const int cc = (threadIdx.x & 15) * 8;    // 8 columns
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint16_t* base = Q + (static_cast<size_t>(h) * n + static_cast<size_t>(I) * kBlk) * kD;
  for (int rr = rg; rr < kBlk; rr += 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(rr) * kD + cc);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[2 * k] += __uint_as_float(w[k] << 16);
      acc[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) part[rg][cc + k] = acc[k];
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int g = 0; g < 8; ++g) s += part[g][threadIdx.x];
  qbar[(static_cast<size_t>(h) * nb + I) * kD + threadIdx.x] = s * (1.f / kBlk);
}

// Kbar for every KV head that serves at least one PE query head.
__global__ void __launch_bounds__(128) pe_pool_k_kernel(const uint16_t* __restrict__ K,
                                                        const uint8_t* __restrict__ route,
                                                        int n, int nb, int hq, int hkv,
                                                        int group, float* kbar) {
  const int hk = blockIdx.y, I = blockIdx.x;
  const int bidx = hk / hkv, kvh = hk % hkv;
  bool any_pe = false;
  for (int g = 0; g < group; ++g) any_pe |= route[bidx * hq + kvh * group + g] == 0;
  if (!any_pe) return;
  __shared__ float part[8][kD];
  const int rg = threadIdx.x >> 4;
  const int cc = (threadIdx.x & 15) * 8;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint16_t* base = K + (static_cast<size_t>(hk) * n + static_cast<size_t>(I) * kBlk) * kD;
  for (int rr = rg; rr < kBlk; rr += 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(rr) * kD + cc);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[2 * k] += __uint_as_float(w[k] << 16);
      acc[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) part[rg][cc + k] = acc[k];
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int g = 0; g < 8; ++g) s += part[g][threadIdx.x];
  kbar[(static_cast<size_t>(hk) * nb + I) * kD + threadIdx.x] = s * (1.f / kBlk);
}

// ---------------------------------------------------------------- pooled logits
// logits[I][K] = Qbar_I . Kbar_K / sqrt(d) for K <= I, in 128 x 128 tiles (fp32 FMA).  Each
// thread accumulates 8 x 8 outputs (rows ty + 16i, columns tx + 16j), two columns per
// packed f32x2 FMA, so a step over d takes 16 shared-memory loads and 32 FMA instructions,
// and the loads of a warp fall in distinct banks (the tiles are stored transposed,
// [d][row], with a row pitch of 129 floats).
constexpr int kPT = 128;
__global__ void __launch_bounds__(256) pe_scores_kernel(const float* __restrict__ qbar,
                                                        const float* __restrict__ kbar,
                                                        const uint8_t* __restrict__ route,
                                                        int nb, int hq, int hkv, int group,
                                                        float scale, float* pev) {
  const int h = blockIdx.z;
  const int I0 = blockIdx.y * kPT, K0 = blockIdx.x * kPT;
  if (route[h] || K0 > I0 + kPT - 1) return;
  const int hk = (h / hq) * hkv + (h % hq) / group;
  __shared__ float sq[32][kPT + 1], sk[32][kPT + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float2 acc[8][4];  // acc[i][j] = outputs (row ty + 16i, columns tx + 32j, tx + 32j + 16)
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);
  for (int d0 = 0; d0 < kD; d0 += 32) {
    for (int i = threadIdx.x; i < kPT * 32; i += 256) {
      const int row = i >> 5, dd = i & 31;
      const int I = I0 + row, K = K0 + row;
      sq[dd][row] = I < nb ? qbar[(static_cast<size_t>(h) * nb + I) * kD + d0 + dd] : 0.f;
      sk[dd][row] = K < nb ? kbar[(static_cast<size_t>(hk) * nb + K) * kD + d0 + dd] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int dd = 0; dd < 32; ++dd) {
      float a[8];
      float2 b[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = sq[dd][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = make_float2(sk[dd][tx + 32 * j], sk[dd][tx + 32 * j + 16]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int I = I0 + ty + 16 * i, K = K0 + tx + 32 * j;
      if (I < nb && K <= I) pev[(static_cast<size_t>(h) * nb + I) * nb + K] = acc[i][j].x * scale;
      if (I < nb && K + 16 <= I)
        pev[(static_cast<size_t>(h) * nb + I) * nb + K + 16] = acc[i][j].y * scale;
    }
}

// v[I][K] = softmax_{K <= I}(logits[I]) / N_b, in place.
__global__ void __launch_bounds__(256) pe_softmax_kernel(const uint8_t* __restrict__ route,
                                                         int nb, float* pev) {
  const int h = blockIdx.y, I = blockIdx.x;
  if (route[h]) return;
  __shared__ float red[8];
  __shared__ float bc;
  float* row = pev + (static_cast<size_t>(h) * nb + I) * nb;
  const int len = I + 1;
  float mx = -FLT_MAX;
  for (int K = threadIdx.x; K < len; K += 256) mx = fmaxf(mx, row[K]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = red[0];
    for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
    bc = m;
  }
  __syncthreads();
  mx = bc;
  float s = 0.f;
  for (int K = threadIdx.x; K < len; K += 256) s += expf(row[K] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += red[i];
    bc = 1.f / (t * static_cast<float>(nb));
  }
  __syncthreads();
  const float inv = bc;
  for (int K = threadIdx.x; K < len; K += 256) row[K] = expf(row[K] - mx) * inv;
}

// ---------------------------------------------------------------- radix select
__global__ void pe_radix_init_kernel(PeState* pe, unsigned long long* hist_cnt,
                                     double* hist_mass) {
  const int h = blockIdx.x;
  if (threadIdx.x == 0) {
    PeState s{};
    pe[h] = s;
  }
  hist_cnt[h * 256 + threadIdx.x] = 0;
  hist_mass[h * 256 + threadIdx.x] = 0.0;
}

constexpr int kHistRows = 16;
__global__ void __launch_bounds__(256) pe_hist_kernel(const float* __restrict__ pev,
                                                      const uint8_t* __restrict__ route,
                                                      const PeState* __restrict__ pe, int nb,
                                                      int shift, unsigned long long* hist_cnt,
                                                      double* hist_mass) {
  const int h = blockIdx.y;
  if (route[h]) return;
  const PeState st = pe[h];
  if (st.select_all) return;
  // Per-warp histograms with native fp32 shared-memory atomics (later passes see many
  // values in few bins, so one shared copy serialises the warps); the CTA's partial
  // masses (each at most a few percent of the total) are combined in fp64 in global
  // memory.
  __shared__ unsigned int scnt[8][256];
  __shared__ float smass[8][256];
  const int wp = threadIdx.x >> 5;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    scnt[w][threadIdx.x] = 0;
    smass[w][threadIdx.x] = 0.f;
  }
  __syncthreads();
  // Each thread caches two (bin, count, fp32 mass) entries and flushes one to the shared
  // histogram only when a third bin appears: the early passes see long runs of one bin,
  // the later ones values alternating between neighbouring bins.
  uint32_t b0 = 0xFFFFFFFFu, b1 = 0xFFFFFFFFu, c0 = 0, c1 = 0;
  float m0 = 0.f, m1 = 0.f;
  auto take = [&](float v) {
    const uint32_t bits = __float_as_uint(v);
    if ((bits & st.decided) != st.prefix) return;
    const uint32_t bin = (bits >> shift) & 255u;
    if (bin == b0) {
      ++c0;
      m0 += v;
    } else if (bin == b1) {
      ++c1;
      m1 += v;
    } else {
      if (c1) {
        atomicAdd(&scnt[wp][b1], c1);
        atomicAdd(&smass[wp][b1], m1);
      }
      b1 = b0;
      c1 = c0;
      m1 = m0;
      b0 = bin;
      c0 = 1;
      m0 = v;
    }
  };
  const int I0 = blockIdx.x * kHistRows;
  for (int I = I0; I < min(nb, I0 + kHistRows); ++I) {
    const float* row = pev + (static_cast<size_t>(h) * nb + I) * nb;
    const int len = I + 1;
    if ((nb & 3) == 0) {
      // rows start on 16-byte boundaries: two float4 loads in flight per thread
      const float4* row4 = reinterpret_cast<const float4*>(row);
      const int n4 = len >> 2;
      int q = threadIdx.x;
      for (; q + 256 < n4; q += 512) {
        const float4 x = row4[q], y = row4[q + 256];
        take(x.x); take(x.y); take(x.z); take(x.w);
        take(y.x); take(y.y); take(y.z); take(y.w);
      }
      if (q < n4) {
        const float4 x = row4[q];
        take(x.x); take(x.y); take(x.z); take(x.w);
      }
      const int K = (n4 << 2) + threadIdx.x;
      if (K < len) take(row[K]);
    } else {
      for (int K = threadIdx.x; K < len; K += 256) take(row[K]);
    }
  }
  if (c0) {
    atomicAdd(&scnt[wp][b0], c0);
    atomicAdd(&smass[wp][b0], m0);
  }
  if (c1) {
    atomicAdd(&scnt[wp][b1], c1);
    atomicAdd(&smass[wp][b1], m1);
  }
  __syncthreads();
  unsigned int c = 0;
  double m = 0.0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    c += scnt[w][threadIdx.x];
    m += static_cast<double>(smass[w][threadIdx.x]);
  }
  if (c) {
    atomicAdd(&hist_cnt[h * 256 + threadIdx.x], static_cast<unsigned long long>(c));
    atomicAdd(&hist_mass[h * 256 + threadIdx.x], m);
  }
}

// Picks the digit whose bin crosses the remaining target; one thread per head.
__global__ void pe_digit_kernel(const uint8_t* __restrict__ route, int pass, float gamma,
                                PeState* pe, unsigned long long* hist_cnt, double* hist_mass) {
  const int h = blockIdx.x;
  if (route[h] == 0 && threadIdx.x == 0) {
    PeState st = pe[h];
    if (!st.select_all) {
      const int shift = 24 - 8 * pass;
      const double rem = static_cast<double>(gamma) - st.mass_above;
      double cum = 0.0;
      int chosen = -1, lowest = -1;
      for (int bin = 255; bin >= 0; --bin) {
        const unsigned long long c = hist_cnt[h * 256 + bin];
        if (!c) continue;
        const double m = hist_mass[h * 256 + bin];
        if (cum + m >= rem) {
          chosen = bin;
          break;
        }
        cum += m;
        lowest = bin;
      }
      if (chosen < 0) {
        if (pass == 0 || lowest < 0) {
          st.select_all = 1;  // the whole triangle holds less than gamma
        } else {
          chosen = lowest;
          cum -= hist_mass[h * 256 + lowest];
        }
      }
      if (!st.select_all) {
        st.mass_above += cum;
        st.prefix |= static_cast<uint32_t>(chosen) << shift;
        st.decided |= 255u << shift;
        if (pass == 3) {
          st.thresh = st.prefix;
          st.count_eq = hist_cnt[h * 256 + chosen];
          const double vt = static_cast<double>(__uint_as_float(st.thresh));
          const double rem2 = static_cast<double>(gamma) - st.mass_above;
          unsigned long long need = st.count_eq;
          if (vt > 0.0) {
            const double q = ceil(rem2 / vt);
            need = q < 1.0 ? 1ull : static_cast<unsigned long long>(q);
          }
          st.need_eq = need < st.count_eq ? need : st.count_eq;
        }
      }
      pe[h] = st;
    }
  }
  __syncthreads();
  hist_cnt[h * 256 + threadIdx.x] = 0;
  hist_mass[h * 256 + threadIdx.x] = 0.0;
}

// Number of items equal to the threshold in each PE row (for flat-order tie ranks).
__global__ void __launch_bounds__(256) pe_eqcount_kernel(const float* __restrict__ pev,
                                                         const uint8_t* __restrict__ route,
                                                         const PeState* __restrict__ pe,
                                                         int nb, int64_t* eq_off) {
  const int h = blockIdx.y, I = blockIdx.x;
  if (route[h]) return;
  const PeState st = pe[h];
  if (st.select_all || st.need_eq >= st.count_eq) return;  // no tie ranks needed
  __shared__ int red[8];
  int c = 0;
  {
    const float* row = pev + (static_cast<size_t>(h) * nb + I) * nb;
    for (int K = threadIdx.x; K <= I; K += 256) c += __float_as_uint(row[K]) == st.thresh;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int i = 0; i < 8; ++i) t += red[i];
    eq_off[static_cast<size_t>(h) * (nb + 1) + I] = t;
  }
}

// In-place exclusive scan of the per-row counts of one head (nb <= 8192 entries).
__global__ void __launch_bounds__(1024) pe_eqscan_kernel(const uint8_t* __restrict__ route,
                                                         const PeState* __restrict__ pe, int nb,
                                                         int64_t* eq_off) {
  const int h = blockIdx.x;
  if (route[h]) return;
  const PeState st = pe[h];
  if (st.select_all || st.need_eq >= st.count_eq) return;  // no tie ranks needed
  __shared__ int64_t part[1024];
  int64_t* a = eq_off + static_cast<size_t>(h) * (nb + 1);
  const int per = (nb + 1023) / 1024;
  const int b0 = threadIdx.x * per, b1 = min(nb, b0 + per);
  int64_t s = 0;
  for (int i = b0; i < b1; ++i) s += a[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int64_t t = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += t;
    __syncthreads();
  }
  int64_t run = part[threadIdx.x] - s;
  for (int i = b0; i < b1; ++i) {
    const int64_t c = a[i];
    a[i] = run;
    run += c;
  }
  if (threadIdx.x == 1023) a[nb] = part[1023];
}

// Row masks of PE heads: v > T, or v == T with flat rank < need; plus the diagonal.  A warp
// per row, four 32-key words in flight per lane.  Flat-order tie ranks are needed only
// when some but not all items equal to the threshold are taken (need_eq < count_eq).
__global__ void __launch_bounds__(256) pe_mask_kernel(const float* __restrict__ pev,
                                                      const uint8_t* __restrict__ route,
                                                      const PeState* __restrict__ pe,
                                                      const int64_t* __restrict__ eq_off,
                                                      int nb, int nbw, uint32_t* rowmask,
                                                      int32_t* counts) {
  const int h = blockIdx.y;
  if (route[h]) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int I = blockIdx.x * 8 + warp;
  if (I >= nb) return;
  const PeState st = pe[h];
  const bool all = st.select_all != 0;
  const bool rank_ties = !all && st.need_eq < st.count_eq;
  int64_t eq_base = rank_ties ? eq_off[static_cast<size_t>(h) * (nb + 1) + I] : 0;
  const float* row = pev + (static_cast<size_t>(h) * nb + I) * nb;
  uint32_t* mrow = rowmask + (static_cast<size_t>(h) * nb + I) * nbw;
  const int nw = (I >> 5) + 1;  // words holding keys K <= I
  int selected = 0;
  for (int wd0 = 0; wd0 < nw; wd0 += 4) {
    uint32_t x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int K = (wd0 + u) * 32 + lane;
      x[u] = K <= I ? __float_as_uint(row[K]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int wd = wd0 + u;
      if (wd >= nw) break;
      const bool valid = wd * 32 + lane <= I;
      bool sel = valid && (all || x[u] > st.thresh);
      if (!all) {
        const bool eq = valid && x[u] == st.thresh;
        if (rank_ties) {
          const unsigned beq = __ballot_sync(0xffffffffu, eq);
          const int64_t rank = eq_base + __popc(beq & ((1u << lane) - 1u));
          sel = sel || (eq && rank < static_cast<int64_t>(st.need_eq));
          eq_base += __popc(beq);
        } else {
          sel = sel || eq;
        }
      }
      unsigned word = __ballot_sync(0xffffffffu, sel);
      selected += __popc(word);
      if (wd == (I >> 5)) word |= 1u << (I & 31);
      if (lane == 0) mrow[wd] = word;
    }
  }
  for (int wd = nw + lane; wd < nbw; wd += 32) mrow[wd] = 0u;
  if (lane == 0) {
    atomicAdd(&counts[h * 4 + 0], selected);
    if (selected == 0) atomicAdd(&counts[h * 4 + 1], 1);
  }
}

}  // namespace

cudaError_t launch_pe_index(crisp_ctx ctx, const Shape& s, const crisp_cfg& cfg, const void* Q,
                            const void* K, cudaStream_t st) {
  Workspace& w = ctx->ws;
  const uint16_t* q = static_cast<const uint16_t*>(Q);
  const uint16_t* k = static_cast<const uint16_t*>(K);
  pe_pool_q_kernel<<<dim3(s.nb, s.H), 128, 0, st>>>(q, w.route, s.n, s.nb, w.qbar);
  pe_pool_k_kernel<<<dim3(s.nb, s.Hkv), 128, 0, st>>>(k, w.route, s.n, s.nb, s.hq, s.hkv,
                                                       s.group, w.kbar);
  const int nt = (s.nb + kPT - 1) / kPT;
  pe_scores_kernel<<<dim3(nt, nt, s.H), 256, 0, st>>>(w.qbar, w.kbar, w.route, s.nb, s.hq,
                                                      s.hkv, s.group,
                                                      1.f / sqrtf(static_cast<float>(kD)), w.pev);
  pe_softmax_kernel<<<dim3(s.nb, s.H), 256, 0, st>>>(w.route, s.nb, w.pev);
  pe_radix_init_kernel<<<s.H, 256, 0, st>>>(w.pe, w.hist_cnt, w.hist_mass);
  for (int pass = 0; pass < 4; ++pass) {
    pe_hist_kernel<<<dim3((s.nb + kHistRows - 1) / kHistRows, s.H), 256, 0, st>>>(
        w.pev, w.route, w.pe, s.nb, 24 - 8 * pass, w.hist_cnt, w.hist_mass);
    pe_digit_kernel<<<s.H, 256, 0, st>>>(w.route, pass, cfg.gamma, w.pe, w.hist_cnt,
                                         w.hist_mass);
  }
  pe_eqcount_kernel<<<dim3(s.nb, s.H), 256, 0, st>>>(w.pev, w.route, w.pe, s.nb, w.eq_off);
  pe_eqscan_kernel<<<s.H, 1024, 0, st>>>(w.route, w.pe, s.nb, w.eq_off);
  pe_mask_kernel<<<dim3((s.nb + 7) / 8, s.H), 256, 0, st>>>(w.pev, w.route, w.pe, w.eq_off, s.nb,
                                                            s.nbw, w.rowmask, w.counts);
  return cudaGetLastError();
}

}  // namespace crisp
