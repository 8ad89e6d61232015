// patsearch.cu -- PatSearch proxy attention, C_struct routing and VS index selection.
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top), "Core method" step 1 and "Method step details"
// steps 1-2; Algorithms 2 (PatSearch) and 3 (VSIndex) under "Figures and tables".
//
// Per query head: A_hat = causal Softmax(Q[-b:] K^T / sqrt(d)) (b = 128 rows),
// a_v = column mean, a_s = diagonal mean (delta = query - key position), both pooled by
// blocks of B = 128, C_struct = anchor mass of a_v, VS iff C_struct >= tau.
//
// A_hat is never materialised.  One pass over K (tcgen05 MMA, S in TMEM) records, for
// every proxy row r and key tile t, the tile's row maximum m and two partial sums of
// exp2(s - m): u over keys on or left of the row's diagonal offset, w over the others.
// Because delta = 128*(N_b-1-t) + (r - c) for key column c of tile t, u is exactly the
// row's mass on slash block N_b-1-t and w its mass on slash block N_b-2-t, and u + w its
// mass on vertical block t.  A second, cheap kernel rescales the partials with the
// row's global max and sum, which gives the pooled p_v and p_s directly.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace crisp {

namespace {

constexpr int kProxyThreads = 352;  // warp 0: TMA, warps 1-2: MMA, warps 3-10: epilogue
constexpr int kProxyStages = 4;
static_assert(kProxyStages % 2 == 0, "each K stage must serve tiles of one parity (one MMA issuer)");
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr size_t kProxySmem = 1024 + kTileBytes * (1 + kProxyStages) + 256;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Warp-uniform bounded wait: lane 0 waits, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort, uint64_t tmo) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err, abort, tmo) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Wait for asynchronous work this thread issued, ignoring the abort flag (bounded).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                           uint64_t tmo) {
  volatile int never = 0;
  mbar_wait(bar, parity, err, &never, tmo);
}

struct ProxyArgs {
  int n, nb, hq, hkv, group;
  int w_sink, w_local;
  int tiles_per_cta;
  float scale_log2;
  float* st_m;
  float* st_u;
  float* st_w;
  float* anc;
  uint32_t* err;
  uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kProxyThreads, 1)
    proxy_tile_stats_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK, const ProxyArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sK + kProxyStages * kTileBytes);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kProxyStages;
  uint64_t* s_full = k_empty + kProxyStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* drain = s_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;  // flattened query head
  const int t_begin = blockIdx.y * a.tiles_per_cta;
  const int t_end = min(a.nb, t_begin + a.tiles_per_cta);
  const int ntiles = t_end - t_begin;
  if (ntiles <= 0) return;
  const int hk = (h / a.hq) * a.hkv + (h % a.hq) / a.group;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kProxyStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(drain, 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t tmo = a.timeout_ns;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      const int qrow = h * a.n + a.n - kBlk;
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(sQ, &tmQ, q_full, 0, qrow);
      tma_load_2d(sQ + kTileBytes / 2, &tmQ, q_full, 64, qrow);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kProxyStages;
        if (i >= kProxyStages &&
            !mbar_wait(&k_empty[s], ((i / kProxyStages) + 1) & 1, a.err, abort_flag, tmo))
          break;
        const int krow = hk * a.n + (t_begin + i) * kBlk;
        uint8_t* dst = sK + s * kTileBytes;
        mbar_arrive_expect_tx(&k_full[s], kTileBytes);
        tma_load_2d(dst, &tmK, &k_full[s], 0, krow);
        tma_load_2d(dst + kTileBytes / 2, &tmK, &k_full[s], 64, krow);
        ++issued;
      }
      drain_wait(q_full, 0, a.err, tmo);
      for (int i = max(0, issued - kProxyStages); i < issued; ++i)
        drain_wait(&k_full[i % kProxyStages], (i / kProxyStages) & 1, a.err, tmo);
    }
  } else if (warp <= 2) {
    // Two MMA issuers, warp 1 for the even tiles (S buffer 0), warp 2 for the odd ones:
    // tcgen05.mma issue waits for the tensor core, and after a tile's commits the issuing
    // thread's next barrier wait lasts until that tile's MMAs are done, so one issuer leaves
    // the tensor core idle between tiles.  With an even number of K stages every stage
    // serves tiles of one parity, i.e. one issuer.
    if (lane == 0) {
      if (mbar_wait(q_full, 0, a.err, abort_flag, tmo)) {
        const uint32_t q_base = smem_u32(sQ);
        for (int i = warp - 1; i < ntiles; i += 2) {
          const int s = i % kProxyStages, sb = i & 1;
          if (!mbar_wait(&k_full[s], (i / kProxyStages) & 1, a.err, abort_flag, tmo)) break;
          if (i >= 2 && !mbar_wait(&s_free[sb], ((i >> 1) + 1) & 1, a.err, abort_flag, tmo))
            break;
          tc_fence_after();
          const uint32_t k_base = smem_u32(sK + s * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
            umma_bf16(tmem + sb * 128, sdesc_sw128(q_base + off, 16, 1024),
                      sdesc_sw128(k_base + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[sb]);
          umma_commit(&k_empty[s]);
        }
      }
      umma_commit(drain);
      drain_wait(drain, 0, a.err, tmo);
    }
  } else {
    // Epilogue: two warpgroups, warpgroup e takes the tiles i with (i & 1) == e, i.e. the
    // S buffer e; thread <-> proxy row r (TMEM lane).  Each warpgroup exponentiates
    // against its running row maximum m_run and falls back to the tile's exact maximum
    // only when the sums show the tile exceeds m_run by a lot (the combine kernels accept
    // any per-tile reference maximum).
    const int e = (warp - 3) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t row_taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + e * 128;
    float m_run = -FLT_MAX;
    bool have_m = false;
    for (int i = e; i < ntiles; i += 2) {
      if (!warp_wait(&s_full[e], (i >> 1) & 1, a.err, abort_flag, tmo)) break;
      tc_fence_after();
      // The tile's S row in one TMEM load; the buffer goes straight back to its MMA issuer.
      uint32_t v[128];
      tmem_ld128(row_taddr, v);
      tc_fence_before();
      mbar_arrive(&s_free[e]);
      const int t = t_begin + i;
      const bool last = (t == a.nb - 1);
      const int j0 = t * kBlk;
      // u: keys with c <= r (slash block N_b-1-t); w: keys with c > r (slash block
      // N_b-2-t); the last tile is causal (c <= r only).  Column chunk c4 (32 keys) lies
      // wholly left of the row's offset when c4 < q, wholly right when c4 > q; only the
      // warp's own chunk c4 == q is split per lane.
      auto sums = [&](float m, float& u, float& w) {
        float ua = 0.f, ub = 0.f, wa = 0.f, wb = 0.f;
        const float neg = -m;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          if (c4 < q || (c4 > q && !last)) {
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(v[c4 * 32 + 2 * c]),
                    __uint_as_float(v[c4 * 32 + 2 * c + 1]), a.scale_log2, a.scale_log2, neg, neg);
              fadd2(sa, sb, sa, sb, fast_exp2(x0), fast_exp2(x1));
            }
            if (c4 < q) {
              ua += sa;
              ub += sb;
            } else {
              wa += sa;
              wb += sb;
            }
          } else if (c4 == q) {
            // the warp's own chunk, split per lane by predicated adds into separate sums
            // (the right part is dropped on the causal last tile)
            float la = 0.f, lb = 0.f, ra = 0.f, rb = 0.f;
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(v[c4 * 32 + c]), __uint_as_float(v[c4 * 32 + c + 1]),
                    a.scale_log2, a.scale_log2, neg, neg);
              const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
              if (c <= lane) la += e0; else ra += e0;
              if (c + 1 <= lane) lb += e1; else rb += e1;
            }
            ua += la + lb;
            if (!last) wa += ra + rb;
          }
        }
        u = ua + ub;
        w = wa + wb;
      };
      float u = 0.f, w = 0.f;
      bool slow = !have_m;
      if (!slow) {
        sums(m_run, u, w);
        slow = __any_sync(0xffffffffu, !(u + w <= 32768.f));
      }
      if (slow) {
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = -FLT_MAX;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (!last || c <= r) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(v[c]));
        const float ms = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * a.scale_log2;
        if (!have_m || ms > m_run) m_run = ms;
        have_m = true;
        sums(m_run, u, w);
      }
      // Anchor mass: the first w_sink keys (tile 0) and the last w_local keys (last tile).
      // With windows of one whole tile that is the tile's own u + w (w = 0 on the causal
      // last tile; with N_b = 1 the one tile is both and its keys count once).
      float an = 0.f;
      if ((t == 0 || last) && a.w_sink == kBlk && a.w_local == kBlk) {
        an = u + w;
      } else if (t == 0 || last) {
        const float neg = -m_run;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int j = j0 + c;
          const bool valid = !last || c <= r;
          const bool anchor = (t == 0 && j < a.w_sink) || (last && j >= a.n - a.w_local);
          if (valid && anchor) an += fast_exp2(fmaf(__uint_as_float(v[c]), a.scale_log2, neg));
        }
      }
      const size_t idx = (static_cast<size_t>(h) * a.nb + t) * kBlk + r;
      a.st_m[idx] = m_run;
      a.st_u[idx] = u;
      a.st_w[idx] = w;
      if (t == 0) {
        a.anc[(static_cast<size_t>(h) * 2 + 0) * kBlk + r] = an;
        if (last) a.anc[(static_cast<size_t>(h) * 2 + 1) * kBlk + r] = 0.f;
      } else if (last) {
        a.anc[(static_cast<size_t>(h) * 2 + 1) * kBlk + r] = an;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Row maximum M_r and normaliser Z_r of every proxy row over all key tiles.
__global__ void __launch_bounds__(256) proxy_row_stats_kernel(const float* __restrict__ st_m,
                                                              const float* __restrict__ st_u,
                                                              const float* __restrict__ st_w,
                                                              int nb, float2* part, int* ticket,
                                                              float* rowM, float* rowZ) {
  // kRowSplit CTAs per head each merge a contiguous range of tiles into (max, sum) per row;
  // the last CTA of the head to finish (ticket) merges the kRowSplit partials.
  __shared__ float sM[2][kBlk], sZ[2][kBlk];
  __shared__ int last;
  const int h = blockIdx.y, sp = blockIdx.x;
  const int r = threadIdx.x & 127, slice = threadIdx.x >> 7;
  const int per = (nb + kRowSplit - 1) / kRowSplit;
  const int t0 = sp * per, t1 = min(nb, t0 + per);
  float M = -FLT_MAX, Z = 0.f;
  for (int t = t0 + slice; t < t1; t += 2) {
    const size_t idx = (static_cast<size_t>(h) * nb + t) * kBlk + r;
    const float m = st_m[idx];
    const float sum = st_u[idx] + st_w[idx];
    if (m > M) {
      Z = Z * fast_exp2(M - m) + sum;
      M = m;
    } else {
      Z += sum * fast_exp2(m - M);
    }
  }
  sM[slice][r] = M;
  sZ[slice][r] = Z;
  __syncthreads();
  if (slice == 0) {
    const float Mt = fmaxf(sM[0][r], sM[1][r]);
    const float Zt = sZ[0][r] * fast_exp2(sM[0][r] - Mt) + sZ[1][r] * fast_exp2(sM[1][r] - Mt);
    part[(static_cast<size_t>(h) * kRowSplit + sp) * kBlk + r] = make_float2(Mt, Zt);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&ticket[h], 1) == kRowSplit - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (slice == 0) {
    const float2* p = part + static_cast<size_t>(h) * kRowSplit * kBlk + r;
    float Mt = -FLT_MAX;
    for (int i = 0; i < kRowSplit; ++i) Mt = fmaxf(Mt, __ldcg(&p[i * kBlk]).x);
    float Zt = 0.f;
    for (int i = 0; i < kRowSplit; ++i) {
      const float2 v = __ldcg(&p[i * kBlk]);
      Zt += v.y * fast_exp2(v.x - Mt);
    }
    rowM[h * kBlk + r] = Mt;
    rowZ[h * kBlk + r] = Zt;
  }
  if (threadIdx.x == 0) ticket[h] = 0;
}

// Pooled vertical and slash contributions of every key tile: a warp per tile.
__global__ void __launch_bounds__(256) proxy_pool_kernel(
    const float* __restrict__ st_m, const float* __restrict__ st_u,
    const float* __restrict__ st_w, const float* __restrict__ rowM,
    const float* __restrict__ rowZ, int nb, float inv_b, float* pv, float* pshi, float* pslo) {
  __shared__ float sM[kBlk], sIZ[kBlk];
  const int h = blockIdx.y;
  if (threadIdx.x < kBlk) {
    sM[threadIdx.x] = rowM[h * kBlk + threadIdx.x];
    sIZ[threadIdx.x] = 1.f / rowZ[h * kBlk + threadIdx.x];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= nb) return;
  float su = 0.f, sw = 0.f;
  const size_t base = (static_cast<size_t>(h) * nb + t) * kBlk;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = lane + 32 * k;
    const float e = fast_exp2(st_m[base + r] - sM[r]) * sIZ[r];
    su += st_u[base + r] * e;
    sw += st_w[base + r] * e;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    su += __shfl_xor_sync(0xffffffffu, su, o);
    sw += __shfl_xor_sync(0xffffffffu, sw, o);
  }
  if (lane == 0) {
    pv[static_cast<size_t>(h) * nb + t] = (su + sw) * inv_b;
    pshi[static_cast<size_t>(h) * nb + t] = su * inv_b;
    pslo[static_cast<size_t>(h) * nb + t] = sw * inv_b;
  }
}

struct RouteArgs {
  int nb;
  // 1: this kernel also merges the per-tile statistics into the row maxima and sums and
  // pools them by tile (what proxy_row_stats and proxy_pool do), for N_b <= kFuseRowsNb
  int fuse_rows;
  const float* st_u;
  const float* st_w;
  int n2;  // power of two >= nb (sort width)
  float inv_b, tau, alpha, gamma;
  int kmin_blocks;
  uint32_t flags;
  const float* st_m;
  const float* anc;
  const float* rowM;
  const float* rowZ;
  float* pv;  // read, or written by this kernel when fuse_rows
  const float* pshi;
  const float* pslo;
  float* ps;
  float* cstruct;
  uint8_t* route;
  float* mu;
  int32_t* counts;
  int32_t* near;  // [H][3]: near-threshold route, VS blocks, (PE pairs: pe_index.cu)
  uint8_t* selv;
  uint8_t* sels;
  uint32_t* selbits;  // [H][2*nbw+1] (may be null: crisp_route_static)
};

__device__ float block_sum_1024(float x, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = lane < (blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

__device__ float block_min_1024(float x, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fminf(x, __shfl_xor_sync(0xffffffffu, x, o));
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = lane < (blockDim.x >> 5) ? red[lane] : FLT_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t = fminf(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

__device__ int block_count_1024(int x, int* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  int t = lane < (blockDim.x >> 5) ? red[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

// Larger value wins; equal values go to the lower index.
__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Blocks with p > thr, then (if fewer than kmin) the largest remaining ones until
// k = clip(count, kmin, nb) are kept.  Returns count and k.  Up to kWarpPadNb blocks one
// warp adds the padding; above it the whole block takes one argmax per added block.
constexpr int kWarpPadNb = 256;
__device__ void select_direction(const float* p, uint8_t* sel, int nb, float thr, int kmin,
                                 int* red, float* redf, int* out_c, int* out_k) {
  int local = 0;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) {
    const uint8_t s = p[J] > thr ? 1 : 0;
    sel[J] = s;
    local += s;
  }
  const int c = block_count_1024(local, red);
  const int k = min(max(c, kmin), nb);
  if (k > c && nb <= kWarpPadNb) {
    // The same blocks, picked by one warp without block barriers: lane l holds blocks
    // l, l + 32, ... (at most 8), and each step takes the argmax (score descending, index
    // ascending) of the unselected ones by shuffles.
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      float pv[8];
      uint32_t avail = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int J = lane + 32 * j;
        pv[j] = -1.f;
        if (J < nb && !sel[J]) {
          pv[j] = p[J];
          avail |= 1u << j;
        }
      }
      for (int it = c; it < k; ++it) {
        float bv = -1.f;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (avail & (1u << j)) better(bv, bi, pv[j], lane + 32 * j);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
          better(bv, bi, v2, i2);
        }
        if (bi < 0 || bi >= nb) break;  // every lane holds the same winner
        if ((bi & 31) == lane) {
          avail &= ~(1u << (bi >> 5));
          sel[bi] = 1;
        }
      }
    }
    __syncthreads();
    *out_c = c;
    *out_k = k;
    return;
  }
  for (int it = c; it < k; ++it) {
    float bv = -1.f;
    int bi = 0x7fffffff;
    for (int J = threadIdx.x; J < nb; J += blockDim.x)
      if (!sel[J]) better(bv, bi, p[J], J);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      better(bv, bi, v2, i2);
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
      redf[threadIdx.x >> 5] = bv;
      red[threadIdx.x >> 5] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float fv = redf[0];
      int fi = red[0];
      for (int wi = 1; wi < (int)(blockDim.x >> 5); ++wi) better(fv, fi, redf[wi], red[wi]);
      if (fi >= 0 && fi < nb) sel[fi] = 1;
    }
    __syncthreads();
  }
  *out_c = c;
  *out_k = k;
}


// Keys that sort ascending as (score descending, index ascending); scores are >= 0, so
// their bit patterns order like the values.
__device__ __forceinline__ uint64_t desc_key(float v, int idx) {
  return (static_cast<uint64_t>(0xFFFFFFFFu - __float_as_uint(v)) << 32) |
         static_cast<uint32_t>(idx);
}
__device__ __forceinline__ float key_value(uint64_t k) {
  return __uint_as_float(0xFFFFFFFFu - static_cast<uint32_t>(k >> 32));
}

// Bitonic sort (ascending) of keys for p[lo .. lo+cnt) into keys[0 .. n2); the padding
// keys sort last.  Whole block; ends synchronised.
__device__ void sort_desc(const float* p, int lo, int cnt, uint64_t* keys, int n2) {
  for (int i = threadIdx.x; i < n2; i += blockDim.x)
    keys[i] = i < cnt ? desc_key(p[lo + i], lo + i) : ~0ull;
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Median of the non-anchor scores p[1 .. nb-2] (mean of the two middle values for an
// even count); 0 when N_b <= 2.
__device__ float median_floor(const float* p, int nb, uint64_t* keys, int n2) {
  if (nb <= 2) return 0.f;
  const int cnt = nb - 2;
  sort_desc(p, 1, cnt, keys, n2);
  const float hi = key_value(keys[(cnt - 1) / 2]);
  const float lo = key_value(keys[cnt / 2]);
  __syncthreads();
  return 0.5f * (hi + lo);
}

// FlexPrefill-style budget: the smallest prefix of the scores sorted in descending
// order (ties: lower index) whose fp64 running sum reaches gamma (all blocks if it never
// does), padded to kmin; marks the chosen blocks in sel.
__device__ void select_gamma_cumsum(const float* p, uint8_t* sel, int nb, float gamma, int kmin,
                                    uint64_t* keys, int n2, double* part, int* first,
                                    int* out_c, int* out_k) {
  sort_desc(p, 0, nb, keys, n2);
  const int per = (nb + blockDim.x - 1) / blockDim.x;
  const int b0 = threadIdx.x * per, b1 = min(nb, b0 + per);
  double s = 0.0;
  for (int i = b0; i < b1; ++i) s += static_cast<double>(key_value(keys[i]));
  part[threadIdx.x] = s;
  if (threadIdx.x == 0) *first = nb;
  __syncthreads();
  for (int off = 1; off < static_cast<int>(blockDim.x); off <<= 1) {
    const double t = threadIdx.x >= static_cast<unsigned>(off) ? part[threadIdx.x - off] : 0.0;
    __syncthreads();
    part[threadIdx.x] += t;
    __syncthreads();
  }
  double run = part[threadIdx.x] - s;
  for (int i = b0; i < b1; ++i) {
    run += static_cast<double>(key_value(keys[i]));
    if (run >= static_cast<double>(gamma)) {
      atomicMin(first, i + 1);
      break;
    }
  }
  __syncthreads();
  const int c = *first;
  const int k = min(max(c, kmin), nb);
  for (int i = threadIdx.x; i < nb; i += blockDim.x) sel[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += blockDim.x) sel[static_cast<uint32_t>(keys[i])] = 1;
  __syncthreads();
  *out_c = c;
  *out_k = k;
}

// Short sequences: the route kernel merges the per-tile statistics itself (one launch
// instead of three); the same formulas as proxy_row_stats and proxy_pool.
constexpr int kFuseRowsNb = 256;

__global__ void __launch_bounds__(1024) route_vs_select_kernel(const RouteArgs a) {
  extern __shared__ uint64_t sdyn64[];
  uint64_t* keys = sdyn64;                                  // [n2]
  float* spv = reinterpret_cast<float*>(keys + a.n2);       // [nb]
  float* sps = spv + a.nb;                                  // [nb]
  uint8_t* ssv = reinterpret_cast<uint8_t*>(sps + a.nb);    // [nb]
  uint8_t* sss = ssv + a.nb;                                // [nb]
  __shared__ int red[32];
  __shared__ float redf[32];
  __shared__ double part[1024];
  __shared__ int first;
  __shared__ float sRowM[kBlk], sRowZ[kBlk], sRowIZ[kBlk];
  const int h = blockIdx.x;
  const int nb = a.nb;
  const size_t hb = static_cast<size_t>(h) * nb;
  // C_struct's operands (written by the tile kernel) load first: they do not depend on the
  // row merge below, so their latency overlaps it.
  float anc0 = 0.f, anc1 = 0.f, stm0 = 0.f, stm1 = 0.f, rowm = 0.f, rowz = 1.f;
  if (threadIdx.x < kBlk) {
    const int r = threadIdx.x;
    anc0 = a.anc[(static_cast<size_t>(h) * 2) * kBlk + r];
    stm0 = a.st_m[hb * kBlk + r];
    if (nb > 1) {
      anc1 = a.anc[(static_cast<size_t>(h) * 2 + 1) * kBlk + r];
      stm1 = a.st_m[(hb + nb - 1) * kBlk + r];
    }
    if (!a.fuse_rows) {
      rowm = a.rowM[h * kBlk + r];
      rowz = a.rowZ[h * kBlk + r];
    }
  }

  if (a.fuse_rows) {
    // Row maximum and normaliser of every proxy row over all tiles (8 slices of tiles
    // merged online, then the slices), then the pooled contributions of every tile.
    float* pM = reinterpret_cast<float*>(part);  // [8][128] (part's bytes, unused yet)
    float* pZ = pM + 8 * kBlk;
    const int r = threadIdx.x & (kBlk - 1), slice = threadIdx.x >> 7;
    // Eight tiles' loads are issued before their merge steps; a missing tile is
    // (-FLT_MAX, 0), which adds exactly 0 to Z.
    float M = -FLT_MAX, Z = 0.f;
    for (int t0 = slice; t0 < nb; t0 += 64) {
      float mm[8], ss[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = t0 + 8 * j;
        mm[j] = -FLT_MAX;
        ss[j] = 0.f;
        if (t < nb) {
          const size_t idx = (hb + t) * kBlk + r;
          mm[j] = a.st_m[idx];
          ss[j] = a.st_u[idx] + a.st_w[idx];
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (mm[j] > M) {
          Z = Z * fast_exp2(M - mm[j]) + ss[j];
          M = mm[j];
        } else {
          Z += ss[j] * fast_exp2(mm[j] - M);
        }
      }
    }
    pM[slice * kBlk + r] = M;
    pZ[slice * kBlk + r] = Z;
    __syncthreads();
    if (threadIdx.x < kBlk) {
      float Mt = -FLT_MAX;
      for (int i = 0; i < 8; ++i) Mt = fmaxf(Mt, pM[i * kBlk + r]);
      float Zt = 0.f;
      for (int i = 0; i < 8; ++i) Zt += pZ[i * kBlk + r] * fast_exp2(pM[i * kBlk + r] - Mt);
      sRowM[r] = Mt;
      sRowZ[r] = Zt;
      sRowIZ[r] = 1.f / Zt;
    }
    __syncthreads();
    // p_v of every tile into spv (and global), the slash halves of each tile into the sort
    // keys' bytes (2 * n2 >= 2 * N_b floats, unused until a flag's sort).  A warp takes two
    // tiles per step, all their loads first.
    float* slo = reinterpret_cast<float*>(keys);
    float* shi = slo + nb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < nb; t += 64) {
      float xm[2][4], xu[2][4], xw[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tt = t + 32 * j;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          xm[j][k] = 0.f;
          xu[j][k] = 0.f;
          xw[j][k] = 0.f;
          if (tt < nb) {
            const size_t idx = (hb + tt) * kBlk + lane + 32 * k;
            xm[j][k] = a.st_m[idx];
            xu[j][k] = a.st_u[idx];
            xw[j][k] = a.st_w[idx];
          }
        }
      }
      float su[2] = {0.f, 0.f}, sw[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = lane + 32 * k;
          const float e = fast_exp2(xm[j][k] - sRowM[rr]) * sRowIZ[rr];  // as proxy_pool
          su[j] += xu[j][k] * e;
          sw[j] += xw[j][k] * e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          su[j] += __shfl_xor_sync(0xffffffffu, su[j], o);
          sw[j] += __shfl_xor_sync(0xffffffffu, sw[j], o);
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tt = t + 32 * j;
          if (tt < nb) {
            const float pv = (su[j] + sw[j]) * a.inv_b;
            a.pv[hb + tt] = pv;
            spv[tt] = pv;
            shi[tt] = su[j] * a.inv_b;
            slo[tt] = sw[j] * a.inv_b;
          }
        }
      }
    }
    __syncthreads();
    // p_s[J] = hi part of tile N_b-1-J + lo part of N_b-2-J
    for (int J = threadIdx.x; J < nb; J += blockDim.x) {
      float s = shi[nb - 1 - J];
      if (J <= nb - 2) s += slo[nb - 2 - J];
      sps[J] = s;
      a.ps[hb + J] = s;
    }
    __syncthreads();
  }

  // C_struct = (1/b) sum_r (anchor mass of row r) -- "Core method" step 1, Algorithm 2.
  float c = 0.f;
  if (threadIdx.x < kBlk) {
    const int r = threadIdx.x;
    const float M = a.fuse_rows ? sRowM[r] : rowm;
    const float iz = 1.f / (a.fuse_rows ? sRowZ[r] : rowz);
    c = anc0 * fast_exp2(stm0 - M);
    if (nb > 1) c += anc1 * fast_exp2(stm1 - M);
    c *= iz;
  }
  const float C = block_sum_1024(c, redf) * a.inv_b;
  bool vs = C >= a.tau;
  if (a.flags & CRISP_FLAG_FORCE_VS) vs = true;
  if (a.flags & CRISP_FLAG_FORCE_PE) vs = false;

  // p_v[J] = tile J's vertical mass; p_s[J] = hi part of tile N_b-1-J + lo part of N_b-2-J.
  if (!a.fuse_rows) {
    for (int J = threadIdx.x; J < nb; J += blockDim.x) {
      spv[J] = a.pv[hb + J];
      float s = a.pshi[hb + (nb - 1 - J)];
      if (J <= nb - 2) s += a.pslo[hb + (nb - 2 - J)];
      sps[J] = s;
      a.ps[hb + J] = s;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.cstruct[h] = C;
    a.route[h] = vs ? 1 : 0;
    for (int i = 0; i < 4; ++i) a.counts[h * 4 + i] = 0;
    // near-threshold counts: the route's here, the VS blocks' below, the PE pairs' in the
    // PE mask kernel
    a.near[h * 3 + 0] = fabsf(C - a.tau) <= 1e-3f * fabsf(a.tau) ? 1 : 0;
    a.near[h * 3 + 1] = 0;
    a.near[h * 3 + 2] = 0;
  }
  if (!vs) {
    for (int J = threadIdx.x; J < nb; J += blockDim.x) {
      a.selv[hb + J] = 0;
      a.sels[hb + J] = 0;
    }
    if (threadIdx.x == 0) {
      a.mu[h * 2] = 0.f;
      a.mu[h * 2 + 1] = 0.f;
    }
    return;
  }
  // Noise floor mu_d = max(1 - p_d[0] - p_d[N_b-1], 0)/(N_b-2)  (Algorithm 3), or the
  // median of the non-anchor scores with CRISP_FLAG_MEDIAN_FLOOR.
  float mu_v, mu_s;
  if (a.flags & CRISP_FLAG_MEDIAN_FLOOR) {
    mu_v = median_floor(spv, nb, keys, a.n2);
    mu_s = median_floor(sps, nb, keys, a.n2);
  } else {
    mu_v = nb > 2 ? fmaxf(1.f - spv[0] - spv[nb - 1], 0.f) / (nb - 2) : 0.f;
    mu_s = nb > 2 ? fmaxf(1.f - sps[0] - sps[nb - 1], 0.f) / (nb - 2) : 0.f;
  }
  int cv, kv, cs, ks;
  if (a.flags & CRISP_FLAG_VS_GAMMA_CUMSUM) {
    select_gamma_cumsum(spv, ssv, nb, a.gamma, a.kmin_blocks, keys, a.n2, part, &first, &cv, &kv);
    select_gamma_cumsum(sps, sss, nb, a.gamma, a.kmin_blocks, keys, a.n2, part, &first, &cs, &ks);
  } else {
    select_direction(spv, ssv, nb, a.alpha * mu_v, a.kmin_blocks, red, redf, &cv, &kv);
    __syncthreads();
    select_direction(sps, sss, nb, a.alpha * mu_s, a.kmin_blocks, red, redf, &cs, &ks);
  }
  __syncthreads();
  // Near-threshold blocks: within 1e-3 of alpha * mu_d (floor rule), or of the smallest kept
  // score where the k_min padding (or the gamma-cumsum rule) decided the set.
  const bool gamma_rule = (a.flags & CRISP_FLAG_VS_GAMMA_CUMSUM) != 0;
  const bool pad_v = gamma_rule || kv > cv, pad_s = gamma_rule || ks > cs;
  float kth_v = FLT_MAX, kth_s = FLT_MAX;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) {
    if (ssv[J]) kth_v = fminf(kth_v, spv[J]);
    if (sss[J]) kth_s = fminf(kth_s, sps[J]);
  }
  kth_v = block_min_1024(kth_v, redf);
  kth_s = block_min_1024(kth_s, redf);
  const float thr_v = a.alpha * mu_v, thr_s = a.alpha * mu_s;
  int near = 0;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) {
    bool nv = !gamma_rule && fabsf(spv[J] - thr_v) <= 1e-3f * thr_v;
    bool ns = !gamma_rule && fabsf(sps[J] - thr_s) <= 1e-3f * thr_s;
    nv |= pad_v && fabsf(spv[J] - kth_v) <= 1e-3f * kth_v;
    ns |= pad_s && fabsf(sps[J] - kth_s) <= 1e-3f * kth_s;
    near += (nv ? 1 : 0) + (ns ? 1 : 0);
  }
  near = block_count_1024(near, red);
  for (int J = threadIdx.x; J < nb; J += blockDim.x) {
    a.selv[hb + J] = ssv[J];
    a.sels[hb + J] = sss[J];
  }
  // The two sets as bit words for the row masks (csr.cu): S_v in block order, S_s reversed
  // (bit x = slash block N_b-1-x), so that a row's slash keys are one funnel shift.
  if (a.selbits) {
    const int nbw = (nb + 31) / 32;
    uint32_t* out = a.selbits + static_cast<size_t>(h) * (2 * nbw + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int wd = warp; wd <= nbw; wd += blockDim.x >> 5) {
      const int x = wd * 32 + lane;
      const unsigned wv = __ballot_sync(0xffffffffu, wd < nbw && x < nb && ssv[x] != 0);
      const unsigned ws = __ballot_sync(0xffffffffu, x < nb && sss[nb - 1 - x] != 0);
      if (lane == 0) {
        if (wd < nbw) out[wd] = wv;
        out[nbw + wd] = ws;
      }
    }
  }
  if (threadIdx.x == 0) {
    a.near[h * 3 + 1] = near;
    a.mu[h * 2] = mu_v;
    a.mu[h * 2 + 1] = mu_s;
    a.counts[h * 4 + 0] = cv;
    a.counts[h * 4 + 1] = cs;
    a.counts[h * 4 + 2] = kv;
    a.counts[h * 4 + 3] = ks;
  }
}

}  // namespace

cudaError_t launch_patsearch(crisp_ctx ctx, const Shape& s, const crisp_cfg& cfg,
                             const CUtensorMap& tmQ, const CUtensorMap& tmK, cudaStream_t st) {
  Workspace& w = ctx->ws;
  ProxyArgs a;
  a.n = s.n;
  a.nb = s.nb;
  a.hq = s.hq;
  a.hkv = s.hkv;
  a.group = s.group;
  a.w_sink = cfg.w_sink;
  a.w_local = cfg.w_local;
  // CTAs (one per SM at a time) over (head, chunk of key tiles): the chunk length that
  // minimises waves x (per-CTA setup + tiles per CTA), the setup (barriers, TMEM, the Q
  // tile, the pipeline's fill and drain) costing about kProxySetupTiles tiles.  Long
  // sequences get ~4 waves of long chunks (the tail balanced); short ones one wave of fewer,
  // longer CTAs rather than many CTAs of a few tiles that are mostly setup.
  constexpr int kProxySetupTiles = 6;
  int64_t best_cost = -1;
  int tpc_best = s.nb;
  for (int c = 1; c <= s.nb; ++c) {
    const int tpc = (s.nb + c - 1) / c;
    if (c > 1 && tpc == (s.nb + c - 2) / (c - 1)) continue;  // same chunk length as c - 1
    const int64_t ctas = static_cast<int64_t>(s.H) * ((s.nb + tpc - 1) / tpc);
    const int64_t waves = (ctas + ctx->num_sms - 1) / ctx->num_sms;
    const int64_t cost = waves * (kProxySetupTiles + tpc);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      tpc_best = tpc;
    }
  }
  a.tiles_per_cta = tpc_best;
  const int nchunks = (s.nb + a.tiles_per_cta - 1) / a.tiles_per_cta;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kD));
  a.st_m = w.st_m;
  a.st_u = w.st_u;
  a.st_w = w.st_w;
  a.anc = w.anc;
  a.err = w.err;
  a.timeout_ns = ctx->timeout_ns;
  const bool fuse = s.nb <= kFuseRowsNb;
  {
    PhaseRange range("PatSearch");
    proxy_tile_stats_kernel<<<dim3(s.H, nchunks), kProxyThreads, kProxySmem, st>>>(tmQ, tmK, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!fuse) {
      proxy_row_stats_kernel<<<dim3(kRowSplit, s.H), 256, 0, st>>>(w.st_m, w.st_u, w.st_w, s.nb,
                                                                   w.row_part, w.row_ticket,
                                                                   w.rowM, w.rowZ);
      proxy_pool_kernel<<<dim3((s.nb + 7) / 8, s.H), 256, 0, st>>>(
          w.st_m, w.st_u, w.st_w, w.rowM, w.rowZ, s.nb, 1.f / kBlk, w.pv, w.pshi, w.pslo);
    }
  }
  RouteArgs r;
  r.nb = s.nb;
  r.fuse_rows = fuse ? 1 : 0;
  r.st_u = w.st_u;
  r.st_w = w.st_w;
  r.inv_b = 1.f / kBlk;
  r.tau = cfg.tau_proxy;
  r.alpha = cfg.alpha;
  r.gamma = cfg.gamma;
  r.n2 = 1;
  while (r.n2 < s.nb) r.n2 <<= 1;
  r.kmin_blocks = (cfg.k_min_tokens + kBlk - 1) / kBlk;
  r.flags = cfg.flags;
  r.st_m = w.st_m;
  r.anc = w.anc;
  r.rowM = w.rowM;
  r.rowZ = w.rowZ;
  r.pv = w.pv;
  r.pshi = w.pshi;
  r.pslo = w.pslo;
  r.ps = w.ps;
  r.cstruct = w.cstruct;
  r.route = w.route;
  r.mu = w.mu;
  r.counts = w.counts;
  r.near = w.near;
  r.selv = w.selv;
  r.sels = w.sels;
  r.selbits = w.selbits;
  const size_t dyn = static_cast<size_t>(r.n2) * sizeof(uint64_t) +
                    static_cast<size_t>(s.nb) * (2 * sizeof(float) + 2);
  PhaseRange range("VS");
  route_vs_select_kernel<<<s.H, 1024, dyn, st>>>(r);
  return cudaGetLastError();
}

int patsearch_launches(int nb) { return nb <= kFuseRowsNb ? 2 : 4; }

cudaError_t init_patsearch_attributes() {
  cudaError_t e = cudaFuncSetAttribute(proxy_tile_stats_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kProxySmem));
  if (e != cudaSuccess) return e;
  // nb <= 8192: 64 KB of sort keys + 80 KB of scores and flags (+ 8.4 KB static)
  return cudaFuncSetAttribute(route_vs_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              160 * 1024);
}

}  // namespace crisp

// ---------------------------------------------------------------------------------------
// crisp_route_static: the routing step with no device allocation.
//
// Some callers cannot call cudaMalloc: a plug-in running inside a host engine that owns
// every byte of device memory through its own pool, or a latency-critical loop where the
// implicit device synchronisation of an allocation is not acceptable.  This entry point
// runs the same PatSearch kernels as crisp_select, but its scratch is the fixed array
// below, which lives in every GPU's memory from the time the library is loaded until
// the process exits.  It holds at most kStaticMaxHeads query heads and
// kStaticMaxTiles (query head, key tile) pairs, i.e. batch*hq*(n/128) <= 8192: for
// example 32 heads at 32k tokens or 8 heads at 128k tokens.  About 15 MB.
// ---------------------------------------------------------------------------------------
#include <mutex>

namespace crisp {
namespace {

constexpr int64_t kStaticMaxTiles = 8192;
constexpr int64_t kStaticMaxHeads = 128;

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
constexpr size_t kOffStM = 0;
constexpr size_t kOffStU = kOffStM + align256(sizeof(float) * kStaticMaxTiles * kBlk);
constexpr size_t kOffStW = kOffStU + align256(sizeof(float) * kStaticMaxTiles * kBlk);
constexpr size_t kOffAnc = kOffStW + align256(sizeof(float) * kStaticMaxTiles * kBlk);
constexpr size_t kOffRowM = kOffAnc + align256(sizeof(float) * kStaticMaxHeads * 2 * kBlk);
constexpr size_t kOffRowZ = kOffRowM + align256(sizeof(float) * kStaticMaxHeads * kBlk);
constexpr size_t kOffPv = kOffRowZ + align256(sizeof(float) * kStaticMaxHeads * kBlk);
constexpr size_t kOffPshi = kOffPv + align256(sizeof(float) * kStaticMaxTiles);
constexpr size_t kOffPslo = kOffPshi + align256(sizeof(float) * kStaticMaxTiles);
constexpr size_t kOffPs = kOffPslo + align256(sizeof(float) * kStaticMaxTiles);
constexpr size_t kOffMu = kOffPs + align256(sizeof(float) * kStaticMaxTiles);
constexpr size_t kOffCounts = kOffMu + align256(sizeof(float) * kStaticMaxHeads * 2);
constexpr size_t kOffNear = kOffCounts + align256(sizeof(int32_t) * kStaticMaxHeads * 4);
constexpr size_t kOffSelv = kOffNear + align256(sizeof(int32_t) * kStaticMaxHeads * 3);
constexpr size_t kOffSels = kOffSelv + align256(kStaticMaxTiles);
constexpr size_t kOffPart = kOffSels + align256(kStaticMaxTiles);
constexpr size_t kOffTicket = kOffPart + align256(sizeof(float2) * kStaticMaxHeads * kRowSplit * kBlk);
constexpr size_t kOffErr = kOffTicket + align256(sizeof(int) * kStaticMaxHeads);
constexpr size_t kStaticBytes = kOffErr + 256;

// The scratch of crisp_route_static.  In host code this name is only a stand-in: the
// device address comes from cudaGetSymbolAddress (below) and is what the kernels get.
static __device__ __align__(256) unsigned char g_route_scratch[kStaticBytes];

struct StaticSetup {
  bool done = false;
  crisp_status status = CRISP_OK;
  unsigned char* scratch = nullptr;  // device address of g_route_scratch on this device
  EncodeTiledFn encode = nullptr;
  int num_sms = 0;
};
constexpr int kMaxDevices = 64;
StaticSetup g_static_setup[kMaxDevices];
std::mutex g_static_mu;

// Once per device, with that device current: resolve the scratch address and the other
// per-device state.  Allocates nothing.  Only a completed setup is kept (and the permanent
// answer for a device of another architecture); a failure of any step leaves the device
// unset, so the next call tries again.
crisp_status static_setup(int dev, StaticSetup** out) {
  if (dev < 0 || dev >= kMaxDevices) return CRISP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_static_mu);
  StaticSetup& s = g_static_setup[dev];
  *out = &s;
  if (s.done) return s.status;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return CRISP_ERR_CUDA;
  }
  if (major != 10 || minor != 3) {  // the kernels are built for sm_103a only
    s.status = CRISP_ERR_UNSUPPORTED;
    s.done = true;
    return s.status;
  }
  unsigned char* scratch = nullptr;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&scratch), g_route_scratch) != cudaSuccess ||
      !scratch ||
      cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn || init_patsearch_attributes() != cudaSuccess) {
    cudaGetLastError();
    return CRISP_ERR_CUDA;
  }
  s.scratch = scratch;
  s.encode = reinterpret_cast<EncodeTiledFn>(fn);
  s.num_sms = sms;
  s.status = CRISP_OK;
  s.done = true;
  return CRISP_OK;
}

bool static_map(EncodeTiledFn encode, CUtensorMap* map, const void* base, int64_t rows) {
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(kD) * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace
}  // namespace crisp

extern "C" crisp_status crisp_route_static(const crisp_dims* dims, const void* Q, const void* K,
                                           const crisp_cfg* cfg, uint8_t* route_vs,
                                           float* c_struct, uint32_t* status, void* stream) {
  using namespace crisp;
  if (!dims || !cfg || !Q || !K || !route_vs || !c_struct || !status)
    return CRISP_ERR_INVALID_ARG;
  // The shape and parameter rules of crisp_select, then the scratch limits.
  crisp_status chk = check_dims(dims);
  if (chk == CRISP_OK) chk = check_cfg(cfg);
  if (chk != CRISP_OK) return chk;
  if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K)) & 15u)
    return CRISP_ERR_INVALID_ARG;
  const Shape s = make_shape(*dims);
  // Sizes beyond the static scratch are rejected before any work is queued.
  if (s.H > kStaticMaxHeads || static_cast<int64_t>(s.H) * s.nb > kStaticMaxTiles)
    return CRISP_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CRISP_ERR_CUDA;
  StaticSetup* su = nullptr;
  crisp_status st = static_setup(dev, &su);
  if (st != CRISP_OK) return st;

  // A context on the stack whose workspace points into the static scratch, except the
  // two outputs, which are the caller's.
  crisp_ctx_s c;
  c.device = dev;
  c.num_sms = su->num_sms;
  c.encode = su->encode;
  Workspace& w = c.ws;
  unsigned char* b = su->scratch;
  w.st_m = reinterpret_cast<float*>(b + kOffStM);
  w.st_u = reinterpret_cast<float*>(b + kOffStU);
  w.st_w = reinterpret_cast<float*>(b + kOffStW);
  w.anc = reinterpret_cast<float*>(b + kOffAnc);
  w.rowM = reinterpret_cast<float*>(b + kOffRowM);
  w.rowZ = reinterpret_cast<float*>(b + kOffRowZ);
  w.pv = reinterpret_cast<float*>(b + kOffPv);
  w.pshi = reinterpret_cast<float*>(b + kOffPshi);
  w.pslo = reinterpret_cast<float*>(b + kOffPslo);
  w.ps = reinterpret_cast<float*>(b + kOffPs);
  w.mu = reinterpret_cast<float*>(b + kOffMu);
  w.counts = reinterpret_cast<int32_t*>(b + kOffCounts);
  w.near = reinterpret_cast<int32_t*>(b + kOffNear);
  w.selv = b + kOffSelv;
  w.sels = b + kOffSels;
  w.row_part = reinterpret_cast<float2*>(b + kOffPart);
  w.row_ticket = reinterpret_cast<int*>(b + kOffTicket);
  w.err = reinterpret_cast<uint32_t*>(b + kOffErr);
  w.cstruct = c_struct;
  w.route = route_vs;

  CUtensorMap tmQ, tmK;
  if (!static_map(su->encode, &tmQ, Q, static_cast<int64_t>(s.H) * s.n) ||
      !static_map(su->encode, &tmK, K, static_cast<int64_t>(s.Hkv) * s.n))
    return CRISP_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // The error word and the row-statistics tickets are the only scratch that must start at
  // zero (the tickets also return to zero after every use); every other scratch value is
  // written before it is read.
  if (cudaMemsetAsync(w.err, 0, sizeof(uint32_t), cs) != cudaSuccess ||
      cudaMemsetAsync(w.row_ticket, 0, sizeof(int) * s.H, cs) != cudaSuccess)
    return CRISP_ERR_CUDA;
  if (launch_patsearch(&c, s, *cfg, tmQ, tmK, cs) != cudaSuccess) return CRISP_ERR_CUDA;
  if (cudaMemcpyAsync(status, w.err, sizeof(uint32_t), cudaMemcpyDeviceToDevice, cs) !=
      cudaSuccess)
    return CRISP_ERR_CUDA;
  return CRISP_OK;
}
