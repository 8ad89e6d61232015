// pe_index.cu -- PEIndex (GlobalAdaptive) selection for heads routed PE.
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top), "Method step details" step 3 and Algorithm 4
// (PEIndex) under "Figures and tables": pool all queries and keys by block, softmax the
// pooled scores, normalise and flatten, sort, and keep the top pairs until their
// cumulative mass reaches gamma ("Prerequisites", the cumulative coverage rule).
//
// The pooled softmax runs on the tensor cores (pe_prob_kernel: the block means as bf16
// hi/lo pairs, three MMA chains per tile, fp32 accumulate in TMEM) and writes v directly.
// The sort is a radix select on the fp32 bit patterns of the (positive) flattened scores
// with fixed-point mass per digit: four 8-bit passes find the threshold value T with
// mass(v > T) < gamma <= mass(v >= T); items equal to T are then taken in flat-index
// order (I*N_b + K) until the running mass reaches gamma.  Every PE row also gets its
// diagonal pair, so that no query block is left without keys.
#include <cuda_bf16.h>

#include <algorithm>
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace crisp {
namespace {

// ---------------------------------------------------------------- block means
// The pooled logits Qbar_I . Kbar_K / sqrt(d) are formed on the tensor cores from bf16
// pairs: x = hi + lo with hi = bf16(x) and lo = bf16(x - hi) (16 significant bits), and
// Qbar . Kbar ~ hi_q.hi_k + hi_q.lo_k + lo_q.hi_k (the dropped lo.lo term and the split's
// residue are ~2^-16 of |Qbar||Kbar|).  Qbar is scaled by log2(e)/sqrt(d) before the split,
// so the product is the logit in base 2.  Layout: a [2][rows][128] bf16 plane pair
// (hi rows first, then lo rows), rows = heads x N_b.
__device__ __forceinline__ void split_store(uint16_t* hi_plane, size_t lo_offset, size_t idx,
                                            float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
  hi_plane[idx] = __bfloat16_as_ushort(hi);
  hi_plane[lo_offset + idx] = __bfloat16_as_ushort(lo);
}

// Block means of the PE heads' queries and of the KV heads that serve them, one launch:
// grid (H + Hkv, N_b) (heads on x: H + Hkv may pass the 65535 limit of y).  y < H: Qbar[y][I][:] = mean of the 128 rows of query block I of a
// PE head, times log2(e)/sqrt(d); y >= H: Kbar[y-H][I][:] for a KV head with at least one
// PE query head.  Both are split into bf16 pairs.
__global__ void __launch_bounds__(128) pe_pool_kernel(const uint16_t* __restrict__ Q,
                                                      const uint16_t* __restrict__ K,
                                                      const uint8_t* __restrict__ route, int n,
                                                      int nb, int H, int hq, int hkv, int group,
                                                      int Hkv, float q_scale, uint16_t* qs,
                                                      uint16_t* ks, int* pe_list) {
  const int y = blockIdx.x, I = blockIdx.y;
  // the PE head list is rebuilt by pe_radix_init_kernel, which runs after this kernel
  if (y == 0 && I == 0 && threadIdx.x == 0) pe_list[0] = 0;
  const bool is_q = y < H;
  const uint16_t* src;
  if (is_q) {
    if (route[y]) return;
    src = Q + (static_cast<size_t>(y) * n + static_cast<size_t>(I) * kBlk) * kD;
  } else {
    const int hk = y - H;
    const int bidx = hk / hkv, kvh = hk % hkv;
    bool any_pe = false;
    for (int g = 0; g < group; ++g) any_pe |= route[bidx * hq + kvh * group + g] == 0;
    if (!any_pe) return;
    src = K + (static_cast<size_t>(hk) * n + static_cast<size_t>(I) * kBlk) * kD;
  }
  __shared__ float part[8][kD];
  const int rg = threadIdx.x >> 4;          // row group 0..7
  const int cc = (threadIdx.x & 15) * 8;    // 8 columns
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int rr = rg; rr < kBlk; rr += 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(rr) * kD + cc);
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
  if (is_q)
    split_store(qs, static_cast<size_t>(H) * nb * kD,
                (static_cast<size_t>(y) * nb + I) * kD + threadIdx.x, s * (1.f / kBlk) * q_scale);
  else
    split_store(ks, static_cast<size_t>(Hkv) * nb * kD,
                (static_cast<size_t>(y - H) * nb + I) * kD + threadIdx.x, s * (1.f / kBlk));
}

// ---------------------------------------------------------------- pooled softmax
// v[I][K] = softmax_{K <= I}(Qbar_I . Kbar_K / sqrt(d)) / N_b for one PE head and one tile
// of 128 query blocks I (row tile t), written row-major into the head's N_b x N_b square.
//
// One CTA per (head, row tile), longest rows first.  Warp 0 loads the row tile's Qbar pair
// once and streams the Kbar pairs of key tiles 0..t twice through a 2-stage ring (TMA, one
// 3-D copy per 32 KB plane tile); warp 1 issues three bf16 MMA chains per key tile
// (hi.hi + hi.lo + lo.hi, M = N = 128, K = 128) into one of two TMEM S buffers; warps 2-9
// are two warpgroups that take alternate key tiles, thread <-> row (TMEM lane).  Pass 0
// (the first t+1 jobs) keeps each row's running maximum and sum of 2^(s - m); the two
// warpgroups then merge their partial (m, sum) per row through shared memory; pass 1 (the
// next t+1 jobs, same MMAs) writes 2^(s - M) / (Z N_b).  Each epilogue warp stages its 32
// rows 16 keys at a time in shared memory and lane 0 hands the box to a TMA store (3-D
// map {N_b, N_b, heads}: rows and keys past N_b are clipped by the copy); the diagonal
// tile's keys K > I are written as 0 (never read).  Without the map (N_b % 4 != 0: row
// pitch not a multiple of 16 bytes) the warp stores through a pitch-17 staging tile,
// 16 consecutive keys of two rows per instruction, keys K <= I only.
constexpr int kPeThreads = 320;
constexpr int kPeBStages = 2;
constexpr uint32_t kIdescPe = idesc_bf16_f32(128, 128, false, false);
constexpr int kPeStagePerWarp = 32 * 17;   // floats (store path without TMA)
constexpr int kPeBoxBytes = 32 * 16 * 4;    // one TMA store box: 32 rows x 16 keys
constexpr size_t kPeStageBytes = 8 * 2 * kPeBoxBytes;  // two boxes per epilogue warp
constexpr size_t kPeSmem = 2 * kTileBytes + kPeBStages * 2 * kTileBytes + kPeStageBytes +
                           2 * kBlk * sizeof(float2) + 256;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort, uint64_t tmo) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err, abort, tmo) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                           uint64_t tmo) {
  volatile int never = 0;
  mbar_wait(bar, parity, err, &never, tmo);
}

struct PeProbArgs {
  const uint8_t* route;
  int nb, nt, hq, hkv, group;
  int q_lo_rows;  // row offset of the lo plane in the Qbar map (heads x N_b)
  int k_lo_rows;  // same for the Kbar map
  float inv_nb;
  int tma_out;  // 1: v leaves through TMA stores (tmO valid: N_b % 4 == 0)
  float* pev;
  uint32_t* err;
  uint64_t timeout_ns;
};

__global__ void __launch_bounds__(kPeThreads, 1)
    pe_prob_kernel(const __grid_constant__ CUtensorMap tmQs,
                   const __grid_constant__ CUtensorMap tmKs,
                   const __grid_constant__ CUtensorMap tmO, const PeProbArgs a) {
  const int h = blockIdx.x;
  if (a.route[h]) return;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrRange);
    return;
  }
  const int t = a.nt - 1 - static_cast<int>(blockIdx.y);  // row tile
  const int T = t + 1;                                    // key tiles 0..t
  const int jobs = 2 * T;                                 // pass 0, then pass 1
  uint8_t* sA = smem_raw;                                 // Qbar hi | lo
  uint8_t* sB = sA + 2 * kTileBytes;                      // per stage: Kbar hi | lo
  float* stage = reinterpret_cast<float*>(sB + kPeBStages * 2 * kTileBytes);
  float2* xchg = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(stage) + kPeStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(xchg + 2 * kBlk);
  uint64_t* a_full = bars;
  uint64_t* b_full = bars + 1;   // [kPeBStages]
  uint64_t* b_empty = bars + 3;  // [kPeBStages]
  uint64_t* s_full = bars + 5;   // [2]
  uint64_t* s_free = bars + 7;   // [2]
  uint64_t* x_ready = bars + 9;  // both warpgroups' pass-0 row statistics are in xchg
  uint64_t* drain = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = (h / a.hq) * a.hkv + (h % a.hq) / a.group;
  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    for (int s = 0; s < kPeBStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(x_ready, 256);
    mbar_init(drain, 1);
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
      tma_prefetch_desc(&tmQs);
      tma_prefetch_desc(&tmKs);
      const int qrow = h * a.nb + t * kBlk;
      mbar_arrive_expect_tx(a_full, 2 * kTileBytes);
      tma_load_3d(sA, &tmQs, a_full, 0, qrow, 0);
      tma_load_3d(sA + kTileBytes, &tmQs, a_full, 0, a.q_lo_rows + qrow, 0);
      int issued = 0;
      for (int j = 0; j < jobs; ++j) {
        const int s = j & 1;
        if (j >= kPeBStages &&
            !mbar_wait(&b_empty[s], ((j >> 1) + 1) & 1, a.err, abort_flag, tmo))
          break;
        const int krow = hk * a.nb + (j < T ? j : j - T) * kBlk;
        uint8_t* dst = sB + s * 2 * kTileBytes;
        mbar_arrive_expect_tx(&b_full[s], 2 * kTileBytes);
        tma_load_3d(dst, &tmKs, &b_full[s], 0, krow, 0);
        tma_load_3d(dst + kTileBytes, &tmKs, &b_full[s], 0, a.k_lo_rows + krow, 0);
        ++issued;
      }
      drain_wait(a_full, 0, a.err, tmo);
      for (int j = max(0, issued - kPeBStages); j < issued; ++j)
        drain_wait(&b_full[j & 1], (j >> 1) & 1, a.err, tmo);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (mbar_wait(a_full, 0, a.err, abort_flag, tmo)) {
        const uint32_t a_hi = smem_u32(sA), a_lo = a_hi + kTileBytes;
        for (int j = 0; j < jobs; ++j) {
          const int s = j & 1;  // B stage and S buffer
          if (!mbar_wait(&b_full[s], (j >> 1) & 1, a.err, abort_flag, tmo)) break;
          if (j >= 2 && !mbar_wait(&s_free[s], ((j >> 1) + 1) & 1, a.err, abort_flag, tmo))
            break;
          tc_fence_after();
          const uint32_t b_hi = smem_u32(sB + s * 2 * kTileBytes), b_lo = b_hi + kTileBytes;
          const uint32_t d = tmem + s * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
            umma_bf16(d, sdesc_sw128(a_hi + off, 16, 1024), sdesc_sw128(b_hi + off, 16, 1024),
                      kIdescPe, kk > 0 ? 1u : 0u);
            umma_bf16(d, sdesc_sw128(a_hi + off, 16, 1024), sdesc_sw128(b_lo + off, 16, 1024),
                      kIdescPe, 1u);
            umma_bf16(d, sdesc_sw128(a_lo + off, 16, 1024), sdesc_sw128(b_hi + off, 16, 1024),
                      kIdescPe, 1u);
          }
          umma_commit(&s_full[s]);
          umma_commit(&b_empty[s]);
        }
      }
      umma_commit(drain);
      drain_wait(drain, 0, a.err, tmo);
    }
  } else {
    const int e = (warp - 2) >> 2;  // warpgroup: jobs j with (j & 1) == e, S buffer e
    const int q = warp & 3;         // TMEM lane quarter
    const int r = q * 32 + lane;
    const int I = t * kBlk + r;
    const bool row_ok = I < a.nb;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + e * 128;
    bool ok = true;
    float m_run = -FLT_MAX, z = 0.f;
    for (int j = e; j < T; j += 2) {
      if (!warp_wait(&s_full[e], (j >> 1) & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[128];
      tmem_ld128(taddr, v);
      tc_fence_before();
      mbar_arrive(&s_free[e]);
      const int lim = row_ok ? (j == t ? r : kBlk - 1) : -1;  // keys c <= lim are in the row
      if (lim == kBlk - 1) {
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = -FLT_MAX;
#pragma unroll
        for (int c = 0; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(v[c]));
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float mn = fmaxf(m_run, mt);
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x0, x1;
          fadd2(x0, x1, __uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]), -mn, -mn);
          fadd2(sa, sb, sa, sb, fast_exp2(x0), fast_exp2(x1));
        }
        z = z * fast_exp2(m_run - mn) + (sa + sb);
        m_run = mn;
      } else if (lim >= 0) {
        float mt = -FLT_MAX;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c <= lim) mt = fmaxf(mt, __uint_as_float(v[c]));
        const float mn = fmaxf(m_run, mt);
        float sa = 0.f;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c <= lim) sa += fast_exp2(__uint_as_float(v[c]) - mn);
        z = z * fast_exp2(m_run - mn) + sa;
        m_run = mn;
      }
    }
    // Merge the two warpgroups' row statistics (every epilogue thread arrives once).
    xchg[e * kBlk + r] = make_float2(m_run, z);
    mbar_arrive(x_ready);
    ok = warp_wait(x_ready, 0, a.err, abort_flag, tmo) && ok;
    if (ok) {
      const float2 p0 = xchg[r], p1 = xchg[kBlk + r];
      const float M = fmaxf(p0.x, p1.x);
      const float Z = p0.y * fast_exp2(p0.x - M) + p1.y * fast_exp2(p1.x - M);
      const float inv = a.inv_nb / Z;
      float* out = a.pev + static_cast<size_t>(h) * a.nb * a.nb;
      const int half = lane >> 4, col = lane & 15;
      // TMA path: per warp two 2 KB boxes [32 rows][16 keys] in the 64-byte swizzled layout
      // (16-byte chunk i of row rr at chunk i ^ ((rr >> 1) & 3)), stored by lane 0.
      uint8_t* box = reinterpret_cast<uint8_t*>(stage) + (warp - 2) * 2 * kPeBoxBytes;
      // Fallback: a [32 rows][16 keys] tile with row pitch 17, stored by the whole warp.
      float* st = stage + (warp - 2) * kPeStagePerWarp;
      int nbox = 0;
      for (int j = T + ((T & 1) != e ? 1 : 0); j < jobs; j += 2) {
        if (!warp_wait(&s_full[e], (j >> 1) & 1, a.err, abort_flag, tmo)) break;
        tc_fence_after();
        uint32_t v[128];
        tmem_ld128(taddr, v);
        tc_fence_before();
        mbar_arrive(&s_free[e]);
        const int kt = j - T;
        const int lim = kt == t ? r : kBlk - 1;  // keys c <= lim are in the row (diagonal tile)
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          float y[16];
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            float x0, x1;
            fadd2(x0, x1, __uint_as_float(v[c16 * 16 + c]), __uint_as_float(v[c16 * 16 + c + 1]),
                  -M, -M);
            ffma2(y[c], y[c + 1], fast_exp2(x0), fast_exp2(x1), inv, inv, 0.f, 0.f);
            if (c16 * 16 + c > lim) y[c] = 0.f;
            if (c16 * 16 + c + 1 > lim) y[c + 1] = 0.f;
          }
          if (a.tma_out) {
            uint8_t* b = box + (nbox & 1) * kPeBoxBytes;
            if (lane == 0 && nbox >= 2) bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<float4*>(b + lane * 64 + 16 * (i ^ ((lane >> 1) & 3))) =
                  make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmO, b, kt * kBlk + c16 * 16, t * kBlk + q * 32, h);
              bulk_commit_group();
            }
            ++nbox;
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) st[lane * 17 + c] = y[c];
            __syncwarp();
            // lanes 0-15 store 16 keys of row rr, lanes 16-31 those of row rr + 1
            const int K = kt * kBlk + c16 * 16 + col;
#pragma unroll 4
            for (int rr = 0; rr < 32; rr += 2) {
              const int row = rr + half;
              const int Ir = t * kBlk + q * 32 + row;
              const float yv = st[row * 17 + col];
              if (Ir < a.nb && K <= Ir) out[static_cast<size_t>(Ir) * a.nb + K] = yv;
            }
            __syncwarp();
          }
        }
      }
      if (lane == 0 && nbox > 0) bulk_wait_group<0>();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------- radix select
__global__ void pe_radix_init_kernel(const uint8_t* __restrict__ route, PeState* pe,
                                     unsigned long long* hist_cnt,
                                     unsigned long long* hist_mass, int* pe_list) {
  const int h = blockIdx.x;
  if (threadIdx.x == 0) {
    PeState s{};
    pe[h] = s;
    // the list of PE heads that the histogram, tie-count and mask kernels walk (its order
    // does not matter: every item's arithmetic is its own, and the bin sums are integers)
    if (!route[h]) pe_list[1 + atomicAdd(&pe_list[0], 1)] = h;
  }
  hist_cnt[h * 256 + threadIdx.x] = 0;
  hist_mass[h * 256 + threadIdx.x] = 0ull;
}

// A non-negative fp32 mass in units of 2^-56 from its bits (integer arithmetic only): the
// value is mant * 2^(e - 150), so the fixed-point number is mant shifted by e - 94; exact
// whenever m * 2^56 is an integer (m >= 2^-33), otherwise rounded half up; 0 below 2^-126.
// Masses here are at most ~1; anything from 2^7 up saturates at 2^63.
__device__ __forceinline__ unsigned long long mass_fixed(float m) {
  const uint32_t b = __float_as_uint(m) & 0x7FFFFFFFu;
  const int e = static_cast<int>(b >> 23);
  if (e == 0) return 0ull;
  const unsigned long long mant = (b & 0x7FFFFFu) | 0x800000u;
  const int sh = e - 94;
  if (sh > 39) return 1ull << 63;
  if (sh >= 0) return mant << sh;
  if (sh < -24) return 0ull;
  return (mant + (1ull << (-sh - 1))) >> (-sh);
}

// The histogram, tie-count and mask kernels walk items of 8 PE rows (a warp per row) of
// the listed PE heads with a grid of resident CTAs (the occupancy of each kernel, found
// once at context creation), longest rows first across all heads: a grid over every
// (head, row chunk) launched as many CTAs that only returned for the VS heads (at 512k,
// 12288 of 16384), at ~1.5 ns each.
constexpr int kPeRowsPerItem = 8;
int g_hist_ctas_per_sm = 1, g_eqcount_ctas_per_sm = 1, g_mask_ctas_per_sm = 1;

__device__ __forceinline__ int pe_items(const int* pe_list, int nb) {
  return pe_list[0] * ((nb + kPeRowsPerItem - 1) / kPeRowsPerItem);
}
// Item -> (head, first row): chunks in descending order, the heads interleaved.
__device__ __forceinline__ void pe_item(const int* pe_list, int nb, int item, int& h, int& I0) {
  const int npe = pe_list[0];
  const int chunks = (nb + kPeRowsPerItem - 1) / kPeRowsPerItem;
  h = pe_list[1 + item % npe];
  I0 = (chunks - 1 - item / npe) * kPeRowsPerItem;
}

__global__ void __launch_bounds__(256) pe_hist_kernel(const float* __restrict__ pev,
                                                      const PeState* __restrict__ pe,
                                                      const int* __restrict__ pe_list, int nb,
                                                      int shift, unsigned long long* hist_cnt,
                                                      unsigned long long* hist_mass) {
  // Per-warp histograms with native fp32 shared-memory atomics (later passes see many
  // values in few bins, so one shared copy serialises the warps); the CTA's partial
  // masses (each at most a few percent of the total) go to global memory in fixed point.
  __shared__ unsigned int scnt[8][256];
  __shared__ float smass[8][256];
  const int wp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = pe_items(pe_list, nb);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    int h, I0;
    pe_item(pe_list, nb, item, h, I0);
    const PeState st = pe[h];
    if (st.select_all) continue;  // the same for the whole CTA
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
    // A warp per row (its own histogram copy, so no cross-warp contention): four coalesced
    // float4 loads in flight per lane, the warps of a CTA on neighbouring rows.
    const int I = I0 + wp;
    if (I < nb) {
      const float* row = pev + (static_cast<size_t>(h) * nb + I) * nb;
      const int len = I + 1;
      if ((nb & 3) == 0) {
        // rows start on 16-byte boundaries
        const float4* row4 = reinterpret_cast<const float4*>(row);
        const int n4 = len >> 2;
        int q = lane;
        for (; q + 96 < n4; q += 128) {
          const float4 x = row4[q], y = row4[q + 32], z = row4[q + 64], u = row4[q + 96];
          take(x.x); take(x.y); take(x.z); take(x.w);
          take(y.x); take(y.y); take(y.z); take(y.w);
          take(z.x); take(z.y); take(z.z); take(z.w);
          take(u.x); take(u.y); take(u.z); take(u.w);
        }
        for (; q < n4; q += 32) {
          const float4 x = row4[q];
          take(x.x); take(x.y); take(x.z); take(x.w);
        }
        const int K = (n4 << 2) + lane;
        if (K < len) take(row[K]);
      } else {
        for (int K = lane; K < len; K += 32) take(row[K]);
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
    float m = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      c += scnt[w][threadIdx.x];
      m += smass[w][threadIdx.x];
    }
    if (c) {
      atomicAdd(&hist_cnt[h * 256 + threadIdx.x], static_cast<unsigned long long>(c));
      atomicAdd(&hist_mass[h * 256 + threadIdx.x], mass_fixed(m));
    }
    __syncthreads();  // the copies are read before the next item clears them
  }
}

// gamma in mass units.
__device__ __forceinline__ unsigned long long gamma_fixed(float gamma) {
  return mass_fixed(gamma);
}

// The digit pick of one radix pass, by all threads of a CTA (blockDim.x >= 256): thread
// t < 256 holds bin 255 - t (count c, fixed-point mass m), so the bins run from the top
// down with the threads.  The masses are non-negative, so the running sum from the top
// never decreases and exactly one non-empty bin takes it from below the remaining target
// rem to rem or above (the bin at which a walk from the top bin down stops); that bin
// reports itself.  bin = -1: no bin reaches rem.  Ends synchronised.
struct DigitPick {
  unsigned long long wsum[8];  // mass per 32 bins
  int bin;
  unsigned long long above;    // mass of the bins above the chosen one
  unsigned long long cnt;      // items in the chosen bin
};

__device__ void pick_crossing(int t, unsigned long long c, unsigned long long m,
                              unsigned long long rem, DigitPick* dp) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long incl = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (t < 256 && lane == 31) dp->wsum[w] = incl;
  if (threadIdx.x == 0) dp->bin = -1;
  __syncthreads();
  if (t < 256) {
    unsigned long long excl = incl - m;
    for (int k = 0; k < w; ++k) excl += dp->wsum[k];
    if (c && excl < rem && m >= rem - excl) {
      dp->bin = 255 - t;
      dp->above = excl;
      dp->cnt = c;
    }
  }
  __syncthreads();
}

// The state after a pass's digit; pass 3 also fixes the threshold and how many of the items
// equal to it the cut takes (ceil of the remaining mass over the threshold value, at least
// one, at most all of them).
__device__ void finish_digit(PeState& st, int pass, float gamma, int chosen,
                             unsigned long long above, unsigned long long cnt) {
  const int shift = 24 - 8 * pass;
  st.above += above;
  st.prefix |= static_cast<uint32_t>(chosen) << shift;
  st.decided |= 255u << shift;
  if (pass == 3) {
    st.thresh = st.prefix;
    st.count_eq = cnt;
    const double vt = static_cast<double>(__uint_as_float(st.thresh));
    const double rem2 = static_cast<double>(gamma_fixed(gamma) - st.above) * 0x1p-56;
    unsigned long long need = st.count_eq;
    if (vt > 0.0) {
      const double q = ceil(rem2 / vt);
      need = q < 1.0 ? 1ull : static_cast<unsigned long long>(q);
    }
    st.need_eq = need < st.count_eq ? need : st.count_eq;
  }
}

// Picks a pass's digit for every PE head (one CTA of 256 threads per head, thread t on bin
// 255 - t), then clears the head's histogram for the next pass.
__global__ void __launch_bounds__(256) pe_digit_kernel(const uint8_t* __restrict__ route,
                                                       int pass, float gamma, PeState* pe,
                                                       unsigned long long* hist_cnt,
                                                       unsigned long long* hist_mass) {
  __shared__ DigitPick dp;
  const int h = blockIdx.x, t = threadIdx.x;
  const unsigned long long c = hist_cnt[h * 256 + 255 - t], m = hist_mass[h * 256 + 255 - t];
  if (route[h] == 0) {
    PeState st = pe[h];  // the same for the whole CTA
    if (!st.select_all) {
      pick_crossing(t, c, m, gamma_fixed(gamma) - st.above, &dp);
      if (t == 0) {
        int chosen = dp.bin;
        unsigned long long above = dp.above, cnt = dp.cnt;
        if (chosen < 0) {
          // no bin reaches the target (the triangle's rounded mass falls short of gamma):
          // the first pass takes the whole triangle, a later one the lowest non-empty bin
          unsigned long long total = 0;
          for (int k = 0; k < 8; ++k) total += dp.wsum[k];
          for (int bin = 0; bin < 256 && chosen < 0; ++bin)
            if (hist_cnt[h * 256 + bin]) chosen = bin;
          if (pass == 0 || chosen < 0) {
            st.select_all = 1;
          } else {
            above = total - hist_mass[h * 256 + chosen];
            cnt = hist_cnt[h * 256 + chosen];
          }
        }
        if (!st.select_all) finish_digit(st, pass, gamma, chosen, above, cnt);
        pe[h] = st;
      }
    }
  }
  __syncthreads();
  hist_cnt[h * 256 + t] = 0;
  hist_mass[h * 256 + t] = 0ull;
}

// Number of items equal to the threshold in each PE row (for flat-order tie ranks): a warp
// per row, four coalesced float4 loads in flight per lane.
__global__ void __launch_bounds__(256) pe_eqcount_kernel(const float* __restrict__ pev,
                                                         const PeState* __restrict__ pe,
                                                         const int* __restrict__ pe_list,
                                                         int nb, int64_t* eq_off) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = pe_items(pe_list, nb);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    int h, I0;
    pe_item(pe_list, nb, item, h, I0);
    const PeState st = pe[h];
    if (st.select_all || st.need_eq >= st.count_eq) continue;  // no tie ranks needed
    const int I = I0 + warp;
    if (I >= nb) continue;
    const uint32_t* row =
        reinterpret_cast<const uint32_t*>(pev + (static_cast<size_t>(h) * nb + I) * nb);
    const int len = I + 1;
    int c = 0;
    auto cnt = [&](uint32_t b) { c += b == st.thresh ? 1 : 0; };
    if ((nb & 3) == 0) {
      // rows start on 16-byte boundaries: four float4 loads in flight per lane
      const uint4* row4 = reinterpret_cast<const uint4*>(row);
      const int n4 = len >> 2;
      int q = lane;
      for (; q + 96 < n4; q += 128) {
        const uint4 x = row4[q], y = row4[q + 32], z = row4[q + 64], u = row4[q + 96];
        cnt(x.x); cnt(x.y); cnt(x.z); cnt(x.w);
        cnt(y.x); cnt(y.y); cnt(y.z); cnt(y.w);
        cnt(z.x); cnt(z.y); cnt(z.z); cnt(z.w);
        cnt(u.x); cnt(u.y); cnt(u.z); cnt(u.w);
      }
      for (; q < n4; q += 32) {
        const uint4 x = row4[q];
        cnt(x.x); cnt(x.y); cnt(x.z); cnt(x.w);
      }
      const int K = (n4 << 2) + lane;
      if (K < len) cnt(row[K]);
    } else {
      for (int K = lane; K < len; K += 32) cnt(row[K]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) eq_off[static_cast<size_t>(h) * (nb + 1) + I] = c;
  }
}

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
// per row: 128-key groups as one float4 per lane (four groups in flight) when no tie ranks
// are needed, else four 32-key words in flight per lane with ballots in key order.
// Flat-order tie ranks are needed only when some but not all items equal to the threshold
// are taken (need_eq < count_eq).
constexpr int kMaskWords = 4;

__global__ void __launch_bounds__(256) pe_mask_kernel(const float* __restrict__ pev,
                                                      const PeState* __restrict__ pe,
                                                      const int* __restrict__ pe_list,
                                                      const int64_t* __restrict__ eq_off,
                                                      int nb, int nbw, uint32_t* rowmask,
                                                      int32_t* counts, int32_t* near) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = pe_items(pe_list, nb);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    int h, I0;
    pe_item(pe_list, nb, item, h, I0);
    const int I = I0 + warp;
    if (I >= nb) continue;
    const PeState st = pe[h];
    const bool all = st.select_all != 0;
    const bool rank_ties = !all && st.need_eq < st.count_eq;
    int64_t eq_base = rank_ties ? eq_off[static_cast<size_t>(h) * (nb + 1) + I] : 0;
    const float* row = pev + (static_cast<size_t>(h) * nb + I) * nb;
    uint32_t* mrow = rowmask + (static_cast<size_t>(h) * nb + I) * nbw;
    const int nw = (I >> 5) + 1;  // words holding keys K <= I
    int selected = 0;
    // near-threshold pairs: |v - T| <= 1e-3 T (none counted when the whole triangle is kept)
    const float T = __uint_as_float(st.thresh);
    int near_cnt = 0;
    if (!rank_ties && (nb & 3) == 0) {
      // Every item equal to T is kept (or the whole triangle is): 128-key groups read as one
      // float4 per lane, four groups in flight.  Lane l holds keys 4l..4l+3 of a group, i.e.
      // nibble l & 7 of the group's word l >> 3; three xor shuffles OR the eight nibbles of
      // each word together.
      const float4* row4 = reinterpret_cast<const float4*>(row);
      const int ng = (I >> 7) + 1;  // groups holding keys K <= I
      for (int g0 = 0; g0 < ng; g0 += 4) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = g0 + u;
          x[u] = (g < ng && g * 128 + 4 * lane <= I) ? row4[g * 32 + lane]
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int g = g0 + u;
          if (g >= ng) break;
          const int K0 = g * 128 + 4 * lane;
          const float xe[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
          uint32_t nib = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const bool valid = K0 + e <= I;
            const uint32_t b = __float_as_uint(xe[e]);
            nib |= (valid && (all || b >= st.thresh)) ? (1u << e) : 0u;
            near_cnt += (valid && !all && fabsf(xe[e] - T) <= 1e-3f * T) ? 1 : 0;
          }
          selected += __popc(nib);
          uint32_t word = nib << (4 * (lane & 7));
          word |= __shfl_xor_sync(0xffffffffu, word, 1);
          word |= __shfl_xor_sync(0xffffffffu, word, 2);
          word |= __shfl_xor_sync(0xffffffffu, word, 4);
          const int wd = g * 4 + (lane >> 3);
          if ((lane & 7) == 0 && wd < nw) {
            if (wd == (I >> 5)) word |= 1u << (I & 31);
            mrow[wd] = word;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) selected += __shfl_xor_sync(0xffffffffu, selected, o);
    } else {
      // tie ranks (or rows not 16-byte aligned): a 32-key word per step, ballots in key order
      for (int wd0 = 0; wd0 < nw; wd0 += kMaskWords) {
        uint32_t x[kMaskWords];
#pragma unroll
        for (int u = 0; u < kMaskWords; ++u) {
          const int K = (wd0 + u) * 32 + lane;
          x[u] = K <= I ? __float_as_uint(row[K]) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kMaskWords; ++u) {
          const int wd = wd0 + u;
          if (wd >= nw) break;
          const bool valid = wd * 32 + lane <= I;
          bool sel = valid && (all || x[u] > st.thresh);
          near_cnt += (valid && !all && fabsf(__uint_as_float(x[u]) - T) <= 1e-3f * T) ? 1 : 0;
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
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) near_cnt += __shfl_xor_sync(0xffffffffu, near_cnt, o);
    if (lane == 0) {
      if (near_cnt) atomicAdd(&near[h * 3 + 2], near_cnt);
      atomicAdd(&counts[h * 4 + 0], selected);
      if (selected == 0) atomicAdd(&counts[h * 4 + 1], 1);
    }
  }
}

// ---------------------------------------------------------------- short sequences
// N_b <= kSmallNb: the whole gamma cut of a PE head in one CTA, the triangle held in shared
// memory (flattened row by row: pair (I, K) at I (I + 1) / 2 + K, the flat order of the
// cut's ties).  Same steps and rules as the multi-kernel path above: four 8-bit radix
// passes with fixed-point bin masses and the same digit pick, flat-order tie ranks when
// only some of the items equal to the threshold are taken, then the row masks (plus the
// diagonal), the kept-pair and rescued-row counts and the near-threshold count.  One
// launch instead of twelve, which matters at short lengths, where each launch costs about
// as much as its work.
constexpr int kSmallNb = 256;
constexpr int kSmallThreads = 1024;
constexpr int kSmallCopies = 8;  // shared histogram copies (one per 4 warps)

__host__ __device__ constexpr size_t small_select_smem(int nb) {
  // flattened triangle (fp32 bits), then the kept-pair bit array with one spare word
  return (static_cast<size_t>(nb) * (nb + 1) / 2 + (static_cast<size_t>(nb) * (nb + 1) / 2 + 31) / 32 + 2) *
         sizeof(uint32_t);
}

__global__ void __launch_bounds__(kSmallThreads, 1)
    pe_select_small_kernel(const float* __restrict__ pev, const uint8_t* __restrict__ route,
                           int nb, int nbw, float gamma, uint32_t* rowmask, int32_t* counts,
                           int32_t* near) {
  const int h = blockIdx.x;
  if (route[h]) return;
  extern __shared__ uint32_t s_dyn[];
  const int T = nb * (nb + 1) / 2;
  uint32_t* sv = s_dyn;                  // [T]
  uint32_t* sbits = s_dyn + T;           // [ceil(T / 32) + 2]
  __shared__ uint32_t scnt[kSmallCopies][256];
  __shared__ float smass[kSmallCopies][256];
  __shared__ int s_red[32];
  __shared__ PeState s_st;
  __shared__ DigitPick s_pick;
  __shared__ int s_sel_total, s_rescued;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // 1. the triangle into shared memory, a warp per row
  for (int I = warp; I < nb; I += kSmallThreads / 32) {
    const uint32_t* row = reinterpret_cast<const uint32_t*>(pev + (static_cast<size_t>(h) * nb + I) * nb);
    uint32_t* dst = sv + I * (I + 1) / 2;
    for (int K = lane; K <= I; K += 32) dst[K] = row[K];
  }
  const int nwords = (T + 31) / 32 + 2;
  for (int i = tid; i < nwords; i += kSmallThreads) sbits[i] = 0u;
  if (tid == 0) {
    PeState z{};
    s_st = z;
    s_sel_total = 0;
    s_rescued = 0;
  }
  __syncthreads();

  // 2. four radix passes over the fp32 bit patterns (positive values: bits order like values)
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < kSmallCopies * 256; i += kSmallThreads) {
      (&scnt[0][0])[i] = 0u;
      (&smass[0][0])[i] = 0.f;
    }
    __syncthreads();
    const PeState st = s_st;
    if (st.select_all) break;  // uniform: every thread read the same state
    const int copy = warp & (kSmallCopies - 1);
    // Values of a head crowd into few bins (the high digits above all), so a warp whose
    // matching lanes share a bin adds once (lane count, shuffle-summed mass); otherwise each
    // lane adds its own value.
    for (int i0 = 0; i0 < T; i0 += kSmallThreads) {
      const int i = i0 + tid;
      const uint32_t bits = i < T ? sv[i] : 0u;
      const bool match = i < T && (bits & st.decided) == st.prefix;
      const uint32_t bin = (bits >> shift) & 255u;
      const unsigned m = __ballot_sync(0xffffffffu, match);
      if (m == 0) continue;
      const uint32_t b0 = __shfl_sync(0xffffffffu, bin, __ffs(m) - 1);
      if (__all_sync(0xffffffffu, !match || bin == b0)) {
        float x = match ? __uint_as_float(bits) : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) {
          atomicAdd(&scnt[copy][b0], static_cast<uint32_t>(__popc(m)));
          atomicAdd(&smass[copy][b0], x);
        }
      } else if (match) {
        atomicAdd(&scnt[copy][bin], 1u);
        atomicAdd(&smass[copy][bin], __uint_as_float(bits));
      }
    }
    __syncthreads();
    // the copies combined per bin, thread t on bin 255 - t, then the parallel digit pick
    unsigned long long pc = 0, pm = 0;
    if (tid < 256) {
      uint32_t cc = 0;
      float mm = 0.f;
#pragma unroll
      for (int k = 0; k < kSmallCopies; ++k) {
        cc += scnt[k][255 - tid];
        mm += smass[k][255 - tid];
      }
      pc = cc;
      pm = mass_fixed(mm);
    }
    pick_crossing(tid, pc, pm, gamma_fixed(gamma) - st.above, &s_pick);
    if (tid == 0) {
      PeState ns = st;
      int chosen = s_pick.bin;
      unsigned long long above = s_pick.above, cnt = s_pick.cnt;
      if (chosen < 0) {
        // no bin reaches the target: as in pe_digit_kernel (the copies are still intact)
        unsigned long long total = 0;
        for (int k = 0; k < 8; ++k) total += s_pick.wsum[k];
        for (int bin = 0; bin < 256 && chosen < 0; ++bin) {
          uint32_t cc = 0;
          float mm = 0.f;
          for (int k = 0; k < kSmallCopies; ++k) {
            cc += scnt[k][bin];
            mm += smass[k][bin];
          }
          if (cc) {
            chosen = bin;
            cnt = cc;
            above = total - mass_fixed(mm);
          }
        }
        if (pass == 0 || chosen < 0) ns.select_all = 1;
      }
      if (!ns.select_all) finish_digit(ns, pass, gamma, chosen, above, cnt);
      s_st = ns;
    }
    __syncthreads();
  }
  __syncthreads();
  const PeState st = s_st;
  const bool all = st.select_all != 0;
  const bool rank_ties = !all && st.need_eq < st.count_eq;
  const float Tv = __uint_as_float(st.thresh);

  // 3. kept pairs as bits in flat order.  Without tie ranks (all items equal to the
  // threshold are kept, or the whole triangle is) a warp builds a 32-pair word from one
  // coalesced read (lane k: pair 32 w + k) and a ballot; with them, every thread owns whole
  // words of a contiguous range and the ranks come from a scan of the per-thread tie counts.
  const int words = (T + 31) / 32;
  int near_cnt = 0;
  if (!rank_ties) {
    for (int wd = warp; wd < words; wd += kSmallThreads / 32) {
      const int f = wd * 32 + lane;
      const uint32_t bits = f < T ? sv[f] : 0u;
      const bool sel = f < T && (all || bits >= st.thresh);
      if (f < T && !all && fabsf(__uint_as_float(bits) - Tv) <= 1e-3f * Tv) ++near_cnt;
      const unsigned word = __ballot_sync(0xffffffffu, sel);
      if (lane == 0) sbits[wd] = word;
    }
  } else {
    const int wper = (words + kSmallThreads - 1) / kSmallThreads;
    const int f0 = min(T, tid * wper * 32), f1 = min(T, (tid + 1) * wper * 32);
    int eq = 0;
    for (int f = f0; f < f1; ++f) eq += sv[f] == st.thresh ? 1 : 0;
    // exclusive scan of eq over the threads
    int incl = eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_red[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = s_red[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_red[lane] = w;
    }
    __syncthreads();
    long long rank = (warp > 0 ? s_red[warp - 1] : 0) + incl - eq;
    for (int f = f0; f < f1; f += 32) {
      uint32_t word = 0;
      for (int k = 0; k < 32 && f + k < f1; ++k) {
        const uint32_t bits = sv[f + k];
        bool sel = all || bits > st.thresh;
        if (!all && bits == st.thresh) {
          sel = rank < static_cast<long long>(st.need_eq);
          ++rank;
        }
        if (!all && fabsf(__uint_as_float(bits) - Tv) <= 1e-3f * Tv) ++near_cnt;
        if (sel) word |= 1u << k;
      }
      sbits[f >> 5] = word;
    }
  }
  __syncthreads();

  // 4. row masks (a warp per row: lane = 32-key word), kept-pair and rescued-row counts
  for (int I = warp; I < nb; I += kSmallThreads / 32) {
    const int base = I * (I + 1) / 2;
    int selected = 0;
    for (int wd0 = 0; wd0 < nbw; wd0 += 32) {
      const int wd = wd0 + lane;
      uint32_t word = 0;
      if (wd < nbw && wd * 32 <= I) {
        const int o = base + wd * 32;
        word = __funnelshift_r(sbits[o >> 5], sbits[(o >> 5) + 1], o & 31);
        const int top = I - wd * 32;  // keys 0..top of this word are in the row
        if (top < 31) word &= (2u << top) - 1u;
        selected += __popc(word);
        if (top < 32) word |= 1u << top;  // the diagonal
      }
      if (wd < nbw) rowmask[(static_cast<size_t>(h) * nb + I) * nbw + wd] = word;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) selected += __shfl_xor_sync(0xffffffffu, selected, o);
    if (lane == 0) {
      atomicAdd(&s_sel_total, selected);
      if (selected == 0) atomicAdd(&s_rescued, 1);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) near_cnt += __shfl_xor_sync(0xffffffffu, near_cnt, o);
  if (lane == 0 && near_cnt) atomicAdd(&near[h * 3 + 2], near_cnt);
  __syncthreads();
  if (tid == 0) {
    counts[h * 4 + 0] = s_sel_total;
    counts[h * 4 + 1] = s_rescued;
  }
}

}  // namespace

cudaError_t init_pe_attributes() {
  cudaError_t e = cudaFuncSetAttribute(pe_prob_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kPeSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(pe_select_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(small_select_smem(kSmallNb)));
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_hist_ctas_per_sm, pe_hist_kernel, 256, 0);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_eqcount_ctas_per_sm, pe_eqcount_kernel,
                                                    256, 0);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_mask_ctas_per_sm, pe_mask_kernel, 256,
                                                       0);
}

int pe_select_launches(int nb) { return nb <= kSmallNb ? 1 : 12; }

cudaError_t launch_pe_index(crisp_ctx ctx, const Shape& s, const crisp_cfg& cfg, const void* Q,
                            const void* K, const CUtensorMap& tmQs, const CUtensorMap& tmKs,
                            const CUtensorMap& tmO, bool tma_out, cudaStream_t st) {
  Workspace& w = ctx->ws;
  const uint16_t* q = static_cast<const uint16_t*>(Q);
  const uint16_t* k = static_cast<const uint16_t*>(K);
  pe_pool_kernel<<<dim3(s.H + s.Hkv, s.nb), 128, 0, st>>>(
      q, k, w.route, s.n, s.nb, s.H, s.hq, s.hkv, s.group, s.Hkv,
      1.4426950408889634f / sqrtf(static_cast<float>(kD)), w.qs, w.ks, w.pe_list);
  PeProbArgs pa;
  pa.route = w.route;
  pa.nb = s.nb;
  pa.nt = (s.nb + kBlk - 1) / kBlk;
  pa.hq = s.hq;
  pa.hkv = s.hkv;
  pa.group = s.group;
  pa.q_lo_rows = s.H * s.nb;
  pa.k_lo_rows = s.Hkv * s.nb;
  pa.inv_nb = 1.f / static_cast<float>(s.nb);
  pa.pev = w.pev;
  pa.err = w.err;
  pa.timeout_ns = ctx->timeout_ns;
  pa.tma_out = tma_out ? 1 : 0;
  pe_prob_kernel<<<dim3(s.H, pa.nt), kPeThreads, kPeSmem, st>>>(tmQs, tmKs, tmO, pa);
  if (s.nb <= kSmallNb) {
    pe_select_small_kernel<<<s.H, kSmallThreads, small_select_smem(s.nb), st>>>(
        w.pev, w.route, s.nb, s.nbw, cfg.gamma, w.rowmask, w.counts, w.near);
    return cudaGetLastError();
  }
  pe_radix_init_kernel<<<s.H, 256, 0, st>>>(w.route, w.pe, w.hist_cnt, w.hist_mass,
                                             w.pe_list);
  // at most one CTA per item of the largest possible list (every head a PE head)
  const int64_t items = static_cast<int64_t>(s.H) * ((s.nb + kPeRowsPerItem - 1) / kPeRowsPerItem);
  auto resident = [&](int per_sm) {
    return static_cast<int>(std::min<int64_t>(
        items, static_cast<int64_t>(ctx->num_sms) * std::max(per_sm, 1)));
  };
  for (int pass = 0; pass < 4; ++pass) {
    pe_hist_kernel<<<resident(g_hist_ctas_per_sm), 256, 0, st>>>(
        w.pev, w.pe, w.pe_list, s.nb, 24 - 8 * pass, w.hist_cnt, w.hist_mass);
    pe_digit_kernel<<<s.H, 256, 0, st>>>(w.route, pass, cfg.gamma, w.pe, w.hist_cnt,
                                         w.hist_mass);
  }
  pe_eqcount_kernel<<<resident(g_eqcount_ctas_per_sm), 256, 0, st>>>(w.pev, w.pe, w.pe_list,
                                                                      s.nb, w.eq_off);
  pe_eqscan_kernel<<<s.H, 1024, 0, st>>>(w.route, w.pe, s.nb, w.eq_off);
  pe_mask_kernel<<<resident(g_mask_ctas_per_sm), 256, 0, st>>>(
      w.pev, w.pe, w.pe_list, w.eq_off, s.nb, s.nbw, w.rowmask, w.counts, w.near);
  return cudaGetLastError();
}

}  // namespace crisp
