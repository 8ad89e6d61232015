// attention.cu -- exact causal attention over selected key blocks (and the dense case).
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top): "Prerequisites" defines
// A(Q,K,V,S) = Softmax(QK^T/sqrt(d) + M_S) V and notes that CRISP computes exact softmax
// attention on the selected blocks, compatible with FlashAttention-style tiling;
// "Method step details" step 4 applies it to the selected index set.  With every key
// block K <= I selected this is dense causal attention, the speedup denominator.
//
// One CTA per (query head, query block I) work item, 6 warps:
//   warp 0  TMA producer: Q tile once, then K_j and V_j of each selected key block into a
//           two-stage ring;
//   warp 1  MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM S buffers, and
//           O += P_j V_j into the TMEM O accumulator (tcgen05, bf16 in, fp32 accumulate);
//   warps 2-5  softmax: thread <-> query row (TMEM lane).  Online softmax in the exp2
//           domain; the running max is only raised when a block exceeds it by more than
//           2^8, so O is rescaled (TMEM load, scale, store) rarely; P_j is written to
//           shared memory as bf16 in the swizzled K-major layout the MMA reads.
// S_{j+1} is computed while the softmax works on S_j.  All waits are bounded.
#include <cuda_bf16.h>

#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace crisp {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);   // Q K^T
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);   // P V (V is MN-major)
constexpr size_t kSmem = 1024 + kTileBytes * 2 + kStages * 2 * kTileBytes + 256;
constexpr float kRescaleLog2 = 8.0f;  // raise the running max only past a factor 2^8
constexpr uint32_t kTmemCols = 512;   // S0 [0,128) S1 [128,256) O [256,384)

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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

struct AttnArgs {
  int n, nb, H, hq, hkv, group;
  float scale_log2;
  const int64_t* row_ptr;  // CSR of the selection (sparse mode)
  const int32_t* col;
  int dense;
  uint16_t* O;
  uint32_t* err;
  uint64_t timeout_ns;
  uint32_t debug;
};

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sP = smem + kTileBytes;
  uint8_t* sKV = smem + 2 * kTileBytes;  // stage s: K at +2s*T, V at +(2s+1)*T
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + kStages * 2 * kTileBytes);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2]
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work item: longest rows first (I descending), heads of a GQA group adjacent.
  const int item = blockIdx.x;
  const int h = item % a.H;
  const int I = a.nb - 1 - item / a.H;
  const int hk = (h / a.hq) * a.hkv + (h % a.hq) / a.group;
  int64_t beg = 0;
  int L;
  if (a.dense) {
    L = I + 1;
  } else {
    beg = a.row_ptr[static_cast<int64_t>(h) * a.nb + I];
    L = static_cast<int>(a.row_ptr[static_cast<int64_t>(h) * a.nb + I + 1] - beg);
  }
  const uint64_t tmo = a.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_O = tmem + 256;

  if (warp == 0) {
    if (lane == 0 && L > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int qrow = h * a.n + I * kBlk;
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(sQ, &tmQ, q_full, 0, qrow);
      tma_load_2d(sQ + kTileBytes / 2, &tmQ, q_full, 64, qrow);
      int issued = 0;
      for (int j = 0; j < L; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            !mbar_wait(&kv_empty[s], ((j / kStages) + 1) & 1, a.err, abort_flag, tmo))
          break;
        int kb = a.dense ? j : a.col[beg + j];
        if (kb < 0 || kb > I) {
          atomicOr(a.err, kErrRange);
          kb = I;
        }
        const int krow = hk * a.n + kb * kBlk;
        uint8_t* dK = sKV + (2 * s) * kTileBytes;
        uint8_t* dV = dK + kTileBytes;
        mbar_arrive_expect_tx(&kv_full[s], 2 * kTileBytes);
        tma_load_2d(dK, &tmK, &kv_full[s], 0, krow);
        tma_load_2d(dK + kTileBytes / 2, &tmK, &kv_full[s], 64, krow);
        tma_load_2d(dV, &tmV, &kv_full[s], 0, krow);
        tma_load_2d(dV + kTileBytes / 2, &tmV, &kv_full[s], 64, krow);
        ++issued;
      }
      drain_wait(q_full, 0, a.err, tmo);
      for (int j = max(0, issued - kStages); j < issued; ++j)
        drain_wait(&kv_full[j % kStages], (j / kStages) & 1, a.err, tmo);
    }
  } else if (warp == 1) {
    if (lane == 0 && L > 0) {
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t p_base = smem_u32(sP);
      auto issue_s = [&](int j) {
        const int s = j % kStages;
        const uint32_t k_base = smem_u32(sKV + (2 * s) * kTileBytes);
        const uint32_t d = tmem + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
          umma_bf16(d, sdesc_sw128(q_base + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024),
                    kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
      };
      bool ok = mbar_wait(q_full, 0, a.err, abort_flag, tmo) &&
                mbar_wait(&kv_full[0], 0, a.err, abort_flag, tmo);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        for (int j = 0; j < L; ++j) {
          if (j + 1 < L) {
            if (!mbar_wait(&kv_full[(j + 1) % kStages], ((j + 1) / kStages) & 1, a.err,
                           abort_flag, tmo))
              break;
            tc_fence_after();
            issue_s(j + 1);
          }
          if (!mbar_wait(p_full, j & 1, a.err, abort_flag, tmo)) break;
          tc_fence_after();
          const int s = j % kStages;
          const uint32_t v_base = smem_u32(sKV + (2 * s + 1) * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
            // B = V_j rows kk*16.. (keys), MN-major: 64-column regions 16 KB apart (LBO),
            // 8-row groups 1024 B apart (SBO).
            umma_bf16(tmem_O, sdesc_sw128(p_base + aoff, 16, 1024),
                      sdesc_sw128(v_base + kk * 2048, kTileBytes / 2, 1024), kIdescPV,
                      (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(o_done);
          umma_commit(&kv_empty[s]);
        }
      }
      umma_commit(drain);
      drain_wait(drain, 0, a.err, tmo);
    }
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint16_t* orow = a.O + (static_cast<size_t>(h) * a.n + static_cast<size_t>(I) * kBlk + r) * kD;
    float m_run = -FLT_MAX, l_run = 0.f;
    bool ok = L > 0;
    for (int j = 0; j < L && ok; ++j) {
      if (!warp_wait(&s_full[j & 1], (j >> 1) & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + (j & 1) * 128 + c * 32, v[c]);
      const int kb = a.dense ? j : a.col[beg + j];
      const bool diag = (kb == I);
      float mloc = -FLT_MAX;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float s2 = __uint_as_float(v[c4][c]) * a.scale_log2;
          if (diag && (c4 * 32 + c) > r) s2 = -FLT_MAX;
          v[c4][c] = __float_as_uint(s2);
          mloc = fmaxf(mloc, s2);
        }
      float alpha = 1.f;
      if (mloc > m_run + kRescaleLog2 || j == 0) {
        const float m_new = fmaxf(m_run, mloc);
        alpha = (j == 0) ? 0.f : fast_exp2(m_run - m_new);
        m_run = m_new;
      }
      float rs = 0.f;
      uint32_t pk[4][16];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float s0 = __uint_as_float(v[c4][2 * c]);
          const float s1 = __uint_as_float(v[c4][2 * c + 1]);
          const float p0 = s0 == -FLT_MAX ? 0.f : fast_exp2(s0 - m_run);
          const float p1 = s1 == -FLT_MAX ? 0.f : fast_exp2(s1 - m_run);
          rs += p0 + p1;
          pk[c4][c] = pack_bf16(p0, p1);
        }
      l_run = l_run * alpha + rs;
      if (j > 0 && !warp_wait(o_done, (j - 1) & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      // P_j -> shared memory, 128-byte swizzled K-major (keys are the K dimension).
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        const uint32_t off = (c16 >> 3) * (kTileBytes / 2) + r * 128 +
                             ((static_cast<uint32_t>(c16 & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(sP + off) =
            make_uint4(pk[c16 >> 2][(c16 & 3) * 4 + 0], pk[c16 >> 2][(c16 & 3) * 4 + 1],
                       pk[c16 >> 2][(c16 & 3) * 4 + 2], pk[c16 >> 2][(c16 & 3) * 4 + 3]);
      }
      fence_proxy_async_smem();
      if (j > 0 && !__all_sync(0xffffffffu, alpha == 1.f)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem_O + lane_off + c * 32, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tmem_O + lane_off + c * 32, o);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      const bool drop = (a.debug & CRISP_DEBUG_DROP_ARRIVE) && blockIdx.x == 0 && j == L - 1;
      if (!drop) mbar_arrive(p_full);
    }
    if (ok && warp_wait(o_done, (L - 1) & 1, a.err, abort_flag, tmo)) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem_O + lane_off + c * 32, o);
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          uint4 pkt;
          pkt.x = pack_bf16(__uint_as_float(o[k + 0]) * inv_l, __uint_as_float(o[k + 1]) * inv_l);
          pkt.y = pack_bf16(__uint_as_float(o[k + 2]) * inv_l, __uint_as_float(o[k + 3]) * inv_l);
          pkt.z = pack_bf16(__uint_as_float(o[k + 4]) * inv_l, __uint_as_float(o[k + 5]) * inv_l);
          pkt.w = pack_bf16(__uint_as_float(o[k + 6]) * inv_l, __uint_as_float(o[k + 7]) * inv_l);
          *reinterpret_cast<uint4*>(orow + c * 32 + k) = pkt;
        }
      }
    } else {
      // No output could be formed (empty row or an aborted wait): write zeros.
      for (int k = 0; k < kD; k += 8) *reinterpret_cast<uint4*>(orow + k) = make_uint4(0, 0, 0, 0);
      if (L <= 0) atomicOr(a.err, kErrRange);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attention(crisp_ctx ctx, const Shape& s, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV, void* O, bool dense,
                             cudaStream_t st) {
  AttnArgs a;
  a.n = s.n;
  a.nb = s.nb;
  a.H = s.H;
  a.hq = s.hq;
  a.hkv = s.hkv;
  a.group = s.group;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kD));
  a.row_ptr = ctx->ws.row_ptr;
  a.col = ctx->ws.col;
  a.dense = dense ? 1 : 0;
  a.O = static_cast<uint16_t*>(O);
  a.err = ctx->ws.err;
  a.timeout_ns = (ctx->debug_flags & CRISP_DEBUG_DROP_ARRIVE) ? 50000000ull : ctx->timeout_ns;
  a.debug = ctx->debug_flags;
  const unsigned items = static_cast<unsigned>(s.H) * static_cast<unsigned>(s.nb);
  attention_kernel<<<items, kThreads, kSmem, st>>>(tmQ, tmK, tmV, a);
  return cudaGetLastError();
}

cudaError_t init_attention_attributes() {
  return cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmem));
}

}  // namespace crisp
