// jsd.cu -- FlexPrefill's JSD routing signal, the one CRISP's C_struct replaces.
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top), "Prerequisites", JSD: FlexPrefill compares the
// "pool first, then softmax" distribution a_bar with the "softmax first, then average"
// distribution a_hat through D_JS = 1/2 KL(a_hat || m) + 1/2 KL(a_bar || m),
// m = (a_hat + a_bar)/2, and routes VS when D_JS >= tau; it costs a pooled product per
// head, a second softmax and two KL passes ("Motivation").  Here a_hat is the pooled
// proxy attention p_v that crisp_select already computed, and a_bar is the softmax over
// key blocks of (mean of the last 128 queries) . (block mean of the keys) / sqrt(d).
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace crisp {
namespace {

// Kbar[hk][J][:] = mean of the 128 keys of block J, for every KV head.
__global__ void __launch_bounds__(128) jsd_pool_k_kernel(const uint16_t* __restrict__ K, int n,
                                                         int nb, float* kbar) {
  const int hk = blockIdx.y, J = blockIdx.x;
  __shared__ float part[8][kD];
  const int rg = threadIdx.x >> 4;
  const int cc = (threadIdx.x & 15) * 8;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint16_t* base = K + (static_cast<size_t>(hk) * n + static_cast<size_t>(J) * kBlk) * kD;
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
  kbar[(static_cast<size_t>(hk) * nb + J) * kD + threadIdx.x] = s * (1.f / kBlk);
}

__device__ double block_sum_d(double x, double* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  double t = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

__device__ float block_max_f(float x, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : -FLT_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

// One CTA (1024 threads) per query head; dynamic shared memory holds nb logits.
__global__ void __launch_bounds__(1024) jsd_kernel(const uint16_t* __restrict__ Q,
                                                   const float* __restrict__ kbar,
                                                   const float* __restrict__ pv, int n, int nb,
                                                   int hq, int hkv, int group, float scale,
                                                   float tau, float* d_js, uint8_t* route) {
  extern __shared__ float slog[];  // [nb]
  __shared__ float qpart[8][kD];
  __shared__ float qbar[kD];
  __shared__ float redf[32];
  __shared__ double redd[32];
  const int h = blockIdx.x;
  const int hk = (h / hq) * hkv + (h % hq) / group;
  // mean of the last 128 query rows
  {
    const int c = threadIdx.x & 127, g = threadIdx.x >> 7;
    const uint16_t* base = Q + (static_cast<size_t>(h) * n + (n - kBlk)) * kD;
    float s = 0.f;
    for (int rr = g; rr < kBlk; rr += 8)
      s += __uint_as_float(static_cast<uint32_t>(base[static_cast<size_t>(rr) * kD + c]) << 16);
    qpart[g][c] = s;
    __syncthreads();
    if (threadIdx.x < kD) {
      float t = 0.f;
      for (int i = 0; i < 8; ++i) t += qpart[i][threadIdx.x];
      qbar[threadIdx.x] = t * (1.f / kBlk);
    }
    __syncthreads();
  }
  // block logits: a warp per key block, lanes over the head dimension
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int J = warp; J < nb; J += 32) {
    const float4 kv = *reinterpret_cast<const float4*>(kbar + (static_cast<size_t>(hk) * nb + J) * kD + lane * 4);
    float s = kv.x * qbar[lane * 4] + kv.y * qbar[lane * 4 + 1] + kv.z * qbar[lane * 4 + 2] +
              kv.w * qbar[lane * 4 + 3];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) slog[J] = s * scale;
  }
  __syncthreads();
  float mx = -FLT_MAX;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) mx = fmaxf(mx, slog[J]);
  mx = block_max_f(mx, redf);
  double z = 0.0;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) z += exp(static_cast<double>(slog[J] - mx));
  z = block_sum_d(z, redd);
  // D_JS in fp64 with 0 log 0 = 0
  double acc = 0.0;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) {
    const double ab = exp(static_cast<double>(slog[J] - mx)) / z;
    const double ah = static_cast<double>(pv[static_cast<size_t>(h) * nb + J]);
    const double m = 0.5 * (ab + ah);
    if (ah > 0.0) acc += 0.5 * ah * log(ah / m);
    if (ab > 0.0) acc += 0.5 * ab * log(ab / m);
  }
  acc = block_sum_d(acc, redd);
  if (threadIdx.x == 0) {
    d_js[h] = static_cast<float>(acc);
    route[h] = acc >= static_cast<double>(tau) ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_jsd(crisp_ctx ctx, const Shape& s, const void* Q, const void* K, float tau,
                       float* d_js, uint8_t* route, cudaStream_t st) {
  Workspace& w = ctx->ws;
  jsd_pool_k_kernel<<<dim3(s.nb, s.Hkv), 128, 0, st>>>(static_cast<const uint16_t*>(K), s.n,
                                                      s.nb, w.kbar);
  jsd_kernel<<<s.H, 1024, static_cast<size_t>(s.nb) * sizeof(float), st>>>(
      static_cast<const uint16_t*>(Q), w.kbar, w.pv, s.n, s.nb, s.hq, s.hkv, s.group,
      1.f / sqrtf(static_cast<float>(kD)), tau, d_js, route);
  return cudaGetLastError();
}

}  // namespace crisp
