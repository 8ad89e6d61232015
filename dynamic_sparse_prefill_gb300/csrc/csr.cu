// csr.cu -- per-query-block key-block lists (the index set S of the masked attention).
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top), Algorithm 3 (VSIndex) under "Figures and
// tables" returns S_v u S_s u {0, N_b-1}; "Prerequisites" defines the mask M_S of
// A(Q,K,V,S).  For a VS head, query block I keeps key block K <= I when K is a selected
// vertical block, when I-K is a selected slash block, when K = 0 (sink) or K = I (local
// window, the diagonal).  PE rows come from pe_index.cu.  Rows are stored as bitmasks
// over key blocks, then compacted into CSR with ascending key blocks.
#include "internal.h"
#include "ptx.cuh"

namespace crisp {
namespace {

constexpr int kRowsPerCta = 16;

__global__ void __launch_bounds__(256) vs_rowmask_kernel(const uint8_t* __restrict__ route,
                                                         const uint8_t* __restrict__ selv,
                                                         const uint8_t* __restrict__ sels,
                                                         int nb, int nbw, uint32_t* rowmask) {
  extern __shared__ uint8_t ssel[];
  const int h = blockIdx.y;
  if (!route[h]) return;
  uint8_t* sv = ssel;
  uint8_t* ss = ssel + nb;
  for (int J = threadIdx.x; J < nb; J += blockDim.x) {
    sv[J] = selv[static_cast<size_t>(h) * nb + J];
    ss[J] = sels[static_cast<size_t>(h) * nb + J];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int I = blockIdx.x * kRowsPerCta + warp; I < min(nb, (blockIdx.x + 1) * kRowsPerCta);
       I += 8) {
    uint32_t* mrow = rowmask + (static_cast<size_t>(h) * nb + I) * nbw;
    for (int wd = 0; wd < nbw; ++wd) {
      const int K = wd * 32 + lane;
      bool on = false;
      if (K <= I) on = (K == 0) || (K == I) || sv[K] || ss[I - K];
      const unsigned word = __ballot_sync(0xffffffffu, on);
      if (lane == 0) mrow[wd] = word;
    }
  }
}

// row_cnt[row] = number of key blocks in the row's mask; a warp per row.
__global__ void __launch_bounds__(256) csr_count_kernel(const uint32_t* __restrict__ rowmask,
                                                        int64_t rows, int nbw, int64_t* row_cnt) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint32_t* m = rowmask + row * nbw;
  int c = 0;
  for (int wd = lane; wd < nbw; wd += 32) c += __popc(m[wd]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if (lane == 0) row_cnt[row] = c;
}

// Exclusive scan of row_cnt into row_ptr (rows+1 entries) with one CTA.
__global__ void __launch_bounds__(1024) csr_scan_kernel(const int64_t* __restrict__ row_cnt,
                                                        int64_t rows, int64_t* row_ptr) {
  __shared__ int64_t part[1024];
  const int64_t per = (rows + 1023) / 1024;
  const int64_t b0 = threadIdx.x * per, b1 = min(rows, b0 + per);
  int64_t s = 0;
  for (int64_t i = b0; i < b1; ++i) s += row_cnt[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int64_t t = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += t;
    __syncthreads();
  }
  int64_t run = part[threadIdx.x] - s;
  for (int64_t i = b0; i < b1; ++i) {
    row_ptr[i] = run;
    run += row_cnt[i];
  }
  if (threadIdx.x == 1023) row_ptr[rows] = part[1023];
}

// col[row_ptr[row] + k] = k-th set bit of the row's mask (ascending); a warp per row.
__global__ void __launch_bounds__(256) csr_fill_kernel(const uint32_t* __restrict__ rowmask,
                                                       const int64_t* __restrict__ row_ptr,
                                                       int64_t rows, int nbw, int32_t* col) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint32_t* m = rowmask + row * nbw;
  int64_t off = row_ptr[row];
  for (int wd0 = 0; wd0 < nbw; wd0 += 32) {
    const int wd = wd0 + lane;
    uint32_t bits = wd < nbw ? m[wd] : 0u;
    const int c = __popc(bits);
    int pre = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += t;
    }
    const int total = __shfl_sync(0xffffffffu, pre, 31);
    int64_t pos = off + pre - c;
    while (bits) {
      const int b = __ffs(bits) - 1;
      col[pos++] = wd * 32 + b;
      bits &= bits - 1;
    }
    off += total;
  }
}

}  // namespace

cudaError_t launch_build_csr(crisp_ctx ctx, const Shape& s, cudaStream_t st) {
  Workspace& w = ctx->ws;
  vs_rowmask_kernel<<<dim3((s.nb + kRowsPerCta - 1) / kRowsPerCta, s.H), 256, 2 * s.nb, st>>>(
      w.route, w.selv, w.sels, s.nb, s.nbw, w.rowmask);
  const int64_t rows = static_cast<int64_t>(s.H) * s.nb;
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  csr_count_kernel<<<grid, 256, 0, st>>>(w.rowmask, rows, s.nbw, w.row_cnt);
  csr_scan_kernel<<<1, 1024, 0, st>>>(w.row_cnt, rows, w.row_ptr);
  csr_fill_kernel<<<grid, 256, 0, st>>>(w.rowmask, w.row_ptr, rows, s.nbw, w.col);
  return cudaGetLastError();
}

}  // namespace crisp
