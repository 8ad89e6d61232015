// csr.cu -- per-query-block key-block lists (the index set S of the masked attention).
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top), Algorithm 3 (VSIndex) under "Figures and
// tables" returns S_v u S_s u {0, N_b-1}; "Prerequisites" defines the mask M_S of
// A(Q,K,V,S).  For a VS head, query block I keeps key block K <= I when K is a selected
// vertical block, when I-K is a selected slash block, when K = 0 (sink) or K = I (local
// window, the diagonal).  PE rows come from pe_index.cu as bitmasks over key blocks; VS
// rows are computed word by word from the head's S_v and S_s bit words where they are
// counted and compacted into CSR with ascending key blocks.
#include "internal.h"
#include "ptx.cuh"

namespace crisp {
namespace {

// A 32-key word of query block I's key set.  VS heads: computed from the head's bit words
// (written once by the route kernel: S_v in block order, then S_s reversed, bit x =
// sels[N_b-1-x]); for query block I, key K <= I is a slash key iff sels[I-K], i.e. bit
// N_b-1-I+K of the reversed array, so a word is a 64-bit funnel shift of that array, plus
// the sink block 0 and the diagonal I.  PE heads: the mask pe_index.cu wrote.  No word has
// a bit above the diagonal, and no caller asks for a word past the diagonal's ((I >> 5) + 1
// words for query block I).
__device__ __forceinline__ uint32_t row_word(bool vs, const uint32_t* __restrict__ sb,
                                             const uint32_t* __restrict__ m, int nb, int nbw,
                                             int I, int wd) {
  if (!vs) return m[wd];
  const int K0 = wd * 32;
  const int sh = nb - 1 - I + K0;  // bit of the reversed array for K = K0 (<= nb - 1)
  uint32_t out = sb[wd] | __funnelshift_r(sb[nbw + (sh >> 5)], sb[nbw + (sh >> 5) + 1], sh & 31);
  if (wd == 0) out |= 1u;  // the sink block
  const int top = I - K0;  // bits 0..top are keys K <= I
  if (top < 31) out &= (2u << top) - 1u;
  if (top < 32) out |= 1u << top;  // the diagonal block
  return out;
}

// Counts the blocks of 1024 rows (a warp per row, or a thread per row when a row mask is
// at most 16 words) and scans them inside the CTA: row_ptr[row] = offset within the CTA's
// rows, blk[b] = the CTA's total.
__global__ void __launch_bounds__(1024) csr_count_scan_kernel(const uint8_t* __restrict__ route,
                                                              const uint32_t* __restrict__ selbits,
                                                              const uint32_t* __restrict__ rowmask,
                                                              int64_t rows, int nb, int nbw,
                                                              int64_t* row_ptr, int64_t* blk) {
  __shared__ int cnt[1024];
  __shared__ int wsum[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 1024;
  if (nbw <= 16) {
    const int64_t row = r0 + threadIdx.x;
    int c = 0;
    if (row < rows) {
      const int h = static_cast<int>(row) / nb, I = static_cast<int>(row) % nb;
      const bool vs = route[h] != 0;
      const uint32_t* sb = selbits + static_cast<size_t>(h) * (2 * nbw + 1);
      const uint32_t* m = rowmask + row * nbw;
      const int nw = I / 32 + 1;
      for (int wd = 0; wd < nw; ++wd) c += __popc(row_word(vs, sb, m, nb, nbw, I, wd));
    }
    cnt[threadIdx.x] = c;
  } else {
    // A warp counts its 32 rows four at a time, every word of the four loaded before any
    // is counted (N_b <= 8192: at most 8 words per lane and row).
    for (int i0 = warp; i0 < 1024; i0 += 32 * 4) {
      uint32_t wv[4][8];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int64_t row = r0 + i0 + 32 * r;
        const int h = static_cast<int>(row) / nb, I = static_cast<int>(row) % nb;
        const int nw = row < rows ? I / 32 + 1 : 0;
        const bool vs = row < rows && route[h] != 0;
        const uint32_t* sb = selbits + static_cast<size_t>(h) * (2 * nbw + 1);
        const uint32_t* m = rowmask + row * nbw;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int wd = j * 32 + lane;
          wv[r][j] = wd < nw ? row_word(vs, sb, m, nb, nbw, I, wd) : 0u;
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        int c = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) c += __popc(wv[r][j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0) cnt[i0 + 32 * r] = c;
      }
    }
  }
  __syncthreads();
  const int c = cnt[threadIdx.x];
  int pre = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, pre, o);
    if (lane >= o) pre += t;
  }
  if (lane == 31) wsum[warp] = pre;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    wsum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int64_t row = r0 + threadIdx.x;
  if (row < rows) row_ptr[row] = (warp > 0 ? wsum[warp - 1] : 0) + pre - c;
  if (threadIdx.x == 1023) blk[blockIdx.x] = wsum[31];
}

// Exclusive scan of the per-CTA totals (one CTA); row_ptr[rows] = nnz.
__global__ void __launch_bounds__(1024) csr_blk_scan_kernel(int64_t* blk, int nblk, int64_t rows,
                                                            int64_t* row_ptr) {
  __shared__ int64_t part[1024];
  const int per = (nblk + 1023) / 1024;
  const int b0 = threadIdx.x * per, b1 = min(nblk, b0 + per);
  int64_t s = 0;
  for (int i = b0; i < b1; ++i) s += blk[i];
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
    const int64_t c = blk[i];
    blk[i] = run;
    run += c;
  }
  if (threadIdx.x == 1023) row_ptr[rows] = part[1023];
}

// col[row_ptr[row] + k] = k-th set bit of the row's mask (ascending); a warp per row.
// Finishes row_ptr (adds the CTA offset of the scan).  Lanes load 32 words at a time; then
// the warp walks the nonzero ones, every lane writing the index of its bit if set, so each
// word's entries are stored by consecutive lanes to consecutive addresses.
__global__ void __launch_bounds__(256) csr_fill_kernel(const uint8_t* __restrict__ route,
                                                       const uint32_t* __restrict__ selbits,
                                                       const uint32_t* __restrict__ rowmask,
                                                       int64_t* row_ptr,
                                                       const int64_t* __restrict__ blk,
                                                       int64_t rows, int nb, int nbw,
                                                       int raw_blk, int32_t* col) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (row >= rows) return;
  // raw_blk: blk holds each 1024-row block's total, not yet scanned (at most 32 blocks):
  // the row's base is the sum of the totals of the blocks before its own.
  int64_t base;
  if (raw_blk) {
    int64_t x = lane < static_cast<int>(row >> 10) ? blk[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    base = x;
  } else {
    base = blk[row >> 10];
  }
  int64_t off = row_ptr[row] + base;
  __syncwarp();
  if (lane == 0) row_ptr[row] = off;
  const uint32_t* m = rowmask + row * nbw;
  const int h = static_cast<int>(row) / nb, I = static_cast<int>(row) % nb;
  const int nw = (I >> 5) + 1;
  const bool vs = route[h] != 0;
  const uint32_t* sb = selbits + static_cast<size_t>(h) * (2 * nbw + 1);
  // The row's mask words all load at once (N_b <= 8192: at most 8 per lane), so a row
  // waits for one memory latency, not one per 32-word chunk.
  constexpr int kWordsPerLane = 8;
  uint32_t wv[kWordsPerLane];
#pragma unroll
  for (int j = 0; j < kWordsPerLane; ++j) {
    const int wd = j * 32 + lane;
    wv[j] = wd < nw ? row_word(vs, sb, m, nb, nbw, I, wd) : 0u;
  }
  // A row whose mask holds every key block K <= I (masks have no bits above I) is written
  // as 0..I with 16-byte stores where the offset allows: the usual row of a PE head.
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < kWordsPerLane; ++j) cnt += __popc(wv[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (raw_blk && row == rows - 1 && lane == 0) row_ptr[rows] = off + cnt;  // nnz
  if (cnt == I + 1) {
    const int mis = static_cast<int>((4 - (off & 3)) & 3);  // elements before a 16-byte boundary
    const int head = mis < I + 1 ? mis : I + 1;
    if (lane < head) col[off + lane] = lane;
    const int body = (I + 1 - head) >> 2;
    int4* dst4 = reinterpret_cast<int4*>(col + off + head);
    for (int i = lane; i < body; i += 32) {
      const int k0 = head + 4 * i;
      dst4[i] = make_int4(k0, k0 + 1, k0 + 2, k0 + 3);
    }
    for (int k = head + 4 * body + lane; k <= I; k += 32) col[off + k] = k;
    return;
  }
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kWordsPerLane; ++j) {
    const int wd0 = j * 32;
    if (wd0 >= nw) break;
    const uint32_t bits = wv[j];
    int pre = __popc(bits);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += t;
    }
    const int total = __shfl_sync(0xffffffffu, pre, 31);
    unsigned nz = __ballot_sync(0xffffffffu, bits != 0u);
    while (nz) {
      const int src = __ffs(nz) - 1;
      nz &= nz - 1u;
      const uint32_t w = __shfl_sync(0xffffffffu, bits, src);
      const int base = __shfl_sync(0xffffffffu, pre, src) - __popc(w);
      if (w & (1u << lane)) col[off + base + __popc(w & lt)] = (wd0 + src) * 32 + lane;
    }
    off += total;
  }
}

}  // namespace

bool csr_raw_blocks(int64_t rows) { return (rows + 1023) / 1024 <= 32; }

int csr_launches(int64_t rows) { return csr_raw_blocks(rows) ? 2 : 3; }

cudaError_t launch_build_csr(crisp_ctx ctx, const Shape& s, cudaStream_t st) {
  Workspace& w = ctx->ws;
  const int64_t rows = static_cast<int64_t>(s.H) * s.nb;
  const int nblk = static_cast<int>((rows + 1023) / 1024);
  csr_count_scan_kernel<<<nblk, 1024, 0, st>>>(w.route, w.selbits, w.rowmask, rows, s.nb, s.nbw,
                                                w.row_ptr, w.scan_blk);
  // Up to 32 blocks of rows the fill kernel sums the block totals itself (one launch fewer).
  const int raw_blk = csr_raw_blocks(rows) ? 1 : 0;
  if (!raw_blk) csr_blk_scan_kernel<<<1, 1024, 0, st>>>(w.scan_blk, nblk, rows, w.row_ptr);
  csr_fill_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      w.route, w.selbits, w.rowmask, w.row_ptr, w.scan_blk, rows, s.nb, s.nbw, raw_blk, w.col);
  return cudaGetLastError();
}

}  // namespace crisp
