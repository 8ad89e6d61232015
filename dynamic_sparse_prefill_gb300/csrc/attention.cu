// attention.cu -- exact causal attention over selected key blocks (and the dense case).
//
// CRISP ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-
// Motivated Routing", paper.rainbus.top): "Prerequisites" defines
// A(Q,K,V,S) = Softmax(QK^T/sqrt(d) + M_S) V and notes that CRISP computes exact softmax
// attention on the selected blocks, compatible with FlashAttention-style tiling;
// "Method step details" step 4 applies it to the selected index set.  With every key
// block K <= I selected this is dense causal attention, the speedup denominator.
//
// Two persistent kernels, one CTA per SM, over work items (query head h, query block I)
// in an order that keeps each launch's KV heads together, longest row first across them
// (one KV head per launch at long lengths, a few at short ones).  The fast kernel
// hands items out dynamically (a per-launch counter and a shared-memory item ring, see
// ItemFeed); the rescue kernel walks its short list in static serpentine waves (see
// get_item).  Both use the same warp roles:
//   warps 0-3  softmax of "tile 0" and warps 4-7 of "tile 1": the tiles take alternate
//              key blocks (by the CTA-wide block index in the fast kernel, by the index
//              within the row in the rescue kernel);
//   warp 8     TMA producer of the item's Q tile and K_j (4-slot ring in the fast
//              kernel, 3-slot in the rescue kernel);
//   warp 9     MMA issuer (one thread, tcgen05): S = Q K_j^T into TMEM (and, in the
//              rescue kernel, O += P V_j with P read from TMEM);
//   warp 10    TMA producer of V_j (2-slot ring), so K prefetch never waits on a V slot;
//   warp 11    (fast kernel) the second MMA issuer: O += P V_j.
// The softmax warpgroups take registers from the loader warpgroup (setmaxnreg).
//
// attention_kernel (every item): each tile has its own S and P buffers in TMEM and the
// two tiles accumulate into one O, exponentiating against one reference per row (the
// larger of the exact maxima of the tiles' first blocks).  A tile's next S is computed
// while its softmax still works on the previous one, so the tensor core never waits for
// a P to be written before it can start the next S.  Rows whose P could overflow against
// the reference are listed for the rescue pass.
//
// attention_rescue_kernel (the listed rows only; normally none): each tile keeps its own
// running max, sum and O accumulator, P overwrites its S buffer, and the epilogue merges
// the two partial softmaxes exactly.  The running max is raised (with a TMEM rescale of
// O) when a block exceeds it by more than 2^8, so any finite input is handled.
// All waits are bounded (see ptx.cuh); nothing traps.
#include <cuda_bf16.h>

#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace crisp {
namespace {

// Warpgroups: WG0 (warps 0-3) softmax of tile 0, WG1 (warps 4-7) softmax of tile 1,
// WG2 (warps 8-11): warp 8 Q/K producer, warp 9 MMA issuer, warp 10 V producer.
constexpr int kThreads = 384;
// Register split: launched at kLaunchRegs per thread (the host checks the compiled
// count), the softmax warpgroups grow and WG2 shrinks; the sum must fit the launch
// allocation.  The fast pass: 128 * (2 * 224 + 56) = 64512 = 384 * 168.  The rescue pass
// (heavier softmax, with O rescaling): 128 * (2 * 232 + 40) = 64512.
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kSoftmaxRegs = 224;
constexpr uint32_t kLoaderRegs = 56;
constexpr uint32_t kRescueSoftmaxRegs = 232;
constexpr uint32_t kRescueLoaderRegs = 40;
static_assert(128 * (2 * kSoftmaxRegs + kLoaderRegs) <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
static_assert(128 * (2 * kRescueSoftmaxRegs + kRescueLoaderRegs) <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);   // Q K^T
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);   // P V (V MN-major)
constexpr size_t kMLBytes = 2 * 2 * kBlk * 2 * sizeof(float);         // [parity][tile][row][m,l]
constexpr size_t kSmem = 1024 + kTileBytes * (1 + kKStages + kVStages) + kMLBytes + 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLazySum = 32768.0f;  // 128 columns x 2^8
constexpr uint32_t kTmemCols = 512;  // S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512)

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

// Row maximum of the 128 raw logits of an S row (columns c > r masked on the diagonal).
template <bool kDiag>
__device__ __forceinline__ float row_max(const uint32_t (&v)[128], int r) {
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = -FLT_MAX;
#pragma unroll
  for (int c = 0; c < 128; ++c)
    if (!kDiag || c <= r) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(v[c]));
  return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// P = exp2(s * scale - m) for the 128 columns of an S row, packed to bf16 pairs in place
// (v[c] <- (p[2c], p[2c+1]); elements 2c, 2c+1 are read before index c is written).
// Returns the row sum of P.
template <bool kDiag>
__device__ __forceinline__ float exp_pack(uint32_t (&v)[128], float scale, float m, int r) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const float neg = -m;
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    float x0, x1;
    ffma2(x0, x1, __uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]), scale, scale, neg, neg);
    if (kDiag) {
      x0 = 2 * c <= r ? x0 : -INFINITY;
      x1 = 2 * c + 1 <= r ? x1 : -INFINITY;
    }
    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
    const int a = (c & 3) * 2;
    fadd2(acc[a], acc[a + 1], acc[a], acc[a + 1], p0, p1);
    v[c] = pack_bf16(p0, p1);
  }
  fadd2(acc[0], acc[1], acc[0], acc[1], acc[2], acc[3]);
  fadd2(acc[4], acc[5], acc[4], acc[5], acc[6], acc[7]);
  fadd2(acc[0], acc[1], acc[0], acc[1], acc[4], acc[5]);
  return acc[0] + acc[1];
}

struct AttnArgs {
  int n, nb, H, hq, hkv, group;
  int num_items;
  int item_base;  // the launch covers entries [item_base, item_base + num_items) of the order
  float scale_log2;
  const int64_t* row_ptr;  // CSR of the selection (sparse mode)
  const int32_t* col;
  const int32_t* order;    // sparse mode: rows by descending length
  int dense;
  uint16_t* O;
  uint32_t* err;
  uint64_t timeout_ns;
  uint32_t debug;
  // Rescue pass: items are the rows listed in list[0 .. *list_count) (set by the fast pass).
  const int32_t* list;
  const int* list_count;
  // Fast pass: rows whose probabilities could overflow against the row's reference
  // maximum are appended here for the rescue pass.
  int32_t* redo;
  int* redo_count;
  // Fast pass: the launch's work counter (items are handed out in order, see ring_take).
  int* work_ctr;
};

struct Item {
  int h, I, hk, L;
  int64_t beg;
  int diag;  // the row's last block is its diagonal (fast pass; only it can be: rows are
             // strictly ascending within [0, I])
};

// Item at position ke of the launch's order: a listed row (rescue pass), a row of the
// sparse order, or the dense enumeration (within a launch's KV heads: query block
// descending, then KV head, the group's q-heads adjacent).
__device__ __forceinline__ Item item_of(const AttnArgs& a, int ke) {
  Item it;
  if (a.list != nullptr) {
    const int row = a.list[ke];
    it.h = row / a.nb;
    it.I = row % a.nb;
  } else if (a.dense) {
    const int per_I = a.num_items / a.nb;  // rows per query block in this launch
    const int local = ke - a.item_base;
    const int r = local % per_I;
    const int hk_all = a.item_base / (a.group * a.nb) + r / a.group;
    it.I = a.nb - 1 - local / per_I;
    it.h = (hk_all / a.hkv) * a.hq + (hk_all % a.hkv) * a.group + r % a.group;
  } else {
    const int row = a.order[ke];
    it.h = row / a.nb;
    it.I = row % a.nb;
  }
  it.hk = (it.h / a.hq) * a.hkv + (it.h % a.hq) / a.group;
  if (a.dense) {
    it.beg = 0;
    it.L = it.I + 1;
  } else {
    const int64_t row = static_cast<int64_t>(it.h) * a.nb + it.I;
    it.beg = a.row_ptr[row];
    it.L = static_cast<int>(a.row_ptr[row + 1] - it.beg);
  }
  return it;
}

// Work item k of a CTA's static round-robin sequence (k = blockIdx.x + i * G): items are
// taken in waves of G consecutive entries of the order, odd waves in reverse
// (serpentine), so each CTA's total stays balanced.  Used by the rescue pass.
__device__ __forceinline__ Item get_item(const AttnArgs& a, int k, int G, int num_items) {
  const int m = k / G, pos = k % G;
  const int base = m * G;
  const int wsize = min(G, num_items - base);
  const int ke = ((m & 1) ? base + wsize - 1 - pos : k) + a.item_base;
  return item_of(a, ke);
}

__device__ __forceinline__ int block_of(const AttnArgs& a, const Item& it, int j) {
  return a.dense ? j : a.col[it.beg + j];
}

// TMA producer of the items' Q tiles and key blocks K_j (one thread): Q is reloaded once
// the MMA warp has committed the item's last S (q_empty); K_j goes into a kKStages-slot
// ring whose slots the consumer releases on k_empty.  Column indices outside [0, I] are
// replaced by I and flagged (kErrRange).
template <int kKS>
__device__ __forceinline__ void produce_qk(const AttnArgs& a, int num_items, const CUtensorMap* tmQ,
                                           const CUtensorMap* tmK, uint8_t* sQ, uint8_t* sK,
                                           uint64_t* q_full, uint64_t* q_empty, uint64_t* k_full,
                                           uint64_t* k_empty, volatile int* abort_flag,
                                           uint64_t tmo) {
  tma_prefetch_desc(tmQ);
  tma_prefetch_desc(tmK);
  int gk = 0, item_idx = 0, q_loads = 0;
  bool ok = true;
  for (int k = blockIdx.x; k < num_items && ok; k += gridDim.x, ++item_idx) {
    const Item it = get_item(a, k, gridDim.x, num_items);
    if (item_idx > 0 && !mbar_wait(q_empty, (item_idx - 1) & 1, a.err, abort_flag, tmo)) {
      ok = false;
      break;
    }
    const int qrow = it.h * a.n + it.I * kBlk;
    mbar_arrive_expect_tx(q_full, kTileBytes);
    tma_load_3d(sQ, tmQ, q_full, 0, qrow, 0);
    ++q_loads;
    for (int j = 0; j < it.L; ++j) {
      int kb = block_of(a, it, j);
      if (kb < 0 || kb > it.I) {
        atomicOr(a.err, kErrRange);
        kb = it.I;
      }
      const int s = gk % kKS;
      if (gk >= kKS &&
          !mbar_wait(&k_empty[s], ((gk / kKS) + 1) & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      uint8_t* dst = sK + s * kTileBytes;
      const int row = it.hk * a.n + kb * kBlk;
      mbar_arrive_expect_tx(&k_full[s], kTileBytes);
      tma_load_3d(dst, tmK, &k_full[s], 0, row, 0);
      ++gk;
    }
  }
  // Let every copy still in flight land before the CTA can exit.
  if (q_loads > 0) drain_wait(q_full, (q_loads - 1) & 1, a.err, tmo);
  for (int g = max(0, gk - kKS); g < gk; ++g)
    drain_wait(&k_full[g % kKS], (g / kKS) & 1, a.err, tmo);
}

// TMA producer of the value blocks V_j (one thread) into a kVS-slot ring, released by the
// commit after the P.V MMAs that read the slot (v_empty).  Both producers load each tile
// with one 3-D copy (see tma_load_3d).
template <int kVS>
__device__ __forceinline__ void produce_v(const AttnArgs& a, int num_items, const CUtensorMap* tmV,
                                          uint8_t* sV, uint64_t* v_full, uint64_t* v_empty,
                                          volatile int* abort_flag, uint64_t tmo) {
  tma_prefetch_desc(tmV);
  int gv = 0;
  bool ok = true;
  for (int k = blockIdx.x; k < num_items && ok; k += gridDim.x) {
    const Item it = get_item(a, k, gridDim.x, num_items);
    for (int j = 0; j < it.L; ++j) {
      int kb = block_of(a, it, j);
      if (kb < 0 || kb > it.I) kb = it.I;
      const int s = gv % kVS;
      if (gv >= kVS &&
          !mbar_wait(&v_empty[s], ((gv / kVS) + 1) & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      uint8_t* dst = sV + s * kTileBytes;
      const int row = it.hk * a.n + kb * kBlk;
      mbar_arrive_expect_tx(&v_full[s], kTileBytes);
      tma_load_3d(dst, tmV, &v_full[s], 0, row, 0);
      ++gv;
    }
  }
  for (int g = max(0, gv - kVS); g < gv; ++g)
    drain_wait(&v_full[g % kVS], (g / kVS) & 1, a.err, tmo);
}

// ---------------------------------------------------------------------------------------
// Dynamic item feed of the fast pass.  The Q/K producer takes the next position of the
// launch's order from a global counter when it starts an item (so CTAs that finish early
// take more items: longest-first greedy balancing, since the order is longest first) and
// publishes it in a kItemRing-slot ring in shared memory; every other role reads the
// ring in order and releases the slot.  -1 ends the stream.
constexpr int kItemRing = 4;
constexpr int kItemReaders = 11;  // V producer, S issuer, P.V issuer, 8 softmax warps

// A ring slot: the item's position in the launch's order and the item decoded by the
// producer (the readers then need no global loads to start it).
struct FeedItem {
  int k, h, I, hk, L, diag;
  long long beg;
};

struct ItemFeed {
  volatile FeedItem* slot;
  uint64_t* full;   // [kItemRing] count 1
  uint64_t* empty;  // [kItemRing] count kItemReaders
};

__device__ __forceinline__ int read_slot(volatile FeedItem* e, Item& it) {
  it.h = e->h;
  it.I = e->I;
  it.hk = e->hk;
  it.L = e->L;
  it.diag = e->diag;
  it.beg = e->beg;
  return e->k;
}

// One thread: the idx-th item of the stream (-1: end), or -2 if a wait ran out.
__device__ __forceinline__ int feed_next(const ItemFeed& f, int idx, Item& it, uint32_t* err,
                                         volatile int* abort_flag, uint64_t tmo) {
  const int s = idx % kItemRing;
  if (!mbar_wait(&f.full[s], (idx / kItemRing) & 1, err, abort_flag, tmo)) return -2;
  const int k = read_slot(&f.slot[s], it);
  mbar_arrive(&f.empty[s]);
  return k;
}

// A whole warp: the same, one release per warp.
__device__ __forceinline__ int feed_next_warp(const ItemFeed& f, int idx, Item& it,
                                              uint32_t* err, volatile int* abort_flag,
                                              uint64_t tmo) {
  const int s = idx % kItemRing;
  if (!warp_wait(&f.full[s], (idx / kItemRing) & 1, err, abort_flag, tmo)) return -2;
  const int k = read_slot(&f.slot[s], it);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&f.empty[s]);
  return k;
}

// The fast pass's Q/K producer: takes items from the counter, publishes them, and loads
// Q and the K blocks exactly as produce_qk does for its static sequence.
template <int kKS>
__device__ __forceinline__ void produce_qk_feed(const AttnArgs& a, int num_items,
                                                const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                                uint8_t* sQ, uint8_t* sK, uint64_t* q_full,
                                                uint64_t* q_empty, uint64_t* k_full,
                                                uint64_t* k_empty, const ItemFeed& feed,
                                                volatile int* abort_flag, uint64_t tmo) {
  tma_prefetch_desc(tmQ);
  tma_prefetch_desc(tmK);
  int gk = 0, q_loads = 0;
  bool ok = true;
  for (int item_idx = 0; ok; ++item_idx) {
    const int s = item_idx % kItemRing;
    if (item_idx >= kItemRing &&
        !mbar_wait(&feed.empty[s], ((item_idx / kItemRing) - 1) & 1, a.err, abort_flag, tmo))
      break;
    int k = atomicAdd(a.work_ctr, 1);
    if (k >= num_items) k = -1;
    Item it{};
    if (k >= 0) {
      it = item_of(a, a.item_base + k);
      it.diag = it.L > 0 && block_of(a, it, it.L - 1) == it.I ? 1 : 0;
    }
    volatile FeedItem* e = &feed.slot[s];
    e->h = it.h;
    e->I = it.I;
    e->hk = it.hk;
    e->L = it.L;
    e->diag = it.diag;
    e->beg = it.beg;
    e->k = k;
    mbar_arrive(&feed.full[s]);
    if (k < 0) break;
    if (item_idx > 0 && !mbar_wait(q_empty, (item_idx - 1) & 1, a.err, abort_flag, tmo)) break;
    const int qrow = it.h * a.n + it.I * kBlk;
    mbar_arrive_expect_tx(q_full, kTileBytes);
    tma_load_3d(sQ, tmQ, q_full, 0, qrow, 0);
    ++q_loads;
    for (int j = 0; j < it.L; ++j) {
      int kb = block_of(a, it, j);
      if (kb < 0 || kb > it.I) {
        atomicOr(a.err, kErrRange);
        kb = it.I;
      }
      const int ks = gk % kKS;
      if (gk >= kKS && !mbar_wait(&k_empty[ks], ((gk / kKS) + 1) & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&k_full[ks], kTileBytes);
      tma_load_3d(sK + ks * kTileBytes, tmK, &k_full[ks], 0, it.hk * a.n + kb * kBlk, 0);
      ++gk;
    }
  }
  if (q_loads > 0) drain_wait(q_full, (q_loads - 1) & 1, a.err, tmo);
  for (int g = max(0, gk - kKS); g < gk; ++g)
    drain_wait(&k_full[g % kKS], (g / kKS) & 1, a.err, tmo);
}

// The fast pass's V producer: the items of the feed, in order.
template <int kVS>
__device__ __forceinline__ void produce_v_feed(const AttnArgs& a, const CUtensorMap* tmV,
                                               uint8_t* sV, uint64_t* v_full, uint64_t* v_empty,
                                               const ItemFeed& feed, volatile int* abort_flag,
                                               uint64_t tmo) {
  tma_prefetch_desc(tmV);
  int gv = 0;
  bool ok = true;
  for (int item_idx = 0; ok; ++item_idx) {
    Item it;
    const int k = feed_next(feed, item_idx, it, a.err, abort_flag, tmo);
    if (k < 0) break;
    for (int j = 0; j < it.L; ++j) {
      int kb = block_of(a, it, j);
      if (kb < 0 || kb > it.I) kb = it.I;
      const int s = gv % kVS;
      if (gv >= kVS && !mbar_wait(&v_empty[s], ((gv / kVS) + 1) & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&v_full[s], kTileBytes);
      tma_load_3d(sV + s * kTileBytes, tmV, &v_full[s], 0, it.hk * a.n + kb * kBlk, 0);
      ++gv;
    }
  }
  for (int g = max(0, gv - kVS); g < gv; ++g)
    drain_wait(&v_full[g % kVS], (g / kVS) & 1, a.err, tmo);
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_rescue_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  // The rescue pass is launched on a full grid before the number of listed rows is known.
  const int num_items = a.list_count != nullptr ? *a.list_count : a.num_items;
  if (static_cast<int>(blockIdx.x) >= num_items) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTileBytes;
  uint8_t* sV = sK + kKStages * kTileBytes;
  float* sML = reinterpret_cast<float*>(sV + kVStages * kTileBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sML) + kMLBytes);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;    // [3]
  uint64_t* k_empty = bars + 5;   // [3]
  uint64_t* v_full = bars + 8;    // [2]
  uint64_t* v_empty = bars + 10;  // [2]
  uint64_t* s_full = bars + 12;   // [2] per tile
  uint64_t* p_full = bars + 14;   // [2] per tile
  uint64_t* o_done = bars + 16;
  uint64_t* o_free = bars + 17;
  uint64_t* ml_ready = bars + 18;
  uint64_t* drain = bars + 19;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
    }
    mbar_init(o_done, 1);
    mbar_init(o_free, 256);
    mbar_init(ml_ready, 256);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 8) {
    regs_decrease<kRescueLoaderRegs>();
  if (warp == 8) {
    if (lane == 0)
      produce_qk<kKStages>(a, num_items, &tmQ, &tmK, sQ, sK, q_full, q_empty, k_full, k_empty,
                           abort_flag, tmo);
  } else if (warp == 10) {
    if (lane == 0) produce_v<kVStages>(a, num_items, &tmV, sV, v_full, v_empty, abort_flag, tmo);
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_u32(sQ);
      int gk = 0, gv = 0, item_idx = 0;
      int cnt[2] = {0, 0};
      bool ok = true;
      for (int k = blockIdx.x; k < num_items && ok; k += gridDim.x, ++item_idx) {
        const Item it = get_item(a, k, gridDim.x, num_items);
        if (!mbar_wait(q_full, item_idx & 1, a.err, abort_flag, tmo)) {
          ok = false;
          break;
        }
        bool first_pv = true;
        auto do_pv = [&](int jj) -> bool {
          const int tt = jj & 1;
          if (!mbar_wait(&p_full[tt], cnt[tt] & 1, a.err, abort_flag, tmo)) return false;
          ++cnt[tt];
          if (first_pv) {
            if (item_idx > 0 &&
                !mbar_wait(o_free, (item_idx - 1) & 1, a.err, abort_flag, tmo))
              return false;
            first_pv = false;
          }
          const int s = gv % kVStages;
          if (!mbar_wait(&v_full[s], (gv / kVStages) & 1, a.err, abort_flag, tmo)) return false;
          tc_fence_after();
          const uint32_t v_base = smem_u32(sV + s * kTileBytes);
          const uint32_t d = tmem + 256 + tt * 128;
          const uint32_t p = tmem + tt * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // B = V rows 16kk.. (keys): MN-major, 64-column regions 16 KB apart (LBO),
            // 8-row groups 1024 B apart (SBO).  A = P from TMEM, 8 columns per K step.
            umma_bf16_tmem_a(d, p + kk * 8, sdesc_sw128(v_base + kk * 2048, kTileBytes / 2, 1024),
                             kIdescPV, (jj >= 2 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&v_empty[s]);
          ++gv;
          return true;
        };
        for (int j = 0; j < it.L && ok; ++j) {
          const int t = j & 1;
          const int s = gk % kKStages;
          if (!mbar_wait(&k_full[s], (gk / kKStages) & 1, a.err, abort_flag, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_base = smem_u32(sK + s * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
            umma_bf16(tmem + t * 128, sdesc_sw128(q_base + off, 16, 1024),
                      sdesc_sw128(k_base + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
          }
          // (the K slot is released by the softmax warpgroup when it sees s_full: one
          // tcgen05.commit less per block)
          umma_commit(&s_full[t]);
          ++gk;
          if (j == it.L - 1) umma_commit(q_empty);
          if (j >= 1 && !do_pv(j - 1)) ok = false;
        }
        if (ok && it.L > 0) {
          if (!do_pv(it.L - 1)) ok = false;
          umma_commit(o_done);
        }
      }
      umma_commit(drain);
      drain_wait(drain, 0, a.err, tmo);
    }
  }
  } else {
    regs_increase<kRescueSoftmaxRegs>();
    // ------------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;         // tile: 0 for warps 0-3, 1 for warps 4-7
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;     // query row within the block
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + t * 128;
    const uint32_t o_addr = tmem + lane_off + 256 + t * 128;
    int ns = 0, item_idx = 0, gbase = 0;  // gbase: CTA-wide index of the item's first block
    bool ok = true;
    for (int k = blockIdx.x; k < num_items && ok; k += gridDim.x, ++item_idx) {
      const Item it = get_item(a, k, gridDim.x, num_items);
      float m_run = -FLT_MAX, l_run = 0.f;
      for (int jj = t; jj < it.L; jj += 2) {
        if (!warp_wait(&s_full[t], ns & 1, a.err, abort_flag, tmo)) {
          ok = false;
          break;
        }
        ++ns;
        tc_fence_after();
        // S_j is complete, so K_j's ring slot is free again.
        if ((warp & 3) == 0 && lane == 0) mbar_arrive(&k_empty[(gbase + jj) % kKStages]);
        const bool diag = block_of(a, it, jj) == it.I;
        const bool first = (jj == t);
        // The whole S row in one TMEM round trip.
        uint32_t v[128];
        tmem_ld128(s_addr, v);
        float alpha = 1.f, rs = 0.f;
        bool rescale = false;
        // Fast path: exponentiate against the running max without recomputing the row
        // maximum; accepted while every P stays below kLazySum.  Otherwise (and for the
        // tile's first block of the item) reload S, take the exact row maximum and raise
        // the running max when the block exceeds it by more than 2^kRescaleLog2.
        bool slow = first;
        if (!first) {
          rs = diag ? exp_pack<true>(v, a.scale_log2, m_run, r)
                    : exp_pack<false>(v, a.scale_log2, m_run, r);
          slow = __any_sync(0xffffffffu, !(rs <= kLazySum));
          if (slow) tmem_ld128(s_addr, v);
        }
        if (slow) {
          const float ms = (diag ? row_max<true>(v, r) : row_max<false>(v, r)) * a.scale_log2;
          if (first) {
            m_run = ms;
          } else if (ms > m_run + kRescaleLog2) {
            alpha = fast_exp2(m_run - ms);
            m_run = ms;
            rescale = true;
          }
          rs = diag ? exp_pack<true>(v, a.scale_log2, m_run, r)
                    : exp_pack<false>(v, a.scale_log2, m_run, r);
        }
        l_run = l_run * alpha + rs;
        tmem_st64p(s_addr, v);
        // s_full of this block implies the tile's previous P.V has completed, so O may
        // be rescaled here without another wait.
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(o_addr + c * 32, o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
            tmem_st32(o_addr + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        const bool drop = (a.debug & CRISP_DEBUG_DROP_ARRIVE) && blockIdx.x == 0 &&
                          item_idx == 0 && jj + 2 >= it.L;
        if (!drop) mbar_arrive(&p_full[t]);
      }
      gbase += it.L;
      if (!ok) break;
      // ---- epilogue: merge the two tiles' partial softmaxes, write this tile's half
      const int par = item_idx & 1;
      float* my = sML + ((par * 2 + t) * kBlk + r) * 2;
      const float* other = sML + ((par * 2 + (t ^ 1)) * kBlk + r) * 2;
      my[0] = m_run;
      my[1] = l_run;
      mbar_arrive(ml_ready);
      if (!warp_wait(ml_ready, item_idx & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      const float m_o = other[0], l_o = other[1];
      if (!warp_wait(o_done, item_idx & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float mA = t == 0 ? m_run : m_o, lA = t == 0 ? l_run : l_o;
      const float mB = t == 0 ? m_o : m_run, lB = t == 0 ? l_o : l_run;
      const bool hasB = it.L >= 2;
      const float m = hasB ? fmaxf(mA, mB) : mA;
      const float aA = fast_exp2(mA - m);
      const float aB = hasB ? fast_exp2(mB - m) : 0.f;
      const float inv = 1.f / (lA * aA + lB * aB);
      const float wA = aA * inv, wB = aB * inv;
      uint16_t* orow = a.O + (static_cast<size_t>(it.h) * a.n + static_cast<size_t>(it.I) * kBlk + r) * kD + t * 64;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t oa[32], ob[32];
        tmem_ld32(tmem + lane_off + 256 + t * 64 + hh * 32, oa);
        if (hasB) tmem_ld32(tmem + lane_off + 384 + t * 64 + hh * 32, ob);
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          float f[8];
#pragma unroll
          for (int x = 0; x < 8; ++x)
            f[x] = __uint_as_float(oa[c + x]) * wA + (hasB ? __uint_as_float(ob[c + x]) * wB : 0.f);
          uint4 pkt;
          pkt.x = pack_bf16(f[0], f[1]);
          pkt.y = pack_bf16(f[2], f[3]);
          pkt.z = pack_bf16(f[4], f[5]);
          pkt.w = pack_bf16(f[6], f[7]);
          *reinterpret_cast<uint4*>(orow + hh * 32 + c) = pkt;
        }
      }
      tc_fence_before();
      mbar_arrive(o_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// Fast pass.  TMEM: S0 [0,128) S1 [128,256) O [256,384) P0 [384,448) P1 [448,512).
// Each tile's P has its own columns, so the MMA warp computes a tile's next S block as
// soon as that tile's softmax has loaded the previous one, while the softmax is still
// exponentiating it: the tensor core always holds queued work.  The price is one O
// accumulator for both tiles, so both exponentiate against one reference per row: the
// larger of the exact row maxima of the two tiles' first blocks, exchanged once per item.
// The reference is never above the row's true maximum, so the largest P of the row is at
// least 1 and nothing that matters underflows; a block whose P row sum passes 2^64 (a logit
// more than 64 log2-units above the reference) marks its item for the rescue pass, which
// recomputes the item with per-tile running maxima.
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;
constexpr float kOverflowSum = 18446744073709551616.0f;  // 2^64
constexpr size_t kXBytes = 2 * 2 * kBlk * sizeof(float) + 16;  // row max, row sum per tile; flag
// Deeper K and V rings than the rescue pass: the dynamic shared memory must then start on
// a 1024-byte boundary (the 128-byte swizzle atoms), which the kernel checks instead of
// padding.
constexpr int kFastKStages = 4;
constexpr int kFastVStages = 2;
// Blocks alternate between the tiles by their CTA-wide index g (g & 1), so a tile's previous
// block is always g - 2 and the V slot of block g is P_t's slot too: one commit after P.V
// (v_empty[g & 1]) frees both the V slot and the P buffer.
static_assert(kFastVStages == 2, "v_empty doubles as the P buffers' release");
constexpr size_t kSmemFast = kTileBytes * (1 + kFastKStages + kFastVStages) + kXBytes + 512;

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrRange);
    return;
  }
  uint8_t* sQ = smem_raw;
  uint8_t* sK = sQ + kTileBytes;
  uint8_t* sV = sK + kFastKStages * kTileBytes;
  float* sXM = reinterpret_cast<float*>(sV + kFastVStages * kTileBytes);  // [tile][row] first-block max
  float* sXL = sXM + 2 * kBlk;                                         // [tile][row] row sum
  volatile int* sRedo = reinterpret_cast<volatile int*>(sXL + 2 * kBlk);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sXM) + kXBytes);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;                   // [kFastKStages]
  uint64_t* k_empty = k_full + kFastKStages;     // [kFastKStages]
  uint64_t* v_full = k_empty + kFastKStages;     // [kFastVStages]
  uint64_t* v_empty = v_full + kFastVStages;     // [kFastVStages]
  uint64_t* s_full = v_empty + kFastVStages;     // [2] S_t holds the tile's next block
  uint64_t* s_free = s_full + 2;                 // [2] the tile's softmax has loaded S_t
  uint64_t* p_full = s_free + 2;                 // [2] P_t written
  uint64_t* o_done = p_full + 2;
  uint64_t* o_free = o_done + 1;
  uint64_t* x_ready = o_free + 1;                // both tiles' first-block maxima are in sXM
  uint64_t* l_ready = x_ready + 1;               // both tiles' row sums are in sXL
  uint64_t* drain = l_ready + 1;                 // [2] one per MMA-issuing thread
  uint64_t* feed_full = drain + 2;               // [kItemRing]
  uint64_t* feed_empty = feed_full + kItemRing;  // [kItemRing]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(feed_empty + kItemRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const ItemFeed feed{reinterpret_cast<volatile FeedItem*>(tmem_slot + 2), feed_full, feed_empty};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t tmo = a.timeout_ns;
  const int num_items = a.num_items;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kFastKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kFastVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 4);   // one arrive per warp of the tile
      mbar_init(&p_full[t], 4);
    }
    mbar_init(o_done, 1);
    mbar_init(o_free, 8);       // one arrive per softmax warp
    mbar_init(x_ready, 8);
    mbar_init(l_ready, 8);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&feed_full[i], 1);
      mbar_init(&feed_empty[i], kItemReaders);
    }
    *sRedo = 0;
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 8) {
    regs_decrease<kLoaderRegs>();
    if (warp == 8) {
      if (lane == 0)
        produce_qk_feed<kFastKStages>(a, num_items, &tmQ, &tmK, sQ, sK, q_full, q_empty, k_full,
                                      k_empty, feed, abort_flag, tmo);
    } else if (warp == 10) {
      if (lane == 0)
        produce_v_feed<kFastVStages>(a, &tmV, sV, v_full, v_empty, feed, abort_flag, tmo);
    } else if (warp == 9) {
      // ---------------------------------------------------------------- S issuer
      // S_j = Q K_j^T into tile (j & 1)'s buffer, as soon as the tile's softmax has loaded
      // the buffer's previous block.  tcgen05.mma issue waits for the tensor core, so S
      // and P.V come from two threads: neither stream stalls the other while it waits.
      if (lane == 0) {
        const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16, 1024);
        // Block g goes to tile g & 1; the tile's previous block is g - 2, so its buffer and
        // barrier phases follow from g alone (phase of block g: (g >> 1) & 1).
        int gk = 0, item_idx = 0;
        bool ok = true;
        for (; ok; ++item_idx) {
          Item it;
          const int kf = feed_next(feed, item_idx, it, a.err, abort_flag, tmo);
          if (kf < 0) break;
          if (!mbar_wait(q_full, item_idx & 1, a.err, abort_flag, tmo)) {
            ok = false;
            break;
          }
          for (int j = 0; j < it.L; ++j) {
            const int t = gk & 1;
            const int s = gk % kFastKStages;
            if ((gk >= 2 && !mbar_wait(&s_free[t], ((gk - 2) >> 1) & 1, a.err, abort_flag, tmo)) ||
                !mbar_wait(&k_full[s], (gk / kFastKStages) & 1, a.err, abort_flag, tmo)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // Descriptors advance by byte offset >> 4 in the start-address field.
            const uint64_t dK = dK0 + static_cast<uint64_t>(s * (kTileBytes >> 4));
            const uint32_t d = tmem + t * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = ((kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32) >> 4;
              umma_bf16(d, dQ + off, dK + off, kIdescS, kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[t]);
            if (j == it.L - 1) umma_commit(q_empty);
            ++gk;
          }
        }
        umma_commit(&drain[0]);
        drain_wait(&drain[0], 0, a.err, tmo);
      }
    } else {
      // ---------------------------------------------------------------- P.V issuer (warp 11)
      // O += P_j V_j once P_j is written; the item's first group overwrites O, after the
      // previous item's epilogue has read it (o_free).
      if (lane == 0) {
        const uint64_t dV0 = sdesc_sw128(smem_u32(sV), kTileBytes / 2, 1024);
        int gv = 0, item_idx = 0;
        bool ok = true;
        for (; ok; ++item_idx) {
          Item it;
          const int kf = feed_next(feed, item_idx, it, a.err, abort_flag, tmo);
          if (kf < 0) break;
          for (int j = 0; j < it.L; ++j) {
            const int t = gv & 1;
            const int s = gv % kFastVStages;  // == t
            if (!mbar_wait(&p_full[t], (gv >> 1) & 1, a.err, abort_flag, tmo) ||
                (j == 0 && item_idx > 0 &&
                 !mbar_wait(o_free, (item_idx - 1) & 1, a.err, abort_flag, tmo)) ||
                !mbar_wait(&v_full[s], (gv / kFastVStages) & 1, a.err, abort_flag, tmo)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t dV = dV0 + static_cast<uint64_t>(s * (kTileBytes >> 4));
            const uint32_t p = tmem + kColP + t * 64;
            // B = V rows 16kk.. (keys): MN-major, 64-column regions 16 KB apart (LBO),
            // 8-row groups 1024 B apart (SBO).  A = P_t from TMEM, 8 columns per K step.
            umma_bf16_tmem_a(tmem + kColO, p, dV, kIdescPV, j > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 1; kk < 8; ++kk)
              umma_bf16_tmem_a(tmem + kColO, p + kk * 8, dV + ((kk * 2048) >> 4), kIdescPV, 1u);
            umma_commit(&v_empty[s]);
            ++gv;
          }
          if (ok) umma_commit(o_done);
        }
        umma_commit(&drain[1]);
        drain_wait(&drain[1], 0, a.err, tmo);
      }
    }
  } else {
    regs_increase<kSoftmaxRegs>();
    // ------------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;         // tile: 0 for warps 0-3, 1 for warps 4-7
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;     // query row within the block
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + t * 128;
    const uint32_t p_addr = tmem + lane_off + kColP + t * 64;
    int item_idx = 0, gbase = 0;  // gbase: CTA-wide index of the item's first block
    bool ok = true;
    uint32_t v[128];
    // Waits for the tile's next S block, loads it, hands the S buffer back to the MMA warp
    // and releases K_j's ring slot (S_j complete means K_j has been read).
    auto load_s = [&](int jj) -> bool {
      if (!warp_wait(&s_full[t], ((gbase + jj) >> 1) & 1, a.err, abort_flag, tmo)) return false;
      tc_fence_after();
      if (q == 0 && lane == 0) mbar_arrive(&k_empty[(gbase + jj) % kFastKStages]);
      tmem_ld128(s_addr, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[t]);
      return true;
    };
    for (; ok; ++item_idx) {
      Item it;
      const int kf = feed_next_warp(feed, item_idx, it, a.err, abort_flag, tmo);
      if (kf < 0) break;
      const int j0 = (t ^ gbase) & 1;  // this tile's first block: (gbase + j0) & 1 == t
      // Row reference: the larger of the two tiles' first-block row maxima.
      float mfirst = -FLT_MAX;
      if (j0 < it.L) {
        if (!load_s(j0)) {
          ok = false;
          break;
        }
        mfirst = (it.diag && j0 == it.L - 1 ? row_max<true>(v, r) : row_max<false>(v, r)) *
                 a.scale_log2;
      }
      sXM[t * kBlk + r] = mfirst;
      __syncwarp();
      if (lane == 0) mbar_arrive(x_ready);
      if (!warp_wait(x_ready, item_idx & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      const float M = fmaxf(sXM[r], sXM[kBlk + r]);
      float l = 0.f;
      bool ovf = false;
      for (int jj = j0; jj < it.L; jj += 2) {
        if (jj != j0 && !load_s(jj)) {
          ok = false;
          break;
        }
        const float rs = it.diag && jj == it.L - 1 ? exp_pack<true>(v, a.scale_log2, M, r)
                                                     : exp_pack<false>(v, a.scale_log2, M, r);
        ovf |= !(rs <= kOverflowSum);
        l += rs;
        // P_t last held block g - 2: wait for its P.V group (v_empty[t] completes once per
        // group of the blocks g' with g' & 1 == t, block g' completing phase g' / 2).
        const int g = gbase + jj;
        if (g >= 2 && !warp_wait(&v_empty[t], ((g - 2) >> 1) & 1, a.err, abort_flag, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st64p(p_addr, v);
        tmem_st_wait();
        tc_fence_before();
        const bool drop = (a.debug & CRISP_DEBUG_DROP_ARRIVE) && blockIdx.x == 0 &&
                          item_idx == 0 && jj + 2 >= it.L;
        __syncwarp();
        if (!drop && lane == 0) mbar_arrive(&p_full[t]);
      }
      gbase += it.L;
      if (!ok) break;
      // ---- epilogue: O / (l_0 + l_1); this tile writes columns [64t, 64t + 64)
      sXL[t * kBlk + r] = l;
      if (ovf) *sRedo = 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(l_ready);
      if (!warp_wait(l_ready, item_idx & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      const float inv = 1.f / (sXL[r] + sXL[kBlk + r]);
      if (threadIdx.x == 0 && *sRedo) {
        *sRedo = 0;
        a.redo[atomicAdd(a.redo_count, 1)] = it.h * a.nb + it.I;
      }
      if (!warp_wait(o_done, item_idx & 1, a.err, abort_flag, tmo)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint16_t* orow = a.O + (static_cast<size_t>(it.h) * a.n + static_cast<size_t>(it.I) * kBlk + r) * kD + t * 64;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kColO + t * 64 + hh * 32, o);
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint4 pkt;
          pkt.x = pack_bf16(__uint_as_float(o[c + 0]) * inv, __uint_as_float(o[c + 1]) * inv);
          pkt.y = pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
          pkt.z = pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
          pkt.w = pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + hh * 32 + c) = pkt;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Counting sort of the selection's rows into the work order of the fast kernel, a launch
// being `per` consecutive KV heads.  Within a launch: rows longer than kShortRow blocks by
// exact length, longest first (the long rows of PE heads: each streams its KV head's blocks
// from the first one up); then the short rows (VS heads) by length class, longest class
// first, and within a class by band of query blocks, so that rows whose local blocks
// overlap (neighbouring query blocks, and the query heads that share the KV head) run close
// together in time and find those blocks in L2.  Rows with the same key keep no particular
// order.
constexpr int kShortRow = 64;
constexpr int kShortClasses = kShortRow / 8;
constexpr int kBands = 32;
static_assert(kShortClasses * kBands == kOrderShortBins, "work-order bins of the short rows");
__host__ __device__ constexpr int order_bins_per_launch(int nb) {
  return nb + 1 + kShortClasses * kBands;
}
__device__ __forceinline__ int order_key(const int64_t* row_ptr, int row, int nb, int hq, int hkv,
                                         int group, int per) {
  const int h = row / nb, I = row % nb;
  const int hk = (h / hq) * hkv + (h % hq) / group;
  const int len = static_cast<int>(row_ptr[row + 1] - row_ptr[row]);
  const int base = (hk / per) * order_bins_per_launch(nb);
  if (len > kShortRow) return base + (nb - len);
  const int cls = (max(len, 1) - 1) >> 3;  // 0 .. kShortClasses - 1
  const int band = static_cast<int>((static_cast<int64_t>(I) * kBands) / nb);
  return base + (nb + 1) + (kShortClasses - 1 - cls) * kBands + band;
}

__global__ void order_hist_kernel(const int64_t* __restrict__ row_ptr, int rows, int nb, int hq,
                                  int hkv, int group, int per, int* hist) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row < rows) atomicAdd(&hist[order_key(row_ptr, row, nb, hq, hkv, group, per)], 1);
}

// In-place exclusive scan of nbins counts (one CTA).
__global__ void __launch_bounds__(1024) order_scan_kernel(int* hist, int nbins) {
  __shared__ int part[1024];
  const int per = (nbins + 1023) / 1024;
  const int p0 = threadIdx.x * per, p1 = min(nbins, p0 + per);
  int s = 0;
  for (int p = p0; p < p1; ++p) s += hist[p];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int t = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += t;
    __syncthreads();
  }
  int run = part[threadIdx.x] - s;
  for (int p = p0; p < p1; ++p) {
    const int c = hist[p];
    hist[p] = run;
    run += c;
  }
}

__global__ void order_scatter_kernel(const int64_t* __restrict__ row_ptr, int rows, int nb, int hq,
                                     int hkv, int group, int per, int* cursor, int32_t* order) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row < rows)
    order[atomicAdd(&cursor[order_key(row_ptr, row, nb, hq, hkv, group, per)], 1)] = row;
}

// The same counting sort in one CTA for short sequences (rows <= kOrderSmallRows and the
// histogram in shared memory): one launch instead of a memset and three.
constexpr int kOrderSmallRows = 16384;
constexpr int kOrderSmallBins = 12288;
__global__ void __launch_bounds__(1024) order_small_kernel(const int64_t* __restrict__ row_ptr,
                                                           int rows, int nb, int hq, int hkv,
                                                           int group, int per, int nbins,
                                                           int32_t* order) {
  extern __shared__ int hist[];  // [nbins]
  __shared__ int part[1024];
  for (int i = threadIdx.x; i < nbins; i += 1024) hist[i] = 0;
  __syncthreads();
  for (int row = threadIdx.x; row < rows; row += 1024)
    atomicAdd(&hist[order_key(row_ptr, row, nb, hq, hkv, group, per)], 1);
  __syncthreads();
  const int pc = (nbins + 1023) / 1024;
  const int p0 = threadIdx.x * pc, p1 = min(nbins, p0 + pc);
  int s = 0;
  for (int p = p0; p < p1; ++p) s += hist[p];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int t = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += t;
    __syncthreads();
  }
  int run = part[threadIdx.x] - s;
  for (int p = p0; p < p1; ++p) {
    const int c = hist[p];
    hist[p] = run;
    run += c;
  }
  __syncthreads();
  for (int row = threadIdx.x; row < rows; row += 1024)
    order[atomicAdd(&hist[order_key(row_ptr, row, nb, hq, hkv, group, per)], 1)] = row;
}

}  // namespace

// Launches of the attention work order for these shapes (1 or 3).
int order_launches(const Shape& s, int num_sms) {
  const int per = attention_kv_heads_per_launch(s, num_sms);
  const int nlaunch = (s.Hkv + per - 1) / per;
  const int64_t rows = static_cast<int64_t>(s.H) * s.nb;
  const int64_t nbins = static_cast<int64_t>(nlaunch) * order_bins_per_launch(s.nb);
  return rows <= kOrderSmallRows && nbins <= kOrderSmallBins ? 1 : 3;
}

// KV heads per launch of the fast kernel: enough rows for 8 per SM, and beyond that as many
// KV heads as keep their K and V (2 x n x 128 x 2 bytes each) within 48 MB of L2, so that
// short sequences run in few launches (each launch pays a start and a tail).
int attention_kv_heads_per_launch(const Shape& s, int num_sms) {
  const int per_kv = s.group * s.nb;
  int per = (8 * num_sms + per_kv - 1) / per_kv;
  const int64_t kv_bytes = 2ll * s.n * kD * 2;
  const int l2_fit = static_cast<int>((48ll << 20) / kv_bytes);
  per = per > l2_fit ? per : l2_fit;
  return per < 1 ? 1 : (per > s.Hkv ? s.Hkv : per);
}

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
  a.num_items = s.H * s.nb;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kD));
  a.row_ptr = ctx->ws.row_ptr;
  a.col = ctx->ws.col;
  a.order = ctx->ws.order;
  a.dense = dense ? 1 : 0;
  // One launch per group of `per` KV heads (every KV head owns group * N_b rows): all CTAs
  // of a launch then stream the same few KV heads' blocks, which keeps them in L2 (at 512k
  // tokens, 3x less DRAM traffic than one launch over every head).
  const int per_kv = s.group * s.nb;
  const int per = attention_kv_heads_per_launch(s, ctx->num_sms);
  const int nlaunch = (s.Hkv + per - 1) / per;
  if (!dense && order_launches(s, ctx->num_sms) == 1) {
    PhaseRange range("work order");
    const int rows = s.H * s.nb;
    const int nbins = nlaunch * order_bins_per_launch(s.nb);
    order_small_kernel<<<1, 1024, sizeof(int) * nbins, st>>>(ctx->ws.row_ptr, rows, s.nb, s.hq,
                                                             s.hkv, s.group, per, nbins,
                                                             ctx->ws.order);
  } else if (!dense) {
    PhaseRange range("work order");
    const int rows = s.H * s.nb;
    const int nbins = nlaunch * order_bins_per_launch(s.nb);
    cudaError_t e = cudaMemsetAsync(ctx->ws.len_hist, 0, sizeof(int) * nbins, st);
    if (e != cudaSuccess) return e;
    order_hist_kernel<<<(rows + 255) / 256, 256, 0, st>>>(ctx->ws.row_ptr, rows, s.nb, s.hq, s.hkv,
                                                          s.group, per, ctx->ws.len_hist);
    order_scan_kernel<<<1, 1024, 0, st>>>(ctx->ws.len_hist, nbins);
    order_scatter_kernel<<<(rows + 255) / 256, 256, 0, st>>>(ctx->ws.row_ptr, rows, s.nb, s.hq,
                                                             s.hkv, s.group, per,
                                                             ctx->ws.len_hist, ctx->ws.order);
  }
  a.O = static_cast<uint16_t*>(O);
  a.err = ctx->ws.err;
  a.timeout_ns = (ctx->debug_flags & CRISP_DEBUG_DROP_ARRIVE) ? 50000000ull : ctx->timeout_ns;
  a.debug = ctx->debug_flags;
  a.list = nullptr;
  a.list_count = nullptr;
  a.redo = ctx->ws.redo;
  a.redo_count = ctx->ws.redo_count;
  PhaseRange range("attention");
  cudaError_t e = cudaMemsetAsync(ctx->ws.redo_count, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ctx->ws.work_ctr, 0, sizeof(int) * nlaunch, st);
  if (e != cudaSuccess) return e;
  for (int g0 = 0; g0 < s.Hkv; g0 += per) {
    const int m = min(per, s.Hkv - g0);
    a.item_base = g0 * per_kv;
    a.num_items = m * per_kv;
    a.work_ctr = ctx->ws.work_ctr + g0 / per;
    const int grid = a.num_items < ctx->num_sms ? a.num_items : ctx->num_sms;
    attention_kernel<<<grid, kThreads, kSmemFast, st>>>(tmQ, tmK, tmV, a);
  }
  // Rescue pass over the rows the fast pass listed (usually none: each CTA then reads the
  // count and returns).
  AttnArgs r = a;
  r.item_base = 0;
  r.list = ctx->ws.redo;
  r.list_count = ctx->ws.redo_count;
  r.redo = nullptr;
  r.redo_count = nullptr;
  r.work_ctr = nullptr;
  attention_rescue_kernel<<<ctx->num_sms, kThreads, kSmem, st>>>(tmQ, tmK, tmV, r);
  return cudaGetLastError();
}

cudaError_t init_attention_attributes() {
  // setmaxnreg.inc waits until the registers it asks for are free, so the split must fit
  // in what the CTA is launched with: refuse to run a build whose count differs.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, attention_kernel);
  if (e != cudaSuccess) return e;
  if (static_cast<uint32_t>(fa.numRegs) != kLaunchRegs) return cudaErrorInvalidKernelImage;
  e = cudaFuncGetAttributes(&fa, attention_rescue_kernel);
  if (e != cudaSuccess) return e;
  if (static_cast<uint32_t>(fa.numRegs) != kLaunchRegs) return cudaErrorInvalidKernelImage;
  e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemFast));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attention_rescue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmem));
}

}  // namespace crisp
