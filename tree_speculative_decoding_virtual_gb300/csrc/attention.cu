// a2: tree-masked attention for every draft-tree node in one pass.
//
// "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on Ascend NPUs",
// technical summary 2.3: the teacher evaluates all speculative nodes at once
// under a tree attention mask that lets node k attend only to its own
// ancestor path (itself included), with no leakage across branches.
// "Speculative Decoding Hierárquico: Medusa, EAGLE-2 e Multi-Token
// Prediction", Medusa section: parallel nodes attend only to their direct
// ancestors.
//
// Layout of the work.  For one (sequence b, kv head) the query rows are the
// tree nodes times the q heads of that kv group, packed node-major
// (row = node * g + head-in-group), so the GQA group shares every K/V tile.
// A block owns 128 or 256 such rows and one split of the key range (split-KV,
// sized to fill the GPU).  K/V tiles come straight from the paged cache by
// TMA; Q K^T and P V run on the tensor cores (tcgen05.mma, bf16 in, fp32
// accumulate in tensor memory) with an online softmax between them.  Tiles
// that lie wholly inside the committed prefix are visible to every row and
// skip masking; tiles that reach the tree tail apply each row's ancestor
// bitmask.  The splits of one key range are merged into the bf16 output.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "sm100_ptx.cuh"
#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const uint16_t *q;
  const uint16_t *k;
  const uint16_t *v;
  const int32_t *table;
  int max_blocks, num_blocks;
  const int32_t *prefix_len;
  const int32_t *n_nodes;
  const uint32_t *mask;
  const int32_t *err;
  int N_max, Hq, Hkv, g, W, max_slots;
  float scale_log2;
  int chunk, splits, row_tiles, rows_pad;  // the host's uniform split of the key range
  // plan_mode 1: the uniform split; partials [B*Hkv][splits][rows_pad].
  // plan_mode 2: the split is planned on the device from the actual lengths
  // (tree_attn_plan_kernel); the grid is one block per work item (grid_items
  // of them) and item k's partials are rows [k * kTcRows, (k + 1) * kTcRows).
  int B, plan_mode, nsm, grid_items;
  int rpb;           // query rows per block: 256 (two row tiles) or 128 (one)
  int4 *plan_out;    // plan_mode 2: per sequence (first item, splits, chunk in key tiles, row tiles)
  int4 *plan_items;  // plan_mode 2: per block of the grid, its item (tree_attn_plan_kernel)
  uint16_t *part_o;  // fp16 partial rows [..][D]: the split's O / (l * c)
  int part_keep;     // 1: more blocks than fit at once, so the K/V streamed after a
                     // block's partial rows would evict them: they are stored with
                     // an evict-last L2 policy and dropped from L2 by the merge
  float4 *part_ml;   // one per partial row: (reference max in log2 units, sum l, scale c, 0)
  uint16_t *out;
  float *lse;
  int32_t *status;
  uint64_t wait_limit_ns;
  int test_stall;  // wait on a barrier nothing signals (exercises the timeout path)
  int direct;      // 1: one split per key range; rows go straight to the output
  // Reading through a deferred commit (all null: the plain layout).  Logical
  // slot s in [remap_base[b], remap_base[b] + remap_len[b]) of sequence b is
  // physical slot remap_src[b * remap_stride + s - remap_base[b]]; the tree's
  // node j is at physical slot tail_base[b] + j (null: P_b + j).
  const int32_t *remap_src, *remap_base, *remap_len, *tail_base;
  int remap_stride;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
// Power of two c with |x| / c < 1 for every |x| <= amax (1 when amax is 0).
// Split partials are stored as fp16 values of O / (l c): always in range, with
// an 11-bit significand, whatever the magnitude of V.
__device__ __forceinline__ float pow2_above(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 1.f;
  const int e = ((__float_as_uint(amax) >> 23) & 0xFF) - 127 + 1;  // 2^e > amax
  return __uint_as_float((uint32_t)(min(max(e, -126), 127) + 127) << 23);
}

// Sequence-level validity from the input lengths and records alone (no
// error flag: that one comes from the ancestor pass).
__device__ __forceinline__ bool seq_shape_ok(const AttnParams &p, int b, int &P, int &nb) {
  P = p.prefix_len[b];
  nb = p.n_nodes ? p.n_nodes[b] : p.N_max;
  if (nb < 1 || nb > p.N_max) return false;
  if (P < 0 || (long)P + nb > (long)p.max_slots || (long)P + nb > (long)p.max_blocks * kPage)
    return false;
  if (p.tail_base) {  // the tree at its own base must fit the sequence's table
    const int T = p.tail_base[b];
    if (T < 0 || (long)T + nb > (long)p.max_blocks * kPage) return false;
  }
  if (p.remap_len) {
    const int rb = p.remap_base[b], rl = p.remap_len[b];
    if (rl < 0 || rl > p.remap_stride || (rl > 0 && (rb < 0 || (long)rb + rl > (long)P))) return false;
  }
  return true;
}

// Sequence-level validity shared by the split and combine kernels.
__device__ __forceinline__ bool seq_ok(const AttnParams &p, int b, int &P, int &nb) {
  const bool shape = seq_shape_ok(p, b, P, nb);
  return shape && !(p.err && p.err[b] != 0);
}


// ===========================================================================
// tcgen05 path.  One block = up to 256 query rows (two 128-row tiles, A and
// B) x one split of the key range of one (sequence, kv head), walked in
// 128-key tiles.  Both row tiles consume every K/V tile, so each K/V byte
// brought to the SM feeds 256 rows (the GQA group of up to 256/g nodes).
//   warp 0:    reads the split's block ids; lane 0 then loads K tiles with
//              TMA into a 2-stage ring (a stage is refilled once both
//              Q K^T that read it completed)
//   warp 10:   lane 0 loads V tiles the same way (refilled once both P V
//              that read a stage completed); a warp of its own, so K and V
//              loads never wait on each other.  With two row tiles the
//              stages are released by row tile B's softmax group: S_Bj is
//              committed after every MMA that reads K_j or V_{j-1}
//   warp 1:    owns 512 TMEM columns; lane 0 issues every MMA and does
//              nothing else (it paces the tensor core): with two row tiles
//              its only waits are for P, since row tile A's softmax group
//              checks that V_j and K_{j+1} have landed before it hands over
//              P_Aj
//   warps 2-5: softmax of row tile A, warps 6-9: of row tile B; one TMEM lane
//              (= one query row) per thread
// Per 128-key tile j and row tile t:
//   S_tj = Q_t K_j^T  (M=128, N=128, K=D; A and B K-major) -> TMEM
//   P_tj = exp2(S_tj * scale * log2e - m) as bf16          -> TMEM, over S_tj
//   O_t += P_tj V_j   (M=128, N=D, K=128; A from TMEM, V read MN-major)
// The MMAs of a row tile form one chain (S_t0, P_t0 V_0, S_t1, P_t1 V_1, ...)
// and the two chains alternate on the tensor core, so the softmax of one row
// tile runs while the other's MMAs execute.  S_{t,j+1} is issued right
// behind P_tj V_j and MMAs complete in issue order, so when the softmax sees
// S_tj complete, every earlier MMA of the row tile has completed too: O may
// be rescaled and S_tj overwritten by P_tj with no further wait.  P is taken
// against a reference max m per row, raised lazily: the tile's max is
// computed only while the row has no reference yet or when its P would sum
// above 2^64 (a score more than 57 above m), and only then are m moved and O
// and the row sums rescaled (in TMEM).  Each row decides this on its own
// scores alone, so a row's result does not depend on the other rows of its
// warp.  Every sum stays far from fp32 overflow and P keeps its relative
// precision, so the result is the same softmax.  A tile's row is handled in two 64-key halves;
// if the second half raises m, the first half's P (already in TMEM) is
// rescaled too.  (The tile max is ALU work that the MMA-issuing warp, which
// shares an SM sub-partition with a softmax warp of each group, would wait
// behind.)
// K and V tiles are read straight from the paged cache by TMA (4-D view
// [block][kv head][slot][D], 128-byte swizzle): when the eight 16-slot
// blocks of a tile are consecutive one box fetches them, otherwise one box
// per block.  The epilogue writes O / (l c) in fp16 (c a power of two per
// row), staged in shared memory and stored with one bulk copy, plus the
// row's (max, sum, c).
// Every wait is bounded; on expiry the block flags TSD_STATUS_TIMEOUT, drains
// what it issued, frees its tensor memory and returns.
// ===========================================================================

constexpr int kTcThreads = 352;     // 11 warps
constexpr int kTcBM = 128;          // rows of one row tile (one MMA M)
constexpr int kTcRows = 256;        // rows of one block (two row tiles)
constexpr int kTcBN = 128;          // keys per tile
constexpr int kTcPagesPerTile = kTcBN / kPage;
constexpr int kTcStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 100 ms
constexpr int kTcMaxPages = 512;    // block ids of one split held in shared memory

template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;                   // 128-byte column blocks of a row
  static constexpr uint32_t kQHalf = kTcBM * 128;          // one column block of a Q row tile
  static constexpr uint32_t kQTile = kTcBM * D * 2;        // one Q row tile
  static constexpr uint32_t kKVHalf = kTcBN * 128;         // one column block of a K/V tile
  static constexpr uint32_t kTile = kTcBN * D * 2;         // one K or V tile
  static constexpr uint32_t kQ = 0;                        // Q_A, Q_B
  static constexpr uint32_t kK = 2 * kQTile;
  static constexpr uint32_t kV = kK + kTcStages * kTile;
  static constexpr uint32_t kBytes = kV + kTcStages * kTile;
  static constexpr uint32_t kAlloc = kBytes + 1024;        // + alignment slack
  static constexpr uint32_t kStaging = kK;                 // epilogue reuses the K/V rings
  static_assert(2 * kTcStages * kTile >= kTcRows * D * 2, "epilogue staging fits the rings");
  // per row tile t: S_t (128 columns; P_t, bf16 pairs, overwrites its first
  // 64) at t * 256, O_t (D columns) at t * 256 + 128
  static constexpr uint32_t kTmemS = 0;
  static constexpr uint32_t kTmemO = 128;
  static constexpr uint32_t kTmemTile = 256;
};

// Device-side split plan (plan_mode 2), for batches of up to kPlanMaxSeq
// sequences.  The work of (sequence b, kv head, row tile) is its key range of
// t_b = ceil((P_b + N_b) / 128) tiles.  For a chunk bound C (in tiles) the
// range is cut into n_b = ceil(t_b / C) pieces of ceil(t_b / n_b) tiles; each
// piece is one work item (one block).  With one resident block per SM the
// estimated time is waves x (longest piece + kPlanFixedTiles), waves =
// ceil(items / SMs); the plan takes the C (1..64) of least estimate (ties:
// the larger C), with items <= the grid and n_b <= kMaxSplits.  For a batch
// of equal lengths this is the host's uniform split; for ragged lengths long
// sequences get more pieces, so they no longer set the kernel's duration.
// Items are numbered by sequence (sequences with longer pieces first), then
// kv head, split, row tile.
constexpr int kPlanMaxSeq = 64;
constexpr int kMaxSplits = 32;                               // pieces of one key range
constexpr int kPlanMaxChunk = kTcMaxPages * kPage / kTcBN;   // 64 key tiles per item
constexpr int kPlanFixedTiles = 4;                           // per-item set-up + partials
constexpr int kPlanGroups = 5;                               // thread groups over the sequences
constexpr int kPlanMinTiles = 16;  // uniform blocks shorter than this keep the uniform split
constexpr int kSmallBlockTiles = 31;  // 256-row blocks of at most this many key tiles: use 128 rows
static_assert(kPlanMaxChunk == 64, "the plan key keeps C in 6 bits");

struct TcPlanShared {
  int tiles[kPlanMaxSeq];  // t_b (0: sequence skipped)
  int rtc[kPlanMaxSeq];    // row tiles that hold valid rows
  int items[kPlanMaxChunk], longest[kPlanMaxChunk], most[kPlanMaxChunk];  // per C
  unsigned best;  // (estimate << 6) | (64 - C), minimised (estimate clamped to 26 bits)
  int mine, first;          // this block's sequence (-1: none) and its first item
};

struct TcShared {
  int32_t pages[kTcMaxPages];  // block ids of the split
  uint64_t k_full[kTcStages], k_empty[kTcStages], v_full[kTcStages], v_empty[kTcStages];
  uint64_t s_full[2], p_full[2], o_final[2], q_full[2];
  uint64_t drain, never;
  float4 mrg[kTcBM];           // group 1's (m, l_sum, l_ex, -) per row (kv2)
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool tc_wait(uint64_t &bar, uint32_t parity, uint64_t limit,
                                        volatile int *abort) {
  using namespace sm100;
  if (mbar_wait(smem_addr(&bar), parity, limit)) return true;
  *abort = 1;
  return false;
}

// The device plan (see TcPlanShared), computed once per launch by one block
// of kTcThreads threads before the split kernel.  It writes
//   plan_seq[b]    (first item, splits n_b, chunk in key tiles, row tiles)
//   plan_items[k]  for every block k of the split kernel's grid: (b, kv head,
//                  rt | split << 5 | chunk << 11 | N_b << 18, P_b), or b = -1
//                  when block k has no item
// and reports sequences whose lengths do not fit (TSD_STATUS_BAD_LEN).
__global__ void __launch_bounds__(kTcThreads) tree_attn_plan_kernel(const AttnParams p) {
  __shared__ TcPlanShared ps;
  __shared__ int s_P[kPlanMaxSeq], s_nb[kPlanMaxSeq], s_first[kPlanMaxSeq + 1];
  __shared__ int s_chunk[kPlanMaxSeq], s_items[kPlanMaxSeq], s_n[kPlanMaxSeq], s_order[kPlanMaxSeq];
  pdl_trigger();
  const int tid = threadIdx.x;
  const int B = p.B;
  for (int i = tid; i < kPlanMaxChunk; i += blockDim.x) {
    ps.items[i] = 0;
    ps.longest[i] = 0;
    ps.most[i] = 0;
  }
  if (tid == 0) ps.best = ~0u;
  pdl_wait();
  if (tid < B) {
    int P, nb;
    const bool ok = seq_ok(p, tid, P, nb);
    ps.tiles[tid] = ok ? (P + nb + kTcBN - 1) / kTcBN : 0;
    ps.rtc[tid] = ok ? (nb * p.g + p.rpb - 1) / p.rpb : 0;
    s_P[tid] = P;
    s_nb[tid] = nb;
    if (!ok && p.status) {
      const int e = p.err ? p.err[tid] : 0;
      const int nbb = p.n_nodes ? p.n_nodes[tid] : p.N_max;
      if (e == 0 && nbb >= 1 && nbb <= p.N_max) atomicOr(p.status, TSD_STATUS_BAD_LEN);
    }
  }
  __syncthreads();
  // candidate C = 1 + (tid % 64); kPlanGroups groups of 64 threads share the sequences
  if (tid < kPlanGroups * kPlanMaxChunk) {
    const int ci = tid % kPlanMaxChunk;
    const int C = ci + 1;
    int items = 0, longest = 0, most = 0;
    for (int s = tid / kPlanMaxChunk; s < B; s += kPlanGroups) {
      const int t = ps.tiles[s];
      if (t == 0) continue;
      const int n = (t + C - 1) / C;
      items += p.Hkv * ps.rtc[s] * n;
      longest = max(longest, (t + n - 1) / n);
      most = max(most, n);
    }
    if (items > 0) {
      atomicAdd(&ps.items[ci], items);
      atomicMax(&ps.longest[ci], longest);
      atomicMax(&ps.most[ci], most);
    }
  }
  __syncthreads();
  if (tid < kPlanMaxChunk) {  // two full warps: one candidate per lane
    const int items = ps.items[tid];
    unsigned key = ~0u;
    if (items > 0 && items <= p.grid_items && ps.most[tid] <= kMaxSplits) {
      const long waves = (items + p.nsm - 1) / p.nsm;
      const long est = min(waves * (long)(ps.longest[tid] + kPlanFixedTiles), (1L << 26) - 1);
      key = ((unsigned)est << 6) | (unsigned)(kPlanMaxChunk - 1 - tid);
    }
    key = __reduce_min_sync(0xffffffffu, key);
    if ((tid & 31) == 0) atomicMin(&ps.best, key);
  }
  __syncthreads();
  // (no candidate: no sequence has work; every block gets b = -1)
  const int C = ps.best == ~0u ? 0 : kPlanMaxChunk - (int)(ps.best & 63u);
  // Items are numbered sequence by sequence, the sequences taken in order of
  // decreasing piece length (ties: increasing b), so the blocks dispatched
  // first get the longest pieces and the short ones fill in behind them; a
  // batch of equal lengths keeps the order b = 0, 1, ...
  if (tid < B) {
    const int t = C > 0 ? ps.tiles[tid] : 0;
    const int n = t > 0 ? (t + C - 1) / C : 0;
    s_chunk[tid] = n > 0 ? (t + n - 1) / n : 0;
    s_items[tid] = n > 0 ? p.Hkv * ps.rtc[tid] * n : 0;
    s_n[tid] = n;
  }
  __syncthreads();
  if (tid < B) {
    const int c = s_chunk[tid];
    int rank = 0;
    for (int s = 0; s < B; ++s) rank += (s_chunk[s] > c || (s_chunk[s] == c && s < tid)) ? 1 : 0;
    s_order[rank] = tid;
  }
  __syncthreads();
  if (tid < 32) {  // exclusive scan of the items in rank order, two ranks per lane
    const int r0 = 2 * tid, r1 = 2 * tid + 1;
    const int i0 = r0 < B ? s_items[s_order[r0]] : 0;
    const int i1 = r1 < B ? s_items[s_order[r1]] : 0;
    int incl = i0 + i1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += y;
    }
    const int f0 = incl - i0 - i1;
    if (r0 < B) s_first[s_order[r0]] = f0;
    if (r1 < B) s_first[s_order[r1]] = f0 + i0;
    if (tid == 31) s_first[kPlanMaxSeq] = incl;
  }
  __syncthreads();
  if (tid < B) p.plan_out[tid] = make_int4(s_first[tid], s_n[tid], s_chunk[tid], ps.rtc[tid]);
  __syncthreads();
  const int total = s_first[kPlanMaxSeq];
  for (int k = tid; k < p.grid_items; k += blockDim.x) {
    int4 e = make_int4(-1, 0, 0, 0);
    if (k < total) {
      // the sequence whose items contain k: first items grow with the rank,
      // so it is the last rank whose first item is <= k (sequences without
      // items rank last, their first item being the total, so the search
      // never stops on one)
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_first[s_order[mid]] <= k) lo = mid; else hi = mid - 1;
      }
      while (lo > 0 && ps.tiles[s_order[lo]] == 0) --lo;
      const int b = s_order[lo];
      const int t = ps.tiles[b];
      const int rtc = ps.rtc[b];
      const int n = (t + C - 1) / C;
      const int chunk = (t + n - 1) / n;
      const int local = k - s_first[b];
      const int rt = local % rtc;
      const int split = (local / rtc) % n;
      const int hkv = local / rtc / n;
      e = make_int4(b, hkv, rt | (split << 5) | (chunk << 11) | (s_nb[b] << 18), s_P[b]);
    }
    p.plan_items[k] = e;
  }
}

// Visibility of 32 consecutive key slots for one query row: bit i covers the
// slot whose tail index (slot - P) is j0 + i.  Prefix slots (j0 + i < 0) are
// visible; tail slot j is visible iff bit j of the row's ancestor mask is set;
// slots at or past the split's end (i >= remaining) are not.
__device__ __forceinline__ uint32_t visible_bits(const uint32_t *mrow, int W, int j0, int remaining,
                                                 bool row_valid) {
  uint32_t bits;
  if (j0 <= -32) {
    bits = 0xFFFFFFFFu;
  } else if (j0 < 0) {
    const int sh = -j0;  // 1..31 prefix slots first
    const uint32_t tail = row_valid ? __ldg(mrow) : 0u;
    bits = ((1u << sh) - 1u) | (tail << sh);
  } else if (!row_valid) {
    bits = 0u;
  } else {
    const int w0 = j0 >> 5;
    const uint32_t lo = w0 < W ? __ldg(mrow + w0) : 0u;
    const uint32_t hi = w0 + 1 < W ? __ldg(mrow + w0 + 1) : 0u;
    bits = __funnelshift_r(lo, hi, j0 & 31);
  }
  if (remaining < 32) bits &= remaining <= 0 ? 0u : ((1u << remaining) - 1u);
  return bits;
}

// Before the previous kernel on the stream has finished (programmatic launch),
// start pulling this block's inputs into L2: its Q rows, and the K/V of the
// first blocks of its split.  Only lines are prefetched (through the load/
// store unit: queuing prefetch boxes on the TMA unit delayed the real tile
// loads behind them); nothing read here is used, so inputs the previous
// kernel is still writing are harmless (L2 is the point of coherence for
// their later writes).
constexpr int kPrefetchPages = 16;  // 2 tiles of 128 keys

template <int D>
__device__ __forceinline__ void attn_prefetch(const AttnParams &p, int b, int hkv, int rt,
                                              int split, int warp, int lane) {
  using namespace sm100;
  const int P = p.prefix_len[b];
  const int nb = p.n_nodes ? p.n_nodes[b] : p.N_max;
  if (P < 0 || nb < 1 || nb > p.N_max || (long)P + nb > (long)p.max_slots ||
      (long)P + nb > (long)p.max_blocks * kPage)
    return;
  const int k_begin = split * p.chunk;
  if (k_begin >= P + nb) return;
  if (warp < 2) {
    // warp 0 prefetches K, warp 1 V: one 16-slot block of one head is 16*D*2
    // contiguous bytes; lane l covers lines l, l+32, ... of each block
    const uint16_t *cache = warp == 0 ? p.k : p.v;
    const int pg_first = k_begin / kPage;
    const int pg_last = min((min(P + nb, k_begin + p.chunk) - 1) / kPage, pg_first + kPrefetchPages - 1);
    for (int i = pg_first; i <= pg_last; ++i) {
      const int page = p.table[(size_t)b * p.max_blocks + i];
      if (page < 0 || page >= p.num_blocks) continue;
      const char *blk =
          reinterpret_cast<const char *>(cache + ((size_t)page * p.Hkv + hkv) * kPage * D);
      for (int off = lane * 128; off < kPage * D * 2; off += 32 * 128) prefetch_l2(blk + off);
    }
  } else if (warp < 10 && ((warp - 2) >> 2) * kTcBM < p.rpb) {
    const int row = rt * p.rpb + ((warp - 2) >> 2) * kTcBM + (warp & 3) * 32 + lane;
    if (row < nb * p.g) {
      const char *q = reinterpret_cast<const char *>(
          p.q + (((size_t)b * p.N_max + row / p.g) * p.Hq + hkv * p.g + row % p.g) * D);
      for (int off = 0; off < D * 2; off += 128) prefetch_l2(q + off);
    }
  }
}

// ---- uniform split of one piece per key range: rows straight to the output ----
// Output row of block row `row` (within the kv head's rows) of sequence b.
__device__ __forceinline__ size_t out_row(const AttnParams &p, int b, int hkv, int row) {
  return ((size_t)b * p.N_max + row / p.g) * p.Hq + hkv * p.g + row % p.g;
}

// Zeros and lse -inf for rows [row0, row0 + nrows) that are past the
// sequence's valid rows (all of them for a skipped sequence).
template <int D>
__device__ void write_invalid_rows(const AttnParams &p, int b, int hkv, int row0, int nrows,
                                   bool seq_valid, int rows_valid, int tid, int nthreads) {
  const int rows_all = p.N_max * p.g;
  for (int r = tid; r < nrows; r += nthreads) {
    const int row = row0 + r;
    if (row >= rows_all) break;
    if (seq_valid && row < rows_valid) continue;
    const size_t o = out_row(p, b, hkv, row);
    uint4 *dst = reinterpret_cast<uint4 *>(p.out + o * D);
#pragma unroll
    for (int k = 0; k < D / 8; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse) p.lse[o] = -INFINITY;
  }
}

// One row normalised straight from tensor memory: O / l_sum in bf16, lse from
// the fp32 sum (tO: the thread's TMEM lane of O).  Called by whole warps (the
// TMEM loads are warp-collective); only threads whose row is valid store.
template <int D>
__device__ __forceinline__ void write_row_direct(const AttnParams &p, size_t orow, bool valid,
                                                 uint32_t tO, float m, float l_sum, float l_ex) {
  using namespace sm100;
  const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
  uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D);
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(tO + c * 32, o);
    tmem_wait_ld();
    if (valid) {
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const float *f = reinterpret_cast<const float *>(&o[q8 * 8]);
        dst[c * 4 + q8] = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                                     pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
      }
    }
  }
  if (valid && p.lse) p.lse[orow] = l_ex > 0.f ? (m + log2f(l_ex)) * 0.6931471805599453f : -INFINITY;
}

// ---- reading through a deferred commit ----
// Where the keys of one (sequence, kv head) live when a deferred commit's
// record or a tree at its own base is in use.
struct SlotMap {
  const int32_t *trow;  // the sequence's block table row
  const int32_t *rsrc;  // physical slots of logical [rb, rb + rl)
  int rb, rl, P, tb;    // record, prefix length, tree base
  int k_end;            // end of the block's key range
  bool active;          // some logical slot is not at its own physical slot
};

__device__ __forceinline__ SlotMap slot_map(const AttnParams &p, int b, int P, int k_end) {
  SlotMap m;
  m.trow = p.table + (size_t)b * p.max_blocks;
  m.rsrc = p.remap_src ? p.remap_src + (size_t)b * p.remap_stride : nullptr;
  m.rb = p.remap_base ? p.remap_base[b] : 0;
  m.rl = p.remap_len ? p.remap_len[b] : 0;
  m.P = P;
  m.tb = p.tail_base ? p.tail_base[b] : P;
  m.k_end = k_end;
  m.active = (m.rsrc && m.rl > 0) || m.tb != P;
  return m;
}

// Whether logical key tile [ts, ts + bn) holds a slot that is not at its own
// physical slot.
__device__ __forceinline__ bool tile_moved(const SlotMap &m, int ts, int bn) {
  if (!m.active) return false;
  if (m.rl > 0 && ts < m.rb + m.rl && ts + bn > m.rb) return true;
  return m.tb != m.P && ts + bn > m.P;
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

// One key tile (bn slots) of K or V loaded slot by slot by the loader
// thread, into the layout the TMA boxes produce (64-column halves of bn rows,
// 128-byte swizzle), then a proxy fence and one arrival on `bar`.  Slots past
// the key range and slots whose block id is out of range read as zeros (the
// latter also set `bad`).
template <int D, int BN>
__device__ void load_tile_by_slot(const uint16_t *cache, const AttnParams &p, const SlotMap &m,
                                  int hkv, int ts, uint32_t dst, uint32_t bar, bool &bad) {
  using namespace sm100;
  for (int r = 0; r < BN; ++r) {
    const int s = ts + r;
    int phys = s;
    bool valid = s < m.k_end;
    if (valid) {
      if (s >= m.P) phys = m.tb + (s - m.P);
      else if (m.rsrc && s >= m.rb && s < m.rb + m.rl) phys = __ldg(m.rsrc + (s - m.rb));
    }
    int page = 0;
    if (valid) {
      page = phys >= 0 && phys < p.max_blocks * kPage ? __ldg(m.trow + phys / kPage) : -1;
      if (page < 0 || page >= p.num_blocks) {
        bad = true;
        valid = false;
        page = 0;
      }
    }
    const uint16_t *src = cache + (((size_t)page * p.Hkv + hkv) * kPage + (valid ? phys % kPage : 0)) * D;
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        cp_async16_zfill(dst + h * (BN * 128) + sw128_offset(r, c), src + h * 64 + c * 8, valid);
  }
  cp_async_wait_all();
  fence_proxy_async_smem();  // the tensor core reads these rows through the async proxy
  mbar_arrive(bar);
}

// Tile j of K (or V) into stage j % kTcStages of the ring: TMA boxes, or slot
// by slot where the tile holds a slot that is not at its own physical slot.
template <int D>
__device__ __forceinline__ void tc_load_tile(const CUtensorMap *m1, const CUtensorMap *m8,
                                             uint64_t *full, uint32_t ring, const int32_t *pages,
                                             int npg, int hkv, const uint16_t *cache,
                                             const AttnParams &p, const SlotMap &sm, int k_begin,
                                             bool &bad, int j) {
  using namespace sm100;
  using L = TcLayout<D>;
  const int st = j % kTcStages;
  if (tile_moved(sm, k_begin + j * kTcBN, kTcBN)) {
    load_tile_by_slot<D, kTcBN>(cache, p, sm, hkv, k_begin + j * kTcBN, ring + st * L::kTile,
                                smem_addr(&full[st]), bad);
    return;
  }
  const int g0 = j * kTcPagesPerTile;
  int pg[kTcPagesPerTile];
  bool run = true;
#pragma unroll
  for (int g = 0; g < kTcPagesPerTile; ++g) {
    pg[g] = pages[min(g0 + g, npg - 1)];
    run = run && pg[g] == pg[0] + g;
  }
  const uint32_t bar = smem_addr(&full[st]);
  mbar_arrive_expect_tx(bar, L::kTile);
#pragma unroll
  for (int h = 0; h < L::kHalves; ++h) {
    const uint32_t dst = ring + st * L::kTile + h * L::kKVHalf;
    if (run) {
      tma_load_4d(dst, m8, h * 64, 0, hkv, pg[0], bar);
    } else {
#pragma unroll
      for (int g = 0; g < kTcPagesPerTile; ++g)
        tma_load_4d(dst + g * kPage * 128, m1, h * 64, 0, hkv, pg[g], bar);
    }
  }
}

// Arrival of a loader on the MMA thread's hand-off barrier for phase ph: the
// loader's tile has landed and phase ph - 1 has completed (so the arrival
// cannot count toward an earlier phase; phase ph cannot complete without it).
__device__ __forceinline__ bool hand_over(uint64_t *hand, int ph, uint64_t &full, uint32_t parity,
                                          uint64_t lim, volatile int *abort) {
  using namespace sm100;
  if (!tc_wait(full, parity, lim, abort)) return false;
  if (ph > 0 && !tc_wait(*hand, (ph - 1) & 1, lim, abort)) return false;
  mbar_arrive(smem_addr(hand));
  return true;
}

// One loader thread: TMA loads of K (or V) tiles 0..ntiles-1 into a ring,
// waiting for a stage to be released before refilling it, then a drain so no
// copy is in flight when the block exits.  With `hand`, the loader also tells
// the MMA thread (through row tile A's P barrier, phase j) that the tile the
// MMAs after P_Aj read has landed: V_j (lag 0) or K_{j+1} (lag 1; the last
// phase, with no K tile after it, gets a plain arrival).
template <int D>
__device__ __forceinline__ void tc_load_tiles(const CUtensorMap *m1, const CUtensorMap *m8,
                                              uint64_t *full, uint64_t *empty, uint32_t ring,
                                              const int32_t *pages, int npg, int ntiles, int hkv,
                                              uint64_t lim, volatile int *abort,
                                              const uint16_t *cache, const AttnParams &p,
                                              const SlotMap &sm, int k_begin, bool &bad,
                                              uint64_t *hand, int lag) {
  using namespace sm100;
  using L = TcLayout<D>;
  int last_issued[kTcStages];
#pragma unroll
  for (int i = 0; i < kTcStages; ++i) last_issued[i] = -1;
  bool all = true;
  for (int j = 0; j < ntiles; ++j) {
    const int st = j % kTcStages;
    if (*abort || (j >= kTcStages && !tc_wait(empty[st], ((j / kTcStages) - 1) & 1, lim, abort))) {
      all = false;
      break;
    }
    tc_load_tile<D>(m1, m8, full, ring, pages, npg, hkv, cache, p, sm, k_begin, bad, j);
    last_issued[st] = j;
    if (hand && j >= lag && !hand_over(hand, j - lag, full[st], (j / kTcStages) & 1, lim, abort)) {
      all = false;
      break;
    }
  }
  if (hand && lag == 1 && all && ntiles >= 1) {
    const int ph = ntiles - 1;
    if (ph == 0 || tc_wait(*hand, (ph - 1) & 1, lim, abort)) mbar_arrive(smem_addr(hand));
  }
  // drain: the last loads issued into each stage have landed
#pragma unroll
  for (int st = 0; st < kTcStages; ++st)
    if (last_issued[st] >= 0)
      mbar_wait(smem_addr(&full[st]), (last_issued[st] / kTcStages) & 1, kDrainLimitNs);
}

// One S chain (K = D in D / 16 steps) from precomputed descriptors: one
// block of MMA instructions for D = 128.
template <int D>
__device__ __forceinline__ void tc_s_chain(uint32_t d, const uint64_t (&a)[D / 16],
                                           const uint64_t (&b)[D / 16], uint32_t idesc) {
  using namespace sm100;
  if constexpr (D == 128) {
    umma8_ss(d, a, b, idesc, 0u);
  } else {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) umma_bf16(d, a[kk], b[kk], idesc, kk > 0);
  }
}

// S_t = Q_q K^T for the K tile in stage st into the S columns of TMEM tile
// t, then a commit to s_full.  With `peek` nonzero, the phase `parity` of
// that barrier is tested (without waiting) while the last two MMAs are still
// queued, so the test's latency is hidden behind them; returns the result.
// Out of line: one copy of the code for every call site.
template <int D>
__device__ __noinline__ bool tc_issue_s(uint32_t tmem, uint32_t base, int q, int t, int st,
                                        uint32_t s_full, uint32_t peek, uint32_t parity) {
  using namespace sm100;
  using L = TcLayout<D>;
  constexpr uint32_t idS = idesc_bf16_f32(kTcBM, kTcBN, false, false);
  const uint64_t qd = smem_desc_sw128(base + L::kQ + q * L::kQTile, 16, 1024);
  const uint64_t kd = smem_desc_sw128(base + L::kK + st * L::kTile, 16, 1024);
  tc_fence_after();
  bool ready = false;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    if (kk == D / 16 - 2 && peek) ready = mbar_test(peek, parity);
    umma_bf16(tmem + t * L::kTmemTile + L::kTmemS,
              desc_add(qd, (kk >> 2) * L::kQHalf + (kk & 3) * 32),
              desc_add(kd, (kk >> 2) * L::kKVHalf + (kk & 3) * 32), idS, kk > 0);
  }
  umma_commit(s_full);
  return ready;
}

// O_t += P_t V for the V tile in stage st (P read from tensor memory); a
// commit to `final_bar` when it is nonzero.
template <int D>
__device__ __noinline__ void tc_issue_pv(uint32_t tmem, uint32_t base, int t, int st, bool accum,
                                         uint32_t final_bar) {
  using namespace sm100;
  using L = TcLayout<D>;
  constexpr uint32_t idPV = idesc_bf16_f32(kTcBM, D, false, true);
  const uint64_t vd = smem_desc_sw128(base + L::kV + st * L::kTile, L::kKVHalf, 1024);
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < kTcBN / 16; ++kk) {
    umma_bf16_ta(tmem + t * L::kTmemTile + L::kTmemO, tmem + t * L::kTmemTile + L::kTmemS + kk * 8,
                 desc_add(vd, kk * 16 * 128), idPV, (accum || kk > 0) ? 1u : 0u);
  }
  if (final_bar) umma_commit(final_bar);
}

// __launch_bounds__ for 384 threads caps registers at 168, which keeps three
// warps of 168 registers inside one SM sub-partition's register file; the
// kernel runs 352 threads.
template <int D>
__global__ void __launch_bounds__(384, 1)
tree_attn_split_tc(const AttnParams p, const __grid_constant__ CUtensorMap map_k1,
                   const __grid_constant__ CUtensorMap map_k8, const __grid_constant__ CUtensorMap map_v1,
                   const __grid_constant__ CUtensorMap map_v8) {
  using namespace sm100;
  using L = TcLayout<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ TcShared sh;

  pdl_trigger();
  // The work item: (row tile, split, sequence x kv head) from the grid for the
  // uniform split; under the device plan the grid is one block per item and
  // the item is known only once the plan kernel (the previous grid) has
  // finished, so until then (b, hkv, rt, split) is the uniform split's guess,
  // used for the prefetch.
  const bool planned = p.plan_mode == 2;
  const int item = blockIdx.x;
  int rt = planned ? item % p.row_tiles : blockIdx.x;
  int split = planned ? (item / p.row_tiles) % p.splits : blockIdx.y;
  const int zg = planned ? item / (p.row_tiles * p.splits) : blockIdx.z;
  int b = zg / p.Hkv;
  int hkv = zg % p.Hkv;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Under the device plan the grid has room for more items than the plan
  // may make; a block past the first wave starts once the plan kernel has
  // finished, and one with no item leaves before any set-up.
  if (planned && item >= p.nsm) {
    pdl_wait();
    if (__ldcg(&p.plan_items[item]).x < 0) return;
  }

  // Set-up touches no global memory, so it runs while the previous kernel on
  // the stream finishes (programmatic launch); so does the L2 prefetch.
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char *gbase = smem_raw + (base - raw);
  volatile int *abort = &sh.abort;
  const uint64_t lim = p.wait_limit_ns;

  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(smem_addr(&sh.k_full[i]), 1);
      mbar_init(smem_addr(&sh.k_empty[i]), 1);
      mbar_init(smem_addr(&sh.v_full[i]), 1);
      mbar_init(smem_addr(&sh.v_empty[i]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_addr(&sh.s_full[t]), 1);
      mbar_init(smem_addr(&sh.p_full[t]), t == 0 ? 6 : 4);
      mbar_init(smem_addr(&sh.o_final[t]), 1);
      mbar_init(smem_addr(&sh.q_full[t]), 4);
    }
    mbar_init(smem_addr(&sh.drain), 1);
    mbar_init(smem_addr(&sh.never), 1);
    sh.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_k1);
    tma_prefetch_desc(&map_k8);
    tma_prefetch_desc(&map_v1);
    tma_prefetch_desc(&map_v8);
  }
  if (warp == 1) tmem_alloc(smem_addr(&sh.tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  // Blocks of the first wave warm L2 while the previous kernel finishes; a
  // later block starts after that kernel has ended and loads at once.
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  if (b < p.B && lin < p.nsm) attn_prefetch<D>(p, b, hkv, rt, split, warp, lane);
  pdl_wait();

  int P = 0, nb = 0;
  bool run;
  int k_begin, k_end;
  size_t item_row0;  // first partial row of this item
  if (planned) {
    const int4 e = __ldcg(&p.plan_items[item]);
    run = e.x >= 0;
    b = run ? e.x : 0;
    hkv = e.y;
    rt = e.z & 31;
    split = (e.z >> 5) & 63;
    const int chunk = ((e.z >> 11) & 127) * kTcBN;
    nb = (e.z >> 18) & 511;
    P = e.w;
    k_begin = split * chunk;
    k_end = min(P + nb, k_begin + chunk);
    item_row0 = (size_t)item * kTcRows;
  } else {
    run = seq_ok(p, b, P, nb);
    if (!run && rt == 0 && split == 0 && hkv == 0 && tid == 0 && p.status) {
      const int e = p.err ? p.err[b] : 0;
      const int nbb = p.n_nodes ? p.n_nodes[b] : p.N_max;
      if (e == 0 && nbb >= 1 && nbb <= p.N_max) atomicOr(p.status, TSD_STATUS_BAD_LEN);
    }
    k_begin = split * p.chunk;
    k_end = min(P + nb, k_begin + p.chunk);
    item_row0 = ((size_t)zg * p.splits + split) * p.rows_pad + (size_t)rt * p.rpb;
  }
  const bool seq_valid = run;
  const int rows_valid = nb * p.g;
  const int seq_len = P + nb;
  run = run && rt * p.rpb < rows_valid && k_begin < seq_len;
  // row tiles with valid rows
  const int ntile_rows = p.rpb == kTcRows && rt * kTcRows + kTcBM < rows_valid ? 2 : 1;
  const int ntiles = (k_end - k_begin + kTcBN - 1) / kTcBN;
  const int pg_first = k_begin / kPage;
  const int npg = run ? (k_end - 1) / kPage - pg_first + 1 : 0;  // <= kTcMaxPages (host check)
  // One row tile and at least two key tiles: both softmax groups work on the
  // same rows, each on every other key tile, and merge at the end.
  const bool kv2 = ntile_rows == 1 && ntiles >= 2;

  if (!run) {
    // nothing to do for this block: straight to the teardown
  } else if (warp == 0 || warp == 10) {
    // --------------------------- loaders (TMA) ---------------------------
    if (warp == 0) {
      const int32_t *trow = p.table + (size_t)b * p.max_blocks;
      bool bad = false;
      for (int i = lane; i < npg; i += 32) {
        int page = __ldg(trow + pg_first + i);
        if (page < 0 || page >= p.num_blocks) {
          bad = true;
          page = 0;
        }
        sh.pages[i] = page;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0 && p.status) atomicOr(p.status, TSD_STATUS_BAD_PAGE);
    }
    asm volatile("bar.sync 2, 64;\n" ::: "memory");  // block ids visible to both loaders
    if (lane == 0) {
      const SlotMap sm = slot_map(p, b, P, k_end);
      bool bad = false;
      uint64_t *hand = kv2 ? nullptr : &sh.p_full[0];
      if (warp == 0)
        tc_load_tiles<D>(&map_k1, &map_k8, sh.k_full, sh.k_empty, base + L::kK, sh.pages, npg,
                         ntiles, hkv, lim, abort, p.k, p, sm, k_begin, bad, hand, 1);
      else
        tc_load_tiles<D>(&map_v1, &map_v8, sh.v_full, sh.v_empty, base + L::kV, sh.pages, npg,
                         ntiles, hkv, lim, abort, p.v, p, sm, k_begin, bad, hand, 0);
      if (bad && p.status) atomicOr(p.status, TSD_STATUS_BAD_PAGE);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // Fixed order: S_t0 for each row tile, then for every tile j and row tile
    // t: P_tj V_j followed by S_t,j+1.  Every wait is on a barrier at most one
    // phase ahead of the one wanted (the order bounds it), so parities are
    // unambiguous.
    if (lane == 0) {
      // K_j has landed; S_t is free.  Returns whether phase `parity` of `peek`
      // (when nonzero) had completed by the end of the issue.
      auto issue_s = [&](int t, int j, uint32_t peek = 0u, uint32_t parity = 0u) -> bool {
        return tc_issue_s<D>(tmem, base, kv2 ? 0 : t, t, j % kTcStages, smem_addr(&sh.s_full[t]),
                             peek, parity);
      };
      auto issue_pv = [&](int t, int j) {  // V_j has landed; P_tj is in TMEM
        const bool last = kv2 ? j + 2 >= ntiles : j == ntiles - 1;
        tc_issue_pv<D>(tmem, base, t, j % kTcStages, kv2 ? j >= 2 : j > 0,
                       last ? smem_addr(&sh.o_final[t]) : 0u);
      };
      bool ok = !p.test_stall || tc_wait(sh.never, 0, lim, abort);
      if (kv2) {
        // one row tile, two chains over alternate key tiles: tile j goes to
        // TMEM tile (and softmax group) j & 1; K_j is released after S_j, V_j
        // after P V_j
        ok = ok && tc_wait(sh.q_full[0], 0, lim, abort);
        for (int j = 0; ok && j < 2; ++j) {
          ok = tc_wait(sh.k_full[j], 0, lim, abort);
          if (ok) {
            issue_s(j, j);
            umma_commit(smem_addr(&sh.k_empty[j]));
          }
        }
        for (int j = 0; ok && j < ntiles; ++j) {
          const int w = j & 1;
          ok = !*abort && tc_wait(sh.p_full[w], (j >> 1) & 1, lim, abort);
          ok = ok && tc_wait(sh.v_full[j % kTcStages], (j / kTcStages) & 1, lim, abort);
          if (!ok) break;
          issue_pv(w, j);
          umma_commit(smem_addr(&sh.v_empty[j % kTcStages]));
          if (j + 2 < ntiles) {
            ok = tc_wait(sh.k_full[(j + 2) % kTcStages], ((j + 2) / kTcStages) & 1, lim, abort);
            if (ok) {
              issue_s(w, j + 2);
              umma_commit(smem_addr(&sh.k_empty[(j + 2) % kTcStages]));
            }
          }
        }
      } else {
        // one chain per row tile; the two chains alternate on the tensor core.
        // This thread paces the tensor core, so it does nothing else: the K
        // and V stages are released by the last row tile's softmax group, a
        // role that gave up is noticed through the bounded waits, and every
        // MMA descriptor is computed once, here, so that issuing a group of
        // MMAs is one block of MMA instructions.
        constexpr uint32_t idS = idesc_bf16_f32(kTcBM, kTcBN, false, false);
        constexpr uint32_t idPV = idesc_bf16_f32(kTcBM, D, false, true);
        uint64_t qa[2][D / 16], kb[kTcStages][D / 16], vb[kTcStages][kTcBN / 16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint64_t qd = smem_desc_sw128(base + L::kQ + i * L::kQTile, 16, 1024);
          const uint64_t kd = smem_desc_sw128(base + L::kK + i * L::kTile, 16, 1024);
          const uint64_t vd = smem_desc_sw128(base + L::kV + i * L::kTile, L::kKVHalf, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            qa[i][kk] = desc_add(qd, (kk >> 2) * L::kQHalf + (kk & 3) * 32);
            kb[i][kk] = desc_add(kd, (kk >> 2) * L::kKVHalf + (kk & 3) * 32);
          }
#pragma unroll
          for (int kk = 0; kk < kTcBN / 16; ++kk) vb[i][kk] = desc_add(vd, kk * 16 * 128);
        }
        // S_t = Q_t K^T from K stage st, then a commit to s_full[t] (the
        // branches keep every array index a constant)
        auto s_group = [&](int t, int st) {
          const uint32_t d = tmem + t * L::kTmemTile + L::kTmemS;
          tc_fence_after();
          if (t == 0) {
            if (st == 0) tc_s_chain<D>(d, qa[0], kb[0], idS);
            else tc_s_chain<D>(d, qa[0], kb[1], idS);
          } else {
            if (st == 0) tc_s_chain<D>(d, qa[1], kb[0], idS);
            else tc_s_chain<D>(d, qa[1], kb[1], idS);
          }
          umma_commit(smem_addr(&sh.s_full[t]));
        };
        // O_t += P_t V from V stage st (P read from tensor memory)
        auto pv_group = [&](int t, int st, bool accum, bool last) {
          const uint32_t d = tmem + t * L::kTmemTile + L::kTmemO;
          const uint32_t a = tmem + t * L::kTmemTile + L::kTmemS;
          tc_fence_after();
          if (st == 0) umma8_ts(d, a, vb[0], idPV, accum ? 1u : 0u);
          else umma8_ts(d, a, vb[1], idPV, accum ? 1u : 0u);
          if (last) umma_commit(smem_addr(&sh.o_final[t]));
        };
        ok = ok && tc_wait(sh.k_full[0], 0, lim, abort);
        for (int t = 0; ok && t < ntile_rows; ++t) {
          ok = tc_wait(sh.q_full[t], 0, lim, abort);
          if (ok) s_group(t, 0);
        }
        for (int j = 0; ok && j < ntiles; ++j) {
          const bool next = j + 1 < ntiles;
          const int st = j % kTcStages;
          for (int t = 0; ok && t < ntile_rows; ++t) {
            // P_tj is in TMEM (and, for row tile A, V_j and K_{j+1} have landed)
            ok = tc_wait(sh.p_full[t], j & 1, lim, abort);
            if (!ok) break;
            pv_group(t, st, j > 0, !next);
            if (next) s_group(t, st ^ 1);
          }
        }
      }
      // drain: every MMA issued above has completed
      umma_commit(smem_addr(&sh.drain));
      mbar_wait(smem_addr(&sh.drain), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------ softmax ------------------------------
    const int t = (warp - 2) >> 2;                    // group: TMEM tile and barriers
    const int tr = kv2 ? 0 : t;                       // row tile of this group
    const int quarter = warp & 3;                     // TMEM lanes 32*quarter .. +31
    const int rl = quarter * 32 + lane;               // row within the row tile
    const int row = rt * p.rpb + tr * kTcBM + rl;
    const bool active = kv2 || t < ntile_rows;
    const bool rvalid = row < rows_valid;
    const int node = rvalid ? row / p.g : 0;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t *mrow = p.mask + ((size_t)b * p.N_max + node) * p.W;
    const uint32_t tS = tmem + t * L::kTmemTile + L::kTmemS + lane_off;
    const uint32_t tO = tmem + t * L::kTmemTile + L::kTmemO + lane_off;

    // waits are taken by every lane and their outcome made warp-uniform, so the
    // .sync.aligned TMEM accesses below are never reached by a partial warp
    auto warp_wait = [&](uint64_t &bar, uint32_t parity) -> bool {
      const bool got = !*abort && tc_wait(bar, parity, lim, abort);
      return __all_sync(0xffffffffu, got);
    };
    // bf16 pair -> the two values' sum
    auto pair_sum = [](uint32_t w) {
      return __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
    };
    // O (once a P V has written it) and this tile's first-half P, times alpha
    // (threads whose max did not move pass alpha = 1); returns the sum of the
    // first half's P as rounded again
    auto rescale = [&](float alpha, bool with_o, bool with_p) -> float {
      float psum = 0.f;
      if (with_o) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + c * 32, o);
        }
      }
      if (with_p) {
        tmem_wait_st();  // the first half's P stores have landed
        uint32_t q[32];
        tmem_ld32(tS, q);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q[i]));
          q[i] = pack_bf16(f.x * alpha, f.y * alpha);
          psum += pair_sum(q[i]);
        }
        tmem_st32(tS, q);
      }
      tmem_wait_st();
      return psum;
    };
    float m_use = -INFINITY, l_sum = 0.f, l_ex = 0.f;
    bool ok = active;
    if (active && (!kv2 || t == 0)) {
      // Q rows -> shared memory (128-byte swizzle) with cp.async: every copy is
      // in flight at once.  Each warp stages its 32 rows; one instruction
      // covers 32 / (D/8) consecutive rows, so global reads are contiguous.
      // Rows past the valid ones copy row 0 of the sequence (finite, unused).
      const uint32_t qt = base + L::kQ + tr * L::kQTile;
      constexpr int kCh = D / 8;               // 16-byte chunks per row
      constexpr int kRowsPer = 32 / kCh;       // rows per warp instruction
      const int ch = lane % kCh;
#pragma unroll
      for (int i = 0; i < 32 / kRowsPer; ++i) {
        const int r_in = quarter * 32 + i * kRowsPer + lane / kCh;  // row within the tile
        const int grow = rt * p.rpb + tr * kTcBM + r_in;
        const int gr = grow < rows_valid ? grow : 0;
        const uint16_t *src =
            p.q + (((size_t)b * p.N_max + gr / p.g) * p.Hq + hkv * p.g + gr % p.g) * D + ch * 8;
        cp_async_16(qt + (ch >> 3) * L::kQHalf + sw128_offset(r_in, ch & 7), src);
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sh.q_full[t]));
    }
    if (active) {
      const float sc = p.scale_log2;
      // this group's tiles: all of them, or every other one (kv2); u counts them
      for (int u = 0, j = kv2 ? t : 0; j < ntiles; ++u, j += kv2 ? 2 : 1) {
        if (!warp_wait(sh.s_full[t], u & 1)) {
          ok = false;
          break;
        }
        // S_tj is complete, and with it every earlier MMA of this row tile
        tc_fence_after();
        if (!kv2 && t == ntile_rows - 1 && warp == 2 + 4 * t && lane == 0) {
          // S_tj was committed after every other MMA that reads K_j or V_{j-1}
          // (a commit tracks all of the issuing thread's earlier MMAs): both
          // stages can be refilled
          mbar_arrive(smem_addr(&sh.k_empty[j % kTcStages]));
          if (j > 0) mbar_arrive(smem_addr(&sh.v_empty[(j - 1) % kTcStages]));
        }
        const int ts = k_begin + j * kTcBN;
        const bool full = (ts + kTcBN <= P) && (ts + kTcBN <= k_end);
        // Two row sums: l_sum adds P exactly as rounded to bf16 for the P V
        // product, so O / l_sum weighs every key alike; l_ex adds the fp32 P
        // and gives the row's log-sum-exp and its weight against other
        // splits.  Both hold the earlier tiles; lt / lte this tile's.
        float lt = 0.f, lte = 0.f;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {  // 64-key halves (one copy of the code)
          uint32_t r[2][32];
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) tmem_ld32(tS + h * 64 + c2 * 32, r[c2]);
          tmem_wait_ld();
          // masked scores become -inf; the max is taken on raw scores (scale > 0)
          if (!full) {
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const int k0 = ts + h * 64 + c2 * 32;
              const uint32_t vis = visible_bits(mrow, p.W, k0 - P, k_end - k0, rvalid);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (!((vis >> i) & 1u)) r[c2][i] = __float_as_uint(-INFINITY);
            }
          }
          // P is taken against the row's reference max with no max pass.  The
          // exact path takes the tile max and moves the reference (rescaling O
          // and the first half's P) for the rows that need it: a row with no
          // visible key yet, or one whose tile sums above 2^64 (a score more
          // than 57 above the reference, or a non-finite one).  Rows that need
          // nothing keep their reference and recompute the same P, so a row's
          // result depends on its own scores only.  Every P stays below 2^64
          // and a tile's sum below 2^71, far from fp32 overflow.
          const bool none = m_use == -INFINITY;
          bool exact = __all_sync(0xffffffffu, none), trig = false;
          const bool mixed = !exact && __any_sync(0xffffffffu, none);
          uint32_t pk[2][16];  // P as bf16 pairs: column i holds keys 2i, 2i+1 of a chunk
          unsigned long long esum2;
          float ra[2], rc[2];  // rounded P: even / odd keys
#pragma unroll 1
          for (;;) {
            if (exact) {
              // the max with three-input max instructions: 8 chains of 8 values
              float mx[8];
#pragma unroll
              for (int a = 0; a < 8; ++a) {
                const auto v = [&](int i) { return __uint_as_float(r[i >> 5][i & 31]); };
                float m = fmax3(v(a), v(a + 8), v(a + 16));
                m = fmax3(m, v(a + 24), v(a + 32));
                m = fmax3(m, v(a + 40), v(a + 48));
                mx[a] = fmaxf(m, v(a + 56));
              }
              const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]),
                                     fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7])) * sc;
              const float m_new = fmaxf(m_use, mt);
              const bool upd = none ? m_new > -INFINITY : trig;
              const float alpha = upd ? exp2f(m_use - m_new) : 1.f;
              if (__any_sync(0xffffffffu, upd) && (u > 0 || h > 0)) {
                const float s0 = rescale(alpha, u > 0, h > 0);
                if (h > 0 && upd) lt = s0;  // the first half's P as rounded again
              }
              if (upd) {
                l_sum *= alpha;
                l_ex *= alpha;
                lte *= alpha;  // (zero in the first half)
                m_use = m_new;
              }
            }
            const float mb = m_use == -INFINITY ? 0.f : m_use;
            // key pairs on packed fp32: one FMA for both arguments, one add for
            // the fp32 sum
            const unsigned long long sc2 = f2_pack(sc, sc), nmb2 = f2_pack(-mb, -mb);
            esum2 = f2_pack(0.f, 0.f);
            ra[0] = ra[1] = rc[0] = rc[1] = 0.f;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 x = f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c2][2 * i]),
                                                          __uint_as_float(r[c2][2 * i + 1])),
                                                  sc2, nmb2));
                const float a = ex2_approx(x.x);
                const float c = ex2_approx(x.y);
                pk[c2][i] = pack_bf16(a, c);
                esum2 = f2_add(esum2, f2_pack(a, c));
                add_bf16x2(ra[i & 1], rc[i & 1], pk[c2][i]);
              }
            }
            if (exact) break;
            const float2 e = f2_unpack(esum2);
            trig = !none && !(e.x + e.y <= 0x1p64f);
            exact = mixed || __any_sync(0xffffffffu, trig);
            if (!exact) break;
          }
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) tmem_st16(tS + h * 32 + c2 * 16, pk[c2]);
          const float2 es = f2_unpack(esum2);
          lt += (ra[0] + ra[1]) + (rc[0] + rc[1]);
          lte += es.x + es.y;
        }
        l_sum += lt;
        l_ex += lte;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        // p_full[0] counts six arrivals: its four warps and, with two row
        // tiles, the two loaders (V_j and K_{j+1} have landed); else warp 2
        // stands in for the loaders
        if (lane == 0) mbar_arrive_cnt(smem_addr(&sh.p_full[t]), kv2 && warp == 2 ? 3u : 1u);
      }
      if (ok) ok = warp_wait(sh.o_final[t], 0);  // this row tile's last P V
    }

    // ---- epilogue: O / (l c) in fp16 through shared memory, (m, l, c) per row ----
    // Every MMA of the block must be complete before the K/V rings are reused.
    // With kv2, group 1 hands its (m, l_sum, l_ex) to group 0 through shared
    // memory and group 0 folds group 1's O into its own before writing.
    const int nthr = kv2 ? 256 : ntile_rows * 128;
    if (kv2 && t == 1) sh.mrg[rl] = make_float4(m_use, l_sum, l_ex, ok ? 0.f : 1.f);
    if (active) asm volatile("bar.sync 1, %0;\n" ::"r"(nthr) : "memory");
    const bool writer = active && (!kv2 || t == 0);
    const int nwr = kv2 ? 128 : nthr;  // threads that stage rows
    const bool all_ok = __all_sync(0xffffffffu, writer && !*abort);
    if (all_ok && kv2) {
      tc_fence_after();
      const float4 o1 = sh.mrg[rl];
      const float m = fmaxf(m_use, o1.x);
      const float a0 = m_use == -INFINITY ? 0.f : exp2f(m_use - m);
      const float a1 = o1.x == -INFINITY ? 0.f : exp2f(o1.x - m);
      l_sum = a0 * l_sum + a1 * o1.y;
      l_ex = a0 * l_ex + a1 * o1.z;
      m_use = m;
      const uint32_t tO1 = tmem + L::kTmemTile + L::kTmemO + lane_off;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t x[32], y[32];
        tmem_ld32(tO + c * 32, x);
        tmem_ld32(tO1 + c * 32, y);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          x[i] = __float_as_uint(a0 * __uint_as_float(x[i]) + a1 * __uint_as_float(y[i]));
        tmem_st32(tO + c * 32, x);
      }
      tmem_wait_st();
    }
    if (p.direct) {  // one piece per key range: the row straight to the output
      if (all_ok) {
        tc_fence_after();
        const int wrow = rt * p.rpb + tr * kTcBM + rl;
        write_row_direct<D>(p, out_row(p, b, hkv, wrow), wrow < rows_valid, tO, m_use, l_sum, l_ex);
      }
    } else if (all_ok) {
      tc_fence_after();
      float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      float amax = 0.f;  // pass 1: the row's largest |O|
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(o[i])));
      }
      const float cs = pow2_above(amax * inv);
      inv /= cs;
      // staged row-major, 16-byte chunk k of a row at position k ^ (row % (D/8)),
      // so the 32 rows a warp writes at once hit distinct banks
      const int swz_mask = D / 8 - 1;
      unsigned char *srow = gbase + L::kStaging + (size_t)(tr * kTcBM + rl) * D * 2;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {  // pass 2: scale, round to fp16, stage
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          uint4 v;
          v.x = pack_f16(__uint_as_float(o[q8 * 8 + 0]) * inv, __uint_as_float(o[q8 * 8 + 1]) * inv);
          v.y = pack_f16(__uint_as_float(o[q8 * 8 + 2]) * inv, __uint_as_float(o[q8 * 8 + 3]) * inv);
          v.z = pack_f16(__uint_as_float(o[q8 * 8 + 4]) * inv, __uint_as_float(o[q8 * 8 + 5]) * inv);
          v.w = pack_f16(__uint_as_float(o[q8 * 8 + 6]) * inv, __uint_as_float(o[q8 * 8 + 7]) * inv);
          *reinterpret_cast<uint4 *>(srow + (((c * 4 + q8) ^ (rl & swz_mask)) << 4)) = v;
        }
      }
      const size_t prow = item_row0 + tr * kTcBM + rl;
      p.part_ml[prow] = make_float4(m_use, l_ex, cs, 0.f);
      fence_proxy_async_smem();
    }
    if (!p.direct) {
      if (writer) asm volatile("bar.sync 1, %0;\n" ::"r"(nwr) : "memory");
      if (all_ok && warp == 2 && lane == 0) {
        if (p.part_keep)  // kept in L2 ahead of the K/V stream for the merge kernel
          bulk_store_hint(p.part_o + item_row0 * D, base + L::kStaging, (uint32_t)(nwr * D * 2),
                          l2_policy_evict_last());
        else
          bulk_store(p.part_o + item_row0 * D, base + L::kStaging, (uint32_t)(nwr * D * 2));
        bulk_wait_read();
      }
    }
  }

  __syncwarp();  // role code above diverges inside warps; reconverge first
  tc_fence_before();
  __syncthreads();
  if (*abort && tid == 0 && p.status) atomicOr(p.status, TSD_STATUS_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (p.direct)
    write_invalid_rows<D>(p, b, hkv, rt * p.rpb, p.rpb, seq_valid, rows_valid, tid, kTcThreads);
}

// ===========================================================================
// Two blocks per SM, for launches whose blocks all hold one 128-row tile.  A
// block of six warps with 64-key tiles needs 96 KB of shared memory, 256
// tensor-memory columns and 192 threads of at most 168 registers, so two fit
// on an SM: while one sets up, waits for its first tile or writes its
// partials, the other streams.  One chain per block, over a double-buffered S:
//   warp 0:    lane 0 loads K tiles, lane 1 V tiles (TMA into 2-stage rings
//              of 64 keys; one 4-block box per 64-column half when the tile's
//              blocks are consecutive, else one box per block)
//   warp 1:    owns the tensor memory; lane 0 issues every MMA
//   warps 2-5: softmax, one TMEM lane (= one query row) per thread
// Per 64-key tile j: S_j = Q K_j^T into S buffer j & 1 (M=128, N=64); P_j as
// bf16 over that buffer's first 32 columns; O += P_j V_j.  Issue order S_0,
// S_1, P_0 V_0, S_2, P_1 V_1, S_3, ...: S_{j+2} reuses the buffer P_j V_j
// reads (the tensor pipe runs in issue order), and while the softmax works on
// S_j the tensor core computes S_{j+1} and P_{j-1} V_{j-1}.  So a P V may still
// be running when the next tile's softmax raises a row's reference max; the
// rescale of O that the lazy rule then needs first waits for it (pv_done).
// Partials, waits, time-outs and teardown are as in tree_attn_split_tc.
// ===========================================================================
constexpr int kDualThreads = 192;
constexpr int kDualBN = 64;                             // keys per tile
constexpr int kDualPagesPerTile = kDualBN / kPage;      // 4
constexpr uint32_t kDualTmemCols = 256;

template <int D>
struct DualLayout {
  static constexpr int kHalves = D / 64;                 // 128-byte column blocks of a row
  static constexpr uint32_t kQHalf = kTcBM * 128;
  static constexpr uint32_t kQTile = kTcBM * D * 2;
  static constexpr uint32_t kKVHalf = kDualBN * 128;
  static constexpr uint32_t kTile = kDualBN * D * 2;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQTile;
  static constexpr uint32_t kV = kK + 2 * kTile;
  static constexpr uint32_t kBytes = kV + 2 * kTile;
  static constexpr uint32_t kAlloc = kBytes + 1024;      // + alignment slack
  static constexpr uint32_t kStaging = kK;               // the epilogue reuses the K ring
  static_assert(2 * kTile >= kTcBM * D * 2, "epilogue staging fits the K ring");
  static constexpr uint32_t kTmemS = 0;                  // S buffer s at s * kDualBN
  static constexpr uint32_t kTmemO = 2 * kDualBN;
  static_assert(kTmemO + D <= kDualTmemCols, "S buffers and O fit the allocation");
};

struct DualShared {
  int32_t pages[kTcMaxPages];
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2];
  uint64_t pv_done, o_final, q_full, drain, never;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__device__ __forceinline__ void dual_load_tiles(const CUtensorMap *m1, const CUtensorMap *m4,
                                                uint64_t *full, uint64_t *empty, uint32_t ring,
                                                const int32_t *pages, int npg, int ntiles,
                                                int hkv, uint64_t lim, volatile int *abort,
                                                const uint16_t *cache, const AttnParams &p,
                                                const SlotMap &sm, int k_begin, bool &bad) {
  using namespace sm100;
  using L = DualLayout<D>;
  int last_issued[2] = {-1, -1};
  for (int j = 0; j < ntiles && !*abort; ++j) {
    const int st = j & 1;
    if (j >= 2 && !tc_wait(empty[st], ((j >> 1) - 1) & 1, lim, abort)) break;
    if (tile_moved(sm, k_begin + j * kDualBN, kDualBN)) {
      load_tile_by_slot<D, kDualBN>(cache, p, sm, hkv, k_begin + j * kDualBN, ring + st * L::kTile,
                                    smem_addr(&full[st]), bad);
      last_issued[st] = j;
      continue;
    }
    const int g0 = j * kDualPagesPerTile;
    int pg[kDualPagesPerTile];
    bool run = true;
#pragma unroll
    for (int g = 0; g < kDualPagesPerTile; ++g) {
      pg[g] = pages[min(g0 + g, npg - 1)];
      run = run && pg[g] == pg[0] + g;
    }
    const uint32_t bar = smem_addr(&full[st]);
    mbar_arrive_expect_tx(bar, L::kTile);
#pragma unroll
    for (int h = 0; h < L::kHalves; ++h) {
      const uint32_t dst = ring + st * L::kTile + h * L::kKVHalf;
      if (run) {
        tma_load_4d(dst, m4, h * 64, 0, hkv, pg[0], bar);
      } else {
#pragma unroll
        for (int g = 0; g < kDualPagesPerTile; ++g)
          tma_load_4d(dst + g * kPage * 128, m1, h * 64, 0, hkv, pg[g], bar);
      }
    }
    last_issued[st] = j;
  }
#pragma unroll
  for (int st = 0; st < 2; ++st)
    if (last_issued[st] >= 0)
      mbar_wait(smem_addr(&full[st]), (last_issued[st] >> 1) & 1, kDrainLimitNs);
}


template <int D>
__global__ void __launch_bounds__(kDualThreads, 2)
tree_attn_split_dual(const AttnParams p, const __grid_constant__ CUtensorMap map_k1,
                     const __grid_constant__ CUtensorMap map_k4,
                     const __grid_constant__ CUtensorMap map_v1,
                     const __grid_constant__ CUtensorMap map_v4) {
  using namespace sm100;
  using L = DualLayout<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ DualShared sh;

  pdl_trigger();
  // the work item, as in tree_attn_split_tc (the uniform split's guess until
  // the plan may be read)
  const bool planned = p.plan_mode == 2;
  const int item = blockIdx.x;
  int rt = planned ? item % p.row_tiles : blockIdx.x;
  int split = planned ? (item / p.row_tiles) % p.splits : blockIdx.y;
  const int zg = planned ? item / (p.row_tiles * p.splits) : blockIdx.z;
  int b = zg / p.Hkv;
  int hkv = zg % p.Hkv;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Under the device plan the grid has room for more items than the plan
  // may make; a block past the first wave starts once the plan kernel has
  // finished, and one with no item leaves before any set-up.
  if (planned && item >= p.nsm) {
    pdl_wait();
    if (__ldcg(&p.plan_items[item]).x < 0) return;
  }

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char *gbase = smem_raw + (base - raw);
  volatile int *abort = &sh.abort;
  const uint64_t lim = p.wait_limit_ns;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&sh.k_full[i]), 1);
      mbar_init(smem_addr(&sh.k_empty[i]), 1);
      mbar_init(smem_addr(&sh.v_full[i]), 1);
      mbar_init(smem_addr(&sh.v_empty[i]), 1);
      mbar_init(smem_addr(&sh.s_full[i]), 1);
      mbar_init(smem_addr(&sh.p_full[i]), 4);
    }
    mbar_init(smem_addr(&sh.pv_done), 1);
    mbar_init(smem_addr(&sh.o_final), 1);
    mbar_init(smem_addr(&sh.q_full), 4);
    mbar_init(smem_addr(&sh.drain), 1);
    mbar_init(smem_addr(&sh.never), 1);
    sh.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_k1);
    tma_prefetch_desc(&map_k4);
    tma_prefetch_desc(&map_v1);
    tma_prefetch_desc(&map_v4);
  }
  if (warp == 1) tmem_alloc(smem_addr(&sh.tmem_base), kDualTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  // With the uniform split the work item and everything the block reads up
  // to the tree's mask (lengths, block ids, K, V, Q) are inputs, not results
  // of the previous kernel on the stream (the ancestor pass, which releases
  // this grid early): the block streams and computes before it waits for that
  // kernel, and waits only before it reads the mask or the error flag and
  // before its first global write.  Under the device plan the item is known
  // only once the plan kernel (the previous grid) has finished; blocks of its
  // first wave warm L2 meanwhile.
  bool waited = planned;
  if (planned) {
    const int lin = blockIdx.x;
    if (b < p.B && lin < p.nsm) attn_prefetch<D>(p, b, hkv, rt, split, warp, lane);
    pdl_wait();
  }
  auto wait_prev = [&]() {
    if (!waited) {
      pdl_wait();
      waited = true;
    }
  };

  int P = 0, nb = 0;
  bool run;
  int k_begin, k_end;
  size_t item_row0;
  if (planned) {
    const int4 e = __ldcg(&p.plan_items[item]);
    run = e.x >= 0;
    b = run ? e.x : 0;
    hkv = e.y;
    rt = e.z & 31;
    split = (e.z >> 5) & 63;
    const int chunk = ((e.z >> 11) & 127) * kTcBN;
    nb = (e.z >> 18) & 511;
    P = e.w;
    k_begin = split * chunk;
    k_end = min(P + nb, k_begin + chunk);
    item_row0 = (size_t)item * kTcRows;
  } else {
    run = seq_shape_ok(p, b, P, nb);  // the error flag is read after the wait
    k_begin = split * p.chunk;
    k_end = min(P + nb, k_begin + p.chunk);
    item_row0 = ((size_t)zg * p.splits + split) * p.rows_pad + (size_t)rt * p.rpb;
  }
  const bool shape_ok = run;
  const int rows_valid = nb * p.g;
  run = run && rt * p.rpb < rows_valid && k_begin < P + nb;
  const int ntiles = (k_end - k_begin + kDualBN - 1) / kDualBN;
  const int pg_first = k_begin / kPage;
  const int npg = run ? (k_end - 1) / kPage - pg_first + 1 : 0;  // <= kTcMaxPages

  if (!run) {
    // nothing to do for this block
  } else if (warp == 0) {
    // --------------------------- loaders (TMA) ---------------------------
    const int32_t *trow = p.table + (size_t)b * p.max_blocks;
    bool bad = false;
    for (int i = lane; i < npg; i += 32) {
      int page = __ldg(trow + pg_first + i);
      if (page < 0 || page >= p.num_blocks) {
        bad = true;
        page = 0;
      }
      sh.pages[i] = page;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && p.status) atomicOr(p.status, TSD_STATUS_BAD_PAGE);
    __syncwarp();
    if (lane < 2) {
      const SlotMap sm = slot_map(p, b, P, k_end);
      bool bad_slot = false;
      if (lane == 0)
        dual_load_tiles<D>(&map_k1, &map_k4, sh.k_full, sh.k_empty, base + L::kK, sh.pages, npg,
                           ntiles, hkv, lim, abort, p.k, p, sm, k_begin, bad_slot);
      else
        dual_load_tiles<D>(&map_v1, &map_v4, sh.v_full, sh.v_empty, base + L::kV, sh.pages, npg,
                           ntiles, hkv, lim, abort, p.v, p, sm, k_begin, bad_slot);
      if (bad_slot && p.status) atomicOr(p.status, TSD_STATUS_BAD_PAGE);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      // Every MMA descriptor is computed once, here, so that a group of MMAs
      // is one block of MMA instructions (the issuing thread shares its SM
      // sub-partition with busy softmax warps); the K stages are released by
      // the softmax warps, which see each S complete.
      constexpr uint32_t idS = idesc_bf16_f32(kTcBM, kDualBN, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(kTcBM, D, false, true);
      uint64_t qa[D / 16], kb[2][D / 16], vb[2][kDualBN / 16];
      {
        const uint64_t qd = smem_desc_sw128(base + L::kQ, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) qa[kk] = desc_add(qd, (kk >> 2) * L::kQHalf + (kk & 3) * 32);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint64_t kd = smem_desc_sw128(base + L::kK + i * L::kTile, 16, 1024);
          const uint64_t vd = smem_desc_sw128(base + L::kV + i * L::kTile, L::kKVHalf, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) kb[i][kk] = desc_add(kd, (kk >> 2) * L::kKVHalf + (kk & 3) * 32);
#pragma unroll
          for (int kk = 0; kk < kDualBN / 16; ++kk) vb[i][kk] = desc_add(vd, kk * 16 * 128);
        }
      }
      auto issue_s = [&](int j) {  // K_j has landed; S buffer j & 1 is free
        const uint32_t d = tmem + L::kTmemS + (j & 1) * kDualBN;
        tc_fence_after();
        if (j & 1) tc_s_chain<D>(d, qa, kb[1], idS);
        else tc_s_chain<D>(d, qa, kb[0], idS);
        umma_commit(smem_addr(&sh.s_full[j & 1]));
      };
      bool ok = !p.test_stall || tc_wait(sh.never, 0, lim, abort);
      ok = ok && tc_wait(sh.q_full, 0, lim, abort);
      for (int j = 0; ok && j < 2 && j < ntiles; ++j) {
        ok = tc_wait(sh.k_full[j], 0, lim, abort);
        if (ok) issue_s(j);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        const int st = j & 1;
        ok = tc_wait(sh.p_full[st], (j >> 1) & 1, lim, abort);
        ok = ok && tc_wait(sh.v_full[st], (j >> 1) & 1, lim, abort);
        if (!ok) break;
        {
          const uint32_t d = tmem + L::kTmemO, a = tmem + L::kTmemS + st * kDualBN;
          tc_fence_after();
          if (st) umma4_ts(d, a, vb[1], idPV, j > 0 ? 1u : 0u);
          else umma4_ts(d, a, vb[0], idPV, j > 0 ? 1u : 0u);
          umma_commit(smem_addr(&sh.pv_done));
          if (j == ntiles - 1) umma_commit(smem_addr(&sh.o_final));
        }
        umma_commit(smem_addr(&sh.v_empty[st]));
        if (j + 2 < ntiles) {
          ok = tc_wait(sh.k_full[st], ((j + 2) >> 1) & 1, lim, abort);
          if (ok) issue_s(j + 2);
        }
      }
      // drain: every MMA issued above has completed
      umma_commit(smem_addr(&sh.drain));
      mbar_wait(smem_addr(&sh.drain), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------ softmax ------------------------------
    const int quarter = warp & 3;                      // TMEM lanes 32*quarter .. +31
    const int rl = quarter * 32 + lane;                // row within the tile
    const int row = rt * p.rpb + rl;
    const bool rvalid = row < rows_valid;
    const int node = rvalid ? row / p.g : 0;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t *mrow = p.mask + ((size_t)b * p.N_max + node) * p.W;
    const uint32_t tO = tmem + L::kTmemO + lane_off;
    auto warp_wait = [&](uint64_t &bar, uint32_t parity) -> bool {
      const bool got = !*abort && tc_wait(bar, parity, lim, abort);
      return __all_sync(0xffffffffu, got);
    };
    {
      // Q rows -> shared memory (128-byte swizzle), as in tree_attn_split_tc
      const uint32_t qt = base + L::kQ;
      constexpr int kCh = D / 8;
      constexpr int kRowsPer = 32 / kCh;
      const int ch = lane % kCh;
#pragma unroll
      for (int i = 0; i < 32 / kRowsPer; ++i) {
        const int r_in = quarter * 32 + i * kRowsPer + lane / kCh;
        const int grow = rt * p.rpb + r_in;
        const int gr = grow < rows_valid ? grow : 0;
        const uint16_t *src =
            p.q + (((size_t)b * p.N_max + gr / p.g) * p.Hq + hkv * p.g + gr % p.g) * D + ch * 8;
        cp_async_16(qt + (ch >> 3) * L::kQHalf + sw128_offset(r_in, ch & 7), src);
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sh.q_full));
    }
    float m_use = -INFINITY, l_sum = 0.f, l_ex = 0.f;
    bool ok = true;
    const float sc = p.scale_log2;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      if (!warp_wait(sh.s_full[st], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S_j was the last MMA to read K_j (the commit tracks it): the stage can
      // be refilled
      if (warp == 2 && lane == 0) mbar_arrive(smem_addr(&sh.k_empty[st]));
      const uint32_t tS = tmem + L::kTmemS + st * kDualBN + lane_off;
      const int ts = k_begin + j * kDualBN;
      const bool full = (ts + kDualBN <= P) && (ts + kDualBN <= k_end);
      uint32_t r[2][32];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) tmem_ld32(tS + c2 * 32, r[c2]);
      tmem_wait_ld();
      if (!full) {
        wait_prev();  // the mask is the ancestor pass's output
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int k0 = ts + c2 * 32;
          const uint32_t vis = visible_bits(mrow, p.W, k0 - P, k_end - k0, rvalid);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (!((vis >> i) & 1u)) r[c2][i] = __float_as_uint(-INFINITY);
        }
      }
      // P against the reference max, with the exact path (max, reference
      // moved, rescale) for rows that need it, as in tree_attn_split_tc
      const bool none = m_use == -INFINITY;
      bool exact = __all_sync(0xffffffffu, none), failed = false, trig = false;
      const bool mixed = !exact && __any_sync(0xffffffffu, none);
      uint32_t pk[2][16];  // P as bf16 pairs: column i holds keys 2i, 2i+1 of a chunk
      unsigned long long esum2;
      float ra[2], rc[2];  // rounded P: even / odd keys
#pragma unroll 1
      for (;;) {
        if (exact) {
          float mx[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) {
            const auto v = [&](int i) { return __uint_as_float(r[i >> 5][i & 31]); };
            float m = fmax3(v(a), v(a + 8), v(a + 16));
            m = fmax3(m, v(a + 24), v(a + 32));
            m = fmax3(m, v(a + 40), v(a + 48));
            mx[a] = fmaxf(m, v(a + 56));
          }
          const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]),
                                 fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7])) * sc;
          const float m_new = fmaxf(m_use, mt);
          // a row moves its reference only for its own first visible key or
          // its own tile sum above 2^64, never because a neighbour did
          const bool upd = none ? m_new > -INFINITY : trig;
          const float alpha = upd ? exp2f(m_use - m_new) : 1.f;
          if (__any_sync(0xffffffffu, upd) && j > 0) {
            // O holds P V of tiles before j - 1; the one of tile j - 1 may still run
            if (!warp_wait(sh.pv_done, (j - 1) & 1)) {
              failed = true;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + c * 32, o);
            }
          }
          if (upd) {
            l_sum *= alpha;
            l_ex *= alpha;
            m_use = m_new;
          }
        }
        const float mb = m_use == -INFINITY ? 0.f : m_use;
        const unsigned long long sc2 = f2_pack(sc, sc), nmb2 = f2_pack(-mb, -mb);
        esum2 = f2_pack(0.f, 0.f);
        ra[0] = ra[1] = rc[0] = rc[1] = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c2][2 * i]),
                                                      __uint_as_float(r[c2][2 * i + 1])),
                                              sc2, nmb2));
            const float a = ex2_approx(x.x);
            const float c = ex2_approx(x.y);
            pk[c2][i] = pack_bf16(a, c);
            esum2 = f2_add(esum2, f2_pack(a, c));
            add_bf16x2(ra[i & 1], rc[i & 1], pk[c2][i]);
          }
        }
        if (exact) break;
        const float2 e = f2_unpack(esum2);
        trig = !none && !(e.x + e.y <= 0x1p64f);
        exact = mixed || __any_sync(0xffffffffu, trig);
        if (!exact) break;
      }
      if (failed) {
        ok = false;
        break;
      }
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) tmem_st16(tS + c2 * 16, pk[c2]);
      const float2 es = f2_unpack(esum2);
      l_sum += (ra[0] + ra[1]) + (rc[0] + rc[1]);
      l_ex += es.x + es.y;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sh.p_full[st]));
    }
    if (ok) ok = warp_wait(sh.o_final, 0);  // the last P V

    // ---- epilogue: O / (l c) in fp16 through shared memory, (m, l, c) per row ----
    // (global writes only once the previous grid has finished: it may still
    // read what an earlier call wrote here)
    wait_prev();
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    const bool all_ok = __all_sync(0xffffffffu, ok && !*abort);
    if (p.direct) {  // one piece per key range: the row straight to the output
      if (all_ok && !(p.err && p.err[b] != 0)) {
        tc_fence_after();
        write_row_direct<D>(p, out_row(p, b, hkv, row), rvalid, tO, m_use, l_sum, l_ex);
      }
    } else if (all_ok) {
      tc_fence_after();
      float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      float amax = 0.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(o[i])));
      }
      const float cs = pow2_above(amax * inv);
      inv /= cs;
      const int swz_mask = D / 8 - 1;
      unsigned char *srow = gbase + L::kStaging + (size_t)rl * D * 2;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          uint4 v;
          v.x = pack_f16(__uint_as_float(o[q8 * 8 + 0]) * inv, __uint_as_float(o[q8 * 8 + 1]) * inv);
          v.y = pack_f16(__uint_as_float(o[q8 * 8 + 2]) * inv, __uint_as_float(o[q8 * 8 + 3]) * inv);
          v.z = pack_f16(__uint_as_float(o[q8 * 8 + 4]) * inv, __uint_as_float(o[q8 * 8 + 5]) * inv);
          v.w = pack_f16(__uint_as_float(o[q8 * 8 + 6]) * inv, __uint_as_float(o[q8 * 8 + 7]) * inv);
          *reinterpret_cast<uint4 *>(srow + (((c * 4 + q8) ^ (rl & swz_mask)) << 4)) = v;
        }
      }
      p.part_ml[item_row0 + rl] = make_float4(m_use, l_ex, cs, 0.f);
      fence_proxy_async_smem();
    }
    if (!p.direct) {
      asm volatile("bar.sync 1, 128;\n" ::: "memory");
      if (all_ok && warp == 2 && lane == 0) {
        if (p.part_keep)
          bulk_store_hint(p.part_o + item_row0 * D, base + L::kStaging, (uint32_t)(kTcBM * D * 2),
                          l2_policy_evict_last());
        else
          bulk_store(p.part_o + item_row0 * D, base + L::kStaging, (uint32_t)(kTcBM * D * 2));
        bulk_wait_read();
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  wait_prev();
  const bool seq_valid = shape_ok && !(p.err && p.err[b] != 0);
  if (!planned && !shape_ok && rt == 0 && split == 0 && hkv == 0 && tid == 0 && p.status) {
    const int e = p.err ? p.err[b] : 0;
    const int nbb = p.n_nodes ? p.n_nodes[b] : p.N_max;
    if (e == 0 && nbb >= 1 && nbb <= p.N_max) atomicOr(p.status, TSD_STATUS_BAD_LEN);
  }
  if (*abort && tid == 0 && p.status) atomicOr(p.status, TSD_STATUS_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kDualTmemCols);
  }
  if (p.direct)
    write_invalid_rows<D>(p, b, hkv, rt * p.rpb, kTcBM, seq_valid, rows_valid, tid, kDualThreads);
}

// One warp per output row (b, node, q head): merge the splits.  Lane s reads
// split s's (max, sum, scale).  A split's partial row is D/8 16-byte chunks,
// so one warp-wide load covers 32/(D/8) splits: lane l reads chunk l % (D/8)
// of split (l / (D/8)) + round * 32/(D/8).  Every load of every round is
// issued before any is used, so the merge costs one memory round trip; lanes
// holding the same chunk for different splits are then summed by shuffles.
// kDrop: the partials were kept in L2 (part_keep) and are dropped once read.
template <int D, int R, bool kDrop>  // R: rounds of loads per batch (R * 32 / (D/8) splits)
__global__ void __launch_bounds__(256) tree_attn_combine_kernel(const AttnParams p, int B) {
  constexpr int kChunks = D / 8;            // 16-byte chunks of a partial row
  constexpr int kPerRound = 32 / kChunks;   // splits covered by one warp-wide load
  pdl_trigger();
  pdl_wait();
  const int warp = (blockIdx.x * 256 + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long total = (long)B * p.N_max * p.Hq;
  if (warp >= total) return;
  const int hq = warp % p.Hq;
  const int node = (warp / p.Hq) % p.N_max;
  const int b = warp / (p.Hq * p.N_max);
  const int c = lane % kChunks;   // logical chunk of this lane
  const int so = lane / kChunks;  // split offset within a round
  uint16_t *dst = p.out + (size_t)warp * D + c * 8;

  // the device plan of sequence b, loaded beside its lengths (read only when b is valid)
  const int4 plan = p.plan_mode == 2 ? __ldcg(&p.plan_out[b]) : make_int4(0, 0, 0, 0);
  int P, nb;
  const bool ok = seq_ok(p, b, P, nb) && node < nb;
  if (!ok) {
    if (so == 0) *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse && lane == 0) p.lse[warp] = -INFINITY;
    return;
  }
  const int hkv = hq / p.g;
  const int row = node * p.g + (hq % p.g);
  // this row's partial for split 0, the distance between splits, their number
  size_t r0, stride;
  int ns;  // <= kMaxSplits
  if (p.plan_mode == 2) {
    const int4 pl = plan;  // (first item, splits, chunk, row tiles) of sequence b
    r0 = ((size_t)pl.x + (size_t)hkv * pl.y * pl.w + row / p.rpb) * kTcRows + row % p.rpb;
    stride = (size_t)pl.w * kTcRows;
    ns = pl.y;
  } else {
    r0 = (size_t)(b * p.Hkv + hkv) * p.splits * p.rows_pad + row;
    stride = p.rows_pad;
    ns = (P + nb + p.chunk - 1) / p.chunk;
  }
  // partial rows sit at multiples of 16 apart, so every split's copy of this
  // row has the same swizzle phase
  const int pc = c ^ (int)(r0 & (kChunks - 1));
  const float4 ml = lane < ns ? __ldcg(&p.part_ml[r0 + (size_t)lane * stride])
                              : make_float4(-INFINITY, 0.f, 0.f, 0.f);
  // partials in batches of R rounds; every load of a batch is issued before
  // any is used, the first batch before the weights are reduced
  uint4 raw[R];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int sp = s0 + r * kPerRound + so;
      raw[r] = sp < ns ? __ldcg(reinterpret_cast<const uint4 *>(
                             p.part_o + (r0 + (size_t)sp * stride) * D + pc * 8))
                       : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load_batch(0);
  float M = ml.x;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float wl = lane < ns ? exp2f(ml.x - M) * ml.y : 0.f;  // weight of split `lane`
  float L = wl;
  const float w = wl * ml.z;  // the split's partial holds O / (l c)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  float acc[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) acc[x] = 0.f;
  for (int s0 = 0;;) {  // ns is the same for the whole warp
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int sp = s0 + r * kPerRound + so;
      const float ws = __shfl_sync(0xffffffffu, w, sp & 31);
      if (sp < ns) {
        const uint32_t h[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[k]));
          acc[2 * k] += f.x * ws;
          acc[2 * k + 1] += f.y * ws;
        }
        // this row's 128-byte lines of split sp are read by no one else: kept
        // partials are dropped from L2 without a write-back (by the lane
        // holding a line's first chunk)
        if (kDrop && (pc & 7) == 0)
          sm100::discard_l2_line(p.part_o + (r0 + (size_t)sp * stride) * D + pc * 8);
      }
    }
    s0 += R * kPerRound;
    if (s0 >= ns) break;
    load_batch(s0);
  }
#pragma unroll
  for (int off = kChunks; off < 32; off <<= 1)
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[x] += __shfl_xor_sync(0xffffffffu, acc[x], off);
  if (so == 0) {
    const float inv = 1.f / L;
    *reinterpret_cast<uint4 *>(dst) =
        make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                   pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
  }
  if (p.lse && lane == 0) p.lse[warp] = (M + log2f(L)) * 0.6931471805599453f;
}

template <int D>
cudaError_t launch_combine(const AttnParams &p, int B, cudaStream_t s) {
  constexpr int kPerRound = 32 / (D / 8);
  const long rows = (long)B * p.N_max * p.Hq;
  const dim3 grid((unsigned)((rows * 32 + 255) / 256));
  // one batch for the uniform split's count; under the device plan (counts
  // known on the device only) batches of four rounds
  const int rounds = p.plan_mode == 2 ? 4 : (p.splits + kPerRound - 1) / kPerRound;
  if (p.part_keep) {
    if (rounds <= 4) return launch(tree_attn_combine_kernel<D, 4, true>, grid, dim3(256), 0, s, p, B);
    if (rounds <= 8) return launch(tree_attn_combine_kernel<D, 8, true>, grid, dim3(256), 0, s, p, B);
    return launch(tree_attn_combine_kernel<D, 32 / kPerRound, true>, grid, dim3(256), 0, s, p, B);
  }
  if (rounds <= 4) return launch(tree_attn_combine_kernel<D, 4, false>, grid, dim3(256), 0, s, p, B);
  if (rounds <= 8) return launch(tree_attn_combine_kernel<D, 8, false>, grid, dim3(256), 0, s, p, B);
  return launch(tree_attn_combine_kernel<D, 32 / kPerRound, false>, grid, dim3(256), 0, s, p, B);
}

struct AttnPlan {
  int bm, row_tiles, rows_pad, splits, chunk;
  int mode;          // plan_mode (AttnParams): 1 uniform split, 2 device plan
  bool dual;         // tree_attn_split_dual (two blocks per SM) instead of tree_attn_split_tc
  bool direct;       // uniform split of one piece: rows go straight to the output
  long grid_items;   // mode 2: blocks of the 1-D grid
  size_t o_bytes, ml_bytes, plan_bytes;
};

AttnPlan plan_attn(int B, int N_max, int Hq, int Hkv, int D, int max_slots) {
  AttnPlan a;
  const int g = Hq / Hkv;
  const long nsm = sm_count();
  const long max_tiles = (max_slots + kTcBN - 1) / kTcBN;
  // the uniform split for blocks of bm rows: `slots` block slots at once,
  // estimated time = waves x (tiles per block + a fixed cost of about four
  // 128-key tiles for the prologue and partials), plus about two tiles for
  // the merge kernel when a key range has more than one piece
  auto split_for = [&](int bm, long slots, long &per) {
    const long units = (long)B * Hkv * ((N_max * g + bm - 1) / bm);
    long best_s = 1;
    double best_t = 1e30;
    for (long s = 1; s <= max_tiles && s <= kMaxSplits; ++s) {
      const long waves = (units * s + slots - 1) / slots;
      const long pr = (max_tiles + s - 1) / s;
      const double t = (double)waves * (double)(pr + 4) + (s > 1 ? 2.0 : 0.0);
      if (t < best_t - 1e-9) {
        best_t = t;
        best_s = s;
        per = pr;
      }
    }
    return best_s;
  };
  // 128-row blocks (the two-blocks-per-SM kernel; the blocks of one kv
  // head's row tiles run side by side, so L2 serves their shared K/V) unless
  // 256-row blocks would each walk 32 or more key tiles: such long,
  // tensor-bound blocks gain from two row tiles sharing every K/V tile
  // (measured: the 70B shape, 128 rows 0.4% slower; 8B, budgeted and
  // dynamic-tree layers 2-7% faster with 128 rows).
  long per = 0;
  a.bm = kTcRows;
  long best_s = split_for(a.bm, nsm, per);
  if (per <= kSmallBlockTiles && N_max * g > kTcBM) {
    a.bm = kTcBM;
    best_s = split_for(a.bm, nsm, per);
  }
  // Blocks that all hold one 128-row tile run the two-blocks-per-SM kernel:
  // two block slots per SM.
  a.dual = a.bm == kTcBM || N_max * g <= kTcBM;
  if (a.dual) best_s = split_for(a.bm, 2 * nsm, per);
  a.row_tiles = (N_max * g + a.bm - 1) / a.bm;
  a.rows_pad = a.row_tiles * a.bm;
  const long units = (long)B * Hkv * a.row_tiles;
  long chunk = (max_slots + best_s - 1) / best_s;
  chunk = (chunk + kTcBN - 1) / kTcBN * kTcBN;
  if (chunk > (long)kTcMaxPages * kPage) chunk = (long)kTcMaxPages * kPage;
  if (chunk > 64L * kTcBN) chunk = 64L * kTcBN;  // at most 64 tiles per block
  while ((max_slots + chunk - 1) / chunk > kMaxSplits) chunk += kTcBN;
  a.chunk = (int)chunk;
  a.splits = (int)((max_slots + chunk - 1) / chunk);
  if (a.splits < 1) a.splits = 1;
  const long items_u = units * a.splits;  // work items of the uniform split
  // The device plan pays off only when lengths may differ (B > 1) and a
  // uniform block would walk many tiles; it costs one small kernel.
  a.mode = B > 1 && B <= kPlanMaxSeq && (a.chunk / kTcBN) >= kPlanMinTiles ? 2 : 1;
  a.direct = a.mode == 1 && a.splits == 1;
  a.grid_items = items_u;
  size_t rows = a.direct ? 0 : (size_t)B * Hkv * a.splits * a.rows_pad;
  if (a.mode == 2) {
    // room for four waves of shorter pieces per block slot (at least the
    // uniform split's blocks); blocks beyond the plan's items exit at once
    a.grid_items = std::min(std::max(items_u, (a.dual ? 8 : 4) * nsm), units * kMaxSplits);
    rows = (size_t)a.grid_items * kTcRows;
  }
  a.o_bytes = align_up(rows * D * sizeof(uint16_t), 256);
  a.ml_bytes = rows * sizeof(float4);
  a.plan_bytes = a.mode == 2 ? ((size_t)B + (size_t)a.grid_items) * sizeof(int4) : 0;
  return a;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 4-D view [block][kv head][slot][D] of a paged cache; a box covers 64
// columns of 16 slots of `pages` consecutive blocks of one head.
bool make_cache_map(CUtensorMap *m, const uint16_t *cache, int num_blocks, int Hkv, int D,
                    int pages) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPage, (cuuint64_t)Hkv, (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)kPage * D * 2,
                           (cuuint64_t)Hkv * kPage * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kPage, 1, (cuuint32_t)pages};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(cache), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_attn(AttnParams &p, const AttnPlan &a, int B, int num_blocks, cudaStream_t s) {
  const dim3 grid = a.mode == 2 ? dim3((unsigned)a.grid_items)
                                : dim3(p.row_tiles, p.splits, B * p.Hkv);
  const int pages = a.dual ? kDualPagesPerTile : kTcPagesPerTile;
  CUtensorMap k1, kn, v1, vn;
  if (!make_cache_map(&k1, p.k, num_blocks, p.Hkv, D, 1) ||
      !make_cache_map(&kn, p.k, num_blocks, p.Hkv, D, pages) ||
      !make_cache_map(&v1, p.v, num_blocks, p.Hkv, D, 1) ||
      !make_cache_map(&vn, p.v, num_blocks, p.Hkv, D, pages))
    return TSD_ERR_CUDA;
  if (a.mode == 2 && launch(tree_attn_plan_kernel, dim3(1), dim3(kTcThreads), 0, s, p) != cudaSuccess)
    return TSD_ERR_CUDA;
  cudaError_t e;
  if (a.dual) {
    if (!set_smem((const void *)tree_attn_split_dual<D>, DualLayout<D>::kAlloc)) return TSD_ERR_CUDA;
    e = launch(tree_attn_split_dual<D>, grid, dim3(kDualThreads), DualLayout<D>::kAlloc, s, p, k1, kn,
               v1, vn);
  } else {
    if (!set_smem((const void *)tree_attn_split_tc<D>, TcLayout<D>::kAlloc)) return TSD_ERR_CUDA;
    e = launch(tree_attn_split_tc<D>, grid, dim3(kTcThreads), TcLayout<D>::kAlloc, s, p, k1, kn, v1, vn);
  }
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return TSD_ERR_CUDA;
  if (!a.direct && launch_combine<D>(p, B, s) != cudaSuccess) return TSD_ERR_CUDA;
  return TSD_OK;
}

}  // namespace
}  // namespace tsd

static int attn_check_dims(int B, int N_max, int Hq, int Hkv, int D, int max_slots) {
  if (B < 0 || max_slots < 1) return TSD_ERR_ARG;
  if (N_max < 1 || N_max > tsd::kMaxNodes || (D != 64 && D != 128) || Hkv < 1 || Hq < Hkv ||
      Hq % Hkv != 0 || Hq / Hkv > 16 || B > 65535 || (long)B * Hkv > 65535)
    return TSD_ERR_LIMIT;
  // a key range is cut into at most kMaxSplits pieces of at most kPlanMaxChunk tiles
  if ((long)max_slots > (long)tsd::kMaxSplits * tsd::kPlanMaxChunk * tsd::kTcBN) return TSD_ERR_LIMIT;
  return TSD_OK;
}

TSD_API size_t tsd_tree_attn_workspace_bytes(int B, int N_max, int Hq, int Hkv, int D,
                                             int max_slots) {
  if (attn_check_dims(B, N_max, Hq, Hkv, D, max_slots) != TSD_OK || B == 0) return 0;
  const tsd::AttnPlan a = tsd::plan_attn(B, N_max, Hq, Hkv, D, max_slots);
  return a.o_bytes + a.ml_bytes + a.plan_bytes;
}

TSD_API int tsd_tree_attn_launches(int B, int N_max, int Hq, int Hkv, int D, int max_slots) {
  if (attn_check_dims(B, N_max, Hq, Hkv, D, max_slots) != TSD_OK || B == 0) return 0;
  const tsd::AttnPlan a = tsd::plan_attn(B, N_max, Hq, Hkv, D, max_slots);
  return a.mode == 2 ? 3 : a.direct ? 1 : 2;
}

TSD_API int tsd_tree_attn_plan(int B, int N_max, int Hq, int Hkv, int D, int max_slots,
                               int32_t *info) {
  if (!info) return TSD_ERR_ARG;
  const int dims = attn_check_dims(B, N_max, Hq, Hkv, D, max_slots);
  if (dims != TSD_OK) return dims;
  if (B == 0) return TSD_ERR_ARG;
  const tsd::AttnPlan a = tsd::plan_attn(B, N_max, Hq, Hkv, D, max_slots);
  info[0] = a.mode;
  info[1] = a.dual ? 1 : 0;
  info[2] = a.bm;
  info[3] = a.row_tiles;
  info[4] = a.splits;
  info[5] = a.chunk;
  info[6] = (int32_t)(a.mode == 2 ? a.grid_items : (long)a.row_tiles * a.splits * B * Hkv);
  info[7] = a.direct ? 1 : 0;
  return TSD_OK;
}

static int attn_fwd_impl(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                              const int32_t *block_table, int max_blocks, int num_blocks,
                              const int32_t *prefix_len, const int32_t *n_nodes,
                              const uint32_t *mask, const int32_t *err, int B, int N_max, int Hq,
                              int Hkv, int D, int max_slots, float scale, uint16_t *out,
                              float *lse, void *workspace, size_t ws_bytes, int32_t *status,
                              const int32_t *remap_src, int remap_stride,
                              const int32_t *remap_base, const int32_t *remap_len,
                              const int32_t *tail_base, tsd_stream_t stream) {
  using namespace tsd;
  const int dims = attn_check_dims(B, N_max, Hq, Hkv, D, max_slots);
  if (dims != TSD_OK) return dims;
  if (B == 0) return TSD_OK;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !mask || !out)
    return TSD_ERR_ARG;
  if (max_blocks < 1 || num_blocks < 1 || !(scale > 0.f) || !std::isfinite(scale))
    return TSD_ERR_ARG;
  if ((long long)num_blocks * Hkv * kPage > 0x7FFFFFFFLL) return TSD_ERR_LIMIT;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return TSD_ERR_ARG;
  const AttnPlan a = plan_attn(B, N_max, Hq, Hkv, D, max_slots);
  const size_t need = a.o_bytes + a.ml_bytes + a.plan_bytes;
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 16)))
    return TSD_ERR_WORKSPACE;
  AttnParams p;
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.table = block_table;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.prefix_len = prefix_len;
  p.n_nodes = n_nodes;
  p.mask = mask;
  p.err = err;
  p.N_max = N_max;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.W = (N_max + 31) / 32;
  p.max_slots = max_slots;
  p.scale_log2 = scale * kLog2e;
  p.chunk = a.chunk;
  p.splits = a.splits;
  p.row_tiles = a.row_tiles;
  p.rows_pad = a.rows_pad;
  p.rpb = a.bm;
  p.part_o = static_cast<uint16_t *>(workspace);
  p.part_ml = reinterpret_cast<float4 *>(static_cast<char *>(workspace) + a.o_bytes);
  p.plan_out = a.mode == 2 ? reinterpret_cast<int4 *>(static_cast<char *>(workspace) + a.o_bytes +
                                                      a.ml_bytes)
                           : nullptr;
  p.plan_items = a.mode == 2 ? p.plan_out + B : nullptr;
  p.B = B;
  p.plan_mode = a.mode;
  // blocks beyond one resident wave (the two-blocks-per-SM kernel fits two per
  // SM); under the device plan, the host's uniform guess of the item count
  p.part_keep = !a.direct && (long)a.row_tiles * a.splits * B * Hkv >
                                 (long)sm_count() * (a.dual ? 2 : 1);
  p.nsm = sm_count() * (a.dual ? 2 : 1);  // block slots the plan spreads items over
  p.grid_items = (int)a.grid_items;
  p.out = out;
  p.lse = lse;
  p.status = status;
  p.wait_limit_ns = (uint64_t)option(TSD_OPT_WAIT_LIMIT_NS);
  p.test_stall = (int)option(TSD_OPT_TEST_STALL);
  p.direct = a.direct ? 1 : 0;
  p.remap_src = remap_src;
  p.remap_base = remap_base;
  p.remap_len = remap_len;
  p.tail_base = tail_base;
  p.remap_stride = remap_stride;
  return D == 128 ? launch_attn<128>(p, a, B, num_blocks, as_cuda(stream))
                  : launch_attn<64>(p, a, B, num_blocks, as_cuda(stream));
}

TSD_API int tsd_tree_attn_fwd(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                              const int32_t *block_table, int max_blocks, int num_blocks,
                              const int32_t *prefix_len, const int32_t *n_nodes,
                              const uint32_t *mask, const int32_t *err, int B, int N_max, int Hq,
                              int Hkv, int D, int max_slots, float scale, uint16_t *out,
                              float *lse, void *workspace, size_t ws_bytes, int32_t *status,
                              tsd_stream_t stream) {
  return attn_fwd_impl(q, k_cache, v_cache, block_table, max_blocks, num_blocks, prefix_len,
                       n_nodes, mask, err, B, N_max, Hq, Hkv, D, max_slots, scale, out, lse,
                       workspace, ws_bytes, status, nullptr, 0, nullptr, nullptr, nullptr, stream);
}

TSD_API int tsd_tree_attn_fwd_remap(const uint16_t *q, const uint16_t *k_cache,
                                    const uint16_t *v_cache, const int32_t *block_table,
                                    int max_blocks, int num_blocks, const int32_t *prefix_len,
                                    const int32_t *n_nodes, const uint32_t *mask,
                                    const int32_t *err, int B, int N_max, int Hq, int Hkv, int D,
                                    int max_slots, float scale, const int32_t *remap_src,
                                    int remap_stride, const int32_t *remap_base,
                                    const int32_t *remap_len, const int32_t *tail_base,
                                    uint16_t *out, float *lse, void *workspace, size_t ws_bytes,
                                    int32_t *status, tsd_stream_t stream) {
  const bool rec = remap_src || remap_base || remap_len;
  if (rec && (!remap_src || !remap_base || !remap_len || remap_stride < 1 ||
              remap_stride > tsd::kMaxDepth + 1))
    return TSD_ERR_ARG;
  return attn_fwd_impl(q, k_cache, v_cache, block_table, max_blocks, num_blocks, prefix_len,
                       n_nodes, mask, err, B, N_max, Hq, Hkv, D, max_slots, scale, out, lse,
                       workspace, ws_bytes, status, remap_src, remap_stride, remap_base, remap_len,
                       tail_base, stream);
}
