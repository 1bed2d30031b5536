// Commit of one sequence's accepted path, shared by the commit kernel (one
// block per kv head, sequence and layer) and the verify kernel's fused commit
// (the block that finishes a sequence's acceptance search commits it for
// every kv head and layer).
//
// "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on Ascend NPUs",
// technical summary 2.1: path-index commit reorders the cache along the
// accepted path, and the prefix-sharing fast reorder moves only the newly
// accepted segment, only when needed.  Slot P + k of the committed sequence
// receives the entry of tree node path[k] - 1 (slot T + path[k] - 1, T the
// tree's base, by default P); entries already in place are not touched.
#pragma once

#include "tsd_common.cuh"

namespace tsd {

constexpr int kMaxMoves = kMaxDepth + 1;  // k = 0..A, A <= D_max <= 32 (k = 0 moves
                                          // only when the tree has its own base)

// The cache and its bookkeeping, as tsd_kv_commit_path takes them (device
// pointers; tail_base, moved and status may be null).
struct CommitArgs {
  uint16_t *k, *v;
  int num_layers;
  int64_t layer_stride;  // elements between layers' pools
  const int32_t *table;
  int max_blocks, num_blocks;
  const int32_t *prefix_len, *tail_base;
  int Hkv;
  int32_t *new_len, *moved, *status;
};

// Sequence b's moves: entry m goes from slot (src_page, src_slot) to slot
// (dst_page, dst_slot), the same slots in every kv head and layer.
struct CommitMoves {
  int n;
  int src_page[kMaxMoves], src_slot[kMaxMoves], dst_page[kMaxMoves], dst_slot[kMaxMoves];
};

// Plans sequence b's commit in one warp (lane l covers path entry k = l + 1):
// validation, then the block ids of every move, every load of a round
// independent, so the plan costs three dependent rounds (lengths and path,
// block ids, then the copy).  The error reported is the first failing
// entry's, in k order, as a sequential walk would find it.  Writes mv (lane
// 0 the counts), new_len / moved when `report`, and status bits.
__device__ __forceinline__ void commit_plan_warp(const CommitArgs &a, int b, int N_max, int D_max,
                                                 const int32_t *n_nodes, const int32_t *err,
                                                 const int32_t *accept_len, const int32_t *path,
                                                 bool report, CommitMoves &mv, int lane) {
  const int cols = D_max + 1;
  const int P = a.prefix_len[b];
  const int T = a.tail_base ? a.tail_base[b] : P;  // slot of the tree's node 0
  const int nb = n_nodes ? n_nodes[b] : N_max;
  const int eb = err ? err[b] : 0;
  const int A = accept_len[b];
  const int p0 = path[(size_t)b * cols];
  const int k = lane + 1;
  const int pk = k <= D_max ? path[(size_t)b * cols + k] : 0;
  const int32_t *trow = a.table + (size_t)b * a.max_blocks;
  int ok = 1, bad = 0;
  if (eb != 0) {
    ok = 0;
  } else if (P < 0 || T < 0 || nb < 1 || nb > N_max || (long)P + nb > (long)a.max_blocks * kPage ||
             (long)T + nb > (long)a.max_blocks * kPage) {
    ok = 0;
    bad = TSD_STATUS_BAD_LEN;
  } else if (A < 0 || A > D_max || A > nb - 1 || p0 != 1) {
    ok = 0;
    bad = TSD_STATUS_BAD_PATH;
  }
  // per entry (the branches above are uniform: ok is the same in every lane)
  const bool mine = ok && k <= A;
  const int node = pk - 1;
  const bool bad_path = mine && (node < 0 || node >= nb);
  const bool move = mine && !bad_path && T + node != P + k;
  int ps = 0, pd = 0;
  if (move) {
    ps = trow[(T + node) / kPage];
    pd = trow[(P + k) / kPage];
  }
  const bool bad_page = move && (ps < 0 || ps >= a.num_blocks || pd < 0 || pd >= a.num_blocks);
  const unsigned fails = __ballot_sync(0xffffffffu, bad_path || bad_page);
  if (ok && fails) {
    const int first = __ffs(fails) - 1;  // the lowest failing k
    const int kind = __shfl_sync(0xffffffffu, bad_path ? 1 : 2, first);
    ok = 0;
    bad = kind == 1 ? TSD_STATUS_BAD_PATH : TSD_STATUS_BAD_PAGE;
  }
  const unsigned moves = __ballot_sync(0xffffffffu, move);
  int n = ok ? __popc(moves) : 0;
  if (ok && move) {
    const int m = __popc(moves & ((1u << lane) - 1u));
    mv.src_page[m] = ps;
    mv.src_slot[m] = (T + node) % kPage;
    mv.dst_page[m] = pd;
    mv.dst_slot[m] = (P + k) % kPage;
  }
  // the root (k = 0, node 0) moves only when the tree has its own base
  if (ok && T != P) {
    const int rs = trow[T / kPage];
    const int rd = trow[P / kPage];
    if (rs < 0 || rs >= a.num_blocks || rd < 0 || rd >= a.num_blocks) {
      ok = 0;
      bad = TSD_STATUS_BAD_PAGE;
      n = 0;
    } else {
      if (lane == 0) {
        mv.src_page[n] = rs;
        mv.src_slot[n] = T % kPage;
        mv.dst_page[n] = rd;
        mv.dst_slot[n] = P % kPage;
      }
      ++n;
    }
  }
  if (lane == 0) {
    mv.n = n;
    if (bad && a.status) atomicOr(a.status, bad);
    if (report) {
      a.new_len[b] = ok ? P + A + 1 : P;
      if (a.moved) a.moved[b] = n;
    }
  }
}

// Performs the planned moves for kv heads [h0, h0 + nh) of layers [l0, l0 +
// nl) with the block's nthreads threads: every source of a group of whole kv
// heads (K and V, 16-byte vectors) is staged in `stage` (room for `cap`
// entries: cap * D / 8 vectors of K, then as many of V) before any of the
// group's destinations is written, because a destination slot can be the
// source of a later path element of the same head; different heads and
// layers never share a slot.  Called by every thread of the block.
template <int D>
__device__ __forceinline__ void commit_copy(const CommitArgs &a, const CommitMoves &mv, int h0,
                                            int nh, int l0, int nl, uint4 *stage, int cap, int t,
                                            int nthreads) {
  constexpr int kVec = D / 8;  // 16-byte vectors per entry
  const int n = mv.n;
  if (n == 0) return;
  const int per = max(1, cap / n);  // whole heads per group
  uint4 *sk = stage, *sv = stage + (size_t)cap * kVec;
  for (int l = l0; l < l0 + nl; ++l) {
    const size_t base = (size_t)l * (size_t)a.layer_stride;
    const uint4 *kin = reinterpret_cast<const uint4 *>(a.k + base);
    const uint4 *vin = reinterpret_cast<const uint4 *>(a.v + base);
    uint4 *kout = reinterpret_cast<uint4 *>(a.k + base);
    uint4 *vout = reinterpret_cast<uint4 *>(a.v + base);
    for (int hs = h0; hs < h0 + nh; hs += per) {
      const int hc = min(per, h0 + nh - hs);
      const int items = hc * n * kVec;
      for (int x = t; x < items; x += nthreads) {
        const int e = x % kVec, m = (x / kVec) % n, h = hs + x / (n * kVec);
        const size_t src = ((size_t)mv.src_page[m] * a.Hkv + h) * kPage + mv.src_slot[m];
        sk[x] = kin[src * kVec + e];
        sv[x] = vin[src * kVec + e];
      }
      __syncthreads();
      for (int x = t; x < items; x += nthreads) {
        const int e = x % kVec, m = (x / kVec) % n, h = hs + x / (n * kVec);
        const size_t dst = ((size_t)mv.dst_page[m] * a.Hkv + h) * kPage + mv.dst_slot[m];
        kout[dst * kVec + e] = sk[x];
        vout[dst * kVec + e] = sv[x];
      }
      __syncthreads();
    }
  }
}

}  // namespace tsd
