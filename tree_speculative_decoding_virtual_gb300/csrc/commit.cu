// a4: commit of the accepted path's K/V with the prefix-sharing fast reorder.
//
// "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on Ascend NPUs",
// technical summary 2.1: path-index commit reorders the cache along the
// accepted path, and the prefix-sharing fast reorder moves only the newly
// accepted segment, only when needed (length-based commit is the special
// case where every accepted entry is already in place).
//
// One thread block per (kv head, sequence, layer).  The block stages every
// out-of-place source entry (K and V, 16-byte vectors) in shared memory
// before it writes any destination, because a destination slot can be the
// source of a later path element.  Entries already in place are not touched.
// The tree may sit at its own base (tail_base[b]; by default right after the
// prefix), which is how a deferred commit's record is materialised.
//
// Deferred commit (tsd_kv_commit_remap): the same validation, but instead of
// moving anything it records the physical slot of each committed entry; the
// next step's attention reads the committed sequence through that record.

#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxMoves = kMaxDepth + 1;  // k = 0..A, A <= D_max <= 32 (k = 0 moves
                                          // only when the tree has its own base)

// Block id of slot page `i` of sequence b.
__device__ __forceinline__ int trow_entry(const int32_t *block_table, int b, int max_blocks, int i) {
  return block_table[(size_t)b * max_blocks + i];
}

template <int D>
__global__ void __launch_bounds__(kThreads)
commit_kernel(uint16_t *__restrict__ k_cache, uint16_t *__restrict__ v_cache,
              int64_t layer_stride, const int32_t *__restrict__ block_table, int max_blocks,
              int num_blocks, const int32_t *__restrict__ prefix_len,
              const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ accept_len,
              const int32_t *__restrict__ path, const int32_t *__restrict__ err,
              const int32_t *__restrict__ tail_base, int N_max, int Hkv, int D_max,
              int32_t *__restrict__ new_len, int32_t *__restrict__ moved,
              int32_t *__restrict__ status) {
  constexpr int kVec = D / 8;  // 16-byte vectors per entry
  __shared__ uint4 s_k[kMaxMoves][kVec];
  __shared__ uint4 s_v[kMaxMoves][kVec];
  __shared__ long long s_src[kMaxMoves];  // entry index within one layer's pool
  __shared__ long long s_dst[kMaxMoves];
  __shared__ int s_n;

  // No early release of the next kernel: it may be an attention pass, which
  // reads the cache before it waits for this grid.
  pdl_wait();
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int layer = blockIdx.z;
  const int t = threadIdx.x;
  const int cols = D_max + 1;

  // Planning by warp 0, one lane per path entry k = lane + 1 (k <= A <= D_max
  // <= 32): every load of a round is independent, so the plan costs three
  // dependent rounds (lengths and path, block ids, then the copy) rather than
  // two per entry.  The error reported is the first failing entry's, in k
  // order, as a sequential walk would find it.
  if (t < 32) {
    const int lane = t;
    const int P = prefix_len[b];
    const int T = tail_base ? tail_base[b] : P;  // slot of the tree's node 0
    const int nb = n_nodes ? n_nodes[b] : N_max;
    const int eb = err ? err[b] : 0;
    const int A = accept_len[b];
    const int p0 = path[(size_t)b * cols];
    const int k = lane + 1;
    const int pk = k <= D_max ? path[(size_t)b * cols + k] : 0;
    int ok = 1, bad = 0;
    if (eb != 0) {
      ok = 0;
    } else if (P < 0 || T < 0 || nb < 1 || nb > N_max || (long)P + nb > (long)max_blocks * kPage ||
               (long)T + nb > (long)max_blocks * kPage) {
      ok = 0;
      bad = TSD_STATUS_BAD_LEN;
    } else if (A < 0 || A > D_max || A > nb - 1 || p0 != 1) {
      ok = 0;
      bad = TSD_STATUS_BAD_PATH;
    }
    // per entry (uniform branch above: ok is the same in every lane)
    const bool mine = ok && k <= A;
    const int node = pk - 1;
    const bool bad_path = mine && (node < 0 || node >= nb);
    const bool move = mine && !bad_path && T + node != P + k;
    int ps = 0, pd = 0;
    if (move) {
      ps = trow_entry(block_table, b, max_blocks, (T + node) / kPage);
      pd = trow_entry(block_table, b, max_blocks, (P + k) / kPage);
    }
    const bool bad_page = move && (ps < 0 || ps >= num_blocks || pd < 0 || pd >= num_blocks);
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
      const int slot = __popc(moves & ((1u << lane) - 1u));
      const int src = T + node, dst = P + k;
      s_src[slot] = ((long long)ps * Hkv + h) * kPage + src % kPage;
      s_dst[slot] = ((long long)pd * Hkv + h) * kPage + dst % kPage;
    }
    // the root (k = 0, node 0) moves only when the tree has its own base
    if (ok && T != P) {
      const int rs = trow_entry(block_table, b, max_blocks, T / kPage);
      const int rd = trow_entry(block_table, b, max_blocks, P / kPage);
      if (rs < 0 || rs >= num_blocks || rd < 0 || rd >= num_blocks) {
        ok = 0;
        bad = TSD_STATUS_BAD_PAGE;
        n = 0;
      } else {
        if (lane == 0) {
          s_src[n] = ((long long)rs * Hkv + h) * kPage + T % kPage;
          s_dst[n] = ((long long)rd * Hkv + h) * kPage + P % kPage;
        }
        ++n;
      }
    }
    if (lane == 0) {
      s_n = n;
      if (bad && status) atomicOr(status, bad);
      if (h == 0 && layer == 0) {
        new_len[b] = ok ? P + A + 1 : P;
        if (moved) moved[b] = n;
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  if (n == 0) return;

  const size_t base = (size_t)layer * (size_t)layer_stride;
  const uint4 *kin = reinterpret_cast<const uint4 *>(k_cache + base);
  const uint4 *vin = reinterpret_cast<const uint4 *>(v_cache + base);
  for (int x = t; x < n * kVec; x += kThreads) {
    const int m = x / kVec, e = x % kVec;
    s_k[m][e] = kin[(size_t)s_src[m] * kVec + e];
    s_v[m][e] = vin[(size_t)s_src[m] * kVec + e];
  }
  __syncthreads();
  uint4 *kout = reinterpret_cast<uint4 *>(k_cache + base);
  uint4 *vout = reinterpret_cast<uint4 *>(v_cache + base);
  for (int x = t; x < n * kVec; x += kThreads) {
    const int m = x / kVec, e = x % kVec;
    kout[(size_t)s_dst[m] * kVec + e] = s_k[m][e];
    vout[(size_t)s_dst[m] * kVec + e] = s_v[m][e];
  }
}

}  // namespace
}  // namespace tsd

static int commit_launch(uint16_t *k_cache, uint16_t *v_cache, int num_layers, int64_t layer_stride,
                         const int32_t *block_table, int max_blocks, int num_blocks,
                         const int32_t *prefix_len, const int32_t *n_nodes,
                         const int32_t *accept_len, const int32_t *path, const int32_t *err,
                         const int32_t *tail_base, int B, int N_max, int Hkv, int D, int D_max,
                         int32_t *new_len, int32_t *moved, int32_t *status, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0 || num_layers < 0 || Hkv < 1 || max_blocks < 1 || num_blocks < 1) return TSD_ERR_ARG;
  if (D != 64 && D != 128) return TSD_ERR_LIMIT;
  if (N_max < 1 || N_max > kMaxNodes || D_max < 0 || D_max > kMaxDepth || B > 65535 ||
      Hkv > 65535 || num_layers > 65535)
    return TSD_ERR_LIMIT;
  if (B == 0 || num_layers == 0) return TSD_OK;
  if (!k_cache || !v_cache || !block_table || !prefix_len || !accept_len || !path || !new_len)
    return TSD_ERR_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return TSD_ERR_ARG;
  const int64_t pool = (int64_t)num_blocks * Hkv * kPage * D;
  if (num_layers > 1 && (layer_stride < pool || layer_stride % 8 != 0)) return TSD_ERR_ARG;
  dim3 grid(Hkv, B, num_layers);
  const cudaError_t e =
      D == 128 ? launch(commit_kernel<128>, grid, dim3(kThreads), 0, as_cuda(stream), k_cache,
                        v_cache, layer_stride, block_table, max_blocks, num_blocks, prefix_len,
                        n_nodes, accept_len, path, err, tail_base, N_max, Hkv, D_max, new_len,
                        moved, status)
               : launch(commit_kernel<64>, grid, dim3(kThreads), 0, as_cuda(stream), k_cache,
                        v_cache, layer_stride, block_table, max_blocks, num_blocks, prefix_len,
                        n_nodes, accept_len, path, err, tail_base, N_max, Hkv, D_max, new_len,
                        moved, status);
  return e == cudaSuccess ? TSD_OK : TSD_ERR_CUDA;
}

TSD_API int tsd_kv_commit_path(uint16_t *k_cache, uint16_t *v_cache, int num_layers,
                               int64_t layer_stride, const int32_t *block_table, int max_blocks,
                               int num_blocks, const int32_t *prefix_len, const int32_t *n_nodes,
                               const int32_t *accept_len, const int32_t *path, const int32_t *err,
                               int B, int N_max, int Hkv, int D, int D_max, int32_t *new_len,
                               int32_t *moved,
                               int32_t *status, tsd_stream_t stream) {
  return commit_launch(k_cache, v_cache, num_layers, layer_stride, block_table, max_blocks,
                       num_blocks, prefix_len, n_nodes, accept_len, path, err, nullptr, B, N_max,
                       Hkv, D, D_max, new_len, moved, status, stream);
}

TSD_API int tsd_kv_commit_path_from(uint16_t *k_cache, uint16_t *v_cache, int num_layers,
                                    int64_t layer_stride, const int32_t *block_table,
                                    int max_blocks, int num_blocks, const int32_t *prefix_len,
                                    const int32_t *n_nodes, const int32_t *accept_len,
                                    const int32_t *path, const int32_t *err,
                                    const int32_t *tail_base, int B, int N_max, int Hkv, int D,
                                    int D_max, int32_t *new_len, int32_t *moved, int32_t *status,
                                    tsd_stream_t stream) {
  if (!tail_base && B > 0) return TSD_ERR_ARG;
  return commit_launch(k_cache, v_cache, num_layers, layer_stride, block_table, max_blocks,
                       num_blocks, prefix_len, n_nodes, accept_len, path, err, tail_base, B, N_max,
                       Hkv, D, D_max, new_len, moved, status, stream);
}

namespace tsd {
namespace {

// Deferred commit: one warp per sequence; lane l takes path entries k = l and
// k = l + 32.  Validation as in commit_kernel (lengths, root, accepted length,
// node ids); a sequence that fails records nothing.
__global__ void __launch_bounds__(32)
commit_remap_kernel(const int32_t *__restrict__ prefix_len, const int32_t *__restrict__ n_nodes,
                    const int32_t *__restrict__ accept_len, const int32_t *__restrict__ path,
                    const int32_t *__restrict__ err, const int32_t *__restrict__ tail_base, int N_max,
                    int D_max, int32_t *__restrict__ remap_src, int32_t *__restrict__ remap_base,
                    int32_t *__restrict__ remap_len, int32_t *__restrict__ new_len,
                    int32_t *__restrict__ next_tail, int32_t *__restrict__ status) {
  // No early release of the next kernel: it may be an attention pass, which
  // reads the record before it waits for this grid.
  pdl_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  const int cols = D_max + 1;
  const int P = prefix_len[b];
  const int T = tail_base ? tail_base[b] : P;
  const int nb = n_nodes ? n_nodes[b] : N_max;
  const int eb = err ? err[b] : 0;
  const int A = accept_len[b];
  int ok = eb == 0, bad = 0;
  if (ok && (P < 0 || T < 0 || nb < 1 || nb > N_max)) {
    ok = 0;
    bad = TSD_STATUS_BAD_LEN;
  } else if (ok && (A < 0 || A > D_max || A > nb - 1 || path[(size_t)b * cols] != 1)) {
    ok = 0;
    bad = TSD_STATUS_BAD_PATH;
  }
  int node[2] = {0, 0};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int k = lane + 32 * r;
    if (ok && k <= A) node[r] = path[(size_t)b * cols + k] - 1;
  }
  const bool bad_node = ok && ((lane <= A && (node[0] < 0 || node[0] >= nb)) ||
                               (lane + 32 <= A && (node[1] < 0 || node[1] >= nb)));
  if (__any_sync(0xffffffffu, bad_node)) {
    ok = 0;
    bad = TSD_STATUS_BAD_PATH;
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int k = lane + 32 * r;
    if (k < cols) remap_src[(size_t)b * cols + k] = ok && k <= A ? T + node[r] : -1;
  }
  if (lane == 0) {
    remap_base[b] = P;
    remap_len[b] = ok ? A + 1 : 0;
    new_len[b] = ok ? P + A + 1 : P;
    next_tail[b] = ok ? T + nb : T;
    if (bad && status) atomicOr(status, bad);
  }
}

}  // namespace
}  // namespace tsd

TSD_API int tsd_kv_commit_remap(const int32_t *prefix_len, const int32_t *n_nodes,
                                const int32_t *accept_len, const int32_t *path,
                                const int32_t *err, const int32_t *tail_base, int B, int N_max,
                                int D_max, int32_t *remap_src, int32_t *remap_base,
                                int32_t *remap_len, int32_t *new_len, int32_t *next_tail,
                                int32_t *status, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0) return TSD_ERR_ARG;
  if (N_max < 1 || N_max > kMaxNodes || D_max < 0 || D_max > kMaxDepth || B > 65535)
    return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!prefix_len || !accept_len || !path || !remap_src || !remap_base || !remap_len || !new_len ||
      !next_tail)
    return TSD_ERR_ARG;
  return launch(commit_remap_kernel, dim3(B), dim3(32), 0, as_cuda(stream), prefix_len, n_nodes,
                accept_len, path, err, tail_base, N_max, D_max, remap_src, remap_base, remap_len,
                new_len, next_tail, status) == cudaSuccess
             ? TSD_OK
             : TSD_ERR_CUDA;
}
