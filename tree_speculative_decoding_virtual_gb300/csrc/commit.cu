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

#include "commit_core.cuh"
#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kThreads = 128;

// One block per (kv head, sequence, layer): warp 0 plans the sequence's
// moves, then the block stages the head's out-of-place sources and writes
// their destinations (commit_core.cuh).
template <int D>
__global__ void __launch_bounds__(kThreads)
commit_kernel(const CommitArgs a, const int32_t *__restrict__ n_nodes,
              const int32_t *__restrict__ accept_len, const int32_t *__restrict__ path,
              const int32_t *__restrict__ err, int N_max, int D_max) {
  __shared__ CommitMoves mv;
  __shared__ uint4 stage[2 * kMaxMoves * (D / 8)];
  // No early release of the next kernel: it may be an attention pass, which
  // reads the cache before it waits for this grid.
  pdl_wait();
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int layer = blockIdx.z;
  if (threadIdx.x < 32)
    commit_plan_warp(a, b, N_max, D_max, n_nodes, err, accept_len, path, h == 0 && layer == 0, mv,
                     threadIdx.x);
  __syncthreads();
  commit_copy<D>(a, mv, h, 1, layer, 1, stage, kMaxMoves, threadIdx.x, kThreads);
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
  const CommitArgs a{k_cache, v_cache, num_layers, layer_stride, block_table, max_blocks, num_blocks,
                     prefix_len, tail_base, Hkv, new_len, moved, status};
  const cudaError_t e =
      D == 128 ? launch(commit_kernel<128>, grid, dim3(kThreads), 0, as_cuda(stream), a, n_nodes,
                        accept_len, path, err, N_max, D_max)
               : launch(commit_kernel<64>, grid, dim3(kThreads), 0, as_cuda(stream), a, n_nodes,
                        accept_len, path, err, N_max, D_max);
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
