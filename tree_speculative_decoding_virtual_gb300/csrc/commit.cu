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

#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxMoves = kMaxDepth;  // k = 1..A, A <= D_max <= 32

template <int D>
__global__ void __launch_bounds__(kThreads)
commit_kernel(uint16_t *__restrict__ k_cache, uint16_t *__restrict__ v_cache,
              int64_t layer_stride, const int32_t *__restrict__ block_table, int max_blocks,
              int num_blocks, const int32_t *__restrict__ prefix_len,
              const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ accept_len,
              const int32_t *__restrict__ path, const int32_t *__restrict__ err, int N_max,
              int Hkv, int D_max, int32_t *__restrict__ new_len, int32_t *__restrict__ moved,
              int32_t *__restrict__ status) {
  constexpr int kVec = D / 8;  // 16-byte vectors per entry
  __shared__ uint4 s_k[kMaxMoves][kVec];
  __shared__ uint4 s_v[kMaxMoves][kVec];
  __shared__ long long s_src[kMaxMoves];  // entry index within one layer's pool
  __shared__ long long s_dst[kMaxMoves];
  __shared__ int s_n;

  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int layer = blockIdx.z;
  const int t = threadIdx.x;
  const int cols = D_max + 1;

  const int P = prefix_len[b];
  const int nb = n_nodes ? n_nodes[b] : N_max;
  const int eb = err ? err[b] : 0;
  const int A = accept_len[b];
  const int32_t *trow = block_table + (size_t)b * max_blocks;

  if (t == 0) {
    int ok = 1, bad = 0, n = 0;
    if (eb != 0) {
      ok = 0;
    } else if (P < 0 || nb < 1 || nb > N_max || (long)P + nb > (long)max_blocks * kPage) {
      ok = 0;
      bad = TSD_STATUS_BAD_LEN;
    } else if (A < 0 || A > D_max || A > nb - 1 || path[(size_t)b * cols] != 1) {
      ok = 0;
      bad = TSD_STATUS_BAD_PATH;
    } else {
      for (int k = 1; k <= A; ++k) {
        const int node = path[(size_t)b * cols + k] - 1;
        if (node < 0 || node >= nb) {
          ok = 0;
          bad = TSD_STATUS_BAD_PATH;
          break;
        }
        if (node != k) {
          const int src = P + node, dst = P + k;
          const int ps = trow[src / kPage], pd = trow[dst / kPage];
          if (ps < 0 || ps >= num_blocks || pd < 0 || pd >= num_blocks) {
            ok = 0;
            bad = TSD_STATUS_BAD_PAGE;
            break;
          }
          s_src[n] = ((long long)ps * Hkv + h) * kPage + src % kPage;
          s_dst[n] = ((long long)pd * Hkv + h) * kPage + dst % kPage;
          ++n;
        }
      }
    }
    if (!ok) n = 0;
    s_n = n;
    if (bad && status) atomicOr(status, bad);
    if (h == 0 && layer == 0) {
      new_len[b] = ok ? P + A + 1 : P;
      if (moved) moved[b] = n;
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

TSD_API int tsd_kv_commit_path(uint16_t *k_cache, uint16_t *v_cache, int num_layers,
                               int64_t layer_stride, const int32_t *block_table, int max_blocks,
                               int num_blocks, const int32_t *prefix_len, const int32_t *n_nodes,
                               const int32_t *accept_len, const int32_t *path, const int32_t *err,
                               int B, int N_max, int Hkv, int D, int D_max, int32_t *new_len,
                               int32_t *moved,
                               int32_t *status, tsd_stream_t stream) {
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
                        n_nodes, accept_len, path, err, N_max, Hkv, D_max, new_len, moved, status)
               : launch(commit_kernel<64>, grid, dim3(kThreads), 0, as_cuda(stream), k_cache,
                        v_cache, layer_stride, block_table, max_blocks, num_blocks, prefix_len,
                        n_nodes, accept_len, path, err, N_max, Hkv, D_max, new_len, moved, status);
  return e == cudaSuccess ? TSD_OK : TSD_ERR_CUDA;
}
