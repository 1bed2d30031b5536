// a1: accelerator-safe tree tensors.
//
// "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on Ascend NPUs",
// technical summary 2.2: the root's -1 sentinel is replaced by a virtual root
// row 0 so that every device gather index lies in [0, M]; an ancestor index
// table is precomputed; range, acyclicity and validity-closure checks run
// before the fused kernels.
//
// One thread block per sequence, one thread per node, two barriers: the
// parent array is staged in shared memory; then each node checks its own
// parent (root, range, closure) and walks up to the root (at most N_b
// steps, which also detects cycles), writing its ancestor row and bitmask
// row into shared memory as it goes; then the rows are written out with
// coalesced stores (all zero when the sequence is flagged).

#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
ancestors_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ n_nodes,
                 int N_max, int D_max, int W, int32_t *__restrict__ anc,
                 int32_t *__restrict__ depth_out, uint32_t *__restrict__ mask,
                 int32_t *__restrict__ err) {
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_depth[kMaxNodes];
  __shared__ uint32_t s_mask[kMaxNodes * (kMaxNodes / 32)];
  __shared__ int s_serr, s_werr;
  extern __shared__ int s_anc[];  // [(N_max + 1) * (D_max + 1)]

  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  const int cols = D_max + 1;
  const int nb = n_nodes ? n_nodes[b] : N_max;
  const bool count_ok = nb >= 1 && nb <= N_max;

  if (t == 0) {
    s_serr = count_ok ? 0 : TSD_TREE_COUNT;
    s_werr = 0;
  }
  for (int i = t; i < N_max; i += kThreads) s_par[i] = parent[(size_t)b * N_max + i];
  for (int x = t; x < (N_max + 1) * cols; x += kThreads) s_anc[x] = 0;
  for (int x = t; x < N_max * W; x += kThreads) s_mask[x] = 0u;
  __syncthreads();

  if (count_ok) {
    int se = 0, we = 0;
    for (int i = t; i < nb; i += kThreads) {
      // structural checks of this node's own parent: root sentinel, range, closure
      const int p = s_par[i];
      if (i == 0) {
        if (p != -1) se |= TSD_TREE_ROOT;
      } else if (p < 0 || p >= N_max) {
        se |= TSD_TREE_RANGE;
      } else if (p >= nb) {
        se |= TSD_TREE_CLOSURE;
      }
      // walk to the root: depth, cycle and depth checks (a parent outside
      // [0, nb) on the way is some node's structural error; stop there)
      int j = i, steps = 0;
      bool cycle = false, broken = false;
      while (s_par[j] != -1) {
        if (steps == nb) {
          cycle = true;
          break;
        }
        const int pj = s_par[j];
        if (pj < 0 || pj >= nb) {
          broken = true;
          break;
        }
        j = pj;
        ++steps;
      }
      if (cycle)
        we |= TSD_TREE_CYCLE;
      else if (!broken && steps > D_max)
        we |= TSD_TREE_TOO_DEEP;
      s_depth[i] = steps;
      if (!cycle && !broken && steps <= D_max) {
        // ancestor row in safe ids (column d = the depth-d ancestor) and bitmask
        int a = i;
        for (int d = steps; d >= 0; --d) {
          s_anc[(i + 1) * cols + d] = a + 1;
          s_mask[i * W + (a >> 5)] |= 1u << (a & 31);
          a = s_par[a];
        }
      }
    }
    if (se) atomicOr(&s_serr, se);
    if (we) atomicOr(&s_werr, we);
  }
  __syncthreads();
  // range, closure and root errors are reported alone; cycle and depth
  // errors only when those are clear
  const int eb = s_serr ? s_serr : s_werr;

  int32_t *anc_b = anc + (size_t)b * (N_max + 1) * cols;
  for (int x = t; x < (N_max + 1) * cols; x += kThreads) anc_b[x] = eb ? 0 : s_anc[x];
  for (int i = t; i < N_max; i += kThreads)
    depth_out[(size_t)b * N_max + i] = (eb == 0 && i < nb) ? s_depth[i] : 0;
  uint32_t *mask_b = mask + (size_t)b * N_max * W;
  for (int x = t; x < N_max * W; x += kThreads) mask_b[x] = (eb == 0 && x < nb * W) ? s_mask[x] : 0u;
  if (t == 0) err[b] = eb;
}

}  // namespace

}  // namespace tsd

TSD_API int tsd_tree_build_ancestors(const int32_t *parent, const int32_t *n_nodes, int B,
                                     int N_max, int D_max, int32_t *anc, int32_t *depth,
                                     uint32_t *mask, int32_t *err, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0 || N_max < 1 || D_max < 0) return B < 0 ? TSD_ERR_ARG : TSD_ERR_LIMIT;
  if (N_max > kMaxNodes || D_max > kMaxDepth || B > 65535) return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!parent || !anc || !depth || !mask || !err) return TSD_ERR_ARG;
  const int W = (N_max + 31) / 32;
  const size_t smem = sizeof(int) * (size_t)(N_max + 1) * (D_max + 1);
  if (launch(ancestors_kernel, dim3(B), dim3(kThreads), smem, as_cuda(stream), parent, n_nodes,
             N_max, D_max, W, anc, depth, mask, err) != cudaSuccess)
    return TSD_ERR_CUDA;
  return TSD_OK;
}
