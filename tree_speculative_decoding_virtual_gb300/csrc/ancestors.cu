// a1: accelerator-safe tree tensors.
//
// "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on Ascend NPUs",
// technical summary 2.2: the root's -1 sentinel is replaced by a virtual root
// row 0 so that every device gather index lies in [0, M]; an ancestor index
// table is precomputed; range, acyclicity and validity-closure checks run
// before the fused kernels.
//
// One thread block per sequence, one thread per node.  The parent array is
// staged in shared memory; each node walks up to the root (at most N_b
// steps, which also detects cycles), and the ancestor rows are assembled in
// shared memory and written out with coalesced stores.

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
  __shared__ int s_err;
  extern __shared__ int s_anc[];  // [(N_max + 1) * (D_max + 1)]

  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  const int cols = D_max + 1;
  const int nb = n_nodes ? n_nodes[b] : N_max;
  const bool count_ok = nb >= 1 && nb <= N_max;

  if (t == 0) s_err = count_ok ? 0 : TSD_TREE_COUNT;
  for (int i = t; i < N_max; i += kThreads) s_par[i] = parent[(size_t)b * N_max + i];
  for (int x = t; x < (N_max + 1) * cols; x += kThreads) s_anc[x] = 0;
  __syncthreads();

  // structural checks: root sentinel, range, closure
  if (count_ok) {
    int e = 0;
    for (int i = t; i < nb; i += kThreads) {
      const int p = s_par[i];
      if (i == 0) {
        if (p != -1) e |= TSD_TREE_ROOT;
      } else if (p < 0 || p >= N_max) {
        e |= TSD_TREE_RANGE;
      } else if (p >= nb) {
        e |= TSD_TREE_CLOSURE;
      }
    }
    if (e) atomicOr(&s_err, e);
  }
  __syncthreads();

  // walk to the root: depth, cycle and depth checks
  if (s_err == 0) {
    int e = 0;
    for (int i = t; i < nb; i += kThreads) {
      int j = i, steps = 0;
      bool cycle = false;
      while (s_par[j] != -1) {
        if (steps == nb) {
          cycle = true;
          break;
        }
        j = s_par[j];
        ++steps;
      }
      s_depth[i] = steps;
      if (cycle)
        e |= TSD_TREE_CYCLE;
      else if (steps > D_max)
        e |= TSD_TREE_TOO_DEEP;
    }
    if (e) atomicOr(&s_err, e);
  }
  __syncthreads();
  const int eb = s_err;

  // ancestor rows in safe ids: row i+1, column d = safe id of the depth-d ancestor
  if (eb == 0) {
    for (int i = t; i < nb; i += kThreads) {
      int j = i;
      for (int d = s_depth[i]; d >= 0; --d) {
        s_anc[(i + 1) * cols + d] = j + 1;
        j = s_par[j];
      }
    }
  }
  __syncthreads();

  int32_t *anc_b = anc + (size_t)b * (N_max + 1) * cols;
  for (int x = t; x < (N_max + 1) * cols; x += kThreads) anc_b[x] = s_anc[x];

  for (int i = t; i < N_max; i += kThreads) {
    const bool valid = eb == 0 && i < nb;
    const int d = valid ? s_depth[i] : 0;
    depth_out[(size_t)b * N_max + i] = d;
    uint32_t *mrow = mask + ((size_t)b * N_max + i) * W;
    for (int w = 0; w < W; ++w) {
      uint32_t bits = 0;
      if (valid) {
        for (int k = 0; k <= d; ++k) {
          const int a = s_anc[(i + 1) * cols + k] - 1;
          if ((a >> 5) == w) bits |= 1u << (a & 31);
        }
      }
      mrow[w] = bits;
    }
  }
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
