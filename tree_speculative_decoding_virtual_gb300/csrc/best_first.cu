// a5: best-first budgeted draft-tree construction.
//
// "Resumo Técnico: BASTION", Methodology 1 and 2: per-position draft
// marginals q_k(.) from one drafter pass; path score
// rho(i) = prod_{k=1}^{d(i)} q_k(x_ik); the surrogate A_hat(T) = sum rho(i) is
// maximised under a node budget by best-first expansion, which repeatedly
// adds the valid node with the largest rho.
//
// Kernel 1 (one block per (position, sequence)): the M = min(N-1, V) best
// tokens of the position, ranked by (q desc, token id asc).  A 4-pass 8-bit
// radix select finds the M-th largest key; the selection is gathered in
// index order (deterministic) and bitonic-sorted in shared memory.
// Kernel 2 (one block per sequence, one warp expanding): every inserted node
// owns exactly one candidate, its best not-yet-inserted child (the next
// rank at the next position); the child ranks of a node are consumed in
// order because q is sorted.  Each step takes the best candidate with two
// warp max-reductions (rho bits, then (depth, parent) as a tie key).

#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kTopThreads = 1024;
constexpr int kMaxPositions = 64;

// Monotone map of a float to uint32 (+0 and -0 map to the same key).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of one unsigned per thread (blockDim.x == kTopThreads).
__device__ unsigned block_excl_scan(unsigned v, unsigned *s_warp, unsigned *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned w = s_warp[lane];
    unsigned z = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, z, off);
      if (lane >= off) z += y;
    }
    s_warp[lane] = z - w;  // exclusive prefix of warp totals
    if (lane == 31) *total = z;
  }
  __syncthreads();
  const unsigned r = s_warp[warp] + x - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kTopThreads)
topk_kernel(const float *__restrict__ q, int K, int V, int M, int32_t *__restrict__ top_tok,
            float *__restrict__ top_q) {
  __shared__ unsigned hist[256];
  __shared__ unsigned s_prefix, s_remaining, s_total;
  __shared__ unsigned s_warp[32];
  __shared__ unsigned long long s_sel[256];

  pdl_trigger();
  pdl_wait();
  const int k = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const float *row = q + ((size_t)b * K + k) * (size_t)V;

  // radix select: the M-th largest key T and how many keys equal to T to take
  unsigned prefix = 0u, pmask = 0u, remaining = (unsigned)M;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int x = t; x < 256; x += kTopThreads) hist[x] = 0u;
    __syncthreads();
    for (int x = t; x < V; x += kTopThreads) {
      const uint32_t key = order_key(__ldg(row + x));
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (t < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      unsigned c[8], s = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * t - j];
        s += c[j];
      }
      unsigned incl = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
        if (t >= off) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
      const int L = __ffs(hit) - 1;
      if (t == L) {
        unsigned cum = incl - s;
        int j = 0;
        for (; j < 7; ++j) {
          if (cum + c[j] >= remaining) break;
          cum += c[j];
        }
        s_prefix = prefix | ((unsigned)(255 - 8 * t - j) << shift);
        s_remaining = remaining - cum;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    pmask |= 0xFFu << shift;
  }
  const unsigned T = prefix;
  const unsigned need_eq = remaining;
  const unsigned cnt_gt = (unsigned)M - need_eq;

  // gather in index order: contiguous segment per thread
  const int seg = (V + kTopThreads - 1) / kTopThreads;
  const int lo = min(V, t * seg), hi = min(V, lo + seg);
  unsigned n_gt = 0u, n_eq = 0u;
  for (int x = lo; x < hi; ++x) {
    const uint32_t key = order_key(__ldg(row + x));
    n_gt += key > T;
    n_eq += key == T;
  }
  unsigned pos_gt = block_excl_scan(n_gt, s_warp, &s_total);
  unsigned pos_eq = block_excl_scan(n_eq, s_warp, &s_total);
  for (int x = t; x < 256; x += kTopThreads) s_sel[x] = 0ull;
  __syncthreads();
  for (int x = lo; x < hi; ++x) {
    const uint32_t key = order_key(__ldg(row + x));
    const unsigned long long packed =
        ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)x);
    if (key > T) {
      s_sel[pos_gt++] = packed;
    } else if (key == T) {
      if (pos_eq < need_eq) s_sel[cnt_gt + pos_eq] = packed;
      ++pos_eq;
    }
  }
  __syncthreads();

  // bitonic sort, descending: (key desc, index asc)
  for (int size = 2; size <= 256; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (t < 256) {
        const int l = t ^ stride;
        if (l > t) {
          const unsigned long long a = s_sel[t], c = s_sel[l];
          const bool up = (t & size) == 0;
          if (up ? (a < c) : (a > c)) {
            s_sel[t] = c;
            s_sel[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int r = t; r < M; r += kTopThreads) {
    const int idx = (int)(0xFFFFFFFFu - (unsigned)(s_sel[r] & 0xFFFFFFFFull));
    top_tok[((size_t)b * K + k) * M + r] = idx;
    top_q[((size_t)b * K + k) * M + r] = __ldg(row + idx);
  }
}

constexpr int kExpandThreads = 256;
constexpr int kPerLane = kMaxNodes / 32;  // nodes owned by one lane

__global__ void __launch_bounds__(kExpandThreads)
expand_kernel(const int32_t *__restrict__ top_tok, const float *__restrict__ top_q,
              const int32_t *__restrict__ root_token, int K, int M, int N,
              int32_t *__restrict__ parent, int32_t *__restrict__ tokens,
              int32_t *__restrict__ depth, float *__restrict__ rho, double *__restrict__ ahat) {
  extern __shared__ unsigned char smem_raw[];
  float *s_tq = reinterpret_cast<float *>(smem_raw);            // [K][M]
  int32_t *s_tt = reinterpret_cast<int32_t *>(s_tq + (size_t)K * M);  // [K][M]
  __shared__ float s_rho[kMaxNodes];

  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, t = threadIdx.x;
  for (int x = t; x < K * M; x += kExpandThreads) {
    s_tq[x] = top_q[(size_t)b * K * M + x];
    s_tt[x] = top_tok[(size_t)b * K * M + x];
  }
  __syncthreads();
  if (t >= 32) return;
  const int lane = t;
  int32_t *par_b = parent + (size_t)b * N;
  int32_t *tok_b = tokens + (size_t)b * N;
  int32_t *dep_b = depth + (size_t)b * N;
  float *rho_b = rho + (size_t)b * N;

  float o_rho[kPerLane];
  int o_dep[kPerLane], o_nch[kPerLane];
  unsigned c_hi[kPerLane], c_lo[kPerLane];
#pragma unroll
  for (int j = 0; j < kPerLane; ++j) {
    o_rho[j] = 0.f;
    o_dep[j] = 0;
    o_nch[j] = 0;
    c_hi[j] = 0u;
    c_lo[j] = 0u;
  }

  // candidate of owned slot j (node id = lane + 32 j): its best remaining child
  auto refresh = [&](int j) {
    const int node = lane + 32 * j;
    const int d = o_dep[j] + 1;
    const int r = o_nch[j];
    if (node >= N || d > K || r >= M) {
      c_hi[j] = 0u;
      c_lo[j] = 0u;
      return;
    }
    const float rc = __fmul_rn(o_rho[j], s_tq[(d - 1) * M + r]);
    c_hi[j] = __float_as_uint(rc);
    c_lo[j] = ((unsigned)(255 - d) << 16) | (unsigned)(0xFFFF - node);
  };

  if (lane == 0) {
    o_rho[0] = 1.f;
    o_dep[0] = 0;
    o_nch[0] = 0;
    refresh(0);
    par_b[0] = -1;
    tok_b[0] = root_token[b];
    dep_b[0] = 0;
    rho_b[0] = 1.f;
    s_rho[0] = 1.f;
  }

  int filled = N;
  for (int n = 1; n < N; ++n) {
    unsigned bh = 0u, bl = 0u;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j)
      if (c_hi[j] > bh || (c_hi[j] == bh && c_lo[j] > bl)) {
        bh = c_hi[j];
        bl = c_lo[j];
      }
    const unsigned H = __reduce_max_sync(0xffffffffu, bh);
    const unsigned Lo = __reduce_max_sync(0xffffffffu, bh == H ? bl : 0u);
    if (H == 0u && Lo == 0u) {  // no valid node left (host checks make this unreachable)
      filled = n;
      break;
    }
    const int p = 0xFFFF - (int)(Lo & 0xFFFFu);
    const int d = 255 - (int)((Lo >> 16) & 0xFFu);
    const float rn = __uint_as_float(H);
    int tok = 0;
    if (lane == (p & 31)) {
      const int jp = p >> 5;
#pragma unroll
      for (int j = 0; j < kPerLane; ++j)
        if (j == jp) {
          tok = s_tt[(d - 1) * M + o_nch[j]];
          o_nch[j] += 1;
          refresh(j);
        }
    }
    tok = __shfl_sync(0xffffffffu, tok, p & 31);
    if (lane == (n & 31)) {
      const int jn = n >> 5;
#pragma unroll
      for (int j = 0; j < kPerLane; ++j)
        if (j == jn) {
          o_rho[j] = rn;
          o_dep[j] = d;
          o_nch[j] = 0;
          refresh(j);
        }
      par_b[n] = p;
      tok_b[n] = tok;
      dep_b[n] = d;
      rho_b[n] = rn;
      s_rho[n] = rn;
    }
  }
  for (int n = filled + lane; n < N; n += 32) {
    par_b[n] = -1;
    tok_b[n] = -1;
    dep_b[n] = 0;
    rho_b[n] = 0.f;
    s_rho[n] = 0.f;
  }
  __syncwarp();
  if (lane == 0) {
    double s = 0.0;
    for (int n = 1; n < N; ++n) s += (double)s_rho[n];
    ahat[b] = s;
  }
}

struct BestFirstPlan {
  int M;
  size_t tok_bytes, q_bytes;
};

BestFirstPlan plan_best_first(int B, int K, int V, int N) {
  BestFirstPlan p;
  p.M = N - 1 < V ? N - 1 : V;
  p.tok_bytes = align_up(sizeof(int32_t) * (size_t)B * K * (p.M > 0 ? p.M : 1), 256);
  p.q_bytes = sizeof(float) * (size_t)B * K * (p.M > 0 ? p.M : 1);
  return p;
}

// number of distinct non-root nodes available: sum_{d=1..K} V^d, saturated
long long valid_nodes(int K, int V) {
  long long total = 0, level = 1;
  for (int d = 1; d <= K; ++d) {
    level = level > (1LL << 40) / V ? (1LL << 40) : level * V;
    total += level;
    if (total > (1LL << 40)) return 1LL << 40;
  }
  return total;
}

}  // namespace
}  // namespace tsd

TSD_API size_t tsd_best_first_workspace_bytes(int B, int K, int V, int N) {
  if (B <= 0 || K <= 0 || V <= 0 || N <= 0) return 0;
  const tsd::BestFirstPlan p = tsd::plan_best_first(B, K, V, N);
  return p.tok_bytes + p.q_bytes;
}

TSD_API int tsd_best_first_tree_build(const float *q, const int32_t *root_token, int B, int K,
                                      int V, int N, int32_t *parent, int32_t *tokens,
                                      int32_t *depth, float *rho, double *ahat, void *workspace,
                                      size_t ws_bytes, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0) return TSD_ERR_ARG;
  if (K < 1 || K > kMaxPositions || V < 1 || N < 1 || N > kMaxNodes || B > 65535)
    return TSD_ERR_LIMIT;
  if ((long long)N - 1 > valid_nodes(K, V)) return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!q || !root_token || !parent || !tokens || !depth || !rho || !ahat) return TSD_ERR_ARG;
  const BestFirstPlan p = plan_best_first(B, K, V, N);
  if (!workspace || ws_bytes < p.tok_bytes + p.q_bytes || !aligned(workspace, 16))
    return TSD_ERR_WORKSPACE;
  int32_t *top_tok = static_cast<int32_t *>(workspace);
  float *top_q = reinterpret_cast<float *>(static_cast<char *>(workspace) + p.tok_bytes);
  cudaStream_t s = as_cuda(stream);
  if (p.M > 0) {
    if (launch(topk_kernel, dim3(K, B), dim3(kTopThreads), 0, s, q, K, V, p.M, top_tok, top_q) !=
        cudaSuccess)
      return TSD_ERR_CUDA;
  }
  const size_t smem = (size_t)K * (p.M > 0 ? p.M : 0) * (sizeof(float) + sizeof(int32_t));
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return TSD_ERR_CUDA;
  }
  if (launch(expand_kernel, dim3(B), dim3(kExpandThreads), smem, s, top_tok, top_q, root_token, K,
             p.M, N, parent, tokens, depth, rho, ahat) != cudaSuccess)
    return TSD_ERR_CUDA;
  return TSD_OK;
}
