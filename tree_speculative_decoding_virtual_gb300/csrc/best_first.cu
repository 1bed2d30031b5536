// a5: best-first budgeted draft-tree construction.
//
// "Resumo Técnico: BASTION", Methodology 1 and 2: per-position draft
// marginals q_k(.) from one drafter pass; path score
// rho(i) = prod_{k=1}^{d(i)} q_k(x_ik); the surrogate A_hat(T) = sum rho(i) is
// maximised under a node budget by best-first expansion, which repeatedly
// adds the valid node with the largest rho.
//
// Kernel 1 (one block per (position, sequence)): the M = min(N-1, V) best
// tokens of the position, ranked by (q desc, token id asc).  Rows that fit in
// shared memory: the staged threshold filter (topk_stage_kernel: the row
// staged once, a threshold from the warps' sorted thread maxima, a radix
// select over the candidates, warp-run sorts).  Longer rows: the threshold
// filter (topk_filter_kernel: the M-th best of the threads' best keys bounds
// the row's M-th best from below; a second pass keeps the keys above it; a
// bitonic sort ranks them).  Both fall back to a 4-pass 8-bit radix select
// (radix_topk_block: the M-th largest key, a coalesced gather, a bitonic
// sort, ties at the threshold beyond the budget resolved in index order).
// Kernel 2 (one block per sequence, one warp expanding): every inserted node
// owns exactly one candidate, its best not-yet-inserted child (the next
// rank at the next position); the child ranks of a node are consumed in
// order because q is sorted.  Each step takes the best candidate with two
// warp max-reductions (rho bits, then (depth, parent) as a tie key) over
// candidate keys held in shared memory, together with the run of its
// next-ranked siblings that beat every other candidate.

//
// Dynamic draft trees ("Speculative Decoding Hierarquico: Medusa, EAGLE-2 e
// Multi-Token Prediction", EAGLE-2 section: deep where the drafter is
// confident, wide where it is not), built level by level with the path score
// above as node confidence: each frontier node's top-k tokens (a5's top-M kernels on
// its draft row) become its children; one block per sequence scores them,
// writes them to the node pool and keeps the level's k best as the next
// frontier (bitonic sort in shared memory); the rerank kernel keeps the N-1
// best pool nodes, in rank order, with parents re-indexed.

#include "sm100_ptx.cuh"
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

// The ranked top M (<= 256) of one row by radix select, for a block of at
// least 256 threads; writes tok_out[0..M) and q_out[0..M).
__device__ void radix_topk_block(const float *__restrict__ row, int V, int M,
                                 int32_t *__restrict__ tok_out, float *__restrict__ q_out) {
  __shared__ unsigned hist[256];
  __shared__ unsigned s_prefix, s_remaining, s_eq_total;
  __shared__ unsigned s_ngt, s_neq;
  __shared__ unsigned long long s_sel[256];
  const int t = threadIdx.x, nthr = blockDim.x;

  // radix select: the M-th largest key T and how many keys equal to T to take
  unsigned prefix = 0u, pmask = 0u, remaining = (unsigned)M;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int x = t; x < 256; x += nthr) hist[x] = 0u;
    __syncthreads();
    for (int x = t; x < V; x += nthr) {
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
        s_eq_total = c[j];  // after the last pass: the keys equal to T
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    pmask |= 0xFFu << shift;
  }
  const uint32_t T = prefix;
  const unsigned need_eq = remaining;             // keys equal to T to take
  const unsigned cnt_gt = (unsigned)M - need_eq;  // keys greater than T
  // keys equal to T in the whole row (the last pass's bin count)
  const bool all_eq = s_eq_total == need_eq;      // no excess ties at T
  const int lane = t & 31, warp = t >> 5;

  // gather: keys > T (and every key == T when all are taken) land in any
  // order, the sort below orders them
  for (int x = t; x < 256; x += nthr) s_sel[x] = 0ull;
  if (t == 0) {
    s_ngt = 0u;
    s_neq = 0u;
  }
  __syncthreads();
  auto take = [&](uint32_t key, int x) {
    const unsigned long long packed =
        ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)x);
    if (key > T) {
      s_sel[atomicAdd(&s_ngt, 1u)] = packed;
    } else if (key == T && all_eq) {
      s_sel[cnt_gt + atomicAdd(&s_neq, 1u)] = packed;
    }
  };
  for (int x = t; x < V; x += nthr) take(order_key(__ldg(row + x)), x);
  if (!all_eq && warp == 0) {
    // ties at T beyond the budget: the lowest indices win, so warp 0 walks the
    // row in index order, 32 elements at a time
    unsigned taken = 0u;
    for (int x0 = 0; x0 < V && taken < need_eq; x0 += 32) {
      const int x = x0 + lane;
      const bool eq = x < V && order_key(__ldg(row + x)) == T;
      const unsigned bal = __ballot_sync(0xffffffffu, eq);
      const unsigned rank = __popc(bal & ((1u << lane) - 1u));
      if (eq && taken + rank < need_eq)
        s_sel[cnt_gt + taken + rank] =
            ((unsigned long long)T << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)x);
      taken += __popc(bal);
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
  for (int r = t; r < M; r += nthr) {
    const int idx = (int)(0xFFFFFFFFu - (unsigned)(s_sel[r] & 0xFFFFFFFFull));
    tok_out[r] = idx;
    q_out[r] = __ldg(row + idx);
  }
}

__global__ void __launch_bounds__(kTopThreads)
topk_kernel(const float *__restrict__ q, int K, int V, int M, int32_t *__restrict__ top_tok,
            float *__restrict__ top_q) {
  pdl_trigger();
  pdl_wait();
  const int k = blockIdx.x, b = blockIdx.y;
  const size_t o = ((size_t)b * K + k) * M;
  radix_topk_block(q + ((size_t)b * K + k) * (size_t)V, V, M, top_tok + o, top_q + o);
}



constexpr int kExpandThreads = 256;
constexpr int kPerLane = kMaxNodes / 32;  // candidate slots one lane scans

// Candidate key of a node: its best remaining child (rank r at the next
// position), as (rho bits, (255 - child depth) << 16 | (0xFFFF - node)) so
// that a larger key wins under (rho desc, depth asc, parent index asc); 0 when
// the node has no child left.
__device__ __forceinline__ unsigned long long child_key(int node, float rho_node, int dep, int r,
                                                       const float *s_tq, int K, int M, int N) {
  const int d = dep + 1;
  if (node >= N || d > K || r >= M) return 0ull;
  const float rc = __fmul_rn(rho_node, s_tq[(d - 1) * M + r]);
  return ((unsigned long long)__float_as_uint(rc) << 32) |
         (unsigned long long)(((unsigned)(255 - d) << 16) | (unsigned)(0xFFFF - node));
}

__device__ __forceinline__ unsigned long long max_u64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Largest 64-bit key over the warp: two 32-bit max reductions (high word,
// then the low word among the lanes holding that high word).
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {
  const unsigned hi = (unsigned)(k >> 32), lo = (unsigned)k;
  const unsigned H = __reduce_max_sync(0xffffffffu, hi);
  const unsigned L = __reduce_max_sync(0xffffffffu, hi == H ? lo : 0u);
  return ((unsigned long long)H << 32) | L;
}

// One warp per sequence.  Every inserted node owns one candidate key in
// shared memory (its best remaining child).  A step takes the best candidate,
// a child (p, r) of node p at depth d, and with it the longest run of p's
// next-ranked children (p, r+1), (p, r+2), ... that still beat every other
// candidate: the best key outside p's slot, and the first child of (p, r),
// which is the best of the run's own first children (their path scores do not
// increase along the run and a later node loses ties on its parent index).
// Inserting the run in one step therefore gives the order of one-at-a-time
// insertion.  Lane i tests (p, r+i); the run is the ballot's leading ones.
// A_hat, the fp64 sum of the non-root path scores in insertion order, is
// order-independent when every partial sum is exact: all terms are multiples
// of 2^b (b the lowest set bit over the terms) and the sum stays below
// 2^(e+9) (e the largest term's exponent, at most 255 terms), so
// e + 9 - b <= 53 makes every addition exact and the warp adds in any order;
// otherwise lane 0 adds in insertion order.
__global__ void __launch_bounds__(kExpandThreads)
expand_kernel(const int32_t *__restrict__ top_tok, const float *__restrict__ top_q,
              const int32_t *__restrict__ root_token, int K, int M, int N,
              int32_t *__restrict__ parent, int32_t *__restrict__ tokens,
              int32_t *__restrict__ depth, float *__restrict__ rho, double *__restrict__ ahat) {
  extern __shared__ unsigned char smem_raw[];
  float *s_tq = reinterpret_cast<float *>(smem_raw);                  // [K][M]
  int32_t *s_tt = reinterpret_cast<int32_t *>(s_tq + (size_t)K * M);  // [K][M]
  __shared__ unsigned long long s_key[kMaxNodes];
  __shared__ float s_rho[kMaxNodes];
  __shared__ int32_t s_dep[kMaxNodes], s_nch[kMaxNodes], s_par[kMaxNodes], s_tok[kMaxNodes];

  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, t = threadIdx.x;
  {
    // the ranked lists, sixteen loads of each kind in flight per thread (one
    // round trip for K * M <= 4096)
    constexpr int kU = 16;
    const int KM = K * M;
    const float *gq = top_q + (size_t)b * KM;
    const int32_t *gt = top_tok + (size_t)b * KM;
    for (int x0 = t; x0 < KM; x0 += kU * kExpandThreads) {
      float qv[kU];
      int32_t tv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int x = x0 + u * kExpandThreads;
        qv[u] = x < KM ? __ldg(gq + x) : 0.f;
        tv[u] = x < KM ? __ldg(gt + x) : 0;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int x = x0 + u * kExpandThreads;
        if (x < KM) {
          s_tq[x] = qv[u];
          s_tt[x] = tv[u];
        }
      }
    }
  }
  for (int x = t; x < kMaxNodes; x += kExpandThreads) {
    s_key[x] = 0ull;
    s_rho[x] = 0.f;
    s_dep[x] = 0;
    s_nch[x] = 0;
    s_par[x] = -1;
    s_tok[x] = -1;
  }
  __syncthreads();
  if (t >= 32) return;
  const int lane = t;
  if (lane == 0) {
    s_rho[0] = 1.f;
    s_tok[0] = root_token[b];
    s_key[0] = child_key(0, 1.f, 0, 0, s_tq, K, M, N);
  }
  __syncwarp();

  int n = 1;
  for (int step = 1; n < N && step < N; ++step) {  // a step inserts at least one node
    unsigned long long k[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) k[j] = s_key[lane + 32 * j];
    const unsigned long long best =
        warp_max_key(max_u64(max_u64(max_u64(k[0], k[1]), max_u64(k[2], k[3])),
                             max_u64(max_u64(k[4], k[5]), max_u64(k[6], k[7]))));
    if (best == 0ull) break;  // no valid node left (host checks make this unreachable)
    const int p = 0xFFFF - (int)(best & 0xFFFFu);
    const int d = 255 - (int)((best >> 16) & 0xFFu);
    // the best key outside p's slot
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) k[j] = lane + 32 * j == p ? 0ull : k[j];
    const unsigned long long k2 =
        warp_max_key(max_u64(max_u64(max_u64(k[0], k[1]), max_u64(k[2], k[3])),
                             max_u64(max_u64(k[4], k[5]), max_u64(k[6], k[7]))));
    const int r = s_nch[p];
    const float rp = s_rho[p];
    const float *q_row = s_tq + (d - 1) * M;
    // the first child of (p, r), the run's first node
    const unsigned long long fc0 =
        child_key(n, __uint_as_float((unsigned)(best >> 32)), d, 0, s_tq, K, M, N);
    const unsigned long long bound = max_u64(k2, fc0);
    const int ri = r + lane;
    const bool ok = ri < M && n + lane < N;
    float rc = 0.f;
    if (ok) rc = __fmul_rn(rp, q_row[ri]);
    const unsigned long long key =
        ok ? ((unsigned long long)__float_as_uint(rc) << 32) |
                 (unsigned long long)(((unsigned)(255 - d) << 16) | (unsigned)(0xFFFF - p))
           : 0ull;
    const unsigned pass = __ballot_sync(0xffffffffu, key > bound);
    const int run = ~pass ? __ffs(~pass) - 1 : 32;  // lane 0 (the best key) always passes
    if (run == 0) break;
    if (lane < run) {
      const int node = n + lane;
      s_par[node] = p;
      s_tok[node] = s_tt[(d - 1) * M + ri];
      s_dep[node] = d;
      s_rho[node] = rc;
      s_key[node] = child_key(node, rc, d, 0, s_tq, K, M, N);
    }
    if (lane == 0) {
      s_nch[p] = r + run;
      s_key[p] = child_key(p, rp, d - 1, r + run, s_tq, K, M, N);
    }
    n += run;
    __syncwarp();
  }
  const int filled = n;

  // A_hat.  When the sum is exact (e_max + 9 - b_min <= 53) every term is an
  // integer multiple of 2^b_min and the total below 2^53 of them: the terms
  // are added as 64-bit integers (the warp's fp64 pipe is slow on this part)
  // and the total scaled once; otherwise lane 0 adds in insertion order.
  int e_max = -1000, b_min = 1000;
  for (int x = 1 + lane; x < filled; x += 32) {
    const unsigned u = __float_as_uint(s_rho[x]) & 0x7FFFFFFFu;
    if (u == 0u) continue;
    const int e = (int)(u >> 23), m = (int)(u & 0x7FFFFFu);
    const int sig = e ? (m | 0x800000) : m;
    const int lo = (e ? e - 150 : -149) + __ffs(sig) - 1;
    const int ex = e ? e - 127 : -149 + (31 - __clz(m));
    e_max = ex > e_max ? ex : e_max;
    b_min = lo < b_min ? lo : b_min;
  }
  e_max = __reduce_max_sync(0xffffffffu, e_max);
  b_min = __reduce_min_sync(0xffffffffu, b_min);
  double a_hat = 0.0;
  if (e_max == -1000) {
    // every term zero
  } else if (e_max + 9 - b_min <= 53) {
    long long part = 0;
    for (int x = 1 + lane; x < filled; x += 32) {
      const unsigned w = __float_as_uint(s_rho[x]);
      const unsigned u = w & 0x7FFFFFFFu;
      if (u == 0u) continue;
      const int e = (int)(u >> 23), m = (int)(u & 0x7FFFFFu);
      const long long sig = e ? (m | 0x800000) : m;
      const int sh = (e ? e - 150 : -149) - b_min;  // term = sig * 2^sh, sh >= -(trailing zeros)
      const long long term = sh >= 0 ? sig << sh : sig >> -sh;
      part += (w >> 31) ? -term : term;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    a_hat = ldexp((double)part, b_min);
  } else if (lane == 0) {
    for (int x = 1; x < filled; ++x) a_hat += (double)s_rho[x];
  }
  for (int x = lane; x < N; x += 32) {
    const bool ok = x < filled;
    parent[(size_t)b * N + x] = ok ? s_par[x] : -1;
    tokens[(size_t)b * N + x] = ok ? s_tok[x] : -1;
    depth[(size_t)b * N + x] = ok ? s_dep[x] : 0;
    rho[(size_t)b * N + x] = ok ? s_rho[x] : 0.f;
  }
  if (lane == 0) ahat[b] = a_hat;
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

// ---------------------------------------------------------------------------
// Dynamic draft trees.  Pool layout per sequence: root at 0; level 1 at 1..k;
// level l >= 2 at 1 + k + (l-2) k^2 + f k + j (frontier slot f, token rank j).

constexpr int kDynMaxK = 32;         // tokens per expanded node, frontier width
constexpr int kDynMaxPool = 8192;    // pool ids per sequence (rerank sorts them in shared memory)
constexpr int kDynThreads = 1024;

__host__ __device__ inline long dyn_base(int level, int k) {
  return level == 1 ? 1L : 1L + k + (long)(level - 2) * k * k;
}

// Bitonic sort of n (a power of two, <= 2 * blockDim.x * ...) keys in shared
// memory, descending; every thread of the block calls it.
__device__ void bitonic_desc(unsigned long long *keys, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int l = i ^ stride;
        if (l > i) {
          const unsigned long long a = keys[i], c = keys[l];
          const bool up = (i & size) == 0;
          if (up ? (a < c) : (a > c)) {
            keys[i] = c;
            keys[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// One block per sequence: the F * k children of one level.  Child c = f k + j
// of frontier node frontier[f] takes token top_tok[f][j] with score
// fl32(score(parent) * top_q[f][j]); the next frontier is the k best children
// by (score desc, pool id asc).
__global__ void __launch_bounds__(kDynThreads)
dyn_expand_kernel(const int32_t *__restrict__ top_tok, const float *__restrict__ top_q,
                  const int32_t *__restrict__ root_token, const int32_t *__restrict__ frontier,
                  int F, int k, int level, int M_max, int32_t *__restrict__ pool_parent,
                  int32_t *__restrict__ pool_token, int32_t *__restrict__ pool_depth,
                  float *__restrict__ pool_score, int32_t *__restrict__ next_frontier) {
  __shared__ unsigned long long s_key[kDynMaxK * kDynMaxK];
  __shared__ float s_pscore[kDynMaxK];
  __shared__ int32_t s_parent[kDynMaxK];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, t = threadIdx.x;
  const size_t pb = (size_t)b * M_max;
  if (level == 1 && t == 0) {
    pool_parent[pb] = -1;
    pool_token[pb] = root_token[b];
    pool_depth[pb] = 0;
    pool_score[pb] = 1.f;
  }
  if (t < F) {
    // a frontier id outside the pool (not one a previous level wrote) gives
    // children with parent -1 and score 0, which a1 then rejects
    int par = level == 1 ? 0 : frontier[(size_t)b * F + t];
    const bool ok = par >= 0 && par < M_max;
    par = ok ? par : -1;
    s_parent[t] = par;
    s_pscore[t] = level == 1 ? 1.f : (ok ? pool_score[pb + par] : 0.f);
  }
  const int n = F * k;
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  __syncthreads();
  const long base = dyn_base(level, k);
  for (int c = t; c < n2; c += blockDim.x) {
    unsigned long long key = 0ull;
    if (c < n) {
      const int f = c / k;
      const size_t src = ((size_t)b * F + f) * k + (c - f * k);
      const float sc = __fmul_rn(s_pscore[f], top_q[src]);
      const long pid = base + c;
      pool_parent[pb + pid] = s_parent[f];
      pool_token[pb + pid] = top_tok[src];
      pool_depth[pb + pid] = level;
      pool_score[pb + pid] = sc;
      key = ((unsigned long long)order_key(sc) << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)pid);
    }
    s_key[c] = key;
  }
  __syncthreads();
  bitonic_desc(s_key, n2);
  if (t < k) next_frontier[(size_t)b * k + t] = (int32_t)(0xFFFFFFFFu - (unsigned)(s_key[t] & 0xFFFFFFFFull));
}

// One block per sequence: the root and the N-1 best of pool ids 1..M-1 by
// (score desc, depth asc, pool id asc), in that order; parents re-indexed to
// output positions (-1 for the root, and for a node whose parent was not kept,
// which draft probabilities <= 1 rule out).
__global__ void __launch_bounds__(kDynThreads)
dyn_rerank_kernel(const int32_t *__restrict__ pool_parent, const int32_t *__restrict__ pool_token,
                  const int32_t *__restrict__ pool_depth, const float *__restrict__ pool_score,
                  int M, int M_max, int N, int32_t *__restrict__ parent,
                  int32_t *__restrict__ tokens, int32_t *__restrict__ depth,
                  float *__restrict__ score) {
  extern __shared__ unsigned long long s_keys[];  // [n2], then int32 map [M]
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, t = threadIdx.x;
  const size_t pb = (size_t)b * M_max;
  const int n = M - 1;
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  int32_t *s_map = reinterpret_cast<int32_t *>(s_keys + n2);
  for (int i = t; i < n2; i += blockDim.x) {
    unsigned long long key = 0ull;
    if (i < n) {
      const int pid = i + 1;
      const unsigned dk = 31u - (unsigned)min(max(pool_depth[pb + pid], 0), 31);
      key = ((unsigned long long)order_key(pool_score[pb + pid]) << 32) |
            (unsigned long long)((dk << 27) | (0x7FFFFFFu - (unsigned)pid));
    }
    s_keys[i] = key;
  }
  for (int i = t; i < M; i += blockDim.x) s_map[i] = -1;
  __syncthreads();
  bitonic_desc(s_keys, n2);
  const size_t ob = (size_t)b * N;
  if (t == 0) s_map[0] = 0;
  for (int r = t; r < N - 1; r += blockDim.x)
    s_map[0x7FFFFFF - (int)(s_keys[r] & 0x7FFFFFFull)] = r + 1;
  __syncthreads();
  for (int r = t; r < N; r += blockDim.x) {
    const int pid = r == 0 ? 0 : 0x7FFFFFF - (int)(s_keys[r - 1] & 0x7FFFFFFull);
    const int pp = pool_parent[pb + pid];
    parent[ob + r] = (r == 0 || pp < 0 || pp >= M) ? -1 : s_map[pp];
    tokens[ob + r] = pool_token[pb + pid];
    depth[ob + r] = pool_depth[pb + pid];
    score[ob + r] = pool_score[pb + pid];
  }
}

// Ranked top M of every row by a threshold filter (M < kFiltThreads).
// Pass 1: every thread's best key over its elements; the M-th best of those
// per-thread bests, tau, is a lower bound of the row's M-th best key (the M
// best per-thread bests are M distinct elements), so the top M all have keys
// >= tau.  Pass 2 (the row is now in L1/L2) collects the keys >= tau, usually
// little more than M of them, and a bitonic sort ranks them.  Keys are
// (order_key(q) << 32 | ~index), distinct, larger is better: the ranking
// (q desc, token id asc).  More than kFiltCap candidates (not seen with real
// distributions) falls back to the radix select in the same block.
constexpr int kFiltThreads = 512;
constexpr int kFiltCap = 2048;

__global__ void __launch_bounds__(kFiltThreads)
topk_filter_kernel(const float *__restrict__ q, int K, int V, int M, int32_t *__restrict__ top_tok,
                   float *__restrict__ top_q) {
  __shared__ unsigned long long s_best[kFiltThreads];
  __shared__ unsigned long long s_cand[kFiltCap];
  __shared__ unsigned s_count;
  pdl_trigger();
  pdl_wait();
  const int k = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const float *row = q + ((size_t)b * K + k) * (size_t)V;
  const size_t o = ((size_t)b * K + k) * M;
  auto key2 = [](float v, int x) {
    return ((unsigned long long)order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)x);
  };
  // rows of a multiple of 4 floats are read as float4 (16-byte aligned: the
  // caller's q is); others element by element
  const bool vec = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
  const float4 *row4 = reinterpret_cast<const float4 *>(row);
  const int V4 = V >> 2;
  unsigned long long best = 0ull;
  // eight loads per thread issued before any is used
  constexpr int kU = 8;
  if (vec) {
    for (int x0 = t; x0 < V4; x0 += kU * kFiltThreads) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (x0 + u * kFiltThreads < V4) v[u] = __ldg(row4 + x0 + u * kFiltThreads);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int x4 = x0 + u * kFiltThreads;
        if (x4 < V4) {
          const int x = 4 * x4;
          unsigned long long k0 = key2(v[u].x, x), k1 = key2(v[u].y, x + 1),
                             k2 = key2(v[u].z, x + 2), k3 = key2(v[u].w, x + 3);
          k0 = k1 > k0 ? k1 : k0;
          k2 = k3 > k2 ? k3 : k2;
          k0 = k2 > k0 ? k2 : k0;
          best = k0 > best ? k0 : best;
        }
      }
    }
  } else {
    for (int x0 = t; x0 < V; x0 += kU * kFiltThreads) {
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (x0 + u * kFiltThreads < V) v[u] = __ldg(row + x0 + u * kFiltThreads);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int x = x0 + u * kFiltThreads;
        if (x < V) {
          const unsigned long long key = key2(v[u], x);
          best = key > best ? key : best;
        }
      }
    }
  }
  s_best[t] = best;
  if (t == 0) s_count = 0u;
  __syncthreads();
  bitonic_desc(s_best, kFiltThreads);
  const unsigned long long tau = s_best[M - 1];
  auto offer = [&](unsigned long long key) {
    if (key >= tau) {
      const unsigned i = atomicAdd(&s_count, 1u);
      if (i < (unsigned)kFiltCap) s_cand[i] = key;
    }
  };
  if (vec) {
    for (int x0 = t; x0 < V4; x0 += kU * kFiltThreads) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (x0 + u * kFiltThreads < V4) v[u] = __ldg(row4 + x0 + u * kFiltThreads);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int x4 = x0 + u * kFiltThreads;
        if (x4 < V4) {
          const int x = 4 * x4;
          offer(key2(v[u].x, x));
          offer(key2(v[u].y, x + 1));
          offer(key2(v[u].z, x + 2));
          offer(key2(v[u].w, x + 3));
        }
      }
    }
  } else {
    for (int x0 = t; x0 < V; x0 += kU * kFiltThreads) {
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (x0 + u * kFiltThreads < V) v[u] = __ldg(row + x0 + u * kFiltThreads);
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (x0 + u * kFiltThreads < V) offer(key2(v[u], x0 + u * kFiltThreads));
    }
  }
  __syncthreads();
  const int n = (int)s_count;
  if (n > kFiltCap) {  // block-uniform
    radix_topk_block(row, V, M, top_tok + o, top_q + o);
    return;
  }
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  for (int i = n + t; i < n2; i += kFiltThreads) s_cand[i] = 0ull;
  __syncthreads();
  bitonic_desc(s_cand, n2);
  for (int r = t; r < M; r += kFiltThreads) {
    const int idx = (int)(0xFFFFFFFFu - (unsigned)(s_cand[r] & 0xFFFFFFFFull));
    top_tok[o + r] = idx;
    top_q[o + r] = __ldg(row + idx);
  }
}

// The threshold filter with the row staged in shared memory (rows of at most
// kStageMaxV floats): one block of 1024 threads per row.
//  1. The row is read once into shared memory (bulk copies for rows of whole
//     16-byte words, else element loads); each thread keeps the largest of
//     its values (NaN ignored).
//  2. Each warp sorts its 32 thread maxima (shuffles) and takes the
//     ceil(M/32)-th; tau, the least of the warps' values, has at least M
//     non-NaN elements at or above it, so every one of the M best (by order
//     key, index) passes !(v < tau) (NaN always passes).
//  3. The passing elements become 64-bit keys (order key, 0xFFFFFFFF - index)
//     in a candidate list, appended a warp at a time (one atomic per warp).
//  4. A radix select over the candidates (8-bit digits from the top, ending
//     once the digit's bin is taken whole) keeps exactly the M largest keys.
//  5. The kept keys are sorted in runs of 32 (one warp each, shuffles); a key's
//     rank is its place in its run plus, for every other run, the number of
//     its keys above it (binary search).
// More candidates than kStageCap (many ties at tau) fall back to the radix
// select over the row.
constexpr int kStageThreads = 1024;
constexpr int kStageWarps = kStageThreads / 32;
constexpr int kStageMaxV = 40960;  // 160 KB of staged row
constexpr int kStageCap = 2048;
constexpr int kStageMaxM = 511;

// Bitonic sort of one key per lane across the warp, descending.
template <typename T>
__device__ __forceinline__ T warp_sort_desc(T x, int lane) {
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
      const T y = __shfl_xor_sync(0xffffffffu, x, j);
      const bool take_max = ((lane & kk) == 0) == ((lane & j) == 0);
      x = take_max ? (x > y ? x : y) : (x < y ? x : y);
    }
  }
  return x;
}

__global__ void __launch_bounds__(kStageThreads)
topk_stage_kernel(const float *__restrict__ q, int K, int V, int M, int32_t *__restrict__ top_tok,
                  float *__restrict__ top_q, unsigned long long wait_limit_ns) {
  extern __shared__ __align__(16) float s_row[];  // [V]
  __shared__ unsigned long long s_cand[kStageCap];
  __shared__ unsigned long long s_sel[kStageMaxM + 1];
  __shared__ __align__(16) float s_wtau[kStageWarps];
  __shared__ unsigned s_hist[256];
  __shared__ unsigned s_count, s_nsel, s_rem, s_bin_count;
  __shared__ unsigned long long s_prefix;
  __shared__ uint64_t s_bar;
  pdl_trigger();
  const int k = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const float *row = q + ((size_t)b * K + k) * (size_t)V;
  const size_t o = ((size_t)b * K + k) * M;
  const unsigned lane_lt = (1u << lane) - 1u;
  const bool vec = (V & 3) == 0 && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
  const uint32_t bar = sm100::smem_addr(&s_bar);
  if (vec && t == 0) {
    sm100::mbar_init(bar, 1);
    sm100::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();

  // 1. stage the row, then each thread's largest value.  A row of whole
  // 16-byte words arrives by bulk copies (the copy engine keeps far more of it
  // in flight than the threads' own loads); other rows element by element.
  float fmx = -INFINITY;
  const int V4 = V >> 2;
  if (vec) {
    if (t == 0) {
      constexpr uint32_t kChunk = 16384;
      const uint32_t bytes = (uint32_t)V * 4u;
      sm100::mbar_arrive_expect_tx(bar, bytes);
      for (uint32_t off = 0; off < bytes; off += kChunk)
        sm100::bulk_load(sm100::smem_addr(s_row) + off, reinterpret_cast<const char *>(row) + off,
                         bytes - off < kChunk ? bytes - off : kChunk, bar);
    }
    const bool landed = sm100::mbar_wait(bar, 0, wait_limit_ns);
    if (__syncthreads_or(!landed)) {
      // the copy did not land in time: the result from global memory, and a
      // second bounded wait so that no copy is left writing this block's
      // shared memory after it exits
      radix_topk_block(row, V, M, top_tok + o, top_q + o);
      sm100::mbar_wait(bar, 0, wait_limit_ns);
      return;
    }
    const float4 *s_row4 = reinterpret_cast<const float4 *>(s_row);
#pragma unroll 4
    for (int x4 = t; x4 < V4; x4 += kStageThreads) {
      const float4 v = s_row4[x4];
      fmx = fmaxf(fmx, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
    }
  } else {
    constexpr int kU = 8;  // eight loads per thread in flight
    for (int x0 = t; x0 < V; x0 += kU * kStageThreads) {
      float v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (x0 + u * kStageThreads < V) v[u] = __ldg(row + x0 + u * kStageThreads);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (x0 + u * kStageThreads < V) {
          s_row[x0 + u * kStageThreads] = v[u];
          fmx = fmaxf(fmx, v[u]);
        }
      }
    }
  }
  if (t == 0) {
    s_count = 0u;
    s_nsel = 0u;
  }
  // 2. the warp's ceil(M/32)-th largest thread maximum; tau the least of them
  {
    const float x = warp_sort_desc(fmx, lane);
    const int mw = (M + kStageWarps - 1) / kStageWarps;  // 1..16 for M <= 511
    const float wt = __shfl_sync(0xffffffffu, x, mw - 1);
    if (lane == 0) s_wtau[warp] = wt;
  }
  __syncthreads();
  float tau = INFINITY;
#pragma unroll
  for (int w = 0; w < kStageWarps; w += 4) {
    const float4 w4 = *reinterpret_cast<const float4 *>(&s_wtau[w]);
    tau = fminf(tau, fminf(fminf(w4.x, w4.y), fminf(w4.z, w4.w)));
  }

  // 3. candidates: every element with !(v < tau), appended a warp at a time
  auto put = [&](unsigned i, float v, int x) {
    if (i < (unsigned)kStageCap)
      s_cand[i] = ((unsigned long long)order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)x);
  };
  if (vec) {
    const float4 *s_row4 = reinterpret_cast<const float4 *>(s_row);
    // (kept rolled: the append path is long and rarely taken)
#pragma unroll 1
    for (int w0 = warp * 32; w0 < V4; w0 += kStageThreads) {
      {
        const int x4 = w0 + lane;
        unsigned m = 0u;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (x4 < V4) {
          v = s_row4[x4];
          m = (unsigned)!(v.x < tau) | ((unsigned)!(v.y < tau) << 1) | ((unsigned)!(v.z < tau) << 2) |
              ((unsigned)!(v.w < tau) << 3);
        }
        if (__any_sync(0xffffffffu, m != 0u)) {
          const unsigned b0 = __ballot_sync(0xffffffffu, m & 1u), b1 = __ballot_sync(0xffffffffu, m & 2u);
          const unsigned b2 = __ballot_sync(0xffffffffu, m & 4u), b3 = __ballot_sync(0xffffffffu, m & 8u);
          const unsigned c0 = __popc(b0), c1 = __popc(b1), c2 = __popc(b2), c3 = __popc(b3);
          unsigned base = 0u;
          if (lane == 0) base = atomicAdd(&s_count, c0 + c1 + c2 + c3);
          base = __shfl_sync(0xffffffffu, base, 0);
          if (m & 1u) put(base + __popc(b0 & lane_lt), v.x, 4 * x4);
          if (m & 2u) put(base + c0 + __popc(b1 & lane_lt), v.y, 4 * x4 + 1);
          if (m & 4u) put(base + c0 + c1 + __popc(b2 & lane_lt), v.z, 4 * x4 + 2);
          if (m & 8u) put(base + c0 + c1 + c2 + __popc(b3 & lane_lt), v.w, 4 * x4 + 3);
        }
      }
    }
  } else {
    for (int w0 = warp * 32; w0 < V; w0 += kStageThreads) {
      const int x = w0 + lane;
      float v = 0.f;
      bool pass = false;
      if (x < V) {
        v = s_row[x];
        pass = !(v < tau);
      }
      const unsigned bal = __ballot_sync(0xffffffffu, pass);
      if (bal) {
        unsigned base = 0u;
        if (lane == 0) base = atomicAdd(&s_count, (unsigned)__popc(bal));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (pass) put(base + __popc(bal & lane_lt), v, x);
      }
    }
  }
  __syncthreads();
  const int n = (int)s_count;
  if (n > kStageCap) {  // block-uniform
    radix_topk_block(row, V, M, top_tok + o, top_q + o);
    return;
  }

  // 4. the M largest candidates: radix select
  unsigned long long prefix = 0ull, pmask = 0ull;
  if (n > M) {
    unsigned remaining = (unsigned)M;
    for (int shift = 56; shift >= 0; shift -= 8) {
      if (t < 256) s_hist[t] = 0u;
      __syncthreads();
      for (int i = t; i < n; i += kStageThreads) {
        const unsigned long long kk = s_cand[i];
        if ((kk & pmask) == prefix) atomicAdd(&s_hist[(unsigned)(kk >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255-8l .. 248-8l (descending)
        unsigned c[8], sum = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = s_hist[255 - 8 * lane - j];
          sum += c[j];
        }
        unsigned incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
        if (lane == __ffs(hit) - 1) {
          // the first of this lane's bins where the running count reaches
          // `remaining` (unrolled: the counts stay in registers)
          unsigned cum = incl - sum, pick_cum = 0u, pick_c = 0u;
          int pick_j = -1;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (pick_j < 0 && cum + c[j] >= remaining) {
              pick_j = j;
              pick_cum = cum;
              pick_c = c[j];
            }
            cum += c[j];
          }
          s_prefix = prefix | ((unsigned long long)(255 - 8 * lane - pick_j) << shift);
          s_rem = remaining - pick_cum;
          s_bin_count = pick_c;
        }
      }
      __syncthreads();
      prefix = s_prefix;
      remaining = s_rem;
      pmask |= 0xFFull << shift;
      if (s_bin_count == remaining) break;  // the bin is taken whole (block-uniform)
    }
  }
  // kept: every key whose selected digits are >= the prefix (exactly M keys)
  for (int i = t; i < n; i += kStageThreads) {
    const unsigned long long kk = s_cand[i];
    if ((kk & pmask) >= prefix) s_sel[atomicAdd(&s_nsel, 1u)] = kk;
  }
  __syncthreads();

  // 5. runs of 32 sorted by one warp each (padding 0 sorts below every key:
  // a key's low word 0xFFFFFFFF - index is never 0 for index < V), then ranks
  const int runs = (M + 31) >> 5;
  unsigned long long key = 0ull;
  if (warp < runs) {
    const int i = warp * 32 + lane;
    key = warp_sort_desc(i < M ? s_sel[i] : 0ull, lane);
    s_cand[i] = key;  // the candidates are no longer needed
  }
  __syncthreads();
  if (warp < runs && key != 0ull) {
    int rank = lane;
    for (int r = 0; r < runs; ++r) {
      if (r == warp) continue;
      const unsigned long long *run = s_cand + r * 32;
      int pos = 0;  // keys of run r above `key` (the run is descending)
#pragma unroll
      for (int step = 16; step > 0; step >>= 1)
        if (run[pos + step - 1] > key) pos += step;
      pos += run[pos] > key ? 1 : 0;  // the search reaches 31 at most; all 32 above
      rank += pos;
    }
    const int idx = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull));
    top_tok[o + rank] = idx;
    top_q[o + rank] = s_row[idx];
  }
}

// Ranked top M of every row of q [B][K][V]: the staged threshold filter for
// rows that fit in shared memory, else the threshold filter, or the radix
// select for M >= kFiltThreads.
cudaError_t launch_topk(const float *q, int K, int B, int V, int M, int32_t *top_tok, float *top_q,
                        cudaStream_t s) {
  if (M <= kStageMaxM && V <= kStageMaxV) {
    const size_t smem = align_up((size_t)V * sizeof(float), 16);
    if (!set_smem((const void *)topk_stage_kernel, (size_t)kStageMaxV * sizeof(float)))
      return cudaErrorInvalidValue;
    return launch(topk_stage_kernel, dim3(K, B), dim3(kStageThreads), smem, s, q, K, V, M, top_tok,
                  top_q, (unsigned long long)option(TSD_OPT_WAIT_LIMIT_NS));
  }
  if (M < kFiltThreads)
    return launch(topk_filter_kernel, dim3(K, B), dim3(kFiltThreads), 0, s, q, K, V, M, top_tok,
                  top_q);
  return launch(topk_kernel, dim3(K, B), dim3(kTopThreads), 0, s, q, K, V, M, top_tok, top_q);
}

size_t dyn_rerank_smem(int M) {
  int n2 = 1;
  while (n2 < M - 1) n2 <<= 1;
  return (size_t)n2 * sizeof(unsigned long long) + (size_t)M * sizeof(int32_t);
}

}  // namespace
}  // namespace tsd

TSD_API size_t tsd_dynamic_tree_workspace_bytes(int B, int F, int k) {
  if (B <= 0 || F <= 0 || k <= 0 || F > tsd::kDynMaxK || k > tsd::kDynMaxK) return 0;
  return tsd::align_up((size_t)B * F * k * sizeof(int32_t), 256) + (size_t)B * F * k * sizeof(float);
}

TSD_API int tsd_dynamic_tree_expand(const float *q, const int32_t *root_token, int B, int F, int V,
                                    int k, int level, const int32_t *frontier,
                                    int32_t *pool_parent, int32_t *pool_token, int32_t *pool_depth,
                                    float *pool_score, int M_max, int32_t *next_frontier,
                                    void *workspace, size_t ws_bytes, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0) return TSD_ERR_ARG;
  if (k < 1 || k > kDynMaxK || level < 1 || V < k || B > 65535 || M_max < 1 ||
      M_max > kDynMaxPool)
    return TSD_ERR_LIMIT;
  if (F != (level == 1 ? 1 : k)) return TSD_ERR_ARG;
  if (dyn_base(level, k) + (long)F * k > (long)M_max) return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!q || !pool_parent || !pool_token || !pool_depth || !pool_score || !next_frontier)
    return TSD_ERR_ARG;
  if (level == 1 ? !root_token : !frontier) return TSD_ERR_ARG;
  if (frontier && frontier == next_frontier) return TSD_ERR_ARG;
  const size_t tok_bytes = align_up((size_t)B * F * k * sizeof(int32_t), 256);
  if (!workspace || ws_bytes < tok_bytes + (size_t)B * F * k * sizeof(float) ||
      !aligned(workspace, 16))
    return TSD_ERR_WORKSPACE;
  int32_t *top_tok = static_cast<int32_t *>(workspace);
  float *top_q = reinterpret_cast<float *>(static_cast<char *>(workspace) + tok_bytes);
  cudaStream_t s = as_cuda(stream);
  if (launch_topk(q, F, B, V, k, top_tok, top_q, s) != cudaSuccess) return TSD_ERR_CUDA;
  if (launch(dyn_expand_kernel, dim3(B), dim3(kDynThreads), 0, s, top_tok, top_q, root_token,
             frontier, F, k, level, M_max, pool_parent, pool_token, pool_depth, pool_score,
             next_frontier) != cudaSuccess)
    return TSD_ERR_CUDA;
  return TSD_OK;
}

TSD_API int tsd_dynamic_tree_rerank(const int32_t *pool_parent, const int32_t *pool_token,
                                    const int32_t *pool_depth, const float *pool_score, int B,
                                    int M, int M_max, int N, int32_t *parent, int32_t *tokens,
                                    int32_t *depth, float *score, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0) return TSD_ERR_ARG;
  if (N < 1 || N > kMaxNodes || M < N || M > M_max || M_max > kDynMaxPool || B > 65535)
    return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!pool_parent || !pool_token || !pool_depth || !pool_score || !parent || !tokens || !depth ||
      !score)
    return TSD_ERR_ARG;
  const size_t smem = dyn_rerank_smem(M);
  if (!set_smem((const void *)dyn_rerank_kernel, dyn_rerank_smem(kDynMaxPool))) return TSD_ERR_CUDA;
  if (launch(dyn_rerank_kernel, dim3(B), dim3(kDynThreads), smem, as_cuda(stream), pool_parent,
             pool_token, pool_depth, pool_score, M, M_max, N, parent, tokens, depth, score) !=
      cudaSuccess)
    return TSD_ERR_CUDA;
  return TSD_OK;
}

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
  if (p.M > 0 && launch_topk(q, K, B, V, p.M, top_tok, top_q, s) != cudaSuccess) return TSD_ERR_CUDA;
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
