// Stochastic verification of a draft tree by modified rejection sampling.
//
// "Speculative Decoding Hierárquico: Medusa, EAGLE-2 e Multi-Token
// Prediction", section on classic speculative decoding: a drafted token x
// drawn from the draft distribution q is accepted with probability
// min(1, p(x)/q(x)); on rejection a corrective token is drawn from the
// normalised residual max(0, p - q), which keeps the emitted token
// distributed as the target p.  For a tree (the same page's Medusa section:
// every branch is scored in one pass, one path is kept) the children of node
// i are independent draws from q_i, tried in increasing id order, each
// against the residual the previous rejections left; when every child is
// rejected node i draws its token from that residual, and a walk that ends
// at a leaf draws from the leaf's target distribution.
//
// One launch, one thread-block cluster of C CTAs per node; CTA c owns the
// slice [c*S, c*S + S) of the node's vocabulary row.
//
// An internal node brings its target row into shared memory (bulk copies,
// one barrier per chunk; each thread keeps a running max and sum of
// exponentials as the chunks land) and decides its children.  The draft row
// is read only after a rejection.  Per-CTA partial results (max, sum, the
// weight at the next child's token) are exchanged through distributed shared
// memory between cluster barriers, and every control decision is taken from
// those exchanged values with the same instructions in every CTA, so all
// CTAs of a cluster pass the same number of barriers.
//
// A leaf decides nothing; each of its CTAs streams its slice once and records
// the slice's (max, sum of exponentials), which is all a later draw from the
// leaf needs to locate its token.
//
// Every node, and every CTA of a leaf, takes a per-sequence ticket when done;
// the CTA taking the last one walks the accepted children from the root and,
// when the walk ends at a leaf, draws the bonus token there: the recorded
// sums pick the slice holding the draw, and only that slice is read again.

#include <climits>
#include <cmath>

#include "sm100_ptx.cuh"
#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kST = 256;                    // threads per CTA (>= kMaxNodes)
constexpr int kSW = kST / 32;               // warps per CTA
constexpr int kSBatch = 8;                  // 16-byte loads in flight per thread
constexpr int kMaxJ = 32;                   // float4s per thread and slice
constexpr int kMaxS = 4 * kST * kMaxJ;      // floats per CTA slice (128 KB)
constexpr int kMaxCluster = 8;              // portable cluster size
constexpr int kChunks = 4;                  // bulk copies (and barriers) per slice
constexpr float kLog2e = 1.4426950408889634f;

struct __align__(16) Slot {
  float m;    // CTA max of the target logits (first exchange only)
  float s;    // CTA sum of the current weights
  float pub;  // weight (first exchange: raw logit) at the next child's token
  float pad;
};

struct Ctl {
  float m, Z;    // global max of the logits, normaliser of the current level
  float pub;     // exchanged weight at the child under test
  int cstar;     // CTA holding a draw
  float tau;     // draw target inside that CTA
  int fallback;  // no cumulative boundary exceeded the target: last positive
  int tok;
};

struct Smem {
  Slot slot[2][kMaxCluster];  // [round parity][source CTA], written by every CTA of the cluster
  Slot mine;                  // this CTA's contribution to the next exchange
  unsigned long long bar[kChunks];
  float T[kMaxCluster];      // per-CTA totals of the current level, global units
  float wf[kSW], wg[kSW];
  int wi[kSW], wj[kSW];
  Ctl ctl;
  int abort;
};

__device__ __forceinline__ float sum4(const float4 &v) { return (v.x + v.y) + (v.z + v.w); }
__device__ __forceinline__ float max4(const float4 &v) {
  return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
}
// exp(x - m) = 2^(x log2 e - m log2 e): one FMA and the hardware 2^x, with
// ml2 = m log2 e.  x = -inf gives 0.
__device__ __forceinline__ float exp_shift(float x, float ml2) {
  return sm100::ex2_approx(fmaf(x, kLog2e, -ml2));
}
__device__ __forceinline__ float4 exp4(float4 w, float ml2) {
  w.x = exp_shift(w.x, ml2);
  w.y = exp_shift(w.y, ml2);
  w.z = exp_shift(w.z, ml2);
  w.w = exp_shift(w.w, ml2);
  return w;
}

// Element k (a float4 index) of a row slice holding `cnt` valid floats;
// entries past the end read as `fill`.  Loads keep the lines in L2.
__device__ __forceinline__ float4 load_slice4(const float *p, int k, int cnt, int vec, float fill) {
  const int e = 4 * k;
  if (vec && e + 4 <= cnt) return __ldcg(reinterpret_cast<const float4 *>(p) + k);
  float4 r;
  r.x = e < cnt ? __ldcg(p + e) : fill;
  r.y = e + 1 < cnt ? __ldcg(p + e + 1) : fill;
  r.z = e + 2 < cnt ? __ldcg(p + e + 2) : fill;
  r.w = e + 3 < cnt ? __ldcg(p + e + 3) : fill;
  return r;
}

// (m, s) <- merge of two (max, sum of exp(x - max)) pairs; -inf maxima carry
// no mass.
__device__ __forceinline__ void merge_ms(float &m, float &s, float mo, float so) {
  const float mn = fmaxf(m, mo);
  if (mn == -INFINITY) return;
  s = s * sm100::ex2_approx((m - mn) * kLog2e) + so * sm100::ex2_approx((mo - mn) * kLog2e);
  m = mn;
}

// Running (max, sum of exp) of one thread over a group of float4s.
template <int kN>
__device__ __forceinline__ void stats_group(const float4 (&v)[kN], float &m_t, float &s_t) {
  float bm = -INFINITY;
#pragma unroll
  for (int u = 0; u < kN; ++u) bm = fmaxf(bm, max4(v[u]));
  const float mn = fmaxf(m_t, bm);
  if (mn == -INFINITY) return;
  const float ml2 = mn * kLog2e;
  float acc = s_t * sm100::ex2_approx((m_t - mn) * kLog2e);
#pragma unroll
  for (int u = 0; u < kN; ++u) acc += sum4(exp4(v[u], ml2));
  s_t = acc;
  m_t = mn;
}

// CTA (max, sum of exp) from every thread's pair; thread 0 holds the result.
__device__ __forceinline__ void block_ms(Smem &sm, float &m_t, float &s_t) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    merge_ms(m_t, s_t, __shfl_xor_sync(0xffffffffu, m_t, off),
             __shfl_xor_sync(0xffffffffu, s_t, off));
  if ((threadIdx.x & 31) == 0) {
    sm.wf[threadIdx.x >> 5] = m_t;
    sm.wg[threadIdx.x >> 5] = s_t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = sm.wf[0], s = sm.wg[0];
    for (int w = 1; w < kSW; ++w) merge_ms(m, s, sm.wf[w], sm.wg[w]);
    m_t = m;
    s_t = s;
  }
}

// Block sum of one float per thread: butterfly inside each warp, then the
// warp totals in warp order (the same association in every CTA).
__device__ __forceinline__ float block_sum(float v, float *s_w) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < kSW; ++w) r += s_w[w];
  __syncthreads();
  return r;
}

__device__ __forceinline__ void init_bars(Smem &sm) {
  using namespace sm100;
  if (threadIdx.x == 0) {
    sm.abort = 0;
#pragma unroll
    for (int j = 0; j < kChunks; ++j) mbar_init(smem_addr(&sm.bar[j]), 1);
    fence_mbar_init();
  }
  __syncthreads();
}

// This CTA's slice of one target row into R4 (raw logits, -inf past the
// row); thread 0 ends with the slice's (max, sum of exp) in sm.mine.
// One thread issues kChunks bulk copies, each completing its own barrier;
// every thread folds its elements of a chunk into a running (max, sum) once
// the chunk has landed.  A wait that runs out sets sm.abort (the data is then
// unspecified, but the CTA goes on so that the cluster's barriers match).
__device__ __forceinline__ void load_row_stats(Smem &sm, float4 *R4, const float *lrow, int cnt,
                                               int S4, int vec, bool bulk, uint64_t limit_ns,
                                               uint32_t parity) {
  using namespace sm100;
  const int t = threadIdx.x;
  float m_t = -INFINITY, s_t = 0.f;
  if (bulk) {
    const int cnt4 = cnt >> 2;  // cnt is a multiple of 4 on this path
    for (int k = cnt4 + t; k < S4; k += kST)
      R4[k] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (t == 0) {
#pragma unroll
      for (int j = 0; j < kChunks; ++j) {
        const int b0 = cnt4 * j / kChunks, b1 = cnt4 * (j + 1) / kChunks;
        const uint32_t bar = smem_addr(&sm.bar[j]);
        mbar_arrive_expect_tx(bar, (uint32_t)(b1 - b0) * 16u);
        if (b1 > b0) bulk_load(smem_addr(R4 + b0), lrow + 4 * b0, (uint32_t)(b1 - b0) * 16u, bar);
      }
    }
    for (int j = 0; j < kChunks; ++j) {
      const int b0 = cnt4 * j / kChunks, b1 = cnt4 * (j + 1) / kChunks;
      if (!mbar_wait(smem_addr(&sm.bar[j]), parity, limit_ns)) sm.abort = 1;
      for (int k0 = b0 + t; k0 < b1; k0 += 4 * kST) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = k0 + u * kST;
          v[u] = k < b1 ? R4[k] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        stats_group(v, m_t, s_t);
      }
    }
  } else {
    for (int k0 = t; k0 < S4; k0 += kSBatch * kST) {
      float4 v[kSBatch];
#pragma unroll
      for (int u = 0; u < kSBatch; ++u) {
        const int k = k0 + u * kST;
        v[u] = k < S4 ? load_slice4(lrow, k, cnt, vec, -INFINITY)
                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < kSBatch; ++u) {
        const int k = k0 + u * kST;
        if (k < S4) R4[k] = v[u];
      }
      stats_group(v, m_t, s_t);
    }
  }
  block_ms(sm, m_t, s_t);  // its barrier also orders every R4 write before later reads
  if (t == 0) {
    sm.mine.m = m_t;
    sm.mine.s = s_t;
  }
}

// Cluster exchange of round r.  Every CTA pushes sm.mine into slot
// [r & 1][its rank] of every CTA of the cluster (its own included), then the
// cluster barrier; afterwards warp 0 reads its local slots and derives,
// identically in every CTA: the global max (first round), the per-CTA
// totals in global units (sm.T), the normaliser Z (their sum in CTA order)
// and the published weight of CTA `o` (o < 0: none).  The slots of round r
// are written again in round r + 2 only, by CTAs that have passed round
// r + 1's barrier, which every CTA reaches after reading round r's slots.
__device__ __forceinline__ void exchange(Smem &sm, int r, bool first, int C, int o) {
  using namespace sm100;
  const int t = threadIdx.x, lane = t & 31;
  __syncthreads();  // sm.mine is complete
  if (t < C) {
    const Slot v = sm.mine;
    st_dsmem_f4(smem_addr(&sm.slot[r & 1][cluster_ctarank()]), (uint32_t)t,
                make_float4(v.m, v.s, v.pub, 0.f));
  }
  cluster_arrive();
  cluster_wait();
  if (t < 32) {
    float4 sl = make_float4(-INFINITY, 0.f, 0.f, 0.f);
    if (lane < C) {
      const Slot &x = sm.slot[r & 1][lane];
      sl = make_float4(x.m, x.s, x.pub, 0.f);
    }
    float m = sm.ctl.m;
    float T = sl.y;
    if (first) {
      m = sl.x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      T = sl.x == -INFINITY ? 0.f : sl.y * ex2_approx((sl.x - m) * kLog2e);
    }
    float Z = 0.f;
#pragma unroll
    for (int l = 0; l < kMaxCluster; ++l) {
      const float v = __shfl_sync(0xffffffffu, T, l);
      if (l < C) Z += v;
    }
    const float pv = __shfl_sync(0xffffffffu, sl.z, o < 0 ? 0 : o);
    if (lane < C) sm.T[lane] = T;
    if (lane == 0) {
      sm.ctl.m = m;
      sm.ctl.Z = Z;
      sm.ctl.pub = pv;
    }
  }
  __syncthreads();
}

// The CTA holding an inverse-CDF draw with target tau (global units), from
// per-CTA totals sm.T in CTA order (thread 0 only).  When rounding leaves no
// crossing: the last CTA of positive total, in fallback mode.
__device__ __forceinline__ void find_owner(Smem &sm, int C, float tau) {
  float acc = 0.f, tl = 0.f;
  int cs = -1, last_pos = -1;
  for (int l = 0; l < C; ++l) {
    if (sm.T[l] > 0.f) last_pos = l;
    if (cs < 0 && acc + sm.T[l] > tau) {
      cs = l;
      tl = tau - acc;
    }
    acc += sm.T[l];
  }
  sm.ctl.fallback = cs < 0;
  sm.ctl.cstar = cs < 0 ? max(last_pos, 0) : cs;
  sm.ctl.tau = tl;
}

// Inverse-CDF search of one slice for target tl (or, in fallback mode, the
// last element of positive weight); returns lo + the element index.  Thread
// t owns the float4s [t*P, t*P + P) in token order: each thread sums its
// range (visited in a rotated order, so that the 16-byte shared loads of a
// quarter warp fall in distinct banks), one block scan finds the thread whose
// range holds the crossing, and that thread walks its range.  Weights:
// exp(x - m) of raw logits (level0, ml2 = m log2 e) or the stored values.
__device__ __forceinline__ int search_slice(Smem &sm, const float4 *R4, int S4, int lo,
                                             bool level0, float ml2, float tl, bool fb) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  auto weight = [&](float4 w) { return level0 ? exp4(w, ml2) : w; };
  const int P = (S4 + kST - 1) / kST;
  const int k0 = t * P;
  const int n = max(0, min(P, S4 - k0));
  // the range's sum, and its last float4 of positive sum (weights are >= 0)
  float s = 0.f;
  int lastk = -1;
  {
    int ii = t % P;
    for (int i = 0; i < P; ++i, ++ii) {
      if (ii == P) ii = 0;
      if (ii < n) {
        const float s4 = sum4(weight(R4[k0 + ii]));
        s += s4;
        lastk = s4 > 0.f ? max(lastk, k0 + ii) : lastk;
      }
    }
  }
  // inclusive scan of the range sums in thread (= token) order
  float incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sm.wg[warp] = incl;
  __syncthreads();
  float wbase = 0.f;
  for (int ww = 0; ww < warp; ++ww) wbase += sm.wg[ww];
  incl += wbase;
  int cand = INT_MAX;
  if (!fb && n > 0 && incl > tl) {
    // the first positive element whose running sum passes the target;
    // rounding may leave none inside this range: then its last positive
    float a = incl - s;
    int lastp = -1;
    for (int i = 0; i < n && cand == INT_MAX; ++i) {
      const float4 w = weight(R4[k0 + i]);
      const float e4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a += e4[e];
        if (e4[e] > 0.f) {
          lastp = 4 * (k0 + i) + e;
          if (cand == INT_MAX && a > tl) cand = lastp;
        }
      }
    }
    if (cand == INT_MAX && lastp >= 0) cand = lastp;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, off));
    lastk = max(lastk, __shfl_xor_sync(0xffffffffu, lastk, off));
  }
  if (lane == 0) {
    sm.wi[warp] = cand;
    sm.wj[warp] = lastk;
  }
  __syncthreads();
  if (t == 0) {
    int best = INT_MAX, lk = -1;
    for (int ww = 0; ww < kSW; ++ww) {
      best = min(best, sm.wi[ww]);
      lk = max(lk, sm.wj[ww]);
    }
    int e = best;
    if (best == INT_MAX) {
      // no crossing: the slice's last element of positive weight
      e = -1;
      if (lk >= 0) {
        const float4 w = weight(R4[lk]);
        e = w.w > 0.f ? 4 * lk + 3 : w.z > 0.f ? 4 * lk + 2 : w.y > 0.f ? 4 * lk + 1 : 4 * lk;
      }
    }
    sm.ctl.tok = e < 0 ? -1 : lo + e;
  }
  __syncthreads();
  return sm.ctl.tok;
}

// Ticket with release (this thread's earlier stores) and acquire semantics.
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned *p) {
  unsigned r;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;\n" : "=r"(r) : "l"(p) : "memory");
  return r;
}

// Before leaving: a CTA whose copy wait ran out waits (bounded) once more for
// the copies it issued, then reports the timeout.
__device__ __forceinline__ void drain_bulk(Smem &sm, bool issued, uint64_t limit_ns,
                                           int32_t *status, uint32_t parity) {
  using namespace sm100;
  if (threadIdx.x == 0 && issued && sm.abort) {
    for (int j = 0; j < kChunks; ++j) mbar_wait(smem_addr(&sm.bar[j]), parity, limit_ns);
    if (status) atomicOr(status, TSD_STATUS_TIMEOUT);
  }
}

struct Args {
  const float *logits, *qd;
  const int32_t *tokens, *parent, *n_nodes, *err;
  const float *u_accept, *u_draw;
  int N_max, V, S, vec, bulk, D_max;
  uint64_t limit_ns;
  int32_t *next, *draw, *accept_len, *leaf, *path, *bonus;
  unsigned *counter;
  int32_t *status;
};

// The CTA that took sequence b's last ticket (all its threads): walk the
// accepted children from the root and write the walk.  Returns the last node
// when it still needs its draw (a leaf), else -1 (the bonus is then written).
// Every node's results were released before its ticket, and this CTA's
// ticket acquired them.
__device__ int walk_sequence(const Args &a, int b, int nb) {
  __shared__ int s_next[kMaxNodes], s_draw[kMaxNodes];
  __shared__ int s_path[kMaxDepth + 1];
  __shared__ int s_walk[2];
  const int t = threadIdx.x;
  const int N_max = a.N_max;
  __threadfence();
  if (t < nb) {
    s_next[t] = __ldcg(a.next + (size_t)b * N_max + t);
    s_draw[t] = __ldcg(a.draw + (size_t)b * N_max + t);
  }
  __syncthreads();
  if (t == 0) {
    a.counter[b] = 0u;  // zero again for the next call
    int f = 0, A = 0;
    s_path[0] = 1;
    while (A < a.D_max && s_next[f] >= 0) {
      f = s_next[f];
      s_path[++A] = f + 1;
    }
    a.accept_len[b] = A;
    a.leaf[b] = f;
    s_walk[0] = A;
    s_walk[1] = f;
    const bool drawn = s_draw[f] >= 0 || s_next[f] >= 0;
    if (drawn) a.bonus[b] = s_draw[f];
    s_walk[1] = drawn ? -1 : f;
  }
  __syncthreads();
  const int A = s_walk[0];
  for (int k = t; k <= a.D_max; k += kST)
    a.path[(size_t)b * (a.D_max + 1) + k] = k <= A ? s_path[k] : 0;
  const int f = s_walk[1];
  __syncthreads();
  return f;
}

// Round r of the cluster: every CTA learns the leaf (if any) that needs the
// bonus draw, from whichever CTA walked the sequence (one at most).
__device__ __forceinline__ int cluster_leaf_flag(Smem &sm, int r, int C, int mine) {
  using namespace sm100;
  __syncthreads();
  if ((int)threadIdx.x < C)
    st_dsmem_f4(smem_addr(&sm.slot[r & 1][cluster_ctarank()]), threadIdx.x,
                make_float4(__int_as_float(mine), 0.f, 0.f, 0.f));
  cluster_arrive();
  cluster_wait();
  int f = -1;
  for (int l = 0; l < C; ++l) f = max(f, __float_as_int(sm.slot[r & 1][l].m));
  return f;
}

// All CTAs of the cluster: the bonus token of sequence b drawn from the
// target distribution of leaf f (rounds r and r + 1 of the cluster; the
// row copy waits on barrier phase `parity`).
__device__ void leaf_draw(const Args &a, Smem &sm, float4 *R4, int b, int f, int C, int c, int r,
                          uint32_t parity) {
  const size_t row = (size_t)b * a.N_max + f;
  const int lo = c * a.S;
  const int cnt = max(0, min(a.S, a.V - lo));
  const int S4 = a.S >> 2;
  const bool bulk = a.bulk != 0;
  load_row_stats(sm, R4, a.logits + row * (size_t)a.V + lo, cnt, S4, a.vec, bulk, a.limit_ns,
                 parity);
  if (threadIdx.x == 0) sm.mine.pub = 0.f;
  exchange(sm, r, true, C, -1);
  if (threadIdx.x == 0) find_owner(sm, C, __fmul_rn(a.u_draw[row], sm.ctl.Z));
  __syncthreads();
  if (sm.ctl.cstar == c) {
    const int tok = search_slice(sm, R4, S4, lo, true, sm.ctl.m * kLog2e, sm.ctl.tau,
                                 sm.ctl.fallback != 0);
    if (threadIdx.x == 0) {
      a.draw[row] = tok;
      a.bonus[b] = tok;
    }
  }
  drain_bulk(sm, bulk, a.limit_ns, a.status, parity);
  // the exchange's barrier was the last access to another CTA's shared memory
}

__global__ void __launch_bounds__(kST, 3) verify_stochastic_kernel(const Args a) {
  using namespace sm100;
  extern __shared__ float4 R4[];  // this CTA's slice: raw logits, then residual weights
  __shared__ Smem sm;
  __shared__ int s_kid[kMaxNodes], s_ktok[kMaxNodes];
  __shared__ float s_ku[kMaxNodes], s_kq[kMaxNodes];
  __shared__ int s_wcnt[kSW];
  __shared__ int s_last;

  pdl_trigger();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int C = (int)cluster_nctarank(), c = (int)cluster_ctarank();
  const int i = blockIdx.y, b = blockIdx.z;
  const int N_max = a.N_max, V = a.V, S = a.S;
  const size_t row = (size_t)b * N_max + i;
  pdl_wait();

  const int nb = a.n_nodes ? a.n_nodes[b] : N_max;
  const bool seq_ok = a.err[b] == 0 && nb >= 1 && nb <= N_max;
  if (!seq_ok || i >= nb) {  // the whole cluster leaves here: same inputs
    if (c == 0) {
      if (t == 0) {
        a.next[row] = -1;
        a.draw[row] = -1;
      }
      if (!seq_ok && i == 0) {
        for (int k = t; k <= a.D_max; k += kST) a.path[(size_t)b * (a.D_max + 1) + k] = 0;
        if (t == 0) {
          a.accept_len[b] = 0;
          a.leaf[b] = -1;
          a.bonus[b] = -1;
        }
      }
    }
    return;
  }

  // ---- children of node i in increasing id order (tokens outside [0, V)
  //      are skipped), with their uniforms and draft probabilities ----
  int nk;
  {
    int is_kid = 0, tok = 0;
    if (t >= 1 && t < nb) {
      tok = a.tokens[(size_t)b * N_max + t];
      is_kid = a.parent[(size_t)b * N_max + t] == i && tok >= 0 && tok < V;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, is_kid);
    if (lane == 0) s_wcnt[warp] = __popc(bal);
    __syncthreads();
    int base = 0;
    nk = 0;
#pragma unroll
    for (int w = 0; w < kSW; ++w) {
      base += w < warp ? s_wcnt[w] : 0;
      nk += s_wcnt[w];
    }
    if (is_kid) {
      const int pos = base + __popc(bal & ((1u << lane) - 1u));
      s_kid[pos] = t;
      s_ktok[pos] = tok;
      s_ku[pos] = a.u_accept[(size_t)b * N_max + t];
      s_kq[pos] = a.qd[row * (size_t)V + tok];
    }
  }
  const int lo = c * S;
  const int cnt = max(0, min(S, V - lo));
  const int S4 = S >> 2;
  const bool bulk = a.bulk != 0;
  init_bars(sm);  // also publishes the child list
  int round = 0;
  int outcome = -1, tok = -1, settle = 0;

  if (nk > 0) {
    // ---- an internal node: target row, then its children in order; after
    //      each rejection the residual max(0, r - q) replaces the weights ----
    const float *lrow = a.logits + row * (size_t)V + lo;
    const float *qrow = a.qd + row * (size_t)V + lo;
    const float *R = reinterpret_cast<const float *>(R4);
    auto owner = [&](int j) { return j < nk ? s_ktok[j] / S : -1; };

    load_row_stats(sm, R4, lrow, cnt, S4, a.vec, bulk, a.limit_ns, 0);
    if (t == 0) sm.mine.pub = owner(0) == c ? R[s_ktok[0] - lo] : 0.f;
    bool level0 = true;
    exchange(sm, round++, true, C, owner(0));
    for (int j = 0; j < nk; ++j) {
      {
        // child j against the current weights: u * q(x) < w(x) / Z
        const float w = level0 ? exp_shift(sm.ctl.pub, sm.ctl.m * kLog2e) : sm.ctl.pub;
        if (__fmul_rn(s_ku[j], s_kq[j]) < __fdiv_rn(w, sm.ctl.Z)) {
          outcome = s_kid[j];
          break;
        }
      }
      const float ml2 = sm.ctl.m * kLog2e;
      const float invZ = __frcp_rn(sm.ctl.Z);
      float acc = 0.f;
      for (int k0 = t; k0 < S4; k0 += kSBatch * kST) {
        float4 qv[kSBatch];
#pragma unroll
        for (int u = 0; u < kSBatch; ++u) {
          const int k = k0 + u * kST;
          qv[u] = k < S4 ? load_slice4(qrow, k, cnt, a.vec, 0.f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kSBatch; ++u) {
          const int k = k0 + u * kST;
          if (k < S4) {
            float4 w = R4[k];
            if (level0) w = exp4(w, ml2);
            w.x = fmaxf(0.f, fmaf(w.x, invZ, -qv[u].x));
            w.y = fmaxf(0.f, fmaf(w.y, invZ, -qv[u].y));
            w.z = fmaxf(0.f, fmaf(w.z, invZ, -qv[u].z));
            w.w = fmaxf(0.f, fmaf(w.w, invZ, -qv[u].w));
            R4[k] = w;
            acc += sum4(w);
          }
        }
      }
      level0 = false;
      float tot = block_sum(acc, sm.wf);  // also orders the R4 writes before the read below
      if (t == 0) {
        sm.mine.s = tot;
        sm.mine.pub = owner(j + 1) == c ? R[s_ktok[j + 1] - lo] : 0.f;
      }
      exchange(sm, round++, false, C, owner(j + 1));
      if (!(sm.ctl.Z > 0.f)) {
        // no residual mass: r equalled q, and the residual is taken to be q
        float a2 = 0.f;
        for (int k = t; k < S4; k += kST) {
          const float4 w = load_slice4(qrow, k, cnt, a.vec, 0.f);
          R4[k] = w;
          a2 += sum4(w);
        }
        tot = block_sum(a2, sm.wf);
        if (t == 0) {
          sm.mine.s = tot;
          sm.mine.pub = owner(j + 1) == c ? R[s_ktok[j + 1] - lo] : 0.f;
        }
        exchange(sm, round++, false, C, owner(j + 1));
      }
    }
    if (outcome < 0) {
      // every child rejected: draw from the residual
      if (t == 0) find_owner(sm, C, __fmul_rn(a.u_draw[row], sm.ctl.Z));
      __syncthreads();
      settle = sm.ctl.cstar;
      if (settle == c)
        tok = search_slice(sm, R4, S4, lo, false, 0.f, sm.ctl.tau, sm.ctl.fallback != 0);
    }
    drain_bulk(sm, bulk, a.limit_ns, a.status, 0);
  }

  // ---- the settling CTA records the node and takes a ticket; the one with
  //      the sequence's last ticket walks the tree ----
  int need = -1;
  if (settle == c) {
    if (t == 0) {
      a.next[row] = outcome;
      a.draw[row] = outcome >= 0 ? -1 : tok;
      s_last = ticket_acq_rel(&a.counter[b]) == (unsigned)(nb - 1);
    }
    __syncthreads();
    if (s_last) need = walk_sequence(a, b, nb);
  }
  // ---- a walk that ended at a leaf: this cluster draws the bonus token ----
  const int f = cluster_leaf_flag(sm, round++, C, need);
  if (f >= 0) leaf_draw(a, sm, R4, b, f, C, c, round, nk > 0 ? 1u : 0u);
}

struct StochPlan {
  int C;        // CTAs per node (cluster size)
  int S;        // floats of the row per CTA
  size_t smem;  // dynamic shared memory per CTA
};

// Clusters of size C with `smem` bytes per CTA that fit on the device at once
// (cached per device and shape).
int resident_clusters(int C, size_t smem) {
  struct Entry {
    int dev, C;
    size_t smem;
    int n;
  };
  static Entry cache[64];
  static int used = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int e = 0; e < used; ++e)
    if (cache[e].dev == dev && cache[e].C == C && cache[e].smem == smem) return cache[e].n;
  if (!set_smem(reinterpret_cast<const void *>(verify_stochastic_kernel), (size_t)kMaxS * 4))
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, 1, 1);
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_stochastic_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (used < 64) cache[used++] = {dev, C, smem, n};
  return n;
}

// Cluster size: the fewest waves of node clusters times the per-CTA row
// length (plus a fixed per-node cost), over the portable sizes.
bool plan_stochastic(int B, int N_max, int V, StochPlan *out) {
  const long rows = (long)B * N_max;
  double best = 0.0;
  bool found = false;
  for (int C = 1; C <= kMaxCluster; ++C) {
    const int S = (int)align_up((size_t)((V + C - 1) / C), 4);
    if (S > kMaxS) continue;
    const size_t smem = (size_t)S * 4;
    const int n = resident_clusters(C, smem);
    if (n <= 0) continue;
    const long waves = (rows + n - 1) / n;
    const double cost = (double)waves * ((double)S + 4096.0);
    if (!found || cost < best) {
      best = cost;
      *out = {C, S, smem};
      found = true;
    }
  }
  return found;
}

bool disjoint(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return true;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x + na <= y || y + nb <= x;
}

size_t counter_bytes(int B) { return align_up(sizeof(unsigned) * (size_t)B, 256); }

}  // namespace
}  // namespace tsd

TSD_API size_t tsd_tree_verify_stochastic_workspace_bytes(int B, int N_max, int V) {
  (void)N_max;
  (void)V;
  if (B <= 0) return 0;
  return tsd::counter_bytes(B);
}

TSD_API int tsd_tree_verify_stochastic(const float *logits, const float *q_draft,
                                       const int32_t *tokens, const int32_t *parent,
                                       const int32_t *n_nodes, const int32_t *err,
                                       const float *u_accept, const float *u_draw, int B,
                                       int N_max, int V, int D_max, int32_t *next, int32_t *draw,
                                       int32_t *accept_len, int32_t *leaf, int32_t *path,
                                       int32_t *bonus, void *workspace, size_t ws_bytes,
                                       int32_t *status, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0 || V < 1) return B < 0 ? TSD_ERR_ARG : TSD_ERR_LIMIT;
  if (N_max < 1 || N_max > kMaxNodes || D_max < 0 || D_max > kMaxDepth || B > 65535 ||
      V > kMaxCluster * kMaxS)
    return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!logits || !q_draft || !tokens || !parent || !err || !u_accept || !u_draw || !next ||
      !draw || !accept_len || !leaf || !path || !bonus)
    return TSD_ERR_ARG;
  const size_t ws_need = tsd_tree_verify_stochastic_workspace_bytes(B, N_max, V);
  if (!workspace || ws_bytes < ws_need || !aligned(workspace, 16)) return TSD_ERR_WORKSPACE;
  // outputs may not overlap any input: every CTA of a node's cluster reads
  // the inputs itself and must see the same values
  const size_t rows = (size_t)B * N_max;
  const size_t big = rows * (size_t)V * 4, small = rows * 4, seq = (size_t)B * 4;
  const void *in[8] = {logits, q_draft, tokens, parent, n_nodes, err, u_accept, u_draw};
  const size_t in_n[8] = {big, big, small, small, n_nodes ? seq : 0, seq, small, small};
  const void *outp[8] = {next, draw, accept_len, leaf, path, bonus, workspace, status};
  const size_t out_n[8] = {small, small, seq, seq, (size_t)B * (D_max + 1) * 4, seq, ws_need,
                           status ? 4u : 0u};
  for (int o = 0; o < 8; ++o)
    for (int k = 0; k < 8; ++k)
      if (!disjoint(outp[o], out_n[o], in[k], in_n[k])) return TSD_ERR_ARG;
  StochPlan p;
  if (!plan_stochastic(B, N_max, V, &p)) return TSD_ERR_CUDA;

  Args a;
  a.logits = logits;
  a.qd = q_draft;
  a.tokens = tokens;
  a.parent = parent;
  a.n_nodes = n_nodes;
  a.err = err;
  a.u_accept = u_accept;
  a.u_draw = u_draw;
  a.N_max = N_max;
  a.V = V;
  a.S = p.S;
  a.vec = (V % 4 == 0) && aligned(logits, 16) && aligned(q_draft, 16);
  a.bulk = a.vec;  // bulk copies: 16-byte aligned rows and slices
  a.D_max = D_max;
  a.limit_ns = (uint64_t)option(TSD_OPT_WAIT_LIMIT_NS);
  a.next = next;
  a.draw = draw;
  a.accept_len = accept_len;
  a.leaf = leaf;
  a.path = path;
  a.bonus = bonus;
  a.counter = static_cast<unsigned *>(workspace);
  a.status = status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.C, N_max, B);
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = as_cuda(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, verify_stochastic_kernel, a) != cudaSuccess) return TSD_ERR_CUDA;
  return TSD_OK;
}

TSD_API int tsd_tree_verify_stochastic_plan(int B, int N_max, int V, int *cluster, int *slice) {
  tsd::StochPlan p;
  if (B < 1 || N_max < 1 || V < 1 || V > tsd::kMaxCluster * tsd::kMaxS) return TSD_ERR_LIMIT;
  if (!tsd::plan_stochastic(B, N_max, V, &p)) return TSD_ERR_CUDA;
  if (cluster) *cluster = p.C;
  if (slice) *slice = p.S;
  return TSD_OK;
}
