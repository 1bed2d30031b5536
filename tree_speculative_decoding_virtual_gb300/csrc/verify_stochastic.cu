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
// rejected (or i is a leaf) node i draws its token from that residual.
//
// Every node is decided from its own target row, draft row, children and
// uniforms, so all nodes of all sequences run at once: one thread-block
// cluster of C CTAs per node, CTA c holding the slice [c*S, c*S + S) of the
// node's vocabulary row in shared memory.  The target row is read from HBM
// once (each thread keeps a running max and sum of exponentials while it
// stores its part); the draft row only when a child is rejected.  Per-CTA
// partial results (max, sum, the weight at the next child's token) are
// exchanged through distributed shared memory between cluster barriers, and
// every control decision is taken from those exchanged values with the same
// instructions in every CTA, so all CTAs of a cluster pass the same number
// of barriers.  The CTA that settles a node takes a per-sequence ticket; the
// one taking the last ticket walks the accepted children from the root.

#include <climits>
#include <cmath>

#include "sm100_ptx.cuh"
#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kST = 256;                    // threads per CTA (>= kMaxNodes)
constexpr int kSW = kST / 32;               // warps per CTA
constexpr int kSBatch = 8;                  // 16-byte loads in flight per thread
constexpr int kMaxJ = 32;                   // float4 rounds per thread
constexpr int kMaxS = 4 * kST * kMaxJ;      // floats per CTA slice (128 KB)
constexpr int kMaxCluster = 8;              // portable cluster size

struct __align__(16) Slot {
  float m;    // CTA max of the target logits (first exchange only)
  float s;    // CTA sum of the current weights
  float pub;  // weight (first exchange: raw logit) at the next child's token
  float pad;
};

struct Ctl {
  float m, Z;         // global max of the logits, normaliser of the current level
  int accept;         // decision for the current child
  int cstar;          // CTA holding the draw
  float tau;          // draw target inside that CTA, in its own units
  int fallback;       // no cumulative boundary exceeded the target: last positive
  int jstar;          // float4 round holding the draw (owner CTA)
  float tau_j;
};

__device__ __forceinline__ float sum4(const float4 &v) { return (v.x + v.y) + (v.z + v.w); }
__device__ __forceinline__ float max4(const float4 &v) {
  return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
}

// Element k (a float4 index) of a row slice holding `cnt` valid floats;
// entries past the end read as `fill`.
template <bool kStream>
__device__ __forceinline__ float4 load_slice4(const float *p, int k, int cnt, int vec, float fill) {
  const int e = 4 * k;
  if (vec && e + 4 <= cnt) {
    const float4 *p4 = reinterpret_cast<const float4 *>(p) + k;
    return kStream ? __ldcs(p4) : __ldcg(p4);
  }
  float4 r;
  r.x = e < cnt ? (kStream ? __ldcs(p + e) : __ldcg(p + e)) : fill;
  r.y = e + 1 < cnt ? (kStream ? __ldcs(p + e + 1) : __ldcg(p + e + 1)) : fill;
  r.z = e + 2 < cnt ? (kStream ? __ldcs(p + e + 2) : __ldcg(p + e + 2)) : fill;
  r.w = e + 3 < cnt ? (kStream ? __ldcs(p + e + 3) : __ldcg(p + e + 3)) : fill;
  return r;
}

// (m, s) <- merge of two (max, sum of exp(x - max)) pairs; -inf maxima carry
// no mass.
__device__ __forceinline__ void merge_ms(float &m, float &s, float mo, float so) {
  const float mn = fmaxf(m, mo);
  if (mn == -INFINITY) return;
  s = s * expf(m - mn) + so * expf(mo - mn);
  m = mn;
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

__global__ void __launch_bounds__(kST, 3)
verify_stochastic_kernel(const float *__restrict__ logits, const float *__restrict__ qd,
                         const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
                         const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ err,
                         const float *__restrict__ u_accept, const float *__restrict__ u_draw,
                         int N_max, int V, int S, int vec, int D_max,
                         int32_t *__restrict__ next_out, int32_t *__restrict__ draw_out,
                         int32_t *__restrict__ accept_len, int32_t *__restrict__ leaf_out,
                         int32_t *__restrict__ path, int32_t *__restrict__ bonus,
                         unsigned *__restrict__ counter) {
  using namespace sm100;
  extern __shared__ float4 R4[];  // this CTA's slice: raw logits, then residual weights
  __shared__ Slot s_slot[2];      // read by the other CTAs of the cluster
  __shared__ int s_kid[kMaxNodes], s_ktok[kMaxNodes];
  __shared__ float s_ku[kMaxNodes], s_kq[kMaxNodes];
  __shared__ int s_wcnt[kSW];
  __shared__ float s_wf[kSW], s_wg[kSW];
  __shared__ float s_T[kMaxCluster];  // per-CTA totals of the current level, global units
  __shared__ float s_rw[kMaxJ][kSW];
  __shared__ int s_wi[kSW];
  __shared__ Ctl s_ctl;
  __shared__ int s_next[kMaxNodes];
  __shared__ int s_path[kMaxDepth + 1];
  __shared__ bool s_last;

  pdl_trigger();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int C = (int)cluster_nctarank(), c = (int)cluster_ctarank();
  const int i = blockIdx.y, b = blockIdx.z;
  const size_t row = (size_t)b * N_max + i;
  pdl_wait();

  const int nb = n_nodes ? n_nodes[b] : N_max;
  const bool seq_ok = err[b] == 0 && nb >= 1 && nb <= N_max;
  if (!seq_ok || i >= nb) {  // the whole cluster leaves here: same inputs
    if (c == 0) {
      if (t == 0) {
        next_out[row] = -1;
        draw_out[row] = -1;
      }
      if (!seq_ok && i == 0) {
        for (int k = t; k <= D_max; k += kST) path[(size_t)b * (D_max + 1) + k] = 0;
        if (t == 0) {
          accept_len[b] = 0;
          leaf_out[b] = -1;
          bonus[b] = -1;
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
      tok = tokens[(size_t)b * N_max + t];
      is_kid = parent[(size_t)b * N_max + t] == i && tok >= 0 && tok < V;
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
      s_ku[pos] = u_accept[(size_t)b * N_max + t];
      s_kq[pos] = qd[row * (size_t)V + tok];
    }
  }

  const int lo = c * S;
  const int cnt = max(0, min(S, V - lo));
  const int S4 = S >> 2;
  const float *lrow = logits + row * (size_t)V + lo;
  const float *qrow = qd + row * (size_t)V + lo;

  // ---- pass 1: the target logits into shared memory, with this thread's
  //      running (max, sum of exp(x - max)) ----
  float m_t = -INFINITY, s_t = 0.f;
  for (int k0 = t; k0 < S4; k0 += kSBatch * kST) {
    float4 v[kSBatch];
#pragma unroll
    for (int u = 0; u < kSBatch; ++u) {
      const int k = k0 + u * kST;
      v[u] = k < S4 ? load_slice4<true>(lrow, k, cnt, vec, -INFINITY)
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    float bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kSBatch; ++u) {
      const int k = k0 + u * kST;
      if (k < S4) R4[k] = v[u];
      bm = fmaxf(bm, max4(v[u]));
    }
    const float mn = fmaxf(m_t, bm);
    if (mn != -INFINITY) {
      float acc = s_t * expf(m_t - mn);
#pragma unroll
      for (int u = 0; u < kSBatch; ++u)
        acc += (expf(v[u].x - mn) + expf(v[u].y - mn)) + (expf(v[u].z - mn) + expf(v[u].w - mn));
      s_t = acc;
      m_t = mn;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    merge_ms(m_t, s_t, __shfl_xor_sync(0xffffffffu, m_t, off),
             __shfl_xor_sync(0xffffffffu, s_t, off));
  if (lane == 0) {
    s_wf[warp] = m_t;
    s_wg[warp] = s_t;
  }
  __syncthreads();

  // token x of child j lives in CTA x / S
  auto owner = [&](int j) { return j < nk ? s_ktok[j] / S : -1; };
  const float *R = reinterpret_cast<const float *>(R4);

  if (t == 0) {
    float m = s_wf[0], s = s_wg[0];
    for (int w = 1; w < kSW; ++w) merge_ms(m, s, s_wf[w], s_wg[w]);
    Slot sl;
    sl.m = m;
    sl.s = s;
    sl.pub = owner(0) == c ? R[s_ktok[0] - lo] : 0.f;
    sl.pad = 0.f;
    s_slot[0] = sl;
  }

  // Cluster exchange of round `r` (slot r & 1), then the decision for child
  // j at this level.  `first`: the slots carry per-CTA (max, sum of exp);
  // the weight at x is exp(logit - m) / Z.  Warp 0 reads every CTA's slot and
  // computes the same values in every CTA; the others wait on the block
  // barrier.  A slot written in round r is overwritten in round r + 2 only,
  // after every CTA has passed round r + 1's barrier, i.e. finished reading.
  auto exchange = [&](int r, bool first, int j) {
    cluster_arrive();
    cluster_wait();
    if (warp == 0) {
      float4 sl = make_float4(-INFINITY, 0.f, 0.f, 0.f);
      if (lane < C) sl = ld_dsmem_f4(smem_addr(&s_slot[r & 1]), (uint32_t)lane);
      float m = s_ctl.m;
      float T = sl.y;
      if (first) {
        m = sl.x;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        T = sl.x == -INFINITY ? 0.f : sl.y * expf(sl.x - m);
      }
      float Z = 0.f;
#pragma unroll
      for (int l = 0; l < kMaxCluster; ++l) {
        const float v = __shfl_sync(0xffffffffu, T, l);
        if (l < C) Z += v;
      }
      const int o = owner(j);
      const float pub = __shfl_sync(0xffffffffu, sl.z, o < 0 ? 0 : o);
      if (lane < C) s_T[lane] = T;
      if (lane == 0) {
        s_ctl.m = m;
        s_ctl.Z = Z;
        int acc = 0;
        if (j < nk) {
          const float w = first ? expf(pub - m) : pub;
          acc = __fmul_rn(s_ku[j], s_kq[j]) < __fdiv_rn(w, Z);
        }
        s_ctl.accept = acc;
      }
    }
    __syncthreads();
  };

  int round = 0;
  exchange(round++, true, 0);
  bool level0 = true;
  int outcome = -1;

  // ---- children in order; after each rejection the residual
  //      max(0, r - q) replaces the weights ----
  for (int j = 0; j < nk; ++j) {
    if (s_ctl.accept) {
      outcome = s_kid[j];
      break;
    }
    const float m = s_ctl.m;
    const float invZ = __frcp_rn(s_ctl.Z);
    float acc = 0.f;
    for (int k0 = t; k0 < S4; k0 += kSBatch * kST) {
      float4 qv[kSBatch];
#pragma unroll
      for (int u = 0; u < kSBatch; ++u) {
        const int k = k0 + u * kST;
        qv[u] = k < S4 ? load_slice4<false>(qrow, k, cnt, vec, 0.f) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kSBatch; ++u) {
        const int k = k0 + u * kST;
        if (k < S4) {
          float4 w = R4[k];
          if (level0) {
            w.x = expf(w.x - m);
            w.y = expf(w.y - m);
            w.z = expf(w.z - m);
            w.w = expf(w.w - m);
          }
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
    float tot = block_sum(acc, s_wf);  // also orders the R4 writes before the read below
    if (t == 0) {
      Slot sl;
      sl.m = 0.f;
      sl.s = tot;
      sl.pub = owner(j + 1) == c ? R[s_ktok[j + 1] - lo] : 0.f;
      sl.pad = 0.f;
      s_slot[round & 1] = sl;
    }
    exchange(round++, false, j + 1);
    if (!(s_ctl.Z > 0.f)) {
      // no residual mass: r equalled q, and the residual is taken to be q
      float a2 = 0.f;
      for (int k = t; k < S4; k += kST) {
        const float4 w = load_slice4<false>(qrow, k, cnt, vec, 0.f);
        R4[k] = w;
        a2 += sum4(w);
      }
      tot = block_sum(a2, s_wf);
      if (t == 0) {
        Slot sl;
        sl.m = 0.f;
        sl.s = tot;
        sl.pub = owner(j + 1) == c ? R[s_ktok[j + 1] - lo] : 0.f;
        sl.pad = 0.f;
        s_slot[round & 1] = sl;
      }
      exchange(round++, false, j + 1);
    }
  }

  // every remote read of this cluster is done: arrive at the exit barrier now,
  // wait for the others only before leaving
  cluster_arrive();

  int settle = -1;  // the CTA that writes the node's result and takes the ticket
  int tok = -1;
  if (outcome >= 0) {
    settle = 0;
  } else {
    // ---- draw from the current weights by inverse CDF in token order ----
    const float Z = s_ctl.Z;
    const float m = s_ctl.m;
    if (t == 0) {
      const float tau = __fmul_rn(u_draw[row], Z);
      float acc = 0.f;
      int cs = -1, last_pos = -1;
      float tl = 0.f;
      for (int l = 0; l < C; ++l) {
        if (s_T[l] > 0.f) last_pos = l;
        if (cs < 0 && acc + s_T[l] > tau) {
          cs = l;
          tl = tau - acc;
        }
        acc += s_T[l];
      }
      s_ctl.fallback = cs < 0;
      if (cs < 0) cs = max(last_pos, 0);
      s_ctl.cstar = cs;
      // in the owner's own units: the first level's weights are exp(x - m)
      // there as well, so no rescale is needed
      s_ctl.tau = tl;
    }
    __syncthreads();
    settle = s_ctl.cstar;
    if (settle == c) {
      const bool fb0 = s_ctl.fallback;
      const float tau = s_ctl.tau;
      auto weight = [&](float4 w) {
        if (level0) {
          w.x = expf(w.x - m);
          w.y = expf(w.y - m);
          w.z = expf(w.z - m);
          w.w = expf(w.w - m);
        }
        return w;
      };
      // totals of every float4 round (round jr = float4 indices [jr*kST, jr*kST + kST))
      const int J = (S4 + kST - 1) / kST;
      for (int jr = 0; jr < J; ++jr) {
        const int k = jr * kST + t;
        float s = k < S4 ? sum4(weight(R4[k])) : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) s_rw[jr][warp] = s;
      }
      __syncthreads();
      if (t == 0) {
        float acc = 0.f;
        int js = -1, last_pos = -1;
        float tj = 0.f;
        for (int jr = 0; jr < J; ++jr) {
          float rt = 0.f;
          for (int w = 0; w < kSW; ++w) rt += s_rw[jr][w];
          if (rt > 0.f) last_pos = jr;
          if (!fb0 && js < 0 && acc + rt > tau) {
            js = jr;
            tj = tau - acc;
          }
          acc += rt;
        }
        s_ctl.fallback = fb0 || js < 0;
        s_ctl.jstar = js < 0 ? max(last_pos, 0) : js;
        s_ctl.tau_j = tj;
      }
      __syncthreads();
      const bool fb = s_ctl.fallback;
      const int k = s_ctl.jstar * kST + t;
      const float4 w = k < S4 ? weight(R4[k]) : make_float4(0.f, 0.f, 0.f, 0.f);
      // inclusive scan of the float4 sums over the round, in thread order
      const float s = sum4(w);
      float incl = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (lane == 31) s_wg[warp] = incl;
      __syncthreads();
      float wbase = 0.f;
      for (int ww = 0; ww < warp; ++ww) wbase += s_wg[ww];
      incl += wbase;
      const float excl = incl - s;
      int cand = INT_MAX;
      if (!fb && incl > s_ctl.tau_j) {
        // first element whose running sum passes the target; rounding may
        // leave none inside this float4, then its last positive element
        const float tj = s_ctl.tau_j;
        float a = excl;
        const float e4[4] = {w.x, w.y, w.z, w.w};
        int pick = -1, lastp = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          a += e4[e];
          if (e4[e] > 0.f) lastp = e;
          if (pick < 0 && e4[e] > 0.f && a > tj) pick = e;
        }
        if (pick < 0) pick = lastp;
        if (pick >= 0) cand = k * 4 + pick;
      }
      // fallback candidate: the round's last element of positive weight
      int lastpos = -1;
      if (w.w > 0.f) lastpos = k * 4 + 3;
      else if (w.z > 0.f) lastpos = k * 4 + 2;
      else if (w.y > 0.f) lastpos = k * 4 + 1;
      else if (w.x > 0.f) lastpos = k * 4;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, off));
        lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
      }
      if (lane == 0) {
        s_wcnt[warp] = cand;
        s_wi[warp] = lastpos;
      }
      __syncthreads();
      if (t == 0) {
        int best = INT_MAX, lp = -1;
        for (int ww = 0; ww < kSW; ++ww) {
          best = min(best, s_wcnt[ww]);
          lp = max(lp, s_wi[ww]);
        }
        const int e = best != INT_MAX ? best : lp;
        s_wcnt[0] = e < 0 ? -1 : lo + e;
      }
      __syncthreads();
      tok = s_wcnt[0];
    }
  }

  // ---- the settling CTA records the node and takes the sequence's ticket ----
  if (settle == c) {
    if (t == 0) {
      next_out[row] = outcome;
      draw_out[row] = outcome >= 0 ? -1 : tok;
      __threadfence();
      const unsigned ticket = atomicAdd(&counter[b], 1u);
      s_last = ticket == (unsigned)(nb - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (t < nb) s_next[t] = __ldcg(next_out + (size_t)b * N_max + t);
      __syncthreads();
      if (t == 0) {
        counter[b] = 0u;  // zero again for the next call
        int f = 0, A = 0;
        s_path[0] = 1;
        while (A < D_max && s_next[f] >= 0) {
          f = s_next[f];
          s_path[++A] = f + 1;
        }
        accept_len[b] = A;
        leaf_out[b] = f;
        bonus[b] = __ldcg(draw_out + (size_t)b * N_max + f);
        s_wcnt[0] = A;
      }
      __syncthreads();
      const int A = s_wcnt[0];
      for (int k = t; k <= D_max; k += kST) path[(size_t)b * (D_max + 1) + k] = k <= A ? s_path[k] : 0;
    }
  }
  cluster_wait();
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

}  // namespace
}  // namespace tsd

TSD_API size_t tsd_tree_verify_stochastic_workspace_bytes(int B, int N_max, int V) {
  (void)N_max;
  (void)V;
  if (B <= 0) return 0;
  return tsd::align_up(sizeof(unsigned) * (size_t)B, 256);
}

TSD_API int tsd_tree_verify_stochastic(const float *logits, const float *q_draft,
                                       const int32_t *tokens, const int32_t *parent,
                                       const int32_t *n_nodes, const int32_t *err,
                                       const float *u_accept, const float *u_draw, int B,
                                       int N_max, int V, int D_max, int32_t *next, int32_t *draw,
                                       int32_t *accept_len, int32_t *leaf, int32_t *path,
                                       int32_t *bonus, void *workspace, size_t ws_bytes,
                                       tsd_stream_t stream) {
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
  const void *outp[7] = {next, draw, accept_len, leaf, path, bonus, workspace};
  const size_t out_n[7] = {small, small, seq, seq, (size_t)B * (D_max + 1) * 4, seq, ws_need};
  for (int o = 0; o < 7; ++o)
    for (int k = 0; k < 8; ++k)
      if (!disjoint(outp[o], out_n[o], in[k], in_n[k])) return TSD_ERR_ARG;
  StochPlan p;
  if (!plan_stochastic(B, N_max, V, &p)) return TSD_ERR_CUDA;
  const int vec = (V % 4 == 0) && aligned(logits, 16) && aligned(q_draft, 16);

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
  if (cudaLaunchKernelEx(&cfg, verify_stochastic_kernel, logits, q_draft, tokens, parent, n_nodes,
                         err, u_accept, u_draw, N_max, V, p.S, vec, D_max, next, draw, accept_len,
                         leaf, path, bonus, static_cast<unsigned *>(workspace)) != cudaSuccess)
    return TSD_ERR_CUDA;
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
