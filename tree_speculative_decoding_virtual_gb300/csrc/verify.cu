// a3: greedy verification of a draft tree.
//
// "Speculative Decoding Hierárquico: Medusa, EAGLE-2 e Multi-Token
// Prediction", Medusa section: the target evaluates all branches in one
// parallel pass and the longest valid path is kept.  Greedy acceptance: a
// draft token is accepted when it equals the target's most likely token at
// its parent, and its parent was accepted.
//
// One fused launch.  Grid (chunk, node, sequence): each block scans one
// chunk of one logits row with 16-byte streaming loads and writes its
// (max, first index) partial.  The block that retires a sequence's last
// chunk (ticket counter per sequence, no waiting) reduces the partials of
// every row, evaluates acceptance with the ancestor bitmasks, and writes
// leaf / accept_len / path / bonus.  The counter is reset by that block, so
// the workspace is zero again when the launch ends.

#include <climits>
#include <cmath>

#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;  // independent 16-byte loads in flight per thread

struct Partial {
  float v;
  int idx;
};

// (v, i) beats (bv, bi): larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }

__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

__global__ void __launch_bounds__(kThreads)
verify_greedy_kernel(const float *__restrict__ logits, const int32_t *__restrict__ tokens,
                     const int32_t *__restrict__ parent, const int32_t *__restrict__ anc,
                     const int32_t *__restrict__ depth, const uint32_t *__restrict__ mask,
                     const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ err,
                     int N_max, int V, int D_max, int W, int chunk, int C, int vec_ok,
                     int32_t *__restrict__ argmax_out, int32_t *__restrict__ accept_len,
                     int32_t *__restrict__ leaf_out, int32_t *__restrict__ path,
                     int32_t *__restrict__ bonus, Partial *__restrict__ part,
                     unsigned *__restrict__ counter) {
  pdl_trigger();
  const int c = blockIdx.x;
  const int i = blockIdx.y;
  const int b = blockIdx.z;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int warp = t >> 5;
  {
    // while the previous kernel finishes, pull this block's logits chunk into
    // L2 (lines only; nothing read here is used)
    const int nb_hint = n_nodes ? n_nodes[b] : N_max;
    if (i < nb_hint) {
      const char *row = reinterpret_cast<const char *>(logits + ((size_t)b * N_max + i) * (size_t)V);
      const long lo = (long)c * chunk * 4, hi = min((long)V, (long)(c + 1) * chunk) * 4;
      for (long off = lo + (long)t * 128; off < hi; off += (long)kThreads * 128) prefetch_l2(row + off);
    }
  }
  pdl_wait();

  const int nb = n_nodes ? n_nodes[b] : N_max;
  const int eb = err ? err[b] : 0;
  const bool seq_ok = eb == 0 && nb >= 1 && nb <= N_max;

  __shared__ float s_v[kThreads / 32];
  __shared__ int s_i[kThreads / 32];
  __shared__ bool s_last;

  // The first block of each sequence pulls the acceptance inputs into L2 so
  // the block that finishes the sequence finds them there.
  if (c == 0 && i == 0 && seq_ok) {
    const char *lines[4] = {reinterpret_cast<const char *>(tokens + (size_t)b * N_max),
                            reinterpret_cast<const char *>(parent + (size_t)b * N_max),
                            reinterpret_cast<const char *>(depth + (size_t)b * N_max),
                            reinterpret_cast<const char *>(mask + (size_t)b * N_max * W)};
    const int bytes[4] = {N_max * 4, N_max * 4, N_max * 4, N_max * W * 4};
    for (int a = 0; a < 4; ++a)
      for (int off = t * 128; off < bytes[a]; off += kThreads * 128) prefetch_l2(lines[a] + off);
    const char *ab = reinterpret_cast<const char *>(anc + (size_t)b * (N_max + 1) * (D_max + 1));
    for (int off = t * 128; off < (N_max + 1) * (D_max + 1) * 4; off += kThreads * 128)
      prefetch_l2(ab + off);
  }

  // ---- phase 1: argmax of one chunk of row (b, i) ----
  if (seq_ok && i < nb) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    const float *row = logits + ((size_t)b * N_max + i) * (size_t)V;
    const int lo = c * chunk;
    const int hi = min(V, lo + chunk);
    if (vec_ok) {
      // passes of kBatch independent 16-byte loads per thread
      const float4 *r4 = reinterpret_cast<const float4 *>(row + lo);
      const int n4 = (hi - lo) >> 2;
      for (int k0 = 0; k0 < n4; k0 += kBatch * kThreads) {
        float4 a[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int k = k0 + u * kThreads + t;
          a[u] = k < n4 ? ld_stream(r4 + k) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int k = k0 + u * kThreads + t;
          if (k < n4) {
            const int x = lo + 4 * k;
            if (better(a[u].x, x, bv, bi)) { bv = a[u].x; bi = x; }
            if (better(a[u].y, x + 1, bv, bi)) { bv = a[u].y; bi = x + 1; }
            if (better(a[u].z, x + 2, bv, bi)) { bv = a[u].z; bi = x + 2; }
            if (better(a[u].w, x + 3, bv, bi)) { bv = a[u].w; bi = x + 3; }
          }
        }
      }
      for (int x = lo + 4 * n4 + t; x < hi; x += kThreads) {
        const float v = __ldcs(row + x);
        if (better(v, x, bv, bi)) { bv = v; bi = x; }
      }
    } else {
      for (int x = lo + t; x < hi; x += kThreads) {
        const float v = __ldcs(row + x);
        if (better(v, x, bv, bi)) { bv = v; bi = x; }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) { s_v[warp] = bv; s_i[warp] = bi; }
    __syncthreads();
    if (t == 0) {
      for (int w = 1; w < kThreads / 32; ++w)
        if (better(s_v[w], s_i[w], bv, bi)) { bv = s_v[w]; bi = s_i[w]; }
      Partial pr;
      pr.v = bv;
      pr.idx = bi;
      part[((size_t)b * N_max + i) * C + c] = pr;
    }
  }

  // ---- retire this block; the last one of sequence b continues ----
  if (t == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(&counter[b], 1u);
    s_last = ticket == (unsigned)(N_max * C - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (t == 0) counter[b] = 0u;

  // ---- phase 2: acceptance search for sequence b (one node per thread) ----
  __shared__ int s_am[kMaxNodes];
  __shared__ uint32_t s_match[kMaxNodes / 32];
  __shared__ int s_key[kThreads / 32];

  const int cols = D_max + 1;
  // independent loads first, so their latencies overlap
  int my_parent = 0, my_token = 0, my_depth = 0;
  uint32_t my_mask[kMaxNodes / 32];
  if (seq_ok && t < nb) {
    my_parent = parent[(size_t)b * N_max + t];
    my_token = tokens[(size_t)b * N_max + t];
    my_depth = depth[(size_t)b * N_max + t];
#pragma unroll
    for (int w = 0; w < kMaxNodes / 32; ++w)
      my_mask[w] = w < W ? mask[((size_t)b * N_max + t) * W + w] : 0u;
  }
  int am = -1;
  if (seq_ok && t < nb) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    const Partial *pr = part + ((size_t)b * N_max + t) * C;
    for (int k = 0; k < C; ++k) {
      const float v = __ldcg(&pr[k].v);
      const int x = __ldcg(&pr[k].idx);
      if (better(v, x, bv, bi)) { bv = v; bi = x; }
    }
    am = bi;
  }
  if (t < kMaxNodes) s_am[t] = am;
  if (t < N_max) argmax_out[(size_t)b * N_max + t] = am;
  __syncthreads();

  // matched(i): root, or token equals the target's choice at the parent
  bool match = false;
  if (seq_ok && t < nb) {
    match = t == 0 || my_token == s_am[my_parent];
  }
  const unsigned ballot = __ballot_sync(0xffffffffu, match);
  if (lane == 0 && warp < kMaxNodes / 32) s_match[warp] = ballot;
  __syncthreads();

  // accepted(i): every node on the ancestor path (bitmask row) matched
  int key = -1;
  if (seq_ok && t < nb) {
    bool acc = true;
#pragma unroll
    for (int w = 0; w < kMaxNodes / 32; ++w)
      acc = acc && (w >= W || (my_mask[w] & ~s_match[w]) == 0u);
    if (acc) key = (my_depth << 16) | (0xFFFF - t);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
  if (lane == 0) s_key[warp] = key;
  __syncthreads();
  if (warp == 0) {
    key = lane < kThreads / 32 ? s_key[lane] : -1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
    if (lane == 0) s_key[0] = key;
  }
  __syncthreads();
  key = s_key[0];

  if (seq_ok && key >= 0) {
    const int A = key >> 16;
    const int leaf = 0xFFFF - (key & 0xFFFF);
    for (int k = t; k < cols; k += kThreads)
      path[(size_t)b * cols + k] = k <= A ? anc[((size_t)b * (N_max + 1) + leaf + 1) * cols + k] : 0;
    if (t == 0) {
      accept_len[b] = A;
      leaf_out[b] = leaf;
      bonus[b] = s_am[leaf];
    }
  } else {
    for (int k = t; k < cols; k += kThreads) path[(size_t)b * cols + k] = 0;
    if (t == 0) {
      accept_len[b] = 0;
      leaf_out[b] = -1;
      bonus[b] = -1;
    }
  }
}

struct VerifyPlan {
  int chunk;
  int C;
  size_t counter_bytes;
  size_t part_bytes;
};

VerifyPlan plan_verify(int B, int N_max, int V) {
  VerifyPlan p;
  const long rows = (long)B * N_max;
  const long total = rows * (long)V;
  const long resident = 4L * sm_count();  // blocks of 256 threads resident at once
  const long per_pass = (long)kBatch * kThreads * 4;
  long chunk = (total + resident - 1) / resident;
  chunk = (chunk + per_pass - 1) / per_pass * per_pass;  // whole passes
  if (chunk < per_pass) chunk = per_pass;
  if (chunk > V) chunk = (V + 3) / 4 * 4;
  p.chunk = (int)chunk;
  p.C = (int)((V + chunk - 1) / chunk);
  p.counter_bytes = align_up(sizeof(unsigned) * (size_t)B, 256);
  p.part_bytes = sizeof(Partial) * (size_t)B * N_max * p.C;
  return p;
}

}  // namespace
}  // namespace tsd

TSD_API size_t tsd_tree_verify_workspace_bytes(int B, int N_max, int V) {
  if (B <= 0 || N_max <= 0 || V <= 0) return 0;
  const tsd::VerifyPlan p = tsd::plan_verify(B, N_max, V);
  return p.counter_bytes + p.part_bytes;
}

TSD_API int tsd_tree_verify_greedy(const float *logits, const int32_t *tokens,
                                   const int32_t *parent, const int32_t *anc, const int32_t *depth,
                                   const uint32_t *mask, const int32_t *n_nodes, const int32_t *err,
                                   int B, int N_max, int V, int D_max, int32_t *argmax,
                                   int32_t *accept_len, int32_t *leaf, int32_t *path, int32_t *bonus,
                                   void *workspace, size_t ws_bytes, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0 || V < 1) return B < 0 ? TSD_ERR_ARG : TSD_ERR_LIMIT;
  if (N_max < 1 || N_max > kMaxNodes || D_max < 0 || D_max > kMaxDepth || B > 65535)
    return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!logits || !tokens || !parent || !anc || !depth || !mask || !argmax || !accept_len ||
      !leaf || !path || !bonus)
    return TSD_ERR_ARG;
  const VerifyPlan p = plan_verify(B, N_max, V);
  if (!workspace || ws_bytes < p.counter_bytes + p.part_bytes || !aligned(workspace, 16))
    return TSD_ERR_WORKSPACE;
  unsigned *counter = static_cast<unsigned *>(workspace);
  Partial *part = reinterpret_cast<Partial *>(static_cast<char *>(workspace) + p.counter_bytes);
  const int W = (N_max + 31) / 32;
  const int vec_ok = (V % 4 == 0) && aligned(logits, 16);
  if (launch(verify_greedy_kernel, dim3(p.C, N_max, B), dim3(kThreads), 0, as_cuda(stream), logits,
             tokens, parent, anc, depth, mask, n_nodes, err, N_max, V, D_max, W, p.chunk, p.C,
             vec_ok, argmax, accept_len, leaf, path, bonus, part, counter) != cudaSuccess)
    return TSD_ERR_CUDA;
  return TSD_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of tsd_tree_verify_greedy.
//
// Some callers cannot call cudaMalloc: a plugin running inside another
// engine that owns every byte of device memory and hands out no workspace,
// or a latency-critical path where an allocation (which may synchronise the
// device) is not acceptable.  This entry point keeps its scratch (the
// per-sequence tickets and the per-chunk argmax partials) in a fixed array
// in device global memory, loaded with the library: every GPU that loads
// libtsd.so holds kStaticScratchBytes of it until the process exits.
//
// In host code `g_verify_scratch` names a host-side shadow, not device
// memory, so its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.  The first
// call on a device performs that look-up, so make it before any stream
// capture.  All calls share the one array: each call zeroes the tickets on
// its stream before its kernel runs, and calls that overlap on the GPU (two
// streams, or two devices' contexts racing on one array) race on it.
// ---------------------------------------------------------------------------

namespace tsd {
namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;  // 1 MiB
__device__ __align__(256) unsigned char g_verify_scratch[kStaticScratchBytes];

void *static_scratch_ptr() {
  static void *ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace tsd

TSD_API size_t tsd_tree_verify_static_capacity(void) { return tsd::kStaticScratchBytes; }

TSD_API int tsd_tree_verify_greedy_static(const float *logits, const int32_t *tokens,
                                          const int32_t *parent, const int32_t *anc,
                                          const int32_t *depth, const uint32_t *mask,
                                          const int32_t *n_nodes, const int32_t *err, int B,
                                          int N_max, int V, int D_max, int32_t *argmax,
                                          int32_t *accept_len, int32_t *leaf, int32_t *path,
                                          int32_t *bonus, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0 || V < 1) return B < 0 ? TSD_ERR_ARG : TSD_ERR_LIMIT;
  if (N_max < 1 || N_max > kMaxNodes || D_max < 0 || D_max > kMaxDepth || B > 65535)
    return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!logits || !tokens || !parent || !anc || !depth || !mask || !argmax || !accept_len ||
      !leaf || !path || !bonus)
    return TSD_ERR_ARG;
  const VerifyPlan p = plan_verify(B, N_max, V);
  if (p.counter_bytes + p.part_bytes > kStaticScratchBytes) return TSD_ERR_LIMIT;
  void *scratch = static_scratch_ptr();
  if (!scratch) return TSD_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, p.counter_bytes, as_cuda(stream)) != cudaSuccess)
    return TSD_ERR_CUDA;
  unsigned *counter = static_cast<unsigned *>(scratch);
  Partial *part = reinterpret_cast<Partial *>(static_cast<char *>(scratch) + p.counter_bytes);
  const int W = (N_max + 31) / 32;
  const int vec_ok = (V % 4 == 0) && aligned(logits, 16);
  if (launch(verify_greedy_kernel, dim3(p.C, N_max, B), dim3(kThreads), 0, as_cuda(stream), logits,
             tokens, parent, anc, depth, mask, n_nodes, err, N_max, V, D_max, W, p.chunk, p.C,
             vec_ok, argmax, accept_len, leaf, path, bonus, part, counter) != cudaSuccess)
    return TSD_ERR_CUDA;
  return TSD_OK;
}
