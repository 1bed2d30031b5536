// a3: greedy verification of a draft tree.
//
// "Speculative Decoding Hierárquico: Medusa, EAGLE-2 e Multi-Token
// Prediction", Medusa section: the target evaluates all branches in one
// parallel pass and the longest valid path is kept.  Greedy acceptance: a
// draft token is accepted when it equals the target's most likely token at
// its parent, and its parent was accepted.
//
// One fused launch.  Grid (Gs, sequence): the valid rows of sequence b,
// nb * V floats laid end to end, are cut into Gs equal ranges, one per
// block, so every block streams the same number of bytes.  Each thread reads
// its part in passes of 8 independent 16-byte loads (32 KB per block in
// flight, four blocks per SM) and keeps a running (max, first index) for
// each row its range touches (at most two); the block then folds each row's
// candidate into a per-row 64-bit key with one atomicMax (key order = value,
// then lower index).  The block that takes a sequence's last ticket reads
// the row keys (resetting them), evaluates acceptance with the ancestor
// bitmasks and writes leaf / accept_len / path / bonus; it also resets the
// ticket, so the workspace is zero again when the launch ends.

#include <cuda.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "commit_core.cuh"
#include "sm100_ptx.cuh"
#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;        // 16-byte loads in flight per thread
constexpr int kBlocksPerSm = 4;  // 1024 threads x 64 registers per SM
constexpr int kFusedCap = 2 * kMaxMoves;  // staged (K, V) entries of the fused commit

// (v, i) beats (bv, bi): larger value, or equal value and lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Order-preserving 64-bit key: larger value first, then lower index; -0 and
// +0 share one key so they tie on value.
__device__ __forceinline__ unsigned long long arg_key(float v, int i) {
  if (v == 0.f) v = 0.f;
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
}

__device__ __forceinline__ void take4(const float4 &a, int x, float &bv, int &bi) {
  if (better(a.x, x, bv, bi)) { bv = a.x; bi = x; }
  if (better(a.y, x + 1, bv, bi)) { bv = a.y; bi = x + 1; }
  if (better(a.z, x + 2, bv, bi)) { bv = a.z; bi = x + 2; }
  if (better(a.w, x + 3, bv, bi)) { bv = a.w; bi = x + 3; }
}

// CD: 0, or the head dimension of the cache the block that finishes a
// sequence also commits (the fused commit).
template <int CD>
__global__ void __launch_bounds__(kThreads, kBlocksPerSm)
verify_greedy_kernel(const float *__restrict__ logits, const int32_t *__restrict__ tokens,
                     const int32_t *__restrict__ parent, const int32_t *__restrict__ anc,
                     const int32_t *__restrict__ depth, const uint32_t *__restrict__ mask,
                     const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ err,
                     int N_max, int V, int D_max, int W, int vec,
                     int32_t *__restrict__ argmax_out, int32_t *__restrict__ accept_len,
                     int32_t *__restrict__ leaf_out, int32_t *__restrict__ path,
                     int32_t *__restrict__ bonus, unsigned long long *__restrict__ row_key,
                     unsigned *__restrict__ counter, const CommitArgs ca) {
  using namespace sm100;
  __shared__ float s_v[2][kThreads / 32];
  __shared__ int s_i[2][kThreads / 32];
  __shared__ bool s_last;

  // With the fused commit this grid writes the K/V cache, which the next
  // attention pass reads before it waits for its own predecessor: no early
  // release then.
  if (CD == 0) pdl_trigger();
  const int g = blockIdx.x;
  const int Gs = gridDim.x;
  const int b = blockIdx.y;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int warp = t >> 5;
  const float *seq = logits + (size_t)b * N_max * (size_t)V;
  {
    // while the previous kernel finishes, pull the first pass of this
    // block's range into L2 (lines only; nothing read here is used)
    const int nb_hint = n_nodes ? n_nodes[b] : N_max;
    if (nb_hint >= 1 && nb_hint <= N_max) {
      const long total = (long)nb_hint * V;
      const long lo = (total * g / Gs) & ~3L;
      const long hi = min(g + 1 == Gs ? total : (total * (g + 1) / Gs) & ~3L,
                          lo + (long)kBatch * kThreads * 4);
      const char *base = reinterpret_cast<const char *>(seq);
      for (long off = lo * 4 + (long)t * 128; off < hi * 4; off += (long)kThreads * 128)
        prefetch_l2(base + off);
      if constexpr (CD != 0) {
        // the fused commit's inputs (lengths, the tree's block ids, the tree's
        // K and V: the only entries a commit can move), each block a slice,
        // so that the block that commits finds them in L2
        const int P = ca.prefix_len[b];
        if (P >= 0 && (long)P + nb_hint <= (long)ca.max_blocks * kPage) {
          const int32_t *trow = ca.table + (size_t)b * ca.max_blocks;
          const int pg0 = P / kPage, pg1 = (P + nb_hint - 1) / kPage;
          const long entries = (long)(P + nb_hint - pg0 * kPage) * ca.Hkv;  // slots x heads
          for (long x = (long)g * kThreads + t; x < entries * 4; x += (long)Gs * kThreads) {
            const int line = (int)(x & 3);  // four 128-byte lines of K and of V per entry
            const long en = x >> 2;
            const int slot = pg0 * kPage + (int)(en / ca.Hkv), h = (int)(en % ca.Hkv);
            const int page = trow[slot / kPage];
            if (page < 0 || page >= ca.num_blocks || slot / kPage > pg1) continue;
            const size_t off = (((size_t)page * ca.Hkv + h) * kPage + slot % kPage) * CD * 2;
            for (int l = 0; l < ca.num_layers && l < 2; ++l) {
              const size_t lb = (size_t)l * (size_t)ca.layer_stride * 2;
              if (line * 128 < CD * 2) {
                prefetch_l2(reinterpret_cast<const char *>(ca.k) + lb + off + line * 128);
                prefetch_l2(reinterpret_cast<const char *>(ca.v) + lb + off + line * 128);
              }
            }
          }
        }
      }
    }
  }
  pdl_wait();

  const int nb = n_nodes ? n_nodes[b] : N_max;
  const int eb = err ? err[b] : 0;
  const bool seq_ok = eb == 0 && nb >= 1 && nb <= N_max;

  // Block-wide fold of up to two candidates (rows r and r + 1) into the row
  // keys.  Every thread calls it with the same `two`.
  auto fold = [&](int r, bool two, float v0, int i0, float v1, int i1) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov0 = __shfl_xor_sync(0xffffffffu, v0, off);
      const int oi0 = __shfl_xor_sync(0xffffffffu, i0, off);
      if (better(ov0, oi0, v0, i0)) { v0 = ov0; i0 = oi0; }
      const float ov1 = __shfl_xor_sync(0xffffffffu, v1, off);
      const int oi1 = __shfl_xor_sync(0xffffffffu, i1, off);
      if (better(ov1, oi1, v1, i1)) { v1 = ov1; i1 = oi1; }
    }
    if (lane == 0) {
      s_v[0][warp] = v0; s_i[0][warp] = i0;
      s_v[1][warp] = v1; s_i[1][warp] = i1;
    }
    __syncthreads();
    if (t < 2 && (t == 0 || two)) {
      float bv = s_v[t][0];
      int bi = s_i[t][0];
      for (int w = 1; w < kThreads / 32; ++w)
        if (better(s_v[t][w], s_i[t][w], bv, bi)) { bv = s_v[t][w]; bi = s_i[t][w]; }
      atomicMax(&row_key[(size_t)b * N_max + r + t], arg_key(bv, bi));
    }
    __syncthreads();
  };

  // ---- phase 1: argmax over this block's range of the sequence's rows ----
  if (seq_ok) {
    const long total = (long)nb * V;
    const long lo = (total * g / Gs) & ~3L;
    const long hi = g + 1 == Gs ? total : (total * (g + 1) / Gs) & ~3L;
    if (lo < hi && vec && hi - lo <= V) {
      // the range touches rows r0 and (if it crosses end0) r0 + 1; a float4
      // never straddles a row end since V is a multiple of 4
      const int r0 = (int)(lo / V);
      const long end0 = (long)(r0 + 1) * V;
      const bool two = hi > end0;
      float v0 = -INFINITY, v1 = -INFINITY;
      int i0 = INT_MAX, i1 = INT_MAX;
      // 32-bit offsets from the range start: the range is at most one row
      const float4 *src = reinterpret_cast<const float4 *>(seq) + (lo >> 2);
      const int n4 = (int)((hi - lo) >> 2);
      const int e4 = (int)((end0 - lo) >> 2);  // first float4 of row r0 + 1
      const int x0 = (int)(lo - (long)r0 * V);  // column of src[0] in row r0
      const int x1 = (int)(lo - end0);          // ... and in row r0 + 1 (negative)
      constexpr int kStride = kBatch * kThreads;
      const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      // passes of kBatch independent loads per thread; once a pass's loads
      // are issued, one thread asks the copy engine to pull the next pass into
      // L2 (inside a verify step the stream then holds its rate against the
      // write-backs of the attention that ran before it)
      float4 a[kBatch];
      for (int p4 = 0; p4 < n4; p4 += kStride) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int q = p4 + u * kThreads + t;
          a[u] = q < n4 ? __ldcs(src + q) : ninf;
        }
        if (t == 0 && p4 + kStride < n4)
          bulk_prefetch_l2(src + p4 + kStride, (uint32_t)min(kStride, n4 - p4 - kStride) * 16u);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int q = p4 + u * kThreads + t;
          if (q < n4) {
            if (q < e4)
              take4(a[u], x0 + 4 * q, v0, i0);
            else
              take4(a[u], x1 + 4 * q, v1, i1);
          }
        }
      }
      fold(r0, two, v0, i0, v1, i1);
    } else if (lo < hi) {
      // general case (rows shorter than the range, or unaligned rows): one
      // row segment at a time with plain loads
      for (long p = lo; p < hi;) {
        const int r = (int)(p / V);
        const long e = min(hi, (long)(r + 1) * V);
        float bv = -INFINITY;
        int bi = INT_MAX;
        const long rs = (long)r * V;
        if (vec) {  // p, e and the row start are multiples of 4
          const float4 *s4 = reinterpret_cast<const float4 *>(seq);
          for (long q = (p >> 2) + t; q < (e >> 2); q += kThreads)
            take4(__ldcs(s4 + q), (int)(4 * q - rs), bv, bi);
        } else {
          for (long q = p + t; q < e; q += kThreads) {
            const float v = __ldcs(seq + q);
            if (better(v, (int)(q - rs), bv, bi)) { bv = v; bi = (int)(q - rs); }
          }
        }
        fold(r, false, bv, bi, -INFINITY, INT_MAX);
        p = e;
      }
    }
  }

  // ---- retire this block; the last one of sequence b continues ----
  if (t == 0) {
    __threadfence();
    const unsigned ticket = atomicAdd(&counter[b], 1u);
    s_last = ticket == (unsigned)(Gs - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (t == 0) counter[b] = 0u;

  // ---- phase 2: acceptance search for sequence b (one node per thread) ----
  __shared__ int s_am[kMaxNodes];
  __shared__ int s_par[kMaxNodes];
  __shared__ uint32_t s_match[kMaxNodes / 32];
  __shared__ int s_key[kThreads / 32];

  const int cols = D_max + 1;
  // independent loads first, so their latencies overlap
  int my_parent = 0, my_token = 0, my_depth = 0;
  unsigned long long my_key = 0ull;
  uint32_t my_mask[kMaxNodes / 32];
  if (seq_ok && t < nb) {
    my_key = __ldcg(&row_key[(size_t)b * N_max + t]);
    my_parent = parent[(size_t)b * N_max + t];
    my_token = tokens[(size_t)b * N_max + t];
    my_depth = depth[(size_t)b * N_max + t];
#pragma unroll
    for (int w = 0; w < kMaxNodes / 32; ++w)
      my_mask[w] = w < W ? mask[((size_t)b * N_max + t) * W + w] : 0u;
  }
  int am = -1;
  if (seq_ok && t < nb) {
    row_key[(size_t)b * N_max + t] = 0ull;  // zero again for the next call
    am = my_key ? (int)(0xFFFFFFFFu - (uint32_t)(my_key & 0xFFFFFFFFull)) : -1;
  }
  if (t < kMaxNodes) {
    s_am[t] = am;
    s_par[t] = (seq_ok && t < nb) ? my_parent : -1;
  }
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
    if (t == 0) {
      // path[k] = safe id of the leaf's depth-k ancestor (its ancestor-table
      // row), walked up the parents already in shared memory: the accepted
      // leaf's chain is valid and A = its depth, so no global round trip
      int a = leaf;
      for (int k = A; k >= 0; --k) {
        path[(size_t)b * cols + k] = a + 1;
        a = a >= 0 && a < kMaxNodes ? s_par[a] : -1;
      }
    }
    for (int k = A + 1 + t; k < cols; k += kThreads) path[(size_t)b * cols + k] = 0;
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
  if constexpr (CD != 0) {
    // ---- phase 3 (fused commit): the accepted path's K/V of sequence b, every
    // kv head and layer, exactly as tsd_kv_commit_path would commit it from
    // the accept_len / path rows just written ----
    __shared__ CommitMoves mv;
    extern __shared__ uint4 stage[];
    __syncthreads();  // this block's accept_len / path writes are visible to it
    if (warp == 0)
      commit_plan_warp(ca, b, N_max, D_max, n_nodes, err, accept_len, path, true, mv, lane);
    __syncthreads();
    commit_copy<CD>(ca, mv, 0, ca.Hkv, 0, ca.num_layers, stage, kFusedCap, t, kThreads);
  }
}

struct VerifyPlan {
  int Gs;                // blocks per sequence
  size_t counter_bytes;  // one ticket per sequence
  size_t key_bytes;      // one 64-bit argmax key per row
};

VerifyPlan plan_verify(int B, int N_max, int V) {
  VerifyPlan p;
  // about one resident wave of blocks, each with at least 4096 floats; at
  // least N_max blocks per sequence, so a block's range spans at most two rows
  const long resident = (long)kBlocksPerSm * sm_count();
  long gs = resident / B;
  const long min_chunks = ((long)N_max * V + 4095) / 4096;
  if (gs > min_chunks) gs = min_chunks;
  if (gs < N_max) gs = N_max;
  if (gs > 65535) gs = 65535;
  p.Gs = (int)gs;
  p.counter_bytes = align_up(sizeof(unsigned) * (size_t)B, 256);
  p.key_bytes = sizeof(unsigned long long) * (size_t)B * N_max;
  return p;
}

// cd: 0 (no commit) or the cache's head dimension (64, 128) with `ca` set.
int launch_verify(const float *logits, const int32_t *tokens, const int32_t *parent,
                  const int32_t *anc, const int32_t *depth, const uint32_t *mask,
                  const int32_t *n_nodes, const int32_t *err, int B, int N_max, int V, int D_max,
                  int32_t *argmax, int32_t *accept_len, int32_t *leaf, int32_t *path,
                  int32_t *bonus, void *scratch, const VerifyPlan &p, cudaStream_t s,
                  int cd = 0, const CommitArgs &ca = CommitArgs{}) {
  unsigned *counter = static_cast<unsigned *>(scratch);
  unsigned long long *keys =
      reinterpret_cast<unsigned long long *>(static_cast<char *>(scratch) + p.counter_bytes);
  const int W = (N_max + 31) / 32;
  const int vec = (V % 4 == 0) && aligned(logits, 16);
  const dim3 grid(p.Gs, B);
  cudaError_t e;
  if (cd == 0) {
    e = launch(verify_greedy_kernel<0>, grid, dim3(kThreads), 0, s, logits, tokens, parent, anc,
               depth, mask, n_nodes, err, N_max, V, D_max, W, vec, argmax, accept_len, leaf, path,
               bonus, keys, counter, ca);
  } else {
    const size_t smem = 2 * (size_t)kFusedCap * (cd / 8) * sizeof(uint4);
    const void *k = cd == 128 ? reinterpret_cast<const void *>(verify_greedy_kernel<128>)
                              : reinterpret_cast<const void *>(verify_greedy_kernel<64>);
    if (!set_smem(k, smem)) return TSD_ERR_CUDA;
    e = cd == 128 ? launch(verify_greedy_kernel<128>, grid, dim3(kThreads), smem, s, logits, tokens,
                           parent, anc, depth, mask, n_nodes, err, N_max, V, D_max, W, vec, argmax,
                           accept_len, leaf, path, bonus, keys, counter, ca)
                  : launch(verify_greedy_kernel<64>, grid, dim3(kThreads), smem, s, logits, tokens,
                           parent, anc, depth, mask, n_nodes, err, N_max, V, D_max, W, vec, argmax,
                           accept_len, leaf, path, bonus, keys, counter, ca);
  }
  return e == cudaSuccess ? TSD_OK : TSD_ERR_CUDA;
}

}  // namespace
}  // namespace tsd

TSD_API size_t tsd_tree_verify_workspace_bytes(int B, int N_max, int V) {
  if (B <= 0 || N_max <= 0 || V <= 0) return 0;
  const tsd::VerifyPlan p = tsd::plan_verify(B, N_max, V);
  return p.counter_bytes + p.key_bytes;
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
  if (!workspace || ws_bytes < p.counter_bytes + p.key_bytes || !aligned(workspace, 16))
    return TSD_ERR_WORKSPACE;
  return launch_verify(logits, tokens, parent, anc, depth, mask, n_nodes, err, B, N_max, V, D_max,
                       argmax, accept_len, leaf, path, bonus, workspace, p, as_cuda(stream));
}

TSD_API int tsd_tree_verify_greedy_commit(
    const float *logits, const int32_t *tokens, const int32_t *parent, const int32_t *anc,
    const int32_t *depth, const uint32_t *mask, const int32_t *n_nodes, const int32_t *err, int B,
    int N_max, int V, int D_max, int32_t *argmax, int32_t *accept_len, int32_t *leaf, int32_t *path,
    int32_t *bonus, void *workspace, size_t ws_bytes, uint16_t *k_cache, uint16_t *v_cache,
    int num_layers, int64_t layer_stride, const int32_t *block_table, int max_blocks,
    int num_blocks, const int32_t *prefix_len, int Hkv, int D, int32_t *new_len, int32_t *moved,
    int32_t *status, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0 || V < 1) return B < 0 ? TSD_ERR_ARG : TSD_ERR_LIMIT;
  if (N_max < 1 || N_max > kMaxNodes || D_max < 0 || D_max > kMaxDepth || B > 65535)
    return TSD_ERR_LIMIT;
  if (num_layers < 0 || Hkv < 1 || max_blocks < 1 || num_blocks < 1) return TSD_ERR_ARG;
  if (D != 64 && D != 128) return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!logits || !tokens || !parent || !anc || !depth || !mask || !argmax || !accept_len ||
      !leaf || !path || !bonus)
    return TSD_ERR_ARG;
  if (num_layers > 0 && (!k_cache || !v_cache || !block_table || !prefix_len || !new_len))
    return TSD_ERR_ARG;
  if (num_layers > 0 && (!aligned(k_cache, 16) || !aligned(v_cache, 16))) return TSD_ERR_ARG;
  const int64_t pool = (int64_t)num_blocks * Hkv * kPage * D;
  if (num_layers > 1 && (layer_stride < pool || layer_stride % 8 != 0)) return TSD_ERR_ARG;
  const VerifyPlan p = plan_verify(B, N_max, V);
  if (!workspace || ws_bytes < p.counter_bytes + p.key_bytes || !aligned(workspace, 16))
    return TSD_ERR_WORKSPACE;
  if (num_layers == 0 || B == 1) {
    // One sequence: its commit would run in a single block after the search
    // (measured slower than the commit kernel's block per head), so the two
    // kernels are launched back to back instead.
    const int rc = launch_verify(logits, tokens, parent, anc, depth, mask, n_nodes, err, B, N_max,
                                 V, D_max, argmax, accept_len, leaf, path, bonus, workspace, p,
                                 as_cuda(stream));
    if (rc != TSD_OK || num_layers == 0) return rc;
    return tsd_kv_commit_path(k_cache, v_cache, num_layers, layer_stride, block_table, max_blocks,
                              num_blocks, prefix_len, n_nodes, accept_len, path, err, B, N_max, Hkv,
                              D, D_max, new_len, moved, status, stream);
  }
  const CommitArgs ca{k_cache, v_cache, num_layers, layer_stride, block_table, max_blocks,
                      num_blocks, prefix_len, nullptr, Hkv, new_len, moved, status};
  return launch_verify(logits, tokens, parent, anc, depth, mask, n_nodes, err, B, N_max, V, D_max,
                       argmax, accept_len, leaf, path, bonus, workspace, p, as_cuda(stream), D, ca);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of tsd_tree_verify_greedy.
//
// Some callers cannot call cudaMalloc: a plugin running inside another
// engine that owns every byte of device memory and hands out no workspace,
// or a latency-critical path where an allocation (which may synchronise the
// device) is not acceptable.  This entry point keeps its scratch (the
// per-sequence tickets and the per-row argmax keys) in a fixed array
// in device global memory, loaded with the library: every GPU that loads
// libtsd.so holds its own kStaticScratchBytes instance until the process
// exits.
//
// In host code `g_verify_scratch` names a host-side shadow, not device
// memory, so its device address is looked up with cudaGetSymbolAddress (with
// the device current) and cached per device, together with the id of the
// CUDA context it belongs to: after a device reset the context, and with it
// the address, changes, and the next call looks it up again.  The look-up is
// serialised by a mutex, so host threads may make their first calls at
// once.  The first call on a device (and the first after a reset) performs
// that look-up, so make it before any stream capture.  All calls on one
// device share its array: each call zeroes the tickets and row keys it uses
// on its stream before its kernel runs, and calls that overlap on the same
// device (two streams) race on it.
// ---------------------------------------------------------------------------

namespace tsd {
namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;  // 1 MiB per device
__device__ __align__(256) unsigned char g_verify_scratch[kStaticScratchBytes];

// Id of the calling thread's current CUDA context (0 when it cannot be read).
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

void *static_scratch_ptr() {
  struct Entry {
    unsigned long long ctx;
    void *ptr;
  };
  static std::mutex mu;
  static Entry cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();  // 0 before the context exists
  if (cache[dev].ptr && ctx != 0 && cache[dev].ctx == ctx) return cache[dev].ptr;
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess) return nullptr;
  cache[dev] = Entry{current_context_id(), p};  // the look-up made the context current
  return p;
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
  if (p.counter_bytes + p.key_bytes > kStaticScratchBytes) return TSD_ERR_LIMIT;
  void *scratch = static_scratch_ptr();
  if (!scratch) return TSD_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, p.counter_bytes + p.key_bytes, as_cuda(stream)) != cudaSuccess)
    return TSD_ERR_CUDA;
  return launch_verify(logits, tokens, parent, anc, depth, mask, n_nodes, err, B, N_max, V, D_max,
                       argmax, accept_len, leaf, path, bonus, scratch, p, as_cuda(stream));
}
