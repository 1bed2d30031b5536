// a2: tree-masked attention for every draft-tree node in one pass.
//
// "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on Ascend NPUs",
// technical summary 2.3: the teacher evaluates all speculative nodes at once
// under a tree attention mask that lets node k attend only to its own
// ancestor path (itself included), with no leakage across branches.
// "Speculative Decoding Hierárquico: Medusa, EAGLE-2 e Multi-Token
// Prediction", Medusa section: parallel nodes attend only to their direct
// ancestors.
//
// Layout of the work.  For one (sequence b, kv head) the query rows are the
// tree nodes times the q heads of that kv group, packed node-major
// (row = node * g + head-in-group), so the GQA group shares every K/V tile.
// A block owns 64 such rows and one split of the key range (split-KV, sized
// to fill the GPU); keys are read straight from the paged cache with 16-byte
// cp.async (double-buffered, XOR-swizzled rows).  Q K^T and P V run on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) with an online
// softmax in registers.  Tiles that lie wholly inside the committed prefix
// are visible to every row and skip masking; tiles that reach the tree tail
// read each row's ancestor bitmask word by word.  Each split writes fp32
// partials (O, running max, running sum); a combine kernel merges them,
// normalises and rounds to bf16.

#include <cuda_bf16.h>

#include <cmath>

#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kBM = 64;  // query rows per block
constexpr int kBN = 64;  // keys per tile
constexpr int kAttnThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const uint16_t *q;
  const uint16_t *k;
  const uint16_t *v;
  const int32_t *table;
  int max_blocks, num_blocks;
  const int32_t *prefix_len;
  const int32_t *n_nodes;
  const uint32_t *mask;
  const int32_t *err;
  int N_max, Hq, Hkv, g, W, max_slots;
  float scale_log2;
  int chunk, splits, row_tiles, rows_pad;
  float *part_o;    // [B*Hkv][splits][rows_pad][D]
  float2 *part_ml;  // [B*Hkv][splits][rows_pad]  (max in log2 units, sum)
  uint16_t *out;
  float *lse;
  int32_t *status;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                        uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                          uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// byte offset of 16-byte chunk `ch` of row `row` in a swizzled [rows][D] bf16 tile
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)((row * (D / 8) + (ch ^ (row & 7))) * 16);
}

// Sequence-level validity shared by the split and combine kernels.
__device__ __forceinline__ bool seq_ok(const AttnParams &p, int b, int &P, int &nb) {
  P = p.prefix_len[b];
  nb = p.n_nodes ? p.n_nodes[b] : p.N_max;
  const int e = p.err ? p.err[b] : 0;
  if (e != 0 || nb < 1 || nb > p.N_max) return false;
  if (P < 0 || (long)P + nb > (long)p.max_slots || (long)P + nb > (long)p.max_blocks * kPage)
    return false;
  return true;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads)
tree_attn_split_kernel(const AttnParams p) {
  constexpr int kCh = D / 8;    // 16-byte chunks per row
  constexpr int kKT = D / 16;   // k-steps of Q K^T
  constexpr int kDT = D / 8;    // n-tiles of P V
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *sQ = smem;
  unsigned char *sK = smem + kBM * D * 2;
  unsigned char *sV = sK + 2 * kBN * D * 2;

  const int rt = blockIdx.x;
  const int split = blockIdx.y;
  const int z = blockIdx.z;
  const int b = z / p.Hkv;
  const int hkv = z % p.Hkv;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  int P, nb;
  const bool ok = seq_ok(p, b, P, nb);
  if (!ok) {
    if (rt == 0 && split == 0 && hkv == 0 && tid == 0 && p.status) {
      const int e = p.err ? p.err[b] : 0;
      const int nbb = p.n_nodes ? p.n_nodes[b] : p.N_max;
      if (e == 0 && nbb >= 1 && nbb <= p.N_max) atomicOr(p.status, TSD_STATUS_BAD_LEN);
    }
    return;
  }
  const int rows_valid = nb * p.g;
  if (rt * kBM >= rows_valid) return;
  const int seq_len = P + nb;
  const int k_begin = split * p.chunk;
  if (k_begin >= seq_len) return;
  const int k_end = min(seq_len, k_begin + p.chunk);
  const int ntiles = (k_end - k_begin + kBN - 1) / kBN;
  const int32_t *trow = p.table + (size_t)b * p.max_blocks;

  // ---- Q tile (rows rt*64 .. +63), zero-filled past the valid rows ----
  for (int c = tid; c < kBM * kCh; c += kAttnThreads) {
    const int r = c / kCh, ch = c % kCh;
    const int row = rt * kBM + r;
    const bool valid = row < rows_valid;
    const int node = valid ? row / p.g : 0;
    const int head = hkv * p.g + (valid ? row % p.g : 0);
    const uint16_t *src = p.q + (((size_t)b * p.N_max + node) * p.Hq + head) * D + ch * 8;
    cp_async16(smem_u32(sQ) + swz<D>(r, ch), src, valid);
  }

  bool bad_page = false;
  auto load_tile = [&](int stage, int ts) {
    for (int c = tid; c < kBN * kCh; c += kAttnThreads) {
      const int r = c / kCh, ch = c % kCh;
      const int slot = ts + r;
      bool valid = slot < k_end;
      int page = 0;
      if (valid) {
        page = __ldg(trow + slot / kPage);
        if (page < 0 || page >= p.num_blocks) {
          bad_page = true;
          valid = false;
          page = 0;
        }
      }
      const size_t off = (((size_t)page * p.Hkv + hkv) * kPage + slot % kPage) * D + ch * 8;
      cp_async16(smem_u32(sK + stage * kBN * D * 2) + swz<D>(r, ch), p.k + off, valid);
      cp_async16(smem_u32(sV + stage * kBN * D * 2) + swz<D>(r, ch), p.v + off, valid);
    }
  };

  load_tile(0, k_begin);
  cp_async_commit();

  // per-thread rows: ra (accumulator regs 0,1) and rb (regs 2,3)
  const int ra_local = warp * 16 + (lane >> 2);
  const int ra = rt * kBM + ra_local;
  const int rb = ra + 8;
  const int node_a = ra < rows_valid ? ra / p.g : -1;
  const int node_b = rb < rows_valid ? rb / p.g : -1;
  const uint32_t *mask_a = p.mask + ((size_t)b * p.N_max + (node_a < 0 ? 0 : node_a)) * p.W;
  const uint32_t *mask_b = p.mask + ((size_t)b * p.N_max + (node_b < 0 ? 0 : node_b)) * p.W;

  uint32_t qf[kKT][4];
  float o[kDT][4];
#pragma unroll
  for (int i = 0; i < kDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  for (int it = 0; it < ntiles; ++it) {
    const int ts = k_begin + it * kBN;
    if (it + 1 < ntiles) {
      load_tile((it + 1) & 1, ts + kBN);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < kKT; ++kk)
        ldsm_x4(qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                smem_u32(sQ) + swz<D>(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)));
    }
    const uint32_t kbase = smem_u32(sK + (it & 1) * kBN * D * 2);
    const uint32_t vbase = smem_u32(sV + (it & 1) * kBN * D * 2);

    // S = Q K^T for this warp's 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kKT; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3,
                kbase + swz<D>(np * 16 + (lane & 7) + ((lane >> 4) << 3),
                               kk * 2 + ((lane >> 3) & 1)));
        mma_bf16(s[2 * np], qf[kk], b0, b1);
        mma_bf16(s[2 * np + 1], qf[kk], b2, b3);
      }
    }

    // scale, mask, online softmax
    const bool full = (ts + kBN <= P) && (ts + kBN <= k_end);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[nt][e] * p.scale_log2;
        if (!full) {
          const int slot = ts + nt * 8 + 2 * (lane & 3) + (e & 1);
          bool vis = slot < k_end;
          if (vis && slot >= P) {
            const int j = slot - P;
            const int node = (e < 2) ? node_a : node_b;
            const uint32_t *mrow = (e < 2) ? mask_a : mask_b;
            vis = node >= 0 && ((__ldg(mrow + (j >> 5)) >> (j & 31)) & 1u);
          }
          if (!vis) x = -INFINITY;
        }
        s[nt][e] = x;
      }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    }
    float alpha[2], muse[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mnew = fmaxf(m_run[h], mx[h]);
      muse[h] = mnew == -INFINITY ? 0.f : mnew;
      alpha[h] = exp2f(m_run[h] - muse[h]);
      m_run[h] = mnew;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - muse[0]);
      s[nt][1] = exp2f(s[nt][1] - muse[0]);
      s[nt][2] = exp2f(s[nt][2] - muse[1]);
      s[nt][3] = exp2f(s[nt][3] - muse[1]);
      rs[0] += s[nt][0] + s[nt][1];
      rs[1] += s[nt][2] + s[nt][3];
    }
    l_run[0] = l_run[0] * alpha[0] + rs[0];
    l_run[1] = l_run[1] * alpha[1] + rs[1];
#pragma unroll
    for (int dt = 0; dt < kDT; ++dt) {
      o[dt][0] *= alpha[0];
      o[dt][1] *= alpha[0];
      o[dt][2] *= alpha[1];
      o[dt][3] *= alpha[1];
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < kDT / 2; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3,
                  vbase + swz<D>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                 2 * dp + (lane >> 4)));
        mma_bf16(o[2 * dp], a, b0, b1);
        mma_bf16(o[2 * dp + 1], a, b2, b3);
      }
    }
    __syncthreads();  // this stage is refilled by the next iteration's prefetch
  }

  if (bad_page && p.status) atomicOr(p.status, TSD_STATUS_BAD_PAGE);

  // ---- write the split's partials ----
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  const size_t base = ((size_t)z * p.splits + split) * p.rows_pad + rt * kBM;
  float *po = p.part_o + base * D;
  const int ca = 2 * (lane & 3);
#pragma unroll
  for (int dt = 0; dt < kDT; ++dt) {
    *reinterpret_cast<float2 *>(po + (size_t)ra_local * D + dt * 8 + ca) =
        make_float2(o[dt][0], o[dt][1]);
    *reinterpret_cast<float2 *>(po + (size_t)(ra_local + 8) * D + dt * 8 + ca) =
        make_float2(o[dt][2], o[dt][3]);
  }
  if ((lane & 3) == 0) {
    p.part_ml[base + ra_local] = make_float2(m_run[0], l_run[0]);
    p.part_ml[base + ra_local + 8] = make_float2(m_run[1], l_run[1]);
  }
}

// One warp per output row (b, node, q head): merge the splits.
template <int D>
__global__ void __launch_bounds__(256) tree_attn_combine_kernel(const AttnParams p, int B) {
  constexpr int kPer = D / 32;
  const int warp = (blockIdx.x * 256 + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long total = (long)B * p.N_max * p.Hq;
  if (warp >= total) return;
  const int hq = warp % p.Hq;
  const int node = (warp / p.Hq) % p.N_max;
  const int b = warp / (p.Hq * p.N_max);
  uint16_t *dst = p.out + (size_t)warp * D + lane * kPer;

  int P, nb;
  const bool ok = seq_ok(p, b, P, nb) && node < nb;
  if (!ok) {
#pragma unroll
    for (int x = 0; x < kPer; ++x) dst[x] = 0;
    if (p.lse && lane == 0) p.lse[warp] = -INFINITY;
    return;
  }
  const int hkv = hq / p.g;
  const int row = node * p.g + (hq % p.g);
  const int z = b * p.Hkv + hkv;
  const int ns = (P + nb + p.chunk - 1) / p.chunk;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) {
    const float2 ml = p.part_ml[((size_t)z * p.splits + s) * p.rows_pad + row];
    M = fmaxf(M, ml.x);
  }
  float L = 0.f;
  float acc[kPer];
#pragma unroll
  for (int x = 0; x < kPer; ++x) acc[x] = 0.f;
  for (int s = 0; s < ns; ++s) {
    const size_t r = ((size_t)z * p.splits + s) * p.rows_pad + row;
    const float2 ml = p.part_ml[r];
    const float w = exp2f(ml.x - M);
    L += ml.y * w;
    const float *src = p.part_o + r * D + lane * kPer;
#pragma unroll
    for (int x = 0; x < kPer; ++x) acc[x] += src[x] * w;
  }
  const float inv = 1.f / L;
#pragma unroll
  for (int x = 0; x < kPer; ++x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(acc[x] * inv);
    dst[x] = *reinterpret_cast<const uint16_t *>(&h);
  }
  if (p.lse && lane == 0) p.lse[warp] = (M + log2f(L)) * 0.6931471805599453f;
}

struct AttnPlan {
  int row_tiles, rows_pad, splits, chunk;
  size_t o_bytes, ml_bytes;
};

AttnPlan plan_attn(int B, int N_max, int Hq, int Hkv, int D, int max_slots) {
  AttnPlan a;
  const int g = Hq / Hkv;
  a.row_tiles = (N_max * g + kBM - 1) / kBM;
  a.rows_pad = a.row_tiles * kBM;
  const long units = (long)B * Hkv * a.row_tiles;
  const long target = 2L * sm_count();
  long splits = (target + units - 1) / units;
  const long max_splits = (max_slots + kBN - 1) / kBN;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  long chunk = (max_slots + splits - 1) / splits;
  chunk = (chunk + kBN - 1) / kBN * kBN;
  if (chunk < kBN) chunk = kBN;
  a.chunk = (int)chunk;
  a.splits = (int)((max_slots + chunk - 1) / chunk);
  if (a.splits < 1) a.splits = 1;
  const size_t rows = (size_t)B * Hkv * a.splits * a.rows_pad;
  a.o_bytes = align_up(rows * D * sizeof(float), 256);
  a.ml_bytes = rows * sizeof(float2);
  return a;
}

template <int D>
int launch_attn(AttnParams &p, int B, cudaStream_t s) {
  const size_t smem = (size_t)(kBM + 4 * kBN) * D * 2;
  static unsigned long long configured = 0ull;  // one bit per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TSD_ERR_CUDA;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    if (cudaFuncSetAttribute(tree_attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return TSD_ERR_CUDA;
    configured |= bit;
  }
  dim3 grid(p.row_tiles, p.splits, B * p.Hkv);
  tree_attn_split_kernel<D><<<grid, kAttnThreads, smem, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return TSD_ERR_CUDA;
  const long rows = (long)B * p.N_max * p.Hq;
  const int blocks = (int)((rows * 32 + 255) / 256);
  tree_attn_combine_kernel<D><<<blocks, 256, 0, s>>>(p, B);
  return launch_status();
}

}  // namespace
}  // namespace tsd

static int attn_check_dims(int B, int N_max, int Hq, int Hkv, int D, int max_slots) {
  if (B < 0 || max_slots < 1) return TSD_ERR_ARG;
  if (N_max < 1 || N_max > tsd::kMaxNodes || (D != 64 && D != 128) || Hkv < 1 || Hq < Hkv ||
      Hq % Hkv != 0 || Hq / Hkv > 16 || B > 65535 || (long)B * Hkv > 65535)
    return TSD_ERR_LIMIT;
  return TSD_OK;
}

TSD_API size_t tsd_tree_attn_workspace_bytes(int B, int N_max, int Hq, int Hkv, int D,
                                             int max_slots) {
  if (attn_check_dims(B, N_max, Hq, Hkv, D, max_slots) != TSD_OK || B == 0) return 0;
  const tsd::AttnPlan a = tsd::plan_attn(B, N_max, Hq, Hkv, D, max_slots);
  return a.o_bytes + a.ml_bytes;
}

TSD_API int tsd_tree_attn_fwd(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                              const int32_t *block_table, int max_blocks, int num_blocks,
                              const int32_t *prefix_len, const int32_t *n_nodes,
                              const uint32_t *mask, const int32_t *err, int B, int N_max, int Hq,
                              int Hkv, int D, int max_slots, float scale, uint16_t *out,
                              float *lse, void *workspace, size_t ws_bytes, int32_t *status,
                              tsd_stream_t stream) {
  using namespace tsd;
  const int dims = attn_check_dims(B, N_max, Hq, Hkv, D, max_slots);
  if (dims != TSD_OK) return dims;
  if (B == 0) return TSD_OK;
  if (!q || !k_cache || !v_cache || !block_table || !prefix_len || !mask || !out)
    return TSD_ERR_ARG;
  if (max_blocks < 1 || num_blocks < 1 || !(scale > 0.f) || !std::isfinite(scale))
    return TSD_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return TSD_ERR_ARG;
  const AttnPlan a = plan_attn(B, N_max, Hq, Hkv, D, max_slots);
  if (!workspace || ws_bytes < a.o_bytes + a.ml_bytes || !aligned(workspace, 16))
    return TSD_ERR_WORKSPACE;
  AttnParams p;
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.table = block_table;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.prefix_len = prefix_len;
  p.n_nodes = n_nodes;
  p.mask = mask;
  p.err = err;
  p.N_max = N_max;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.W = (N_max + 31) / 32;
  p.max_slots = max_slots;
  p.scale_log2 = scale * kLog2e;
  p.chunk = a.chunk;
  p.splits = a.splits;
  p.row_tiles = a.row_tiles;
  p.rows_pad = a.rows_pad;
  p.part_o = static_cast<float *>(workspace);
  p.part_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + a.o_bytes);
  p.out = out;
  p.lse = lse;
  p.status = status;
  return D == 128 ? launch_attn<128>(p, B, as_cuda(stream)) : launch_attn<64>(p, B, as_cuda(stream));
}
